// attention_pair.cu — dense bidirectional attention for a full recompute step (every position
// attends to every cached key), on pairs of SMs with the 2-CTA tensor-core products.
//
// EntropyCache, gist.science pt summary §2 ("Decisão de Pulo"): a step whose decoded tokens are
// too uncertain recomputes every position; pt §1 ("Atenção Bidirecional") and zh §1: dLLMs attend
// bidirectionally, so no mask. The first forward of a generation block is full by definition,
// so the caller knows these steps ahead; ec_dense_attention serves them.
//   out[b, r, h] = sum_j softmax_j(scale <q[b, r, h], k[b, j, h/g]>) v[b, j, h/g],  r, j < L
//
// Why pairs: one CTA per SM with a single MMA-issuing thread spends its block period issuing
// products and waiting for its own 64 KB K/V stage. Here a cluster of 2 CTAs takes two 128-row
// tiles of one (sequence, KV head), and the leader's MMA thread issues M = 256 products
// (tcgen05.mma.cta_group::2): A (the queries, or P from tensor memory) is split by rows, each CTA
// supplying its own tile, and B (K, or V) by columns, each CTA loading half of every K/V block
// (64 keys of K, 64 of the 128 dims of V). So each issued product covers both tiles, and each SM
// streams half the K/V bytes per tile.
// Roles per CTA (6 warps):
//   warp 0      TMA: this CTA's query tile once per item, its halves of K and V per block of 128
//               keys, into a ring of stages; the loads complete on the leader's barriers (the
//               .cta_group::2 load form), which count the bytes of both CTAs.
//   warp 1      allocates 512 TMEM columns (both CTAs, one collective allocation); in the leader,
//               one lane issues S = Q K^T into a TMEM S buffer and O += P V with P read from
//               TMEM, and commits to barriers in both CTAs at once (multicast).
//   warps 2..5  softmax and epilogue for this CTA's 128 rows, as in the partial-attention kernel
//               (one TMEM lane per row, lazy rescale, P written over the S buffer); each warp tells
//               the leader when its P rows (and, per item, its O rows) are done: in the leader
//               directly, in the peer through a local barrier whose completion the peer's warp 1
//               forwards with one remote arrival (cheaper than four warps arriving remotely).
// GQA packs the g query heads of a KV head into the 128 rows (floor(128 / g) positions per tile).
// Every wait is bounded and reports EC_DEVERR_TIMEOUT.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "ec_common.cuh"
#include "ec_internal.h"

namespace ec {
namespace {

constexpr int D = 128;           // head size (V is split by dims over the pair: 64 each)
constexpr int kBlockM = 128;     // packed query rows per CTA tile (TMEM lanes)
constexpr int kBlockN = 128;     // keys per block
constexpr int kHalfN = 64;       // keys of K (and dims of V) each CTA loads per block
constexpr int kThreads = 192;    // warp 0 TMA, warp 1 MMA (the peer's: P relay), warps 2-5 softmax + epilogue
constexpr uint32_t kTmemCols = 512;
constexpr int kSBuf = 3;         // S/P buffers in TMEM
constexpr int kKvStages = 5;     // K/V stages in shared memory
constexpr uint32_t kTmemO = 384;  // O accumulator at columns [384, 512)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.f;
constexpr int kMaxClusters = 128;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per pipeline wait
constexpr uint16_t kPairMask = 3;                 // both CTAs of the pair

constexpr int kAtomBytes = 128 * 128;             // 128 rows x 128 bytes (64 bf16)
constexpr int kQBytes = 2 * kAtomBytes;           // 128 query rows x 128 dims
constexpr int kKHalfBytes = 2 * (kHalfN * 128);   // 64 keys x 128 dims, two 64-dim atoms of 8 KB
constexpr int kVHalfBytes = kBlockN * 128;        // 128 keys x 64 dims, one atom
constexpr int kStageBytes = kKHalfBytes + kVHalfBytes;
constexpr int kQOff = 0;
constexpr int kStageOff = kQBytes;
constexpr int kBarOff = kStageOff + kKvStages * kStageBytes;

struct Bars {
  uint64_t q_full, q_empty;                      // q_full: leader only (both tiles' bytes)
  uint64_t kv_full[kKvStages], kv_empty[kKvStages];  // kv_full: leader only (both halves' bytes)
  uint64_t s_full[kSBuf], s_free[kSBuf];
  uint64_t p_full[kSBuf];                        // leader only: its 4 softmax warps + the peer's relay
  uint64_t o_full, o_free;                       // o_free: leader only: its 4 softmax warps + the peer's relay
  uint64_t p_local[kSBuf], o_local;              // peer only: its 4 softmax warps, relayed to the leader
  uint32_t tmem_base;
  int abort;
};
constexpr int kDynSmem = kBarOff + static_cast<int>(sizeof(Bars)) + 1024;  // + slack for 1024-byte alignment
static_assert(kDynSmem <= 227 * 1024, "shared memory");

// One K step (16 keys or 16 dims) of the operand tiles: the query tile's atoms are 16 KB apart,
// the K half's 8 KB; within an atom a step is 32 bytes. The V half advances 16 rows of 128 bytes.
__host__ __device__ constexpr uint32_t step_q(int kk) { return (kk >> 2) * (kAtomBytes / 16) + (kk & 3) * 2; }
__host__ __device__ constexpr uint32_t step_k(int kk) { return (kk >> 2) * (kHalfN * 128 / 16) + (kk & 3) * 2; }
constexpr uint32_t kStepPV = 16 * 128 / 16;
constexpr uint32_t kDescHi = sdesc_hi(1024);

EC_DEV void umma_ss_pair(uint32_t d_tmem, uint32_t a_lo, uint32_t b_lo, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 da, db;\n\t"
      "mov.b64 da, {%1, %3};\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], da, db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_lo), "r"(b_lo), "r"(kDescHi), "r"(idesc), "r"(accumulate)
      : "memory");
}

EC_DEV void umma_ts_pair(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_lo, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t.reg .b64 db;\n\t"
      "mov.b64 db, {%2, %3};\n\t"
      "setp.ne.b32 p, %5, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], [%1], db, %4, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "r"(b_lo), "r"(kDescHi), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` in both CTAs of the pair when the leader's tensor-core work issued so far
// is done.
EC_DEV void commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(kPairMask)
      : "memory");
}

// A tile load that completes on a barrier of either CTA of the pair (cluster address).
EC_DEV void tma_pair_4d(void* dst, const CUtensorMap* tm, uint32_t bar, int c0, int c1, int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
EC_DEV void tma_pair_5d(void* dst, const CUtensorMap* tm, uint32_t bar, int c0, int c1, int c2, int c3, int c4) {
  asm volatile(
      "cp.async.bulk.tensor.5d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6, %7}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(c4)
      : "memory");
}

// A bounded wait on a barrier of this CTA that the peer CTA also completes (its loads' bytes or
// its warps' arrivals): acquire at cluster scope. Gives up like mbar_wait_bounded.
EC_DEV bool try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
EC_DEV bool wait_cluster_bounded(uint64_t* bar, uint32_t parity, volatile int* abort, int32_t* dev_err) {
  if (try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (try_wait_cluster(bar, parity)) return true;
    if ((i & 63u) == 0u) {
      if (*abort) return false;
      if (global_timer_ns() - t0 > kWaitLimitNs) {
        *abort = 1;
        report_error(dev_err, EC_DEVERR_TIMEOUT);
        return false;
      }
    }
  }
}

// One arrival of a warp that has finished its rows (lane 0, after the warp's preceding
// tensor-memory stores were fenced): in the leader on the leader's barrier; in the peer on the
// peer's local barrier, which the peer's relay thread forwards to the leader with one remote
// arrival (the warps' own arrivals stay local and cheap; release/acquire order is transitive).
EC_DEV void arrive_done(uint64_t* leader_bar, uint64_t* local_bar, uint32_t rank) {
  mbar_arrive(rank == 0 ? leader_bar : local_bar);
}
EC_DEV void arrive_remote_leader(uint64_t* bar) {
  const uint32_t remote = dsmem_map(smem_u32(bar), 0);
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(remote) : "memory");
}

struct PairItem {
  int b, kvh, tile;  // this CTA's tile
  bool live;         // the tile exists (an odd tile count leaves the last pair's second CTA idle)
  int ld_tile;       // the tile whose queries this CTA loads (its own, or a live one when idle)
};

// Items are pairs of tiles of one (b, kv head): (b, kvh, pair) in that order.
__device__ __forceinline__ PairItem pair_item(int item, int pairs_per_head, int tiles_per_head, int Hkv, int rank) {
  PairItem it;
  const int bh = item / pairs_per_head;
  const int pr = item - bh * pairs_per_head;
  it.b = bh / Hkv;
  it.kvh = bh - it.b * Hkv;
  it.tile = 2 * pr + rank;
  it.live = it.tile < tiles_per_head;
  it.ld_tile = it.live ? it.tile : tiles_per_head - 1;
  return it;
}

__global__ void __launch_bounds__(kThreads, 1) pair_attention_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, int B, int L, int Hq, int Hkv, int g, int nr, float scale_log2,
    uint16_t* __restrict__ out, int32_t* __restrict__ dev_err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  uint8_t* q_smem = smem + kQOff;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cluster = static_cast<int>(cluster_id_x());
  const int nclusters = static_cast<int>(cluster_count_x());
  const int M_rows = nr * g;
  const int tiles_per_head = (L + nr - 1) / nr;
  const int pairs_per_head = (tiles_per_head + 1) / 2;
  const int n_items = B * Hkv * pairs_per_head;
  const int nblk = (L + kBlockN - 1) / kBlockN;

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int i = 0; i < kKvStages; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
    }
    for (int i = 0; i < kSBuf; ++i) {
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], 1);
      mbar_init(&bars->p_full[i], 5);
      mbar_init(&bars->p_local[i], 4);
    }
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_free, 5);
    mbar_init(&bars->o_local, 4);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 1) {  // one collective allocation of the pair (both CTAs' warp 1)
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&bars->tmem_base)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  cluster_sync_all();  // both CTAs' barriers are initialised before any load or commit reaches them
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort;
  pdl_wait();  // queries and cache may come from the previous kernels in the stream
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t q_full_l = dsmem_map(smem_u32(&bars->q_full), 0);
      bool ok = true;
      uint32_t it = 0;
      for (int n = 0; ok; ++n) {
        const int item = cluster + n * nclusters;
        if (item >= n_items) break;
        const PairItem I = pair_item(item, pairs_per_head, tiles_per_head, Hkv, rank);
        if (n > 0) ok = mbar_wait_bounded(&bars->q_empty, (n - 1) & 1, abort_flag, dev_err, kWaitLimitNs);
        if (!ok) break;
        if (rank == 0) mbar_arrive_expect_tx(&bars->q_full, 2 * 2 * M_rows * 128);  // both tiles, two atoms
        for (int a = 0; a < 2; ++a)
          tma_pair_5d(q_smem + a * kAtomBytes, &tm_q, q_full_l, a * 64, 0, I.kvh, I.ld_tile * nr, I.b);
        for (int j = 0; j < nblk; ++j) {
          const uint32_t cur = it + j, st = cur % kKvStages, u = cur / kKvStages;
          ok = mbar_wait_bounded(&bars->kv_empty[st], (u & 1u) ^ 1u, abort_flag, dev_err, kWaitLimitNs);
          if (!ok) break;
          uint8_t* kst = smem + kStageOff + st * kStageBytes;
          uint8_t* vst = kst + kKHalfBytes;
          const uint32_t full_l = dsmem_map(smem_u32(&bars->kv_full[st]), 0);
          if (rank == 0) mbar_arrive_expect_tx(&bars->kv_full[st], 2 * kStageBytes);
          const int key0 = j * kBlockN;
          for (int a = 0; a < 2; ++a)  // K: keys [key0 + 64 rank, + 64), both 64-dim atoms
            tma_pair_4d(kst + a * (kHalfN * 128), &tm_k, full_l, a * 64, I.kvh, key0 + kHalfN * static_cast<int>(rank), I.b);
          // V: keys [key0, + 128), dims [64 rank, + 64)
          tma_pair_4d(vst, &tm_v, full_l, 64 * static_cast<int>(rank), I.kvh, key0, I.b);
        }
        it += nblk;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (leader)
    if (rank == 0 && lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(256, kBlockN, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(256, D, 1);
      const uint32_t q_lo = sdesc_lo(smem_u32(q_smem), 16);
      // S runs kAhead blocks ahead of PV: QK(j + kAhead) is issued right after PV(j), so the
      // softmax of the next blocks never waits for the handshake of the current one (its S
      // buffer is the one PV(j - 1) released).
      constexpr int kAhead = kSBuf - 1;
      bool ok = true;
      uint32_t it = 0;
      auto issue_qk = [&](int j) -> bool {  // block j of the current item (global block it + j)
        const uint32_t cur = it + j, st = cur % kKvStages, ku = cur / kKvStages;
        const uint32_t sb = cur % kSBuf, su = cur / kSBuf;
        if (!(wait_cluster_bounded(&bars->kv_full[st], ku & 1u, abort_flag, dev_err) &&
              mbar_wait_bounded(&bars->s_free[sb], (su & 1u) ^ 1u, abort_flag, dev_err, kWaitLimitNs)))
          return false;
        tc_fence_after();
        const uint32_t k_lo = sdesc_lo(smem_u32(smem + kStageOff + st * kStageBytes), 16);
        const uint32_t s_col = tmem + sb * kBlockN;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss_pair(s_col, q_lo + step_q(kk), k_lo + step_k(kk), idesc_qk, kk > 0 ? 1u : 0u);
        commit_pair(&bars->s_full[sb]);
        if (j == nblk - 1) commit_pair(&bars->q_empty);  // the item's queries are no longer read
        return true;
      };
      for (int n = 0; ok; ++n) {
        const int item = cluster + n * nclusters;
        if (item >= n_items) break;
        ok = wait_cluster_bounded(&bars->q_full, n & 1, abort_flag, dev_err);
        for (int j = 0; ok && j < kAhead && j < nblk; ++j) ok = issue_qk(j);
        for (int j = 0; ok && j < nblk; ++j) {
          const uint32_t cur = it + j, pst = cur % kKvStages;
          const uint32_t psb = cur % kSBuf, psu = cur / kSBuf;
          if (j == 0 && n > 0) ok = wait_cluster_bounded(&bars->o_free, (n - 1) & 1, abort_flag, dev_err);
          ok = ok && wait_cluster_bounded(&bars->p_full[psb], psu & 1u, abort_flag, dev_err);
          if (!ok) break;
          tc_fence_after();
          const uint32_t v_lo = sdesc_lo(smem_u32(smem + kStageOff + pst * kStageBytes + kKHalfBytes), kAtomBytes);
          const uint32_t p_col = tmem + psb * kBlockN;
#pragma unroll
          for (int kk = 0; kk < kBlockN / 16; ++kk)  // P: 16 keys = 8 TMEM columns per product
            umma_ts_pair(tmem + kTmemO, p_col + kk * 8, v_lo + kk * kStepPV, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
          commit_pair(&bars->kv_empty[pst]);
          commit_pair(&bars->s_free[psb]);
          if (j == nblk - 1) commit_pair(&bars->o_full);
          if (j + kAhead < nblk) ok = issue_qk(j + kAhead);
        }
        it += nblk;
      }
      if (!ok) {  // tell the peer to stop waiting
        *abort_flag = 1;
        const uint32_t peer_abort = dsmem_map(smem_u32(&bars->abort), 1);
        asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(peer_abort), "r"(1) : "memory");
      }
    } else if (rank == 1 && lane == 0) {
      // relay: the peer's softmax warps finished a block's P (or an item's O): one remote arrival
      bool ok = true;
      uint32_t it = 0;
      for (int n = 0; ok; ++n) {
        const int item = cluster + n * nclusters;
        if (item >= n_items) break;
        for (int j = 0; ok && j < nblk; ++j) {
          const uint32_t cur = it + j, sb = cur % kSBuf, su = cur / kSBuf;
          ok = mbar_wait_bounded(&bars->p_local[sb], su & 1u, abort_flag, dev_err, kWaitLimitNs);
          if (ok) arrive_remote_leader(&bars->p_full[sb]);
        }
        it += nblk;
        ok = ok && mbar_wait_bounded(&bars->o_local, n & 1, abort_flag, dev_err, kWaitLimitNs);
        if (ok) arrive_remote_leader(&bars->o_free);
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    const int row = 32 * (warp & 3) + lane;  // TMEM lane = packed query row of this CTA's tile
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    uint32_t it = 0;
    for (int n = 0;; ++n) {
      const int item = cluster + n * nclusters;
      if (item >= n_items) break;
      const PairItem I = pair_item(item, pairs_per_head, tiles_per_head, Hkv, rank);
      float m_used = -INFINITY, l_sum = 0.f;
      bool ok = true;
      for (int j = 0; j < nblk; ++j) {
        const uint32_t cur = it + j, sb = cur % kSBuf, su = cur / kSBuf;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars->s_full[sb], su & 1u, abort_flag, dev_err, kWaitLimitNs));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[kBlockN];
#pragma unroll
        for (int c = 0; c < kBlockN / 32; ++c) EC_TMEM_LD32(tmem + lane_off + sb * kBlockN + c * 32, (sr + c * 32));
        tmem_wait_ld();
        const int nvalid = min(kBlockN, L - j * kBlockN);
        if (nvalid < kBlockN) {  // ragged last block
#pragma unroll
          for (int c = 0; c < kBlockN; ++c)
            if (c >= nvalid) sr[c] = __float_as_uint(-INFINITY);
        }
        float mxs[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mxs[e] = __uint_as_float(sr[e]);
#pragma unroll
        for (int c = 8; c < kBlockN; c += 8)
#pragma unroll
          for (int e = 0; e < 8; ++e) mxs[e] = fmaxf(mxs[e], __uint_as_float(sr[c + e]));
        const float mx = fmaxf(fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])),
                               fmaxf(fmaxf(mxs[4], mxs[5]), fmaxf(mxs[6], mxs[7]))) * scale_log2;
        bool rescale = false;
        float alpha = 1.f;
        if (j == 0) {
          m_used = mx;
        } else if (mx > m_used + kRescaleLog2) {
          alpha = ex2_approx(m_used - mx);
          m_used = mx;
          l_sum *= alpha;
          rescale = true;
        }
        const float neg_m = -m_used;
        float rss[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) rss[e] = 0.f;
        uint32_t pk[kBlockN / 2];
#pragma unroll
        for (int c = 0; c < kBlockN; c += 2) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(sr[c]), scale_log2, neg_m));
          const float p1 = ex2_approx(fmaf(__uint_as_float(sr[c + 1]), scale_log2, neg_m));
          rss[(c >> 1) & 7] += p0 + p1;
          pk[c / 2] = pack_bf16x2(p0, p1);
        }
        l_sum += ((rss[0] + rss[1]) + (rss[2] + rss[3])) + ((rss[4] + rss[5]) + (rss[6] + rss[7]));
        EC_TMEM_ST32(tmem + lane_off + sb * kBlockN, pk);
        EC_TMEM_ST32(tmem + lane_off + sb * kBlockN + 32, (pk + 32));
        tmem_wait_st();
        if (__any_sync(0xffffffffu, rescale)) {
          // O holds the products of blocks 0 .. j-1: wait for the last of them, then scale
          const uint32_t prev = cur - 1;
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars->s_free[prev % kSBuf], (prev / kSBuf) & 1u, abort_flag,
                                                         dev_err, kWaitLimitNs));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            EC_TMEM_LD32(tmem + lane_off + kTmemO + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            EC_TMEM_ST32(tmem + lane_off + kTmemO + c * 32, o);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) arrive_done(&bars->p_full[sb], &bars->p_local[sb], rank);
      }
      it += nblk;
      if (ok) ok = mbar_wait_bounded(&bars->o_full, n & 1, abort_flag, dev_err, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      const int rl = row / g, jh = row - rl * g;
      const int pos = I.tile * nr + rl;
      const bool valid_row = I.live && row < M_rows && pos < L;
      const float inv_l = 1.f / l_sum;
      uint16_t* orow = out + ((static_cast<int64_t>(I.b) * L + pos) * Hq + I.kvh * g + jh) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        EC_TMEM_LD32(tmem + lane_off + kTmemO + c * 32, o);
        tmem_wait_ld();
        if (valid_row) {
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint4 v;
            v.x = pack_bf16x2(__uint_as_float(o[8 * q + 0]) * inv_l, __uint_as_float(o[8 * q + 1]) * inv_l);
            v.y = pack_bf16x2(__uint_as_float(o[8 * q + 2]) * inv_l, __uint_as_float(o[8 * q + 3]) * inv_l);
            v.z = pack_bf16x2(__uint_as_float(o[8 * q + 4]) * inv_l, __uint_as_float(o[8 * q + 5]) * inv_l);
            v.w = pack_bf16x2(__uint_as_float(o[8 * q + 6]) * inv_l, __uint_as_float(o[8 * q + 7]) * inv_l);
            *reinterpret_cast<uint4*>(orow + c * 32 + 8 * q) = v;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) arrive_done(&bars->o_free, &bars->o_local, rank);
    }
  }

  // ---------------------------------------------------------------------- teardown
  tc_fence_before();
  cluster_sync_all();  // no product of the pair is pending and no CTA still reads its TMEM
  if (warp == 1) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

// ---------------------------------------------------------------------------------- host

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

bool encode(EncodeTiledFn enc, CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
            const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  const cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims,
             strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_dense_attention(const ec_params& p, const void* q, const void* k_cache, const void* v_cache,
                                   float scale, void* out, int32_t* dev_err, cudaStream_t s, ec_status* status) {
  *status = EC_OK;
  if (p.D != D) {
    *status = EC_ERR_UNSUPPORTED;
    return cudaErrorInvalidValue;
  }
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) {
    *status = EC_ERR_CUDA;
    return cudaErrorNotSupported;
  }
  const int g = p.Hq / p.Hkv;
  const int nr = kBlockM / g;
  CUtensorMap tq, tk, tv;
  // queries [B, L, Hkv, g, D] (the g heads of a KV head are adjacent), box {64 dims, g, 1, nr, 1}
  const cuuint64_t qd[5] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(g), static_cast<cuuint64_t>(p.Hkv),
                            static_cast<cuuint64_t>(p.L), static_cast<cuuint64_t>(p.B)};
  const cuuint64_t qs[4] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(g) * D * 2,
                            static_cast<cuuint64_t>(p.Hq) * D * 2, static_cast<cuuint64_t>(p.L) * p.Hq * D * 2};
  const cuuint32_t qb[5] = {64, static_cast<cuuint32_t>(g), 1, static_cast<cuuint32_t>(nr), 1};
  // cache [B, L, Hkv, D]: K in boxes of 64 keys x 64 dims, V in boxes of 128 keys x 64 dims
  const cuuint64_t kd[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(p.Hkv), static_cast<cuuint64_t>(p.L),
                            static_cast<cuuint64_t>(p.B)};
  const cuuint64_t ks[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(p.Hkv) * D * 2,
                            static_cast<cuuint64_t>(p.L) * p.Hkv * D * 2};
  const cuuint32_t kb[4] = {64, 1, static_cast<cuuint32_t>(kHalfN), 1};
  const cuuint32_t vb[4] = {64, 1, static_cast<cuuint32_t>(kBlockN), 1};
  if (!encode(enc, &tq, q, 5, qd, qs, qb) || !encode(enc, &tk, k_cache, 4, kd, ks, kb) ||
      !encode(enc, &tv, v_cache, 4, kd, ks, vb)) {
    *status = EC_ERR_INVALID_ARG;
    return cudaErrorInvalidValue;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kDynSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;  // the occupancy query sees the cluster shape only
  int mc = 0;
  cudaError_t e = cached_per_device(
      1000 + D, &mc,
      [](int* n_out, void* ctx) -> cudaError_t {
        cudaLaunchConfig_t* c = static_cast<cudaLaunchConfig_t*>(ctx);
        int sms = 0;
        cudaError_t r = current_device_sms(&sms);
        if (r == cudaSuccess)
          r = cudaFuncSetAttribute(pair_attention_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
        if (r != cudaSuccess) return r;
        c->gridDim = dim3(std::min(sms, 2 * kMaxClusters) / 2 * 2);
        int n = 0;
        r = cudaOccupancyMaxActiveClusters(&n, pair_attention_kernel, c);
        if (r != cudaSuccess) return r;
        if (n < 1) return cudaErrorInvalidConfiguration;
        *n_out = std::min(n, kMaxClusters);
        return cudaSuccess;
      },
      &cfg);
  if (e != cudaSuccess) {
    *status = EC_ERR_CUDA;
    return e;
  }
  const int64_t items = static_cast<int64_t>(p.B) * p.Hkv * (((p.L + nr - 1) / nr + 1) / 2);
  const int nclusters = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(mc, items)));
  cfg.gridDim = dim3(2 * nclusters);
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, pair_attention_kernel, tq, tk, tv, p.B, p.L, p.Hq, p.Hkv, g, nr, scale * kLog2e,
                         static_cast<uint16_t*>(out), dev_err);
  if (e != cudaSuccess) *status = EC_ERR_CUDA;
  return e;
}

}  // namespace ec
