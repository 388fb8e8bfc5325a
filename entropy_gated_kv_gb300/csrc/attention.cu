// attention.cu — stage (d) of the EntropyCache step: bidirectional attention of the
// recompute rows against every cached K/V row, on the 5th-generation tensor cores.
//
// EntropyCache, gist.science pt summary §1 ("Atenção Bidirecional") and zh summary §1: dLLMs
// attend bidirectionally, so a recomputed row attends to all L positions, none masked; zh
// §2.2: the partial forward recomputes only the recompute set and reads the rest from the
// cache; pt §2: a full recompute refreshes every row (R = L: dense attention).
//   out[b, r, h] = sum_j softmax_j(scale <q[b, r, h], k[b, j, h/g]>) v[b, j, h/g],  r < R[b]
//
// Structure (one CTA per SM, persistent, 6 warps):
//   warp 0      TMA producer: the query tile once per work item, then K and V blocks of
//               128 keys into a 3-stage ring (128-byte swizzle, mbarrier transaction counts).
//   warp 1      allocates 512 TMEM columns; one lane issues tcgen05.mma: S = Q K^T into one
//               of three TMEM S buffers, and O += P V into the TMEM O accumulator with P read
//               from TMEM; completion is signalled with tcgen05.commit on mbarriers.
//   warps 2..5  softmax and epilogue, one TMEM lane (= one packed query row) per thread:
//               tcgen05.ld of the S row, online softmax in base 2 with a lazy rescale of O
//               (only when the running max grows by more than 2^8), P in bf16 written back
//               over the first half of the S buffer with tcgen05.st (no shared memory).
// Grouped-query attention packs the g = Hq / Hkv query heads of one KV head into the 128 MMA
// rows (floor(128 / g) query rows per tile), so K/V are read once per KV head.
// Work items (b, kv head, row tile, KV split) are derived on the device from R[], so the
// kernel needs no host synchronisation. CTAs are launched in clusters of 4. When there are
// no more row tiles than clusters (a partial step), the 4 CTAs of a cluster share one tile and
// each takes a quarter of the key range; each stages its unnormalised partial (O, running max,
// running sum) in its own shared memory; after a cluster barrier each CTA pushes every peer
// the 32 rows that peer merges with one bulk shared-to-shared copy (the async copy engine,
// completion counted on the peer's mbarrier), and merges its own 32 rows by log-sum-exp
// weights from local shared memory — the split-KV-then-merge idea of "Prefilling-dLLM"
// (gist.science pt summary, "Otimização de Kernel de Atenção"), with the merge kept on chip. Otherwise (a full step)
// every CTA works through whole tiles on its own.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "ec_common.cuh"
#include "ec_internal.h"

namespace ec {
namespace {

constexpr int kBlockM = 128;  // packed query rows per tile (TMEM lanes)
constexpr int kBlockN = 128;  // keys per KV block
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 512;
constexpr int kStages = 3;        // K/V blocks in flight, and S/P buffers in TMEM
constexpr uint32_t kTmemS = 0;    // S buffer i at columns [128 i, 128 i + 128); P (bf16) over its first 64
constexpr uint32_t kTmemO = 384;  // O accumulator at columns [384, 384 + D)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.f;
constexpr int kMaxGrid = 256;
constexpr int kCluster = 4;  // CTAs per cluster = KV splits of a shared tile
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per pipeline wait
// Operand descriptors: every tile is 128-byte swizzled with 8-row groups 1024 bytes apart. One
// K step of 16 keys / dims advances a K-major tile by 32 bytes within a 64-element atom (the
// next atom is 16 KB further), and the MN-major V tile by 16 rows of 128 bytes.
constexpr uint32_t kDescHi = sdesc_hi(1024);
__host__ __device__ constexpr uint32_t step_qk(int kk) { return (kk >> 2) * (128 * 128 / 16) + (kk & 3) * 2; }
constexpr uint32_t kStepPV = 16 * 128 / 16;

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[kStages], s_free[kStages];  // s_free: the PV product that read P from the buffer is done
  uint64_t p_full[kStages];
  uint64_t o_full, o_free;
  uint64_t recv;  // split merge: bytes pushed into this CTA by its cluster peers
  uint32_t tmem_base;
  int abort;
};

template <int D>
struct Layout {
  static constexpr int kAtoms = D / 64;                  // 64 bf16 = 128 bytes per swizzle row
  static constexpr int kAtomBytes = 128 * 128;           // 128 rows x 128 bytes
  static constexpr int kQBytes = kAtoms * kAtomBytes;
  static constexpr int kKVBytes = kAtoms * kAtomBytes;   // one of K or V for one block
  static constexpr int kStageBytes = 2 * kKVBytes;
  static constexpr int kQOff = 0;
  static constexpr int kStageOff = kQOff + kQBytes;
  static constexpr int kBarOff = kStageOff + kStages * kStageBytes;
  static constexpr int kBytes = kBarOff + static_cast<int>(sizeof(Bars));
  static constexpr int kDynSmem = kBytes + 1024;  // slack for 1024-byte alignment
};

struct Plan {
  int tiles;   // row tiles over all (b, kv head)
  int splits;  // key splits per tile
  int bps;     // KV blocks per split
  int nkv;     // KV blocks per sequence
  int r_lane;  // B <= 32: clamped R[lane] (0 past B), so items decode without reading R again
};

struct Item {
  int b, kvh, r0, nrows, kb0, nblk, kv_end, tile, split;
};

__device__ __forceinline__ int clamp_r(int r, int L) { return min(max(r, 0), L); }

__device__ __forceinline__ int warp_sum(int v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}

// Whole warp; every warp of every CTA computes the same plan. With no more tiles than
// clusters, each cluster shares one tile over kCluster key splits; otherwise no split.
__device__ Plan make_plan(const int32_t* R, int B, int L, int Lk, int Hkv, int nr, int nclusters) {
  const int lane = threadIdx.x & 31;
  int t = 0, r_lane = 0;
  for (int b = lane; b < B; b += 32) {
    const int rb = clamp_r(__ldcg(R + b), L);
    if (b == lane) r_lane = rb;
    t += Hkv * ((rb + nr - 1) / nr);
  }
  t = warp_sum(t);
  Plan p;
  p.r_lane = r_lane;
  p.tiles = t;
  p.nkv = (Lk + kBlockN - 1) / kBlockN;
  const int s = (t > 0 && t <= nclusters) ? min(kCluster, p.nkv) : 1;
  p.bps = (p.nkv + s - 1) / s;
  p.splits = (p.nkv + p.bps - 1) / p.bps;
  return p;
}

// The k-th work item of this CTA, or -1. Split plans give cluster c the tile c and its CTA of
// rank r the split r; unsplit plans deal tiles round-robin over all CTAs.
__device__ __forceinline__ int cta_item(int k, const Plan& pl, int cluster, int rank, int nclusters) {
  if (pl.splits > 1) return (k == 0 && cluster < pl.tiles && rank < pl.splits) ? cluster * pl.splits + rank : -1;
  const int item = static_cast<int>(blockIdx.x) + k * static_cast<int>(gridDim.x);
  return item < pl.tiles ? item : -1;
}

// Whole warp. Items are ordered (b, kv head, row tile, split).
__device__ Item decode_item(int item, const Plan& pl, const int32_t* R, int B, int L, int Lk, int Hkv, int nr) {
  const int lane = threadIdx.x & 31;
  Item it{};
  const int tile = item / pl.splits;
  it.tile = tile;
  it.split = item - tile * pl.splits;
  int base = 0;
  for (int b0 = 0; b0 < B; b0 += 32) {
    const int b = b0 + lane;
    const int rb = b >= B ? 0 : (B <= 32 ? pl.r_lane : clamp_r(__ldcg(R + b), L));
    const int tb = b < B ? Hkv * ((rb + nr - 1) / nr) : 0;
    int incl = tb;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (tile < base + total) {
      const unsigned hit = __ballot_sync(0xffffffffu, base + incl > tile);
      const int src = __ffs(hit) - 1;
      const int excl = __shfl_sync(0xffffffffu, incl - tb, src);
      const int rsel = __shfl_sync(0xffffffffu, rb, src);
      const int mt_count = (rsel + nr - 1) / nr;
      const int within = tile - base - excl;
      it.b = b0 + src;
      it.kvh = within / mt_count;
      const int mt = within - it.kvh * mt_count;
      it.r0 = mt * nr;
      it.nrows = min(nr, rsel - it.r0);
      break;
    }
    base += total;
  }
  it.kb0 = it.split * pl.bps;
  const int kb1 = min(pl.nkv, it.kb0 + pl.bps);
  it.nblk = kb1 - it.kb0;
  it.kv_end = min(Lk, kb1 * kBlockN);
  return it;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) attention_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, const int32_t* __restrict__ R, int B, int L, int Lk, int Hq, int Hkv, int g,
    int nr, float scale_log2, uint16_t* __restrict__ out, int32_t* __restrict__ dev_err, int plan_early) {
  using LY = Layout<D>;
  // A staged partial row: O as D bf16 (unnormalised; one more rounding than the fp32
  // accumulator, far below the output's own bf16 rounding after the merge), then the running
  // max and running sum as fp32, padded to 16 bytes.
  constexpr int kRowBytes = 2 * D + 16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + LY::kBarOff);
  uint8_t* q_smem = smem + LY::kQOff;
  // Split partials reuse the K/V stages once every CTA of the cluster is past its compute:
  // `send` holds this CTA's 128 partial rows, grouped by the peer that merges them; `recv`
  // holds the kBlockM / kCluster rows this CTA merges, one slice per peer.
  constexpr int kSliceRows = kBlockM / kCluster;
  constexpr uint32_t kSliceBytes = kSliceRows * kRowBytes;
  uint8_t* send = smem + LY::kStageOff;
  uint8_t* recv = send + kBlockM * kRowBytes;
  static_assert(LY::kStageOff + 2 * kBlockM * kRowBytes <= LY::kBarOff, "split buffers overlap barriers");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M_rows = nr * g;
  const int cluster = static_cast<int>(cluster_id_x());
  const int rank = static_cast<int>(cluster_ctarank());
  const int nclusters = static_cast<int>(cluster_count_x());

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
      mbar_init(&bars->s_full[i], 1);
      mbar_init(&bars->s_free[i], 1);
      mbar_init(&bars->p_full[i], 128);
    }
    mbar_init(&bars->o_full, 1);
    mbar_init(&bars->o_free, 128);
    mbar_init(&bars->recv, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort;

  // Everything above overlaps the previous kernel; Q and the cache are read after the wait.
  // Inside a step (plan_early) R was written by the select kernel, which finished before the
  // scatter kernel released this one, so the plan is made before the wait (R is read through
  // L2); standalone, R may come from the previous kernel.
  if (!plan_early) pdl_wait();
  const Plan pl = make_plan(R, B, L, Lk, Hkv, nr, nclusters);
  if (plan_early) pdl_wait();
  pdl_launch_dependents();
  const bool split_mode = pl.splits > 1;
  Item split_item{};  // the shared tile's item, kept by the softmax warps for the merge
  split_item.nrows = -1;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    uint32_t it = 0;
    for (int n = 0;; ++n) {
      const int item = cta_item(n, pl, cluster, rank, nclusters);
      if (item < 0) break;
      const Item I = decode_item(item, pl, R, B, L, Lk, Hkv, nr);
      int ok = 1;
      if (lane == 0) {
        if (n > 0) ok = mbar_wait_bounded(&bars->q_empty, (n - 1) & 1, abort_flag, dev_err, kWaitLimitNs);
        if (ok) {
          mbar_arrive_expect_tx(&bars->q_full, LY::kAtoms * M_rows * 128);
          for (int a = 0; a < LY::kAtoms; ++a)
            tma_load_5d(q_smem + a * LY::kAtomBytes, &tm_q, &bars->q_full, a * 64, 0, I.kvh, I.r0, I.b);
        }
        for (int j = 0; ok && j < I.nblk; ++j) {
          const uint32_t cur = it + j, slot = cur % kStages, u = cur / kStages;
          ok = mbar_wait_bounded(&bars->kv_empty[slot], (u & 1u) ^ 1u, abort_flag, dev_err, kWaitLimitNs);
          if (!ok) break;
          uint8_t* kst = smem + LY::kStageOff + slot * LY::kStageBytes;
          uint8_t* vst = kst + LY::kKVBytes;
          mbar_arrive_expect_tx(&bars->kv_full[slot], LY::kStageBytes);
          const int key0 = (I.kb0 + j) * kBlockN;
          for (int a = 0; a < LY::kAtoms; ++a)
            tma_load_4d(kst + a * LY::kAtomBytes, &tm_k, &bars->kv_full[slot], a * 64, I.kvh, key0, I.b);
          for (int a = 0; a < LY::kAtoms; ++a)
            tma_load_4d(vst + a * LY::kAtomBytes, &tm_v, &bars->kv_full[slot], a * 64, I.kvh, key0, I.b);
        }
      }
      it += I.nblk;
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kBlockN, 0);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 1);
    const uint32_t q_lo = sdesc_lo(smem_u32(q_smem), 16);
    uint32_t it = 0;
    for (int n = 0;; ++n) {
      const int item = cta_item(n, pl, cluster, rank, nclusters);
      if (item < 0) break;
      const Item I = decode_item(item, pl, R, B, L, Lk, Hkv, nr);
      int ok = 1;
      if (lane == 0) {
        ok = mbar_wait_bounded(&bars->q_full, n & 1, abort_flag, dev_err, kWaitLimitNs);
        for (int j = 0; ok && j <= I.nblk; ++j) {
          if (j < I.nblk) {
            const uint32_t cur = it + j, slot = cur % kStages, u = cur / kStages;
            ok = mbar_wait_bounded(&bars->kv_full[slot], u & 1u, abort_flag, dev_err, kWaitLimitNs) &&
                 mbar_wait_bounded(&bars->s_free[slot], (u & 1u) ^ 1u, abort_flag, dev_err, kWaitLimitNs);
            if (!ok) break;
            tc_fence_after();
            const uint32_t k_lo = sdesc_lo(smem_u32(smem + LY::kStageOff + slot * LY::kStageBytes), 16);
            const uint32_t s_col = tmem + kTmemS + slot * kBlockN;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk)
              umma_ss(s_col, q_lo + step_qk(kk), k_lo + step_qk(kk), kDescHi, idesc_qk, kk > 0 ? 1u : 0u);
            umma_commit(&bars->s_full[slot]);
            if (j == I.nblk - 1) umma_commit(&bars->q_empty);
          }
          if (j >= 1) {
            const uint32_t prev = it + j - 1, ps = prev % kStages, pu = prev / kStages;
            if (j == 1 && n > 0)
              ok = mbar_wait_bounded(&bars->o_free, (n - 1) & 1, abort_flag, dev_err, kWaitLimitNs);
            ok = ok && mbar_wait_bounded(&bars->p_full[ps], pu & 1u, abort_flag, dev_err, kWaitLimitNs);
            if (!ok) break;
            tc_fence_after();
            const uint32_t v_lo =
                sdesc_lo(smem_u32(smem + LY::kStageOff + ps * LY::kStageBytes + LY::kKVBytes), LY::kAtomBytes);
            const uint32_t p_col = tmem + kTmemS + ps * kBlockN;
            const uint32_t acc0 = j > 1 ? 1u : 0u;
#pragma unroll
            for (int kk = 0; kk < kBlockN / 16; ++kk)  // P: 16 keys = 8 TMEM columns per product
              umma_ts(tmem + kTmemO, p_col + kk * 8, v_lo + kk * kStepPV, kDescHi, idesc_pv, kk > 0 ? 1u : acc0);
            umma_commit(&bars->kv_empty[ps]);
            umma_commit(&bars->s_free[ps]);
            if (j == I.nblk) umma_commit(&bars->o_full);
          }
        }
      }
      it += I.nblk;
      if (!__shfl_sync(0xffffffffu, ok, 0)) break;
    }
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    const int row = 32 * (warp & 3) + lane;  // TMEM lane = packed query row
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    uint32_t it = 0;
    bool staged = false;
    for (int n = 0;; ++n) {
      const int item = cta_item(n, pl, cluster, rank, nclusters);
      if (item < 0) break;
      const Item I = decode_item(item, pl, R, B, L, Lk, Hkv, nr);
      if (split_mode) split_item = I;
      float m_used = -INFINITY, l_sum = 0.f;
      bool ok = true;
      for (int j = 0; j < I.nblk; ++j) {
        const uint32_t cur = it + j, slot = cur % kStages, u = cur / kStages;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars->s_full[slot], u & 1u, abort_flag, dev_err, kWaitLimitNs));
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[kBlockN];
#pragma unroll
        for (int c = 0; c < kBlockN / 32; ++c) EC_TMEM_LD32(tmem + lane_off + kTmemS + slot * kBlockN + c * 32, (sr + c * 32));
        tmem_wait_ld();

        // Row max of the raw scores (scale > 0 commutes with max), 8 independent chains.
        const int nvalid = min(kBlockN, I.kv_end - (I.kb0 + j) * kBlockN);
        if (nvalid < kBlockN) {  // ragged last block of the key range
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
        // p = 2^(s * scale * log2(e) - m_used); row sum over 8 independent chains.
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
        const float rs = ((rss[0] + rss[1]) + (rss[2] + rss[3])) + ((rss[4] + rss[5]) + (rss[6] + rss[7]));
        l_sum += rs;
        // P (bf16) over the first 64 columns of this S buffer: the PV product reads it from TMEM.
        EC_TMEM_ST32(tmem + lane_off + kTmemS + slot * kBlockN, pk);
        EC_TMEM_ST32(tmem + lane_off + kTmemS + slot * kBlockN + 32, (pk + 32));
        tmem_wait_st();
        // tcgen05.ld/st are warp-collective: the whole warp rescales when any of its rows
        // needs it (alpha = 1 for the others).
        if (__any_sync(0xffffffffu, rescale)) {
          // O holds the products of blocks 0 .. j-1; wait for the last of them (its buffer's
          // release), then scale.
          const uint32_t prev = cur - 1;
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars->s_free[prev % kStages], (prev / kStages) & 1u, abort_flag,
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
        mbar_arrive(&bars->p_full[slot]);
      }
      it += I.nblk;
      if (ok) ok = mbar_wait_bounded(&bars->o_full, n & 1, abort_flag, dev_err, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      if (!split_mode) {
        // Whole key range: normalise and write this row.
        const int rl = row / g, jh = row - rl * g;
        const bool valid_row = row < M_rows && rl < I.nrows;
        const float inv_l = 1.f / l_sum;
        uint16_t* orow = out + ((static_cast<int64_t>(I.b) * L + I.r0 + rl) * Hq + I.kvh * g + jh) * D;
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
      } else {
        // One split of a shared tile: stage the unnormalised partial for the cluster merge.
        // Every K/V load of this CTA has been consumed (o_full), so the stages are free.
        uint8_t* ro = send + row * kRowBytes;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          EC_TMEM_LD32(tmem + lane_off + kTmemO + c * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<uint4*>(ro + 2 * (c * 32 + 8 * q)) =
                make_uint4(pack_bf16x2(__uint_as_float(o[8 * q + 0]), __uint_as_float(o[8 * q + 1])),
                           pack_bf16x2(__uint_as_float(o[8 * q + 2]), __uint_as_float(o[8 * q + 3])),
                           pack_bf16x2(__uint_as_float(o[8 * q + 4]), __uint_as_float(o[8 * q + 5])),
                           pack_bf16x2(__uint_as_float(o[8 * q + 6]), __uint_as_float(o[8 * q + 7])));
        }
        reinterpret_cast<float*>(ro + 2 * D)[0] = m_used;
        reinterpret_cast<float*>(ro + 2 * D)[1] = l_sum;
        staged = true;
      }
      tc_fence_before();
      mbar_arrive(&bars->o_free);
    }
    if (split_mode && !staged) {  // no split of its own (or a failed one): contribute nothing
      reinterpret_cast<float*>(send + row * kRowBytes + 2 * D)[0] = -INFINITY;
      reinterpret_cast<float*>(send + row * kRowBytes + 2 * D)[1] = 0.f;
    }
    if (split_mode) fence_proxy_async_smem();  // the bulk copies below read `send`
  }

  // ---------------------------------------------------------------------- cluster merge
  if (split_mode) {
    if (threadIdx.x == 0) mbar_arrive_expect_tx(&bars->recv, (kCluster - 1) * kSliceBytes);
    cluster_sync_all();  // every CTA has staged its partial and armed its receive barrier
    if (threadIdx.x == 0) {
      // push each peer the slice of rows it merges (the own slice stays in `send`)
      for (int d = 1; d < kCluster; ++d) {
        const uint32_t dst = (rank + d) % kCluster;
        const uint32_t dst_recv = dsmem_map(smem_u32(recv + rank * kSliceBytes), dst);
        bulk_copy_s2cluster(dst_recv, send + dst * kSliceBytes, kSliceBytes,
                            dsmem_map(smem_u32(&bars->recv), dst));
      }
    }
    // The barrier that keeps every CTA alive until the pushes out of its `send` have landed is
    // split: a CTA's merging threads arrive once their own receive barrier is complete (every
    // push into them has finished reading its source), the others right away, and everyone
    // waits at teardown, so the barrier's latency overlaps the merge.
    if (warp < 2) cluster_arrive_release();
    if (warp >= 2) {
      const bool got = __all_sync(0xffffffffu, mbar_wait_bounded(&bars->recv, 0, abort_flag, dev_err, kWaitLimitNs));
      cluster_arrive_release();
      if (got && cluster < pl.tiles) {
        // the tile is shared by the cluster; CTAs without a split of their own decode it here
        const Item I = split_item.nrows >= 0 ? split_item : decode_item(cluster * pl.splits, pl, R, B, L, Lk, Hkv, nr);
        constexpr int kCols = D / 4;  // four threads per row, kCols columns each
        const int t = threadIdx.x - 64;
        const int srow = t >> 2;  // row within this CTA's slice
        const int prow = rank * kSliceRows + srow;
        const int col0 = (t & 3) * kCols;
        const uint8_t* src[kCluster];
#pragma unroll
        for (int sidx = 0; sidx < kCluster; ++sidx)
          src[sidx] = (sidx == rank) ? send + prow * kRowBytes : recv + (sidx * kSliceRows + srow) * kRowBytes;
        float wgt[kCluster], ls[kCluster];
        float mmax = -INFINITY;
#pragma unroll
        for (int sidx = 0; sidx < kCluster; ++sidx) {
          wgt[sidx] = reinterpret_cast<const float*>(src[sidx] + 2 * D)[0];
          ls[sidx] = reinterpret_cast<const float*>(src[sidx] + 2 * D)[1];
          if (ls[sidx] > 0.f) mmax = fmaxf(mmax, wgt[sidx]);
        }
        float lsum = 0.f;
#pragma unroll
        for (int sidx = 0; sidx < kCluster; ++sidx) {
          wgt[sidx] = ls[sidx] > 0.f ? ex2_approx(wgt[sidx] - mmax) : 0.f;  // weight of split sidx
          lsum = fmaf(wgt[sidx], ls[sidx], lsum);
        }
        const float inv_l = 1.f / lsum;
        float acc[kCols];
#pragma unroll
        for (int e = 0; e < kCols; ++e) acc[e] = 0.f;
#pragma unroll
        for (int sidx = 0; sidx < kCluster; ++sidx) {
          if (wgt[sidx] == 0.f) continue;  // an empty split may hold stale values
          const uint4* o8 = reinterpret_cast<const uint4*>(src[sidx] + 2 * col0);
#pragma unroll
          for (int q = 0; q < kCols / 8; ++q) {
            const uint4 v = o8[q];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              acc[8 * q + 2 * e] = fmaf(wgt[sidx], bf16lo_to_f32(w[e]), acc[8 * q + 2 * e]);
              acc[8 * q + 2 * e + 1] = fmaf(wgt[sidx], bf16hi_to_f32(w[e]), acc[8 * q + 2 * e + 1]);
            }
          }
        }
        const int rl = prow / g, jh = prow - rl * g;
        if (prow < M_rows && rl < I.nrows && !*abort_flag) {
          uint16_t* orow = out + ((static_cast<int64_t>(I.b) * L + I.r0 + rl) * Hq + I.kvh * g + jh) * D + col0;
#pragma unroll
          for (int q = 0; q < kCols / 8; ++q) {
            uint4 v;
            v.x = pack_bf16x2(acc[8 * q + 0] * inv_l, acc[8 * q + 1] * inv_l);
            v.y = pack_bf16x2(acc[8 * q + 2] * inv_l, acc[8 * q + 3] * inv_l);
            v.z = pack_bf16x2(acc[8 * q + 4] * inv_l, acc[8 * q + 5] * inv_l);
            v.w = pack_bf16x2(acc[8 * q + 6] * inv_l, acc[8 * q + 7] * inv_l);
            *reinterpret_cast<uint4*>(orow + 8 * q) = v;
          }
        }
      }
    }
    cluster_wait_acquire();  // every push out of this CTA has landed before it leaves
  }

  // ---------------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------------- host

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
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

bool encode_map(EncodeTiledFn enc, CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                const cuuint64_t* strides_bytes, const cuuint32_t* box) {
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base),
                         dims, strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_impl(const ec_params& p, const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* R, float scale, void* out, void* ws, int32_t* dev_err, bool plan_early,
                        cudaStream_t s, ec_status* status) {
  using LY = Layout<D>;
  EncodeTiledFn enc = get_encode_fn();
  if (enc == nullptr) {
    *status = EC_ERR_CUDA;
    return cudaErrorNotSupported;
  }
  const int g = p.Hq / p.Hkv;
  const int nr = kBlockM / g;
  CUtensorMap tq, tk, tv;
  const cuuint64_t qd[5] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(g), static_cast<cuuint64_t>(p.Hkv),
                            static_cast<cuuint64_t>(p.L), static_cast<cuuint64_t>(p.B)};
  const cuuint64_t qs[4] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(g) * D * 2,
                            static_cast<cuuint64_t>(p.Hq) * D * 2, static_cast<cuuint64_t>(p.L) * p.Hq * D * 2};
  const cuuint32_t qb[5] = {64, static_cast<cuuint32_t>(g), 1, static_cast<cuuint32_t>(nr), 1};
  // keys [0, Lk): the whole cache, or up to the end of the gate's scope (block-causal); rows
  // past Lk read as zeros through the map and are masked out of the softmax
  const int Lk = scope_hi(p);
  const cuuint64_t kd[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(p.Hkv), static_cast<cuuint64_t>(Lk),
                            static_cast<cuuint64_t>(p.B)};
  const cuuint64_t ks[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(p.Hkv) * D * 2,
                            static_cast<cuuint64_t>(p.L) * p.Hkv * D * 2};
  const cuuint32_t kb[4] = {64, 1, static_cast<cuuint32_t>(kBlockN), 1};
  if (!encode_map(enc, &tq, q, 5, qd, qs, qb) || !encode_map(enc, &tk, k_cache, 4, kd, ks, kb) ||
      !encode_map(enc, &tv, v_cache, 4, kd, ks, kb)) {
    *status = EC_ERR_INVALID_ARG;
    return cudaErrorInvalidValue;
  }
  // Clusters of kCluster CTAs, one CTA per SM (shared memory bound), as many clusters as
  // fit on the device at once (the kernel is persistent); counted once per device and head size.
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = LY::kDynSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;  // the occupancy query sees the cluster shape only
  int mc = 0;
  cudaError_t e = cached_per_device(
      D, &mc,
      [](int* n_out, void* ctx) -> cudaError_t {
        cudaLaunchConfig_t* c = static_cast<cudaLaunchConfig_t*>(ctx);
        int sms = 0;
        cudaError_t r = current_device_sms(&sms);
        if (r == cudaSuccess)
          r = cudaFuncSetAttribute(attention_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, LY::kDynSmem);
        if (r != cudaSuccess) return r;
        c->gridDim = dim3(std::min(sms, kMaxGrid) / kCluster * kCluster);
        int n = 0;
        r = cudaOccupancyMaxActiveClusters(&n, attention_kernel<D>, c);
        if (r != cudaSuccess) return r;
        if (n < 1) return cudaErrorInvalidConfiguration;
        *n_out = std::min(n, kMaxGrid / kCluster);
        return cudaSuccess;
      },
      &cfg);
  if (e != cudaSuccess) {
    *status = EC_ERR_CUDA;
    return e;
  }
  cfg.gridDim = dim3(mc * kCluster);
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, attention_kernel<D>, tq, tk, tv, R, p.B, p.L, Lk, p.Hq, p.Hkv, g, nr, scale * kLog2e,
                         static_cast<uint16_t*>(out), dev_err, plan_early ? 1 : 0);
  if (e != cudaSuccess) *status = EC_ERR_CUDA;
  return e;
}

}  // namespace

size_t attention_workspace_bytes(const ec_params& p) {
  (void)p;
  return 256;  // the split merge runs on chip; the workspace is reserved for future use
}

cudaError_t launch_partial_attention(const ec_params& p, const void* q, const void* k_cache,
                                     const void* v_cache, const int32_t* R, float scale, void* out, void* ws,
                                     int32_t* dev_err, bool plan_early, cudaStream_t s, ec_status* status) {
  *status = EC_OK;
  if (p.D == 128) return launch_impl<128>(p, q, k_cache, v_cache, R, scale, out, ws, dev_err, plan_early, s, status);
  return launch_impl<64>(p, q, k_cache, v_cache, R, scale, out, ws, dev_err, plan_early, s, status);
}

}  // namespace ec
