// attention_dense.cu — dense bidirectional attention for a full recompute step (every position
// attends to every cached key), two query tiles per CTA with a softmax warpgroup per tile.
//
// EntropyCache, gist.science pt summary §2 ("Decisão de Pulo"): a step whose decoded tokens are
// too uncertain recomputes every position; pt §1 ("Atenção Bidirecional") and zh §1: dLLMs attend
// bidirectionally, so no mask. The first forward of a generation block is full by definition,
// so the caller knows these steps ahead; ec_dense_attention serves them.
//   out[b, r, h] = sum_j softmax_j(scale <q[b, r, h], k[b, j, h/g]>) v[b, j, h/g],  r, j < L
//
// Why this shape: with one query tile per CTA (the partial-attention kernel) the period of a
// key block is the softmax of that block (one warp per SM sub-partition, its exponentials and
// TMEM round trips in series), and the tensor pipe idles about 40% of it. Here a CTA takes two
// 128-row tiles of one (sequence, KV head), which share every K/V block, and each tile has its
// own softmax warpgroup: while one tile's softmax runs, the tensor pipe works on the other
// tile's PV and next S products. Per tile the chain is S -> softmax -> PV -> next S (one S
// buffer per tile: TMEM holds two S and two O accumulators). The softmax reads its S row in
// 64-column chunks (the row max first, then the exponentials), so a thread needs about 120
// registers: three warpgroups' worth of threads get at most 168 each.
// Roles (10 warps, one CTA per SM, persistent over work items, no clusters):
//   warp 0      TMA: both query tiles once per item, then K and V blocks of 128 keys into two
//               64 KB stages (128-byte swizzle, mbarrier transaction counts).
//   warp 1      allocates 512 TMEM columns; one lane issues S = Q K^T into the tile's S buffer
//               and O += P V with P read from TMEM, and commits each to its barrier. TMEM: tile
//               t's S buffer at columns 128 t, its O accumulator at 256 + 128 t.
//   warps 2..5  softmax and epilogue of tile 0, warps 6..9 of tile 1: one TMEM lane (= one packed
//               query row) per thread; online softmax in base 2 with a lazy rescale of O (only
//               when the running max grows by more than 2^8), P in bf16 written back over the
//               first half of the S buffer.
// GQA packs the g query heads of a KV head into the 128 rows (floor(128 / g) positions per tile).
// Every wait is bounded and reports EC_DEVERR_TIMEOUT.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "ec_common.cuh"
#include "ec_internal.h"

namespace ec {
namespace {

constexpr int D = 128;           // head size
constexpr int kBlockM = 128;     // packed query rows per tile (TMEM lanes)
constexpr int kBlockN = 128;     // keys per K/V block (one TMA stage)
constexpr int kSubN = 128;       // keys per S product and softmax step (64 measured slower)
constexpr int kNBuf = kBlockN / kSubN;  // S buffers per tile = sub-blocks per K/V block
constexpr int kThreads = 320;    // warp 0 TMA, warp 1 MMA, warps 2-5 / 6-9 softmax of tile 0 / 1
constexpr int kMaxRegs = 168;    // per thread: registers are granted per 4 warps, 65536 / (3 x 128) = 170
constexpr uint32_t kTmemCols = 512;
constexpr int kStages = 2;       // K/V blocks in flight
constexpr uint32_t kTmemO = 256;  // tile t's O accumulator at [256 + 128 t, 384 + 128 t)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kRescaleLog2 = 8.f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s per pipeline wait

constexpr int kAtomBytes = 128 * 128;   // 128 rows x 128 bytes (64 bf16)
constexpr int kQBytes = 2 * kAtomBytes;  // one tile: 128 rows x 128 dims
constexpr int kKVBytes = 2 * kAtomBytes;  // K (or V) of one block: 128 keys x 128 dims
constexpr int kStageBytes = 2 * kKVBytes;
constexpr int kQOff = 0;
constexpr int kStageOff = kQOff + 2 * kQBytes;
constexpr int kBarOff = kStageOff + kStages * kStageBytes;

struct Bars {
  uint64_t q_full, q_empty;
  uint64_t kv_full[kStages], kv_empty[kStages];
  uint64_t s_full[2][kNBuf], s_free[2][kNBuf];  // [tile][S buffer]; s_free: the PV product that read P is done
  uint64_t p_full[2][kNBuf];
  uint64_t o_full, o_free[2];
  uint32_t tmem_base;
  int abort;
};
constexpr int kDynSmem = kBarOff + static_cast<int>(sizeof(Bars)) + 1024;  // slack for 1024-byte alignment

// Operand descriptors (128-byte swizzle, 8-row groups 1024 bytes apart): one K step of 16 dims
// advances a K-major tile by 32 bytes within a 64-dim atom (the next atom is 16 KB further); a
// sub-block of kSubN keys starts kSubN rows into each atom; one K step of 16 keys advances the
// MN-major V tile by 16 rows of 128 bytes.
constexpr uint32_t kDescHi = sdesc_hi(1024);
__host__ __device__ constexpr uint32_t step_qk(int kk) { return (kk >> 2) * (128 * 128 / 16) + (kk & 3) * 2; }
constexpr uint32_t kStepPV = 16 * 128 / 16;
constexpr uint32_t kSubK = kSubN * 128;  // bytes from one sub-block's keys to the next within a K block

struct Item {
  int b, kvh, r0, nrows0, nrows1;
};

// Items are (b, kv head, pair of consecutive row tiles), in that order.
__device__ __forceinline__ Item decode_item(int item, int Hkv, int L, int nr) {
  const int pairs = ((L + nr - 1) / nr + 1) / 2;
  Item it;
  const int bk = item / pairs;
  const int md = item - bk * pairs;
  it.b = bk / Hkv;
  it.kvh = bk - it.b * Hkv;
  it.r0 = md * 2 * nr;
  it.nrows0 = min(nr, L - it.r0);
  it.nrows1 = max(0, min(nr, L - it.r0 - nr));
  return it;
}

__global__ void __maxnreg__(kMaxRegs) dense_tiles_kernel(
    const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
    const __grid_constant__ CUtensorMap tm_v, int B, int L, int Hq, int Hkv, int g, int nr, float scale_log2,
    uint16_t* __restrict__ out, int32_t* __restrict__ dev_err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Bars* bars = reinterpret_cast<Bars*>(smem + kBarOff);
  uint8_t* q_smem = smem + kQOff;
  uint8_t* stage0 = smem + kStageOff;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int M_rows = nr * g;
  const int nblk = (L + kBlockN - 1) / kBlockN;
  // sub-blocks per item: all of every block, so that each S buffer is used once per block (a
  // sub-block past L reads zeros and is masked out of the softmax)
  const int nsub = kNBuf * nblk;
  const int items = B * Hkv * (((L + nr - 1) / nr + 1) / 2);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    mbar_init(&bars->q_empty, 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&bars->kv_full[i], 1);
      mbar_init(&bars->kv_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      for (int h = 0; h < kNBuf; ++h) {
        mbar_init(&bars->s_full[t][h], 1);
        mbar_init(&bars->s_free[t][h], 1);
        mbar_init(&bars->p_full[t][h], 128);
      }
      mbar_init(&bars->o_free[t], 128);
    }
    mbar_init(&bars->o_full, 1);
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
  pdl_wait();  // Q and the cache may come from the previous kernel in the stream
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;  // K/V blocks loaded so far
      bool ok = true;
      for (int n = 0, item = blockIdx.x; ok && item < items; ++n, item += gridDim.x) {
        const Item I = decode_item(item, Hkv, L, nr);
        if (n > 0) ok = mbar_wait_bounded(&bars->q_empty, (n - 1) & 1, abort_flag, dev_err, kWaitLimitNs);
        if (!ok) break;
        mbar_arrive_expect_tx(&bars->q_full, 2 * 2 * M_rows * 128);
        for (int t = 0; t < 2; ++t)
          for (int a = 0; a < 2; ++a)
            tma_load_5d(q_smem + t * kQBytes + a * kAtomBytes, &tm_q, &bars->q_full, a * 64, 0, I.kvh, I.r0 + t * nr,
                        I.b);
        for (int j = 0; j < nblk; ++j) {
          const uint32_t cur = it + j, slot = cur % kStages, u = cur / kStages;
          ok = mbar_wait_bounded(&bars->kv_empty[slot], (u & 1u) ^ 1u, abort_flag, dev_err, kWaitLimitNs);
          if (!ok) break;
          uint8_t* kst = stage0 + slot * kStageBytes;
          uint8_t* vst = kst + kKVBytes;
          mbar_arrive_expect_tx(&bars->kv_full[slot], kStageBytes);
          for (int a = 0; a < 2; ++a)
            tma_load_4d(kst + a * kAtomBytes, &tm_k, &bars->kv_full[slot], a * 64, I.kvh, j * kBlockN, I.b);
          for (int a = 0; a < 2; ++a)
            tma_load_4d(vst + a * kAtomBytes, &tm_v, &bars->kv_full[slot], a * 64, I.kvh, j * kBlockN, I.b);
        }
        it += nblk;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    // Per item: both tiles' S of the first block, then per block and tile t: PV_t of the block,
    // then S_t of the next block into the buffer that PV_t has just released.
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(128, kSubN, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, D, 1);
      const uint32_t q_lo0 = sdesc_lo(smem_u32(q_smem), 16);
      const uint32_t q_lo1 = sdesc_lo(smem_u32(q_smem + kQBytes), 16);
      uint32_t it = 0;  // K/V blocks consumed so far
      bool ok = true;
      // S_t = Q_t K^T for sub-block h of K/V block kb (in stage kb % kStages) into tile t's buffer h.
      auto issue_qk = [&](int t, uint32_t kb, int h) {
        const uint32_t k_lo = sdesc_lo(smem_u32(stage0 + (kb % kStages) * kStageBytes + h * kSubK), 16);
        const uint32_t s_col = tmem + (t * kNBuf + h) * kSubN;
        const uint32_t ql = t ? q_lo1 : q_lo0;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          umma_ss(s_col, ql + step_qk(kk), k_lo + step_qk(kk), kDescHi, idesc_qk, kk > 0 ? 1u : 0u);
        umma_commit(&bars->s_full[t][h]);
      };
      for (int n = 0, item = blockIdx.x; ok && item < items; ++n, item += gridDim.x) {
        // prologue: both tiles' S of the first block's sub-blocks
        ok = mbar_wait_bounded(&bars->q_full, n & 1, abort_flag, dev_err, kWaitLimitNs) &&
             mbar_wait_bounded(&bars->kv_full[it % kStages], (it / kStages) & 1u, abort_flag, dev_err, kWaitLimitNs);
        for (int s = 0; ok && s < kNBuf; ++s) {
          for (int t = 0; ok && t < 2; ++t) {
            // the buffer's previous use: the previous item's last block (use it - 1)
            ok = mbar_wait_bounded(&bars->s_free[t][s], (it & 1u) ^ 1u, abort_flag, dev_err, kWaitLimitNs);
            if (!ok) break;
            tc_fence_after();
            issue_qk(t, it, s);
          }
        }
        if (ok && nsub <= kNBuf) umma_commit(&bars->q_empty);
        for (int s = 0; ok && s < nsub; ++s) {
          const int h = s % kNBuf;
          const uint32_t kb = it + s / kNBuf;  // this sub-block's K/V block
          const uint32_t use = kb;             // use count of buffer h of either tile (one use per block)
          const uint32_t v_lo = sdesc_lo(smem_u32(stage0 + (kb % kStages) * kStageBytes + kKVBytes), kAtomBytes);
          for (int t = 0; ok && t < 2; ++t) {
            if (s == 0 && n > 0) ok = mbar_wait_bounded(&bars->o_free[t], (n - 1) & 1, abort_flag, dev_err, kWaitLimitNs);
            ok = ok && mbar_wait_bounded(&bars->p_full[t][h], use & 1u, abort_flag, dev_err, kWaitLimitNs);
            if (!ok) break;
            tc_fence_after();
            const uint32_t p_col = tmem + (t * kNBuf + h) * kSubN;
            const uint32_t o_col = tmem + kTmemO + t * kBlockM;
#pragma unroll
            for (int kk = 0; kk < kSubN / 16; ++kk)  // P: 16 keys = 8 TMEM columns per product
              umma_ts(o_col, p_col + kk * 8, v_lo + (h * (kSubN / 16) + kk) * kStepPV, kDescHi, idesc_pv,
                      (s > 0 || kk > 0) ? 1u : 0u);
            umma_commit(&bars->s_free[t][h]);
            if (t == 1 && h == kNBuf - 1) umma_commit(&bars->kv_empty[kb % kStages]);
            if (t == 1 && s == nsub - 1) umma_commit(&bars->o_full);
            if (s + kNBuf < nsub) {  // the S product one block ahead, into the buffer just read
              const uint32_t kbn = kb + 1;
              if (t == 0 && h == 0)
                ok = mbar_wait_bounded(&bars->kv_full[kbn % kStages], (kbn / kStages) & 1u, abort_flag, dev_err,
                                       kWaitLimitNs);
              ok = ok && mbar_wait_bounded(&bars->s_free[t][h], use & 1u, abort_flag, dev_err, kWaitLimitNs);
              if (!ok) break;
              tc_fence_after();
              issue_qk(t, kbn, h);
              if (t == 1 && s + kNBuf == nsub - 1) umma_commit(&bars->q_empty);
            }
          }
        }
        it += nblk;
      }
    }
  } else {
    // ------------------------------------------------------------------ softmax + epilogue
    const int t = (warp - 2) >> 2;           // tile of this warpgroup
    const int row = 32 * (warp & 3) + lane;  // TMEM lane = packed query row
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t o_col = tmem + lane_off + kTmemO + t * kBlockM;
    uint32_t it = 0;
    bool ok = true;
    for (int n = 0, item = blockIdx.x; ok && item < items; ++n, item += gridDim.x) {
      const Item I = decode_item(item, Hkv, L, nr);
      float m_used = -INFINITY, l_sum = 0.f;
      for (int s = 0; ok && s < nsub; ++s) {
        const int h = s % kNBuf;
        const uint32_t use = it + s / kNBuf;
        ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars->s_full[t][h], use & 1u, abort_flag, dev_err, kWaitLimitNs));
        if (!ok) break;
        tc_fence_after();
        const uint32_t s_col = tmem + lane_off + (t * kNBuf + h) * kSubN;
        const int nvalid = min(kSubN, L - s * kSubN);  // may be <= 0: a sub-block past L
        // The S row in chunks of 64 columns (64 registers): pass 1 takes the row max of the raw
        // scores (scale > 0 commutes with max) over 8 independent chains, pass 2 reloads each
        // chunk (a sub-block of 64 keys keeps its one chunk) for the exponentials.
        uint32_t sr[64];
        auto load_chunk = [&](int c0) {
          EC_TMEM_LD32(s_col + c0, sr);
          EC_TMEM_LD32(s_col + c0 + 32, (sr + 32));
          tmem_wait_ld();
          if (c0 + 64 > nvalid) {  // ragged last sub-block of the key range
#pragma unroll
            for (int c = 0; c < 64; ++c)
              if (c0 + c >= nvalid) sr[c] = __float_as_uint(-INFINITY);
          }
        };
        float mxs[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) mxs[e] = -INFINITY;
#pragma unroll 1
        for (int c0 = 0; c0 < kSubN; c0 += 64) {
          load_chunk(c0);
#pragma unroll
          for (int c = 0; c < 64; c += 8)
#pragma unroll
            for (int e = 0; e < 8; ++e) mxs[e] = fmaxf(mxs[e], __uint_as_float(sr[c + e]));
        }
        const float mx = fmaxf(fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])),
                               fmaxf(fmaxf(mxs[4], mxs[5]), fmaxf(mxs[6], mxs[7]))) * scale_log2;
        bool rescale = false;
        float alpha = 1.f;
        if (s == 0) {
          m_used = mx;
        } else if (mx > m_used + kRescaleLog2) {
          alpha = ex2_approx(m_used - mx);
          m_used = mx;
          l_sum *= alpha;
          rescale = true;
        }
        // p = 2^(s * scale * log2(e) - m_used); row sum over 8 independent chains. P (bf16) goes
        // over the first half of this S buffer (chunk c0 to columns c0 / 2, already read), where
        // the PV product reads it from TMEM.
        const float neg_m = -m_used;
        float rss[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) rss[e] = 0.f;
#pragma unroll 1
        for (int c0 = 0; c0 < kSubN; c0 += 64) {
          if (kSubN > 64) load_chunk(c0);
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            const float p0 = ex2_approx(fmaf(__uint_as_float(sr[c]), scale_log2, neg_m));
            const float p1 = ex2_approx(fmaf(__uint_as_float(sr[c + 1]), scale_log2, neg_m));
            rss[(c >> 1) & 7] += p0 + p1;
            pk[c / 2] = pack_bf16x2(p0, p1);
          }
          EC_TMEM_ST32(s_col + c0 / 2, pk);
        }
        l_sum += ((rss[0] + rss[1]) + (rss[2] + rss[3])) + ((rss[4] + rss[5]) + (rss[6] + rss[7]));
        tmem_wait_st();
        // tcgen05.ld/st are warp-collective: the whole warp rescales when any of its rows
        // needs it (alpha = 1 for the others).
        if (__any_sync(0xffffffffu, rescale)) {
          // O holds the products of sub-blocks 0 .. s-1; wait for the last of them (the release
          // of the buffer of sub-block s - 1), then scale.
          const uint32_t pu = it + (s - 1) / kNBuf;
          ok = __all_sync(0xffffffffu, mbar_wait_bounded(&bars->s_free[t][(s - 1) % kNBuf], pu & 1u, abort_flag,
                                                         dev_err, kWaitLimitNs));
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            EC_TMEM_LD32(o_col + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            EC_TMEM_ST32(o_col + c * 32, o);
          }
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(&bars->p_full[t][h]);
      }
      it += nblk;
      if (ok) ok = mbar_wait_bounded(&bars->o_full, n & 1, abort_flag, dev_err, kWaitLimitNs);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      // Normalise and write this thread's row of the tile.
      const int nrows = t ? I.nrows1 : I.nrows0;
      const int rl = row / g, jh = row - rl * g;
      const bool valid_row = row < M_rows && rl < nrows;
      const float inv_l = 1.f / l_sum;
      uint16_t* orow = out + ((static_cast<int64_t>(I.b) * L + I.r0 + t * nr + rl) * Hq + I.kvh * g + jh) * D;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        EC_TMEM_LD32(o_col + c * 32, o);
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
      mbar_arrive(&bars->o_free[t]);
    }
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
  cuuint32_t es[5] = {1, 1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, static_cast<cuuint32_t>(rank), const_cast<void*>(base), dims,
             strides_bytes, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_dense_attention_tiles(const ec_params& p, const void* q, const void* k_cache, const void* v_cache,
                                         float scale, void* out, int32_t* dev_err, cudaStream_t s,
                                         ec_status* status) {
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
  // cache [B, L, Hkv, D] in boxes of 128 keys x 64 dims (keys past L read as zeros)
  const cuuint64_t kd[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(p.Hkv), static_cast<cuuint64_t>(p.L),
                            static_cast<cuuint64_t>(p.B)};
  const cuuint64_t ks[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(p.Hkv) * D * 2,
                            static_cast<cuuint64_t>(p.L) * p.Hkv * D * 2};
  const cuuint32_t kb[4] = {64, 1, static_cast<cuuint32_t>(kBlockN), 1};
  if (!encode(enc, &tq, q, 5, qd, qs, qb) || !encode(enc, &tk, k_cache, 4, kd, ks, kb) ||
      !encode(enc, &tv, v_cache, 4, kd, ks, kb)) {
    *status = EC_ERR_INVALID_ARG;
    return cudaErrorInvalidValue;
  }
  int sms = 0;
  cudaError_t e = cached_per_device(
      2000 + D, &sms,
      [](int* n_out, void*) -> cudaError_t {
        cudaError_t r = current_device_sms(n_out);
        if (r == cudaSuccess)
          r = cudaFuncSetAttribute(dense_tiles_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kDynSmem);
        return r;
      },
      nullptr);
  if (e != cudaSuccess) {
    *status = EC_ERR_CUDA;
    return e;
  }
  const int64_t items = static_cast<int64_t>(p.B) * p.Hkv * (((p.L + nr - 1) / nr + 1) / 2);
  if (items > INT32_MAX) {
    *status = EC_ERR_UNSUPPORTED;
    return cudaErrorInvalidValue;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>(sms, items))));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kDynSmem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, dense_tiles_kernel, tq, tk, tv, p.B, p.L, p.Hq, p.Hkv, g, nr, scale * kLog2e,
                         static_cast<uint16_t*>(out), dev_err);
  if (e != cudaSuccess) *status = EC_ERR_CUDA;
  return e;
}

}  // namespace ec
