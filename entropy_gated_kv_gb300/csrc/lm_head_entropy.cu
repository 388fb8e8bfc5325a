// lm_head_entropy.cu — the output projection of the candidate rows fused with stage (a) of
// the EntropyCache step: logits = hidden · Wᵀ, then per row the greedy decode, the Shannon
// entropy and the log-confidence of the decoded token, without the logits ever reaching
// memory.
//
// The pages define stage (a) on the logits of the masked candidates (EntropyCache,
// gist.science zh summary §2.2: decode each candidate and take the entropy of its softmax);
// producing those logits is the model's last matrix product, which the pages leave to the
// model. Fusing the two is this library's design, with no counterpart in the pages.
//
// Design (HBM-bound on W: V x d_model bf16 is read once; the candidate rows are few):
//   - Swap-AB tcgen05 GEMM: M = 128 vocabulary rows of W (A, K-major), N = the candidate rows
//     padded to a multiple of 32 (B, K-major), K = d_model in tiles of 64 (one 128-byte
//     swizzle atom per row). TMA loads both operands into a ring of stages; one thread issues
//     tcgen05.mma (bf16 in, fp32 accumulate) into a double-buffered TMEM accumulator, so the
//     epilogue of one vocabulary tile overlaps the products of the next.
//   - Persistent CTAs, one per SM, vocabulary tiles dealt round-robin.
//   - Epilogue (4 warps): tcgen05.ld of 32 candidates x 128 vocabulary rows, transposed through
//     shared memory; thread (candidate c, quarter q) keeps a running (max, index, S, T) over its
//     32 vocabulary rows of every tile (S = sum 2^d, T = sum d 2^d, d = (x - max) log2 e, as in
//     the decode kernels). The four quarters merge once, after the last tile, into one partial
//     per (candidate, CTA); a second kernel merges the CTAs' partials and writes the results.
#include <cuda.h>

#include <algorithm>
#include <climits>
#include <mutex>

#include "ec_common.cuh"
#include "ec_internal.h"
#include "entropy_merge.cuh"

namespace ec {
namespace {

constexpr int kThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kTileV = 128;    // vocabulary rows per tile (MMA M)
constexpr int kTileK = 64;     // d_model elements per stage (one 128-byte swizzle atom)
constexpr int kMaxN = 256;     // candidate rows (MMA N, padded to a multiple of 32)
constexpr int kMaxGrid = 1024;
constexpr uint32_t kABytes = kTileV * kTileK * 2;  // 16 KB
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: far beyond any legitimate wait
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kDescHi = sdesc_hi(1024);  // 8 rows of 128 B between core-matrix groups

struct Bars {
  uint64_t full[8];
  uint64_t empty[8];
  uint64_t acc_full[2];
  uint64_t acc_empty[2];
  uint32_t tmem_base;
  int abort;
  int epi_ok;  // the epilogue's shared verdict on its latest wait
};

// Shared-memory layout for N padded candidates and S stages.
struct Layout {
  int n_pad, stages;
  uint32_t b_bytes, stage_bytes, a_off, b_off, t_off, p_off, bar_off, total;
};

__host__ __device__ inline Layout make_layout(int n_pad) {
  Layout l;
  l.n_pad = n_pad;
  l.b_bytes = static_cast<uint32_t>(n_pad) * kTileK * 2;
  l.stage_bytes = kABytes + l.b_bytes;
  const uint32_t budget = 200u * 1024u;  // stages, plus 16 KB transpose and 8 KB partials
  int s = static_cast<int>(budget / l.stage_bytes);
  l.stages = s < 2 ? 2 : (s > 8 ? 8 : s);
  l.a_off = 0;
  l.b_off = l.stages * kABytes;
  l.t_off = l.b_off + l.stages * l.b_bytes;           // transpose buffer, 32 x 129 floats
  l.p_off = l.t_off + 32 * 129 * 4;                   // quarter partials, 4 x 32 EntPart
  l.bar_off = (l.p_off + 4 * 32 * 16 + 15) & ~15u;
  l.total = l.bar_off + static_cast<uint32_t>(sizeof(Bars));
  return l;
}

__device__ __forceinline__ void tma_load_2d(void* dst, const void* tmap, uint64_t* bar, int c0, int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
      : "memory");
}

// Folds 32 logits x[0..31] of vocabulary rows v0.. (the first nvalid valid) into a running
// (max, index, S, T). S and T are relative to the running max; the lowest index wins ties.
__device__ __forceinline__ void fold32(const float* x, int v0, int nvalid, EntPart& st) {
  float m = -INFINITY;
  int mi = INT_MAX;
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (i < nvalid && (x[i] > m || mi == INT_MAX)) {
      m = x[i];
      mi = v0 + i;
    }
  const float m_old = st.m;
  ent_argmax_merge(st.m, st.i, m, mi);
  if (st.m > m_old && st.s > 0.f) {
    const float d = (m_old - st.m) * kLog2e;
    const float f = ex2_approx(d);
    st.t = f * fmaf(d, st.s, st.t);
    st.s *= f;
  }
  const float M2 = st.m == -INFINITY ? 0.f : st.m * kLog2e;
  float s0 = 0.f, s1 = 0.f, t0 = 0.f, t1 = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    if (i < nvalid) {
      const float d = fmaxf(fmaf(x[i], kLog2e, -M2), -127.f);
      const float p = ex2_approx(d);
      if (i & 1) {
        s1 += p;
        t1 = fmaf(p, d, t1);
      } else {
        s0 += p;
        t0 = fmaf(p, d, t0);
      }
    }
  }
  st.s += s0 + s1;
  st.t += t0 + t1;
}

__global__ void __launch_bounds__(kThreads, 1) lm_head_kernel(const __grid_constant__ CUtensorMap tm_w,
                                                               const __grid_constant__ CUtensorMap tm_h,
                                                               int n_rows, int n_pad, int d_model, int V,
                                                               ChunkPartial* __restrict__ partials,
                                                               int32_t* __restrict__ dev_err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const Layout ly = make_layout(n_pad);
  Bars* bars = reinterpret_cast<Bars*>(smem + ly.bar_off);
  float* sT = reinterpret_cast<float*>(smem + ly.t_off);
  EntPart* sP = reinterpret_cast<EntPart*>(smem + ly.p_off);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int S = ly.stages;
  const int n_tiles = (V + kTileV - 1) / kTileV;
  const int n_k = d_model / kTileK;
  const int n_chunks = n_pad / 32;
  const uint32_t tmem_cols = n_pad * 2 <= 32 ? 32u : (n_pad * 2 <= 64 ? 64u : (n_pad * 2 <= 128 ? 128u : (n_pad * 2 <= 256 ? 256u : 512u)));

  if (threadIdx.x == 0) {
    for (int i = 0; i < S; ++i) {
      mbar_init(&bars->full[i], 1);
      mbar_init(&bars->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bars->acc_full[i], 1);
      mbar_init(&bars->acc_empty[i], 128);
    }
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_w);
    prefetch_tmap(&tm_h);
  }
  if (warp == 1) {
    tmem_alloc(&bars->tmem_base, tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bars->tmem_base;
  volatile int* abort_flag = &bars->abort;
  pdl_wait();  // hidden rows may come from the previous kernel in the stream
  pdl_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      uint32_t it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x) {
        for (int kt = 0; kt < n_k; ++kt, ++it) {
          const uint32_t s = it % S, u = it / S;
          if (!(ok = mbar_wait_bounded(&bars->empty[s], (u & 1u) ^ 1u, abort_flag, dev_err, kWaitLimitNs))) break;
          mbar_arrive_expect_tx(&bars->full[s], ly.stage_bytes);
          tma_load_2d(smem + ly.a_off + s * kABytes, &tm_w, &bars->full[s], kt * kTileK, tile * kTileV);
          tma_load_2d(smem + ly.b_off + s * ly.b_bytes, &tm_h, &bars->full[s], kt * kTileK, 0);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(128, static_cast<uint32_t>(n_pad), 0);
      uint32_t it = 0;
      bool ok = true;
      int n = 0;
      for (int tile = blockIdx.x; ok && tile < n_tiles; tile += gridDim.x, ++n) {
        const int buf = n & 1;
        const uint32_t use = static_cast<uint32_t>(n >> 1);
        if (!(ok = mbar_wait_bounded(&bars->acc_empty[buf], (use & 1u) ^ 1u, abort_flag, dev_err, kWaitLimitNs))) break;
        tc_fence_after();
        const uint32_t d_col = tmem + static_cast<uint32_t>(buf * n_pad);
        for (int kt = 0; kt < n_k; ++kt, ++it) {
          const uint32_t s = it % S, u = it / S;
          if (!(ok = mbar_wait_bounded(&bars->full[s], u & 1u, abort_flag, dev_err, kWaitLimitNs))) break;
          tc_fence_after();
          const uint32_t a_lo = sdesc_lo(smem_u32(smem + ly.a_off + s * kABytes), 16);
          const uint32_t b_lo = sdesc_lo(smem_u32(smem + ly.b_off + s * ly.b_bytes), 16);
#pragma unroll
          for (int kk = 0; kk < kTileK / 16; ++kk)  // 16 elements = 32 bytes = 2 descriptor units
            umma_ss(d_col, a_lo + 2 * kk, b_lo + 2 * kk, kDescHi, idesc, (kt > 0 || kk > 0) ? 1u : 0u);
          umma_commit(&bars->empty[s]);
        }
        if (ok) umma_commit(&bars->acc_full[buf]);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int et = threadIdx.x - 64;        // 0..127
    const int q = warp - 2;                 // the warp's quarter of vocabulary rows
    const int row = 32 * (warp & 3) + lane;  // the TMEM lane this thread reads (tcgen05 warp rule)
    const uint32_t lane_off = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    EntPart st[kMaxN / 32];
#pragma unroll
    for (int c = 0; c < kMaxN / 32; ++c) st[c] = EntPart{-INFINITY, INT_MAX, 0.f, 0.f};
    bool ok = true;
    int n = 0;
    for (int tile = blockIdx.x; tile < n_tiles; tile += gridDim.x, ++n) {
      const int buf = n & 1;
      const uint32_t use = static_cast<uint32_t>(n >> 1);
      // one thread waits and the four warps take its verdict together, so that none of them
      // can be left at a named barrier that the others have abandoned
      named_bar_sync(1, 128);  // the previous verdict has been read by everyone
      if (et == 0) bars->epi_ok = mbar_wait_bounded(&bars->acc_full[buf], use & 1u, abort_flag, dev_err, kWaitLimitNs) ? 1 : 0;
      named_bar_sync(1, 128);
      ok = bars->epi_ok != 0;
      if (!ok) break;
      tc_fence_after();
      for (int ch = 0; ch < n_chunks; ++ch) {
        uint32_t r[32];
        EC_TMEM_LD32(tmem + lane_off + static_cast<uint32_t>(buf * n_pad + ch * 32), r);
        tmem_wait_ld();
        if (ch == n_chunks - 1) {  // the accumulator buffer may be overwritten now
          tc_fence_before();
          mbar_arrive(&bars->acc_empty[buf]);
        }
        named_bar_sync(1, 128);  // the transpose buffer is free
#pragma unroll
        for (int c = 0; c < 32; ++c) sT[c * 129 + row] = __uint_as_float(r[c]);
        named_bar_sync(1, 128);
        // thread (candidate lane, quarter q) folds its 32 vocabulary rows of this tile
        float x[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) x[i] = sT[lane * 129 + q * 32 + i];
        const int v0 = tile * kTileV + q * 32;
        const int nvalid = min(32, V - v0);
#pragma unroll
        for (int c = 0; c < kMaxN / 32; ++c)
          if (c == ch && nvalid > 0) fold32(x, v0, nvalid, st[c]);
      }
    }
    // merge the four quarters of each candidate and publish one partial per (candidate, CTA)
    for (int ch = 0; ch < n_chunks; ++ch) {
      EntPart mine{-INFINITY, INT_MAX, 0.f, 0.f};
#pragma unroll
      for (int c = 0; c < kMaxN / 32; ++c)
        if (c == ch) mine = st[c];
      named_bar_sync(1, 128);
      sP[q * 32 + lane] = mine;
      named_bar_sync(1, 128);
      if (q == 0) {
        EntPart p = sP[lane];
#pragma unroll
        for (int k = 1; k < 4; ++k) ent_part_merge(p, sP[k * 32 + lane]);
        const int cand = ch * 32 + lane;
        if (cand < n_rows) {
          if (!ok || *abort_flag) p = EntPart{NAN, -1, 1.f, NAN};  // a failed wait: the row reads NaN
          partials[static_cast<int64_t>(cand) * gridDim.x + blockIdx.x] = ChunkPartial{p.m, p.i, p.s, p.t};
        }
      }
    }
  }

  // ---------------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// One warp per candidate row: merge the CTAs' partials (in CTA order per lane) and finish.
__global__ void __launch_bounds__(256) lm_head_merge_kernel(const ChunkPartial* __restrict__ partials, int n_rows,
                                                            int nparts, int32_t* __restrict__ ids,
                                                            float* __restrict__ entropy, float* __restrict__ log_conf) {
  pdl_wait();
  pdl_launch_dependents();
  const int row = blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= n_rows) return;
  EntPart p{-INFINITY, INT_MAX, 0.f, 0.f};
  const ChunkPartial* rp = partials + static_cast<int64_t>(row) * nparts;
  for (int c = lane; c < nparts; c += 32)
    ent_part_merge(p, EntPart{__ldcg(&rp[c].m), __ldcg(&rp[c].idx), __ldcg(&rp[c].s), __ldcg(&rp[c].t)});
  p = ent_warp_merge(p);
  if (lane == 0) {
    ids[row] = p.i;
    ent_finish(p, entropy[row], log_conf[row]);
  }
}

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

// A 2D bf16 tensor map over a row-major [rows, cols] matrix, box {64, box_rows}, 128-byte
// swizzle, zero fill outside the matrix.
bool map_2d(EncodeTiledFn enc, CUtensorMap* m, const void* base, int64_t rows, int64_t cols, uint32_t box_rows) {
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {static_cast<cuuint32_t>(kTileK), box_rows};
  const cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

size_t lm_head_workspace_bytes(int32_t n_rows) {
  return align_up(static_cast<size_t>(n_rows > 0 ? n_rows : 0) * kMaxGrid * sizeof(ChunkPartial), 256);
}

int32_t lm_head_max_rows() { return kMaxN; }

cudaError_t launch_lm_head_entropy(const void* hidden, const void* weight, int32_t n_rows, int32_t d_model, int32_t V,
                                   int32_t* ids, float* entropy, float* log_conf, void* ws, int32_t* dev_err,
                                   cudaStream_t s) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return cudaErrorNotSupported;
  const int n_pad = (n_rows + 31) / 32 * 32;
  CUtensorMap tw, th;
  if (!map_2d(enc, &tw, weight, V, d_model, kTileV) || !map_2d(enc, &th, hidden, n_rows, d_model, static_cast<uint32_t>(n_pad)))
    return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const Layout ly = make_layout(n_pad);
  const size_t smem = ly.total + 1024;
  e = cudaFuncSetAttribute(lm_head_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  const int n_tiles = (V + kTileV - 1) / kTileV;
  const int grid = std::max(1, std::min({sms, n_tiles, kMaxGrid}));
  auto* parts = static_cast<ChunkPartial*>(ws);
  e = launch_pdl(lm_head_kernel, dim3(grid), dim3(kThreads), smem, s, tw, th, n_rows, n_pad, d_model, V, parts, dev_err);
  if (e != cudaSuccess) return e;
  return launch_pdl(lm_head_merge_kernel, dim3((n_rows + 7) / 8), dim3(256), 0, s, static_cast<const ChunkPartial*>(parts),
                    n_rows, grid, ids, entropy, log_conf);
}

}  // namespace ec
