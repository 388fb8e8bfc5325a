// entropy_decode.cu — stage (a) of the EntropyCache step: fused softmax, greedy decode and
// Shannon entropy over the V-wide logits of each candidate row.
//
// Defines, per row i (EntropyCache, gist.science zh summary §2.2, the max-entropy
// equation's inner term; decode = greedy argmax):
//   ids[i] = lowest j attaining max_j x_ij
//   entropy[i] = -sum_j p_ij ln p_ij,  p_ij = softmax_j(x_ij)
//   log_conf[i] = ln p_{i, ids[i]} = -ln S_i,  S_i = sum_j exp(x_ij - max)
//
// Design (HBM-bound: every logit is read exactly once).
//   - Split-V: the row is cut into chunks of kThreads * kVecPerThread 16-byte vectors; one
//     CTA per (row, chunk), so a 32 x 126464 bf16 problem runs as 512 CTAs and issues all of
//     its loads in the first wave. Each thread issues all its 16-byte streaming loads before
//     any arithmetic.
//   - Two passes over registers: (1) max and lowest index over the raw stored values (exact,
//     no rescaling before comparison), block-reduced; (2) S = sum 2^d and T = sum d 2^d with
//     d = (x - M) log2(e) relative to the block max M, block-reduced. H = ln2 (log2 S - T/S).
//   - Chunks of a row merge in the last CTA to finish (a counter per row, no spinning): it
//     rescales every chunk's (S, T) to the row max, picks the row argmax with the
//     lower-index tie rule, writes the row result and returns the counter to zero.
#include <climits>

#include "ec_common.cuh"
#include "ec_internal.h"

namespace ec {
namespace {

constexpr int kThreads = 256;
constexpr int kVecPerThread = 4;
constexpr int kWarps = kThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <int DT>
struct Elem;
template <>
struct Elem<EC_F32> {
  static constexpr int kPerVec = 4;
  static constexpr int kBytes = 4;
};
template <>
struct Elem<EC_BF16> {
  static constexpr int kPerVec = 8;
  static constexpr int kBytes = 2;
};

template <int DT>
constexpr int chunk_elems() {
  return kThreads * kVecPerThread * Elem<DT>::kPerVec;
}

__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

template <int DT>
__device__ __forceinline__ void unpack(const uint4& v, float* x) {
  if constexpr (DT == EC_F32) {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
  } else {
    x[0] = bf16lo_to_f32(v.x);
    x[1] = bf16hi_to_f32(v.x);
    x[2] = bf16lo_to_f32(v.y);
    x[3] = bf16hi_to_f32(v.y);
    x[4] = bf16lo_to_f32(v.z);
    x[5] = bf16hi_to_f32(v.z);
    x[6] = bf16lo_to_f32(v.w);
    x[7] = bf16hi_to_f32(v.w);
  }
}

template <int DT>
__device__ __forceinline__ float load_one(const char* row, int64_t j) {
  if constexpr (DT == EC_F32) {
    return __ldg(reinterpret_cast<const float*>(row) + j);
  } else {
    const uint16_t u = __ldg(reinterpret_cast<const unsigned short*>(row) + j);
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
  }
}

// Larger value wins; equal values: lower index wins.
__device__ __forceinline__ void argmax_merge(float& m, int& i, float m2, int i2) {
  if (m2 > m || (m2 == m && i2 < i)) {
    m = m2;
    i = i2;
  }
}

__device__ __forceinline__ void warp_argmax(float& m, int& i) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, off);
    argmax_merge(m, i, m2, i2);
  }
}

__device__ __forceinline__ void warp_sum2(float& a, float& b) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    a += __shfl_xor_sync(0xffffffffu, a, off);
    b += __shfl_xor_sync(0xffffffffu, b, off);
  }
}

struct BlockScratch {
  float m[kWarps];
  int i[kWarps];
  float s[kWarps];
  float t[kWarps];
  float bm;
  int bi;
  float bs;
  float bt;
  int last;
};

__device__ __forceinline__ void block_argmax(float& m, int& i, BlockScratch& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  warp_argmax(m, i);
  if (lane == 0) {
    sh.m[warp] = m;
    sh.i[warp] = i;
  }
  __syncthreads();
  if (warp == 0) {
    m = lane < kWarps ? sh.m[lane] : -INFINITY;
    i = lane < kWarps ? sh.i[lane] : INT_MAX;
    warp_argmax(m, i);
    if (lane == 0) {
      sh.bm = m;
      sh.bi = i;
    }
  }
  __syncthreads();
  m = sh.bm;
  i = sh.bi;
}

__device__ __forceinline__ void block_sum2(float& a, float& b, BlockScratch& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  warp_sum2(a, b);
  if (lane == 0) {
    sh.s[warp] = a;
    sh.t[warp] = b;
  }
  __syncthreads();
  if (warp == 0) {
    a = lane < kWarps ? sh.s[lane] : 0.f;
    b = lane < kWarps ? sh.t[lane] : 0.f;
    warp_sum2(a, b);
    if (lane == 0) {
      sh.bs = a;
      sh.bt = b;
    }
  }
  __syncthreads();
  a = sh.bs;
  b = sh.bt;
}

__device__ __forceinline__ void write_row(int row, float m_unused, int idx, float S, float T, int32_t* ids,
                                          float* entropy, float* log_conf) {
  (void)m_unused;
  const float l2s = lg2_approx(S);
  ids[row] = idx;
  entropy[row] = kLn2 * (l2s - T / S);
  log_conf[row] = -kLn2 * l2s;
}

struct EntArgs {
  const char* logits;
  int64_t row_stride_bytes;
  int32_t V, nchunks;
  int32_t* ids;
  float* entropy;
  float* log_conf;
  ChunkPartial* partials;
  uint32_t* counters;
  const int32_t* row_count;
  int32_t rows_per_group;
};

// One (row, vocabulary chunk) per CTA. Returns the row whose final result this CTA wrote (the
// only chunk of the row, or its last chunk to finish), else -1. Uniform over the CTA.
template <int DT>
__device__ __forceinline__ int entropy_chunk(
    int64_t bid, const char* __restrict__ logits, int64_t row_stride_bytes, int32_t V, int32_t nchunks,
    int32_t* __restrict__ ids, float* __restrict__ entropy, float* __restrict__ log_conf,
    ChunkPartial* __restrict__ partials, uint32_t* __restrict__ counters, const int32_t* __restrict__ row_count,
    int32_t rows_per_group, BlockScratch& sh) {
  constexpr int PV = Elem<DT>::kPerVec;
  constexpr int EB = Elem<DT>::kBytes;
  constexpr int CE = chunk_elems<DT>();
  const int row = static_cast<int>(bid / nchunks);
  const int chunk = static_cast<int>(bid - static_cast<int64_t>(row) * nchunks);
  if (row_count != nullptr) {
    const int grp = row / rows_per_group;
    if (row - grp * rows_per_group >= __ldg(row_count + grp)) return -1;  // whole row skipped
  }
  const char* rowp = logits + static_cast<int64_t>(row) * row_stride_bytes;
  const int64_t c0 = static_cast<int64_t>(chunk) * CE;
  const int64_t c1 = min(static_cast<int64_t>(V), c0 + CE);
  const int nvec = static_cast<int>((c1 - c0) / PV);
  const int64_t tail0 = c0 + static_cast<int64_t>(nvec) * PV;
  const int ntail = static_cast<int>(c1 - tail0);

  // Issue every load of this thread before any arithmetic.
  uint4 v[kVecPerThread];
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const int vi = threadIdx.x + u * kThreads;
    if (vi < nvec) v[u] = ld_stream_v4(rowp + (c0 + static_cast<int64_t>(vi) * PV) * EB);
  }
  float xt = -INFINITY;
  const bool has_tail = threadIdx.x < ntail;
  if (has_tail) xt = load_one<DT>(rowp, tail0 + threadIdx.x);

  // Pass 1: max of the raw values, lowest index (this thread scans increasing j).
  float m = -INFINITY;
  int mi = INT_MAX;
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const int vi = threadIdx.x + u * kThreads;
    if (vi < nvec) {
      float x[PV];
      unpack<DT>(v[u], x);
      const int jb = static_cast<int>(c0) + vi * PV;
#pragma unroll
      for (int e = 0; e < PV; ++e) {
        if (x[e] > m || mi == INT_MAX) {
          m = x[e];
          mi = jb + e;
        }
      }
    }
  }
  if (has_tail && (xt > m || mi == INT_MAX)) {
    m = xt;
    mi = static_cast<int>(tail0) + threadIdx.x;
  }
  block_argmax(m, mi, sh);

  // Pass 2: S = sum 2^d, T = sum d 2^d, d = (x - M) log2 e; d clamped at -127 so that
  // -inf logits give 2^d = 0 (flushed) and d 2^d = 0.
  const float M2 = m * kLog2e;
  float S = 0.f, T = 0.f;
#pragma unroll
  for (int u = 0; u < kVecPerThread; ++u) {
    const int vi = threadIdx.x + u * kThreads;
    if (vi < nvec) {
      float x[PV];
      unpack<DT>(v[u], x);
#pragma unroll
      for (int e = 0; e < PV; ++e) {
        const float d = fmaxf(fmaf(x[e], kLog2e, -M2), -127.f);
        const float p = ex2_approx(d);
        S += p;
        T = fmaf(p, d, T);
      }
    }
  }
  if (has_tail) {
    const float d = fmaxf(fmaf(xt, kLog2e, -M2), -127.f);
    const float p = ex2_approx(d);
    S += p;
    T = fmaf(p, d, T);
  }
  block_sum2(S, T, sh);

  if (nchunks == 1) {
    if (threadIdx.x == 0) write_row(row, m, mi, S, T, ids, entropy, log_conf);
    return row;
  }

  // Publish this chunk; the last chunk of the row to finish merges.
  if (threadIdx.x == 0) {
    partials[static_cast<int64_t>(row) * nchunks + chunk] = ChunkPartial{m, mi, S, T};
    __threadfence();
    const uint32_t done = atomicAdd(counters + row, 1u);
    sh.last = (done == static_cast<uint32_t>(nchunks - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!sh.last) return -1;
  __threadfence();

  const ChunkPartial* rp = partials + static_cast<int64_t>(row) * nchunks;
  float rm = -INFINITY;
  int ri = INT_MAX;
  for (int c = threadIdx.x; c < nchunks; c += kThreads) {
    const float cm = __ldcg(&rp[c].m);
    const int ci = __ldcg(&rp[c].idx);
    argmax_merge(rm, ri, cm, ci);
  }
  block_argmax(rm, ri, sh);
  const float R2 = rm * kLog2e;
  float RS = 0.f, RT = 0.f;
  for (int c = threadIdx.x; c < nchunks; c += kThreads) {
    const float cs = __ldcg(&rp[c].s);
    if (cs > 0.f) {
      const float delta = __ldcg(&rp[c].m) * kLog2e - R2;
      const float f = ex2_approx(delta);
      RS = fmaf(f, cs, RS);
      RT = fmaf(f, fmaf(delta, cs, __ldcg(&rp[c].t)), RT);
    }
  }
  block_sum2(RS, RT, sh);
  if (threadIdx.x == 0) {
    write_row(row, rm, ri, RS, RT, ids, entropy, log_conf);
    counters[row] = 0u;  // ready for the next call
  }
  return row;
}

template <int DT>
__global__ void __launch_bounds__(kThreads) entropy_decode_kernel(EntArgs a) {
  __shared__ BlockScratch sh;
  pdl_wait();  // logits and row counts may come from the previous kernel in the stream
  pdl_launch_dependents();
  entropy_chunk<DT>(blockIdx.x, a.logits, a.row_stride_bytes, a.V, a.nchunks, a.ids, a.entropy, a.log_conf,
                    a.partials, a.counters, a.row_count, a.rows_per_group, sh);
}

}  // namespace

int entropy_chunk_elems(int32_t dtype) {
  return dtype == EC_F32 ? chunk_elems<EC_F32>() : chunk_elems<EC_BF16>();
}

int32_t entropy_num_chunks(int32_t V, int32_t dtype) {
  const int ce = entropy_chunk_elems(dtype);
  return static_cast<int32_t>((static_cast<int64_t>(V) + ce - 1) / ce);
}

size_t entropy_workspace_bytes(int32_t n_rows, int32_t V, int32_t dtype) {
  const size_t nch = static_cast<size_t>(entropy_num_chunks(V, dtype));
  const size_t rows = static_cast<size_t>(n_rows > 0 ? n_rows : 0);
  return align_up(rows * nch * sizeof(ChunkPartial), 256) + align_up(rows * sizeof(uint32_t), 256);
}

cudaError_t launch_entropy_decode(const void* logits, int64_t row_stride, int32_t n_rows, int32_t V,
                                  int32_t dtype, int32_t* ids, float* entropy, float* log_conf, void* ws,
                                  const int32_t* row_count, int32_t rows_per_group, cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const int32_t nch = entropy_num_chunks(V, dtype);
  const size_t rows = static_cast<size_t>(n_rows);
  auto* partials = static_cast<ChunkPartial*>(ws);
  auto* counters = reinterpret_cast<uint32_t*>(static_cast<char*>(ws) +
                                               align_up(rows * nch * sizeof(ChunkPartial), 256));
  const int64_t nblocks = static_cast<int64_t>(n_rows) * nch;
  if (nblocks > INT_MAX) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(nblocks));
  const EntArgs a{static_cast<const char*>(logits), row_stride * (dtype == EC_F32 ? 4 : 2), V, nch, ids, entropy,
                  log_conf, partials, counters, row_count, rows_per_group};
  if (dtype == EC_F32) return launch_pdl(entropy_decode_kernel<EC_F32>, grid, dim3(kThreads), 0, s, a);
  return launch_pdl(entropy_decode_kernel<EC_BF16>, grid, dim3(kThreads), 0, s, a);
}

}  // namespace ec
