// entropy_decode.cu — stage (a) of the EntropyCache step: fused softmax, greedy decode and
// Shannon entropy over the V-wide logits of each candidate row.
//
// Defines, per row i (EntropyCache, gist.science zh summary §2.2, the max-entropy
// equation's inner term; decode = greedy argmax):
//   ids[i] = lowest j attaining max_j x_ij
//   entropy[i] = -sum_j p_ij ln p_ij,  p_ij = softmax_j(x_ij)
//   log_conf[i] = ln p_{i, ids[i]} = -ln S_i,  S_i = sum_j exp(x_ij - max)
//
// Design (HBM-bound: every logit is read exactly once; at the sizes of one decoding step the
// kernel's latency matters as much as its bandwidth). Two launch shapes share the per-stretch
// reduction (sub_chunk):
//   - Two passes over registers per stretch: (1) max and lowest index over the raw stored
//     values (exact, no rescaling before comparison), block-reduced; (2) S = sum 2^d and
//     T = sum d 2^d with d = (x - M) log2(e) relative to the stretch max M, block-reduced.
//     Stretches combine by rescaling S and T to the larger max (entropy_merge.cuh).
//     H = ln2 (log2 S - T/S). Each thread issues all its 16-byte streaming loads of a
//     stretch before any arithmetic.
//   - Few rows (the whole problem within about one wave), when the caller allows it (the
//     standalone entry; not the chained step, see launch_entropy_decode): one cluster of up to
//     8 CTAs per row, CTA r owning a contiguous slice of the row; the slices merge on chip:
//     each CTA leaves its (max, index, S, T) in shared memory and, after one cluster barrier,
//     the first CTA reads them through distributed shared memory and writes the row result.
//     A 32 x 126464 bf16 problem runs as 256 CTAs with one global round trip.
//   - Many rows: one CTA per (row, 8192-element chunk), so every load is in flight at once;
//     each chunk publishes its partial to the workspace and the last chunk of a row to finish
//     (a counter per row, no spinning) merges them, writes the row result and returns the
//     counter to zero.
#include <algorithm>
#include <climits>

#include "ec_common.cuh"
#include "ec_internal.h"
#include "entropy_merge.cuh"

namespace ec {
namespace {

constexpr int kThreads = 256;
constexpr int kSplitVec = 4;    // 16-byte vectors per thread, one CTA per (row, chunk)
constexpr int kClusterVec = 8;  // 16-byte vectors per thread per stretch, cluster path
constexpr int kMaxCluster = 8;  // CTAs per row (portable cluster size)
constexpr int kClusterCtasPerSm = 4;  // cluster path while rows x cluster <= this x SMs
constexpr int kWarps = kThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;

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
constexpr int chunk_elems() {  // the split path's chunk (the workspace is sized by it)
  return kThreads * kSplitVec * Elem<DT>::kPerVec;
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

__device__ __forceinline__ void warp_argmax(float& m, int& i) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, off);
    const int i2 = __shfl_xor_sync(0xffffffffu, i, off);
    ent_argmax_merge(m, i, m2, i2);
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

using Part = EntPart;

__device__ __forceinline__ void write_row(int row, const Part& p, int32_t* ids, float* entropy, float* log_conf) {
  ids[row] = p.i;
  ent_finish(p, entropy[row], log_conf[row]);
}

struct EntArgs {
  const char* logits;
  int64_t row_stride_bytes;
  int32_t V, nchunks;  // nchunks: split path only
  int32_t* ids;
  float* entropy;
  float* log_conf;
  ChunkPartial* partials;  // split path only
  uint32_t* counters;      // split path only
  int32_t publish_only;    // split path: write each chunk's partial and stop (the reader merges)
  const int32_t* row_count;
  int32_t rows_per_group;
};

// Rows past their group's count are skipped (uniform over a CTA and over a cluster).
__device__ __forceinline__ bool row_skipped(const EntArgs& a, int row) {
  if (a.row_count == nullptr) return false;
  const int grp = row / a.rows_per_group;
  return row - grp * a.rows_per_group >= __ldg(a.row_count + grp);
}

// One stretch [c0, c1) of a row (c0 a multiple of the vector width, at most NV vectors per
// thread plus a tail of fewer than one vector at the row's end); uniform over the CTA.
template <int DT, int NV>
__device__ __forceinline__ Part sub_chunk(const char* __restrict__ rowp, int64_t c0, int64_t c1, BlockScratch& sh) {
  constexpr int PV = Elem<DT>::kPerVec;
  constexpr int EB = Elem<DT>::kBytes;
  const int nvec = static_cast<int>((c1 - c0) / PV);
  const int64_t tail0 = c0 + static_cast<int64_t>(nvec) * PV;
  const int ntail = static_cast<int>(c1 - tail0);

  // Issue every load of this thread before any arithmetic.
  uint4 v[NV];
#pragma unroll
  for (int u = 0; u < NV; ++u) {
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
  for (int u = 0; u < NV; ++u) {
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
  for (int u = 0; u < NV; ++u) {
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
  return Part{m, mi, S, T};
}

// Split path: one (row, chunk) per CTA; the last chunk of a row to finish merges the row.
template <int DT>
__global__ void __launch_bounds__(kThreads) entropy_split_kernel(EntArgs a) {
  constexpr int CE = chunk_elems<DT>();
  __shared__ BlockScratch sh;
  __shared__ int last;
  pdl_wait();  // logits and row counts may come from the previous kernel in the stream
  pdl_launch_dependents();
  const int64_t bid = blockIdx.x;
  const int row = static_cast<int>(bid / a.nchunks);
  const int chunk = static_cast<int>(bid - static_cast<int64_t>(row) * a.nchunks);
  if (row_skipped(a, row)) return;
  const char* rowp = a.logits + static_cast<int64_t>(row) * a.row_stride_bytes;
  const int64_t c0 = static_cast<int64_t>(chunk) * CE;
  const Part p = sub_chunk<DT, kSplitVec>(rowp, c0, min(static_cast<int64_t>(a.V), c0 + CE), sh);
  if (a.publish_only) {  // the step's select kernel merges the chunks of each row itself
    if (threadIdx.x == 0) a.partials[static_cast<int64_t>(row) * a.nchunks + chunk] = ChunkPartial{p.m, p.i, p.s, p.t};
    return;
  }
  if (a.nchunks == 1) {
    if (threadIdx.x == 0) write_row(row, p, a.ids, a.entropy, a.log_conf);
    return;
  }
  // Publish this chunk; the last chunk of the row to finish merges.
  if (threadIdx.x == 0) {
    a.partials[static_cast<int64_t>(row) * a.nchunks + chunk] = ChunkPartial{p.m, p.i, p.s, p.t};
    __threadfence();
    const uint32_t done = atomicAdd(a.counters + row, 1u);
    last = (done == static_cast<uint32_t>(a.nchunks - 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!last || threadIdx.x >= 32) return;
  __threadfence();
  const ChunkPartial* rp = a.partials + static_cast<int64_t>(row) * a.nchunks;
  Part r{-INFINITY, INT_MAX, 0.f, 0.f};
  for (int c = threadIdx.x; c < a.nchunks; c += 32)  // chunks in increasing order per lane
    ent_part_merge(r, Part{__ldcg(&rp[c].m), __ldcg(&rp[c].idx), __ldcg(&rp[c].s), __ldcg(&rp[c].t)});
  r = ent_warp_merge(r);
  if (threadIdx.x == 0) {
    write_row(row, r, a.ids, a.entropy, a.log_conf);
    a.counters[row] = 0u;  // ready for the next call
  }
}

// Cluster path: one cluster per row; CTA `rank` of the cluster reduces its slice, the
// cluster's first CTA merges the slices and writes the row result.
template <int DT>
__global__ void __launch_bounds__(kThreads) entropy_cluster_kernel(EntArgs a) {
  constexpr int PV = Elem<DT>::kPerVec;
  constexpr int64_t kSub = static_cast<int64_t>(kThreads) * kClusterVec * PV;  // elements per stretch
  __shared__ BlockScratch sh;
  __shared__ __align__(16) Part slice;
  pdl_wait();  // logits and row counts may come from the previous kernel in the stream
  pdl_launch_dependents();
  const int csize = static_cast<int>(cluster_size());
  const int rank = static_cast<int>(cluster_ctarank());
  const int row = static_cast<int>(cluster_id_x());
  if (row_skipped(a, row)) return;  // the whole cluster skips the row
  const char* rowp = a.logits + static_cast<int64_t>(row) * a.row_stride_bytes;
  // slice of this CTA: whole vectors, the last slice takes the remainder (and the tail)
  const int64_t nvec_row = (static_cast<int64_t>(a.V) + PV - 1) / PV;
  const int64_t w = ((nvec_row + csize - 1) / csize) * PV;
  const int64_t lo = min(static_cast<int64_t>(a.V), static_cast<int64_t>(rank) * w);
  const int64_t hi = min(static_cast<int64_t>(a.V), lo + w);
  // equal sub-chunks of at most kSub elements (whole vectors except the last)
  const int64_t nsub = (hi - lo + kSub - 1) / kSub;
  const int64_t step = nsub > 0 ? ((hi - lo + nsub - 1) / nsub + PV - 1) / PV * PV : 0;
  Part acc{-INFINITY, INT_MAX, 0.f, 0.f};
  for (int64_t c0 = lo; c0 < hi; c0 += step) {
    const Part p = sub_chunk<DT, kClusterVec>(rowp, c0, min(hi, c0 + step), sh);
    ent_part_merge(acc, p);
  }
  if (threadIdx.x == 0) slice = acc;
  cluster_sync_all();  // every slice result is in its CTA's shared memory
  if (rank == 0 && threadIdx.x < 32) {
    const int lane = threadIdx.x;
    Part p{-INFINITY, INT_MAX, 0.f, 0.f};
    if (lane < csize) {
      const float4 q = dsmem_ld_f4(dsmem_map(smem_u32(&slice), static_cast<uint32_t>(lane)));
      p = Part{q.x, __float_as_int(q.y), q.z, q.w};
    }
#pragma unroll
    for (int off = 1; off < kMaxCluster; off <<= 1) {
      const Part o{__shfl_xor_sync(0xffffffffu, p.m, off), __shfl_xor_sync(0xffffffffu, p.i, off),
                   __shfl_xor_sync(0xffffffffu, p.s, off), __shfl_xor_sync(0xffffffffu, p.t, off)};
      ent_part_merge(p, o);
    }
    if (lane == 0) write_row(row, p, a.ids, a.entropy, a.log_conf);
  }
  cluster_sync_all();  // peers keep their shared memory until it has been read
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
                                  const int32_t* row_count, int32_t rows_per_group, bool allow_cluster,
                                  bool publish_only, cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const bool f32 = dtype == EC_F32;
  const int per_vec = f32 ? Elem<EC_F32>::kPerVec : Elem<EC_BF16>::kPerVec;
  const int64_t nvec = (static_cast<int64_t>(V) + per_vec - 1) / per_vec;
  const int64_t per_cta = static_cast<int64_t>(kThreads) * kClusterVec;
  const int csize = static_cast<int>(std::min<int64_t>(kMaxCluster, std::max<int64_t>(1, (nvec + per_cta - 1) / per_cta)));
  const int32_t nch = entropy_num_chunks(V, dtype);
  const size_t rows = static_cast<size_t>(n_rows);
  EntArgs a{static_cast<const char*>(logits), row_stride * (f32 ? 4 : 2), V, nch, ids, entropy, log_conf,
            static_cast<ChunkPartial*>(ws),
            reinterpret_cast<uint32_t*>(static_cast<char*>(ws) + align_up(rows * nch * sizeof(ChunkPartial), 256)),
            publish_only ? 1 : 0, row_count, rows_per_group};
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int64_t cluster_ctas = static_cast<int64_t>(n_rows) * csize;
  if (!publish_only &&
      ((allow_cluster && cluster_ctas <= static_cast<int64_t>(kClusterCtasPerSm) * sms) || nch == 1 || ws == nullptr)) {
    if (cluster_ctas > INT_MAX) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(cluster_ctas));
    if (f32) return launch_pdl_cluster(entropy_cluster_kernel<EC_F32>, grid, dim3(kThreads), 0, csize, s, a);
    return launch_pdl_cluster(entropy_cluster_kernel<EC_BF16>, grid, dim3(kThreads), 0, csize, s, a);
  }
  const int64_t nblocks = static_cast<int64_t>(n_rows) * nch;
  if (nblocks > INT_MAX) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(nblocks));
  if (f32) return launch_pdl(entropy_split_kernel<EC_F32>, grid, dim3(kThreads), 0, s, a);
  return launch_pdl(entropy_split_kernel<EC_BF16>, grid, dim3(kThreads), 0, s, a);
}

}  // namespace ec
