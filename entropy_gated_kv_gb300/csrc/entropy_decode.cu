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
//   - Problems of 32 MB and more, outside a step: one persistent CTA of 16 warps per SM; each warp streams a
//     contiguous run of the same chunks through a ring of three 4 KB shared-memory stages
//     filled by bulk async copies (cp.async.bulk, completion on an mbarrier), keeps a running
//     (max, index, S, T) per lane and merges once per row segment; the segments publish in
//     the chunk layout above, so the workspace and its readers are the same. Pass 1 takes the
//     lane maximum with packed bf16x2 max and looks for its index only when it beats the
//     running one; pass 2 uses the paired fp32 instructions (fma.rn.f32x2 / add.rn.f32x2).
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
  int32_t n_rows;    // streaming path: rows of the problem
  int32_t* dev_err;  // may be null: where a timed-out wait is reported
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

// ---- streaming path (large problems) ----------------------------------------------------
// One persistent CTA per SM. Each warp owns a contiguous run of (row, chunk) units (the
// split path's chunks, so the workspace layout is the same) and streams it through its own
// ring of kStreamStages shared-memory stages of kSubBytes, filled by bulk async copies, so
// loads never wait for arithmetic or for a block-wide reduction. Each lane keeps a running
// (max, index, S, T) over its share of the run; a warp merge happens once per row segment.
// The first chunk of a segment holds the segment's merged partial and its other chunks an
// empty one, so the per-chunk partial array reads exactly as the split path's.
constexpr int kStreamWarps = 16;
constexpr int kStreamThreads = kStreamWarps * 32;
constexpr int kStreamStages = 3;
constexpr int kSubBytes = 4096;
constexpr int kSubVecPerLane = kSubBytes / 16 / 32;
constexpr uint64_t kStreamWaitNs = 1000000000ull;  // 1 s: a bulk copy from HBM never takes this long
// Problems at least this large take the streaming path (smaller ones are latency-bound and
// finish sooner with every load of the problem in flight at once).
constexpr int64_t kStreamMinBytes = 32ll << 20;

struct StreamShared {
  uint64_t full[kStreamWarps][kStreamStages];
  int abort;
};

template <int DT>
constexpr size_t stream_smem_bytes() {
  return 1024 + static_cast<size_t>(kStreamWarps) * kStreamStages * kSubBytes + sizeof(StreamShared);
}

// Position in a warp's run: chunk `chunk` of row `row`, sub-stretch `s` of that chunk.
// Runs are walked without divisions: the chunks' sub-stretch counts are all kFullSubs except
// the last chunk of a row (last_subs).
struct StreamPos {
  int row, chunk, s;
};

struct StreamGeom {
  int nchunks, last_subs, row_end, chunk_end;  // the run ends before (row_end, chunk_end)
  __device__ __forceinline__ bool before_end(const StreamPos& p) const {
    return p.row < row_end || (p.row == row_end && p.chunk < chunk_end);
  }
  __device__ __forceinline__ int subs(int chunk) const;
};

template <int DT>
constexpr int full_subs() {
  return chunk_elems<DT>() * Elem<DT>::kBytes / kSubBytes;
}
static_assert(full_subs<EC_BF16>() == full_subs<EC_F32>(), "one sub-stretch count per whole chunk");
__device__ __forceinline__ int StreamGeom::subs(int chunk) const {
  return chunk == nchunks - 1 ? last_subs : full_subs<EC_BF16>();
}

// Moves p forward to the first position at or after it whose row is not skipped.
__device__ __forceinline__ void skip_dead_rows(const EntArgs& a, const StreamGeom& g, StreamPos& p) {
  while (g.before_end(p) && row_skipped(a, p.row)) {
    ++p.row;
    p.chunk = 0;
    p.s = 0;
  }
}

__device__ __forceinline__ void stream_advance(const EntArgs& a, const StreamGeom& g, StreamPos& p) {
  if (++p.s < g.subs(p.chunk)) return;
  p.s = 0;
  if (++p.chunk == g.nchunks) {
    p.chunk = 0;
    ++p.row;
    skip_dead_rows(a, g, p);
  }
}

// Element range [e0, e1) of sub-stretch p, and the bytes its bulk copy moves (whole 16-byte
// vectors; the remaining e1 - e0 - bytes / element-size elements are read directly).
template <int DT>
__device__ __forceinline__ void sub_range(const EntArgs& a, const StreamPos& p, int& e0, int& e1, uint32_t& bytes) {
  constexpr int CE = chunk_elems<DT>();
  constexpr int SE = kSubBytes / Elem<DT>::kBytes;
  e0 = p.chunk * CE + p.s * SE;
  e1 = min(a.V, min((p.chunk + 1) * CE, e0 + SE));
  bytes = static_cast<uint32_t>((e1 - e0) * Elem<DT>::kBytes) & ~15u;
}

// Largest of the elements of one 16-byte vector.
template <int DT>
__device__ __forceinline__ float vec_max(const uint4& v) {
  if constexpr (DT == EC_F32) {
    return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)), fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
  } else {
    uint32_t a, b, c;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(v.x), "r"(v.y));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(b) : "r"(v.z), "r"(v.w));
    asm("max.bf16x2 %0, %1, %2;" : "=r"(c) : "r"(a), "r"(b));
    return fmaxf(bf16lo_to_f32(c), bf16hi_to_f32(c));
  }
}

// Merged summary of one row segment [c_first, c_last] (chunks of `row`) held by a warp:
// published as the segment's first chunk's partial (empty partials for its other chunks),
// or written as the row result when the segment is the whole row. Outside publish-only mode
// the warp that completes a row's chunk count merges the row, as on the split path.
// poisoned: the warp gave up waiting for its copies; the segment is published as a part
// that turns the row's entropy into NaN.
__device__ __forceinline__ void stream_finish_segment(const EntArgs& a, int row, int c_first, int c_last, EntPart p,
                                                      bool poisoned) {
  const int lane = threadIdx.x & 31;
  p = ent_warp_merge(p);
  if (poisoned) p = EntPart{NAN, -1, 1.f, NAN};
  const int nseg = c_last - c_first + 1;
  if (!a.publish_only && nseg == a.nchunks) {
    if (lane == 0) write_row(row, p, a.ids, a.entropy, a.log_conf);
    return;
  }
  ChunkPartial* rp = a.partials + static_cast<int64_t>(row) * a.nchunks;
  if (lane == 0) rp[c_first] = ChunkPartial{p.m, p.i, p.s, p.t};
  for (int c = c_first + 1 + lane; c <= c_last; c += 32) rp[c] = ChunkPartial{-INFINITY, INT_MAX, 0.f, 0.f};
  if (a.publish_only) return;
  __threadfence();
  __syncwarp();
  uint32_t done = 0;
  if (lane == 0) done = atomicAdd(a.counters + row, static_cast<uint32_t>(nseg));
  done = __shfl_sync(0xffffffffu, done, 0);
  if (done + static_cast<uint32_t>(nseg) != static_cast<uint32_t>(a.nchunks)) return;
  __threadfence();
  EntPart r{-INFINITY, INT_MAX, 0.f, 0.f};
  for (int c = lane; c < a.nchunks; c += 32)  // chunks in increasing order per lane
    ent_part_merge(r, EntPart{__ldcg(&rp[c].m), __ldcg(&rp[c].idx), __ldcg(&rp[c].s), __ldcg(&rp[c].t)});
  r = ent_warp_merge(r);
  if (lane == 0) {
    write_row(row, r, a.ids, a.entropy, a.log_conf);
    a.counters[row] = 0u;  // ready for the next call
  }
}

// Packed helpers for the streaming path: bf16x2 maximum (a NaN operand yields the other one)
// and the sm_100 paired fp32 operations, two lanes of arithmetic per instruction.
__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unf2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Logits below this are treated as -inf by the sums (2^d is 0 for them either way); keeping
// d finite makes d 2^d exactly 0 instead of -inf * 0.
constexpr uint32_t kClampBf16x2 = 0xF149F149u;  // (-9.95e29, -9.95e29) as bf16
constexpr float kClampF32 = -1e30f;

// Pass 2 over one pair of elements: S += 2^d, T += d 2^d with d = x log2 e - M2.
__device__ __forceinline__ void st_pair(uint64_t x, uint64_t l2e, uint64_t nm, uint64_t& s, uint64_t& t) {
  const uint64_t d = fma2(x, l2e, nm);
  float dl, dh;
  unf2(d, dl, dh);
  const uint64_t p = f2(ex2_approx(dl), ex2_approx(dh));
  s = add2(s, p);
  t = fma2(p, d, t);
}

// A whole stretch of kSubBytes (every lane holds kSubVecPerLane vectors, no tail), folded
// into the lane's running (am, ai, S, T). Pass 1 takes only the lane's maximum; the index is
// looked for only when that maximum beats the running one (rare once a row is under way).
template <int DT>
__device__ __forceinline__ void stream_full_sub(const uint4* __restrict__ sv, int e0, int lane, float& am, int& ai,
                                                float& S, float& T) {
  constexpr int PV = Elem<DT>::kPerVec;
  uint4 v[kSubVecPerLane];
#pragma unroll
  for (int k = 0; k < kSubVecPerLane; ++k) v[k] = sv[lane + 32 * k];
  float m;
  if constexpr (DT == EC_BF16) {
    uint32_t a = bmax2(v[0].x, v[0].y), b = bmax2(v[0].z, v[0].w);
#pragma unroll
    for (int k = 1; k < kSubVecPerLane; ++k) {
      a = bmax2(a, bmax2(v[k].x, v[k].y));
      b = bmax2(b, bmax2(v[k].z, v[k].w));
    }
    const uint32_t c = bmax2(a, b);
    m = fmaxf(bf16lo_to_f32(c), bf16hi_to_f32(c));
  } else {
    float a = fmaxf(__uint_as_float(v[0].x), __uint_as_float(v[0].y));
    float b = fmaxf(__uint_as_float(v[0].z), __uint_as_float(v[0].w));
#pragma unroll
    for (int k = 1; k < kSubVecPerLane; ++k) {
      a = fmaxf(a, fmaxf(__uint_as_float(v[k].x), __uint_as_float(v[k].y)));
      b = fmaxf(b, fmaxf(__uint_as_float(v[k].z), __uint_as_float(v[k].w)));
    }
    m = fmaxf(a, b);
  }
  if (m > am || ai == INT_MAX) {  // a new running maximum (or the lane's first stretch)
    int mi = INT_MAX;
#pragma unroll
    for (int k = kSubVecPerLane - 1; k >= 0; --k) {
      float x[PV];
      unpack<DT>(v[k], x);
#pragma unroll
      for (int e = PV - 1; e >= 0; --e)
        if (x[e] == m || (m == -INFINITY && !(x[e] > m))) mi = e0 + (lane + 32 * k) * PV + e;
    }
    const float am_old = am;
    am = m;
    ai = mi;
    if (am > am_old && S > 0.f) {  // S and T are relative to the running maximum
      const float d = (am_old - am) * kLog2e;
      const float f = ex2_approx(d);
      T = f * fmaf(d, S, T);
      S *= f;
    }
  }
  const float M2 = am == -INFINITY ? 0.f : am * kLog2e;
  const uint64_t l2e = f2(kLog2e, kLog2e), nm = f2(-M2, -M2);
  uint64_t sa = 0, sb = 0, ta = 0, tb = 0;  // two accumulator pairs (0 is +0.0f, +0.0f)
#pragma unroll
  for (int k = 0; k < kSubVecPerLane; ++k) {
    if constexpr (DT == EC_BF16) {
      const uint32_t w[4] = {v[k].x, v[k].y, v[k].z, v[k].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t c = bmax2(w[j], kClampBf16x2);
        const uint64_t x = f2(bf16lo_to_f32(c), bf16hi_to_f32(c));
        if (j & 1) st_pair(x, l2e, nm, sb, tb);
        else st_pair(x, l2e, nm, sa, ta);
      }
    } else {
      const uint64_t x0 = f2(fmaxf(__uint_as_float(v[k].x), kClampF32), fmaxf(__uint_as_float(v[k].y), kClampF32));
      const uint64_t x1 = f2(fmaxf(__uint_as_float(v[k].z), kClampF32), fmaxf(__uint_as_float(v[k].w), kClampF32));
      st_pair(x0, l2e, nm, sa, ta);
      st_pair(x1, l2e, nm, sb, tb);
    }
  }
  float s0, s1, t0, t1;
  unf2(add2(sa, sb), s0, s1);
  unf2(add2(ta, tb), t0, t1);
  S += s0 + s1;
  T += t0 + t1;
}

template <int DT>
__global__ void __launch_bounds__(kStreamThreads, 1) entropy_stream_kernel(EntArgs a) {
  constexpr int PV = Elem<DT>::kPerVec;
  constexpr int EB = Elem<DT>::kBytes;
  constexpr int CE = chunk_elems<DT>();
  extern __shared__ uint8_t smem_raw[];
  uint8_t* stages = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  StreamShared* sh = reinterpret_cast<StreamShared*>(stages + kStreamWarps * kStreamStages * kSubBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x < kStreamWarps * kStreamStages) mbar_init(&sh->full[0][0] + threadIdx.x, 1);
  if (threadIdx.x == 0) sh->abort = 0;
  fence_mbar_init();
  __syncthreads();
  pdl_wait();  // logits and row counts may come from the previous kernel in the stream
  pdl_launch_dependents();

  // This warp's run of units [u_begin, u_end), unit = row * nchunks + chunk.
  const int64_t U = static_cast<int64_t>(a.n_rows) * a.nchunks;
  const int64_t NW = static_cast<int64_t>(gridDim.x) * kStreamWarps;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kStreamWarps + warp;
  const int64_t u_begin = U * gw / NW, u_end = U * (gw + 1) / NW;
  StreamGeom g;
  g.nchunks = a.nchunks;
  g.last_subs = ((a.V - (a.nchunks - 1) * CE) * EB + kSubBytes - 1) / kSubBytes;
  g.row_end = static_cast<int>(u_end / a.nchunks);
  g.chunk_end = static_cast<int>(u_end - static_cast<int64_t>(g.row_end) * a.nchunks);
  StreamPos start{static_cast<int>(u_begin / a.nchunks), 0, 0};
  start.chunk = static_cast<int>(u_begin - static_cast<int64_t>(start.row) * a.nchunks);
  if (g.before_end(start) && row_skipped(a, start.row)) {
    start.chunk = g.nchunks - 1;
    start.s = g.subs(start.chunk) - 1;
    stream_advance(a, g, start);  // moves on to the next live row
  }
  uint8_t* ring = stages + warp * kStreamStages * kSubBytes;
  uint64_t* full = sh->full[warp];
  volatile int* abort_flag = &sh->abort;
  const uint64_t pol = l2_policy_evict_first();

  // Issue side (lane 0 copies; every lane keeps the same bookkeeping).
  StreamPos issue = start;
  uint32_t n_issued = 0;
  auto issue_one = [&]() {
    int e0, e1;
    uint32_t bytes;
    sub_range<DT>(a, issue, e0, e1, bytes);
    const uint32_t slot = n_issued % kStreamStages;
    if (lane == 0) {
      mbar_arrive_expect_tx(&full[slot], bytes);
      if (bytes > 0) {
        const char* src = a.logits + static_cast<int64_t>(issue.row) * a.row_stride_bytes + static_cast<int64_t>(e0) * EB;
        bulk_load_g2s(ring + slot * kSubBytes, src, bytes, &full[slot], pol);
      }
    }
    ++n_issued;
    stream_advance(a, g, issue);
  };
  for (int k = 0; k < kStreamStages && g.before_end(issue); ++k) issue_one();

  // Consume side.
  StreamPos cur = start;
  uint32_t q = 0;
  bool poisoned = false;
  int seg_row = -1, seg_c0 = 0;
  float am = -INFINITY, S = 0.f, T = 0.f;
  int ai = INT_MAX;
  while (g.before_end(cur)) {
    const int row = cur.row, chunk = cur.chunk;
    if (row != seg_row) {  // a new row segment
      seg_row = row;
      seg_c0 = chunk;
      am = -INFINITY;
      ai = INT_MAX;
      S = 0.f;
      T = 0.f;
    }
    const uint32_t slot = q % kStreamStages;
    if (!poisoned) {
      const bool ok = mbar_wait_bounded(&full[slot], (q / kStreamStages) & 1u, abort_flag, a.dev_err, kStreamWaitNs);
      poisoned = !__all_sync(0xffffffffu, ok);
    }
    int e0, e1;
    uint32_t bytes;
    sub_range<DT>(a, cur, e0, e1, bytes);
    if (!poisoned && bytes == kSubBytes) {
      stream_full_sub<DT>(reinterpret_cast<const uint4*>(ring + slot * kSubBytes), e0, lane, am, ai, S, T);
    } else if (!poisoned) {  // the ragged last stretch of a row
      const uint4* sv = reinterpret_cast<const uint4*>(ring + slot * kSubBytes);
      const int nvec = static_cast<int>(bytes / 16);
      uint4 v[kSubVecPerLane];
#pragma unroll
      for (int k = 0; k < kSubVecPerLane; ++k)
        if (lane + 32 * k < nvec) v[k] = sv[lane + 32 * k];
      const int tb = e0 + nvec * PV;  // elements past the last whole vector (row end only)
      const bool has_tail = lane < e1 - tb;
      const float xt = has_tail
                           ? load_one<DT>(a.logits + static_cast<int64_t>(row) * a.row_stride_bytes, tb + lane)
                           : -INFINITY;
      // pass 1: the lane's largest vector maximum (the earliest vector on ties), then the
      // lowest index attaining it inside that vector
      float m = -INFINITY;
      int kb = 0;
#pragma unroll
      for (int k = 0; k < kSubVecPerLane; ++k) {
        if (lane + 32 * k < nvec) {
          const float vm = vec_max<DT>(v[k]);
          if (vm > m) {
            m = vm;
            kb = k;
          }
        }
      }
      int mi = INT_MAX;
      if (lane + 32 * kb < nvec) {
        uint4 w = v[0];
#pragma unroll
        for (int k = 1; k < kSubVecPerLane; ++k)
          if (k == kb) w = v[k];
        float x[PV];
        unpack<DT>(w, x);
        const int jb = e0 + (lane + 32 * kb) * PV;
#pragma unroll
        for (int e = PV - 1; e >= 0; --e)
          if (x[e] == m || (m == -INFINITY && !(x[e] > m))) mi = jb + e;
      }
      if (has_tail && (xt > m || mi == INT_MAX)) {
        m = xt;
        mi = tb + lane;
      }
      // S and T stay relative to the lane's running maximum am; rescale them when it grows
      const float am_old = am;
      ent_argmax_merge(am, ai, m, mi);
      if (am > am_old && S > 0.f) {
        const float d = (am_old - am) * kLog2e;
        const float f = ex2_approx(d);
        T = f * fmaf(d, S, T);
        S *= f;
      }
      // pass 2: S += 2^d, T += d 2^d, d = (x - am) log2 e clamped at -127 (2^d flushes to 0)
      const float M2 = am * kLog2e;
      float S1 = 0.f, T1 = 0.f;
#pragma unroll
      for (int k = 0; k < kSubVecPerLane; ++k) {
        if (lane + 32 * k < nvec) {
          float x[PV];
          unpack<DT>(v[k], x);
#pragma unroll
          for (int e = 0; e < PV; ++e) {
            const float d = fmaxf(fmaf(x[e], kLog2e, -M2), -127.f);
            const float p = ex2_approx(d);
            if (e & 1) {
              S1 += p;
              T1 = fmaf(p, d, T1);
            } else {
              S += p;
              T = fmaf(p, d, T);
            }
          }
        }
      }
      if (has_tail) {
        const float d = fmaxf(fmaf(xt, kLog2e, -M2), -127.f);
        const float p = ex2_approx(d);
        S += p;
        T = fmaf(p, d, T);
      }
      S += S1;
      T += T1;
    }
    __syncwarp();  // every lane is done with this stage
    if (!poisoned && g.before_end(issue)) {
      fence_proxy_async_smem();  // the stage's reads come before the copy that refills it
      issue_one();
    }
    ++q;
    stream_advance(a, g, cur);
    if (!g.before_end(cur) || cur.row != row)
      stream_finish_segment(a, row, seg_c0, chunk, EntPart{am, ai, S, T}, poisoned);
  }
  if (poisoned && lane == 0) {  // let the copies still in flight land before the CTA exits
    int local_abort = 0;
    for (uint32_t k = q; k < n_issued; ++k)
      mbar_wait_bounded(&full[k % kStreamStages], (k / kStreamStages) & 1u, &local_abort, nullptr, kStreamWaitNs);
  }
}

}  // namespace

int entropy_chunk_elems(int32_t dtype) {
  return dtype == EC_F32 ? chunk_elems<EC_F32>() : chunk_elems<EC_BF16>();
}

int32_t entropy_num_chunks(int32_t V, int32_t dtype) {
  const int ce = entropy_chunk_elems(dtype);
  return static_cast<int32_t>((static_cast<int64_t>(V) + ce - 1) / ce);
}

template <int DT>
cudaError_t launch_stream(int grid, cudaStream_t s, const EntArgs& a) {
  const cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(entropy_stream_kernel<DT>), stream_smem_bytes<DT>());
  if (e != cudaSuccess) return e;
  return launch_pdl(entropy_stream_kernel<DT>, dim3(grid), dim3(kStreamThreads), stream_smem_bytes<DT>(), s, a);
}

size_t entropy_workspace_bytes(int32_t n_rows, int32_t V, int32_t dtype) {
  const size_t nch = static_cast<size_t>(entropy_num_chunks(V, dtype));
  const size_t rows = static_cast<size_t>(n_rows > 0 ? n_rows : 0);
  return align_up(rows * nch * sizeof(ChunkPartial), 256) + align_up(rows * sizeof(uint32_t), 256);
}

cudaError_t launch_entropy_decode(const void* logits, int64_t row_stride, int32_t n_rows, int32_t V,
                                  int32_t dtype, int32_t* ids, float* entropy, float* log_conf, void* ws,
                                  const int32_t* row_count, int32_t rows_per_group, bool allow_cluster,
                                  bool publish_only, int32_t* dev_err, cudaStream_t s) {
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
            publish_only ? 1 : 0, row_count, rows_per_group, n_rows, dev_err};
  int sms = 0;
  const cudaError_t e = current_device_sms(&sms);
  if (e != cudaSuccess) return e;
  const int64_t total_bytes = static_cast<int64_t>(n_rows) * V * (f32 ? 4 : 2);
  // not in publish-only mode (inside a step): the persistent CTAs cannot start beside the
  // previous kernel, and the split CTAs can
  if (!publish_only && ws != nullptr && nch > 1 && total_bytes >= kStreamMinBytes) {
    const int64_t units = static_cast<int64_t>(n_rows) * nch;
    const int grid = static_cast<int>(std::min<int64_t>(sms, (units + kStreamWarps - 1) / kStreamWarps));
    if (f32) return launch_stream<EC_F32>(grid, s, a);
    return launch_stream<EC_BF16>(grid, s, a);
  }
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
