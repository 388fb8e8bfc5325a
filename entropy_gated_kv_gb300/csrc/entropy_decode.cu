// entropy_decode.cu — stage (a) of the EntropyCache step: fused softmax, greedy decode and
// Shannon entropy over the V-wide logits of each candidate row.
//
// Defines, per row i (EntropyCache, gist.science zh summary §2.2, the max-entropy
// equation's inner term; decode = greedy argmax):
//   ids[i] = lowest j attaining max_j x_ij
//   entropy[i] = -sum_j p_ij ln p_ij,  p_ij = softmax_j(x_ij)
//   log_conf[i] = ln p_{i, ids[i]} = -ln S_i,  S_i = sum_j exp(x_ij - max)
//
// Design (HBM-bound: every logit is read exactly once). The unit of work is a piece of a row:
// 32 lanes x 4 sixteen-byte vectors (1024 bf16 or 512 fp32 elements), reduced by one warp with
// no CTA barrier:
//   - pass 1: each lane's maximum (a bf16x2 max tree for bf16), then the warp's maximum with one
//     redux.sync; only the lanes holding that maximum look for their lowest index, and a
//     redux.sync minimum picks the warp's lowest;
//   - pass 2: S = sum 2^d and T = sum d 2^d with d = (x - M) log2(e) relative to the warp's
//     maximum M (paired fp32 instructions, two elements each), summed over the warp by
//     shuffles; H = ln2 (log2 S - T/S).
// The 8 warps of a CTA take the 8 pieces of a chunk (8192 bf16 / 4096 fp32 elements), merge
// them in shared memory and publish the chunk's (max, index, S, T) to the workspace; rows are
// merged by rescaling (entropy_merge.cuh): by a merge kernel (one warp per row), or inside a
// step by the select kernel. Launch shapes:
//   - split: one CTA per chunk, every load in flight at once (the shape of the fastest plain
//     read of these sizes on this GPU: 2.7 us for 8 MB, 11.9 us for 78 MB);
//   - few rows outside a step (the whole problem within about one wave): one cluster of up to
//     8 CTAs per row, its warps on double-width pieces (8 vectors per lane); each CTA merges
//     its warps in shared memory and the first CTA merges the CTAs through distributed shared
//     memory, so no workspace is needed.
#include <algorithm>
#include <climits>

#include "ec_common.cuh"
#include "ec_internal.h"
#include "entropy_merge.cuh"

namespace ec {
namespace {

constexpr int kThreads = 256;  // 8 warps per CTA
constexpr int kWarps = kThreads / 32;
constexpr int kLaneVec = 4;     // 16-byte vectors per lane per piece (the split launch in a step)
constexpr int kAloneVec = 6;    // the split launch outside a step (many rows: fewer, larger pieces)
constexpr int kWideVec = 8;     // the cluster launch's double-width pieces
// Pass 2 in scalar fp32 or on the paired f32x2 instructions, per launch: the form each launch
// measured faster in (the split launch paired, the cluster launch scalar).
constexpr bool kSplitScalar = false;
constexpr bool kWideScalar = true;
constexpr int kMaxCluster = 8;  // CTAs per row (portable cluster size)
constexpr int kClusterCtasPerSmBf16 = 4;  // cluster path while rows x cluster <= this x SMs (all resident;
constexpr int kClusterCtasPerSmF32 = 2;   // the cluster kernel's launch bounds per type)
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

template <int DT, int LV = kLaneVec>
constexpr int piece_elems() {  // elements of one piece (the workspace holds one partial per piece)
  return 32 * LV * Elem<DT>::kPerVec;
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

// Packed helpers: bf16x2 maximum (a NaN operand yields the other one) and the sm_100 paired
// fp32 operations, two lanes of arithmetic per instruction.
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
// Warp-wide maximum of a float, one instruction.
__device__ __forceinline__ float warp_max_f32(float v) {
  float r;
  asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
  return r;
}

// Logits below this are treated as -inf by the sums (2^d is 0 for them either way); keeping
// d finite makes d 2^d exactly 0 instead of -inf * 0.
constexpr uint32_t kClampBf16x2 = 0xF149F149u;  // (-9.95e29, -9.95e29) as bf16
constexpr float kClampF32 = -1e30f;
constexpr uint32_t kNegInfBf16x2 = 0xFF80FF80u;
constexpr uint32_t kNegInfF32 = 0xFF800000u;

// Pass 2 over one pair of elements: S += 2^d, T += d 2^d with d = x log2 e - M2.
__device__ __forceinline__ void st_pair(uint64_t x, uint64_t l2e, uint64_t nm, uint64_t& s, uint64_t& t) {
  const uint64_t d = fma2(x, l2e, nm);
  float dl, dh;
  unf2(d, dl, dh);
  const uint64_t p = f2(ex2_approx(dl), ex2_approx(dh));
  s = add2(s, p);
  t = fma2(p, d, t);
}

using Part = EntPart;

__device__ __forceinline__ void write_row(int row, const Part& p, int32_t* ids, float* entropy, float* log_conf) {
  ids[row] = p.i;
  ent_finish(p, entropy[row], log_conf[row]);
}

struct EntArgs {
  const char* logits;
  int64_t row_stride_bytes;
  int32_t V, nparts;  // nparts: chunks (8 pieces) per row, the partials per row in the workspace
  int32_t* ids;
  float* entropy;
  float* log_conf;
  ChunkPartial* partials;  // [n_rows][nparts]
  const int32_t* row_count;
  int32_t rows_per_group;
  int32_t n_rows;
};

// Rows past their group's count are skipped (uniform over a CTA and over a cluster).
__device__ __forceinline__ bool row_skipped(const EntArgs& a, int row) {
  if (a.row_count == nullptr) return false;
  const int grp = row / a.rows_per_group;
  return row - grp * a.rows_per_group >= __ldg(a.row_count + grp);
}

// One lane's share of a piece [base, end) of a row: vector u of lane L holds the elements
// from base + PV (L + 32 u) on (PV = 8 for bf16, 4 for fp32), so a warp reads 512 contiguous
// bytes per u. Vectors past the piece hold -inf. The row's last few elements, when V is not a
// multiple of the vector width, are the piece's tail: lane t < ntail holds element tail0 + t.
template <int DT, int LV = kLaneVec>
struct Piece {
  uint4 v[LV];
  float xt;
  int nvec;   // whole vectors in the piece
  int ntail;  // elements after them (fewer than one vector; the row's end only)
  int base;   // first element of the piece
};

template <int DT, int LV>
__device__ __forceinline__ void piece_geometry(Piece<DT, LV>& pc, int V, int base) {
  constexpr int PV = Elem<DT>::kPerVec;
  const int end = min(V, base + piece_elems<DT, LV>());
  pc.base = base;
  pc.nvec = (end - base) / PV;
  pc.ntail = end - base - pc.nvec * PV;
}

template <int DT>
__device__ __forceinline__ uint4 neg_inf_vec() {
  constexpr uint32_t n = DT == EC_BF16 ? kNegInfBf16x2 : kNegInfF32;
  return make_uint4(n, n, n, n);
}

// Loads a piece with plain 16-byte streaming loads (every load of the lane issued at once).
template <int DT, int LV>
__device__ __forceinline__ void load_piece(Piece<DT, LV>& pc, const char* __restrict__ rowp, int V, int base) {
  constexpr int PV = Elem<DT>::kPerVec;
  constexpr int EB = Elem<DT>::kBytes;
  const int lane = threadIdx.x & 31;
  piece_geometry(pc, V, base);
#pragma unroll
  for (int u = 0; u < LV; ++u) {
    const int j = lane + 32 * u;
    pc.v[u] = j < pc.nvec ? ld_stream_v4(rowp + (static_cast<int64_t>(base) + j * PV) * EB) : neg_inf_vec<DT>();
  }
  pc.xt = lane < pc.ntail ? load_one<DT>(rowp, base + pc.nvec * PV + lane) : -INFINITY;
}

// Largest element of one vector.
template <int DT>
__device__ __forceinline__ float vec_max(const uint4& v) {
  if constexpr (DT == EC_F32) {
    return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)), fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
  } else {
    const uint32_t c = bmax2(bmax2(v.x, v.y), bmax2(v.z, v.w));
    return fmaxf(bf16lo_to_f32(c), bf16hi_to_f32(c));
  }
}

// The warp's (max, lowest index, S, T) over one piece; every lane returns it. Whole warp.
template <int DT, int LV, bool SCALAR>
__device__ __forceinline__ Part reduce_piece(const Piece<DT, LV>& pc) {
  constexpr int PV = Elem<DT>::kPerVec;
  const int lane = threadIdx.x & 31;
  const int nmine = lane < pc.nvec ? min(LV, (pc.nvec - lane + 31) / 32) : 0;
  const bool has_tail = lane < pc.ntail;

  // pass 1: the lane's maximum, the warp's maximum, the warp's lowest index attaining it
  float vm[LV];
#pragma unroll
  for (int u = 0; u < LV; ++u) vm[u] = vec_max<DT>(pc.v[u]);
  float m = vm[0];
#pragma unroll
  for (int u = 1; u < LV; ++u) m = fmaxf(m, vm[u]);
  if (has_tail) m = fmaxf(m, pc.xt);
  const float M = warp_max_f32(m);
  uint32_t idx = 0x7FFFFFFFu;
  if (m == M && (nmine > 0 || has_tail)) {  // this lane holds the maximum: its first occurrence
    int ub = -1;
#pragma unroll
    for (int u = LV - 1; u >= 0; --u)
      if (u < nmine && vm[u] == M) ub = u;
    if (ub >= 0) {
      uint4 w = pc.v[0];
#pragma unroll
      for (int u = 1; u < LV; ++u)
        if (u == ub) w = pc.v[u];
      float x[PV];
      unpack<DT>(w, x);
      int e0 = PV - 1;
#pragma unroll
      for (int e = PV - 1; e >= 0; --e)
        if (x[e] == M) e0 = e;
      idx = static_cast<uint32_t>(pc.base + (lane + 32 * ub) * PV + e0);
    } else {
      idx = static_cast<uint32_t>(pc.base + pc.nvec * PV + lane);  // the tail element
    }
  }
  idx = __reduce_min_sync(0xffffffffu, idx);

  // pass 2: S = sum 2^d, T = sum d 2^d, d = x log2 e - M log2 e (-inf clamped, giving 0)
  const float M2 = M == -INFINITY ? 0.f : M * kLog2e;
  const uint64_t l2e = f2(kLog2e, kLog2e), nm = f2(-M2, -M2);
  uint64_t sa = 0, sb = 0, ta = 0, tb = 0;  // two accumulator pairs (0 is +0.0f, +0.0f)
  float q0 = 0.f, q1 = 0.f, r0 = 0.f, r1 = 0.f;  // scalar accumulators (double-width pieces)
#pragma unroll
  for (int u = 0; u < LV; ++u) {
    if constexpr (DT == EC_BF16 && SCALAR) {
      const uint32_t w[4] = {pc.v[u].x, pc.v[u].y, pc.v[u].z, pc.v[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t cl = bmax2(w[j], kClampBf16x2);
        const float dl = fmaf(bf16lo_to_f32(cl), kLog2e, -M2), dh = fmaf(bf16hi_to_f32(cl), kLog2e, -M2);
        const float pl = ex2_approx(dl), ph = ex2_approx(dh);
        q0 += pl;
        q1 += ph;
        r0 = fmaf(pl, dl, r0);
        r1 = fmaf(ph, dh, r1);
      }
    } else if constexpr (DT == EC_BF16) {
      const uint32_t w[4] = {pc.v[u].x, pc.v[u].y, pc.v[u].z, pc.v[u].w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t cl = bmax2(w[j], kClampBf16x2);
        const uint64_t x = f2(bf16lo_to_f32(cl), bf16hi_to_f32(cl));
        if (j & 1) st_pair(x, l2e, nm, sb, tb);
        else st_pair(x, l2e, nm, sa, ta);
      }
    } else {
      const uint64_t x0 = f2(fmaxf(__uint_as_float(pc.v[u].x), kClampF32), fmaxf(__uint_as_float(pc.v[u].y), kClampF32));
      const uint64_t x1 = f2(fmaxf(__uint_as_float(pc.v[u].z), kClampF32), fmaxf(__uint_as_float(pc.v[u].w), kClampF32));
      st_pair(x0, l2e, nm, sa, ta);
      st_pair(x1, l2e, nm, sb, tb);
    }
  }
  float s0, s1, t0, t1;
  unf2(add2(sa, sb), s0, s1);
  unf2(add2(ta, tb), t0, t1);
  float S = s0 + s1 + (q0 + q1), T = t0 + t1 + (r0 + r1);
  if (has_tail) {
    const float d = fmaxf(fmaf(pc.xt, kLog2e, -M2), -127.f);
    const float p = ex2_approx(d);
    S += p;
    T = fmaf(p, d, T);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    S += __shfl_xor_sync(0xffffffffu, S, off);
    T += __shfl_xor_sync(0xffffffffu, T, off);
  }
  return Part{M, static_cast<int>(idx), S, T};
}

// Merges the 8 warps' parts of one chunk (8 consecutive pieces) in shared memory and
// publishes the chunk's partial. All threads of the CTA; `has` is false for a warp whose
// piece lies past the row's end.
__device__ __forceinline__ void publish_chunk(const EntArgs& a, int row, int chunk, const Part& p, bool has,
                                              Part* wpart) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (lane == 0) wpart[warp] = has ? p : Part{-INFINITY, INT_MAX, 0.f, 0.f};
  __syncthreads();
  if (warp == 0) {
    Part q = lane < kWarps ? wpart[lane] : Part{-INFINITY, INT_MAX, 0.f, 0.f};
#pragma unroll
    for (int off = 1; off < kWarps; off <<= 1) {
      const Part o{__shfl_xor_sync(0xffffffffu, q.m, off), __shfl_xor_sync(0xffffffffu, q.i, off),
                   __shfl_xor_sync(0xffffffffu, q.s, off), __shfl_xor_sync(0xffffffffu, q.t, off)};
      ent_part_merge(q, o);
    }
    if (lane == 0) a.partials[static_cast<int64_t>(row) * a.nparts + chunk] = ChunkPartial{q.m, q.i, q.s, q.t};
  }
}

// Split path: CTA (row, c) takes chunk c of the row (pieces 8 c .. 8 c + 7, one per warp, of
// LV vectors per lane). Every instantiation is held to 6 resident CTAs per SM (at most 40
// registers). For the standalone launch (kAloneVec pieces, many rows) that keeps more loads in
// flight per SM (measured faster at 78 MB: 18.9 -> 18.1 us); the step's 4-vector pieces need no
// more than that anyway (39 registers unbounded; a bound of 1 CTA let them grow to 67 and slowed
// the step).
template <int DT, int LV>
__global__ void __launch_bounds__(kThreads, 6) entropy_split_kernel(EntArgs a) {
  __shared__ Part wpart[kWarps];
  pdl_wait();  // logits and row counts may come from the previous kernel in the stream
  pdl_launch_dependents();
  const int row = static_cast<int>(blockIdx.x) / a.nparts;  // the grid has fewer than 2^31 CTAs
  const int chunk = static_cast<int>(blockIdx.x) - row * a.nparts;
  if (row_skipped(a, row)) return;  // uniform over the CTA
  const int base = (chunk * kWarps + static_cast<int>(threadIdx.x >> 5)) * piece_elems<DT, LV>();
  const bool has = base < a.V;  // uniform over the warp
  Part p{};
  if (has) {
    Piece<DT, LV> pc;
    load_piece(pc, a.logits + static_cast<int64_t>(row) * a.row_stride_bytes, a.V, base);
    p = reduce_piece<DT, LV, kSplitScalar>(pc);
  }
  publish_chunk(a, row, chunk, p, has, wpart);
}

// Waits for the first phase of a barrier that other CTAs of the cluster complete with remote
// stores (acquire at cluster scope: their data is visible once it returns true). Gives up after
// kLandedWaitNs of wall time (the stores are issued right after a cluster barrier, so this
// never binds unless the hardware misbehaves).
constexpr uint64_t kLandedWaitNs = 1000000000ull;
__device__ __forceinline__ bool wait_landed(uint64_t* bar) {
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 0;; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], 0;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar))
        : "memory");
    if (done) return true;
    if ((i & 63u) == 63u && global_timer_ns() - t0 > kLandedWaitNs) return false;
  }
}

// Cluster path: one cluster per row; CTA `rank` of the cluster takes a contiguous run of the
// row's double-width pieces (8 vectors per lane, 2048 bf16 elements), its warps take every
// 8th piece of the run (at the sizes it serves, one piece each, all loads in flight at once),
// and the 8 warps merge in shared memory. Each other CTA then pushes its 16-byte partial into
// the first CTA's shared memory with one asynchronous remote store, counted on the first CTA's
// barrier, and exits; the first CTA merges the cluster's partials and writes the row. The one
// cluster barrier (which publishes the first CTA's barrier before any store into it) is
// arrived at on entry and waited on only before the store, so it overlaps the loads. bf16 is
// held to 4 CTAs per SM (64 registers): measured faster than 2 (127) or 3 (79) at 32 rows of
// 126464. fp32 keeps 2 (at 64 registers it spills, and the 32-row fp32 decode slowed).
template <int DT>
__global__ void __launch_bounds__(kThreads, DT == EC_BF16 ? 4 : 2) entropy_cluster_kernel(EntArgs a) {
  __shared__ __align__(16) Part wpart[kWarps];
  __shared__ __align__(16) Part slices[kMaxCluster];  // the first CTA: one partial per CTA of the cluster
  __shared__ __align__(8) uint64_t landed;            // the first CTA: the other CTAs' partials are in
  pdl_wait();  // logits and row counts may come from the previous kernel in the stream
  pdl_launch_dependents();
  const int csize = static_cast<int>(cluster_size());
  const int rank = static_cast<int>(cluster_ctarank());
  const int row = static_cast<int>(cluster_id_x());
  if (row_skipped(a, row)) return;  // the whole cluster skips the row
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (rank == 0 && threadIdx.x == 0) {
    mbar_init(&landed, 1);
    fence_mbar_init();
  }
  cluster_arrive_release();
  const char* rowp = a.logits + static_cast<int64_t>(row) * a.row_stride_bytes;
  constexpr int LV = kWideVec;
  constexpr int PE = piece_elems<DT, LV>();
  const int nwide = (a.V + PE - 1) / PE;
  const int per = (nwide + csize - 1) / csize;
  const int p0 = rank * per, p1 = min(nwide, p0 + per);
  Part acc{-INFINITY, INT_MAX, 0.f, 0.f};
  for (int piece = p0 + warp; piece < p1; piece += kWarps) {
    Piece<DT, LV> pc;
    load_piece(pc, rowp, a.V, piece * PE);
    ent_part_merge(acc, reduce_piece<DT, LV, kWideScalar>(pc));
  }
  if (lane == 0) wpart[warp] = acc;
  __syncthreads();
  cluster_wait_acquire();  // the first CTA's barrier is initialised
  if (warp != 0) return;
  Part p = lane < kWarps ? wpart[lane] : Part{-INFINITY, INT_MAX, 0.f, 0.f};
#pragma unroll
  for (int off = 1; off < kWarps; off <<= 1) {
    const Part o{__shfl_xor_sync(0xffffffffu, p.m, off), __shfl_xor_sync(0xffffffffu, p.i, off),
                 __shfl_xor_sync(0xffffffffu, p.s, off), __shfl_xor_sync(0xffffffffu, p.t, off)};
    ent_part_merge(p, o);
  }
  if (rank != 0) {
    if (lane == 0)
      st_async_v4(dsmem_map(smem_u32(&slices[rank]), 0u),
                  make_uint4(__float_as_uint(p.m), static_cast<uint32_t>(p.i), __float_as_uint(p.s),
                             __float_as_uint(p.t)),
                  dsmem_map(smem_u32(&landed), 0u));
    return;
  }
  if (lane == 0) {
    slices[0] = p;
    mbar_arrive_expect_tx(&landed, static_cast<uint32_t>(csize - 1) * 16u);
  }
  __syncwarp();
  if (!__all_sync(0xffffffffu, wait_landed(&landed))) {
    // a partial never arrived: mark the row (the decode entries carry no error word)
    if (lane == 0) {
      a.ids[row] = -1;
      a.entropy[row] = __int_as_float(0x7FC00000);
      a.log_conf[row] = __int_as_float(0x7FC00000);
    }
    return;
  }
  Part q = Part{-INFINITY, INT_MAX, 0.f, 0.f};
  if (lane < csize) q = slices[lane];
#pragma unroll
  for (int off = 1; off < kMaxCluster; off <<= 1) {
    const Part o{__shfl_xor_sync(0xffffffffu, q.m, off), __shfl_xor_sync(0xffffffffu, q.i, off),
                 __shfl_xor_sync(0xffffffffu, q.s, off), __shfl_xor_sync(0xffffffffu, q.t, off)};
    ent_part_merge(q, o);
  }
  if (lane == 0) write_row(row, q, a.ids, a.entropy, a.log_conf);
}

// Merges each row's chunk partials (one warp per row) and writes the row's results.
__global__ void __launch_bounds__(256) entropy_merge_kernel(EntArgs a) {
  pdl_wait();  // the partials come from the previous kernel
  pdl_launch_dependents();
  const int row = static_cast<int>(blockIdx.x) * 8 + static_cast<int>(threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= a.n_rows || row_skipped(a, row)) return;
  const ChunkPartial* rp = a.partials + static_cast<int64_t>(row) * a.nparts;
  Part r{-INFINITY, INT_MAX, 0.f, 0.f};
  for (int c = lane; c < a.nparts; c += 32)  // chunks in increasing order per lane
    ent_part_merge(r, Part{__ldcg(&rp[c].m), __ldcg(&rp[c].idx), __ldcg(&rp[c].s), __ldcg(&rp[c].t)});
  r = ent_warp_merge(r);
  if (lane == 0) write_row(row, r, a.ids, a.entropy, a.log_conf);
}

}  // namespace

int32_t entropy_num_chunks(int32_t V, int32_t dtype) {
  const int ce = kWarps * (dtype == EC_F32 ? piece_elems<EC_F32>() : piece_elems<EC_BF16>());
  return static_cast<int32_t>((static_cast<int64_t>(V) + ce - 1) / ce);
}

size_t entropy_workspace_bytes(int32_t n_rows, int32_t V, int32_t dtype) {
  const size_t np = static_cast<size_t>(entropy_num_chunks(V, dtype));
  const size_t rows = static_cast<size_t>(n_rows > 0 ? n_rows : 0);
  return align_up(rows * np * sizeof(ChunkPartial), 256);
}

cudaError_t launch_entropy_decode(const void* logits, int64_t row_stride, int32_t n_rows, int32_t V,
                                  int32_t dtype, int32_t* ids, float* entropy, float* log_conf, void* ws,
                                  const int32_t* row_count, int32_t rows_per_group, bool allow_cluster,
                                  bool publish_only, cudaStream_t s) {
  if (n_rows == 0) return cudaSuccess;
  const bool f32 = dtype == EC_F32;
  const int32_t np = entropy_num_chunks(V, dtype);
  const EntArgs a{static_cast<const char*>(logits), row_stride * (f32 ? 4 : 2), V, np, ids, entropy, log_conf,
                  static_cast<ChunkPartial*>(ws), row_count, rows_per_group, n_rows};
  int sms = 0;
  cudaError_t e = current_device_sms(&sms);
  if (e != cudaSuccess) return e;
  // the cluster launch: CTAs of 8 double-width pieces, at most kMaxCluster per row
  const int64_t wide = kWarps * (f32 ? piece_elems<EC_F32, kWideVec>() : piece_elems<EC_BF16, kWideVec>());
  const int csize = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(kMaxCluster, (V + wide - 1) / wide)));
  const int64_t cluster_ctas = static_cast<int64_t>(n_rows) * csize;
  const int per_sm = f32 ? kClusterCtasPerSmF32 : kClusterCtasPerSmBf16;
  if (!publish_only && (ws == nullptr || (allow_cluster && cluster_ctas <= static_cast<int64_t>(per_sm) * sms))) {
    // few rows, or no workspace: merge on chip, write the rows
    if (cluster_ctas > INT_MAX) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(cluster_ctas));
    if (f32) return launch_pdl_cluster(entropy_cluster_kernel<EC_F32>, grid, dim3(kThreads), 0, csize, s, a);
    return launch_pdl_cluster(entropy_cluster_kernel<EC_BF16>, grid, dim3(kThreads), 0, csize, s, a);
  }
  const int64_t units = static_cast<int64_t>(n_rows) * np;
  if (units > INT_MAX) return cudaErrorInvalidValue;
  const dim3 grid(static_cast<unsigned>(units));
  // outside a step: chunks of the wider pieces (fewer partials than the workspace holds)
  const int64_t ce_alone = kWarps * (f32 ? piece_elems<EC_F32, kAloneVec>() : piece_elems<EC_BF16, kAloneVec>());
  EntArgs a_alone = a;
  a_alone.nparts = static_cast<int32_t>((static_cast<int64_t>(V) + ce_alone - 1) / ce_alone);
  const dim3 grid_alone(static_cast<unsigned>(static_cast<int64_t>(n_rows) * a_alone.nparts));
  // inside a step (publish only) the pieces have the width the select kernel's merge expects;
  // outside, many rows take the wider pieces (measured faster at 78 MB, slower in the step)
  if (publish_only)
    e = f32 ? launch_pdl(entropy_split_kernel<EC_F32, kLaneVec>, grid, dim3(kThreads), 0, s, a)
            : launch_pdl(entropy_split_kernel<EC_BF16, kLaneVec>, grid, dim3(kThreads), 0, s, a);
  else
    e = f32 ? launch_pdl(entropy_split_kernel<EC_F32, kAloneVec>, grid_alone, dim3(kThreads), 0, s, a_alone)
            : launch_pdl(entropy_split_kernel<EC_BF16, kAloneVec>, grid_alone, dim3(kThreads), 0, s, a_alone);
  if (e != cudaSuccess || publish_only) return e;
  return launch_pdl(entropy_merge_kernel, dim3((n_rows + 7) / 8), dim3(256), 0, s, a_alone);
}

}  // namespace ec
