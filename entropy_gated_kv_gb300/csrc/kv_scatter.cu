// kv_scatter.cu — K/V cache refresh of the recompute set (stage (c) of the EntropyCache
// step) and, inside a whole step, the gather of the recompute rows' queries.
//
// EntropyCache, gist.science zh summary §2.2 (partial forward): only the recompute set gets
// fresh K/V, every other position is read from the cache; a full forward refreshes all rows.
//   k_cache[b, idx[b, r]] = k_new[b, src]   (src = r, or idx[b, r] when the fresh rows are
//   v_cache[b, idx[b, r]] = v_new[b, src]    indexed by position), for r < R[b]
//   q_dst[b, r] = q_src[b, idx[b, r]]        (optional)
//
// A pure copy (HBM-bound, bytes = 2 reads + 2 writes of R * Hkv * D bf16, plus the query
// rows). One warp per row; each lane moves 16-byte vectors, four loads in flight before the
// stores. The grid is sized from L and the batch (R lives on the device) and warps stride
// over the rows.
#include "ec_common.cuh"
#include "ec_internal.h"

namespace ec {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

__device__ __forceinline__ uint4 ld_nc(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// Copies n16 16-byte vectors from src to dst with the 32 lanes of a warp.
__device__ __forceinline__ void warp_copy(uint4* __restrict__ dst, const uint4* __restrict__ src, int n16, int lane) {
  int c = lane;
  for (; c + 96 < n16; c += 128) {
    const uint4 a = ld_nc(src + c), b2 = ld_nc(src + c + 32), d = ld_nc(src + c + 64), e = ld_nc(src + c + 96);
    dst[c] = a;
    dst[c + 32] = b2;
    dst[c + 64] = d;
    dst[c + 96] = e;
  }
  for (; c < n16; c += 32) dst[c] = ld_nc(src + c);
}

__global__ void __launch_bounds__(kThreads) kv_scatter_kernel(
    int32_t L, int32_t kv_row16, int32_t q_row16, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, int32_t src_by_position,
    const int32_t* __restrict__ idx, const int32_t* __restrict__ R, const uint4* __restrict__ q_src,
    uint4* __restrict__ q_dst, int32_t* __restrict__ dev_err) {
  const int b = blockIdx.y;
  const int lane = threadIdx.x & 31;
  const int Rb = __ldg(R + b);
  if (Rb < 0 || Rb > L) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report_error(dev_err, EC_DEVERR_BAD_R);
    return;
  }
  const int64_t rowL = static_cast<int64_t>(b) * L;
  const int gw = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int nw = gridDim.x * kWarps;
  for (int r = gw; r < Rb; r += nw) {
    const int pos = __ldg(idx + rowL + r);
    if (pos < 0 || pos >= L) {
      if (lane == 0) report_error(dev_err, EC_DEVERR_BAD_IDX);
      continue;
    }
    const int src = src_by_position ? pos : r;
    const int64_t dst_off = (rowL + pos) * kv_row16;
    const int64_t src_off = (rowL + src) * kv_row16;
    warp_copy(k_cache + dst_off, k_new + src_off, kv_row16, lane);
    warp_copy(v_cache + dst_off, v_new + src_off, kv_row16, lane);
    if (q_dst != nullptr) warp_copy(q_dst + (rowL + r) * q_row16, q_src + (rowL + pos) * q_row16, q_row16, lane);
  }
}

}  // namespace

cudaError_t launch_kv_scatter(const ec_params& p, void* k_cache, void* v_cache, const void* k_new,
                              const void* v_new, int32_t src_by_position, const int32_t* idx,
                              const int32_t* R, const void* q_src, void* q_dst, int32_t* dev_err,
                              cudaStream_t s) {
  const int32_t kv_row16 = p.Hkv * p.D * 2 / 16;
  const int32_t q_row16 = p.Hq * p.D * 2 / 16;
  const int64_t want = (static_cast<int64_t>(p.L) + kWarps - 1) / kWarps;
  const int64_t cap = std::max<int64_t>(1, 2432 / (static_cast<int64_t>(p.B) * kWarps));
  const int gx = static_cast<int>(std::max<int64_t>(1, std::min(want, cap)));
  const dim3 grid(gx, p.B);
  kv_scatter_kernel<<<grid, kThreads, 0, s>>>(p.L, kv_row16, q_row16, static_cast<uint4*>(k_cache),
                                              static_cast<uint4*>(v_cache), static_cast<const uint4*>(k_new),
                                              static_cast<const uint4*>(v_new), src_by_position, idx, R,
                                              static_cast<const uint4*>(q_src), static_cast<uint4*>(q_dst),
                                              dev_err);
  return cudaGetLastError();
}

}  // namespace ec
