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
// rows). One CTA per row with the whole row's loads in flight before its stores.
#include <algorithm>

#include "ec_common.cuh"
#include "ec_internal.h"

namespace ec {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxVecPerThread = 8;  // 16-byte vectors held per thread before the stores

__device__ __forceinline__ uint4 ld_nc(const uint4* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// One CTA moves one recompute row at a time: the K row, the V row and (optionally) the query
// row form one list of 16-byte vectors; each thread loads up to kMaxVecPerThread of them
// before storing any, so a whole row is in flight at once.
__global__ void __launch_bounds__(kThreads) kv_scatter_kernel(
    int32_t L, int32_t kv_row16, int32_t q_row16, uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
    const uint4* __restrict__ k_new, const uint4* __restrict__ v_new, int32_t src_by_position,
    const int32_t* __restrict__ idx, const int32_t* __restrict__ R, const uint4* __restrict__ q_src,
    uint4* __restrict__ q_dst, int32_t* __restrict__ dev_err) {
  const int b = blockIdx.y;
  pdl_wait();  // idx / R and the fresh rows may come from the previous kernels in the stream
  pdl_launch_dependents();
  const int Rb = __ldg(R + b);
  if (Rb < 0 || Rb > L) {
    if (blockIdx.x == 0 && threadIdx.x == 0) report_error(dev_err, EC_DEVERR_BAD_R);
    return;
  }
  const int64_t rowL = static_cast<int64_t>(b) * L;
  const int nq = q_dst != nullptr ? q_row16 : 0;
  const int total = 2 * kv_row16 + nq;
  for (int r = blockIdx.x; r < Rb; r += gridDim.x) {
    const int pos = __ldg(idx + rowL + r);
    if (pos < 0 || pos >= L) {
      if (threadIdx.x == 0) report_error(dev_err, EC_DEVERR_BAD_IDX);
      continue;
    }
    const int src = src_by_position ? pos : r;
    const int64_t dst_kv = (rowL + pos) * kv_row16;
    const int64_t src_kv = (rowL + src) * kv_row16;
    const int64_t dst_q = (rowL + r) * q_row16;
    const int64_t src_q = (rowL + pos) * q_row16;
    for (int base = 0; base < total; base += kThreads * kMaxVecPerThread) {
      uint4 v[kMaxVecPerThread];
#pragma unroll
      for (int u = 0; u < kMaxVecPerThread; ++u) {
        const int e = base + threadIdx.x + u * kThreads;
        if (e < kv_row16) v[u] = ld_nc(k_new + src_kv + e);
        else if (e < 2 * kv_row16) v[u] = ld_nc(v_new + src_kv + (e - kv_row16));
        else if (e < total) v[u] = ld_nc(q_src + src_q + (e - 2 * kv_row16));
      }
#pragma unroll
      for (int u = 0; u < kMaxVecPerThread; ++u) {
        const int e = base + threadIdx.x + u * kThreads;
        if (e < kv_row16) k_cache[dst_kv + e] = v[u];
        else if (e < 2 * kv_row16) v_cache[dst_kv + (e - kv_row16)] = v[u];
        else if (e < total) q_dst[dst_q + (e - 2 * kv_row16)] = v[u];
      }
    }
  }
}

}  // namespace

cudaError_t launch_kv_scatter(const ec_params& p, void* k_cache, void* v_cache, const void* k_new,
                              const void* v_new, int32_t src_by_position, const int32_t* idx,
                              const int32_t* R, const void* q_src, void* q_dst, int32_t* dev_err,
                              cudaStream_t s) {
  const int32_t kv_row16 = p.Hkv * p.D * 2 / 16;
  const int32_t q_row16 = p.Hq * p.D * 2 / 16;
  // one CTA per recompute row, at most two per SM in total so the whole grid is resident at
  // once (the next kernel can then launch early); R lives on the device, so CTAs stride over
  // the rows
  int sms = 0;
  const cudaError_t e = current_device_sms(&sms);
  if (e != cudaSuccess) return e;
  const int64_t cap = std::max<int64_t>(1, 2 * static_cast<int64_t>(sms) / p.B);
  const int gx = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(p.L, cap)));
  const dim3 grid(gx, p.B);
  return launch_pdl(kv_scatter_kernel, grid, dim3(kThreads), 0, s, p.L, kv_row16, q_row16,
                    static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), static_cast<const uint4*>(k_new),
                    static_cast<const uint4*>(v_new), src_by_position, idx, R, static_cast<const uint4*>(q_src),
                    static_cast<uint4*>(q_dst), dev_err);
}

}  // namespace ec
