// select_recompute.cu — stages (b) and (c) of the EntropyCache step as a kernel of their own
// (ec_select_recompute, and inside ec_step): one CTA per sequence runs select_prefetch and
// select_finish (select_device.cuh).
#include <cmath>

#include "ec_internal.h"
#include "select_device.cuh"

namespace ec {
namespace {

constexpr int kThreads = 512;

__global__ void __launch_bounds__(kThreads) select_recompute_kernel(SelArgs a) {
  extern __shared__ __align__(16) uint8_t dyn[];
  if (a.prefetch_early) {
    select_prefetch<kThreads>(a, blockIdx.x, dyn);
    pdl_wait();  // the decode results come from the previous kernel
    pdl_launch_dependents();
  } else {
    pdl_wait();  // decode results and state may come from the previous kernels in the stream
    pdl_launch_dependents();
    select_prefetch<kThreads>(a, blockIdx.x, dyn);
  }
  select_finish<kThreads>(a, blockIdx.x, dyn);
}

// Candidates of a step for block-wise or sliding-window decoding, one CTA per sequence: the
// masked positions of the window [w0, w0 + width), ascending. Block mode: w0 = start.
// Sliding mode: w0 = the first masked position at or after start (L if none).
constexpr int kCandThreads = 256;

__global__ void __launch_bounds__(kCandThreads) candidates_kernel(const uint8_t* __restrict__ mask, int L, int C_max,
                                                                  int mode, int start, int width,
                                                                  int32_t* __restrict__ cand_pos,
                                                                  int32_t* __restrict__ cand_count) {
  __shared__ int first;
  __shared__ int warp_n[kCandThreads / 32];
  __shared__ int carry;
  pdl_wait();  // the mask comes from the previous step's select kernel
  pdl_launch_dependents();
  const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint8_t* m = mask + static_cast<int64_t>(b) * L;
  int w0 = start;
  if (mode == EC_CAND_SLIDING) {
    if (tid == 0) first = L;
    __syncthreads();
    for (int p0 = start; p0 < L; p0 += kCandThreads) {
      const int p = p0 + tid;
      const bool hit = p < L && m[p] != 0;
      if (hit) atomicMin(&first, p);
      if (__syncthreads_or(hit)) break;
    }
    w0 = first;
  }
  if (tid == 0) carry = 0;
  __syncthreads();
  const int hi = min(L, w0 + width);
  int32_t* out = cand_pos + static_cast<int64_t>(b) * C_max;
  for (int p0 = w0; p0 < hi; p0 += kCandThreads) {  // compaction, ascending
    const int p = p0 + tid;
    const bool hit = p < hi && m[p] != 0;
    const unsigned bal = __ballot_sync(0xffffffffu, hit);
    if (lane == 0) warp_n[warp] = __popc(bal);
    __syncthreads();
    int before = carry, tot = 0;
    for (int w = 0; w < kCandThreads / 32; ++w) {
      if (w < warp) before += warp_n[w];
      tot += warp_n[w];
    }
    if (hit) out[before + __popc(bal & ((1u << lane) - 1u))] = p;
    __syncthreads();
    if (tid == 0) carry += tot;
    __syncthreads();
  }
  for (int i = carry + tid; i < C_max; i += kCandThreads) out[i] = -1;
  if (tid == 0) cand_count[b] = carry;
}

}  // namespace

cudaError_t launch_candidates(const ec_params& p, const uint8_t* mask, int32_t mode, int32_t start, int32_t width,
                              int32_t* cand_pos, int32_t* cand_count, cudaStream_t s) {
  return launch_pdl(candidates_kernel, dim3(p.B), dim3(kCandThreads), 0, s, mask, p.L, p.C_max, mode, start, width,
                    cand_pos, cand_count);
}

SelArgs make_sel_args(const ec_params& p, const ec_state& st, const int32_t* cand_pos, const int32_t* cand_count,
                      const int32_t* ids, const float* entropy, const float* log_conf, bool prefetch_early,
                      const ChunkPartial* partials, int32_t nchunks) {
  SelArgs a;
  a.prefetch_early = prefetch_early ? 1 : 0;
  a.partials = partials;
  a.nchunks = nchunks;
  a.L = p.L;
  a.scope_lo = scope_lo(p);
  a.scope_hi = scope_hi(p);
  a.C_max = p.C_max;
  a.k = p.k;
  a.n_dec = p.n_dec;
  a.tau = p.tau;
  a.log_thresh = p.conf_threshold > 0.f ? logf(p.conf_threshold) : -INFINITY;
  a.cand_pos = cand_pos;
  a.cand_count = cand_count;
  a.ids = ids;
  a.entropy = entropy;
  a.log_conf = log_conf;
  a.tokens = st.tokens;
  a.mask = st.mask;
  a.ring = st.ring;
  a.ring_head = st.ring_head;
  a.ring_count = st.ring_count;
  a.dec_pos = st.dec_pos;
  a.E = st.E;
  a.flag = st.flag;
  a.idx = st.idx;
  a.R = st.R;
  a.dev_err = st.dev_err;
  return a;
}

size_t select_smem_bytes(const ec_params& p) { return static_cast<size_t>(sel_layout(p.L, p.C_max, p.k).total); }

cudaError_t launch_select_recompute(const ec_params& p, const ec_state& st, const int32_t* cand_pos,
                                    const int32_t* cand_count, const int32_t* ids, const float* entropy,
                                    const float* log_conf, bool prefetch_early, const ChunkPartial* partials,
                                    int32_t nchunks, cudaStream_t s) {
  const size_t smem = select_smem_bytes(p);
  const cudaError_t e = ensure_dyn_smem(reinterpret_cast<const void*>(select_recompute_kernel), smem);
  if (e != cudaSuccess) return e;
  return launch_pdl(select_recompute_kernel, dim3(p.B), dim3(kThreads), smem, s,
                    make_sel_args(p, st, cand_pos, cand_count, ids, entropy, log_conf, prefetch_early, partials,
                                  nchunks));
}

}  // namespace ec
