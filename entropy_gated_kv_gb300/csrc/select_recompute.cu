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

}  // namespace

SelArgs make_sel_args(const ec_params& p, const ec_state& st, const int32_t* cand_pos, const int32_t* cand_count,
                      const int32_t* ids, const float* entropy, const float* log_conf, bool prefetch_early,
                      const ChunkPartial* partials, int32_t nchunks) {
  SelArgs a;
  a.prefetch_early = prefetch_early ? 1 : 0;
  a.partials = partials;
  a.nchunks = nchunks;
  a.L = p.L;
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
