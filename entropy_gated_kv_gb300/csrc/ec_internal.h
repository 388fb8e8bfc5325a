// ec_internal.h — launchers shared between the kernel files and the C-ABI layer.
#pragma once

#include <cstddef>
#include <utility>
#include <cstdint>
#include <cuda_runtime.h>

#include "entropycache.h"

namespace ec {

// ---- entropy_decode ---------------------------------------------------------------------
// Partial result of one piece of one row (entropy_decode.cu: 1024 bf16 or 512 fp32
// elements): raw max logit, its (lowest) index, and S = sum 2^d, T = sum d 2^d with
// d = (x - max) * log2(e).
struct ChunkPartial {
  float m;
  int32_t idx;
  float s;
  float t;
};

// Pieces per row: the partials per row that a publishing launch writes to the workspace.
int32_t entropy_num_chunks(int32_t V, int32_t dtype);
size_t entropy_workspace_bytes(int32_t n_rows, int32_t V, int32_t dtype);
// row_count (may be null): rows r with (r % rows_per_group) >= row_count[r / rows_per_group]
// are skipped (their outputs are left untouched). allow_cluster: few rows may take the
// one-cluster-per-row launch, which merges on chip (lowest latency on an idle GPU); without
// it, or with many rows, the split launch (or, from 32 MB, the pipelined one) publishes one
// partial per piece to the workspace and a merge kernel writes the rows. publish_only: the
// partials are left in the workspace for the next kernel to merge (ids / entropy / log_conf
// are not written). No workspace contents need to be initialised.
cudaError_t launch_entropy_decode(const void* logits, int64_t row_stride, int32_t n_rows, int32_t V,
                                  int32_t dtype, int32_t* ids, float* entropy, float* log_conf, void* ws,
                                  const int32_t* row_count, int32_t rows_per_group, bool allow_cluster,
                                  bool publish_only, cudaStream_t s);

// ---- output projection fused with the decode (lm_head_entropy.cu) -------------------------
size_t lm_head_workspace_bytes(int32_t n_rows);
int32_t lm_head_max_rows();
cudaError_t launch_lm_head_entropy(const void* hidden, const void* weight, int32_t n_rows, int32_t d_model, int32_t V,
                                   int32_t* ids, float* entropy, float* log_conf, void* ws, int32_t* dev_err,
                                   cudaStream_t s);

// ---- select_recompute ---------------------------------------------------------------------
struct SelArgs;
SelArgs make_sel_args(const ec_params& p, const ec_state& st, const int32_t* cand_pos, const int32_t* cand_count,
                      const int32_t* ids, const float* entropy, const float* log_conf, bool prefetch_early,
                      const ChunkPartial* partials, int32_t nchunks);
size_t select_smem_bytes(const ec_params& p);
// prefetch_early: stage the decode state before the grid dependency wait; partials (may be
// null): merge the decode kernel's per-chunk partials instead of reading ids / entropy /
// log_conf (see SelArgs).
cudaError_t launch_select_recompute(const ec_params& p, const ec_state& st, const int32_t* cand_pos,
                                    const int32_t* cand_count, const int32_t* ids, const float* entropy,
                                    const float* log_conf, bool prefetch_early, const ChunkPartial* partials,
                                    int32_t nchunks, cudaStream_t s);

// Candidate positions for block-wise / sliding-window decoding (EC_CAND_BLOCK / _SLIDING).
cudaError_t launch_candidates(const ec_params& p, const uint8_t* mask, int32_t mode, int32_t start, int32_t width,
                              int32_t* cand_pos, int32_t* cand_count, cudaStream_t s);

// ---- kv_scatter (+ optional query gather) -------------------------------------------------
cudaError_t launch_kv_scatter(const ec_params& p, void* k_cache, void* v_cache, const void* k_new,
                              const void* v_new, int32_t src_by_position, const int32_t* idx,
                              const int32_t* R, const void* q_src, void* q_dst, int32_t* dev_err,
                              cudaStream_t s);

// ---- partial attention --------------------------------------------------------------------
size_t attention_workspace_bytes(const ec_params& p);
// plan_early: R is final when the kernel starts (inside a step: written by the select kernel
// two launches earlier), so the work plan is made before the grid dependency wait.
cudaError_t launch_partial_attention(const ec_params& p, const void* q, const void* k_cache,
                                     const void* v_cache, const int32_t* R, float scale, void* out, void* ws,
                                     int32_t* dev_err, bool plan_early, cudaStream_t s, ec_status* status);

// ---- dense attention, two query tiles per CTA (attention_dense.cu): every position against
// every key ---------------------------------------------------------------------------------
cudaError_t launch_dense_attention_tiles(const ec_params& p, const void* q, const void* k_cache, const void* v_cache,
                                         float scale, void* out, int32_t* dev_err, cudaStream_t s,
                                         ec_status* status);

// ---- the partial forward of one layer (layer_forward.cu) ----------------------------------
size_t layer_forward_workspace_bytes(const ec_params& p, int32_t d_ff);
cudaError_t launch_layer_forward(const ec_params& p, const ec_layer& w, const int32_t* idx, const int32_t* R,
                                 const void* x_src, void* k_cache, void* v_cache, void* y, void* ws,
                                 int32_t* dev_err, cudaStream_t s, ec_status* status);
cudaError_t launch_rope_table(int32_t L, int32_t D, float theta, float* cs, float* sn, cudaStream_t s);

// ---- measurement aid (read_floor.cu) ---------------------------------------------------------
cudaError_t launch_read_floor(const void* buf, size_t bytes, uint32_t* sink, cudaStream_t s);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// The gate's scope [lo, hi): the whole sequence unless the caller set one (ec_params).
inline bool has_scope(const ec_params& p) { return p.scope_lo != 0 || p.scope_hi != 0; }
inline int32_t scope_lo(const ec_params& p) { return has_scope(p) ? p.scope_lo : 0; }
inline int32_t scope_hi(const ec_params& p) { return has_scope(p) ? p.scope_hi : p.L; }

// ---- per-device launch configuration (ec_api.cu) -------------------------------------------
// Kernel attributes and device properties apply per device, and the entry points may be
// called from several host threads and on several devices, so every cached value is kept
// per device behind a lock.
// SM count of the current device.
cudaError_t current_device_sms(int* sms);
// Raises `func`'s dynamic shared-memory limit on the current device to at least `bytes`.
cudaError_t ensure_dyn_smem(const void* func, size_t bytes);
// A value computed once per (current device, key) by `make` (which returns cudaSuccess and
// sets *value, or an error that is returned and not cached).
cudaError_t cached_per_device(int key, int* value, cudaError_t (*make)(int* value, void* ctx), void* ctx);

}  // namespace ec

namespace ec {

// Launches `kernel` with programmatic stream serialization, so it may begin while the
// previous kernel in the stream finishes; the kernel itself calls pdl_wait() before reading
// its inputs.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// launch_pdl with thread-block clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, int cluster_x,
                               cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(cluster_x);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace ec
