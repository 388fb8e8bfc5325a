// ec_api.cu — the C ABI of the EntropyCache step library: host-side validation, workspace
// layout and the composition of the stages into one denoising step.
//
// Every entry point validates its arguments on the host before launching anything, returns
// an ec_status and never throws. The library allocates no memory.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "ec_common.cuh"
#include "ec_internal.h"
#include "entropycache.h"

namespace ec {

static std::mutex g_cfg_mutex;
static std::map<std::pair<int, const void*>, size_t> g_dyn_smem;  // (device, kernel) -> configured bytes
static std::map<std::pair<int, int>, int> g_cached;               // (device, key) -> value

cudaError_t current_device_sms(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  return cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
}

cudaError_t ensure_dyn_smem(const void* func, size_t bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_cfg_mutex);
  size_t& have = g_dyn_smem[{dev, func}];
  if (bytes <= have) return cudaSuccess;
  if (bytes > 48 * 1024) {
    e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
    if (e != cudaSuccess) return e;
  }
  have = bytes;
  return cudaSuccess;
}

cudaError_t cached_per_device(int key, int* value, cudaError_t (*make)(int* value, void* ctx), void* ctx) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_cfg_mutex);
  auto it = g_cached.find({dev, key});
  if (it != g_cached.end()) {
    *value = it->second;
    return cudaSuccess;
  }
  int v = 0;
  e = make(&v, ctx);
  if (e != cudaSuccess) return e;
  g_cached[{dev, key}] = v;
  *value = v;
  return cudaSuccess;
}

}  // namespace ec

using namespace ec;

namespace {

constexpr int32_t kMaxB = 4096;
constexpr int32_t kMaxL = 1 << 20;
constexpr int32_t kMaxV = 1 << 30;
constexpr int32_t kMaxCmax = 1024;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The byte ranges [a, a + na) and [b, b + nb) share a byte (addresses compared, never read).
bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}
size_t q_bytes(const ec_params& p) { return static_cast<size_t>(p.B) * p.L * p.Hq * p.D * 2; }
size_t kv_bytes(const ec_params& p) { return static_cast<size_t>(p.B) * p.L * p.Hkv * p.D * 2; }

// The attention writes out ([B, L, Hq, D]) while it reads q, k_cache and v_cache.
bool attention_io_overlap(const ec_params& p, const void* q, const void* k, const void* v, const void* out) {
  const size_t nq = q_bytes(p), nkv = kv_bytes(p);
  return overlaps(out, nq, q, nq) || overlaps(out, nq, k, nkv) || overlaps(out, nq, v, nkv);
}

// The scatter writes both caches while it reads the fresh rows ([B, L, Hkv, D] each).
bool scatter_io_overlap(const ec_params& p, const void* kc, const void* vc, const void* kn, const void* vn) {
  const size_t n = kv_bytes(p);
  return overlaps(kc, n, vc, n) || overlaps(kc, n, kn, n) || overlaps(kc, n, vn, n) || overlaps(vc, n, kn, n) ||
         overlaps(vc, n, vn, n);
}

ec_status cuda_status(cudaError_t e) { return e == cudaSuccess ? EC_OK : EC_ERR_CUDA; }

// Shape checks common to the stages that need them. `what` selects the groups checked.
enum : int { kCheckDecode = 1, kCheckSelect = 2, kCheckAttn = 4 };

ec_status check_params(const ec_params* p, int what) {
  if (p == nullptr) return EC_ERR_INVALID_ARG;
  if (p->B < 1 || p->B > kMaxB || p->L < 1 || p->L > kMaxL) return EC_ERR_INVALID_ARG;
  if (has_scope(*p) && !(p->scope_lo >= 0 && p->scope_lo < p->scope_hi && p->scope_hi <= p->L))
    return EC_ERR_INVALID_ARG;
  if (what & kCheckDecode) {
    if (p->V < 1 || p->V > kMaxV) return EC_ERR_INVALID_ARG;
    if (p->logits_dtype != EC_F32 && p->logits_dtype != EC_BF16) return EC_ERR_INVALID_ARG;
  }
  if (what & kCheckSelect) {
    if (p->C_max < 1 || p->C_max > std::min(p->L, kMaxCmax)) return EC_ERR_INVALID_ARG;
    if (p->k < 1 || p->k > p->L) return EC_ERR_INVALID_ARG;
    if (p->n_dec < 1 || p->n_dec > p->C_max) return EC_ERR_INVALID_ARG;
    if (p->tau != p->tau) return EC_ERR_INVALID_ARG;  // NaN threshold
    if (!(p->conf_threshold <= 1.f)) return EC_ERR_INVALID_ARG;  // NaN, or above any probability
  }
  if (what & kCheckAttn) {
    if (p->Hq < 1 || p->Hkv < 1 || p->Hq % p->Hkv != 0) return EC_ERR_INVALID_ARG;
    if (p->Hq / p->Hkv > 128) return EC_ERR_UNSUPPORTED;
    if (p->D != 64 && p->D != 128) return EC_ERR_UNSUPPORTED;
    const int64_t g = p->Hq / p->Hkv;
    const int64_t nr = 128 / g;
    const int64_t tiles = static_cast<int64_t>(p->B) * p->Hkv * ((p->L + nr - 1) / nr);
    if (tiles > (1ll << 30)) return EC_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(p->Hq) * p->D * p->L * p->B > (1ll << 40)) return EC_ERR_UNSUPPORTED;
  }
  return EC_OK;
}

ec_status check_state(const ec_state* st) {
  if (st == nullptr) return EC_ERR_INVALID_ARG;
  if (!st->tokens || !st->mask || !st->ring || !st->ring_head || !st->ring_count || !st->dec_pos || !st->E ||
      !st->flag || !st->idx || !st->R)
    return EC_ERR_INVALID_ARG;
  if (!aligned16(st->mask)) return EC_ERR_INVALID_ARG;  // the mask row is read with 16-byte loads
  return EC_OK;
}

// ---- ec_step workspace layout --------------------------------------------------------
struct StepLayout {
  size_t k1, ids, ent, conf, qbuf, attn, total;
};

StepLayout step_layout(const ec_params& p) {
  StepLayout s{};
  const size_t rows = static_cast<size_t>(p.B) * p.C_max;
  size_t off = 0;
  s.k1 = off;
  off += align_up(entropy_workspace_bytes(static_cast<int32_t>(rows), p.V, p.logits_dtype), 256);
  s.ids = off;
  off += align_up(rows * 4, 256);
  s.ent = off;
  off += align_up(rows * 4, 256);
  s.conf = off;
  off += align_up(rows * 4, 256);
  s.qbuf = off;
  off += align_up(static_cast<size_t>(p.B) * p.L * p.Hq * p.D * 2, 256);
  s.attn = off;
  off += align_up(attention_workspace_bytes(p), 256);
  s.total = off;
  return s;
}

// One CTA: thread 0 waits for a phase of a barrier on which nothing ever arrives.
__global__ void selftest_wait_kernel(int32_t* dev_err, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort;
  if (threadIdx.x == 0) {
    abort = 0;
    ec::mbar_init(&bar, 1);
    ec::fence_mbar_init();
    ec::mbar_wait_bounded(&bar, 0, &abort, dev_err, limit_ns);
  }
}

}  // namespace

extern "C" {

const char* ec_status_string(ec_status st) {
  switch (st) {
    case EC_OK: return "EC_OK";
    case EC_ERR_INVALID_ARG: return "EC_ERR_INVALID_ARG";
    case EC_ERR_UNSUPPORTED: return "EC_ERR_UNSUPPORTED";
    case EC_ERR_CUDA: return "EC_ERR_CUDA";
    case EC_ERR_DEVICE_CHECK: return "EC_ERR_DEVICE_CHECK";
    case EC_ERR_TIMEOUT: return "EC_ERR_TIMEOUT";
    default: return "EC_ERR_UNKNOWN";
  }
}

int32_t ec_version(void) { return 100; }

ec_status ec_read_device_error(const int32_t* dev_err, int32_t* host_word, ec_stream_t stream) {
  if (dev_err == nullptr) return EC_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int32_t w = 0;
  cudaError_t e = cudaMemcpyAsync(&w, dev_err, sizeof(w), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return EC_ERR_CUDA;
  if (host_word != nullptr) *host_word = w;
  if (w == 0) return EC_OK;
  return (w & EC_DEVERR_TIMEOUT) ? EC_ERR_TIMEOUT : EC_ERR_DEVICE_CHECK;
}

ec_status ec_selftest_bounded_wait(int32_t* dev_err, uint64_t limit_ns, ec_stream_t stream) {
  if (dev_err == nullptr || limit_ns < 1 || limit_ns > 10000000000ull) return EC_ERR_INVALID_ARG;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_err, limit_ns);
  return cuda_status(cudaGetLastError());
}

// ---- (a) ----------------------------------------------------------------------------------
size_t ec_entropy_decode_workspace_size(int32_t n_rows, int32_t V, int32_t dtype) {
  if (n_rows < 0 || V < 1 || V > kMaxV || (dtype != EC_F32 && dtype != EC_BF16)) return 0;
  return entropy_workspace_bytes(n_rows, V, dtype);
}

ec_status ec_entropy_decode(const void* logits, int64_t row_stride, int32_t n_rows, int32_t V, int32_t dtype,
                            int32_t* ids, float* entropy, float* log_conf, void* ws, size_t ws_bytes,
                            ec_stream_t stream) {
  if (dtype != EC_F32 && dtype != EC_BF16) return EC_ERR_INVALID_ARG;
  if (V < 1 || V > kMaxV || n_rows < 0 || row_stride < V) return EC_ERR_INVALID_ARG;
  if (n_rows == 0) return EC_OK;
  const int64_t esize = dtype == EC_F32 ? 4 : 2;
  if ((row_stride * esize) % 16 != 0) return EC_ERR_INVALID_ARG;
  if (!logits || !ids || !entropy || !log_conf || !aligned16(logits)) return EC_ERR_INVALID_ARG;
  if (static_cast<int64_t>(n_rows) * entropy_num_chunks(V, dtype) > INT32_MAX) return EC_ERR_UNSUPPORTED;
  const size_t need = entropy_workspace_bytes(n_rows, V, dtype);
  if (ws == nullptr || ws_bytes < need || !aligned16(ws)) return EC_ERR_INVALID_ARG;
  return cuda_status(launch_entropy_decode(logits, row_stride, n_rows, V, dtype, ids, entropy, log_conf, ws,
                                           nullptr, 1, true, false, static_cast<cudaStream_t>(stream)));
}

// ---- (a) from the hidden states ----------------------------------------------------------------
size_t ec_lm_head_entropy_workspace_size(int32_t n_rows) {
  if (n_rows < 1 || n_rows > lm_head_max_rows()) return 0;
  return lm_head_workspace_bytes(n_rows);
}

ec_status ec_lm_head_entropy(const void* hidden, const void* weight, int32_t n_rows, int32_t d_model, int32_t V,
                             int32_t* ids, float* entropy, float* log_conf, void* ws, size_t ws_bytes,
                             ec_stream_t stream) {
  if (n_rows < 1 || n_rows > lm_head_max_rows()) return EC_ERR_INVALID_ARG;
  if (d_model < 64 || d_model > 65536 || d_model % 64 != 0 || V < 1 || V > kMaxV) return EC_ERR_INVALID_ARG;
  if (!hidden || !weight || !ids || !entropy || !log_conf || !ws) return EC_ERR_INVALID_ARG;
  if (!aligned16(hidden) || !aligned16(weight) || !aligned16(ws)) return EC_ERR_INVALID_ARG;
  if (ws_bytes < lm_head_workspace_bytes(n_rows)) return EC_ERR_INVALID_ARG;
  return cuda_status(launch_lm_head_entropy(hidden, weight, n_rows, d_model, V, ids, entropy, log_conf, ws, nullptr,
                                            static_cast<cudaStream_t>(stream)));
}

// ---- (b)+(c) --------------------------------------------------------------------------------
ec_status ec_select_recompute(const ec_params* p, const ec_state* st, const int32_t* cand_pos,
                              const int32_t* cand_count, const int32_t* ids, const float* entropy,
                              const float* log_conf, ec_stream_t stream) {
  ec_status r = check_params(p, kCheckSelect);
  if (r != EC_OK) return r;
  if ((r = check_state(st)) != EC_OK) return r;
  if (!cand_pos || !cand_count || !ids || !entropy || !log_conf) return EC_ERR_INVALID_ARG;
  return cuda_status(launch_select_recompute(*p, *st, cand_pos, cand_count, ids, entropy, log_conf, false, nullptr,
                                             0, static_cast<cudaStream_t>(stream)));
}

// ---- candidates for block-wise / sliding-window decoding -----------------------------------------
ec_status ec_candidates(const ec_params* p, const ec_state* st, int32_t mode, int32_t start, int32_t width,
                        int32_t* cand_pos, int32_t* cand_count, ec_stream_t stream) {
  ec_status r = check_params(p, kCheckSelect);
  if (r != EC_OK) return r;
  if (st == nullptr || st->mask == nullptr || !cand_pos || !cand_count) return EC_ERR_INVALID_ARG;
  if (mode != EC_CAND_BLOCK && mode != EC_CAND_SLIDING) return EC_ERR_INVALID_ARG;
  if (start < 0 || start >= p->L || width < 1 || width > p->C_max) return EC_ERR_INVALID_ARG;
  return cuda_status(launch_candidates(*p, st->mask, mode, start, width, cand_pos, cand_count,
                                       static_cast<cudaStream_t>(stream)));
}

// ---- (c) scatter ------------------------------------------------------------------------------
ec_status ec_kv_scatter(const ec_params* p, void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                        int32_t src_by_position, const int32_t* idx, const int32_t* R, int32_t* dev_err,
                        ec_stream_t stream) {
  if (p == nullptr) return EC_ERR_INVALID_ARG;
  if (p->B < 1 || p->B > kMaxB || p->L < 1 || p->L > kMaxL || p->Hkv < 1) return EC_ERR_INVALID_ARG;
  if (p->D != 64 && p->D != 128) return EC_ERR_UNSUPPORTED;
  if (src_by_position != 0 && src_by_position != 1) return EC_ERR_INVALID_ARG;
  if (!k_cache || !v_cache || !k_new || !v_new || !idx || !R) return EC_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new))
    return EC_ERR_INVALID_ARG;
  if (scatter_io_overlap(*p, k_cache, v_cache, k_new, v_new)) return EC_ERR_INVALID_ARG;
  return cuda_status(launch_kv_scatter(*p, k_cache, v_cache, k_new, v_new, src_by_position, idx, R, nullptr,
                                       nullptr, dev_err, static_cast<cudaStream_t>(stream)));
}

// ---- (d) ----------------------------------------------------------------------------------------
size_t ec_partial_attention_workspace_size(const ec_params* p) {
  if (check_params(p, kCheckAttn) != EC_OK) return 0;
  return attention_workspace_bytes(*p);
}

ec_status ec_dense_attention(const ec_params* p, const void* q, const void* k_cache, const void* v_cache,
                             float scale, void* out, int32_t* dev_err, ec_stream_t stream) {
  ec_status r = check_params(p, kCheckAttn);
  if (r != EC_OK) return r;
  if (!q || !k_cache || !v_cache || !out) return EC_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out)) return EC_ERR_INVALID_ARG;
  if (!(scale == scale)) return EC_ERR_INVALID_ARG;
  if (p->D != 128) return EC_ERR_UNSUPPORTED;
  if (attention_io_overlap(*p, q, k_cache, v_cache, out)) return EC_ERR_INVALID_ARG;
  ec_status st = EC_OK;
  launch_dense_attention_tiles(*p, q, k_cache, v_cache, scale, out, dev_err, static_cast<cudaStream_t>(stream), &st);
  return st;
}

ec_status ec_partial_attention(const ec_params* p, const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* R, float scale, void* out, void* ws, size_t ws_bytes,
                               int32_t* dev_err, ec_stream_t stream) {
  ec_status r = check_params(p, kCheckAttn);
  if (r != EC_OK) return r;
  if (!q || !k_cache || !v_cache || !R || !out || !ws) return EC_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) || !aligned16(ws))
    return EC_ERR_INVALID_ARG;
  if (ws_bytes < attention_workspace_bytes(*p)) return EC_ERR_INVALID_ARG;
  if (!(scale == scale)) return EC_ERR_INVALID_ARG;
  if (attention_io_overlap(*p, q, k_cache, v_cache, out)) return EC_ERR_INVALID_ARG;
  ec_status st = EC_OK;
  launch_partial_attention(*p, q, k_cache, v_cache, R, scale, out, ws, dev_err, false, static_cast<cudaStream_t>(stream),
                           &st);
  return st;
}

// ---- the partial forward of one layer --------------------------------------------------------------
namespace {
ec_status check_layer(const ec_params* p, const ec_layer* w) {
  ec_status r = check_params(p, kCheckAttn);
  if (r != EC_OK) return r;
  if (w == nullptr) return EC_ERR_INVALID_ARG;
  const int64_t d = static_cast<int64_t>(p->Hq) * p->D, kvf = static_cast<int64_t>(p->Hkv) * p->D;
  if (d % 128 != 0 || d > 8192 || kvf % 128 != 0) return EC_ERR_UNSUPPORTED;
  if (w->d_ff < 64 || w->d_ff % 64 != 0 || w->d_ff > 65536) return EC_ERR_INVALID_ARG;
  if (!(w->eps > 0.f)) return EC_ERR_INVALID_ARG;
  const void* ptrs[] = {w->wq, w->wk, w->wv, w->wo, w->wg, w->wu, w->wd, w->gamma1, w->gamma2, w->rope_cos, w->rope_sin};
  for (const void* q : ptrs)
    if (q == nullptr || !aligned16(q)) return EC_ERR_INVALID_ARG;
  return EC_OK;
}
}  // namespace

size_t ec_layer_forward_workspace_size(const ec_params* p, int32_t d_ff) {
  if (check_params(p, kCheckAttn) != EC_OK || d_ff < 64 || d_ff % 64 != 0) return 0;
  return layer_forward_workspace_bytes(*p, d_ff);
}

ec_status ec_layer_forward(const ec_params* p, const ec_layer* w, const int32_t* idx, const int32_t* R,
                           const void* x_src, void* k_cache, void* v_cache, void* y, void* ws, size_t ws_bytes,
                           int32_t* dev_err, ec_stream_t stream) {
  ec_status r = check_layer(p, w);
  if (r != EC_OK) return r;
  if (!idx || !R || !x_src || !k_cache || !v_cache || !y || !ws) return EC_ERR_INVALID_ARG;
  if (!aligned16(x_src) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(y) || !aligned16(ws))
    return EC_ERR_INVALID_ARG;
  if (ws_bytes < layer_forward_workspace_bytes(*p, w->d_ff)) return EC_ERR_INVALID_ARG;
  ec_status st = EC_OK;
  launch_layer_forward(*p, *w, idx, R, x_src, k_cache, v_cache, y, ws, dev_err, static_cast<cudaStream_t>(stream), &st);
  return st;
}

ec_status ec_rope_table(int32_t L, int32_t D, float theta, float* rope_cos, float* rope_sin, ec_stream_t stream) {
  if (L < 1 || L > kMaxL || D < 2 || D > 256 || D % 2 != 0 || !(theta > 0.f)) return EC_ERR_INVALID_ARG;
  if (!rope_cos || !rope_sin) return EC_ERR_INVALID_ARG;
  return cuda_status(launch_rope_table(L, D, theta, rope_cos, rope_sin, static_cast<cudaStream_t>(stream)));
}

// ---- measurement aid -----------------------------------------------------------------------------
ec_status ec_read_floor(const void* buf, size_t bytes, uint32_t* sink, ec_stream_t stream) {
  if (buf == nullptr || sink == nullptr || !aligned16(buf) || bytes % 16 != 0 || bytes > (size_t(1) << 40))
    return EC_ERR_INVALID_ARG;
  return cuda_status(launch_read_floor(buf, bytes, sink, static_cast<cudaStream_t>(stream)));
}

// ---- whole step ---------------------------------------------------------------------------------
size_t ec_step_workspace_size(const ec_params* p) {
  if (check_params(p, kCheckDecode | kCheckSelect | kCheckAttn) != EC_OK) return 0;
  return step_layout(*p).total;
}

ec_status ec_step(const ec_params* p, const ec_state* st, const void* logits, const int32_t* cand_pos,
                  const int32_t* cand_count, int32_t n_layers, void* const* k_cache, void* const* v_cache,
                  const void* const* k_src, const void* const* v_src, const void* const* q_src, void* const* out,
                  float scale, void* ws, size_t ws_bytes, ec_stream_t stream) {
  ec_status r = check_params(p, kCheckDecode | kCheckSelect | kCheckAttn);
  if (r != EC_OK) return r;
  if ((r = check_state(st)) != EC_OK) return r;
  const int64_t esize = p->logits_dtype == EC_F32 ? 4 : 2;
  if ((static_cast<int64_t>(p->V) * esize) % 16 != 0) return EC_ERR_INVALID_ARG;
  if (!logits || !aligned16(logits) || !cand_pos || !cand_count || !ws || !aligned16(ws)) return EC_ERR_INVALID_ARG;
  if (n_layers < 0 || (n_layers > 0 && (!k_cache || !v_cache || !k_src || !v_src || !q_src || !out)))
    return EC_ERR_INVALID_ARG;
  if (!(scale == scale)) return EC_ERR_INVALID_ARG;
  for (int32_t l = 0; l < n_layers; ++l) {
    if (!k_cache[l] || !v_cache[l] || !k_src[l] || !v_src[l] || !q_src[l] || !out[l]) return EC_ERR_INVALID_ARG;
    if (!aligned16(k_cache[l]) || !aligned16(v_cache[l]) || !aligned16(k_src[l]) || !aligned16(v_src[l]) ||
        !aligned16(q_src[l]) || !aligned16(out[l]))
      return EC_ERR_INVALID_ARG;
    if (scatter_io_overlap(*p, k_cache[l], v_cache[l], k_src[l], v_src[l]) ||
        attention_io_overlap(*p, q_src[l], k_cache[l], v_cache[l], out[l]))
      return EC_ERR_INVALID_ARG;
  }
  const StepLayout lay = step_layout(*p);
  if (ws_bytes < lay.total) return EC_ERR_INVALID_ARG;
  char* w = static_cast<char*>(ws);
  auto* ids = reinterpret_cast<int32_t*>(w + lay.ids);
  auto* ent = reinterpret_cast<float*>(w + lay.ent);
  auto* conf = reinterpret_cast<float*>(w + lay.conf);
  cudaStream_t s = static_cast<cudaStream_t>(stream);

  // stages (a)-(c): decode + entropy of the candidate rows, then the select stage
  cudaError_t e = launch_entropy_decode(logits, p->V, p->B * p->C_max, p->V, p->logits_dtype, ids, ent, conf,
                                        w + lay.k1, cand_count, p->C_max, false, true, s);
  // the decode kernel waits for every earlier kernel before it releases this one, so the select
  // kernel may stage the state before its own wait
  if (e == cudaSuccess)
    e = launch_select_recompute(*p, *st, cand_pos, cand_count, ids, ent, conf, true,
                                reinterpret_cast<const ChunkPartial*>(w + lay.k1), entropy_num_chunks(p->V, p->logits_dtype),
                                s);
  if (e != cudaSuccess) return EC_ERR_CUDA;
  // Entropies are non-negative (an empty decode set counts 0, a NaN counts as full), so with
  // tau < 0 the gate fires on every step. Without a scope every step then recomputes every
  // position in order (idx is the identity), and the attention is the dense one for every
  // sequence: the two-tile kernel reads the position-indexed queries where they are, and the
  // scatter kernel refreshes the cache only (no query gather).
  const bool always_full = p->tau < 0.f && !has_scope(*p) && p->D == 128;
  for (int32_t l = 0; l < n_layers; ++l) {
    e = launch_kv_scatter(*p, k_cache[l], v_cache[l], k_src[l], v_src[l], 1, st->idx, st->R,
                          always_full ? nullptr : q_src[l], always_full ? nullptr : w + lay.qbuf, st->dev_err, s);
    if (e != cudaSuccess) return EC_ERR_CUDA;
    ec_status as = EC_OK;
    if (always_full)
      launch_dense_attention_tiles(*p, q_src[l], k_cache[l], v_cache[l], scale, out[l], st->dev_err, s, &as);
    else
      launch_partial_attention(*p, w + lay.qbuf, k_cache[l], v_cache[l], st->R, scale, out[l], w + lay.attn,
                               st->dev_err, true, s, &as);
    if (as != EC_OK) return as;
  }
  return EC_OK;
}

}  // extern "C"
