// entropy_decode_noalloc.cu — stage (a) for callers that cannot allocate device memory.
//
// ec_entropy_decode keeps the per-chunk partial results of its split-vocabulary reduction in
// a workspace the caller allocates. Some callers cannot provide one: a plugin or custom-op
// interface of a serving runtime hands the op its input and output tensors but no allocator,
// and latency-critical code may not call cudaMalloc at all because it synchronises the whole
// device. ec_entropy_decode_noalloc runs the same kernel with its scratch in a fixed array
// that the library itself places in device memory, so such a caller passes only inputs and
// outputs.
//
// The array (EC_NOALLOC_SCRATCH_BYTES) exists on every GPU that loads the library and stays
// there until the process exits. Its device address is looked up once per device, on the
// first call made with that device current. Every call shares it and it keeps the last
// call's contents; no call needs it to start in any particular state (every partial result a
// call reads back is one it wrote first), and calls that overlap on the GPU race with each
// other.
#include <mutex>

#include "ec_internal.h"

namespace {

constexpr size_t kScratchBytes = EC_NOALLOC_SCRATCH_BYTES;

// The scratch: one partial result per (row, vocabulary piece).
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device; set up once per device. In host code
// the name g_scratch is only a host-side stand-in, so the address must come from here.
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" ec_status ec_entropy_decode_noalloc(const void* logits, int64_t row_stride, int32_t n_rows, int32_t V,
                                               int32_t dtype, int32_t* ids, float* entropy, float* log_conf,
                                               ec_stream_t stream) {
  if (dtype != EC_F32 && dtype != EC_BF16) return EC_ERR_INVALID_ARG;
  if (V < 1 || V > (1 << 30) || n_rows < 0 || row_stride < V) return EC_ERR_INVALID_ARG;
  if (n_rows == 0) return EC_OK;
  const int64_t esize = dtype == EC_F32 ? 4 : 2;
  if ((row_stride * esize) % 16 != 0) return EC_ERR_INVALID_ARG;
  if (!logits || !ids || !entropy || !log_conf || !aligned16(logits)) return EC_ERR_INVALID_ARG;
  const int32_t nch = ec::entropy_num_chunks(V, dtype);
  if (static_cast<int64_t>(n_rows) * nch > INT32_MAX) return EC_ERR_UNSUPPORTED;
  if (ec::entropy_workspace_bytes(n_rows, V, dtype) > kScratchBytes) return EC_ERR_UNSUPPORTED;  // too large

  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return EC_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = ec::launch_entropy_decode(logits, row_stride, n_rows, V, dtype, ids, entropy, log_conf,
                                                  scratch, nullptr, 1, true, false, s);
  return e == cudaSuccess ? EC_OK : EC_ERR_CUDA;
}
