// select_recompute.cu — stages (b) and (c) of the EntropyCache step: commit the decoded
// tokens, gate on their maximum entropy, push them onto the decode history and build the
// recompute set.
//
// EntropyCache, gist.science zh summary §2.2 ("skip decision and selection"): if the
// maximum entropy E_{t+1} of the newly decoded tokens exceeds tau the next forward is a
// full one, otherwise it recomputes the current masked tokens plus the k most recently
// decoded tokens, taken from a decode history; §2.3: the history costs O(k) memory.
//
// One CTA per sequence. Candidates live in shared memory (C_max <= 1024); the commit set is
// found by ranking (O(C^2) comparisons, tiny for the block sizes in use). The recompute set
// is built as an L-bit bitmap in shared memory (mask bits OR the last-k history bits) and
// compacted in ascending order with a block-wide prefix sum over the words' popcounts.
#include <cmath>

#include "ec_common.cuh"
#include "ec_internal.h"

namespace ec {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCand = 1024;
constexpr int kPerThread = kMaxCand / kThreads;  // candidates handled per thread

struct SelShared {
  int pos[kMaxCand];
  float conf[kMaxCand];
  unsigned char valid[kMaxCand];
  unsigned char chosen[kMaxCand];
  int warp_tmp[kWarps];
  float warp_e[kWarps];
  int warp_nan[kWarps];
  int n_dec_eff;
  int head;
  int count;
  int full;
  int carry;
};

// Candidate j outranks candidate i: higher confidence; equal confidence, smaller position.
__device__ __forceinline__ bool outranks(float cj, int pj, float ci, int pi) {
  return cj > ci || (cj == ci && pj < pi);
}

__device__ __forceinline__ int block_sum_int(int v, SelShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if (lane == 0) sh.warp_tmp[warp] = v;
  __syncthreads();
  int tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) tot += sh.warp_tmp[w];
  __syncthreads();
  return tot;
}

// Exclusive prefix sum over the block; *total receives the block sum.
__device__ __forceinline__ int block_exclusive_scan(int v, int* total, SelShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) sh.warp_tmp[warp] = incl;
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    const int t = sh.warp_tmp[w];
    if (w < warp) before += t;
    tot += t;
  }
  __syncthreads();
  *total = tot;
  return before + incl - v;
}

__global__ void __launch_bounds__(kThreads) select_recompute_kernel(
    int32_t L, int32_t C_max, int32_t k, int32_t n_dec, float tau, const int32_t* __restrict__ cand_pos,
    const int32_t* __restrict__ cand_count, const int32_t* __restrict__ ids, const float* __restrict__ entropy,
    const float* __restrict__ log_conf, int32_t* __restrict__ tokens, uint8_t* __restrict__ mask,
    int32_t* __restrict__ ring, int32_t* __restrict__ ring_head, int32_t* __restrict__ ring_count,
    int32_t* __restrict__ dec_pos, float* __restrict__ E_out, uint8_t* __restrict__ flag_out,
    int32_t* __restrict__ idx, int32_t* __restrict__ R_out, int32_t* __restrict__ dev_err) {
  extern __shared__ uint32_t bitmap[];  // ceil(L / 32) words
  __shared__ SelShared sh;
  const int b = blockIdx.x;
  const int tid = threadIdx.x;
  const int64_t rowL = static_cast<int64_t>(b) * L;
  const int64_t rowC = static_cast<int64_t>(b) * C_max;

  if (tid == 0) {
    int h = ring_head[b], c = ring_count[b];
    if (h < 0 || h >= k || c < 0 || c > k) {
      report_error(dev_err, EC_DEVERR_BAD_R);
      h = min(max(h, 0), k - 1);
      c = min(max(c, 0), k);
    }
    sh.head = h;
    sh.count = c;
  }
  int count = __ldg(cand_count + b);
  if (count < 0 || count > C_max) {
    if (tid == 0) report_error(dev_err, EC_DEVERR_BAD_R);
    count = min(max(count, 0), C_max);
  }

  // 1. Load candidates; a position outside [0, L) or not masked is invalid.
#pragma unroll
  for (int q = 0; q < kPerThread; ++q) {
    const int i = tid + q * kThreads;
    if (i < count) {
      const int p = __ldg(cand_pos + rowC + i);
      const bool in_range = p >= 0 && p < L;
      const bool ok = in_range && mask[rowL + p] != 0;
      float c = __ldg(log_conf + rowC + i);
      if (isnan(c)) c = -INFINITY;  // NaN confidence ranks lowest
      sh.pos[i] = in_range ? p : -1;
      sh.conf[i] = c;
      sh.valid[i] = ok ? 1 : 0;
      if (!ok) report_error(dev_err, EC_DEVERR_BAD_CAND_POS);
    }
  }
  __syncthreads();
  // A position listed twice keeps only its first occurrence.
  unsigned char dup[kPerThread];
#pragma unroll
  for (int q = 0; q < kPerThread; ++q) {
    const int i = tid + q * kThreads;
    dup[q] = 0;
    if (i < count && sh.valid[i]) {
      for (int j = 0; j < i; ++j)
        if (sh.valid[j] && sh.pos[j] == sh.pos[i]) {
          dup[q] = 1;
          break;
        }
    }
  }
  __syncthreads();
  int nvalid_local = 0;
#pragma unroll
  for (int q = 0; q < kPerThread; ++q) {
    const int i = tid + q * kThreads;
    if (i < count) {
      if (dup[q]) {
        sh.valid[i] = 0;
        report_error(dev_err, EC_DEVERR_BAD_CAND_POS);
      }
      nvalid_local += sh.valid[i];
    }
  }
  __syncthreads();
  const int nvalid = block_sum_int(nvalid_local, sh);
  const int nD = min(n_dec, nvalid);

  // 2. D = the nD best-ranked valid candidates.
#pragma unroll
  for (int q = 0; q < kPerThread; ++q) {
    const int i = tid + q * kThreads;
    if (i < count) {
      int rank = 0;
      if (sh.valid[i]) {
        const float ci = sh.conf[i];
        const int pi = sh.pos[i];
        for (int j = 0; j < count; ++j)
          if (j != i && sh.valid[j] && outranks(sh.conf[j], sh.pos[j], ci, pi)) ++rank;
      }
      sh.chosen[i] = (sh.valid[i] && rank < nD) ? 1 : 0;
    }
  }
  __syncthreads();

  // 3. Commit, record dec_pos in ascending position order, push onto the ring, reduce E.
  const int head0 = sh.head;
  float emax = -INFINITY;
  int any_nan = 0;
#pragma unroll
  for (int q = 0; q < kPerThread; ++q) {
    const int i = tid + q * kThreads;
    if (i < count && sh.chosen[i]) {
      const int p = sh.pos[i];
      int ord = 0;
      for (int j = 0; j < count; ++j)
        if (sh.chosen[j] && sh.pos[j] < p) ++ord;
      tokens[rowL + p] = __ldg(ids + rowC + i);
      mask[rowL + p] = 0;
      dec_pos[static_cast<int64_t>(b) * n_dec + ord] = p;
      if (ord >= nD - k) ring[static_cast<int64_t>(b) * k + (head0 + ord) % k] = p;
      const float h = __ldg(entropy + rowC + i);
      if (isnan(h)) any_nan = 1;
      else emax = fmaxf(emax, h);
    }
  }
  for (int t = nD + tid; t < n_dec; t += kThreads) dec_pos[static_cast<int64_t>(b) * n_dec + t] = -1;
  {
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      emax = fmaxf(emax, __shfl_xor_sync(0xffffffffu, emax, off));
      any_nan |= __shfl_xor_sync(0xffffffffu, any_nan, off);
    }
    if (lane == 0) {
      sh.warp_e[warp] = emax;
      sh.warp_nan[warp] = any_nan;
    }
  }
  __syncthreads();
  if (tid == 0) {
    float e = -INFINITY;
    int nan_seen = 0;
    for (int w = 0; w < kWarps; ++w) {
      e = fmaxf(e, sh.warp_e[w]);
      nan_seen |= sh.warp_nan[w];
    }
    float E;
    int full;
    if (nD == 0) {
      E = 0.f;  // nothing decoded: E = 0
      full = (E > tau) ? 1 : 0;
    } else if (nan_seen) {
      E = NAN;
      full = 1;
    } else {
      E = e;
      full = (E > tau) ? 1 : 0;
    }
    E_out[b] = E;
    flag_out[b] = static_cast<uint8_t>(full);
    const int head1 = (head0 + nD) % k;
    const int count1 = min(sh.count + nD, k);
    ring_head[b] = head1;
    ring_count[b] = count1;
    sh.head = head1;
    sh.count = count1;
    sh.full = full;
    sh.carry = 0;
  }
  __syncthreads();  // commits, ring writes and the new head/count are visible to the block

  // 4. Recompute set.
  if (sh.full) {
    for (int r = tid; r < L; r += kThreads) idx[rowL + r] = r;
    if (tid == 0) R_out[b] = L;
    return;
  }
  const int nwords = (L + 31) >> 5;
  {
    const int lane = tid & 31, warp = tid >> 5;
    for (int p0 = warp << 5; p0 < L; p0 += kThreads) {  // one warp per 32 positions
      const int p = p0 + lane;
      const bool m = p < L && mask[rowL + p] != 0;
      const uint32_t bits = __ballot_sync(0xffffffffu, m);
      if (lane == 0) bitmap[p0 >> 5] = bits;
    }
  }
  __syncthreads();
  const int head1 = sh.head, count1 = sh.count;
  for (int t = tid; t < count1; t += kThreads) {
    const int p = ring[static_cast<int64_t>(b) * k + ((head1 - 1 - t) % k + k) % k];
    if (p >= 0 && p < L) atomicOr(&bitmap[p >> 5], 1u << (p & 31));
    else report_error(dev_err, EC_DEVERR_BAD_IDX);
  }
  __syncthreads();
  for (int base = 0; base < nwords; base += kThreads) {
    const int w = base + tid;
    const uint32_t bits = (w < nwords) ? bitmap[w] : 0u;
    int total = 0;
    const int off = block_exclusive_scan(__popc(bits), &total, sh);
    int o = sh.carry + off;
    uint32_t rest = bits;
    while (rest) {
      const int bit = __ffs(rest) - 1;
      idx[rowL + o++] = (w << 5) + bit;
      rest &= rest - 1;
    }
    __syncthreads();
    if (tid == 0) sh.carry += total;
    __syncthreads();
  }
  if (tid == 0) R_out[b] = sh.carry;
}

}  // namespace

cudaError_t launch_select_recompute(const ec_params& p, const ec_state& st, const int32_t* cand_pos,
                                    const int32_t* cand_count, const int32_t* ids, const float* entropy,
                                    const float* log_conf, cudaStream_t s) {
  const size_t smem = static_cast<size_t>((p.L + 31) / 32) * sizeof(uint32_t);
  static size_t configured = 0;
  if (smem > 48 * 1024 && smem > configured) {
    cudaError_t e = cudaFuncSetAttribute(select_recompute_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    configured = smem;
  }
  select_recompute_kernel<<<p.B, kThreads, smem, s>>>(
      p.L, p.C_max, p.k, p.n_dec, p.tau, cand_pos, cand_count, ids, entropy, log_conf, st.tokens, st.mask, st.ring,
      st.ring_head, st.ring_count, st.dec_pos, st.E, st.flag, st.idx, st.R, st.dev_err);
  return cudaGetLastError();
}

}  // namespace ec
