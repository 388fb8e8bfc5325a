// select_recompute.cu — stages (b) and (c) of the EntropyCache step: commit the decoded
// tokens, gate on their maximum entropy, push them onto the decode history and build the
// recompute set.
//
// EntropyCache, gist.science zh summary §2.2 ("skip decision and selection"): if the
// maximum entropy E_{t+1} of the newly decoded tokens exceeds tau the next forward is a
// full one, otherwise it recomputes the current masked tokens plus the k most recently
// decoded tokens, taken from a decode history; §2.3: the history costs O(k) memory.
//
// One CTA per sequence. The mask row becomes an L-bit bitmap in shared memory, the
// candidates (C_max <= 1024) and the history (k <= 4096) are staged there too, all in one read
// phase. The commit set is found by ranking (O(C^2) comparisons, tiny for the block sizes in
// use); the committed bits are cleared, the last-k history bits set, and the bitmap is
// compacted in ascending order with a block-wide prefix sum over the words' popcounts.
#include <climits>
#include <cmath>

#include "ec_common.cuh"
#include "ec_internal.h"

namespace ec {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCand = 1024;
constexpr int kPerThread = kMaxCand / kThreads;  // candidates handled per thread
constexpr int kMaxRingSmem = 4096;               // histories up to this length live in smem

struct SelShared {
  int pos[kMaxCand];
  float conf[kMaxCand];
  float ent[kMaxCand];
  int id[kMaxCand];
  unsigned char valid[kMaxCand];
  unsigned char chosen[kMaxCand];
  int ring[kMaxRingSmem];
  int warp_tmp[kWarps];
  float warp_e[kWarps];
  int warp_nan[kWarps];
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

__device__ __forceinline__ bool bit_set(const uint32_t* bm, int p) { return (bm[p >> 5] >> (p & 31)) & 1u; }

// 32 mask bytes -> one bitmap word (bit t set when byte t is non-zero).
__device__ __forceinline__ uint32_t bytes_to_bits(uint4 lo, uint4 hi) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint32_t bits = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q)
#pragma unroll
    for (int e = 0; e < 4; ++e) bits |= (((w[q] >> (8 * e)) & 0xFFu) != 0u ? 1u : 0u) << (4 * q + e);
  return bits;
}

// Warp-wide: the set bits of words [0, nwords) written to idx in ascending order; returns
// the count (nwords <= 32). Lane w computes the prefix count of word w; then, word by word,
// lane j writes bit j — independent iterations, no lane loops over its own bits.
__device__ __forceinline__ int warp_compact(const uint32_t* bitmap, int nwords, int32_t* idx_row, int lane) {
  const uint32_t mine = lane < nwords ? bitmap[lane] : 0u;
  const int c = __popc(mine);
  int incl = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  const int excl = incl - c;
  const uint32_t below = (1u << lane) - 1u;
#pragma unroll 8
  for (int w = 0; w < nwords; ++w) {
    const uint32_t word = __shfl_sync(0xffffffffu, mine, w);
    const int base = __shfl_sync(0xffffffffu, excl, w);
    if ((word >> lane) & 1u) idx_row[base + __popc(word & below)] = (w << 5) + lane;
  }
  return __shfl_sync(0xffffffffu, incl, 31);
}

// Warp argmax over (confidence, -position): the best-ranked lane among `live`, or -1.
__device__ __forceinline__ int warp_best(float c, int p, bool live, int lane) {
  float bc = live ? c : -INFINITY;
  int bp = live ? p : INT_MAX;
  int bl = live ? lane : 32;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float oc = __shfl_xor_sync(0xffffffffu, bc, off);
    const int op = __shfl_xor_sync(0xffffffffu, bp, off);
    const int ol = __shfl_xor_sync(0xffffffffu, bl, off);
    if (ol < 32 && (bl == 32 || outranks(oc, op, bc, bp))) {
      bc = oc;
      bp = op;
      bl = ol;
    }
  }
  return bl < 32 ? bl : -1;
}

// One CTA per sequence. One read phase stages the mask as an L-bit bitmap (16-byte loads),
// the candidates and the history in shared memory. With at most 32 candidates a single warp
// then ranks, commits, gates, pushes the history and edits the bitmap, and for L <= 1024 also
// compacts it: two block barriers in all. Larger candidate lists and sequences use block-wide
// loops.
__global__ void __launch_bounds__(kThreads) select_recompute_kernel(
    int32_t L, int32_t C_max, int32_t k, int32_t n_dec, float tau, const int32_t* __restrict__ cand_pos,
    const int32_t* __restrict__ cand_count, const int32_t* __restrict__ ids, const float* __restrict__ entropy,
    const float* __restrict__ log_conf, int32_t* __restrict__ tokens, uint8_t* __restrict__ mask,
    int32_t* __restrict__ ring, int32_t* __restrict__ ring_head, int32_t* __restrict__ ring_count,
    int32_t* __restrict__ dec_pos, float* __restrict__ E_out, uint8_t* __restrict__ flag_out,
    int32_t* __restrict__ idx, int32_t* __restrict__ R_out, int32_t* __restrict__ dev_err) {
  extern __shared__ uint32_t bitmap[];  // ceil(L / 32) words: the recompute set under construction
  __shared__ SelShared sh;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t rowL = static_cast<int64_t>(b) * L;
  const int64_t rowC = static_cast<int64_t>(b) * C_max;
  int32_t* const ring_g = ring + static_cast<int64_t>(b) * k;
  const bool ring_in_smem = k <= kMaxRingSmem;
  int* const rs = ring_in_smem ? sh.ring : ring_g;
  const int nwords = (L + 31) >> 5;
  const bool fast = C_max <= 32;

  pdl_wait();  // decode results and state may come from the previous kernels in the stream
  pdl_launch_dependents();

  // ---- phase A: every global read, one round trip ------------------------------------------
  if (tid == 0) {
    int h = ring_head[b], c = ring_count[b];
    if (h < 0 || h >= k || c < 0 || c > k) {
      report_error(dev_err, EC_DEVERR_BAD_R);
      h = min(max(h, 0), k - 1);
      c = min(max(c, 0), k);
    }
    sh.head = h;
    sh.count = c;
    sh.carry = 0;
  }
  int count = __ldg(cand_count + b);
  if (count < 0 || count > C_max) {
    if (tid == 0) report_error(dev_err, EC_DEVERR_BAD_R);
    count = min(max(count, 0), C_max);
  }
  if ((L & 15) == 0) {  // 16-byte aligned rows: two vector loads per 32 positions
    const uint4* m4 = reinterpret_cast<const uint4*>(mask + rowL);
    for (int w = tid; w < nwords; w += kThreads) {
      const uint4 lo = m4[2 * w];
      const uint4 hi = (32 * w + 16 < L) ? m4[2 * w + 1] : make_uint4(0, 0, 0, 0);
      bitmap[w] = bytes_to_bits(lo, hi);
    }
  } else {
    for (int p0 = warp << 5; p0 < L; p0 += kThreads) {  // one warp per 32 positions
      const int p = p0 + lane;
      const bool m = p < L && mask[rowL + p] != 0;
      const uint32_t bits = __ballot_sync(0xffffffffu, m);
      if (lane == 0) bitmap[p0 >> 5] = bits;
    }
  }
  if (ring_in_smem)
    for (int t = tid; t < k; t += kThreads) sh.ring[t] = ring_g[t];
#pragma unroll
  for (int q = 0; q < kPerThread; ++q) {  // every field of every candidate row
    const int i = tid + q * kThreads;
    if (i < C_max) {
      const int p = __ldg(cand_pos + rowC + i);
      float c = __ldg(log_conf + rowC + i);
      if (isnan(c)) c = -INFINITY;  // NaN confidence ranks lowest
      sh.pos[i] = (p >= 0 && p < L) ? p : -1;
      sh.conf[i] = c;
      sh.ent[i] = __ldg(entropy + rowC + i);
      sh.id[i] = __ldg(ids + rowC + i);
    }
  }
  __syncthreads();

  // ---- phases B + C: validity, the committed set D, commit, history push, E ---------------
  // B: a candidate is valid if in range, still masked and the first listing of its position;
  //    D = the nD = min(n_dec, #valid) best-ranked valid candidates.
  // C: commit D, record dec_pos in ascending position order, push D onto the ring, reduce E,
  //    gate, and mark the recompute set (clear D's mask bits, set the last-k history bits).
  const int head0 = sh.head;
  if (fast) {
    // One warp holds every candidate: ranking by shuffles, no shared-memory loops.
    if (warp == 0) {
      const bool in = lane < count;
      const int p = in ? sh.pos[lane] : -1;
      const float c = in ? sh.conf[lane] : -INFINITY;
      bool ok = in && p >= 0 && bit_set(bitmap, p);
      const unsigned same = __match_any_sync(0xffffffffu, ok ? p : -2 - lane);
      ok = ok && (__ffs(same) - 1 == lane);  // first listing of its position
      if (in && !ok) report_error(dev_err, EC_DEVERR_BAD_CAND_POS);
      const unsigned vmask = __ballot_sync(0xffffffffu, ok);
      const int nD = min(n_dec, __popc(vmask));
      // D: nD rounds of a warp argmax over the not-yet-chosen valid candidates.
      bool chosen = false;
      for (int r = 0; r < nD; ++r) {
        const int wl = warp_best(c, p, ok && !chosen, lane);
        if (wl == lane) chosen = true;
      }
      const unsigned cmask = __ballot_sync(0xffffffffu, chosen);
      int ord = 0;  // rank of this position among D, ascending
      if (nD > 1) {
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const int pj = __shfl_sync(0xffffffffu, p, j);
          if (((cmask >> j) & 1u) && pj < p) ++ord;
        }
      }
      float emax = -INFINITY;
      int any_nan = 0;
      if (chosen) {
        tokens[rowL + p] = sh.id[lane];
        mask[rowL + p] = 0;
        atomicAnd(&bitmap[p >> 5], ~(1u << (p & 31)));
        dec_pos[static_cast<int64_t>(b) * n_dec + ord] = p;
        if (ord >= nD - k) {  // only the last k of D survive in the history
          const int slot = (head0 + ord) % k;
          rs[slot] = p;
          if (ring_in_smem) ring_g[slot] = p;
        }
        const float h = sh.ent[lane];
        if (isnan(h)) any_nan = 1;
        else emax = fmaxf(emax, h);
      }
      for (int t = nD + lane; t < n_dec; t += 32) dec_pos[static_cast<int64_t>(b) * n_dec + t] = -1;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        emax = fmaxf(emax, __shfl_xor_sync(0xffffffffu, emax, off));
        any_nan |= __shfl_xor_sync(0xffffffffu, any_nan, off);
      }
      const float E = nD == 0 ? 0.f : (any_nan ? NAN : emax);  // nothing decoded: E = 0
      const int full = (nD > 0 && any_nan) ? 1 : (E > tau ? 1 : 0);
      const int head1 = (head0 + nD) % k;
      const int count1 = min(sh.count + nD, k);
      if (lane == 0) {
        E_out[b] = E;
        flag_out[b] = static_cast<uint8_t>(full);
        ring_head[b] = head1;
        ring_count[b] = count1;
        sh.full = full;
      }
      __syncwarp();
      if (!full) {
        for (int t = lane; t < count1; t += 32) {  // the last min(k, count) decoded positions
          const int q = rs[((head1 - 1 - t) % k + k) % k];
          if (q >= 0 && q < L) atomicOr(&bitmap[q >> 5], 1u << (q & 31));
          else report_error(dev_err, EC_DEVERR_BAD_IDX);
        }
        __syncwarp();
        if (nwords <= 32) {
          const int R = warp_compact(bitmap, nwords, idx + rowL, lane);
          if (lane == 0) R_out[b] = R;
        }
      }
    }
  } else {
    int nvalid_local = 0;
#pragma unroll
    for (int q = 0; q < kPerThread; ++q) {
      const int i = tid + q * kThreads;
      if (i < count) {
        const int p = sh.pos[i];
        bool ok = p >= 0 && bit_set(bitmap, p);
        for (int j = 0; ok && j < i; ++j)
          if (sh.pos[j] == p) ok = false;  // a position listed twice keeps its first occurrence
        if (!ok) report_error(dev_err, EC_DEVERR_BAD_CAND_POS);
        sh.valid[i] = ok ? 1 : 0;
        nvalid_local += ok ? 1 : 0;
      }
    }
    const int nD = min(n_dec, block_sum_int(nvalid_local, sh));  // contains __syncthreads
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
        tokens[rowL + p] = sh.id[i];
        mask[rowL + p] = 0;
        atomicAnd(&bitmap[p >> 5], ~(1u << (p & 31)));
        dec_pos[static_cast<int64_t>(b) * n_dec + ord] = p;
        if (ord >= nD - k) {  // only the last k of D survive in the history
          const int slot = (head0 + ord) % k;
          rs[slot] = p;
          if (ring_in_smem) ring_g[slot] = p;
        }
        const float h = sh.ent[i];
        if (isnan(h)) any_nan = 1;
        else emax = fmaxf(emax, h);
      }
    }
    for (int t = nD + tid; t < n_dec; t += kThreads) dec_pos[static_cast<int64_t>(b) * n_dec + t] = -1;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      emax = fmaxf(emax, __shfl_xor_sync(0xffffffffu, emax, off));
      any_nan |= __shfl_xor_sync(0xffffffffu, any_nan, off);
    }
    if (lane == 0) {
      sh.warp_e[warp] = emax;
      sh.warp_nan[warp] = any_nan;
    }
    __syncthreads();
    if (tid == 0) {
      float e = -INFINITY;
      int nan_seen = 0;
      for (int w = 0; w < kWarps; ++w) {
        e = fmaxf(e, sh.warp_e[w]);
        nan_seen |= sh.warp_nan[w];
      }
      const float E = nD == 0 ? 0.f : (nan_seen ? NAN : e);  // nothing decoded: E = 0
      const int full = (nD > 0 && nan_seen) ? 1 : (E > tau ? 1 : 0);
      E_out[b] = E;
      flag_out[b] = static_cast<uint8_t>(full);
      const int head1 = (head0 + nD) % k;
      const int count1 = min(sh.count + nD, k);
      ring_head[b] = head1;
      ring_count[b] = count1;
      sh.head = head1;
      sh.count = count1;
      sh.full = full;
    }
    __syncthreads();
    if (!sh.full) {
      const int head1 = sh.head, count1 = sh.count;
      for (int t = tid; t < count1; t += kThreads) {  // the last min(k, count) decoded positions
        const int q = rs[((head1 - 1 - t) % k + k) % k];
        if (q >= 0 && q < L) atomicOr(&bitmap[q >> 5], 1u << (q & 31));
        else report_error(dev_err, EC_DEVERR_BAD_IDX);
      }
    }
  }
  __syncthreads();

  // ---- phase D: the recompute set ------------------------------------------------------------
  if (sh.full) {
    for (int r = tid; r < L; r += kThreads) idx[rowL + r] = r;
    if (tid == 0) R_out[b] = L;
    return;
  }
  if (fast && nwords <= 32) return;  // warp 0 has compacted already
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
  return launch_pdl(select_recompute_kernel, dim3(p.B), dim3(kThreads), smem, s, p.L, p.C_max, p.k, p.n_dec, p.tau,
                    cand_pos, cand_count, ids, entropy, log_conf, st.tokens, st.mask, st.ring, st.ring_head,
                    st.ring_count, st.dec_pos, st.E, st.flag, st.idx, st.R, st.dev_err);
}

}  // namespace ec
