// select_device.cuh — stages (b) and (c) of the EntropyCache step for one sequence, as a
// device function run by one CTA: commit the decoded tokens, gate on their maximum entropy,
// push them onto the decode history and build the recompute set.
//
// EntropyCache, gist.science zh summary §2.2 ("skip decision and selection"): if the
// maximum entropy E_{t+1} of the newly decoded tokens exceeds tau the next forward is a
// full one, otherwise it recomputes the current masked tokens plus the k most recently
// decoded tokens, taken from a decode history; §2.3: the history costs O(k) memory.
//
// The reads stage the mask as an L-bit bitmap (16-byte loads when rows are 16-byte aligned),
// the candidates and the history in shared memory (select_prefetch needs nothing from this
// step's decode; select_finish reads the decode results). With at
// most 32 candidates a single warp ranks (repeated warp argmax), commits, gates, pushes the
// history and edits the bitmap, and for L <= 1024 also compacts it; larger candidate lists
// and sequences use block-wide loops.
#pragma once

#include <climits>
#include <cmath>

#include "ec_common.cuh"
#include "ec_internal.h"
#include "entropy_merge.cuh"

namespace ec {

struct SelArgs {
  int32_t L, C_max, k, n_dec;
  // The scope of the gate: positions [scope_lo, scope_hi) (the whole sequence [0, L) unless
  // the caller decodes block by block). A full step recomputes the scope; a partial step its
  // masked positions and the recent history entries that lie in it; candidates must lie in it.
  int32_t scope_lo, scope_hi;
  float tau;
  // confidence-threshold commit: ln(conf_threshold), or -inf for the fixed-count commit
  float log_thresh;
  const int32_t* cand_pos;
  const int32_t* cand_count;
  const int32_t* ids;
  const float* entropy;
  const float* log_conf;
  int32_t* tokens;
  uint8_t* mask;
  int32_t* ring;
  int32_t* ring_head;
  int32_t* ring_count;
  int32_t* dec_pos;
  float* E;
  uint8_t* flag;
  int32_t* idx;
  int32_t* R;
  int32_t* dev_err;
  // Stage the decode state before waiting on the previous kernel: only when every kernel that
  // writes the state (mask, ring, candidates) has completed before this launch's predecessor
  // released it (inside a step, where the predecessor is the decode kernel).
  int32_t prefetch_early;
  // Inside a step: the decode kernel's per-chunk partials ([B * C_max][nchunks]), merged here
  // instead of reading ids / entropy / log_conf (null: read those).
  const ChunkPartial* partials;
  int32_t nchunks;
};
static_assert(sizeof(ChunkPartial) == 16, "partials are read as one 16-byte vector");

constexpr int kSelMaxRingSmem = 4096;  // histories up to this length are staged in smem

struct SelHdr {
  int warp_tmp[32];
  float warp_e[32];
  int warp_nan[32];
  int word_off[32];  // fast path: idx offset of each bitmap word (words <= 32)
  int head, count, full, carry;
};

// Offsets (bytes) of the per-sequence shared-memory layout.
struct SelLayout {
  int bitmap, pos, conf, ent, id, valid, chosen, ring, total;
};

__host__ __device__ inline int sel_align16(int x) { return (x + 15) & ~15; }

__host__ __device__ inline SelLayout sel_layout(int L, int C_max, int k) {
  SelLayout s;
  int off = sel_align16(static_cast<int>(sizeof(SelHdr)));
  s.bitmap = off;
  off += sel_align16(((L + 31) / 32) * 4);
  s.pos = off;
  off += sel_align16(C_max * 4);
  s.conf = off;
  off += sel_align16(C_max * 4);
  s.ent = off;
  off += sel_align16(C_max * 4);
  s.id = off;
  off += sel_align16(C_max * 4);
  s.valid = off;
  off += sel_align16(C_max);
  s.chosen = off;
  off += sel_align16(C_max);
  s.ring = off;
  off += k <= kSelMaxRingSmem ? sel_align16(k * 4) : 0;
  s.total = off;
  return s;
}

// Candidate j outranks candidate i: higher confidence; equal confidence, smaller position.
__device__ __forceinline__ bool sel_outranks(float cj, int pj, float ci, int pi) {
  return cj > ci || (cj == ci && pj < pi);
}

template <int NT>
__device__ __forceinline__ int sel_block_sum(int v, SelHdr& h) {
  constexpr int W = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if (lane == 0) h.warp_tmp[warp] = v;
  __syncthreads();
  int tot = 0;
#pragma unroll
  for (int w = 0; w < W; ++w) tot += h.warp_tmp[w];
  __syncthreads();
  return tot;
}

// Exclusive prefix sum over the block; *total receives the block sum.
template <int NT>
__device__ __forceinline__ int sel_block_scan(int v, int* total, SelHdr& h) {
  constexpr int W = NT / 32;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  if (lane == 31) h.warp_tmp[warp] = incl;
  __syncthreads();
  int before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < W; ++w) {
    const int t = h.warp_tmp[w];
    if (w < warp) before += t;
    tot += t;
  }
  __syncthreads();
  *total = tot;
  return before + incl - v;
}

__device__ __forceinline__ bool sel_bit(const uint32_t* bm, int p) { return (bm[p >> 5] >> (p & 31)) & 1u; }

// Bits of bitmap word w (positions 32 w .. 32 w + 31) that lie in [lo, hi).
__device__ __forceinline__ uint32_t sel_scope_bits(int w, int lo, int hi) {
  const int a = max(lo - 32 * w, 0), b = min(hi - 32 * w, 32);
  if (b <= a) return 0u;
  return (b - a == 32 ? 0xFFFFFFFFu : ((1u << (b - a)) - 1u)) << a;
}

// 32 mask bytes -> one bitmap word (bit t set when byte t is non-zero).
__device__ __forceinline__ uint32_t sel_bytes_to_bits(uint4 lo, uint4 hi) {
  const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
  uint32_t bits = 0;
#pragma unroll
  for (int q = 0; q < 8; ++q)
#pragma unroll
    for (int e = 0; e < 4; ++e) bits |= (((w[q] >> (8 * e)) & 0xFFu) != 0u ? 1u : 0u) << (4 * q + e);
  return bits;
}

// Warp argmax over (confidence, -position): the best-ranked lane among `live`, or -1.
__device__ __forceinline__ int sel_warp_best(float c, int p, bool live, int lane) {
  float bc = live ? c : -INFINITY;
  int bp = live ? p : INT_MAX;
  int bl = live ? lane : 32;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float oc = __shfl_xor_sync(0xffffffffu, bc, off);
    const int op = __shfl_xor_sync(0xffffffffu, bp, off);
    const int ol = __shfl_xor_sync(0xffffffffu, bl, off);
    if (ol < 32 && (bl == 32 || sel_outranks(oc, op, bc, bp))) {
      bc = oc;
      bp = op;
      bl = ol;
    }
  }
  return bl < 32 ? bl : -1;
}

// Stage-(b)+(c) reads that do not depend on this step's decode results: the mask bitmap, the
// history and the candidate positions, staged in `dyn` (16-byte aligned, sel_layout(L, C_max,
// k).total bytes). All NT threads of the calling CTA.
template <int NT>
__device__ void select_prefetch(const SelArgs& a, int b, uint8_t* dyn) {
  const int L = a.L, C_max = a.C_max, k = a.k;
  const SelLayout lay = sel_layout(L, C_max, k);
  SelHdr& h = *reinterpret_cast<SelHdr*>(dyn);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(dyn + lay.bitmap);
  int* s_pos = reinterpret_cast<int*>(dyn + lay.pos);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t rowL = static_cast<int64_t>(b) * L;
  const int64_t rowC = static_cast<int64_t>(b) * C_max;
  const int32_t* const ring_g = a.ring + static_cast<int64_t>(b) * k;
  const int nwords = (L + 31) >> 5;
  if (tid == 0) {
    int hd = a.ring_head[b], c = a.ring_count[b];
    if (hd < 0 || hd >= k || c < 0 || c > k) {
      report_error(a.dev_err, EC_DEVERR_BAD_R);
      hd = min(max(hd, 0), k - 1);
      c = min(max(c, 0), k);
    }
    h.head = hd;
    h.count = c;
    h.carry = 0;
  }
  if ((L & 15) == 0) {  // 16-byte aligned rows: two vector loads per 32 positions
    const uint4* m4 = reinterpret_cast<const uint4*>(a.mask + rowL);
    for (int w = tid; w < nwords; w += NT) {
      const uint4 lo = m4[2 * w];
      const uint4 hi = (32 * w + 16 < L) ? m4[2 * w + 1] : make_uint4(0, 0, 0, 0);
      bitmap[w] = sel_bytes_to_bits(lo, hi) & sel_scope_bits(w, a.scope_lo, a.scope_hi);
    }
  } else {
    for (int p0 = warp << 5; p0 < L; p0 += NT) {  // one warp per 32 positions
      const int p = p0 + lane;
      const bool m = p < L && a.mask[rowL + p] != 0;
      const uint32_t bits = __ballot_sync(0xffffffffu, m);
      if (lane == 0) bitmap[p0 >> 5] = bits & sel_scope_bits(p0 >> 5, a.scope_lo, a.scope_hi);
    }
  }
  if (k <= kSelMaxRingSmem) {
    int* rs = reinterpret_cast<int*>(dyn + lay.ring);
    for (int t = tid; t < k; t += NT) rs[t] = ring_g[t];
  }
  for (int i = tid; i < C_max; i += NT) {
    const int p = __ldg(a.cand_pos + rowC + i);
    s_pos[i] = (p >= 0 && p < L) ? p : -1;
  }
}

// The rest of stages (b)+(c) for sequence b, after select_prefetch by the same CTA (no
// barrier needed in between). ids/entropy/log_conf are read through L2: they may have been
// written by other CTAs of the same kernel.
template <int NT>
__device__ void select_finish(const SelArgs& a, int b, uint8_t* dyn) {
  constexpr int W = NT / 32;
  const int L = a.L, C_max = a.C_max, k = a.k, n_dec = a.n_dec;
  const SelLayout lay = sel_layout(L, C_max, k);
  SelHdr& h = *reinterpret_cast<SelHdr*>(dyn);
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(dyn + lay.bitmap);
  int* s_pos = reinterpret_cast<int*>(dyn + lay.pos);
  float* s_conf = reinterpret_cast<float*>(dyn + lay.conf);
  float* s_ent = reinterpret_cast<float*>(dyn + lay.ent);
  int* s_id = reinterpret_cast<int*>(dyn + lay.id);
  unsigned char* s_valid = dyn + lay.valid;
  unsigned char* s_chosen = dyn + lay.chosen;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int64_t rowL = static_cast<int64_t>(b) * L;
  const int64_t rowC = static_cast<int64_t>(b) * C_max;
  int32_t* const ring_g = a.ring + static_cast<int64_t>(b) * k;
  const bool ring_in_smem = k <= kSelMaxRingSmem;
  int* const rs = ring_in_smem ? reinterpret_cast<int*>(dyn + lay.ring) : ring_g;
  const int nwords = (L + 31) >> 5;
  const bool fast = C_max <= 32;

  // ---- phase A (rest): this step's decode results -----------------------------------------
  int count = __ldg(a.cand_count + b);
  if (count < 0 || count > C_max) {
    if (tid == 0) report_error(a.dev_err, EC_DEVERR_BAD_R);
    count = min(max(count, 0), C_max);
  }
  if (a.partials != nullptr) {
    // merge each candidate row's chunks: 16 lanes per row (two rows per warp, all rows of one
    // pass in flight at once), lane k of a group taking chunks k, k + 16, ...
    const int grp = lane >> 4, gl = lane & 15;
    for (int i0 = 2 * warp; i0 < C_max; i0 += 2 * W) {
      const int i = i0 + grp;
      EntPart pt{-INFINITY, INT_MAX, 0.f, 0.f};
      if (i < count) {  // rows past the count were skipped by the decode kernel
        const float4* rp = reinterpret_cast<const float4*>(a.partials + (rowC + i) * a.nchunks);
        for (int c = gl; c < a.nchunks; c += 16) {
          const float4 q = __ldcg(rp + c);
          ent_part_merge(pt, EntPart{q.x, __float_as_int(q.y), q.z, q.w});
        }
      }
      pt = ent_group16_merge(pt);
      if (gl == 0 && i < C_max) {
        float h, c;
        ent_finish(pt, h, c);
        s_conf[i] = isnan(c) ? -INFINITY : c;  // NaN confidence ranks lowest
        s_ent[i] = h;
        s_id[i] = pt.i;
      }
    }
  } else {
    for (int i = tid; i < C_max; i += NT) {
      float c = __ldcg(a.log_conf + rowC + i);
      if (isnan(c)) c = -INFINITY;  // NaN confidence ranks lowest
      s_conf[i] = c;
      s_ent[i] = __ldcg(a.entropy + rowC + i);
      s_id[i] = __ldcg(a.ids + rowC + i);
    }
  }
  __syncthreads();

  // ---- phases B + C: validity, the committed set D, commit, history push, E ---------------
  // B: a candidate is valid if in range, still masked and the first listing of its position;
  //    D = the nD = min(n_dec, #valid) best-ranked valid candidates.
  // C: commit D, record dec_pos in ascending position order, push D onto the ring, reduce E,
  //    gate, and mark the recompute set (clear D's mask bits, set the last-k history bits).
  const int head0 = h.head;
  if (fast) {
    if (warp == 0) {  // one warp holds every candidate
      const bool in = lane < count;
      const int p = in ? s_pos[lane] : -1;
      const float c = in ? s_conf[lane] : -INFINITY;
      bool ok = in && p >= 0 && sel_bit(bitmap, p);
      const unsigned same = __match_any_sync(0xffffffffu, ok ? p : -2 - lane);
      ok = ok && (__ffs(same) - 1 == lane);  // first listing of its position
      if (in && !ok) report_error(a.dev_err, EC_DEVERR_BAD_CAND_POS);
      const unsigned vmask = __ballot_sync(0xffffffffu, ok);
      const int n_above = __popc(__ballot_sync(0xffffffffu, ok && c >= a.log_thresh));
      // the most confident candidates rank first, so the top nD are exactly those above the
      // threshold (at least one when any candidate is valid)
      const int nD = vmask == 0u ? 0 : min(n_dec, max(1, n_above));
      bool chosen = false;  // D: nD rounds of a warp argmax over the remaining valid candidates
      for (int r = 0; r < nD; ++r)
        if (sel_warp_best(c, p, ok && !chosen, lane) == lane) chosen = true;
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
        a.tokens[rowL + p] = s_id[lane];
        a.mask[rowL + p] = 0;
        atomicAnd(&bitmap[p >> 5], ~(1u << (p & 31)));
        a.dec_pos[static_cast<int64_t>(b) * n_dec + ord] = p;
        if (ord >= nD - k) {  // only the last k of D survive in the history
          const int slot = (head0 + ord) % k;
          rs[slot] = p;
          if (ring_in_smem) ring_g[slot] = p;
        }
        const float hv = s_ent[lane];
        if (isnan(hv)) any_nan = 1;
        else emax = fmaxf(emax, hv);
      }
      for (int t = nD + lane; t < n_dec; t += 32) a.dec_pos[static_cast<int64_t>(b) * n_dec + t] = -1;
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        emax = fmaxf(emax, __shfl_xor_sync(0xffffffffu, emax, off));
        any_nan |= __shfl_xor_sync(0xffffffffu, any_nan, off);
      }
      const float E = nD == 0 ? 0.f : (any_nan ? NAN : emax);  // nothing decoded: E = 0
      const int full = (nD > 0 && any_nan) ? 1 : (E > a.tau ? 1 : 0);
      const int head1 = (head0 + nD) % k;
      const int count1 = min(h.count + nD, k);
      if (lane == 0) {
        a.E[b] = E;
        a.flag[b] = static_cast<uint8_t>(full);
        a.ring_head[b] = head1;
        a.ring_count[b] = count1;
        h.full = full;
      }
      __syncwarp();
      if (!full) {
        for (int t = lane; t < count1; t += 32) {  // the last min(k, count) decoded positions
          const int q = rs[((head1 - 1 - t) % k + k) % k];
          if (q < 0 || q >= L) report_error(a.dev_err, EC_DEVERR_BAD_IDX);
          else if (q >= a.scope_lo && q < a.scope_hi) atomicOr(&bitmap[q >> 5], 1u << (q & 31));
        }
        __syncwarp();
        if (nwords <= 32) {  // offsets of each word's bits in idx; every warp writes below
          const uint32_t mine = lane < nwords ? bitmap[lane] : 0u;
          const int c = __popc(mine);
          int incl = c;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const int t = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += t;
          }
          h.word_off[lane] = incl - c;
          if (lane == 31) a.R[b] = incl;
        }
      }
    }
  } else {
    int nvalid_local = 0;  // valid candidates, plus (<< 16) those at or above the threshold
    for (int i = tid; i < count; i += NT) {
      const int p = s_pos[i];
      bool ok = p >= 0 && sel_bit(bitmap, p);
      for (int j = 0; ok && j < i; ++j)
        if (s_pos[j] == p) ok = false;  // a position listed twice keeps its first occurrence
      if (!ok) report_error(a.dev_err, EC_DEVERR_BAD_CAND_POS);
      s_valid[i] = ok ? 1 : 0;
      nvalid_local += ok ? (s_conf[i] >= a.log_thresh ? 0x10001 : 1) : 0;
    }
    const int packed = sel_block_sum<NT>(nvalid_local, h);  // contains __syncthreads
    const int n_valid = packed & 0xFFFF, n_above = packed >> 16;
    const int nD = n_valid == 0 ? 0 : min(n_dec, max(1, n_above));
    for (int i = tid; i < count; i += NT) {
      int rank = 0;
      if (s_valid[i]) {
        const float ci = s_conf[i];
        const int pi = s_pos[i];
        for (int j = 0; j < count; ++j)
          if (j != i && s_valid[j] && sel_outranks(s_conf[j], s_pos[j], ci, pi)) ++rank;
      }
      s_chosen[i] = (s_valid[i] && rank < nD) ? 1 : 0;
    }
    __syncthreads();
    float emax = -INFINITY;
    int any_nan = 0;
    for (int i = tid; i < count; i += NT) {
      if (!s_chosen[i]) continue;
      const int p = s_pos[i];
      int ord = 0;
      for (int j = 0; j < count; ++j)
        if (s_chosen[j] && s_pos[j] < p) ++ord;
      a.tokens[rowL + p] = s_id[i];
      a.mask[rowL + p] = 0;
      atomicAnd(&bitmap[p >> 5], ~(1u << (p & 31)));
      a.dec_pos[static_cast<int64_t>(b) * n_dec + ord] = p;
      if (ord >= nD - k) {  // only the last k of D survive in the history
        const int slot = (head0 + ord) % k;
        rs[slot] = p;
        if (ring_in_smem) ring_g[slot] = p;
      }
      const float hv = s_ent[i];
      if (isnan(hv)) any_nan = 1;
      else emax = fmaxf(emax, hv);
    }
    for (int t = nD + tid; t < n_dec; t += NT) a.dec_pos[static_cast<int64_t>(b) * n_dec + t] = -1;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      emax = fmaxf(emax, __shfl_xor_sync(0xffffffffu, emax, off));
      any_nan |= __shfl_xor_sync(0xffffffffu, any_nan, off);
    }
    if (lane == 0) {
      h.warp_e[warp] = emax;
      h.warp_nan[warp] = any_nan;
    }
    __syncthreads();
    if (tid == 0) {
      float e = -INFINITY;
      int nan_seen = 0;
      for (int w = 0; w < W; ++w) {
        e = fmaxf(e, h.warp_e[w]);
        nan_seen |= h.warp_nan[w];
      }
      const float E = nD == 0 ? 0.f : (nan_seen ? NAN : e);  // nothing decoded: E = 0
      const int full = (nD > 0 && nan_seen) ? 1 : (E > a.tau ? 1 : 0);
      a.E[b] = E;
      a.flag[b] = static_cast<uint8_t>(full);
      const int head1 = (head0 + nD) % k;
      const int count1 = min(h.count + nD, k);
      a.ring_head[b] = head1;
      a.ring_count[b] = count1;
      h.head = head1;
      h.count = count1;
      h.full = full;
    }
    __syncthreads();
    if (!h.full) {
      const int head1 = h.head, count1 = h.count;
      for (int t = tid; t < count1; t += NT) {  // the last min(k, count) decoded positions
        const int q = rs[((head1 - 1 - t) % k + k) % k];
        if (q < 0 || q >= L) report_error(a.dev_err, EC_DEVERR_BAD_IDX);
        else if (q >= a.scope_lo && q < a.scope_hi) atomicOr(&bitmap[q >> 5], 1u << (q & 31));
      }
    }
  }
  __syncthreads();

  // ---- phase D: the recompute set ------------------------------------------------------------
  if (h.full) {  // every position of the scope
    const int lo = a.scope_lo, n = a.scope_hi - a.scope_lo;
    for (int r = tid; r < n; r += NT) a.idx[rowL + r] = lo + r;
    if (tid == 0) a.R[b] = n;
    return;
  }
  if (fast && nwords <= 32) {
    // word w of the bitmap goes to idx[word_off[w] ...]: lane j of a warp writes bit j
    for (int w = warp; w < nwords; w += W) {
      const uint32_t word = bitmap[w];
      if ((word >> lane) & 1u) a.idx[rowL + h.word_off[w] + __popc(word & ((1u << lane) - 1u))] = (w << 5) + lane;
    }
    return;
  }
  for (int base = 0; base < nwords; base += NT) {
    const int w = base + tid;
    const uint32_t bits = (w < nwords) ? bitmap[w] : 0u;
    int total = 0;
    const int off = sel_block_scan<NT>(__popc(bits), &total, h);
    int o = h.carry + off;
    uint32_t rest = bits;
    while (rest) {
      const int bit = __ffs(rest) - 1;
      a.idx[rowL + o++] = (w << 5) + bit;
      rest &= rest - 1;
    }
    __syncthreads();
    if (tid == 0) h.carry += total;
    __syncthreads();
  }
  if (tid == 0) a.R[b] = h.carry;
}

}  // namespace ec

