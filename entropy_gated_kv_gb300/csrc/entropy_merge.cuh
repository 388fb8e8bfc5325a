// entropy_merge.cuh — the combine step of stage (a), shared by the decode kernel (merging the
// stretches of a row) and the select kernel (merging a step's per-chunk partials itself).
//
// A stretch of one logit row is summarised by (m, i, S, T): its maximum m, the lowest index i
// attaining it, S = sum_j 2^d_j and T = sum_j d_j 2^d_j with d_j = (x_j - m) log2(e). For the
// whole row (EntropyCache, gist.science zh summary §2.2: the entropy of each decoded token):
//   H = -sum p ln p = ln2 (log2 S - T / S),   ln p_max = -ln2 log2 S,   id = i.
#pragma once

#include "ec_common.cuh"

namespace ec {

struct EntPart {
  float m;
  int i;
  float s;
  float t;
};

constexpr float kEntLog2e = 1.4426950408889634f;
constexpr float kEntLn2 = 0.6931471805599453f;

// Larger value wins; equal values: lower index wins.
EC_DEV void ent_argmax_merge(float& m, int& i, float m2, int i2) {
  if (m2 > m || (m2 == m && i2 < i)) {
    m = m2;
    i = i2;
  }
}

// Adds stretch b to stretch a: argmax with the lower-index rule (also over stretches whose
// values are all -inf), S and T rescaled to the larger max. S >= 1 whenever a stretch's max
// is finite (its maximum contributes 2^0), so S == 0 marks a stretch without mass.
EC_DEV void ent_part_merge(EntPart& a, const EntPart& b) {
  float m = a.m;
  int i = a.i;
  ent_argmax_merge(m, i, b.m, b.i);
  if (b.s > 0.f) {
    if (a.s > 0.f) {
      const float da = (a.m - m) * kEntLog2e, db = (b.m - m) * kEntLog2e;
      const float fa = ex2_approx(da), fb = ex2_approx(db);
      a.t = fa * fmaf(da, a.s, a.t) + fb * fmaf(db, b.s, b.t);
      a.s = fa * a.s + fb * b.s;
    } else {
      a.s = b.s;
      a.t = b.t;
    }
  }
  a.m = m;
  a.i = i;
}

// Butterfly over a warp: every lane ends with the merge of all lanes' stretches (a fixed
// pairing order, so the result does not depend on timing).
EC_DEV EntPart ent_warp_merge(EntPart p) {
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const EntPart o{__shfl_xor_sync(0xffffffffu, p.m, off), __shfl_xor_sync(0xffffffffu, p.i, off),
                    __shfl_xor_sync(0xffffffffu, p.s, off), __shfl_xor_sync(0xffffffffu, p.t, off)};
    ent_part_merge(p, o);
  }
  return p;
}

// Butterfly within aligned groups of 16 lanes: every lane ends with its group's merge.
EC_DEV EntPart ent_group16_merge(EntPart p) {
#pragma unroll
  for (int off = 1; off < 16; off <<= 1) {
    const EntPart o{__shfl_xor_sync(0xffffffffu, p.m, off), __shfl_xor_sync(0xffffffffu, p.i, off),
                    __shfl_xor_sync(0xffffffffu, p.s, off), __shfl_xor_sync(0xffffffffu, p.t, off)};
    ent_part_merge(p, o);
  }
  return p;
}

// Entropy (nats) and log-probability of the decoded token of a whole row.
EC_DEV void ent_finish(const EntPart& p, float& entropy, float& log_conf) {
  const float l2s = lg2_approx(p.s);
  entropy = kEntLn2 * (l2s - p.t / p.s);
  log_conf = -kEntLn2 * l2s;
}

}  // namespace ec
