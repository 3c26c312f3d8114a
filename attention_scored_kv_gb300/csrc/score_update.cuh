// One step's update of the score tables for one entry and one block: shared by the
// accumulate kernel and the fused accumulate + select kernel, so both write identical
// values.
//
// "Context views at marginal cost", Tier 1: running reductions, O(1) per entry per
// step.  Flash-MoE "Context Optimization", H2O > How It Works, step 1: the token score
// sums the post-softmax weights over all heads (and, here, all layers) and all steps.
// "Per-Head Attention as a Scoring Signal": the block score is the maximum over heads
// (and layers).  Token score x_p = sum_l tau_l[p] (the float32 layer masses added in
// layer order as an exact float32 two-sum pair hi + lo, converted to float64 once at
// the end); block score y_k = max_l beta_l[k]; C += x;
// E <- d*E + (1-d)*x.  The decay of entries not updated for a while is applied lazily:
// each entry keeps the step at which E was last written and a reader multiplies by
// d^(steps elapsed).
#pragma once
#include "kvs_internal.cuh"

namespace kvs {

// EMA value as of step `step - 1` of an entry last written at step `last` (-1: never).
// An entry resident in the previous step (the common case) needs no power at all.
__device__ __forceinline__ double decayed(double e, int32_t last, int32_t step, double dec) {
  if (last < 0) return 0.0;
  const int32_t gap = step - 1 - last;
  if (gap == 0) return e;
  if (gap == 1) return e * dec;
  return e * pow(dec, (double)gap);
}

// Entry p of sequence s, stored in (page, slot), at step `step`; returns its score x.
// The layer sum runs in float32 as an unevaluated pair hi + lo kept exact by the
// two-sum rule (Knuth: s = a + b, bb = s - a, err = (a - (s - bb)) + (b - bb), so that
// s + err == a + b exactly), and becomes one float64 at the end: this part's float64
// rate is low, and ten float64 conversions and adds per entry dominated the update.
// The pair carries about 48 bits, beyond the float64 tables' 1e-4 absolute bar.
__device__ __forceinline__ double update_entry(const Dev& d, int s, int64_t p, int32_t page, int32_t slot,
                                               int32_t step) {
  float hi = 0.f, lo = 0.f;
  for (int l = 0; l < d.L; ++l) {
    const float v = d.tok_mass[(size_t)l * d.slot_layer_elems + (size_t)page * kBlock + slot];
    const float t = __fadd_rn(hi, v);
    const float bb = __fsub_rn(t, hi);
    lo = __fadd_rn(lo, __fadd_rn(__fsub_rn(hi, __fsub_rn(t, bb)), __fsub_rn(v, bb)));
    hi = t;
  }
  const double x = (double)hi + (double)lo;
  const size_t t = (size_t)s * d.max_positions + p;
  const int32_t last = d.last_tok[t];
  const double e_prev = decayed(d.e_tok[t], last, step, d.ema_decay);
  d.c_tok[t] += x;
  d.e_tok[t] = d.ema_decay * e_prev + (1.0 - d.ema_decay) * x;
  d.last_tok[t] = step;
  return x;
}

// Sum of the entry scores x of one block's 16 entries, held by 16 consecutive lanes
// (lane & 15 = entry; entries left out contribute 0).  Every lane of the warp calls it;
// lanes of the block get the sum.  Added in a fixed tree order.
__device__ __forceinline__ double block_entry_sum(double x) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// Block k of sequence s at step `step`, whose entries' scores sum to xsum; returns the
// new cumulative score in *c_new and the new EMA in *e_new.  The token-sum score
// (H2O) accumulates xsum, and the TOVA score is xsum.  Side-car views ("Context views
// at marginal cost", Tier 1): the trajectory ring keeps xsum in slot step % traj_len,
// each profiled layer's sum gains that layer's block mass, and each profiled head's sum
// gains that head's in-block weight of the step.
__device__ __forceinline__ void update_block(const Dev& d, int s, int32_t k, int32_t step, double xsum,
                                             double* c_new, double* e_new) {
  float y = 0.f;
  for (int l = 0; l < d.L; ++l)
    y = fmaxf(y, d.blk_mass[(size_t)l * d.blk_layer_elems + (size_t)s * d.max_blocks + k]);
  const size_t t = (size_t)s * d.max_blocks + k;
  const int32_t last = d.last_blk[t];
  const double e_prev = decayed(d.e_blk[t], last, step, d.ema_decay);
  const double c = d.c_blk[t] + (double)y;
  const double e = d.ema_decay * e_prev + (1.0 - d.ema_decay) * (double)y;
  d.c_blk[t] = c;
  d.e_blk[t] = e;
  d.s_blk[t] += xsum;
  d.t_blk[t] = xsum;
  if (d.traj_len) d.traj[t * d.traj_len + step % d.traj_len] = (float)xsum;
  for (int i = 0; i < d.n_prof; ++i)
    d.prof[t * d.n_prof + i] += (double)d.blk_mass[(size_t)d.prof_layer[i] * d.blk_layer_elems + t];
  for (int j = 0; j < d.n_hprof; ++j) d.hprof[t * d.n_hprof + j] += (double)d.hstep[t * 4 + j];
  d.last_blk[t] = step;
  *c_new = c;
  *e_new = e;
}

}  // namespace kvs
