// Selection keys, shared by the select kernel and the fused accumulate + select kernel.
//
// "Per-Head Attention as a Scoring Signal", Combined placement decision: the highest-
// scoring (sequence, 16-token block) units stay resident.  Flash-MoE "Context
// Optimization", H2O > The Algorithm: sink tokens (the first few) and recent tokens
// (the last quarter of the budget) are always kept.
#pragma once
#include "kvs_internal.cuh"

namespace kvs {

// 64-bit key that orders like the float64 score (protected blocks get ~0, above all).
__device__ __forceinline__ uint64_t order_key(double v) {
  const uint64_t b = (uint64_t)__double_as_longlong(v);
  return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}

// H2O protection of block k of a sequence whose next position is `next`: a sink block
// (it holds one of the first sink tokens) or a recent one (it holds one of the last
// recent tokens).
__device__ __forceinline__ bool protected_block(const Dev& d, int32_t k, int64_t next) {
  const int64_t b0 = (int64_t)k * kBlock, b1 = b0 + kBlock;         // block holds [b0, b1)
  return b0 < d.h2o_sink_tokens || b1 > next - d.h2o_recent_tokens;
}

// Score of block k of sequence s (a kvs_score_kind): the cumulative score, the EMA as
// of step steps_now - 1, the token sum, or the TOVA score of step steps_now - 1 (0 for
// a block that step did not update).  L2ONLY reads the tables through L2 only (they
// were just written by other CTAs).
template <bool L2ONLY>
__device__ __forceinline__ double block_score(const Dev& d, int s, int32_t k, int kind, int32_t steps_now) {
  const size_t t = (size_t)s * d.max_blocks + k;
  double v;
  if (kind == KVS_SCORE_CUMULATIVE) {
    v = L2ONLY ? __ldcg(d.c_blk + t) : d.c_blk[t];
  } else if (kind == KVS_SCORE_TOKEN_SUM) {
    v = L2ONLY ? __ldcg(d.s_blk + t) : d.s_blk[t];
  } else if (kind == KVS_SCORE_TOVA) {
    const int32_t last = L2ONLY ? __ldcg(d.last_blk + t) : d.last_blk[t];
    const double tv = L2ONLY ? __ldcg(d.t_blk + t) : d.t_blk[t];
    v = last == steps_now - 1 ? tv : 0.0;
  } else {
    const int32_t last = L2ONLY ? __ldcg(d.last_blk + t) : d.last_blk[t];
    const double e = L2ONLY ? __ldcg(d.e_blk + t) : d.e_blk[t];
    const int32_t gap = steps_now - 1 - last;
    v = (last < 0) ? 0.0 : (gap == 0 ? e : e * pow(d.ema_decay, (double)gap));
  }
  return v;
}

// Key of the i-th resident block of sequence s (its id and page to *kid, *page): the
// order key of its block_score, ~0 when protected.
template <bool L2ONLY>
__device__ __forceinline__ uint64_t cand_key(const Dev& d, int s, const SeqBlocks& sb, int i, int kind, bool protect,
                                             int32_t steps_now, int32_t* kid, int32_t* page) {
  const int32_t k = block_at(d, s, sb, i, page);
  *kid = k;
  if (protect && protected_block(d, k, sb.next)) return ~0ull;
  return order_key(block_score<L2ONLY>(d, s, k, kind, steps_now));
}

}  // namespace kvs
