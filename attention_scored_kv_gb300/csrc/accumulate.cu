// kvs_accumulate_scores: fold one step's masses of every layer into the score tables.
//
// "Context views at marginal cost", Tier 1: keep running reductions (cumulative and
// EMA, O(1) per entry per step), never the attention matrix.  Flash-MoE "Context
// Optimization", H2O > How It Works, step 1: the token score sums the post-softmax
// weights over all heads (and, here, all layers) and all steps.  "Per-Head Attention
// as a Scoring Signal": the block score is the maximum over heads (and layers).
//
// Token score x_p = sum_l tau_l[p] (float64 sum of the float32 layer masses, layers in
// order); block score y_k = max_l beta_l[k]; C += x; E <- d*E + (1-d)*x.  Entries that
// were not attended this step have x = 0: their C is unchanged and their E decays.
// The decay of such entries is applied lazily: each entry keeps the step at which E
// was last written and any reader multiplies by d^(steps elapsed); a resident entry
// (updated every step) therefore sees exactly the recursive update.
#include "kvs_internal.cuh"

namespace kvs {

namespace {

constexpr int kBlocksPerCta = 16;     // 16 blocks x 16 positions = 256 threads

// EMA value as of step `step - 1` of an entry last written at step `last` (-1: never).
// An entry resident in the previous step (the common case) needs no power at all.
__device__ __forceinline__ double decayed(double e, int32_t last, int32_t step, double dec) {
  if (last < 0) return 0.0;
  const int32_t gap = step - 1 - last;
  if (gap == 0) return e;
  if (gap == 1) return e * dec;
  return e * pow(dec, (double)gap);
}

__global__ void __launch_bounds__(256) accumulate_kernel(Dev d, int seq_begin) {
  const int s = seq_begin + blockIdx.y;
  const SeqBlocks sb = seq_blocks(d, 0, s);
  const int32_t step = d.steps[s];            // read by every CTA before the last ticket
  const int i = blockIdx.x * kBlocksPerCta + (threadIdx.x >> 4);
  const int j = threadIdx.x & 15;
  const double dec = d.ema_decay;
  if (i < sb.n) {
    int32_t page;
    const int32_t k = block_at(d, s, sb, i, &page);
    const int64_t p = (int64_t)k * kBlock + j;
    if (p >= sb.lo && p < sb.next) {
      int32_t slot;
      page = page_of(d, s, p, &slot);
      double x = 0.0;
      for (int l = 0; l < d.L; ++l)
        x += (double)d.tok_mass[(size_t)l * d.slot_layer_elems + (size_t)page * kBlock + slot];
      const size_t t = (size_t)s * d.max_positions + p;
      const int32_t last = d.last_tok[t];
      const double e_prev = decayed(d.e_tok[t], last, step, dec);
      d.c_tok[t] += x;
      d.e_tok[t] = dec * e_prev + (1.0 - dec) * x;
      d.last_tok[t] = step;
    }
    if (j == 0) {
      float y = 0.f;
      for (int l = 0; l < d.L; ++l)
        y = fmaxf(y, d.blk_mass[(size_t)l * d.blk_layer_elems + (size_t)s * d.max_blocks + k]);
      const size_t t = (size_t)s * d.max_blocks + k;
      const int32_t last = d.last_blk[t];
      const double e_prev = decayed(d.e_blk[t], last, step, dec);
      d.c_blk[t] += (double)y;
      d.e_blk[t] = dec * e_prev + (1.0 - dec) * (double)y;
      d.last_blk[t] = step;
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int tk = atomicAdd(&d.acc_tickets[s], 1);
    if (tk == (int)gridDim.x - 1) {
      d.steps[s] = step + 1;
      d.acc_tickets[s] = 0;
      __threadfence();
    }
  }
}

}  // namespace

cudaError_t launch_accumulate(const Dev& d, int seq_begin, int n_seqs, int max_blocks_per_seq,
                              cudaStream_t st) {
  dim3 grid((max_blocks_per_seq + kBlocksPerCta - 1) / kBlocksPerCta, n_seqs);
  if (grid.x == 0) grid.x = 1;
  accumulate_kernel<<<grid, 256, 0, st>>>(d, seq_begin);
  return cudaGetLastError();
}

}  // namespace kvs
