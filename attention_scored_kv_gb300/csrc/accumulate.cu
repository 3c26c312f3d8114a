// kvs_accumulate_scores: fold one step's masses of every layer into the score tables
// (the arithmetic is in score_update.cuh).  Entries that were not attended this step
// have x = 0: their C is unchanged and their E decays, lazily.
#include "score_update.cuh"

namespace kvs {

namespace {

constexpr int kBlocksPerCta = 16;     // 16 blocks x 16 positions = 256 threads

__global__ void __launch_bounds__(256) accumulate_kernel(Dev d, SeqSel sel) {
  const int s = sel.at(blockIdx.y);
  if (!KVS_DCHECK(d, s >= 0 && s < d.max_seqs)) return;
  const SeqBlocks sb = seq_blocks(d, 0, s);
  const int32_t step = d.steps[s];            // read by every CTA before the last ticket
  const int i = blockIdx.x * kBlocksPerCta + (threadIdx.x >> 4);
  const int j = threadIdx.x & 15;
  double x = 0.0;
  int32_t k = -1;
  if (i < sb.n) {
    int32_t page;
    k = block_at(d, s, sb, i, &page);
    const int64_t p = (int64_t)k * kBlock + j;
    if (p >= sb.lo && p < sb.next) {
      int32_t slot;
      page = page_of(d, s, p, &slot);
      x = update_entry(d, s, p, page, slot, step);
    }
  }
  const double xsum = block_entry_sum(x);        // the block's 16 entries are 16 lanes
  if (i < sb.n && j == 0) {
    double c_new, e_new;
    update_block(d, s, k, step, xsum, &c_new, &e_new);
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

cudaError_t launch_accumulate(const Dev& d, SeqSel sel, int n_seqs, int max_blocks_per_seq,
                              cudaStream_t st) {
  dim3 grid((max_blocks_per_seq + kBlocksPerCta - 1) / kBlocksPerCta, n_seqs);
  if (grid.x == 0) grid.x = 1;
  accumulate_kernel<<<grid, 256, 0, st>>>(d, sel);
  return cudaGetLastError();
}

}  // namespace kvs
