// kvs_accumulate_select: kvs_accumulate_scores followed by kvs_select_blocks, in one
// launch, for sequences of at most kRankMax resident blocks.
//
// The grid is the accumulate kernel's: CTAs of 32 blocks x 16 entries per sequence,
// with the same updates (score_update.cuh). Keeping the float64 work spread over many
// SMs matters here, because this part's FP64 rate is low. Each CTA takes a ticket.
// The last CTA of a sequence to finish then selects for it, with the select kernel's
// keys (select_key.cuh), read through L2 because other CTAs have just written them.
// Candidates are enumerated in ascending block id, one per thread. The kept set is the
// candidates whose rank (keys above plus equal keys of lower id) is below k, found as
// the select kernel finds it: a radix select gives the k-th best key T, and the set is
// every key above T, then the first ties with T by id. A stable compaction writes them
// in id order, and H2O eviction rewrites the resident list as the select kernel does.
#include "score_update.cuh"
#include "select_key.cuh"

namespace kvs {

namespace {

constexpr int kBlocksPerCta = 32;
constexpr int kThreads = kBlocksPerCta * kBlock;   // 512
constexpr int kRankMax = kThreads;                 // one candidate per thread

// Exclusive block-wide prefix of one flag per thread; the total goes to *total.
__device__ __forceinline__ int scan_flags(int flag, int32_t* warp_sums, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  if (lane == 0) warp_sums[warp] = __popc(bal);
  __syncthreads();
  int before = 0, tot = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    const int v = warp_sums[w];
    if (w < warp) before += v;
    tot += v;
  }
  __syncthreads();
  *total = tot;
  return before + __popc(bal & ((1u << lane) - 1u));
}

__global__ void __launch_bounds__(kThreads) accumulate_select_kernel(Dev d, SeqSel sel, const int32_t* k_per_seq,
                                                                     int k_uniform, int kind, uint32_t flags,
                                                                     int32_t* keep_ids, int keep_capacity,
                                                                     int32_t* keep_count) {
  __shared__ uint64_t skey[kRankMax];
  __shared__ int32_t sid[kRankMax], spage[kRankMax];
  __shared__ int32_t warp_sums[kThreads / 32];
  __shared__ int32_t is_last;
  __shared__ uint32_t hist[256];
  __shared__ uint64_t s_prefix;
  __shared__ int32_t s_take;
  const int lane_id = threadIdx.x & 31, warp_id = threadIdx.x >> 5;
  const int sl = blockIdx.y, s = sel.at(sl), tid = threadIdx.x;
  if (!KVS_DCHECK(d, s >= 0 && s < d.max_seqs)) return;
  const SeqBlocks sb = seq_blocks(d, 0, s);
  const int32_t step = d.steps[s];            // read by every CTA before the last ticket

  // ---- accumulate, exactly as the accumulate kernel
  const int ib = blockIdx.x * kBlocksPerCta + (tid >> 4), j = tid & 15;
  double x = 0.0;
  int32_t kb = -1;
  if (ib < sb.n) {
    int32_t page;
    kb = block_at(d, s, sb, ib, &page);
    const int64_t p = (int64_t)kb * kBlock + j;
    if (p >= sb.lo && p < sb.next) {
      int32_t slot;
      page = page_of(d, s, p, &slot);
      x = update_entry(d, s, p, page, slot, step);
    }
  }
  const double xsum = block_entry_sum(x);        // the block's 16 entries are 16 lanes
  if (ib < sb.n && j == 0) {
    double c_new, e_new;
    update_block(d, s, kb, step, xsum, &c_new, &e_new);
  }
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int tk = atomicAdd(&d.acc_tickets[s], 1);
    is_last = tk == (int)gridDim.x - 1;
    if (is_last) d.acc_tickets[s] = 0;
  }
  __syncthreads();
  if (!is_last) return;

  // ---- select (the last CTA of the sequence): every CTA's tables are visible
  __threadfence();
  if (tid == 0) d.steps[s] = step + 1;
  const int n = sb.n;
  if (n > kRankMax) {                          // the host sends such launches elsewhere
    if (tid == 0) set_error(d, kErrState);
    return;
  }
  const bool protect = (flags & KVS_SELECT_PROTECT) != 0;
  const bool apply = (flags & KVS_SELECT_APPLY) != 0 && d.mode == KVS_MODE_H2O;
  int prot = 0;
  if (tid < n) {
    int32_t k, page;
    const uint64_t key = cand_key<true>(d, s, sb, tid, kind, protect, step + 1, &k, &page);
    prot = key == ~0ull;
    skey[tid] = key;
    sid[tid] = k;
    spage[tid] = page;
  }
  int n_prot = 0;
  scan_flags(prot, warp_sums, &n_prot);        // also the barrier that publishes the keys
  if (!protect) n_prot = 0;
  int kk = k_per_seq ? k_per_seq[sl] : k_uniform;
  if (kk < 0) kk = 0;
  if (kk < n_prot) kk = n_prot;
  const bool keep_all = kk >= n;
  // Radix select, most significant byte first: T = the kk-th best key and take = how
  // many keys equal to T are kept.  Kept: every key above T, then the first take keys
  // equal to T in id order (thread order).  That is the set whose rank (keys above plus
  // equal keys of lower id) is below kk.
  if (tid == 0) {
    s_prefix = 0;
    s_take = kk;
  }
  uint64_t mask = 0;
  if (!keep_all && kk > 0) {
    for (int shift = 56; shift >= 0; shift -= 8) {
      if (tid < 256) hist[tid] = 0;
      __syncthreads();
      const uint64_t prefix = s_prefix;
      if (tid < n && (skey[tid] & mask) == prefix) atomicAdd(&hist[(skey[tid] >> shift) & 255u], 1u);
      __syncthreads();
      if (warp_id == 0) {
        // lane l holds buckets 255-8l .. 248-8l (descending); the lane whose range holds
        // the take-th largest key finds its bucket
        const int rem = s_take;
        int c8[8], local = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          c8[u] = (int)hist[255 - 8 * lane_id - u];
          local += c8[u];
        }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane_id >= o) incl += v;
        }
        const int excl = incl - local;
        if (excl < rem && rem <= incl) {
          int acc = excl;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            if (acc < rem && acc + c8[u] >= rem) {
              s_prefix = prefix | ((uint64_t)(255 - 8 * lane_id - u) << shift);
              s_take = rem - acc;
            }
            acc += c8[u];
          }
        }
      }
      __syncthreads();
      mask |= 0xFFull << shift;
    }
  }
  const uint64_t T = s_prefix;
  const bool is_t = !keep_all && kk > 0 && tid < n && skey[tid] == T;
  int n_eq = 0;
  const int eq_before = scan_flags(is_t ? 1 : 0, warp_sums, &n_eq);
  const int keep = (tid < n && (keep_all || (kk > 0 && (skey[tid] > T || (is_t && eq_before < s_take))))) ? 1 : 0;
  int kept = 0;
  const int out = scan_flags(keep, warp_sums, &kept);   // candidates in id order = thread order
  if (tid < n) {
    const int32_t k = sid[tid], page = spage[tid];
    if (keep) {
      if (out < keep_capacity) keep_ids[(size_t)sl * keep_capacity + out] = k;
      else set_error(d, kErrCapacity);
      if (apply) {
        d.res_blocks[(size_t)s * d.max_blocks + out] = k;
        d.res_pages[(size_t)s * d.max_blocks + out] = page;
      }
    } else if (apply) {
      d.block_table[(size_t)s * d.max_blocks + k] = -1;
      const int32_t top = atomicAdd(d.free_top, 1);
      d.free_pages[top] = page;
    }
  }
  if (tid == 0) {
    keep_count[sl] = kept;
    if (apply) d.res_count[s] = kept;
  }
}

}  // namespace

int accumulate_select_max_blocks() { return kRankMax; }

cudaError_t launch_accumulate_select(const Dev& d, SeqSel sel, int n_seqs, int max_blocks_per_seq,
                                     const int32_t* k_per_seq, int k_uniform, int score_kind, uint32_t flags,
                                     int32_t* keep_ids, int keep_capacity, int32_t* keep_count, cudaStream_t st) {
  dim3 grid((max_blocks_per_seq + kBlocksPerCta - 1) / kBlocksPerCta, n_seqs);
  if (grid.x == 0) grid.x = 1;
  accumulate_select_kernel<<<grid, kThreads, 0, st>>>(d, sel, k_per_seq, k_uniform, score_kind, flags,
                                                      keep_ids, keep_capacity, keep_count);
  return cudaGetLastError();
}

}  // namespace kvs
