// kvs_select_blocks: per sequence, the top-k resident blocks by score, ties to the
// lower block id, optionally with H2O protection and eviction.
//
// "Per-Head Attention as a Scoring Signal", Combined placement decision: the highest-
// scoring (sequence, 16-token block) units stay resident.  Flash-MoE "Context
// Optimization", H2O > The Algorithm: sink tokens (the first few) and recent tokens
// (the last quarter of the budget) are always kept, the rest of the budget goes to the
// top scorers; eviction runs when the resident count exceeds the budget.
//
// One CTA per sequence.  Candidates are enumerated in ascending block id.  Each gets a
// 64-bit key that orders like its float64 score (protected blocks get the largest
// key); an MSB-first radix select over the key bytes finds the key T of the k-th best
// and how many of the candidates equal to T to take; a stable compaction in id order
// then emits every key > T and the first ties in id order, ascending.
#include "kvs_internal.cuh"

namespace kvs {

namespace {

constexpr int kThreads = 512;

__device__ __forceinline__ uint64_t order_key(double v) {
  const uint64_t b = (uint64_t)__double_as_longlong(v);
  return (b >> 63) ? ~b : (b | 0x8000000000000000ull);
}

struct SelShared {
  uint32_t hist[256];
  int32_t warp_sums[kThreads / 32];
  uint64_t prefix;
  int32_t remaining;
  int32_t n_prot;
  int32_t base;
};

__device__ __forceinline__ uint64_t cand_key(const Dev& d, int s, const SeqBlocks& sb, int i, int kind,
                                             bool protect, int32_t* kid, int32_t* page) {
  const int32_t k = block_at(d, s, sb, i, page);
  *kid = k;
  if (protect) {
    const int64_t b0 = (int64_t)k * kBlock, b1 = b0 + kBlock;       // block holds [b0, b1)
    const bool sink = b0 < d.h2o_sink_tokens;
    const bool recent = b1 > sb.next - d.h2o_recent_tokens;
    if (sink || recent) return ~0ull;
  }
  const size_t t = (size_t)s * d.max_blocks + k;
  double v;
  if (kind == KVS_SCORE_CUMULATIVE) {
    v = d.c_blk[t];
  } else {
    const int32_t last = d.last_blk[t];
    v = (last < 0) ? 0.0 : d.e_blk[t] * pow(d.ema_decay, (double)(d.steps[s] - 1 - last));
  }
  return order_key(v);
}

// Block-wide exclusive scan of one flag per thread; returns the exclusive prefix and
// writes the total to *total.  All threads must call it.
__device__ __forceinline__ int block_scan(int flag, SelShared& sh, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const unsigned bal = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(bal & ((1u << lane) - 1u));
  if (lane == 0) sh.warp_sums[warp] = __popc(bal);
  __syncthreads();
  int before = 0, tot = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    const int v = sh.warp_sums[w];
    if (w < warp) before += v;
    tot += v;
  }
  __syncthreads();
  *total = tot;
  return before + in_warp;
}

__global__ void __launch_bounds__(kThreads) select_kernel(Dev d, int seq_begin, const int32_t* k_per_seq,
                                                            int k_uniform, int kind, uint32_t flags, int32_t* keep_ids,
                                                            int keep_capacity, int32_t* keep_count) {
  __shared__ SelShared sh;
  const int sl = blockIdx.x, s = seq_begin + sl;
  const SeqBlocks sb = seq_blocks(d, 0, s);
  const int n = sb.n;
  const bool protect = (flags & KVS_SELECT_PROTECT) != 0;
  const bool apply = (flags & KVS_SELECT_APPLY) != 0 && d.mode == KVS_MODE_H2O;
  int kk = k_per_seq ? k_per_seq[sl] : k_uniform;
  if (kk < 0) kk = 0;

  // protected count
  if (threadIdx.x == 0) sh.n_prot = 0;
  __syncthreads();
  if (protect) {
    int cnt = 0;
    for (int i = threadIdx.x; i < n; i += kThreads) {
      int32_t k, page;
      cnt += cand_key(d, s, sb, i, kind, true, &k, &page) == ~0ull;
    }
    atomicAdd(&sh.n_prot, cnt);
    __syncthreads();
    if (kk < sh.n_prot) kk = sh.n_prot;
  }
  const bool keep_all = kk >= n;

  // radix select of the kk-th largest key
  if (threadIdx.x == 0) { sh.prefix = 0; sh.remaining = kk; }
  uint64_t mask = 0;
  if (!keep_all) {
    for (int shift = 56; shift >= 0; shift -= 8) {
      for (int b = threadIdx.x; b < 256; b += kThreads) sh.hist[b] = 0;
      __syncthreads();
      const uint64_t prefix = sh.prefix;
      for (int i = threadIdx.x; i < n; i += kThreads) {
        int32_t k, page;
        const uint64_t key = cand_key(d, s, sb, i, kind, protect, &k, &page);
        if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        int rem = sh.remaining;
        for (int b = 255; b >= 0; --b) {
          const int c = (int)sh.hist[b];
          if (c >= rem) { sh.prefix = prefix | ((uint64_t)b << shift); break; }
          rem -= c;
        }
        sh.remaining = rem;
      }
      mask |= 255ull << shift;
      __syncthreads();
    }
  }
  const uint64_t T = sh.prefix;        // key of the kk-th best (all bytes fixed)
  const int take_eq = sh.remaining;    // how many keys == T to keep, lowest ids first

  // stable compaction in id order (chunks of kThreads); eviction rewrites the list
  int kept_before = 0, eq_before = 0;
  if (threadIdx.x == 0) sh.base = 0;
  for (int c0 = 0; c0 < n; c0 += kThreads) {
    const int i = c0 + threadIdx.x;
    int32_t k = -1, page = -1;
    uint64_t key = 0;
    const bool live = i < n;
    if (live) key = cand_key(d, s, sb, i, kind, protect, &k, &page);
    int eq_total;
    const int is_eq = (!keep_all && live && key == T) ? 1 : 0;
    const int eq_rank = eq_before + block_scan(is_eq, sh, &eq_total);
    eq_before += eq_total;
    const int keep = live && (keep_all || key > T || (is_eq && eq_rank < take_eq));
    int kept_total;
    const int out = kept_before + block_scan(keep, sh, &kept_total);
    kept_before += kept_total;
    // every thread has read its candidate before anyone rewrites the list
    __syncthreads();
    if (keep) {
      if (out < keep_capacity) keep_ids[(size_t)sl * keep_capacity + out] = k;
      else set_error(d, kErrCapacity);
      if (apply) {
        d.res_blocks[(size_t)s * d.max_blocks + out] = k;
        d.res_pages[(size_t)s * d.max_blocks + out] = page;
      }
    } else if (live && apply) {
      d.block_table[(size_t)s * d.max_blocks + k] = -1;
      const int32_t top = atomicAdd(d.free_top, 1);
      d.free_pages[top] = page;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    keep_count[sl] = kept_before;
    if (apply) d.res_count[s] = kept_before;
  }
}

}  // namespace

cudaError_t launch_select(const Dev& d, int seq_begin, int n_seqs, const int32_t* k_per_seq,
                          int k_uniform, int score_kind, uint32_t flags, int32_t* keep_ids, int keep_capacity,
                          int32_t* keep_count, cudaStream_t st) {
  select_kernel<<<n_seqs, kThreads, 0, st>>>(d, seq_begin, k_per_seq, k_uniform, score_kind, flags, keep_ids,
                                             keep_capacity, keep_count);
  return cudaGetLastError();
}

}  // namespace kvs
