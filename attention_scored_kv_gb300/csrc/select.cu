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
// key); the keys are kept in shared memory when they fit.  An MSB-first radix select
// over the key bytes (histogram in shared memory, bucket found by one warp scan) finds
// the key T of the k-th best and how many candidates equal to T to take; a stable
// compaction in id order then emits every key > T and the first ties in id order.
#include "select_key.cuh"

namespace kvs {

namespace {

constexpr int kThreads = 512;
constexpr int kSmemCap = 6144;          // candidates whose keys stay in shared memory


struct SelShared {
  uint32_t hist[256];
  int32_t warp_sums[kThreads / 32];
  uint64_t prefix;
  int32_t remaining;
  int32_t n_prot;
};


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

__global__ void __launch_bounds__(kThreads) select_kernel(Dev d, SeqSel sel, const int32_t* k_per_seq,
                                                            int k_uniform, int kind, uint32_t flags, int32_t* keep_ids,
                                                            int keep_capacity, int32_t* keep_count) {
  __shared__ SelShared sh;
  extern __shared__ uint8_t dyn[];
  uint64_t* skey = reinterpret_cast<uint64_t*>(dyn);                 // [kSmemCap]
  int32_t* sid = reinterpret_cast<int32_t*>(skey + kSmemCap);        // [kSmemCap]
  int32_t* spage = sid + kSmemCap;                                   // [kSmemCap]
  const int sl = blockIdx.x, s = sel.at(sl);
  if (!KVS_DCHECK(d, s >= 0 && s < d.max_seqs)) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const SeqBlocks sb = seq_blocks(d, 0, s);
  const int n = sb.n;
  const bool protect = (flags & KVS_SELECT_PROTECT) != 0;
  const bool apply = (flags & KVS_SELECT_APPLY) != 0 && d.mode == KVS_MODE_H2O;
  const bool in_smem = n <= kSmemCap;
  int kk = k_per_seq ? k_per_seq[sl] : k_uniform;
  if (kk < 0) kk = 0;

  // keys (into shared memory when they fit) and the protected count
  if (tid == 0) sh.n_prot = 0;
  __syncthreads();
  int cnt = 0;
  for (int i = tid; i < n; i += kThreads) {
    int32_t k, page;
    const uint64_t key = cand_key<false>(d, s, sb, i, kind, protect, d.steps[s], &k, &page);
    cnt += key == ~0ull;
    if (in_smem) { skey[i] = key; sid[i] = k; spage[i] = page; }
  }
  if (protect) atomicAdd(&sh.n_prot, cnt);
  __syncthreads();
  if (kk < sh.n_prot) kk = sh.n_prot;
  const bool keep_all = kk >= n;

  auto key_of = [&](int i, int32_t* k, int32_t* page) -> uint64_t {
    if (in_smem) { *k = sid[i]; *page = spage[i]; return skey[i]; }
    return cand_key<false>(d, s, sb, i, kind, protect, d.steps[s], k, page);
  };

  // radix select of the kk-th largest key (k = 0 keeps nothing: T above every key)
  if (tid == 0) { sh.prefix = kk > 0 ? 0ull : ~0ull; sh.remaining = 0; }
  if (tid == 0 && kk > 0) sh.remaining = kk;
  uint64_t mask = 0;
  if (!keep_all && kk > 0) {
    for (int shift = 56; shift >= 0; shift -= 8) {
      for (int b = tid; b < 256; b += kThreads) sh.hist[b] = 0;
      __syncthreads();
      const uint64_t prefix = sh.prefix;
      for (int i = tid; i < n; i += kThreads) {
        int32_t k, page;
        const uint64_t key = key_of(i, &k, &page);
        if ((key & mask) == prefix) atomicAdd(&sh.hist[(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      if (warp == 0) {
        // lane l owns buckets 255-8l .. 248-8l (descending); find the bucket holding the
        // remaining-th largest key with one scan over the lanes
        const int rem = sh.remaining;
        int c8[8], local = 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) { c8[u] = (int)sh.hist[255 - 8 * lane - u]; local += c8[u]; }
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int v = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += v;
        }
        const int excl = incl - local;
        const unsigned m = __ballot_sync(0xffffffffu, excl < rem && incl >= rem);
        const int src = m ? __ffs(m) - 1 : 31;
        if (lane == src) {
          int r2 = rem - excl, bucket = 248 - 8 * lane;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            if (c8[u] >= r2) { bucket = 255 - 8 * lane - u; break; }
            r2 -= c8[u];
          }
          sh.prefix = prefix | ((uint64_t)bucket << shift);
          sh.remaining = r2;
        }
      }
      mask |= 255ull << shift;
      __syncthreads();
    }
  }
  const uint64_t T = sh.prefix;        // key of the kk-th best (all bytes fixed)
  const int take_eq = sh.remaining;    // how many keys == T to keep, lowest ids first

  // stable compaction in id order (chunks of kThreads); eviction rewrites the list
  int kept_before = 0, eq_before = 0;
  for (int c0 = 0; c0 < n; c0 += kThreads) {
    const int i = c0 + tid;
    int32_t k = -1, page = -1;
    uint64_t key = 0;
    const bool live = i < n;
    if (live) key = key_of(i, &k, &page);
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
  if (tid == 0) {
    keep_count[sl] = kept_before;
    if (apply) d.res_count[s] = kept_before;
  }
}

// Threshold view ("Context views at marginal cost", Tier 1: a view filters the kept
// table by a_s > theta): one CTA per sequence writes the resident blocks whose score
// exceeds theta, in ascending id, 512 candidates per pass.
__global__ void __launch_bounds__(kThreads) filter_kernel(Dev d, SeqSel sel, int kind, double theta,
                                                            int32_t* ids, int capacity, int32_t* count) {
  __shared__ SelShared sh;
  const int sl = blockIdx.x, s = sel.at(sl), tid = threadIdx.x;
  if (!KVS_DCHECK(d, s >= 0 && s < d.max_seqs)) return;
  const SeqBlocks sb = seq_blocks(d, 0, s);
  const int32_t steps_now = d.steps[s];
  int before = 0;
  for (int base = 0; base < sb.n; base += kThreads) {
    const int i = base + tid;
    int32_t k = -1;
    int pass = 0;
    if (i < sb.n) {
      int32_t page;
      k = block_at(d, s, sb, i, &page);
      pass = block_score<false>(d, s, k, kind, steps_now) > theta;
    }
    int total;
    const int out = before + block_scan(pass, sh, &total);
    if (pass) {
      if (out < capacity) ids[(size_t)sl * capacity + out] = k;
      else set_error(d, kErrCapacity);
    }
    before += total;
  }
  if (tid == 0) count[sl] = before;
}

}  // namespace

cudaError_t launch_filter(const Dev& d, SeqSel sel, int n_seqs, int score_kind, double theta, int32_t* ids,
                          int capacity, int32_t* count, cudaStream_t st) {
  filter_kernel<<<n_seqs, kThreads, 0, st>>>(d, sel, score_kind, theta, ids, capacity, count);
  return cudaGetLastError();
}

cudaError_t launch_select(const Dev& d, SeqSel sel, int n_seqs, const int32_t* k_per_seq,
                          int k_uniform, int score_kind, uint32_t flags, int32_t* keep_ids, int keep_capacity,
                          int32_t* keep_count, cudaStream_t st) {
  const size_t smem = (size_t)kSmemCap * (8 + 4 + 4);
  static std::atomic<unsigned long long> optin{0};   // per device
  const cudaError_t e = smem_optin_once(optin, select_kernel, (int)smem);
  if (e != cudaSuccess) return e;
  select_kernel<<<n_seqs, kThreads, smem, st>>>(d, sel, k_per_seq, k_uniform, score_kind, flags, keep_ids,
                                                keep_capacity, keep_count);
  return cudaGetLastError();
}

}  // namespace kvs
