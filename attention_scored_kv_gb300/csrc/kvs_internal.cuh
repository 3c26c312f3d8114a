// Internal declarations shared by the CUDA translation units of libkvs.
//
// Workspace layout (all regions 256-byte aligned, owned by the caller):
//   per layer l (stride = layer_bytes of each array):
//     K pages, V pages   [num_pages][Hkv][16][D] storage elements
//     K, V scales        [num_pages][16] float        (E4M3 only)
//     positions          [num_pages][16] int64         (-1 = empty slot)
//     token masses       [num_pages][16] float         (entry masses of the last attend)
//     block masses       [max_seqs][max_blocks] float  (block masses of the last attend)
//     next_position      [max_seqs] int64
//     append tickets     [max_seqs] int32
//   shared by all layers:
//     block table, resident block list, resident page list [max_seqs][max_blocks] int32
//     resident count [max_seqs]; free page stack [num_pages] + top
//     score tables C/E per token [max_seqs][max_positions] double, stamp int32;
//     C/E per block [max_seqs][max_blocks] double, stamp int32; steps [max_seqs] int32
//     side-car: trajectory ring [max_seqs][max_blocks][traj_len] float, layer profiles
//     [max_seqs][max_blocks][profiled layers] double, head profiles [max_seqs][max_blocks]
//     [profiled heads] double and their per-step inputs [max_seqs][max_blocks][4] float
//     attend partials: output rows [(grid_max + max_seqs)][Hq][D] float and (m, l) words
//     [(grid_max + max_seqs)][Hq] u64; arrival counters
//     logit scratch (the general kernel, and the tensor kernel when logits do not fit
//     in shared memory); accumulate tickets; the error word.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/kvs.h"

namespace kvs {

constexpr int kBlock = 16;          // tokens per block (placement unit)
constexpr int kGridMax = 256;       // upper bound of persistent attend CTAs (sizing)
constexpr int kPsSeqMax = 512;     // sequences of one prefill-scoring launch

// Device error word bits.
enum : int32_t {
  kErrCapacity = 1,      // H2O page pool empty / position overflow seen on device
  kErrTimeout = 2,       // a bounded wait ran out
  kErrState = 4,         // missing page / inconsistent state seen on device
  kErrBounds = 8,        // a debug-build bounds check failed (the access was skipped)
};

// The attend's per-sequence counters each sit on a 128-byte line of their own: every
// CTA of a sequence polls them, and counters of several sequences on one line made all
// pollers and all atomics contend for it.  Output arrivals at 0, departures at
// kDepartAt, softmax-statistics arrivals at kMlAt.
constexpr int kCounterInts = 96;
constexpr int kDepartAt = 32;
constexpr int kMlAt = 64;

// The sequences of one launch: the i-th is ids[i] (a device list) or begin + i (a
// contiguous range, ids == nullptr).
struct SeqSel {
  int32_t begin;
  const int32_t* ids;
  __device__ __forceinline__ int at(int i) const { return ids ? __ldg(ids + i) : begin + i; }
};

// Options of a tensor-core attend launch (all off by default).
struct AttendOpts {
  const void* k_new = nullptr;       // fused append of one token per sequence
  const void* v_new = nullptr;
  const int32_t* list_ids = nullptr; // block list [n_seqs][list_stride], list_count[n_seqs]
  const int32_t* list_count = nullptr;
  int list_stride = 0;
  float* tok_out = nullptr;          // entry masses also to [n_seqs][max_positions] (optional)
};

struct Dev {
  // shape
  int32_t L, Hq, Hkv, D, G;
  int32_t max_seqs, max_positions, max_blocks;
  int32_t window, mode, num_pages, pages_per_seq;
  int32_t kv_dtype, in_dtype;
  int32_t spin_limit;     // polls of a device wait; -1: no wait (only the last arrival goes on)
  int32_t h2o_sink_tokens, h2o_recent_tokens;
  double ema_decay;
  // per-layer arrays: base pointer + per-layer stride in elements
  uint8_t* k_pages;  uint8_t* v_pages;  size_t page_layer_bytes;  size_t page_bytes;
  float* k_scales;   float* v_scales;   size_t slot_layer_elems;   // num_pages*16
  int64_t* pos;
  float* tok_mass;
  float* blk_mass;   size_t blk_layer_elems;                       // max_seqs*max_blocks
  int64_t* next_pos;                                               // [L][max_seqs]
  int32_t* append_tickets;                                         // [L][max_seqs]
  // shared
  int32_t* block_table;   // [max_seqs][max_blocks]
  int32_t* res_blocks;    // [max_seqs][max_blocks]
  int32_t* res_pages;     // [max_seqs][max_blocks]
  int32_t* res_count;     // [max_seqs]
  int32_t* free_pages;    // [num_pages]
  int32_t* free_top;      // [1]
  double* c_tok; double* e_tok; int32_t* last_tok;   // [max_seqs][max_positions]
  double* c_blk; double* e_blk; int32_t* last_blk;   // [max_seqs][max_blocks]
  double* s_blk; double* t_blk;                      // [max_seqs][max_blocks] summed over entries
  float* traj;  int32_t traj_len;                    // [max_seqs][max_blocks][traj_len] ring of t_blk
  double* prof; int32_t n_prof;                      // [max_seqs][max_blocks][n_prof] layer profiles
  int32_t prof_layer[4];                             // profiled layers, ascending
  // per-head profiles: the attend of layer hprof_layer[j] writes head hprof_head[j]'s
  // in-block weight to hstep [max_seqs][max_blocks][4]; the accumulate adds it to
  // hprof [max_seqs][max_blocks][n_hprof]
  float* hstep; double* hprof; int32_t n_hprof;
  int32_t hprof_layer[4], hprof_head[4];
  // prefill scoring scratch (obs_window > 0), for the S <= kPsSeqMax sequences of one
  // launch and its groups g = (launch slot, KV head): row partials (max, sum) per (CTA +
  // group) slot [kGridMax + S * Hkv][256]; per group the entry sums [S * Hkv][ps_bound][16]
  // and block values [S * Hkv][ps_bound]; group arrival and departure counters
  // [S * Hkv]; KV-head tickets [S][ps_bound]
  float2* ps_part; float* ps_tok; float* ps_blk;
  int32_t* ps_ready; int32_t* ps_done; int32_t* ps_tickets;
  int32_t ps_bound;
  int32_t* steps;                                    // [max_seqs]
  int32_t* acc_tickets;                              // [max_seqs]
  float* partials;        // [records][Hq][D] partial output rows, records = kGridMax + max_seqs
  unsigned long long* part_ml;   // [records][Hq] softmax partials (l bits << 32 | m bits)
  int32_t* counters;      // [max_seqs][kCounterInts]: arrivals at 0, departures at kDepartAt,
                          // statistics arrivals at kMlAt
  float* logit_scratch;   size_t logit_scratch_elems;
  int32_t* err;           // [1]
};

__host__ __device__ inline int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Storage location of absolute position p of sequence s: page and slot in page.
__device__ __forceinline__ int32_t page_of(const Dev& d, int s, int64_t p, int32_t* slot) {
  if (d.mode == KVS_MODE_WINDOW) {
    int64_t w = p % d.window;
    *slot = (int32_t)(w % kBlock);
    return s * d.pages_per_seq + (int32_t)(w / kBlock);
  }
  *slot = (int32_t)(p % kBlock);
  if (d.mode == KVS_MODE_H2O) return d.block_table[(size_t)s * d.max_blocks + p / kBlock];
  return s * d.pages_per_seq + (int32_t)(p / kBlock);
}

// Resident block range of sequence s given next position nxt.
//   NONE / WINDOW: blocks [k0, k0 + n) contiguous in block id; H2O: the resident list.
struct SeqBlocks {
  int64_t next, lo;   // resident positions are lo <= p < next (H2O: within listed blocks)
  int32_t k0, n;      // first block id and block count (H2O: k0 unused)
};

// The same for a given next position (NONE / WINDOW; H2O reads its resident count).
__device__ __forceinline__ SeqBlocks seq_blocks_at(const Dev& d, int s, int64_t next) {
  SeqBlocks r;
  r.next = next;
  r.lo = 0;
  if (d.mode == KVS_MODE_WINDOW && r.next > d.window) r.lo = r.next - d.window;
  if (r.next <= 0) { r.k0 = 0; r.n = 0; return r; }
  if (d.mode == KVS_MODE_H2O) { r.k0 = 0; r.n = d.res_count[s]; return r; }
  r.k0 = (int32_t)(r.lo / kBlock);
  r.n = (int32_t)((r.next - 1) / kBlock) - r.k0 + 1;
  return r;
}

__device__ __forceinline__ SeqBlocks seq_blocks(const Dev& d, int layer, int s) {
  return seq_blocks_at(d, s, d.next_pos[(size_t)layer * d.max_seqs + s]);
}

// Block id and page of the i-th resident block of sequence s.
__device__ __forceinline__ int32_t block_at(const Dev& d, int s, const SeqBlocks& sb, int i,
                                            int32_t* page) {
  if (d.mode == KVS_MODE_H2O) {
    *page = d.res_pages[(size_t)s * d.max_blocks + i];
    return d.res_blocks[(size_t)s * d.max_blocks + i];
  }
  int32_t k = sb.k0 + i;
  int32_t idx = (d.mode == KVS_MODE_WINDOW) ? (k % d.pages_per_seq) : k;
  *page = s * d.pages_per_seq + idx;
  return k;
}

__device__ __forceinline__ void set_error(const Dev& d, int32_t bits) { atomicOr(d.err, bits); }

// Debug builds (KVS_DEBUG) check indices that come from device memory the host could
// not validate (sequence ids of a device list, pages, block ids) before using them: a
// failed check records kErrBounds and the caller skips the access.  Release builds
// compile the checks away.
#ifdef KVS_DEBUG
#define KVS_DCHECK(d, cond) ((cond) ? true : (set_error((d), kErrBounds), false))
#else
#define KVS_DCHECK(d, cond) true
#endif

// Per-head profiles: record head h's in-block weight w of block k of sequence s, when
// (layer, h) is profiled.
__device__ __forceinline__ void record_head(const Dev& d, int layer, int s, int32_t k, int h, float w) {
  for (int j = 0; j < d.n_hprof; ++j)
    if (d.hprof_layer[j] == layer && d.hprof_head[j] == h)
      d.hstep[((size_t)s * d.max_blocks + k) * 4 + j] = w;
}

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ int32_t ld_acquire(const int32_t* p) {
  int32_t v;
  asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Poll *p until it reaches target: at most `limit` polls after the first (limit 0: one
// look only), 32 ns apart for the first 64, then 100 ns apart.
// Returns false when the limit ran out (the caller records kErrTimeout).
__device__ __forceinline__ bool wait_at_least(const int32_t* p, int32_t target, int32_t limit) {
  for (int32_t it = 0;; ++it) {
    if (ld_acquire(p) >= target) return true;
    if (it >= limit) return false;
    __nanosleep(it < 64 ? 32 : 100);    // short sleeps first: arrivals are close
  }
}

}  // namespace kvs

// Host-side entry points of each translation unit (launchers).
#include <atomic>
namespace kvs {
// Dynamic shared-memory opt-in of kernel `fn` to `bytes` on the current device, made
// once per device: the attribute is per device, so `done` keeps one bit per device
// (devices 0..63; others set it on every call).  Two host threads that race on a
// device's first call may both make the call, which sets the same value.
template <typename Kernel>
inline cudaError_t smem_optin_once(std::atomic<unsigned long long>& done, Kernel fn, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_release);
  return e;
}

struct Ctx;
cudaError_t launch_init(const Dev& d, cudaStream_t st);
cudaError_t launch_reset(const Dev& d, SeqSel sel, int n_seqs, cudaStream_t st);
cudaError_t launch_alloc_pages(const Dev& d, int layer, SeqSel sel, int n_seqs, int n_new,
                               cudaStream_t st);
cudaError_t launch_append(const Dev& d, int layer, SeqSel sel, int n_seqs, int n_new,
                          const void* k, const void* v, cudaStream_t st);
cudaError_t launch_attend_general(const Dev& d, int layer, SeqSel sel, int n_seqs,
                                  const void* q, float* out, float* tok_out, cudaStream_t st);
int accumulate_select_max_blocks();
cudaError_t launch_accumulate_select(const Dev& d, SeqSel sel, int n_seqs, int max_blocks_per_seq,
                                     const int32_t* k_per_seq, int k_uniform, int score_kind, uint32_t flags,
                                     int32_t* keep_ids, int keep_capacity, int32_t* keep_count, cudaStream_t st);
cudaError_t launch_accumulate(const Dev& d, SeqSel sel, int n_seqs, int max_blocks_per_seq,
                              cudaStream_t st);
cudaError_t launch_select(const Dev& d, SeqSel sel, int n_seqs, const int32_t* k_per_seq,
                          int k_uniform, int score_kind, uint32_t flags, int32_t* keep_ids, int keep_capacity,
                          int32_t* keep_count, cudaStream_t st);
cudaError_t launch_read_ema(const Dev& d, int what, double* dst, cudaStream_t st);
cudaError_t launch_read_trajectory(const Dev& d, float* dst, cudaStream_t st);
cudaError_t launch_filter(const Dev& d, SeqSel sel, int n_seqs, int score_kind, double theta, int32_t* ids,
                          int capacity, int32_t* count, cudaStream_t st);
cudaError_t launch_clear(const Dev& d, cudaStream_t st);
int prefill_obs_max();
}  // namespace kvs
struct CUtensorMap_st;
namespace kvs {
// k_map: the layer's bf16 K pages with one KV head per box (null for E4M3 caches)
cudaError_t launch_prefill_score(const Dev& d, const CUtensorMap_st* k_map, int layer, SeqSel sel, int n_seqs,
                                 const void* q_obs, int n_obs, int grid, cudaStream_t st);
size_t general_smem_bytes(int Hq, int D);
}  // namespace kvs
