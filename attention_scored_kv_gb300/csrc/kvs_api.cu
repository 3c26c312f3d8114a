// The C ABI of libkvs: argument checks, workspace plan, host shadows, dispatch.
//
// Host shadows: the context keeps next_position per (layer, sequence), the allocation
// frontier and (H2O) a bound on resident blocks per sequence, so every call can be
// checked and sized without reading device memory.  The device holds the truth; a
// replayed CUDA graph advances the device state but not these shadows.
#include <cuda.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cstdlib>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "kvs_internal.cuh"

namespace kvs {
bool tc_supported(int Hq, int Hkv, int D, int kv_dtype, int in_dtype, int window, int mode);
cudaError_t make_page_map(CUtensorMap* map, const void* base, int num_pages, int Hkv, int kv_dtype, int box_heads);
cudaError_t launch_attend_tc(const CUtensorMap& tk, const CUtensorMap& tv, const Dev& d, int layer,
                             SeqSel sel, int n_seqs, const void* q, float* out, const int32_t* bounds, int grid,
                             const AttendOpts& opt, cudaStream_t st);
int tc_grid(int kv_dtype, int Hkv, int sm_count);
size_t static_scratch_limit();
size_t static_scratch_need(const Dev& d, int n_seqs, int grid, size_t* ml_offset);
cudaError_t launch_attend_tc_static(const CUtensorMap& tk, const CUtensorMap& tv, const Dev& d, int layer,
                                    SeqSel sel, int n_seqs, const void* q, float* out, float* tok_out,
                                    const int32_t* bounds, int grid, cudaStream_t st);
}  // namespace kvs

using namespace kvs;

namespace {

constexpr int32_t kDefaultSpin = 5000000;   // ~0.5 s of 100 ns polls

// NVTX ranges around every ABI call, for profiler timelines (Nsight Systems, ncu's
// range filters): on when the environment variable KVS_NVTX is set to anything but
// "0" when the library is first used.  Without an attached tool the calls do nothing.
bool tracing_on() {
  static const bool on = [] {
    const char* v = std::getenv("KVS_NVTX");
    return v && *v && std::strcmp(v, "0") != 0;
  }();
  return on;
}

struct Trace {
  explicit Trace(const char* name) : on(tracing_on()) {
    if (on) nvtxRangePushA(name);
  }
  ~Trace() {
    if (on) nvtxRangePop();
  }
  Trace(const Trace&) = delete;
  Trace& operator=(const Trace&) = delete;
  bool on;
};

struct Plan {
  int mode = 0, pages_per_seq = 0, num_pages = 0, max_blocks = 0, res_blocks_per_seq = 0;
  int recent_tokens = 0;
  size_t page_bytes = 0, logit_elems = 0, total = 0;
  // region offsets
  size_t k_pages, v_pages, k_scales, v_scales, pos, tok_mass, blk_mass, next_pos, app_tickets;
  size_t block_table, res_blocks, res_pages, res_count, free_pages, free_top;
  size_t c_tok, e_tok, last_tok, c_blk, e_blk, last_blk, s_blk, t_blk, traj, prof, hstep, hprof, steps, acc_tickets;
  size_t partials, part_ml, counters, logits, ps_part, ps_tok, ps_blk, ps_ready, ps_done, ps_tickets, err;
  int ps_bound = 0;
};

size_t esize(int dt) { return dt == KVS_F32 ? 4 : (dt == KVS_BF16 ? 2 : 1); }

void put(char* msg, size_t n, const char* fmt, ...) {
  if (!msg || n == 0) return;
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(msg, n, fmt, ap);
  va_end(ap);
}

kvs_status check_config(const kvs_config* c, char* msg, size_t n) {
  if (!c) { put(msg, n, "config is NULL"); return KVS_ERR_INVALID_ARGUMENT; }
  if (c->num_layers < 1) { put(msg, n, "num_layers must be >= 1"); return KVS_ERR_INVALID_ARGUMENT; }
  if (c->num_q_heads < 1 || c->num_kv_heads < 1 || c->num_q_heads % c->num_kv_heads) {
    put(msg, n, "num_q_heads must be a positive multiple of num_kv_heads");
    return KVS_ERR_INVALID_ARGUMENT;
  }
  if (c->head_dim != 16 && c->head_dim != 32 && c->head_dim != 64 && c->head_dim != 128) {
    put(msg, n, "head_dim must be 16, 32, 64 or 128");
    return KVS_ERR_UNSUPPORTED;
  }
  if (c->max_seqs < 1 || c->max_positions < 1) { put(msg, n, "max_seqs and max_positions must be >= 1"); return KVS_ERR_INVALID_ARGUMENT; }
  if (c->max_positions > (1 << 30)) { put(msg, n, "max_positions too large"); return KVS_ERR_UNSUPPORTED; }
  if (c->window < 0) { put(msg, n, "window must be >= 0 (0 = none)"); return KVS_ERR_INVALID_ARGUMENT; }
  if (c->block_tokens != kBlock) { put(msg, n, "block_tokens must be 16"); return KVS_ERR_UNSUPPORTED; }
  if (c->h2o_budget_tokens < 0 || (c->h2o_budget_tokens % kBlock)) {
    put(msg, n, "h2o_budget_tokens must be 0 or a positive multiple of 16");
    return KVS_ERR_INVALID_ARGUMENT;
  }
  if (c->h2o_sink_tokens < 0) { put(msg, n, "h2o_sink_tokens must be >= 0"); return KVS_ERR_INVALID_ARGUMENT; }
  if (!(c->h2o_recent_frac >= 0.0 && c->h2o_recent_frac <= 1.0)) { put(msg, n, "h2o_recent_frac must be in [0, 1]"); return KVS_ERR_INVALID_ARGUMENT; }
  if (!(c->ema_decay >= 0.0 && c->ema_decay < 1.0)) { put(msg, n, "ema_decay must be in [0, 1)"); return KVS_ERR_INVALID_ARGUMENT; }
  if (c->num_pages < 0) { put(msg, n, "num_pages must be >= 0"); return KVS_ERR_INVALID_ARGUMENT; }
  if (c->kernel < 0 || c->kernel > 2) { put(msg, n, "kernel must be a kvs_kernel"); return KVS_ERR_INVALID_ARGUMENT; }
  if (c->spin_limit < -1) { put(msg, n, "spin_limit must be >= -1"); return KVS_ERR_INVALID_ARGUMENT; }
  if (c->kv_dtype < KVS_F32 || c->kv_dtype > KVS_E4M3) { put(msg, n, "kv_dtype must be F32, BF16 or E4M3"); return KVS_ERR_INVALID_ARGUMENT; }
  if (c->in_dtype != KVS_F32 && c->in_dtype != KVS_BF16) { put(msg, n, "in_dtype must be F32 or BF16"); return KVS_ERR_INVALID_ARGUMENT; }
  if (c->kv_dtype == KVS_BF16 && c->in_dtype != KVS_BF16) {
    put(msg, n, "a bf16 cache needs bf16 inputs (f32 would be rounded)");
    return KVS_ERR_UNSUPPORTED;
  }
  if (c->traj_len < 0 || c->traj_len > 256) { put(msg, n, "traj_len must be in [0, 256]"); return KVS_ERR_INVALID_ARGUMENT; }
  if ((c->num_layers < 32 && (c->profile_layers >> c->num_layers)) || __builtin_popcount(c->profile_layers) > 4) {
    put(msg, n, "profile_layers: at most 4 bits, each below num_layers");
    return KVS_ERR_INVALID_ARGUMENT;
  }
  if (c->reserved_i) { put(msg, n, "reserved fields must be 0"); return KVS_ERR_INVALID_ARGUMENT; }
  if (c->n_profile_heads < 0 || c->n_profile_heads > 4) {
    put(msg, n, "n_profile_heads must be in [0, 4]");
    return KVS_ERR_INVALID_ARGUMENT;
  }
  for (int i = 0; i < c->n_profile_heads; ++i) {
    const int l = c->profile_heads[i] >> 16, h = c->profile_heads[i] & 0xffff;
    if (c->profile_heads[i] < 0 || l >= c->num_layers || h >= c->num_q_heads) {
      put(msg, n, "profile_heads[%d]: layer * 65536 + query head, both in range", i);
      return KVS_ERR_INVALID_ARGUMENT;
    }
    for (int j = 0; j < i; ++j)
      if (c->profile_heads[j] == c->profile_heads[i]) { put(msg, n, "profile_heads[%d] repeats a head", i); return KVS_ERR_INVALID_ARGUMENT; }
  }
  for (int i = c->n_profile_heads; i < 4; ++i)
    if (c->profile_heads[i]) { put(msg, n, "unused profile_heads entries must be 0"); return KVS_ERR_INVALID_ARGUMENT; }
  if (c->obs_window < 0 || c->obs_window > prefill_obs_max()) {
    put(msg, n, "obs_window must be in [0, %d]", prefill_obs_max());
    return KVS_ERR_INVALID_ARGUMENT;
  }
  for (int i = 0; i < 2; ++i) if (c->reserved_d[i] != 0.0) { put(msg, n, "reserved fields must be 0"); return KVS_ERR_INVALID_ARGUMENT; }
  const int mode = c->h2o_budget_tokens > 0 ? KVS_MODE_H2O : (c->window > 0 ? KVS_MODE_WINDOW : KVS_MODE_NONE);
  const bool tc = tc_supported(c->num_q_heads, c->num_kv_heads, c->head_dim, c->kv_dtype, c->in_dtype, c->window, mode);
  if (c->obs_window > 0 && !tc) {
    put(msg, n, "SnapKV prefill scoring (obs_window > 0) needs the tensor-core configuration: head_dim 128, 8 query "
                "heads per KV head, bf16 inputs, bf16 or E4M3 storage");
    return KVS_ERR_UNSUPPORTED;
  }
  if (c->kernel == KVS_KERNEL_TENSOR && !tc) {
    put(msg, n, "the tensor-core kernel needs head_dim 128, 8 query heads per KV head (4 or 8 KV heads), bf16 "
                "inputs, bf16 or E4M3 storage and a window that is 0 or a multiple of 16");
    return KVS_ERR_UNSUPPORTED;
  }
  if (msg && n) msg[0] = 0;
  return KVS_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

void make_plan(const kvs_config* c, Plan* p) {
  const size_t L = c->num_layers, B = c->max_seqs, Hq = c->num_q_heads, D = c->head_dim;
  p->mode = c->h2o_budget_tokens > 0 ? KVS_MODE_H2O : (c->window > 0 ? KVS_MODE_WINDOW : KVS_MODE_NONE);
  p->max_blocks = (int)cdiv64(c->max_positions, kBlock);
  if (p->mode == KVS_MODE_WINDOW) {
    p->pages_per_seq = (int)cdiv64(c->window, kBlock);
    p->num_pages = (int)(B * p->pages_per_seq);
    p->res_blocks_per_seq = std::min<int>(p->max_blocks, p->pages_per_seq + 1);
  } else if (p->mode == KVS_MODE_NONE) {
    p->pages_per_seq = p->max_blocks;
    p->num_pages = (int)(B * p->max_blocks);
    p->res_blocks_per_seq = p->max_blocks;
  } else {
    p->pages_per_seq = 0;
    p->num_pages = c->num_pages > 0 ? c->num_pages : (int)(B * p->max_blocks);
    p->res_blocks_per_seq = p->max_blocks;
  }
  p->recent_tokens = (int)std::ceil(c->h2o_recent_frac * c->h2o_budget_tokens);
  p->page_bytes = (size_t)c->num_kv_heads * kBlock * D * esize(c->kv_dtype);
  const size_t NP = p->num_pages, slots = NP * kBlock, MB = p->max_blocks, P = c->max_positions;
  // logits: the general kernel needs [seq][Hq][entries]; the tensor kernel per-CTA shares
  const size_t res_total = std::min<size_t>(B * p->res_blocks_per_seq, p->mode == KVS_MODE_H2O ? NP : SIZE_MAX);
  const size_t gen = B * Hq * (size_t)p->res_blocks_per_seq * kBlock;
  const size_t tcs = (res_total + 2 * (size_t)kGridMax) * (Hq * kBlock + 16);   // + the per-block padding
  p->logit_elems = std::max(gen, tcs);
  size_t o = 0;
  auto take = [&](size_t bytes) { size_t r = o; o = align256(o + bytes); return r; };
  p->k_pages = take(L * NP * p->page_bytes);
  p->v_pages = take(L * NP * p->page_bytes);
  const bool fp8 = c->kv_dtype == KVS_E4M3;
  p->k_scales = take(fp8 ? L * slots * 4 : 0);
  p->v_scales = take(fp8 ? L * slots * 4 : 0);
  p->pos = take(L * slots * 8);
  p->tok_mass = take(L * slots * 4);
  p->blk_mass = take(L * B * MB * 4);
  p->next_pos = take(L * B * 8);
  p->app_tickets = take(L * B * 4);
  p->block_table = take(B * MB * 4);
  p->res_blocks = take(B * MB * 4);
  p->res_pages = take(B * MB * 4);
  p->res_count = take(B * 4);
  p->free_pages = take(NP * 4);
  p->free_top = take(4);
  p->c_tok = take(B * P * 8);
  p->e_tok = take(B * P * 8);
  p->last_tok = take(B * P * 4);
  p->c_blk = take(B * MB * 8);
  p->e_blk = take(B * MB * 8);
  p->s_blk = take(B * MB * 8);
  p->t_blk = take(B * MB * 8);
  p->traj = take(B * MB * (size_t)c->traj_len * 4);
  p->prof = take(B * MB * (size_t)__builtin_popcount(c->profile_layers) * 8);
  p->hstep = take(c->n_profile_heads ? B * MB * 4 * 4 : 0);
  p->hprof = take(B * MB * (size_t)c->n_profile_heads * 8);
  p->last_blk = take(B * MB * 4);
  p->steps = take(B * 4);
  p->acc_tickets = take(B * 4);
  p->partials = take(((size_t)kGridMax + B) * Hq * D * 4);
  p->part_ml = take(((size_t)kGridMax + B) * Hq * 8);
  p->counters = take((size_t)kCounterInts * B * 4);
  p->logits = take(p->logit_elems * 4);
  // prefill scoring scratch, for the at most kPsSeqMax sequences of one launch: row
  // partials per (CTA + group) slot, per group the entry sums and block values, the
  // group arrival and departure counters, per (sequence, block) the KV-head tickets
  const bool ps = c->obs_window > 0;
  const size_t Bp = ps ? std::min<size_t>(B, (size_t)kPsSeqMax) : 0, Hkv = c->num_kv_heads;
  p->ps_bound = ps ? p->res_blocks_per_seq : 0;
  p->ps_part = take(ps ? ((size_t)kGridMax + Bp * Hkv) * 256 * 8 : 0);
  p->ps_tok = take(Bp * Hkv * p->ps_bound * kBlock * 4);
  p->ps_blk = take(Bp * Hkv * p->ps_bound * 4);
  p->ps_ready = take(Bp * Hkv * 4);
  p->ps_done = take(Bp * Hkv * 4);
  p->ps_tickets = take(Bp * p->ps_bound * 4);
  p->err = take(4);
  p->total = o;
}

}  // namespace

struct kvs_ctx {
  kvs_config cfg;
  Plan plan;
  Dev dev;
  int device = 0, sm_count = 0, kernel = KVS_KERNEL_GENERAL, grid = 0;
  std::vector<int64_t> next;        // [L][max_seqs]
  std::vector<int64_t> frontier;    // [max_seqs] max over layers of next (pages allocated below it)
  std::vector<int64_t> h2o_bound;   // [max_seqs] bound on resident blocks (H2O)
  std::vector<int32_t> bounds;      // per-launch scratch: block bound of each sequence
  std::vector<int32_t> sids;        // per-call scratch: the call's sequence ids, in order
  std::vector<uint8_t> seen;        // per-call scratch: repeated-id check [max_seqs]
  std::vector<CUtensorMap> maps;    // [L][2]
  std::vector<CUtensorMap> ps_maps; // [L]: bf16 K pages, one KV head per box (prefill scoring)
  std::string err;
};

namespace {

kvs_status fail(kvs_ctx* ctx, kvs_status s, const char* fmt, ...) {
  if (ctx) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    ctx->err = buf;
  }
  return s;
}

kvs_status cuda_ok(kvs_ctx* ctx, cudaError_t e, const char* what) {
  if (e == cudaSuccess) return KVS_OK;
  return fail(ctx, KVS_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// Check the sequences of a call and put their ids, in call order, in ctx->sids.
kvs_status check_seqs(kvs_ctx* ctx, const kvs_seqs& q) {
  const int B = ctx->cfg.max_seqs;
  if (q.count < 1 || q.count > B) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "sequence count %d outside [1, %d]", q.count, B);
  ctx->sids.resize((size_t)q.count);
  if (!q.h_ids && !q.d_ids) {
    if (q.begin < 0 || (int64_t)q.begin + q.count > B)
      return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "sequence range [%d, %d) outside [0, %d)", q.begin,
                  q.begin + q.count, B);
    for (int i = 0; i < q.count; ++i) ctx->sids[i] = q.begin + i;
    return KVS_OK;
  }
  if (!q.h_ids || !q.d_ids)
    return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "a sequence list needs both its host and its device copy");
  ctx->seen.assign((size_t)B, 0);
  for (int i = 0; i < q.count; ++i) {
    const int32_t s = q.h_ids[i];
    if (s < 0 || s >= B) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "sequence id %d outside [0, %d)", s, B);
    if (ctx->seen[s]) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "sequence id %d listed twice", s);
    ctx->seen[s] = 1;
    ctx->sids[i] = s;
  }
  return KVS_OK;
}

// The kernels' view of the call's sequences.
SeqSel sel_of(const kvs_seqs& q) {
  SeqSel r;
  r.begin = q.d_ids ? 0 : q.begin;
  r.ids = q.d_ids;
  return r;
}

int64_t seq_block_bound(const kvs_ctx* ctx, int s) {
  if (ctx->plan.mode == KVS_MODE_H2O)
    return std::min<int64_t>(ctx->plan.max_blocks, ctx->h2o_bound[s] + 2);
  return ctx->plan.res_blocks_per_seq;
}

}  // namespace

namespace {

// Sections of a score snapshot of n sequences starting at seq_begin, in snapshot order,
// each starting on a 256-byte boundary: the table's first element of seq_begin and the
// bytes of the n sequences' rows.  Returns the number of sections.
constexpr int kSnapSections = 12;
int snapshot_sections(const kvs_ctx* ctx, int seq_begin, int n, void* ptr[kSnapSections], size_t bytes[kSnapSections]) {
  const Dev& d = ctx->dev;
  const size_t P = d.max_positions, MB = d.max_blocks, s0 = seq_begin, TL = d.traj_len, NP = d.n_prof;
  int i = 0;
  auto add = [&](void* p, size_t b) { ptr[i] = p; bytes[i] = b; ++i; };
  add(d.c_tok + s0 * P, n * P * 8);
  add(d.e_tok + s0 * P, n * P * 8);
  add(d.c_blk + s0 * MB, n * MB * 8);
  add(d.e_blk + s0 * MB, n * MB * 8);
  add(d.s_blk + s0 * MB, n * MB * 8);
  add(d.t_blk + s0 * MB, n * MB * 8);
  add(d.prof + s0 * MB * NP, n * MB * NP * 8);
  add(d.hprof + s0 * MB * d.n_hprof, n * MB * (size_t)d.n_hprof * 8);
  add(d.traj + s0 * MB * TL, n * MB * TL * 4);
  add(d.last_tok + s0 * P, n * P * 4);
  add(d.last_blk + s0 * MB, n * MB * 4);
  add(d.steps + s0, (size_t)n * 4);
  return i;
}

size_t round256(size_t b) { return (b + 255) & ~(size_t)255; }

// A snapshot holds one section per table (snapshot_sections order, each 256-byte
// aligned) with the rows of the call's sequences in call order.  A range's rows are
// contiguous in both places (one copy per table); a list's are copied row by row.
kvs_status snapshot_copy(kvs_ctx* ctx, const kvs_seqs& seqs, void* buf, size_t buf_bytes, bool out,
                         kvs_stream_t stream) {
  if (!ctx) return KVS_ERR_INVALID_ARGUMENT;
  kvs_status st = check_seqs(ctx, seqs);
  if (st != KVS_OK) return st;
  const int n = seqs.count;
  const size_t need = kvs_scores_snapshot_bytes(ctx, n);
  if (!buf || buf_bytes < need) return fail(ctx, KVS_ERR_CAPACITY, "snapshot needs %zu bytes", need);
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* b = static_cast<uint8_t*>(buf);
  const bool list = seqs.h_ids != nullptr;
  void* ptr[kSnapSections];
  size_t bytes[kSnapSections];
  const int ns = snapshot_sections(ctx, list ? 0 : seqs.begin, n, ptr, bytes);
  void* row0[kSnapSections];
  size_t rowb[kSnapSections];
  snapshot_sections(ctx, 0, 1, row0, rowb);                  // one sequence's row of each table
  size_t off = 0;
  for (int i = 0; i < ns; ++i) {
    for (int r = 0; r < (list ? n : 1) && bytes[i]; ++r) {
      const size_t len = list ? rowb[i] : bytes[i];
      uint8_t* dev = static_cast<uint8_t*>(list ? row0[i] : ptr[i]) + (list ? (size_t)ctx->sids[r] * rowb[i] : 0);
      uint8_t* host = b + off + (list ? (size_t)r * rowb[i] : 0);
      void* dst = out ? static_cast<void*>(host) : static_cast<void*>(dev);
      const void* src = out ? static_cast<const void*>(dev) : static_cast<const void*>(host);
      st = cuda_ok(ctx, cudaMemcpyAsync(dst, src, len, cudaMemcpyDefault, cs), out ? "export scores" : "import scores");
      if (st != KVS_OK) return st;
    }
    off += round256(bytes[i]);
  }
  return KVS_OK;
}

}  // namespace

namespace {
// Checks shared by the attend entry points: q and out present and 16-byte aligned, the
// optional token-mass output 4-byte aligned.
kvs_status check_attend_buffers(kvs_ctx* ctx, const void* d_q, const float* d_out, const float* d_tok) {
  if (!d_q || !d_out) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "NULL q or out");
  if ((reinterpret_cast<uintptr_t>(d_q) | reinterpret_cast<uintptr_t>(d_out)) & 15)
    return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "q and out must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(d_tok) & 3)
    return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "the token-mass output must be 4-byte aligned");
  return KVS_OK;
}

// Per sequence of the call: not empty in `layer`; its block bound into ctx->bounds.
kvs_status attend_bounds(kvs_ctx* ctx, int32_t layer) {
  const int B = ctx->cfg.max_seqs;
  ctx->bounds.resize(ctx->sids.size());
  for (size_t i = 0; i < ctx->sids.size(); ++i) {
    const int32_t s = ctx->sids[i];
    if (ctx->next[(size_t)layer * B + s] == 0)
      return fail(ctx, KVS_ERR_EMPTY_CACHE, "sequence %d has no entry in layer %d (all-masked row)", s, layer);
    ctx->bounds[i] = (int32_t)seq_block_bound(ctx, s);
  }
  return KVS_OK;
}
}  // namespace

namespace {
// accumulate checks: the layers of every sequence of the call agree on next_position;
// returns the largest block bound through *maxb.
kvs_status accumulate_bounds(kvs_ctx* ctx, int64_t* maxb) {
  const int B = ctx->cfg.max_seqs;
  *maxb = 1;
  for (const int32_t s : ctx->sids) {
    const int64_t n0 = ctx->next[s];
    for (int l = 1; l < ctx->cfg.num_layers; ++l)
      if (ctx->next[(size_t)l * B + s] != n0)
        return fail(ctx, KVS_ERR_STATE, "sequence %d: layers disagree on next_position", s);
    *maxb = std::max(*maxb, seq_block_bound(ctx, s));
  }
  return KVS_OK;
}

kvs_status check_select_args(kvs_ctx* ctx, int32_t score_kind, uint32_t flags, const int32_t* d_k_per_seq,
                             int32_t k_uniform, const int32_t* d_keep_ids, int32_t keep_capacity,
                             const int32_t* d_keep_count) {
  if (score_kind < KVS_SCORE_CUMULATIVE || score_kind > KVS_SCORE_TOVA)
    return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "score_kind must be CUMULATIVE, EMA, TOKEN_SUM or TOVA");
  if (flags & ~(KVS_SELECT_PROTECT | KVS_SELECT_APPLY)) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "unknown flags");
  if ((flags & KVS_SELECT_APPLY) && ctx->plan.mode != KVS_MODE_H2O)
    return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "eviction (KVS_SELECT_APPLY) needs the H2O mode");
  if (!d_k_per_seq && k_uniform < 0) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "k must be >= 0");
  if (!d_keep_ids || !d_keep_count || keep_capacity < 1)
    return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "keep buffers missing or keep_capacity < 1");
  return KVS_OK;
}

// After an eviction with a uniform k: kept <= max(k, protected blocks), protected <=
// sink blocks + recent blocks + 1.
void shrink_h2o_bounds(kvs_ctx* ctx, uint32_t flags, const int32_t* d_k_per_seq, int32_t k_uniform) {
  if (!(flags & KVS_SELECT_APPLY) || d_k_per_seq) return;
  const int64_t prot = cdiv64(ctx->cfg.h2o_sink_tokens, kBlock) + cdiv64(ctx->plan.recent_tokens, kBlock) + 1;
  const int64_t kept = std::max<int64_t>(k_uniform, (flags & KVS_SELECT_PROTECT) ? prot : 0);
  for (const int32_t s : ctx->sids) ctx->h2o_bound[s] = std::min(ctx->h2o_bound[s], kept);
}
}  // namespace

extern "C" {

void kvs_config_init(kvs_config* cfg) {
  Trace trace_("kvs_config_init");
  if (!cfg) return;
  std::memset(cfg, 0, sizeof *cfg);
  cfg->num_layers = 1;
  cfg->num_q_heads = 8;
  cfg->num_kv_heads = 1;
  cfg->head_dim = 128;
  cfg->max_seqs = 1;
  cfg->max_positions = 4096;
  cfg->block_tokens = kBlock;
  cfg->h2o_sink_tokens = 4;
  cfg->h2o_recent_frac = 0.25;
  cfg->ema_decay = 0.9;
  cfg->kv_dtype = KVS_BF16;
  cfg->in_dtype = KVS_BF16;
}

kvs_status kvs_validate_config(const kvs_config* cfg, char* msg, size_t msg_len) {
  Trace trace_("kvs_validate_config");
  return check_config(cfg, msg, msg_len);
}

size_t kvs_workspace_bytes(const kvs_config* cfg) {
  Trace trace_("kvs_workspace_bytes");
  if (check_config(cfg, nullptr, 0) != KVS_OK) return 0;
  Plan p;
  make_plan(cfg, &p);
  return p.total;
}

kvs_status kvs_create(const kvs_config* cfg, void* d_workspace, size_t workspace_bytes, kvs_stream_t stream,
                      kvs_ctx** out) {
  Trace trace_("kvs_create");
  if (!out) return KVS_ERR_INVALID_ARGUMENT;
  *out = nullptr;
  char msg[256];
  kvs_status st = check_config(cfg, msg, sizeof msg);
  if (st != KVS_OK) return st;
  Plan p;
  make_plan(cfg, &p);
  if (!d_workspace || (reinterpret_cast<uintptr_t>(d_workspace) & 255)) return KVS_ERR_INVALID_ARGUMENT;
  if (workspace_bytes < p.total) return KVS_ERR_CAPACITY;
  kvs_ctx* ctx = new (std::nothrow) kvs_ctx();
  if (!ctx) return KVS_ERR_CAPACITY;
  ctx->cfg = *cfg;
  ctx->plan = p;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaGetDevice(&ctx->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&ctx->sm_count, cudaDevAttrMultiProcessorCount, ctx->device) != cudaSuccess) {
    delete ctx;
    return KVS_ERR_CUDA;
  }
  uint8_t* w = static_cast<uint8_t*>(d_workspace);
  Dev& d = ctx->dev;
  std::memset(&d, 0, sizeof d);
  d.L = cfg->num_layers; d.Hq = cfg->num_q_heads; d.Hkv = cfg->num_kv_heads; d.D = cfg->head_dim;
  d.G = cfg->num_q_heads / cfg->num_kv_heads;
  d.max_seqs = cfg->max_seqs; d.max_positions = cfg->max_positions; d.max_blocks = p.max_blocks;
  d.window = cfg->window; d.mode = p.mode; d.num_pages = p.num_pages; d.pages_per_seq = p.pages_per_seq;
  d.kv_dtype = cfg->kv_dtype; d.in_dtype = cfg->in_dtype;
  d.spin_limit = cfg->spin_limit == 0 ? kDefaultSpin : cfg->spin_limit;
  d.h2o_sink_tokens = cfg->h2o_sink_tokens; d.h2o_recent_tokens = p.recent_tokens;
  d.ema_decay = cfg->ema_decay;
  const size_t slots = (size_t)p.num_pages * kBlock;
  d.k_pages = w + p.k_pages; d.v_pages = w + p.v_pages;
  d.page_layer_bytes = (size_t)p.num_pages * p.page_bytes; d.page_bytes = p.page_bytes;
  d.k_scales = cfg->kv_dtype == KVS_E4M3 ? reinterpret_cast<float*>(w + p.k_scales) : nullptr;
  d.v_scales = cfg->kv_dtype == KVS_E4M3 ? reinterpret_cast<float*>(w + p.v_scales) : nullptr;
  d.slot_layer_elems = slots;
  d.pos = reinterpret_cast<int64_t*>(w + p.pos);
  d.tok_mass = reinterpret_cast<float*>(w + p.tok_mass);
  d.blk_mass = reinterpret_cast<float*>(w + p.blk_mass);
  d.blk_layer_elems = (size_t)cfg->max_seqs * p.max_blocks;
  d.next_pos = reinterpret_cast<int64_t*>(w + p.next_pos);
  d.append_tickets = reinterpret_cast<int32_t*>(w + p.app_tickets);
  d.block_table = reinterpret_cast<int32_t*>(w + p.block_table);
  d.res_blocks = reinterpret_cast<int32_t*>(w + p.res_blocks);
  d.res_pages = reinterpret_cast<int32_t*>(w + p.res_pages);
  d.res_count = reinterpret_cast<int32_t*>(w + p.res_count);
  d.free_pages = reinterpret_cast<int32_t*>(w + p.free_pages);
  d.free_top = reinterpret_cast<int32_t*>(w + p.free_top);
  d.c_tok = reinterpret_cast<double*>(w + p.c_tok);
  d.e_tok = reinterpret_cast<double*>(w + p.e_tok);
  d.last_tok = reinterpret_cast<int32_t*>(w + p.last_tok);
  d.c_blk = reinterpret_cast<double*>(w + p.c_blk);
  d.e_blk = reinterpret_cast<double*>(w + p.e_blk);
  d.s_blk = reinterpret_cast<double*>(w + p.s_blk);
  d.t_blk = reinterpret_cast<double*>(w + p.t_blk);
  d.traj = reinterpret_cast<float*>(w + p.traj);
  d.traj_len = cfg->traj_len;
  d.prof = reinterpret_cast<double*>(w + p.prof);
  d.n_prof = 0;
  for (int l = 0; l < cfg->num_layers && l < 32; ++l)
    if (cfg->profile_layers >> l & 1u) d.prof_layer[d.n_prof++] = l;
  d.hstep = reinterpret_cast<float*>(w + p.hstep);
  d.hprof = reinterpret_cast<double*>(w + p.hprof);
  d.n_hprof = cfg->n_profile_heads;
  for (int j = 0; j < cfg->n_profile_heads; ++j) {
    d.hprof_layer[j] = cfg->profile_heads[j] >> 16;
    d.hprof_head[j] = cfg->profile_heads[j] & 0xffff;
  }
  d.last_blk = reinterpret_cast<int32_t*>(w + p.last_blk);
  d.steps = reinterpret_cast<int32_t*>(w + p.steps);
  d.acc_tickets = reinterpret_cast<int32_t*>(w + p.acc_tickets);
  d.partials = reinterpret_cast<float*>(w + p.partials);
  d.part_ml = reinterpret_cast<unsigned long long*>(w + p.part_ml);
  d.counters = reinterpret_cast<int32_t*>(w + p.counters);
  d.logit_scratch = reinterpret_cast<float*>(w + p.logits);
  d.logit_scratch_elems = p.logit_elems;
  d.err = reinterpret_cast<int32_t*>(w + p.err);
  d.ps_part = reinterpret_cast<float2*>(w + p.ps_part);
  d.ps_tok = reinterpret_cast<float*>(w + p.ps_tok);
  d.ps_blk = reinterpret_cast<float*>(w + p.ps_blk);
  d.ps_ready = reinterpret_cast<int32_t*>(w + p.ps_ready);
  d.ps_done = reinterpret_cast<int32_t*>(w + p.ps_done);
  d.ps_tickets = reinterpret_cast<int32_t*>(w + p.ps_tickets);
  d.ps_bound = p.ps_bound;

  const bool tc = tc_supported(cfg->num_q_heads, cfg->num_kv_heads, cfg->head_dim, cfg->kv_dtype, cfg->in_dtype,
                               cfg->window, p.mode);
  ctx->kernel = (cfg->kernel == KVS_KERNEL_GENERAL || !tc) ? KVS_KERNEL_GENERAL : KVS_KERNEL_TENSOR;
  if (ctx->kernel == KVS_KERNEL_TENSOR) {
    ctx->grid = tc_grid(cfg->kv_dtype, cfg->num_kv_heads, ctx->sm_count);
    if (ctx->grid < 1) {
      delete ctx;
      return KVS_ERR_CUDA;
    }
    ctx->maps.resize((size_t)cfg->num_layers * 2);
    for (int l = 0; l < cfg->num_layers; ++l) {
      if (make_page_map(&ctx->maps[2 * l], d.k_pages + l * d.page_layer_bytes, p.num_pages, d.Hkv, d.kv_dtype,
                        d.Hkv) != cudaSuccess ||
          make_page_map(&ctx->maps[2 * l + 1], d.v_pages + l * d.page_layer_bytes, p.num_pages, d.Hkv, d.kv_dtype,
                        d.Hkv) != cudaSuccess) {
        delete ctx;
        return KVS_ERR_CUDA;
      }
    }
    if (cfg->obs_window > 0 && cfg->kv_dtype == KVS_BF16) {
      ctx->ps_maps.resize((size_t)cfg->num_layers);
      for (int l = 0; l < cfg->num_layers; ++l)
        if (make_page_map(&ctx->ps_maps[l], d.k_pages + l * d.page_layer_bytes, p.num_pages, d.Hkv, d.kv_dtype, 1) !=
            cudaSuccess) {
          delete ctx;
          return KVS_ERR_CUDA;
        }
    }
  }
  ctx->next.assign((size_t)cfg->num_layers * cfg->max_seqs, 0);
  ctx->frontier.assign(cfg->max_seqs, 0);
  ctx->h2o_bound.assign(cfg->max_seqs, 0);
  if (cudaMemsetAsync(d_workspace, 0, p.total, s) != cudaSuccess || launch_init(d, s) != cudaSuccess) {
    delete ctx;
    return KVS_ERR_CUDA;
  }
#ifdef KVS_DEBUG
  // Debug builds fill every region that must be written before it is read with 0xFF
  // bytes (NaN as float, NaN pairs as (m, l) words): a read of a stale or never-written
  // element then shows up as a non-finite result.
  {
    const size_t regions[][2] = {{p.tok_mass, p.blk_mass}, {p.blk_mass, p.next_pos}, {p.hstep, p.hprof},
                                 {p.partials, p.counters}, {p.logits, p.ps_part}, {p.ps_part, p.ps_ready}};
    for (const auto& r : regions)
      if (r[1] > r[0] && cudaMemsetAsync(w + r[0], 0xFF, r[1] - r[0], s) != cudaSuccess) {
        delete ctx;
        return KVS_ERR_CUDA;
      }
  }
#endif
  *out = ctx;
  return KVS_OK;
}

kvs_status kvs_destroy(kvs_ctx* ctx) {
  Trace trace_("kvs_destroy");
  if (!ctx) return KVS_ERR_INVALID_ARGUMENT;
  delete ctx;
  return KVS_OK;
}

kvs_status kvs_reset(kvs_ctx* ctx, kvs_seqs seqs, kvs_stream_t stream) {
  Trace trace_("kvs_reset");
  if (!ctx) return KVS_ERR_INVALID_ARGUMENT;
  kvs_status st = check_seqs(ctx, seqs);
  if (st != KVS_OK) return st;
  st = cuda_ok(ctx, launch_reset(ctx->dev, sel_of(seqs), seqs.count, reinterpret_cast<cudaStream_t>(stream)), "reset");
  if (st != KVS_OK) return st;
  for (const int32_t s : ctx->sids) {
    for (int l = 0; l < ctx->cfg.num_layers; ++l) ctx->next[(size_t)l * ctx->cfg.max_seqs + s] = 0;
    ctx->frontier[s] = 0;
    ctx->h2o_bound[s] = 0;
  }
  return KVS_OK;
}

kvs_status kvs_append_kv(kvs_ctx* ctx, int32_t layer, kvs_seqs seqs, int32_t n_new, const void* d_k,
                         const void* d_v, kvs_stream_t stream) {
  Trace trace_("kvs_append_kv");
  if (!ctx) return KVS_ERR_INVALID_ARGUMENT;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "layer %d out of range", layer);
  kvs_status st = check_seqs(ctx, seqs);
  if (st != KVS_OK) return st;
  if (n_new < 1) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "n_new must be >= 1");
  if (!d_k || !d_v) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "NULL K or V");
  const int B = ctx->cfg.max_seqs;
  bool lead = false;
  for (const int32_t s : ctx->sids) {
    const int64_t nx = ctx->next[(size_t)layer * B + s];
    if (nx + n_new > ctx->cfg.max_positions)
      return fail(ctx, KVS_ERR_CAPACITY, "sequence %d: position %lld + %d exceeds max_positions %d", s,
                  (long long)nx, n_new, ctx->cfg.max_positions);
    if (nx + n_new > ctx->frontier[s]) lead = true;
  }
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (ctx->plan.mode == KVS_MODE_H2O && lead) {
    st = cuda_ok(ctx, launch_alloc_pages(ctx->dev, layer, sel_of(seqs), seqs.count, n_new, cs), "page allocation");
    if (st != KVS_OK) return st;
  }
  st = cuda_ok(ctx, launch_append(ctx->dev, layer, sel_of(seqs), seqs.count, n_new, d_k, d_v, cs), "append");
  if (st != KVS_OK) return st;
  for (const int32_t s : ctx->sids) {
    int64_t& nx = ctx->next[(size_t)layer * B + s];
    nx += n_new;
    if (nx > ctx->frontier[s]) {
      const int64_t new_blocks = cdiv64(nx, kBlock) - cdiv64(ctx->frontier[s], kBlock);
      ctx->h2o_bound[s] += new_blocks;
      ctx->frontier[s] = nx;
    }
  }
  return KVS_OK;
}


kvs_status kvs_decode_attend(kvs_ctx* ctx, int32_t layer, kvs_seqs seqs, const void* d_q, float* d_out,
                             float* d_tok_mass_opt, kvs_stream_t stream) {
  Trace trace_("kvs_decode_attend");
  if (!ctx) return KVS_ERR_INVALID_ARGUMENT;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "layer %d out of range", layer);
  kvs_status st = check_seqs(ctx, seqs);
  if (st != KVS_OK) return st;
  st = check_attend_buffers(ctx, d_q, d_out, d_tok_mass_opt);
  if (st != KVS_OK) return st;
  st = attend_bounds(ctx, layer);
  if (st != KVS_OK) return st;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  if (ctx->kernel == KVS_KERNEL_TENSOR) {
    AttendOpts opt;
    opt.tok_out = d_tok_mass_opt;
    st = cuda_ok(ctx, launch_attend_tc(ctx->maps[2 * layer], ctx->maps[2 * layer + 1], ctx->dev, layer, sel_of(seqs),
                                       seqs.count, d_q, d_out, ctx->bounds.data(), ctx->grid, opt, cs),
                 "tensor-core attend");
  } else {
    st = cuda_ok(ctx, launch_attend_general(ctx->dev, layer, sel_of(seqs), seqs.count, d_q, d_out, d_tok_mass_opt, cs),
                 "attend");
  }
  return st;
}

kvs_status kvs_append_attend(kvs_ctx* ctx, int32_t layer, kvs_seqs seqs, const void* d_k, const void* d_v,
                             const void* d_q, float* d_out, float* d_tok_mass_opt, kvs_stream_t stream) {
  Trace trace_("kvs_append_attend");
  if (!ctx) return KVS_ERR_INVALID_ARGUMENT;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "layer %d out of range", layer);
  kvs_status st = check_seqs(ctx, seqs);
  if (st != KVS_OK) return st;
  if (!d_k || !d_v) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "NULL K or V");
  st = check_attend_buffers(ctx, d_q, d_out, d_tok_mass_opt);
  if (st != KVS_OK) return st;
  if (ctx->kernel == KVS_KERNEL_TENSOR) {
    const int B = ctx->cfg.max_seqs;
    ctx->bounds.resize(ctx->sids.size());
    bool lead = false;
    for (size_t i = 0; i < ctx->sids.size(); ++i) {
      const int32_t s = ctx->sids[i];
      const int64_t nx = ctx->next[(size_t)layer * B + s];
      if (nx + 1 > ctx->cfg.max_positions)
        return fail(ctx, KVS_ERR_CAPACITY, "sequence %d: position %lld + 1 exceeds max_positions %d", s,
                    (long long)nx, ctx->cfg.max_positions);
      if (nx + 1 > ctx->frontier[s]) lead = true;
      // H2O: a block the new token opens is counted from the launch on
      const int64_t grow = (ctx->plan.mode == KVS_MODE_H2O && nx + 1 > ctx->frontier[s] && nx % kBlock == 0) ? 1 : 0;
      ctx->bounds[i] = (int32_t)std::min<int64_t>(ctx->plan.max_blocks, seq_block_bound(ctx, s) + grow);
    }
    if (ctx->plan.mode == KVS_MODE_H2O && lead) {
      // H2O: the pages of blocks the new tokens open come from the pool in a small
      // launch of their own first (the fused kernel appends into existing pages)
      st = cuda_ok(ctx, launch_alloc_pages(ctx->dev, layer, sel_of(seqs), seqs.count, 1,
                                           reinterpret_cast<cudaStream_t>(stream)),
                   "page allocation");
      if (st != KVS_OK) return st;
    }
    AttendOpts opt;
    opt.k_new = d_k;
    opt.v_new = d_v;
    opt.tok_out = d_tok_mass_opt;
    const cudaError_t e = launch_attend_tc(ctx->maps[2 * layer], ctx->maps[2 * layer + 1], ctx->dev, layer,
                                           sel_of(seqs), seqs.count, d_q, d_out, ctx->bounds.data(), ctx->grid, opt,
                                           reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaErrorNotSupported) {
      st = cuda_ok(ctx, e, "tensor-core append + attend");
      if (st != KVS_OK) return st;
      for (const int32_t s : ctx->sids) {          // the same shadow update as an append
        int64_t& nx = ctx->next[(size_t)layer * B + s];
        nx += 1;
        if (nx > ctx->frontier[s]) {
          ctx->h2o_bound[s] += cdiv64(nx, kBlock) - cdiv64(ctx->frontier[s], kBlock);
          ctx->frontier[s] = nx;
        }
      }
      return KVS_OK;
    }
  }
  // no single-launch form for this context or launch: the two steps, same results
  st = kvs_append_kv(ctx, layer, seqs, 1, d_k, d_v, stream);
  if (st != KVS_OK) return st;
  return kvs_decode_attend(ctx, layer, seqs, d_q, d_out, d_tok_mass_opt, stream);
}

kvs_status kvs_attend_blocks(kvs_ctx* ctx, int32_t layer, kvs_seqs seqs, const int32_t* d_block_ids,
                             int32_t ids_stride, const int32_t* d_block_count, const void* d_q, float* d_out,
                             kvs_stream_t stream) {
  Trace trace_("kvs_attend_blocks");
  if (!ctx) return KVS_ERR_INVALID_ARGUMENT;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "layer %d out of range", layer);
  kvs_status st = check_seqs(ctx, seqs);
  if (st != KVS_OK) return st;
  if (!d_block_ids || !d_block_count || ids_stride < 1)
    return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "block list missing or ids_stride < 1");
  st = check_attend_buffers(ctx, d_q, d_out, nullptr);
  if (st != KVS_OK) return st;
  if (ctx->kernel != KVS_KERNEL_TENSOR)
    return fail(ctx, KVS_ERR_UNSUPPORTED, "the block-list attend runs on the tensor-core attend only");
  st = attend_bounds(ctx, layer);
  if (st != KVS_OK) return st;
  for (auto& b : ctx->bounds) b = std::min<int32_t>(ids_stride, b);
  AttendOpts opt;
  opt.list_ids = d_block_ids;
  opt.list_count = d_block_count;
  opt.list_stride = ids_stride;
  st = cuda_ok(ctx, launch_attend_tc(ctx->maps[2 * layer], ctx->maps[2 * layer + 1], ctx->dev, layer, sel_of(seqs),
                                     seqs.count, d_q, d_out, ctx->bounds.data(), ctx->grid, opt,
                                     reinterpret_cast<cudaStream_t>(stream)),
               "tensor-core block-list attend");
  return st;
}

kvs_status kvs_prefill_score(kvs_ctx* ctx, int32_t layer, kvs_seqs seqs, const void* d_q_obs, int32_t n_obs,
                             kvs_stream_t stream) {
  Trace trace_("kvs_prefill_score");
  if (!ctx) return KVS_ERR_INVALID_ARGUMENT;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "layer %d out of range", layer);
  kvs_status st = check_seqs(ctx, seqs);
  if (st != KVS_OK) return st;
  if (ctx->cfg.obs_window == 0)
    return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "prefill scoring is off: create the context with obs_window > 0");
  if (n_obs < 1 || n_obs > ctx->cfg.obs_window)
    return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "n_obs must be in [1, obs_window = %d]", ctx->cfg.obs_window);
  if (!d_q_obs || (reinterpret_cast<uintptr_t>(d_q_obs) & 15))
    return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "q_obs must be a 16-byte aligned device pointer");
  const int B = ctx->cfg.max_seqs;
  for (const int32_t s : ctx->sids) {
    const int64_t nx = ctx->next[(size_t)layer * B + s];
    if (nx < n_obs)
      return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "sequence %d holds %lld entries in layer %d, fewer than n_obs", s,
                  (long long)nx, layer);
    if (ctx->plan.mode == KVS_MODE_WINDOW && n_obs > ctx->cfg.window)
      return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "n_obs exceeds the window");
  }
  // one CTA per SM; calls of more than kPsSeqMax sequences run as several launches
  const int grid = std::min(ctx->sm_count, kGridMax);
  st = cuda_ok(ctx, launch_prefill_score(ctx->dev, ctx->ps_maps.empty() ? nullptr : &ctx->ps_maps[layer], layer,
                                         sel_of(seqs), seqs.count, d_q_obs, n_obs, grid,
                                         reinterpret_cast<cudaStream_t>(stream)),
               "prefill score");
  return st;
}

kvs_status kvs_decode_attend_static_scratch(kvs_ctx* ctx, int32_t layer, kvs_seqs seqs, const void* d_q, float* d_out,
                                            float* d_tok_mass_opt, kvs_stream_t stream) {
  Trace trace_("kvs_decode_attend_static_scratch");
  if (!ctx) return KVS_ERR_INVALID_ARGUMENT;
  if (layer < 0 || layer >= ctx->cfg.num_layers) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "layer %d out of range", layer);
  kvs_status st = check_seqs(ctx, seqs);
  if (st != KVS_OK) return st;
  st = check_attend_buffers(ctx, d_q, d_out, d_tok_mass_opt);
  if (st != KVS_OK) return st;
  if (ctx->kernel != KVS_KERNEL_TENSOR)
    return fail(ctx, KVS_ERR_UNSUPPORTED, "the library-owned exchange area serves the tensor-core attend only");
  st = attend_bounds(ctx, layer);
  if (st != KVS_OK) return st;
  size_t off = 0;
  const size_t need = static_scratch_need(ctx->dev, seqs.count, ctx->grid, &off);
  if (need > static_scratch_limit())
    return fail(ctx, KVS_ERR_CAPACITY, "this launch needs %zu bytes of exchange area; the library array holds %zu",
                need, static_scratch_limit());
  const cudaError_t e = launch_attend_tc_static(ctx->maps[2 * layer], ctx->maps[2 * layer + 1], ctx->dev, layer,
                                                sel_of(seqs), seqs.count, d_q, d_out, d_tok_mass_opt,
                                                ctx->bounds.data(), ctx->grid, reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaErrorNotSupported)
    return fail(ctx, KVS_ERR_UNSUPPORTED, "the logits of this launch do not fit on chip");
  return cuda_ok(ctx, e, "tensor-core attend (library exchange area)");
}


kvs_status kvs_accumulate_scores(kvs_ctx* ctx, kvs_seqs seqs, kvs_stream_t stream) {
  Trace trace_("kvs_accumulate_scores");
  if (!ctx) return KVS_ERR_INVALID_ARGUMENT;
  kvs_status st = check_seqs(ctx, seqs);
  if (st != KVS_OK) return st;
  int64_t maxb = 1;
  st = accumulate_bounds(ctx, &maxb);
  if (st != KVS_OK) return st;
  st = cuda_ok(ctx, launch_accumulate(ctx->dev, sel_of(seqs), seqs.count, (int)maxb,
                                      reinterpret_cast<cudaStream_t>(stream)),
               "accumulate");
  return st;
}

kvs_status kvs_select_blocks(kvs_ctx* ctx, kvs_seqs seqs, const int32_t* d_k_per_seq, int32_t k_uniform,
                             int32_t score_kind, uint32_t flags, int32_t* d_keep_ids, int32_t keep_capacity,
                             int32_t* d_keep_count, kvs_stream_t stream) {
  Trace trace_("kvs_select_blocks");
  if (!ctx) return KVS_ERR_INVALID_ARGUMENT;
  kvs_status st = check_seqs(ctx, seqs);
  if (st != KVS_OK) return st;
  st = check_select_args(ctx, score_kind, flags, d_k_per_seq, k_uniform, d_keep_ids, keep_capacity, d_keep_count);
  if (st != KVS_OK) return st;
  st = cuda_ok(ctx, launch_select(ctx->dev, sel_of(seqs), seqs.count, d_k_per_seq, k_uniform, score_kind, flags,
                                  d_keep_ids, keep_capacity, d_keep_count, reinterpret_cast<cudaStream_t>(stream)),
               "select");
  if (st != KVS_OK) return st;
  shrink_h2o_bounds(ctx, flags, d_k_per_seq, k_uniform);
  return KVS_OK;
}

kvs_status kvs_accumulate_select(kvs_ctx* ctx, kvs_seqs seqs, const int32_t* d_k_per_seq, int32_t k_uniform,
                                 int32_t score_kind, uint32_t flags, int32_t* d_keep_ids, int32_t keep_capacity,
                                 int32_t* d_keep_count, kvs_stream_t stream) {
  Trace trace_("kvs_accumulate_select");
  if (!ctx) return KVS_ERR_INVALID_ARGUMENT;
  kvs_status st = check_seqs(ctx, seqs);
  if (st != KVS_OK) return st;
  st = check_select_args(ctx, score_kind, flags, d_k_per_seq, k_uniform, d_keep_ids, keep_capacity, d_keep_count);
  if (st != KVS_OK) return st;
  int64_t maxb = 1;
  st = accumulate_bounds(ctx, &maxb);
  if (st != KVS_OK) return st;
  if (maxb > accumulate_select_max_blocks()) {   // long sequences: the two kernels
    st = kvs_accumulate_scores(ctx, seqs, stream);
    if (st != KVS_OK) return st;
    return kvs_select_blocks(ctx, seqs, d_k_per_seq, k_uniform, score_kind, flags, d_keep_ids, keep_capacity,
                             d_keep_count, stream);
  }
  st = cuda_ok(ctx, launch_accumulate_select(ctx->dev, sel_of(seqs), seqs.count, (int)maxb, d_k_per_seq, k_uniform,
                                             score_kind, flags, d_keep_ids, keep_capacity, d_keep_count,
                                             reinterpret_cast<cudaStream_t>(stream)),
               "accumulate + select");
  if (st != KVS_OK) return st;
  shrink_h2o_bounds(ctx, flags, d_k_per_seq, k_uniform);
  return KVS_OK;
}

kvs_status kvs_filter_blocks(kvs_ctx* ctx, kvs_seqs seqs, int32_t score_kind, double theta, int32_t* d_ids,
                             int32_t capacity, int32_t* d_count, kvs_stream_t stream) {
  Trace trace_("kvs_filter_blocks");
  if (!ctx) return KVS_ERR_INVALID_ARGUMENT;
  kvs_status st = check_seqs(ctx, seqs);
  if (st != KVS_OK) return st;
  if (score_kind < KVS_SCORE_CUMULATIVE || score_kind > KVS_SCORE_TOVA)
    return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "score_kind must be CUMULATIVE, EMA, TOKEN_SUM or TOVA");
  if (theta != theta) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "theta is NaN");
  if (!d_ids || !d_count || capacity < 1)
    return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "output buffers missing or capacity < 1");
  st = cuda_ok(ctx, launch_filter(ctx->dev, sel_of(seqs), seqs.count, score_kind, theta, d_ids, capacity, d_count,
                                  reinterpret_cast<cudaStream_t>(stream)),
               "filter");
  return st;
}

size_t kvs_scores_snapshot_bytes(const kvs_ctx* ctx, int32_t n_seqs) {
  Trace trace_("kvs_scores_snapshot_bytes");
  if (!ctx || n_seqs < 0 || n_seqs > ctx->cfg.max_seqs) return 0;
  void* ptr[kSnapSections];
  size_t bytes[kSnapSections];
  const int ns = snapshot_sections(ctx, 0, n_seqs, ptr, bytes);
  size_t total = 0;
  for (int i = 0; i < ns; ++i) total += round256(bytes[i]);
  return total;
}

kvs_status kvs_export_scores(kvs_ctx* ctx, kvs_seqs seqs, void* dst, size_t dst_bytes, kvs_stream_t stream) {
  Trace trace_("kvs_export_scores");
  return snapshot_copy(ctx, seqs, dst, dst_bytes, true, stream);
}

kvs_status kvs_import_scores(kvs_ctx* ctx, kvs_seqs seqs, const void* src, size_t src_bytes, kvs_stream_t stream) {
  Trace trace_("kvs_import_scores");
  return snapshot_copy(ctx, seqs, const_cast<void*>(src), src_bytes, false, stream);
}

size_t kvs_state_bytes(const kvs_ctx* ctx, int32_t what) {
  Trace trace_("kvs_state_bytes");
  if (!ctx) return 0;
  const size_t slots = (size_t)ctx->plan.num_pages * kBlock, B = ctx->cfg.max_seqs, MB = ctx->plan.max_blocks;
  switch (what) {
    case KVS_STATE_K_PAGES: case KVS_STATE_V_PAGES: return (size_t)ctx->plan.num_pages * ctx->plan.page_bytes;
    case KVS_STATE_K_SCALES: case KVS_STATE_V_SCALES: return ctx->cfg.kv_dtype == KVS_E4M3 ? slots * 4 : 0;
    case KVS_STATE_POSITIONS: return slots * 8;
    case KVS_STATE_NEXT_POSITION: return B * 8;
    case KVS_STATE_TOKEN_MASS: return slots * 4;
    case KVS_STATE_BLOCK_MASS: return B * MB * 4;
    case KVS_STATE_C_TOKEN: case KVS_STATE_E_TOKEN: return B * ctx->cfg.max_positions * 8;
    case KVS_STATE_C_BLOCK: case KVS_STATE_E_BLOCK: case KVS_STATE_S_BLOCK: case KVS_STATE_T_BLOCK: return B * MB * 8;
    case KVS_STATE_STEPS: return B * 4;
    case KVS_STATE_BLOCK_TABLE: return B * MB * 4;
    case KVS_STATE_TRAJECTORY: return B * MB * (size_t)ctx->cfg.traj_len * 4;
    case KVS_STATE_LAYER_PROFILE: return B * MB * (size_t)ctx->dev.n_prof * 8;
    case KVS_STATE_HEAD_PROFILE: return B * MB * (size_t)ctx->dev.n_hprof * 8;
    default: return 0;
  }
}

kvs_status kvs_read_state(kvs_ctx* ctx, int32_t what, int32_t layer, void* d_dst, size_t dst_bytes,
                          kvs_stream_t stream) {
  Trace trace_("kvs_read_state");
  if (!ctx) return KVS_ERR_INVALID_ARGUMENT;
  const size_t n = kvs_state_bytes(ctx, what);
  if (n == 0) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "state item %d not available", what);
  if (!d_dst || dst_bytes < n) return fail(ctx, KVS_ERR_CAPACITY, "destination needs %zu bytes", n);
  if (layer < 0 || layer >= ctx->cfg.num_layers) return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "layer %d out of range", layer);
  const Dev& d = ctx->dev;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  const size_t slots = d.slot_layer_elems;
  const void* src = nullptr;
  switch (what) {
    case KVS_STATE_K_PAGES: src = d.k_pages + layer * d.page_layer_bytes; break;
    case KVS_STATE_V_PAGES: src = d.v_pages + layer * d.page_layer_bytes; break;
    case KVS_STATE_K_SCALES: src = d.k_scales + layer * slots; break;
    case KVS_STATE_V_SCALES: src = d.v_scales + layer * slots; break;
    case KVS_STATE_POSITIONS: src = d.pos + layer * slots; break;
    case KVS_STATE_NEXT_POSITION: src = d.next_pos + (size_t)layer * d.max_seqs; break;
    case KVS_STATE_TOKEN_MASS: src = d.tok_mass + layer * slots; break;
    case KVS_STATE_BLOCK_MASS: src = d.blk_mass + layer * d.blk_layer_elems; break;
    case KVS_STATE_C_TOKEN: src = d.c_tok; break;
    case KVS_STATE_C_BLOCK: src = d.c_blk; break;
    case KVS_STATE_S_BLOCK: src = d.s_blk; break;
    case KVS_STATE_STEPS: src = d.steps; break;
    case KVS_STATE_BLOCK_TABLE: src = d.block_table; break;
    case KVS_STATE_LAYER_PROFILE: src = d.prof; break;
    case KVS_STATE_HEAD_PROFILE: src = d.hprof; break;
    case KVS_STATE_TRAJECTORY:
      return cuda_ok(ctx, launch_read_trajectory(d, static_cast<float*>(d_dst), cs), "read trajectory");
    case KVS_STATE_E_TOKEN: case KVS_STATE_E_BLOCK: case KVS_STATE_T_BLOCK:
      return cuda_ok(ctx, launch_read_ema(d, what, static_cast<double*>(d_dst), cs), "read score");
    default: return fail(ctx, KVS_ERR_INVALID_ARGUMENT, "state item %d", what);
  }
  return cuda_ok(ctx, cudaMemcpyAsync(d_dst, src, n, cudaMemcpyDeviceToDevice, cs), "read state");
}

kvs_status kvs_get_layout(const kvs_ctx* ctx, kvs_layout* out) {
  Trace trace_("kvs_get_layout");
  if (!ctx || !out) return KVS_ERR_INVALID_ARGUMENT;
  std::memset(out, 0, sizeof *out);
  out->mode = ctx->plan.mode;
  out->num_pages = ctx->plan.num_pages;
  out->pages_per_seq = ctx->plan.pages_per_seq;
  out->max_blocks = ctx->plan.max_blocks;
  out->attend_kernel = ctx->kernel;
  out->attend_grid = ctx->grid;
  return KVS_OK;
}

kvs_status kvs_get_status(kvs_ctx* ctx, kvs_stream_t stream) {
  Trace trace_("kvs_get_status");
  if (!ctx) return KVS_ERR_INVALID_ARGUMENT;
  cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
  kvs_status st = cuda_ok(ctx, cudaStreamSynchronize(cs), "synchronise");
  if (st != KVS_OK) return st;
  int32_t e = 0;
  st = cuda_ok(ctx, cudaMemcpy(&e, ctx->dev.err, 4, cudaMemcpyDeviceToHost), "read error word");
  if (st != KVS_OK) return st;
  if (e & kErrTimeout) return fail(ctx, KVS_ERR_TIMEOUT, "a device-side wait ran out (error word 0x%x)", e);
  if (e & kErrCapacity) return fail(ctx, KVS_ERR_CAPACITY, "device capacity exhausted (error word 0x%x)", e);
  if (e & kErrState) return fail(ctx, KVS_ERR_STATE, "inconsistent device state (error word 0x%x)", e);
  if (e & kErrBounds)
    return fail(ctx, KVS_ERR_STATE, "a debug bounds check failed: an index read from device memory was out of "
                                    "range (error word 0x%x)", e);
  return KVS_OK;
}

kvs_status kvs_clear_error(kvs_ctx* ctx, kvs_stream_t stream) {
  Trace trace_("kvs_clear_error");
  if (!ctx) return KVS_ERR_INVALID_ARGUMENT;
  return cuda_ok(ctx, launch_clear(ctx->dev, reinterpret_cast<cudaStream_t>(stream)), "clear error");
}

const char* kvs_last_error(const kvs_ctx* ctx) { Trace trace_("kvs_last_error"); return ctx ? ctx->err.c_str() : ""; }

const char* kvs_status_string(kvs_status s) {
  Trace trace_("kvs_status_string");
  switch (s) {
    case KVS_OK: return "ok";
    case KVS_ERR_INVALID_ARGUMENT: return "invalid argument";
    case KVS_ERR_CAPACITY: return "capacity exceeded";
    case KVS_ERR_EMPTY_CACHE: return "empty cache (all-masked row)";
    case KVS_ERR_CUDA: return "CUDA error";
    case KVS_ERR_TIMEOUT: return "device wait timed out";
    case KVS_ERR_UNSUPPORTED: return "unsupported";
    case KVS_ERR_STATE: return "call order violated";
    default: return "unknown status";
  }
}

uint32_t kvs_build_info(void) {
  Trace trace_("kvs_build_info");
  uint32_t f = tracing_on() ? KVS_BUILD_TRACING : 0u;
#ifdef KVS_DEBUG
  f |= KVS_BUILD_DEBUG_CHECKS;
#endif
  return f;
}

int32_t kvs_abi_version(void) { Trace trace_("kvs_abi_version"); return KVS_ABI_VERSION; }

}  // extern "C"
