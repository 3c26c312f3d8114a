/*
 * kvs.h - C ABI of the attention-scored KV cache decode path (GB300, sm_103a).
 *
 * One decode step over a KV cache that also scores what it attends:
 *
 *   for every layer l:  kvs_append_kv     store the new token's K and V
 *                       kvs_decode_attend attend every query head over the resident
 *                                         entries, write the output, and turn the
 *                                         post-softmax weights into per-token and
 *                                         per-16-token-block masses on chip
 *   once per step:      kvs_accumulate_scores  cumulative + EMA score tables
 *                       kvs_select_blocks      top-k blocks to keep resident
 *
 * Sources (page title, then section):
 *   - Flash-MoE "Context Optimization": FP8 KV Cache > How It Works (E4M3 codes, one
 *     scale = absmax/240 per position, decoded inline during attention); Flag
 *     Ordering (the storage format is fixed before set-up); Sliding Window Attention >
 *     Design (circular slot = position % window); H2O KV Cache Eviction (sink, recent
 *     and heavy-hitter regions; score = post-softmax weights summed over all query
 *     heads and steps); H2O vs Sliding Window (H2O takes priority).
 *   - "Context views at marginal cost": Tier 1 (keep a running reduction - EMA and
 *     cumulative - never the attention matrix); Fact 3 (the QK^T, softmax, V read is
 *     the floor of the method).
 *   - "Per-Head Attention as a Scoring Signal": Fix: score per head, place per block
 *     (a block of 16 tokens stays if any head weights it).
 *   - "LLM mechanics III": sections 1, 3 and 5 (the window includes the current
 *     token; slots, absolute positions and the processed count are kept apart;
 *     invalid windows and all-masked rows are rejected).
 *
 * Conventions
 *   - Every call returns a kvs_status; nothing is thrown across the ABI.  Arguments
 *     are checked on the host before any launch; a call that fails a check launches
 *     nothing and leaves the state unchanged.  kvs_last_error() describes the last
 *     failure of a context.
 *   - Device memory is owned by the caller: kvs_create() takes a workspace of
 *     kvs_workspace_bytes() bytes and keeps non-owning pointers into it until
 *     kvs_destroy().  The library itself never allocates device memory.
 *   - Pointers named d_* are device pointers; h_* are host pointers.  Every launch
 *     goes on the stream given to the call (a cudaStream_t; 0 is the legacy default
 *     stream).  No call synchronises except kvs_get_status().
 *   - Device-side failures (capacity exhausted, a bounded wait that ran out) set an
 *     error word that kvs_get_status() reports and kvs_clear_error() resets.
 *   - The sequences of a call are a kvs_seqs: either a contiguous range of the
 *     max_seqs sequences the cache holds, or a list of distinct sequence ids in any
 *     order (a serving batch whose active sequences are scattered).  Per-sequence
 *     inputs and outputs are packed in the call's order: row i belongs to the i-th
 *     sequence of the range or list.
 *   - Call order per step: kvs_append_kv(l) before kvs_decode_attend(l) for every
 *     layer, kvs_accumulate_scores() after the last layer, then kvs_select_blocks().
 */
#ifndef KVS_H
#define KVS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define KVS_ABI_VERSION 2

#if defined(__GNUC__)
#define KVS_API __attribute__((visibility("default")))
#else
#define KVS_API
#endif

typedef struct kvs_ctx kvs_ctx;
typedef struct CUstream_st* kvs_stream_t;   /* a cudaStream_t */

/* The sequences one call works on.
 *   Range form (h_ids == NULL, d_ids == NULL): sequences begin .. begin + count - 1.
 *   List form (both non-NULL, begin ignored): the `count` sequence ids h_ids[0..count)
 *     in host memory and the same ids, in the same order, in device memory at d_ids.
 *     The library reads h_ids during the call (argument checks, its per-sequence
 *     host bookkeeping and launch plans, so no call has to read device memory); the
 *     kernels it launches read d_ids, which must stay valid until they have run.  The
 *     ids must be distinct and in [0, max_seqs); a list with a bad or repeated id is
 *     rejected (KVS_ERR_INVALID_ARGUMENT) and launches nothing.  The two copies must
 *     hold the same ids: the library cannot check d_ids without a device read.
 * count >= 1 in both forms. */
typedef struct {
  int32_t begin;
  int32_t count;
  const int32_t* h_ids;
  const int32_t* d_ids;
} kvs_seqs;

static inline kvs_seqs kvs_seq_range(int32_t begin, int32_t count) {
  kvs_seqs r;
  r.begin = begin;
  r.count = count;
  r.h_ids = 0;
  r.d_ids = 0;
  return r;
}

static inline kvs_seqs kvs_seq_list(int32_t count, const int32_t* h_ids, const int32_t* d_ids) {
  kvs_seqs r;
  r.begin = 0;
  r.count = count;
  r.h_ids = h_ids;
  r.d_ids = d_ids;
  return r;
}

typedef enum {
  KVS_OK = 0,
  KVS_ERR_INVALID_ARGUMENT = 1, /* a bad pointer, size, id, window or config field */
  KVS_ERR_CAPACITY = 2,         /* positions, pages or an output buffer would overflow */
  KVS_ERR_EMPTY_CACHE = 3,      /* attend with no resident entry: an all-masked row */
  KVS_ERR_CUDA = 4,             /* a CUDA runtime call failed */
  KVS_ERR_TIMEOUT = 5,          /* a device-side bounded wait ran out */
  KVS_ERR_UNSUPPORTED = 6,      /* shape or format not covered by any kernel */
  KVS_ERR_STATE = 7             /* call order violated (e.g. layers disagree) */
} kvs_status;

typedef enum { KVS_F32 = 0, KVS_BF16 = 1, KVS_E4M3 = 2 } kvs_dtype;

/* Block scores a selection can rank by ("Per-Head Attention as a Scoring Signal",
 * Combined placement decision; "Context views at marginal cost", per-system
 * reductions):
 *   CUMULATIVE  sum over steps of the block mass (max over layers and heads of the
 *               in-block weight sum)
 *   EMA         its exponential moving average
 *   TOKEN_SUM   H2O: sum over steps of the entry scores (weights summed over heads and
 *               layers) summed over the block's entries
 *   TOVA        the latest step's entry scores summed over the block's entries (the
 *               latest query's weight; keeping the top k evicts the argmin blocks) */
typedef enum { KVS_SCORE_CUMULATIVE = 0, KVS_SCORE_EMA = 1, KVS_SCORE_TOKEN_SUM = 2,
               KVS_SCORE_TOVA = 3 } kvs_score_kind;

/* Attend kernel choice: AUTO takes the tensor-core kernel when the shape allows it
 * (head_dim 128, 8 query heads per KV head, bf16 inputs, bf16 or E4M3 storage, and
 * a window that is 0 or a multiple of 16), else the general CUDA-core kernel. */
typedef enum { KVS_KERNEL_AUTO = 0, KVS_KERNEL_GENERAL = 1, KVS_KERNEL_TENSOR = 2 } kvs_kernel;

/* Residency mode, derived from the config: H2O when h2o_budget_tokens > 0 (it takes
 * priority over a window), else WINDOW when window > 0, else NONE. */
typedef enum { KVS_MODE_NONE = 0, KVS_MODE_WINDOW = 1, KVS_MODE_H2O = 2 } kvs_mode;

typedef struct {
  int32_t num_layers;        /* >= 1 */
  int32_t num_q_heads;       /* Hq, a multiple of num_kv_heads */
  int32_t num_kv_heads;      /* Hkv; query head h reads KV head h / (Hq / Hkv) */
  int32_t head_dim;          /* D in {16, 32, 64, 128} */
  int32_t max_seqs;          /* sequences held */
  int32_t max_positions;     /* absolute-position capacity of each sequence */
  int32_t window;            /* 0 = none; else >= 1 positions, the current one included */
  int32_t block_tokens;      /* 16 (the only value supported) */
  int32_t h2o_budget_tokens; /* 0 = off; else the resident budget (a multiple of 16) */
  int32_t h2o_sink_tokens;   /* H2O: always keep the blocks of the first N tokens (4) */
  int32_t num_pages;         /* H2O page pool (0 = max_seqs * ceil(max_positions/16)) */
  int32_t kernel;            /* a kvs_kernel */
  int32_t spin_limit;        /* device wait polls: 0 = default (~0.5 s), > 0 = that many, -1 = no poll
                                (a CTA that is not the last to arrive reports KVS_ERR_TIMEOUT) */
  int32_t kv_dtype;          /* storage: KVS_F32, KVS_BF16 or KVS_E4M3 */
  int32_t in_dtype;          /* dtype of Q, K, V inputs: KVS_F32 or KVS_BF16 */
  int32_t traj_len;          /* side-car trajectory ring: the last N steps' TOVA block score
                                per block (0 = off, at most 256) */
  uint32_t profile_layers;   /* side-car layer profiles: bit l set = keep, per block, the
                                sum over steps of layer l's block mass (at most 4 bits) */
  int32_t obs_window;        /* SnapKV prefill scoring: the most observation queries one
                                kvs_prefill_score call takes (1..32); 0 = off */
  int32_t n_profile_heads;   /* side-car per-head profiles: 0..4 profiled query heads */
  int32_t profile_heads[4];  /* each layer * 65536 + query head: keep, per block, the sum over
                                steps of that head's in-block weight in that layer */
  int32_t reserved_i;        /* must be 0 */
  double  h2o_recent_frac;   /* H2O: always keep the last frac * budget tokens (0.25) */
  double  ema_decay;         /* d in E <- d*E + (1-d)*x, in [0, 1) (0.9) */
  double  reserved_d[2];     /* must be 0 */
} kvs_config;

/* Fill *cfg with defaults (block 16, sinks 4, recent 0.25, decay 0.9, bf16). */
KVS_API void kvs_config_init(kvs_config* cfg);

/* Check a config without touching the GPU.  On failure writes a message into msg
 * (if msg_len > 0) and returns KVS_ERR_INVALID_ARGUMENT or KVS_ERR_UNSUPPORTED. */
KVS_API kvs_status kvs_validate_config(const kvs_config* cfg, char* msg, size_t msg_len);

/* Workspace bytes a config needs (0 if the config is invalid).  Host-only. */
KVS_API size_t kvs_workspace_bytes(const kvs_config* cfg);

/* Bind a context to a caller-owned device workspace of at least
 * kvs_workspace_bytes(cfg) bytes (256-byte aligned) on the current device and
 * initialise it (on `stream`).  The config is copied and fixed for the context's
 * life: the storage format decides the workspace layout.  *out receives the
 * context (a host object; free it with kvs_destroy). */
KVS_API kvs_status kvs_create(const kvs_config* cfg, void* d_workspace, size_t workspace_bytes,
                      kvs_stream_t stream, kvs_ctx** out);

/* Free the host object.  The workspace stays the caller's. */
KVS_API kvs_status kvs_destroy(kvs_ctx* ctx);

/* Empty the sequences of `seqs`: next_position = 0 in every layer, score tables
 * zeroed, H2O pages returned to the pool ("LLM mechanics III" §5: the processed count
 * and the positions restart only when a sequence starts over). */
KVS_API kvs_status kvs_reset(kvs_ctx* ctx, kvs_seqs seqs, kvs_stream_t stream);

/* Append n_new tokens to every sequence of `seqs` in layer `layer` (Flash-MoE "Context
 * Optimization", FP8 KV Cache > How It Works, Encoding; Sliding Window Attention >
 * Design; "LLM mechanics III" §1 and §5: absolute positions kept apart from slots).
 * d_k, d_v: [seqs.count][n_new][num_kv_heads][head_dim] in in_dtype, device memory.
 * Token i of sequence s goes to absolute position next_position[layer][s] + i.
 * E4M3 storage quantises each position (all KV heads of one of K or V) with
 * scale = fl32(absmax / 240) and round-to-nearest-even saturating E4M3 codes of
 * fl32(x / scale); absmax 0 gives scale 0 and zero codes.
 * Window mode writes position p to slot p % window; H2O mode writes it to the page
 * of block p / 16.  Errors: KVS_ERR_CAPACITY if a sequence would pass
 * max_positions (or, on the device, if the H2O page pool is empty). */
KVS_API kvs_status kvs_append_kv(kvs_ctx* ctx, int32_t layer, kvs_seqs seqs, int32_t n_new, const void* d_k,
                                 const void* d_v, kvs_stream_t stream);

/* Decode attention of one query per head over the resident entries of layer `layer`
 * ("Context views at marginal cost", §7 Fact 3: the QK^T, softmax, V read; Flash-MoE
 * "Context Optimization", FP8 KV Cache > How It Works, Decoding: E4M3 decoded inline;
 * H2O KV Cache Eviction > How It Works in Flash-MoE, step 1: the post-softmax weights
 * summed across all query heads; "Per-Head Attention as a Scoring Signal", Fix: score
 * per head, place per block).
 * d_q: [seqs.count][num_q_heads][head_dim] in in_dtype; d_out: [seqs.count]
 * [num_q_heads][head_dim] float32, both device memory aligned to 16 bytes.  Logits
 * are q.k/sqrt(D) (k, v decoded inline from E4M3 as code * scale), softmax per head
 * over the resident entries; query head h reads KV head h / (Hq / Hkv).
 * In the same launch, without writing the weights anywhere off chip, the kernel
 * stores the step masses of this layer: per resident entry the sum over query heads
 * of its weight, and per resident 16-token block the maximum over query heads of
 * the head's summed weight in the block (both readable with kvs_read_state).
 * d_tok_mass_opt: NULL, or device float32 [seqs.count][max_positions] that also
 * receives each resident entry's mass at its absolute position (row i for the i-th
 * sequence of the call; elements of positions not resident are left as they were).
 * Errors: KVS_ERR_EMPTY_CACHE if a sequence of the call has no resident entry;
 * KVS_ERR_INVALID_ARGUMENT if d_q or d_out is NULL or not 16-byte aligned, or
 * d_tok_mass_opt is not 4-byte aligned. */
KVS_API kvs_status kvs_decode_attend(kvs_ctx* ctx, int32_t layer, kvs_seqs seqs, const void* d_q, float* d_out,
                                     float* d_tok_mass_opt, kvs_stream_t stream);

/* One decode step of one layer in one call: kvs_append_kv of one new token per
 * sequence (d_k, d_v: [seqs.count][1][num_kv_heads][head_dim] in in_dtype), then
 * kvs_decode_attend (d_q, d_out, d_tok_mass_opt as there).  No page counterpart as a single step: the
 * pages append the decode token and attend over the cache including it, and this call
 * does both.  With the tensor-core attend in NONE or WINDOW mode, and when every
 * sequence of the range can have CTAs of its own, it is one kernel launch.  The CTA
 * holding a sequence's newest block stores the token (the same bytes the append
 * kernel stores) while the others stream, and the sequence's next_position advances
 * when its last CTA leaves.  Otherwise it issues the two calls.  Same results, state
 * and errors as the two calls.  If the launch reports KVS_ERR_TIMEOUT, the token may
 * be stored without next_position having advanced: append it again after
 * kvs_clear_error. */
KVS_API kvs_status kvs_append_attend(kvs_ctx* ctx, int32_t layer, kvs_seqs seqs, const void* d_k,
                                     const void* d_v, const void* d_q, float* d_out, float* d_tok_mass_opt,
                                     kvs_stream_t stream);

/* Tier-2 re-attend ("Context views at marginal cost", Tier 2 and Fact 3): decode
 * attention of one query per head over the cached K and V of a selected subset only.
 * The subset is the resident entries of the listed blocks, for example the keep_ids
 * that kvs_select_blocks returns.  d_block_ids: [seqs.count][ids_stride] int32 block
 * ids (each listed once); d_block_count: [seqs.count] int32, the first count entries of a row
 * are used (clamped to [0, ids_stride]); both device memory.  d_q, d_out as in
 * kvs_decode_attend.  Softmax over the subset; no mass or score is written.  Listed
 * blocks must be resident: with every listed entry outside the resident range the
 * row has no entry and its output is not finite.  A block id out of range, or (H2O)
 * not resident, is reported as KVS_ERR_STATE by kvs_get_status and its entries are
 * left out.
 * Errors: KVS_ERR_UNSUPPORTED unless the context uses the tensor-core attend;
 * KVS_ERR_EMPTY_CACHE as kvs_decode_attend; KVS_ERR_INVALID_ARGUMENT for missing
 * buffers, ids_stride < 1 or unaligned q / out. */
KVS_API kvs_status kvs_attend_blocks(kvs_ctx* ctx, int32_t layer, kvs_seqs seqs, const int32_t* d_block_ids,
                                     int32_t ids_stride, const int32_t* d_block_count, const void* d_q,
                                     float* d_out, kvs_stream_t stream);

/* kvs_decode_attend without any exchange area from the caller.  No page counterpart:
 * this is a deployment variant, not a step of the method.
 *
 * The tensor-core attend needs a per-launch exchange area (one softmax partial per
 * CTA and sequence, three counters per sequence: output arrivals, statistics arrivals
 * and departures).  kvs_decode_attend keeps it in
 * the context's workspace.  This entry point instead uses one fixed array of 8 MiB
 * compiled into the library (a __device__ array each GPU that loads the library holds
 * until the process exits), so the call itself needs no device memory beyond the
 * cache it reads and the q / out buffers it is given.  It is for callers that cannot
 * obtain device memory when they run a decode step: a runtime whose device memory is
 * parcelled out once at start-up by a supervisor, code that must not enter the CUDA
 * allocator (which can synchronise the device and fail under memory pressure), or a
 * caller that wants to hand the library nothing but its inputs and outputs.
 *
 * Same arguments, same results and same errors as kvs_decode_attend, plus:
 *   KVS_ERR_UNSUPPORTED  the context does not use the tensor-core attend, or this
 *                        launch's logits do not fit in shared memory;
 *   KVS_ERR_CAPACITY     the launch needs more than the array holds:
 *                        (grid + seqs.count) * num_q_heads * head_dim * 4
 *                        bytes, rounded up to 256, plus (grid + seqs.count) *
 *                        num_q_heads * 8
 *                        rounded up to 256, plus 384 * max_seqs bytes must be
 *                        <= 8 MiB.
 * The array is shared by every call of every context on the device and keeps the last
 * call's contents; the counters are cleared on `stream` before each launch.  Two such
 * launches that overlap on the GPU (different streams or contexts) race on the array:
 * order them.  The first call on a device looks up the array's device address (a
 * host-side API call, done once per device); make that first call before any stream
 * capture. */
KVS_API kvs_status kvs_decode_attend_static_scratch(kvs_ctx* ctx, int32_t layer, kvs_seqs seqs, const void* d_q,
                                                    float* d_out, float* d_tok_mass_opt, kvs_stream_t stream);

/* SnapKV prefill scoring ("Context views at marginal cost", the per-system
 * reductions: observation window of the prompt's last queries, votes pooled per token
 * and head, max-pool kernel 7).  Call it for a layer once its prompt is appended, in
 * place of the attend of a decode step; kvs_accumulate_scores after the last layer
 * then folds the result into the tables as their first step.
 * d_q_obs: [seqs.count][n_obs][num_q_heads][head_dim] bf16 (device, 16-byte aligned), the
 * queries of the last n_obs positions of each sequence's prompt, oldest first.  Query
 * i, at position next_position - n_obs + i, attends over the resident entries at
 * positions <= its own: logits q.k/sqrt(D), softmax per head.  An entry's vote for
 * head h sums the weights of the n_obs queries of head h.  The votes are max-pooled:
 * at each resident position, the largest vote among the resident positions within 3
 * of it.  The pooled votes replace the layer's step masses: the entry mass is their
 * sum over heads, and the block mass the max over heads of the in-block sum.  E4M3
 * caches convert the bf16 queries to f16 (exact in f16's normal range), as the
 * decode attend does.
 * Needs a context created with obs_window >= n_obs (tensor-core configurations
 * only).  One cooperative kernel launch (a CTA per SM) per 512 sequences of the call:
 * a larger call runs as several launches, in order on the stream.  Errors:
 * KVS_ERR_INVALID_ARGUMENT for n_obs outside [1, obs_window], a sequence holding fewer
 * than n_obs entries, or (window mode) n_obs > window. */
KVS_API kvs_status kvs_prefill_score(kvs_ctx* ctx, int32_t layer, kvs_seqs seqs, const void* d_q_obs,
                                     int32_t n_obs, kvs_stream_t stream);

/* Fold this step's masses of every layer into the score tables of the sequences of
 * `seqs` ("Context views at marginal cost", Tier 1: EMA and Cumulative as running
 * reductions, O(1) per span per step; Flash-MoE "Context Optimization", H2O KV Cache
 * Eviction > How It Works in Flash-MoE, step 1: the scores accumulate over all steps;
 * "Per-Head Attention as a Scoring Signal", Combined placement decision: a block
 * scores as its best head):
 * token score x_p = sum over layers of the entry masses, block score y_k = max over
 * layers of the block masses; for every tracked entry (every position below
 * next_position and every block holding one) C += x and E <- d*E + (1-d)*x, x = 0
 * where nothing was attended this step.  Errors: KVS_ERR_STATE if the layers of a
 * sequence disagree on next_position. */
KVS_API kvs_status kvs_accumulate_scores(kvs_ctx* ctx, kvs_seqs seqs, kvs_stream_t stream);

#define KVS_SELECT_PROTECT 1u  /* H2O: keep the sink and recent blocks first */
#define KVS_SELECT_APPLY   2u  /* H2O: evict the unkept blocks (pages back to the pool) */

/* Top-budget block selection ("Per-Head Attention as a Scoring Signal", worked 128K
 * example: the highest-scoring blocks stay resident; Flash-MoE "Context Optimization",
 * H2O KV Cache Eviction > The Algorithm: sink, recent and heavy-hitter regions).
 * Per sequence of `seqs`, keep the k resident blocks with the highest score
 * (C or E, a kvs_score_kind), ties to the lower block id; all are kept when k >= the
 * resident count.  With KVS_SELECT_PROTECT the blocks holding a sink token (position
 * < h2o_sink_tokens) or a recent token (position >= next_position - ceil(recent_frac
 * * budget)) are kept whatever their score and the rest of k is filled by score; if
 * they alone exceed k, all of them are kept.  k comes from d_k_per_seq ([seqs.count]
 * int32, device) or, when d_k_per_seq is NULL, from k_uniform for every sequence.
 * d_keep_ids: [seqs.count][keep_capacity] int32 (device), ascending block ids;
 * d_keep_count: [seqs.count] int32 (device), the number kept (ids beyond keep_capacity
 * are dropped and flag KVS_ERR_CAPACITY on the device).
 * Errors: KVS_ERR_INVALID_ARGUMENT for APPLY outside H2O mode or a negative k. */
KVS_API kvs_status kvs_select_blocks(kvs_ctx* ctx, kvs_seqs seqs, const int32_t* d_k_per_seq, int32_t k_uniform, int32_t score_kind,
                             uint32_t flags, int32_t* d_keep_ids, int32_t keep_capacity,
                             int32_t* d_keep_count, kvs_stream_t stream);

/* kvs_accumulate_scores followed by kvs_select_blocks (same arguments as the latter),
 * in one launch when every sequence of the call has at most 512 resident blocks.
 * There is no page counterpart as a single step: the pages fold a step's weights into
 * the scores and then pick the blocks to keep, and this call does both.  The tables
 * are updated exactly as the accumulate kernel does, on its grid.  The last CTA of
 * each sequence to finish ranks the blocks just scored: rank = keys above + equal keys
 * with a lower id, which keeps the same set as the radix select.  It then compacts the
 * kept ids in id order.  Longer sequences: the two calls.  Same results, state and
 * errors as the two calls. */
KVS_API kvs_status kvs_accumulate_select(kvs_ctx* ctx, kvs_seqs seqs, const int32_t* d_k_per_seq, int32_t k_uniform, int32_t score_kind,
                                 uint32_t flags, int32_t* d_keep_ids, int32_t keep_capacity,
                                 int32_t* d_keep_count, kvs_stream_t stream);

/* Threshold view ("Context views at marginal cost", Tier 1: a view is a filter of the
 * kept score table, a_s > theta): per sequence of `seqs`, the resident blocks whose
 * block score (a kvs_score_kind, read as kvs_select_blocks reads it) is strictly
 * greater than theta, in ascending id.  d_ids: [seqs.count][capacity] int32 (device);
 * d_count: [seqs.count] int32 (device), the number that passed (ids beyond capacity are
 * dropped and flag KVS_ERR_CAPACITY on the device).  Reads the tables only.
 * Errors: KVS_ERR_INVALID_ARGUMENT for an unknown score kind, a NaN theta or missing
 * buffers. */
KVS_API kvs_status kvs_filter_blocks(kvs_ctx* ctx, kvs_seqs seqs, int32_t score_kind, double theta, int32_t* d_ids, int32_t capacity, int32_t* d_count,
                                     kvs_stream_t stream);

/* Score snapshot (the side-car kept next to the session's KV: "Context views at
 * marginal cost", Tier 1).  Export copies, for the sequences of `seqs` in the call's
 * order, every score table (token and block cumulative, EMA and update stamps,
 * token-sum and TOVA block scores, the trajectory ring, the layer and head profiles) and the
 * step counts into one buffer; import copies such a buffer back into as many
 * sequences (any range or list of the same count).  The
 * buffer is raw and carries no header: it can be imported only into a context created
 * with the same max_positions, traj_len, profile_layers and n_profile_heads (the KV entries and the
 * residency are not part of it).  The buffer may be device memory or host memory
 * (pinned memory keeps the copies asynchronous); it must hold
 * kvs_scores_snapshot_bytes(ctx, seqs.count) bytes.  One cudaMemcpyAsync per table on
 * `stream` (range form) or per table and sequence (list form).  Errors: KVS_ERR_CAPACITY for a short buffer. */
KVS_API size_t kvs_scores_snapshot_bytes(const kvs_ctx* ctx, int32_t n_seqs);
KVS_API kvs_status kvs_export_scores(kvs_ctx* ctx, kvs_seqs seqs, void* dst, size_t dst_bytes,
                                     kvs_stream_t stream);
KVS_API kvs_status kvs_import_scores(kvs_ctx* ctx, kvs_seqs seqs, const void* src, size_t src_bytes,
                                     kvs_stream_t stream);

/* State read-back (tests, inspection).  Copies one array of `layer` (ignored for
 * per-sequence items) into d_dst (device), which must hold kvs_state_bytes(). */
typedef enum {
  KVS_STATE_K_PAGES = 0,     /* [num_pages][Hkv][16][D] storage elements of K */
  KVS_STATE_V_PAGES = 1,     /* same for V */
  KVS_STATE_K_SCALES = 2,    /* [num_pages][16] float32 (E4M3 only) */
  KVS_STATE_V_SCALES = 3,
  KVS_STATE_POSITIONS = 4,   /* [num_pages][16] int64 absolute position per slot, -1 empty */
  KVS_STATE_NEXT_POSITION = 5, /* [max_seqs] int64 */
  KVS_STATE_TOKEN_MASS = 6,  /* [num_pages][16] float32 entry masses of the last attend */
  KVS_STATE_BLOCK_MASS = 7,  /* [max_seqs][max_blocks] float32 block masses of the last attend */
  KVS_STATE_C_TOKEN = 8,     /* [max_seqs][max_positions] float64 cumulative */
  KVS_STATE_E_TOKEN = 9,     /* [max_seqs][max_positions] float64 EMA, as of the last step */
  KVS_STATE_C_BLOCK = 10,    /* [max_seqs][max_blocks] float64 */
  KVS_STATE_E_BLOCK = 11,
  KVS_STATE_STEPS = 12,      /* [max_seqs] int32 accumulate steps done */
  KVS_STATE_BLOCK_TABLE = 13,/* [max_seqs][max_blocks] int32 page of each block, -1 = none */
  KVS_STATE_S_BLOCK = 14,    /* [max_seqs][max_blocks] float64 TOKEN_SUM block score */
  KVS_STATE_T_BLOCK = 15,    /* [max_seqs][max_blocks] float64 TOVA block score of the last step */
  KVS_STATE_TRAJECTORY = 16, /* [max_seqs][max_blocks][traj_len] float32, oldest step first,
                                0 where the block was not updated (traj_len > 0) */
  KVS_STATE_LAYER_PROFILE = 17, /* [max_seqs][max_blocks][profiled layers, ascending] float64 */
  KVS_STATE_HEAD_PROFILE = 18,  /* [max_seqs][max_blocks][n_profile_heads] float64, in
                                   profile_heads order */
  KVS_STATE_COUNT = 19
} kvs_state_item;

KVS_API size_t kvs_state_bytes(const kvs_ctx* ctx, int32_t what);
KVS_API kvs_status kvs_read_state(kvs_ctx* ctx, int32_t what, int32_t layer, void* d_dst, size_t dst_bytes,
                          kvs_stream_t stream);

/* Layout facts: the page of (sequence s, position p) is
 *   NONE:   s * pages_per_seq + p / 16                slot p % 16
 *   WINDOW: s * pages_per_seq + (p % window) / 16     slot (p % window) % 16
 *   H2O:    block_table[s][p / 16]                    slot p % 16          */
typedef struct {
  int32_t mode;              /* a kvs_mode */
  int32_t num_pages;
  int32_t pages_per_seq;     /* NONE and WINDOW modes */
  int32_t max_blocks;        /* ceil(max_positions / 16) */
  int32_t attend_kernel;     /* kvs_kernel the attend launches use */
  int32_t attend_grid;       /* CTAs of one tensor-core attend launch (persistent) */
  int32_t reserved[2];
} kvs_layout;

KVS_API kvs_status kvs_get_layout(const kvs_ctx* ctx, kvs_layout* out);

/* Synchronise `stream` and report the device error word (KVS_OK if clear). */
KVS_API kvs_status kvs_get_status(kvs_ctx* ctx, kvs_stream_t stream);

/* Clear the device error word and the attend arrival counters (after a timeout). */
KVS_API kvs_status kvs_clear_error(kvs_ctx* ctx, kvs_stream_t stream);

/* Message of the last failed call on ctx ("" if none); never NULL. */
KVS_API const char* kvs_last_error(const kvs_ctx* ctx);

KVS_API const char* kvs_status_string(kvs_status s);

KVS_API int32_t kvs_abi_version(void);

#define KVS_BUILD_DEBUG_CHECKS 1u  /* built with KVS_DEBUG: device-side bounds checks that
                                      record KVS_ERR_STATE instead of touching memory out of
                                      range, and scratch poisoned with NaN at kvs_create */
#define KVS_BUILD_TRACING      2u  /* NVTX ranges around every call (environment variable
                                      KVS_NVTX set to anything but "0") */
/* How this library was built and what it emits (KVS_BUILD_* bits). */
KVS_API uint32_t kvs_build_info(void);

#ifdef __cplusplus
}
#endif

#endif /* KVS_H */
