// General decode attend: any head_dim, any GQA group, f32 / bf16 / E4M3 storage, any
// window.  One CTA per sequence, CUDA cores, logits in the workspace scratch.
//
// Serves the shapes the tensor-core kernel does not cover (small heads, f32 caches,
// windows that are not a multiple of 16).  Same arithmetic contract: logits
// q.k/sqrt(D) with k decoded inline (E4M3: code * scale), softmax per query head
// ("Context views at marginal cost", Fact 3), output sum_j a_j v_j, then the step
// masses: per entry the sum over query heads of its weight ("Context Optimization",
// H2O > How It Works, step 1) and per 16-token block the maximum over query heads of
// the head's in-block weight ("Per-Head Attention as a Scoring Signal", Fix: score
// per head, place per block).
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kvs_internal.cuh"

namespace kvs {

namespace {

constexpr int kThreads = 256;
constexpr float kLog2e = 1.4426950408889634f;

template <int KV>
__device__ __forceinline__ float load_kv(const uint8_t* page, int idx) {
  if constexpr (KV == KVS_E4M3) {
    const __half_raw h = __nv_cvt_fp8_to_halfraw(page[idx], __NV_E4M3);
    return __half2float(__half(h));
  } else if constexpr (KV == KVS_BF16) {
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(page)[idx]);
  } else {
    return reinterpret_cast<const float*>(page)[idx];
  }
}

template <int IN>
__device__ __forceinline__ float load_in(const void* p, size_t idx) {
  if constexpr (IN == KVS_BF16) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[idx]);
  else return static_cast<const float*>(p)[idx];
}

__device__ __forceinline__ float block_max(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = red[0];
  for (int w = 1; w < kThreads / 32; ++w) r = fmaxf(r, red[w]);
  return r;
}

__device__ __forceinline__ float block_sum(float v, float* red) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float r = 0.f;
  for (int w = 0; w < kThreads / 32; ++w) r += red[w];   // fixed order: deterministic
  return r;
}

// scratch per sequence: logits [Hq][cap] (log2 domain), cap = entries capacity
template <int KV, int IN>
__global__ void __launch_bounds__(kThreads) attend_general_kernel(Dev d, int layer, SeqSel sel,
                                                                  const void* q, float* out, float* tok_out,
                                                                  int cap) {
  extern __shared__ float sm[];
  float* qs = sm;                                  // [Hq][D]
  float* mh = qs + d.Hq * d.D;                     // [Hq] max
  float* lh = mh + d.Hq;                           // [Hq] sum
  float* red = lh + d.Hq;                          // [32]
  const int sl = blockIdx.x, s = sel.at(sl);
  if (!KVS_DCHECK(d, s >= 0 && s < d.max_seqs)) return;
  const SeqBlocks sb = seq_blocks(d, layer, s);
  const int n = sb.n * kBlock;                     // entries incl. masked ones
  if (n == 0 || n > cap) {
    if (threadIdx.x == 0) set_error(d, kErrState);
    return;
  }
  float* lg = d.logit_scratch + (size_t)sl * d.Hq * cap;
  const int G = d.Hq / d.Hkv;
  const size_t lay_slot = (size_t)layer * d.slot_layer_elems;
  const uint8_t* kpages = d.k_pages + layer * d.page_layer_bytes;
  const uint8_t* vpages = d.v_pages + layer * d.page_layer_bytes;
  const float inv = rsqrtf((float)d.D) * kLog2e;

  for (int i = threadIdx.x; i < d.Hq * d.D; i += kThreads)
    qs[i] = load_in<IN>(q, (size_t)sl * d.Hq * d.D + i);
  __syncthreads();

  // 1. logits (log2 domain) for every (head, entry); masked entries get -inf
  for (int idx = threadIdx.x; idx < d.Hq * n; idx += kThreads) {
    const int h = idx / n, e = idx % n;
    int32_t page;
    const int32_t k = block_at(d, s, sb, e / kBlock, &page);
    const int64_t p = (int64_t)k * kBlock + e % kBlock;
    float v = -INFINITY;
    if (p >= sb.lo && p < sb.next) {
      int32_t slot;
      page = page_of(d, s, p, &slot);
      const int kvh = h / G;
      const uint8_t* kp = kpages + (size_t)page * d.page_bytes;
      const int base = (kvh * kBlock + slot) * d.D;
      float acc = 0.f;
      for (int j = 0; j < d.D; ++j) acc = fmaf(qs[h * d.D + j], load_kv<KV>(kp, base + j), acc);
      const float sc = (KV == KVS_E4M3) ? d.k_scales[lay_slot + (size_t)page * kBlock + slot] : 1.f;
      v = acc * sc * inv;
    }
    lg[(size_t)h * cap + e] = v;
  }
  __syncthreads();

  // 2. per-head max and normaliser
  for (int h = 0; h < d.Hq; ++h) {
    float m = -INFINITY;
    for (int e = threadIdx.x; e < n; e += kThreads) m = fmaxf(m, lg[(size_t)h * cap + e]);
    m = block_max(m, red);
    float l = 0.f;
    for (int e = threadIdx.x; e < n; e += kThreads) l += exp2f(lg[(size_t)h * cap + e] - m);
    l = block_sum(l, red);
    if (threadIdx.x == 0) { mh[h] = m; lh[h] = l; }
    __syncthreads();
  }

  // 3. output: thread per (head, dim), entries in order
  for (int idx = threadIdx.x; idx < d.Hq * d.D; idx += kThreads) {
    const int h = idx / d.D, j = idx % d.D, kvh = h / G;
    const float m = mh[h];
    float acc = 0.f;
    for (int e = 0; e < n; ++e) {
      const float lv = lg[(size_t)h * cap + e];
      if (lv == -INFINITY) continue;
      int32_t page;
      const int32_t k = block_at(d, s, sb, e / kBlock, &page);
      const int64_t p = (int64_t)k * kBlock + e % kBlock;
      int32_t slot;
      page = page_of(d, s, p, &slot);
      const float sc = (KV == KVS_E4M3) ? d.v_scales[lay_slot + (size_t)page * kBlock + slot] : 1.f;
      acc = fmaf(exp2f(lv - m), load_kv<KV>(vpages + (size_t)page * d.page_bytes,
                                            (kvh * kBlock + slot) * d.D + j) * sc, acc);
    }
    out[((size_t)sl * d.Hq + h) * d.D + j] = acc / lh[h];
  }

  // 4. masses
  for (int e = threadIdx.x; e < n; e += kThreads) {
    int32_t page;
    const int32_t k = block_at(d, s, sb, e / kBlock, &page);
    const int64_t p = (int64_t)k * kBlock + e % kBlock;
    if (p < sb.lo || p >= sb.next) continue;
    float tau = 0.f;
    for (int h = 0; h < d.Hq; ++h) tau += exp2f(lg[(size_t)h * cap + e] - mh[h]) / lh[h];
    int32_t slot;
    page = page_of(d, s, p, &slot);
    d.tok_mass[lay_slot + (size_t)page * kBlock + slot] = tau;
    if (tok_out) tok_out[(size_t)sl * d.max_positions + p] = tau;
  }
  for (int i = threadIdx.x; i < sb.n; i += kThreads) {
    int32_t page;
    const int32_t k = block_at(d, s, sb, i, &page);
    float best = 0.f;
    for (int h = 0; h < d.Hq; ++h) {
      float bs = 0.f;
      for (int j = 0; j < kBlock; ++j) bs += exp2f(lg[(size_t)h * cap + i * kBlock + j] - mh[h]) / lh[h];
      best = fmaxf(best, bs);
      record_head(d, layer, s, k, h, bs);
    }
    d.blk_mass[(size_t)layer * d.blk_layer_elems + (size_t)s * d.max_blocks + k] = best;
  }
}

}  // namespace

size_t general_smem_bytes(int Hq, int D) { return ((size_t)Hq * D + 2 * Hq + 32) * sizeof(float); }

cudaError_t launch_attend_general(const Dev& d, int layer, SeqSel sel, int n_seqs,
                                  const void* q, float* out, float* tok_out, cudaStream_t st) {
  const int cap = (int)(d.logit_scratch_elems / ((size_t)n_seqs * d.Hq));
  const size_t smem = general_smem_bytes(d.Hq, d.D);
  const int KV = d.kv_dtype, IN = d.in_dtype;
#define KVS_LAUNCH(A, B)                                                                          \
  do {                                                                                            \
    auto fn = attend_general_kernel<A, B>;                                                        \
    if (smem > 48 * 1024) cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); \
    fn<<<n_seqs, kThreads, smem, st>>>(d, layer, sel, q, out, tok_out, cap);                      \
  } while (0)
  if (KV == KVS_E4M3 && IN == KVS_BF16) KVS_LAUNCH(KVS_E4M3, KVS_BF16);
  else if (KV == KVS_E4M3) KVS_LAUNCH(KVS_E4M3, KVS_F32);
  else if (KV == KVS_BF16) KVS_LAUNCH(KVS_BF16, KVS_BF16);
  else if (IN == KVS_BF16) KVS_LAUNCH(KVS_F32, KVS_BF16);
  else KVS_LAUNCH(KVS_F32, KVS_F32);
#undef KVS_LAUNCH
  return cudaGetLastError();
}

}  // namespace kvs
