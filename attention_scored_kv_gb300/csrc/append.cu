// kvs_append_kv: quantise (E4M3) or copy the new tokens' K and V into their slots.
//
// Flash-MoE "Context Optimization", FP8 KV Cache > How It Works: one scale per
// position (all KV heads of K, and separately of V) = absmax / 240, values divided by
// the scale and rounded to E4M3, the scale stored beside the codes.  The divisions
// are IEEE round-to-nearest (__fdiv_rn) and the code is the hardware's
// round-to-nearest-even, saturating conversion.  Sliding Window Attention > Design:
// window mode writes position p to slot p % window.  "LLM mechanics III", section 5:
// the absolute position is recorded per slot and next_position only ever advances.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kvs_internal.cuh"

namespace kvs {

namespace {

constexpr int kWarps = 8;

template <int IN>
__device__ __forceinline__ void load8(const void* base, size_t elem, float v[8]) {
  if constexpr (IN == KVS_BF16) {
    const uint4 raw = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + elem);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      v[2 * i] = f.x;
      v[2 * i + 1] = f.y;
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(base) + elem);
    const float4 a = p[0], b = p[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// One warp stores one position of one cache (K or V): Hkv*D values, 8 per chunk.
template <int KV, int IN>
__device__ void store_position(const Dev& d, const void* src, size_t src_elem, uint8_t* page_base,
                               float* scale_slot, int slot, int lane) {
  const int n = d.Hkv * d.D;
  const int chunks = n / 8;
  if constexpr (KV == KVS_E4M3) {
    float amax = 0.f;
    for (int c = lane; c < chunks; c += 32) {
      float v[8];
      load8<IN>(src, src_elem + (size_t)c * 8, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = (amax > 0.f) ? __fdiv_rn(amax, 240.0f) : 0.f;
    for (int c = lane; c < chunks; c += 32) {
      float v[8];
      load8<IN>(src, src_elem + (size_t)c * 8, v);
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t code = 0;
        if (scale > 0.f)
          code = (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(v[i], scale), __NV_SATFINITE, __NV_E4M3);
        if (i < 4) lo |= code << (8 * i); else hi |= code << (8 * (i - 4));
      }
      const int e = c * 8, kvh = e / d.D, dd = e % d.D;
      uint8_t* dst = page_base + ((size_t)(kvh * kBlock + slot) * d.D + dd);
      *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
    }
    if (lane == 0) *scale_slot = scale;
  } else if constexpr (KV == KVS_BF16) {
    // bf16 input only (checked on the host)
    for (int c = lane; c < chunks; c += 32) {
      const int e = c * 8, kvh = e / d.D, dd = e % d.D;
      const uint4 raw = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(src) + src_elem + e);
      *reinterpret_cast<uint4*>(page_base + ((size_t)(kvh * kBlock + slot) * d.D + dd) * 2) = raw;
    }
  } else {
    for (int c = lane; c < chunks; c += 32) {
      float v[8];
      load8<IN>(src, src_elem + (size_t)c * 8, v);
      const int e = c * 8, kvh = e / d.D, dd = e % d.D;
      float4* dst = reinterpret_cast<float4*>(page_base + ((size_t)(kvh * kBlock + slot) * d.D + dd) * 4);
      dst[0] = make_float4(v[0], v[1], v[2], v[3]);
      dst[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
  }
}

// grid (ceil(n_new / (kWarps/2)), n_seqs): two warps per new token, one for K, one for V.
template <int KV, int IN>
__global__ void __launch_bounds__(kWarps * 32) append_kernel(Dev d, int layer, int seq_begin, int n_new,
                                                               const void* k_in, const void* v_in) {
  const int s_local = blockIdx.y;
  const int s = seq_begin + s_local;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const size_t np_idx = (size_t)layer * d.max_seqs + s;
  const int64_t next0 = d.next_pos[np_idx];
  const int i = blockIdx.x * (kWarps / 2) + (warp >> 1);   // token; warp pairs split K and V
  const bool is_k = (warp & 1) == 0;
  if (i < n_new) {
    const int64_t p = next0 + i;
    if (p >= d.max_positions) {
      if (lane == 0) set_error(d, kErrCapacity);
    } else if (d.mode == KVS_MODE_WINDOW && i < n_new - d.window) {
      // a later token of this same call takes slot p % window: only the last `window`
      // tokens of a chunk are stored (the circular overwrite, without a write race)
    } else {
      int32_t slot;
      const int32_t page = page_of(d, s, p, &slot);
      if (page < 0 || page >= d.num_pages) {
        if (lane == 0) set_error(d, kErrState);
      } else {
        const size_t src_elem = ((size_t)s_local * n_new + i) * (size_t)d.Hkv * d.D;
        const size_t lay_slot = (size_t)layer * d.slot_layer_elems + (size_t)page * kBlock;
        uint8_t* kp = d.k_pages + layer * d.page_layer_bytes + (size_t)page * d.page_bytes;
        uint8_t* vp = d.v_pages + layer * d.page_layer_bytes + (size_t)page * d.page_bytes;
        if (is_k) {
          store_position<KV, IN>(d, k_in, src_elem, kp, d.k_scales ? d.k_scales + lay_slot + slot : nullptr, slot, lane);
          if (lane == 0) d.pos[lay_slot + slot] = p;
        } else {
          store_position<KV, IN>(d, v_in, src_elem, vp, d.v_scales ? d.v_scales + lay_slot + slot : nullptr, slot, lane);
        }
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // Every CTA of this sequence has read next0 before taking its ticket, so the
    // last ticket holder may advance next_position.
    __threadfence();
    const int t = atomicAdd(&d.append_tickets[np_idx], 1);
    if (t == (int)gridDim.x - 1) {
      d.next_pos[np_idx] = next0 + n_new;
      d.append_tickets[np_idx] = 0;
      __threadfence();
    }
  }
}

// H2O: give every block that the new positions enter a page from the pool, in order,
// and append it to the sequence's resident list.  One thread per sequence.
__global__ void alloc_pages_kernel(Dev d, int layer, int seq_begin, int n_seqs, int n_new) {
  const int sl = blockIdx.x * blockDim.x + threadIdx.x;
  if (sl >= n_seqs) return;
  const int s = seq_begin + sl;
  const int64_t next0 = d.next_pos[(size_t)layer * d.max_seqs + s];
  const int64_t last = next0 + n_new - 1;
  if (n_new <= 0 || last >= d.max_positions) return;   // the append reports capacity
  const size_t base = (size_t)s * d.max_blocks;
  for (int64_t k = next0 / kBlock; k <= last / kBlock; ++k) {
    if (d.block_table[base + k] >= 0) continue;
    const int32_t idx = atomicSub(d.free_top, 1) - 1;
    if (idx < 0) {
      atomicAdd(d.free_top, 1);
      set_error(d, kErrCapacity);
      return;
    }
    const int32_t page = d.free_pages[idx];
    d.block_table[base + k] = page;
    const int32_t n = d.res_count[s];
    d.res_blocks[base + n] = (int32_t)k;
    d.res_pages[base + n] = page;
    d.res_count[s] = n + 1;
    for (int l = 0; l < d.L; ++l)
      for (int j = 0; j < kBlock; ++j) d.pos[(size_t)l * d.slot_layer_elems + (size_t)page * kBlock + j] = -1;
  }
}

}  // namespace

cudaError_t launch_alloc_pages(const Dev& d, int layer, int seq_begin, int n_seqs, int n_new,
                               cudaStream_t st) {
  alloc_pages_kernel<<<(n_seqs + 127) / 128, 128, 0, st>>>(d, layer, seq_begin, n_seqs, n_new);
  return cudaGetLastError();
}

cudaError_t launch_append(const Dev& d, int layer, int seq_begin, int n_seqs, int n_new,
                          const void* k, const void* v, cudaStream_t st) {
  dim3 grid((n_new + kWarps / 2 - 1) / (kWarps / 2), n_seqs);
  const int KV = d.kv_dtype, IN = d.in_dtype;
  if (KV == KVS_E4M3 && IN == KVS_BF16) append_kernel<KVS_E4M3, KVS_BF16><<<grid, kWarps * 32, 0, st>>>(d, layer, seq_begin, n_new, k, v);
  else if (KV == KVS_E4M3 && IN == KVS_F32) append_kernel<KVS_E4M3, KVS_F32><<<grid, kWarps * 32, 0, st>>>(d, layer, seq_begin, n_new, k, v);
  else if (KV == KVS_BF16) append_kernel<KVS_BF16, KVS_BF16><<<grid, kWarps * 32, 0, st>>>(d, layer, seq_begin, n_new, k, v);
  else if (KV == KVS_F32 && IN == KVS_BF16) append_kernel<KVS_F32, KVS_BF16><<<grid, kWarps * 32, 0, st>>>(d, layer, seq_begin, n_new, k, v);
  else append_kernel<KVS_F32, KVS_F32><<<grid, kWarps * 32, 0, st>>>(d, layer, seq_begin, n_new, k, v);
  return cudaGetLastError();
}

}  // namespace kvs
