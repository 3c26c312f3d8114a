// Storing one new position of one cache (K or V) into its slot: shared by the append
// kernel and the tensor-core attend's fused append, so both store identical bytes.
//
// Flash-MoE "Context Optimization", FP8 KV Cache > How It Works: one scale per position
// (all KV heads of K, and separately of V) = absmax / 240, values divided by the scale
// and rounded to E4M3, the scale stored beside the codes.  The divisions are IEEE
// round-to-nearest (__fdiv_rn) and the code is the hardware's round-to-nearest-even,
// saturating conversion.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kvs_internal.cuh"

namespace kvs {

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

// The same store for bf16 input already in registers: lane l holds chunks l, l + 32,
// ... (NCH of them, 8 values each) of the position's Hkv*D values, loaded by
// load_position_bf16.  Same arithmetic as store_position<KV, KVS_BF16>, so the bytes
// are the same.  Used by the fused append, which loads the rows before its own copies
// fill the memory queue.
template <int NCH>
__device__ __forceinline__ void load_position_bf16(const void* src, size_t src_elem, int lane, uint4 (&raw)[NCH]) {
#pragma unroll
  for (int j = 0; j < NCH; ++j)
    raw[j] = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(src) + src_elem + (size_t)(lane + 32 * j) * 8);
}

template <int KV, int NCH>
__device__ void store_position_regs(const Dev& d, const uint4 (&raw)[NCH], uint8_t* page_base, float* scale_slot,
                                    int slot, int lane) {
  if constexpr (KV == KVS_E4M3) {
    float amax = 0.f;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[j]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = (amax > 0.f) ? __fdiv_rn(amax, 240.0f) : 0.f;
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw[j]);
      float v[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h[i]);
        v[2 * i] = f.x;
        v[2 * i + 1] = f.y;
      }
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        uint32_t code = 0;
        if (scale > 0.f)
          code = (uint32_t)__nv_cvt_float_to_fp8(__fdiv_rn(v[i], scale), __NV_SATFINITE, __NV_E4M3);
        if (i < 4) lo |= code << (8 * i); else hi |= code << (8 * (i - 4));
      }
      const int e = (lane + 32 * j) * 8, kvh = e / d.D, dd = e % d.D;
      uint8_t* dst = page_base + ((size_t)(kvh * kBlock + slot) * d.D + dd);
      *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
    }
    if (lane == 0) *scale_slot = scale;
  } else {
    static_assert(KV == KVS_BF16, "bf16 or E4M3 storage");
#pragma unroll
    for (int j = 0; j < NCH; ++j) {
      const int e = (lane + 32 * j) * 8, kvh = e / d.D, dd = e % d.D;
      *reinterpret_cast<uint4*>(page_base + ((size_t)(kvh * kBlock + slot) * d.D + dd) * 2) = raw[j];
    }
  }
}

}  // namespace kvs
