// Tensor-core decode attend with the fused mass epilogue (head_dim 128, 8 query heads
// per KV head, bf16 or E4M3 storage, bf16 queries).
//
// What it computes ("Context views at marginal cost", Fact 3; Flash-MoE "Context
// Optimization", FP8 KV Cache > How It Works and H2O > How It Works; "Per-Head
// Attention as a Scoring Signal", Fix: score per head, place per block): for every
// sequence and query head h, logits s_j = q_h.k_j / sqrt(D) over the resident
// entries (E4M3 keys decoded inline as code * scale), a = softmax(s), output
// o_h = sum_j a_j v_j; then, without writing a anywhere off chip, the entry mass
// sum_h a_hj and the block mass max_h sum_{j in block} a_hj.
//
// How (GB300):
//   * Persistent, cooperative grid of one CTA per SM.  The resident 16-token blocks of
//     all sequences of the launch are laid end to end and split evenly over the CTAs,
//     so a ragged batch balances by construction; a CTA's share is cut into segments
//     (runs of blocks of one sequence).
//   * One producer warp streams each block's K (then V) for all KV heads into a ring
//     of shared-memory stages with TMA tensor copies (128-byte swizzle, L2 evict-first)
//     completed on mbarriers; E4M3 scales arrive by bulk copy on the same barrier.
//   * Eight consumer warps, each bound to one KV head, run QK^T and PV on the tensor
//     cores with mma.sync m16n8k16 (positions on M, the 8 heads of the group on N for
//     QK^T; dimensions on M for PV).  E4M3 codes are decoded to f16 in registers
//     (exact) and fed straight into the MMA fragments; the K scale is applied to the
//     fp32 logits, the V scale is folded into P.  bf16 P is split in two bf16 terms
//     (hi + lo) so the PV product keeps ~16 bits.
//   * Two passes per segment: all K blocks first (logits to shared memory, exact local
//     max), then all V blocks (p = exp2(s - m), written back in place, and PV) - no
//     rescaling of accumulators.
//   * Each CTA publishes (m, l, o) per head and segment, arrives on a per-sequence
//     counter, waits (bounded) until every CTA of the sequence has arrived, combines
//     the global normaliser, converts its own on-chip p into the final weights and
//     reduces them to the entry and block masses; the CTAs of a sequence share the
//     output combine.  The last CTA to leave resets the counters for the next launch.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "kvs_internal.cuh"

namespace kvs {

namespace {

constexpr int kD = 128;
constexpr int kG = 8;
constexpr int kNCW = 8;                 // consumer warps
constexpr int kThreads = (kNCW + 1) * 32;
constexpr int kMbarLimit = 1 << 22;     // polls of an mbarrier before giving up
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kVFold = 256.0f;        // E4M3: p * v_scale * 256 keeps P off f16 subnormals

template <int HKV, bool FP8>
struct Cfg {
  static constexpr int HQ = HKV * kG;
  static constexpr int WPK = kNCW / HKV;                   // consumer warps per KV head
  static constexpr int ESZ = FP8 ? 1 : 2;
  static constexpr int STAGE = HKV * kBlock * kD * ESZ;     // one block of K or V, all heads
  static constexpr int NS = FP8 ? (HKV == 4 ? 10 : 6) : (HKV == 4 ? 6 : 4);
  static constexpr int HALF = HKV * kBlock * 128;           // bf16: bytes of one 64-dim half
};

// ------------------------------------------------------------------ PTX wrappers
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
// Bounded wait for the phase with the given parity; false if the limit ran out.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (int it = 0; it < kMbarLimit; ++it) {
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    if (ok) return true;
  }
  return false;
}
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ uint4 lds128(const uint8_t* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes16) {
  uint32_t r;
  const uint16_t a = (uint16_t)two_codes16;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(a));
  return r;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ void mma_f16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_bf16(float c[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
               : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
               : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// Logit / weight store: per local block i, [HQ][16] floats; the 4-float chunk index of
// a position is XOR-ed with bits of the head so both access patterns spread over banks.
template <int HQ>
__device__ __forceinline__ int lidx(int i, int h, int pos) {
  return (i * HQ + h) * kBlock + ((((pos >> 2) ^ (h >> 1)) & 3) << 2) + (pos & 3);
}

// CTA holding global block x when CTA c holds q + (c < r) blocks.
__device__ __forceinline__ int cta_of(int64_t x, int64_t q, int64_t r) {
  const int64_t big = r * (q + 1);
  return (int)(x < big ? x / (q + 1) : r + (x - big) / q);
}

struct Params {
  int layer, seq_begin, n_seqs, cap;   // cap: blocks per CTA the buffers hold
  const void* q;                       // [n_seqs][HQ][D] bf16
  float* out;                          // [n_seqs][HQ][D]
  float qk_scale;                      // log2(e) / sqrt(D)
};

template <int HKV, bool FP8, bool LSMEM>
__global__ void __launch_bounds__(kThreads, 1)
attend_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                 const Dev d, const Params P) {
  using C = Cfg<HKV, FP8>;
  constexpr int HQ = C::HQ, NS = C::NS, WPK = C::WPK, REC = kD + 2;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* ring = smem;                                           // NS * STAGE
  float* sscale = reinterpret_cast<float*>(ring + NS * C::STAGE); // NS * 16 (E4M3)
  uint64_t* bars = reinterpret_cast<uint64_t*>(sscale + NS * kBlock);   // full[NS], empty[NS]
  int32_t* blk_id = reinterpret_cast<int32_t*>(bars + 2 * NS);
  int32_t* blk_page = blk_id + P.cap;
  int32_t* blk_seq = blk_page + P.cap;
  int32_t* prefix = blk_seq + P.cap;                              // [n_seqs + 1]
  float* mbuf = reinterpret_cast<float*>(prefix + P.n_seqs + 1); // [WPK][HQ]
  float* lbuf = mbuf + WPK * HQ;                                  // [WPK][HQ]
  float* mseg = lbuf + WPK * HQ;                                  // [HQ]
  float* cfac = mseg + HQ;                                        // [HQ]
  float* gmax = cfac + HQ;                                        // [HQ]
  float* ginv = gmax + HQ;                                        // [HQ]
  int32_t* flag = reinterpret_cast<int32_t*>(ginv + HQ);          // [4]
  float* obuf = reinterpret_cast<float*>(flag + 4);               // WPK==2: [HKV][32 regs][32 lanes]
  float* lg_smem = reinterpret_cast<float*>(
      (reinterpret_cast<uintptr_t>(obuf + (WPK == 2 ? HKV * 32 * 32 : 0)) + 15) & ~uintptr_t(15));

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, G = gridDim.x;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + NS);

  // ---------------------------------------------------------------- partition
  if (warp == 0) {
    int run = 0;
    for (int b0 = 0; b0 < P.n_seqs; b0 += 32) {
      const int b = b0 + lane;
      int nb = 0;
      if (b < P.n_seqs) nb = seq_blocks(d, P.layer, P.seq_begin + b).n;
      int incl = nb;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (b < P.n_seqs) prefix[b] = run + incl - nb;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) prefix[P.n_seqs] = run;
  }
  __syncthreads();
  // CTA c takes q + (c < r) consecutive blocks (T = q*G + r): no empty CTA ever sits
  // between two non-empty ones, so a sequence's CTAs are a gap-free range.
  const int64_t T = prefix[P.n_seqs];
  const int64_t q = T / G, r = T % G;
  const int64_t x0 = (int64_t)c * q + (c < r ? c : r);
  const int nblk = (int)(q + (c < r ? 1 : 0));
  if (nblk > P.cap) {                       // the host's bound was too small
    if (tid == 0) set_error(d, kErrCapacity);
    return;
  }
  for (int i = tid; i < nblk; i += kThreads) {
    const int64_t x = x0 + i;
    int lo = 0, hi = P.n_seqs - 1;          // last b with prefix[b] <= x
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= x) lo = mid; else hi = mid - 1;
    }
    const int s = P.seq_begin + lo;
    const SeqBlocks sb = seq_blocks(d, P.layer, s);
    int32_t page;
    blk_id[i] = block_at(d, s, sb, (int)(x - prefix[lo]), &page);
    blk_page[i] = page;
    blk_seq[i] = lo;
  }
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, HKV);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  if (nblk == 0) return;

  float* lgbase = LSMEM ? lg_smem : d.logit_scratch + (size_t)c * P.cap * HQ * kBlock;
  const size_t lay_slot = (size_t)P.layer * d.slot_layer_elems;
  float* partials = d.partials;
  int32_t* arrive = d.counters;
  int32_t* depart = d.counters + d.max_seqs;

  // ================================================================ producer warp
  if (warp == kNCW) {
    if (lane == 0) {
      const uint64_t pol = evict_first_policy();
      uint32_t ctr = 0;
      int i0 = 0;
      while (i0 < nblk) {
        int i1 = i0 + 1;
        while (i1 < nblk && blk_seq[i1] == blk_seq[i0]) ++i1;
        for (int ph = 0; ph < 2; ++ph) {
          const CUtensorMap* map = ph == 0 ? &tmk : &tmv;
          const float* scales = ph == 0 ? d.k_scales : d.v_scales;
          for (int i = i0; i < i1; ++i, ++ctr) {
            const uint32_t st = ctr % NS, round = ctr / NS;
            if (round > 0 && !mbar_wait(empty0 + 8 * st, (round - 1) & 1)) set_error(d, kErrTimeout);
            const uint32_t fb = full0 + 8 * st;
            const uint32_t dst = smem_u32(ring + st * C::STAGE);
            mbar_expect_tx(fb, C::STAGE + (FP8 ? kBlock * 4 : 0));
            if constexpr (FP8) {
              tma_load_4d(dst, map, 0, 0, 0, blk_page[i], fb, pol);
              bulk_load(smem_u32(sscale + st * kBlock), scales + lay_slot + (size_t)blk_page[i] * kBlock,
                        kBlock * 4, fb);
            } else {
              tma_load_4d(dst, map, 0, 0, 0, blk_page[i], fb, pol);
              tma_load_4d(dst + C::HALF, map, 64, 0, 0, blk_page[i], fb, pol);
            }
          }
        }
        i0 = i1;
      }
    }
  } else {
    // ============================================================== consumer warps
    const int kvh = warp % HKV, sub = warp / HKV;
    const int g = lane >> 2, t = lane & 3;
    uint32_t ctr = 0;
    int i0 = 0;
    while (i0 < nblk) {
      int i1 = i0 + 1;
      while (i1 < nblk && blk_seq[i1] == blk_seq[i0]) ++i1;
      const int b = blk_seq[i0], s = P.seq_begin + b;
      const SeqBlocks sb = seq_blocks(d, P.layer, s);

      // Q fragments of head kvh*8 + g (B operand of QK^T)
      uint32_t qf[8][2];
      {
        const __nv_bfloat16* qrow = static_cast<const __nv_bfloat16*>(P.q) + ((size_t)b * HQ + kvh * kG + g) * kD;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          if constexpr (FP8) {
            // dims 32t + 4ks .. +3 (a permutation of the k index shared with the A side)
            const uint2 raw = *reinterpret_cast<const uint2*>(qrow + 32 * t + 4 * ks);
            const __nv_bfloat162* q2 = reinterpret_cast<const __nv_bfloat162*>(&raw);
            const float2 f0 = __bfloat1622float2(q2[0]), f1 = __bfloat1622float2(q2[1]);
            qf[ks][0] = pack_f16(f0.x, f0.y);
            qf[ks][1] = pack_f16(f1.x, f1.y);
          } else {
            qf[ks][0] = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * t);
            qf[ks][1] = *reinterpret_cast<const uint32_t*>(qrow + 16 * ks + 2 * t + 8);
          }
        }
      }

      // ------------------------------------------------------------ pass 1: K
      float mx0 = -INFINITY, mx1 = -INFINITY;      // heads 2t, 2t+1 of this KV group
      for (int i = i0; i < i1; ++i, ++ctr) {
        if ((i & (WPK - 1)) != sub) continue;
        const uint32_t st = ctr % NS, round = ctr / NS;
        if (!mbar_wait(full0 + 8 * st, round & 1)) set_error(d, kErrTimeout);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const uint8_t* stage = ring + st * C::STAGE;
        if constexpr (FP8) {
          const uint8_t* kb = stage + kvh * kBlock * kD;
          const uint4 r0a = lds128(kb + g * kD + (((2 * t) ^ g) << 4));
          const uint4 r0b = lds128(kb + g * kD + (((2 * t + 1) ^ g) << 4));
          const uint4 r1a = lds128(kb + (g + 8) * kD + (((2 * t) ^ g) << 4));
          const uint4 r1b = lds128(kb + (g + 8) * kD + (((2 * t + 1) ^ g) << 4));
          const uint32_t w0[8] = {r0a.x, r0a.y, r0a.z, r0a.w, r0b.x, r0b.y, r0b.z, r0b.w};
          const uint32_t w1[8] = {r1a.x, r1a.y, r1a.z, r1a.w, r1b.x, r1b.y, r1b.z, r1b.w};
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            mma_f16(acc, e4m3x2_to_f16x2(w0[ks] & 0xffffu), e4m3x2_to_f16x2(w1[ks] & 0xffffu),
                    e4m3x2_to_f16x2(w0[ks] >> 16), e4m3x2_to_f16x2(w1[ks] >> 16), qf[ks][0], qf[ks][1]);
          }
        } else {
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const int half = ks >> 2, c0 = (2 * ks) & 7;
            const int m = lane >> 3, row = ((m & 1) << 3) + (lane & 7), chunk = c0 + (m >> 1);
            const uint8_t* base = stage + half * C::HALF + kvh * kBlock * 128;
            uint32_t a0, a1, a2, a3;
            ldsm_x4(smem_u32(base + row * 128 + ((chunk ^ (row & 7)) << 4)), a0, a1, a2, a3);
            mma_bf16(acc, a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
          }
        }
        const int64_t p0 = (int64_t)blk_id[i] * kBlock;
        float sc0 = P.qk_scale, sc1 = P.qk_scale;
        if constexpr (FP8) {
          const float* sk = sscale + st * kBlock;
          sc0 *= sk[g];
          sc1 *= sk[g + 8];
        }
        const bool v0 = p0 + g >= sb.lo && p0 + g < sb.next;
        const bool v1 = p0 + g + 8 >= sb.lo && p0 + g + 8 < sb.next;
        const float s00 = v0 ? acc[0] * sc0 : -INFINITY, s01 = v0 ? acc[1] * sc0 : -INFINITY;
        const float s10 = v1 ? acc[2] * sc1 : -INFINITY, s11 = v1 ? acc[3] * sc1 : -INFINITY;
        const int h0 = kvh * kG + 2 * t;
        lgbase[lidx<HQ>(i, h0, g)] = s00;
        lgbase[lidx<HQ>(i, h0 + 1, g)] = s01;
        lgbase[lidx<HQ>(i, h0, g + 8)] = s10;
        lgbase[lidx<HQ>(i, h0 + 1, g + 8)] = s11;
        mx0 = fmaxf(mx0, fmaxf(s00, s10));
        mx1 = fmaxf(mx1, fmaxf(s01, s11));
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * st);
      }
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      if (g == 0) {
        mbuf[sub * HQ + kvh * kG + 2 * t] = mx0;
        mbuf[sub * HQ + kvh * kG + 2 * t + 1] = mx1;
      }
      named_sync(1, kNCW * 32);
      if (tid < HQ) {
        float m = mbuf[tid];
        for (int w = 1; w < WPK; ++w) m = fmaxf(m, mbuf[w * HQ + tid]);
        mseg[tid] = m;
      }
      named_sync(1, kNCW * 32);

      // ------------------------------------------------------------ pass 2: V
      const int hg = kvh * kG + g;                 // head of this thread's P column
      const float mh = mseg[hg];
      float lsum = 0.f;
      float o[8][4];
#pragma unroll
      for (int mb = 0; mb < 8; ++mb) o[mb][0] = o[mb][1] = o[mb][2] = o[mb][3] = 0.f;
      for (int i = i0; i < i1; ++i, ++ctr) {
        if ((i & (WPK - 1)) != sub) continue;
        const uint32_t st = ctr % NS, round = ctr / NS;
        if (!mbar_wait(full0 + 8 * st, round & 1)) set_error(d, kErrTimeout);
        const uint8_t* stage = ring + st * C::STAGE;
        float2* pa = reinterpret_cast<float2*>(lgbase + lidx<HQ>(i, hg, 2 * t));
        float2* pb = reinterpret_cast<float2*>(lgbase + lidx<HQ>(i, hg, 2 * t + 8));
        const float2 sa = *pa, sbv = *pb;
        const float p0 = exp2f(sa.x - mh), p1 = exp2f(sa.y - mh);
        const float p8 = exp2f(sbv.x - mh), p9 = exp2f(sbv.y - mh);
        lsum += (p0 + p1) + (p8 + p9);
        *pa = make_float2(p0, p1);
        *pb = make_float2(p8, p9);
        if constexpr (FP8) {
          const float* sv = sscale + st * kBlock;
          const uint32_t b0 = pack_f16(p0 * sv[2 * t] * kVFold, p1 * sv[2 * t + 1] * kVFold);
          const uint32_t b1 = pack_f16(p8 * sv[2 * t + 8] * kVFold, p9 * sv[2 * t + 9] * kVFold);
          const uint8_t* vb = stage + kvh * kBlock * kD;
          const uint4 L0 = lds128(vb + (2 * t) * kD + ((g ^ (2 * t)) << 4));
          const uint4 L1 = lds128(vb + (2 * t + 1) * kD + ((g ^ (2 * t + 1)) << 4));
          const uint4 L2 = lds128(vb + (2 * t + 8) * kD + ((g ^ (2 * t)) << 4));
          const uint4 L3 = lds128(vb + (2 * t + 9) * kD + ((g ^ (2 * t + 1)) << 4));
          const uint32_t x0[4] = {L0.x, L0.y, L0.z, L0.w}, y0[4] = {L1.x, L1.y, L1.z, L1.w};
          const uint32_t x2[4] = {L2.x, L2.y, L2.z, L2.w}, y2[4] = {L3.x, L3.y, L3.z, L3.w};
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const uint32_t lo = prmt(x0[w], y0[w], 0x5140), hi = prmt(x0[w], y0[w], 0x7362);
            const uint32_t lo2 = prmt(x2[w], y2[w], 0x5140), hi2 = prmt(x2[w], y2[w], 0x7362);
            mma_f16(o[2 * w], e4m3x2_to_f16x2(lo & 0xffffu), e4m3x2_to_f16x2(lo >> 16),
                    e4m3x2_to_f16x2(lo2 & 0xffffu), e4m3x2_to_f16x2(lo2 >> 16), b0, b1);
            mma_f16(o[2 * w + 1], e4m3x2_to_f16x2(hi & 0xffffu), e4m3x2_to_f16x2(hi >> 16),
                    e4m3x2_to_f16x2(hi2 & 0xffffu), e4m3x2_to_f16x2(hi2 >> 16), b0, b1);
          }
        } else {
          const float h0 = __bfloat162float(__float2bfloat16_rn(p0)), h1 = __bfloat162float(__float2bfloat16_rn(p1));
          const float h8 = __bfloat162float(__float2bfloat16_rn(p8)), h9 = __bfloat162float(__float2bfloat16_rn(p9));
          const uint32_t bh0 = pack_bf16(h0, h1), bh1 = pack_bf16(h8, h9);
          const uint32_t bl0 = pack_bf16(p0 - h0, p1 - h1), bl1 = pack_bf16(p8 - h8, p9 - h9);
#pragma unroll
          for (int mb = 0; mb < 8; ++mb) {
            const int half = mb >> 2, c0 = (2 * mb) & 7;
            const int m = lane >> 3, pos = ((m >> 1) << 3) + (lane & 7), chunk = c0 + (m & 1);
            const uint8_t* base = stage + half * C::HALF + kvh * kBlock * 128;
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(smem_u32(base + pos * 128 + ((chunk ^ (pos & 7)) << 4)), a0, a1, a2, a3);
            mma_bf16(o[mb], a0, a1, a2, a3, bh0, bh1);
            mma_bf16(o[mb], a0, a1, a2, a3, bl0, bl1);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * st);
      }
      // l of head hg: sum over the four lanes sharing g
      lsum += __shfl_xor_sync(0xffffffffu, lsum, 1);
      lsum += __shfl_xor_sync(0xffffffffu, lsum, 2);
      if (t == 0) lbuf[sub * HQ + hg] = lsum;
      if (WPK == 2 && sub == 1) {
#pragma unroll
        for (int mb = 0; mb < 8; ++mb)
#pragma unroll
          for (int r = 0; r < 4; ++r) obuf[(kvh * 32 + mb * 4 + r) * 32 + lane] = o[mb][r];
      }
      named_sync(1, kNCW * 32);
      if (sub == 0) {
        if (WPK == 2) {
#pragma unroll
          for (int mb = 0; mb < 8; ++mb)
#pragma unroll
            for (int r = 0; r < 4; ++r) o[mb][r] += obuf[(kvh * 32 + mb * 4 + r) * 32 + lane];
        }
        const float ofold = FP8 ? 1.0f / kVFold : 1.0f;
        float* rec = partials + (size_t)(c + b) * HQ * REC;
        const int ha = kvh * kG + 2 * t;
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
          int da, db;   // dims of accumulator rows g and g+8
          if constexpr (FP8) { da = 16 * g + 2 * mb; db = da + 1; }
          else { da = 16 * mb + g; db = da + 8; }
          rec[(size_t)ha * REC + 2 + da] = o[mb][0] * ofold;
          rec[(size_t)(ha + 1) * REC + 2 + da] = o[mb][1] * ofold;
          rec[(size_t)ha * REC + 2 + db] = o[mb][2] * ofold;
          rec[(size_t)(ha + 1) * REC + 2 + db] = o[mb][3] * ofold;
        }
        if (lane < kG) {
          const int h = kvh * kG + lane;
          float l = lbuf[h];
          for (int w = 1; w < WPK; ++w) l += lbuf[w * HQ + h];
          rec[(size_t)h * REC + 0] = mseg[h];
          rec[(size_t)h * REC + 1] = l;
        }
      }
      __threadfence();                 // every writer: partials visible GPU-wide ...
      named_sync(1, kNCW * 32);
      if (tid == 0) atomicAdd(&arrive[s], 1);   // ... before the arrival
      i0 = i1;
    }

    // ================================================================ epilogue
    i0 = 0;
    while (i0 < nblk) {
      int i1 = i0 + 1;
      while (i1 < nblk && blk_seq[i1] == blk_seq[i0]) ++i1;
      const int b = blk_seq[i0], s = P.seq_begin + b;
      const SeqBlocks sb = seq_blocks(d, P.layer, s);
      const int cf = cta_of(prefix[b], q, r), cl = cta_of(prefix[b + 1] - 1, q, r);
      const int S = cl - cf + 1;
      if (tid == 0) {
        const bool ok = wait_at_least(&arrive[s], S, d.spin_limit);
        __threadfence();
        flag[0] = ok ? 1 : 0;
        if (!ok) set_error(d, kErrTimeout);
      }
      named_sync(1, kNCW * 32);
      if (!flag[0]) break;
      if (tid < HQ) {
        float M = -INFINITY;
        for (int pc = cf; pc <= cl; ++pc) M = fmaxf(M, __ldcg(partials + ((size_t)(pc + b) * HQ + tid) * REC));
        float L = 0.f;
        for (int pc = cf; pc <= cl; ++pc) {
          const float* r = partials + ((size_t)(pc + b) * HQ + tid) * REC;
          L += __ldcg(r + 1) * exp2f(__ldcg(r) - M);
        }
        const float mown = __ldcg(partials + ((size_t)(c + b) * HQ + tid) * REC);
        cfac[tid] = exp2f(mown - M) / L;
        gmax[tid] = M;
        ginv[tid] = 1.0f / L;
      }
      named_sync(1, kNCW * 32);
      // masses: one warp per block; lanes 0-15 positions x heads [0, HQ/2), 16-31 the rest
      for (int i = i0 + warp; i < i1; i += kNCW) {
        const int j = lane & 15, hh = (lane >> 4) * (HQ / 2);
        float tau = 0.f, bmax = 0.f;
        for (int h = hh; h < hh + HQ / 2; ++h) {
          const float a = lgbase[lidx<HQ>(i, h, j)] * cfac[h];
          tau += a;
          float bs = a;
          bs += __shfl_xor_sync(0xffffffffu, bs, 1);
          bs += __shfl_xor_sync(0xffffffffu, bs, 2);
          bs += __shfl_xor_sync(0xffffffffu, bs, 4);
          bs += __shfl_xor_sync(0xffffffffu, bs, 8);
          bmax = fmaxf(bmax, bs);
        }
        tau += __shfl_xor_sync(0xffffffffu, tau, 16);
        bmax = fmaxf(bmax, __shfl_xor_sync(0xffffffffu, bmax, 16));
        const int64_t p = (int64_t)blk_id[i] * kBlock + j;
        if (lane < 16 && p >= sb.lo && p < sb.next) {
          int32_t slot;
          const int32_t page = page_of(d, s, p, &slot);
          d.tok_mass[lay_slot + (size_t)page * kBlock + slot] = tau;
        }
        if (lane == 0)
          d.blk_mass[(size_t)P.layer * d.blk_layer_elems + (size_t)s * d.max_blocks + blk_id[i]] = bmax;
      }
      // output: this CTA combines heads h with h % S == its rank among the sequence's CTAs
      for (int h = c - cf; h < HQ; h += S) {
        const float M = gmax[h], inv = ginv[h];
        for (int dd = tid; dd < kD; dd += kNCW * 32) {
          float acc = 0.f;
          for (int pc = cf; pc <= cl; ++pc) {
            const float* r = partials + ((size_t)(pc + b) * HQ + h) * REC;
            acc += __ldcg(r + 2 + dd) * exp2f(__ldcg(r) - M);
          }
          P.out[((size_t)b * HQ + h) * kD + dd] = acc * inv;
        }
      }
      named_sync(1, kNCW * 32);
      if (tid == 0) {
        __threadfence();
        if (atomicAdd(&depart[s], 1) == S - 1) {   // last CTA of the sequence to leave
          arrive[s] = 0;
          depart[s] = 0;
          __threadfence();
        }
      }
      i0 = i1;
    }
  }
  __syncthreads();
}

size_t tc_smem_limit() { return 227 * 1024; }

template <int HKV, bool FP8, bool LSMEM>
size_t smem_bytes(int cap, int n_seqs) {
  using C = Cfg<HKV, FP8>;
  size_t b = 1024;                                    // alignment slack
  b += (size_t)C::NS * C::STAGE + C::NS * kBlock * 4 + 2 * C::NS * 8;
  b += (size_t)3 * cap * 4 + (size_t)(n_seqs + 1) * 4;
  b += (size_t)(2 * C::WPK + 4) * C::HQ * 4 + 16;
  b += (C::WPK == 2 ? (size_t)HKV * 32 * 32 * 4 : 0) + 16;
  if (LSMEM) b += (size_t)cap * C::HQ * kBlock * 4;
  return b;
}

template <int HKV, bool FP8, bool LSMEM>
cudaError_t launch_one(const CUtensorMap& tk, const CUtensorMap& tv, const Dev& d, const Params& P, int grid,
                       cudaStream_t st) {
  auto fn = attend_tc_kernel<HKV, FP8, LSMEM>;
  const size_t smem = smem_bytes<HKV, FP8, LSMEM>(P.cap, P.n_seqs);
  static bool attr_set = false;      // one opt-in per instantiation, to the full limit
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tc_smem_limit());
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, tk, tv, d, P);
}

template <int HKV, bool FP8>
cudaError_t launch_pick(const CUtensorMap& tk, const CUtensorMap& tv, const Dev& d, Params P, int grid,
                        size_t smem_limit, cudaStream_t st) {
  if (smem_bytes<HKV, FP8, true>(P.cap, P.n_seqs) <= smem_limit)
    return launch_one<HKV, FP8, true>(tk, tv, d, P, grid, st);
  if (smem_bytes<HKV, FP8, false>(P.cap, P.n_seqs) > smem_limit) return cudaErrorInvalidConfiguration;
  if ((size_t)grid * P.cap * Cfg<HKV, FP8>::HQ * kBlock > d.logit_scratch_elems) return cudaErrorInvalidConfiguration;
  return launch_one<HKV, FP8, false>(tk, tv, d, P, grid, st);
}

}  // namespace

bool tc_supported(int Hq, int Hkv, int D, int kv_dtype, int in_dtype, int window, int mode) {
  if (D != kD || Hq != Hkv * kG || (Hkv != 4 && Hkv != 8)) return false;
  if (in_dtype != KVS_BF16 || (kv_dtype != KVS_BF16 && kv_dtype != KVS_E4M3)) return false;
  if (mode == KVS_MODE_WINDOW && window % kBlock != 0) return false;
  return true;
}

// Tensor map over one layer's pages viewed as [num_pages][Hkv][16][D] elements.
cudaError_t make_page_map(CUtensorMap* map, const void* base, int num_pages, int Hkv, int kv_dtype) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (!encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  const bool fp8 = kv_dtype == KVS_E4M3;
  const int esz = fp8 ? 1 : 2;
  cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)kBlock, (cuuint64_t)Hkv, (cuuint64_t)num_pages};
  cuuint64_t strides[3] = {(cuuint64_t)kD * esz, (cuuint64_t)kBlock * kD * esz, (cuuint64_t)Hkv * kBlock * kD * esz};
  cuuint32_t box[4] = {(cuuint32_t)(fp8 ? 128 : 64), (cuuint32_t)kBlock, (cuuint32_t)Hkv, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = encode(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                      const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Blocks one CTA must hold for a launch whose resident blocks number at most T_bound.
int tc_cap(int64_t T_bound, int grid) { return (int)((T_bound + grid - 1) / grid); }

cudaError_t launch_attend_tc(const CUtensorMap& tk, const CUtensorMap& tv, const Dev& d, int layer,
                             int seq_begin, int n_seqs, const void* q, float* out, int64_t T_bound, int grid,
                             cudaStream_t st) {
  Params P;
  P.layer = layer;
  P.seq_begin = seq_begin;
  P.n_seqs = n_seqs;
  P.cap = tc_cap(T_bound, grid);
  if (P.cap < 1) P.cap = 1;
  P.q = q;
  P.out = out;
  P.qk_scale = kLog2e / sqrtf((float)kD);
  const size_t lim = tc_smem_limit();
  const bool fp8 = d.kv_dtype == KVS_E4M3;
  if (d.Hkv == 4) return fp8 ? launch_pick<4, true>(tk, tv, d, P, grid, lim, st)
                             : launch_pick<4, false>(tk, tv, d, P, grid, lim, st);
  return fp8 ? launch_pick<8, true>(tk, tv, d, P, grid, lim, st) : launch_pick<8, false>(tk, tv, d, P, grid, lim, st);
}

// Largest grid the cooperative launch allows with one CTA per SM.
int tc_grid(int kv_dtype, int Hkv, int sm_count) {
  int per_sm = 0;
  const bool fp8 = kv_dtype == KVS_E4M3;
  const size_t smem = tc_smem_limit();
  cudaError_t e;
  if (Hkv == 4) {
    if (fp8) { auto f = attend_tc_kernel<4, true, false>; cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f, kThreads, smem); }
    else { auto f = attend_tc_kernel<4, false, false>; cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f, kThreads, smem); }
  } else {
    if (fp8) { auto f = attend_tc_kernel<8, true, false>; cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f, kThreads, smem); }
    else { auto f = attend_tc_kernel<8, false, false>; cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem); e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f, kThreads, smem); }
  }
  if (e != cudaSuccess || per_sm < 1) return 0;
  int g = sm_count;          // one CTA per SM: the shares stay equal
  return g > kGridMax ? kGridMax : g;
}

// ----------------------------------------------------------------------------------
// Tensor-core attend with its exchange area in a library-owned array.
//
// The attend launch needs an exchange area: one (m, l, o) record per CTA and sequence
// and two arrival counters per sequence.  kvs_decode_attend takes it from the caller's
// workspace; this variant takes it from the array below, compiled into the library, so
// a call asks the caller for nothing but its inputs and outputs.  The array holds
// kStaticScratchBytes; a launch that needs more is refused.  Every call (every context,
// every stream) shares it and it keeps the last call's contents: the counters are
// cleared on the call's stream before each launch, and two such launches that overlap
// on the GPU race on it.
constexpr size_t kStaticScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_attend_scratch[kStaticScratchBytes];

namespace {
constexpr int kMaxDevices = 64;
void* g_scratch_addr[kMaxDevices] = {};
}  // namespace

size_t static_scratch_limit() { return kStaticScratchBytes; }

// Bytes of the array one launch uses: records for CTA + sequence index < grid + n_seqs,
// then 2 * max_seqs counters (indexed by absolute sequence).
size_t static_scratch_need(const Dev& d, int n_seqs, int grid, size_t* counters_offset) {
  const size_t rec = (size_t)(grid + n_seqs) * d.Hq * (kD + 2) * sizeof(float);
  const size_t off = (rec + 255) & ~size_t(255);
  *counters_offset = off;
  return off + 2 * (size_t)d.max_seqs * sizeof(int32_t);
}

// Device address of the array on the current device, looked up once per device (the
// host-side symbol is only a stand-in, never a device address).
cudaError_t static_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_attend_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

// Returns cudaErrorInvalidValue if the launch needs more than the array holds and
// cudaErrorNotSupported if its logits do not fit in shared memory (that case needs the
// workspace's logit scratch).
cudaError_t launch_attend_tc_static(const CUtensorMap& tk, const CUtensorMap& tv, const Dev& d, int layer,
                                    int seq_begin, int n_seqs, const void* q, float* out, int64_t T_bound,
                                    int grid, cudaStream_t st) {
  size_t counters_off = 0;
  if (static_scratch_need(d, n_seqs, grid, &counters_off) > kStaticScratchBytes) return cudaErrorInvalidValue;
  Params P;
  P.layer = layer;
  P.seq_begin = seq_begin;
  P.n_seqs = n_seqs;
  P.cap = tc_cap(T_bound, grid);
  if (P.cap < 1) P.cap = 1;
  P.q = q;
  P.out = out;
  P.qk_scale = kLog2e / sqrtf((float)kD);
  const bool fp8 = d.kv_dtype == KVS_E4M3;
  const size_t need_smem = d.Hkv == 4 ? (fp8 ? smem_bytes<4, true, true>(P.cap, n_seqs) : smem_bytes<4, false, true>(P.cap, n_seqs))
                                      : (fp8 ? smem_bytes<8, true, true>(P.cap, n_seqs) : smem_bytes<8, false, true>(P.cap, n_seqs));
  if (need_smem > tc_smem_limit()) return cudaErrorNotSupported;
  void* base = nullptr;
  cudaError_t e = static_scratch_address(&base);
  if (e != cudaSuccess) return e;
  Dev dd = d;
  dd.partials = static_cast<float*>(base);
  dd.counters = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(base) + counters_off);
  e = cudaMemsetAsync(dd.counters, 0, 2 * (size_t)d.max_seqs * sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  if (d.Hkv == 4) return fp8 ? launch_one<4, true, true>(tk, tv, dd, P, grid, st) : launch_one<4, false, true>(tk, tv, dd, P, grid, st);
  return fp8 ? launch_one<8, true, true>(tk, tv, dd, P, grid, st) : launch_one<8, false, true>(tk, tv, dd, P, grid, st);
}

}  // namespace kvs
