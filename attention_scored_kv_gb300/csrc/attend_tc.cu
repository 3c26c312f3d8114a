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
//   * Persistent, cooperative grid of one CTA per SM.  When every sequence can have CTAs
//     of its own, the host plans whole CTAs per sequence (sequence b owns CTAs
//     [cst[b], cst[b+1]) and splits its blocks evenly over them, one segment per CTA);
//     otherwise the resident 16-token blocks of all sequences are laid end to end and
//     split evenly over the CTAs on the device, a CTA's share cut into segments (runs
//     of blocks of one sequence).
//   * Ten warps.  One producer warp streams each block's K (then V) for all KV heads
//     into a ring of 48 KB shared-memory stages (three in the whole-CTA plan) with TMA
//     tensor copies (128-byte swizzle, L2 evict-first) completed on mbarriers; E4M3
//     scales arrive by bulk copy on the same barrier.  In the whole-CTA plan it builds
//     its own page list and issues the first copies without waiting for the consumers.
//   * Eight consumer warps, one or two per KV head, run QK^T and PV on the tensor cores
//     with mma.sync m16n8k16 (positions on M, the 8 heads of the group on N for QK^T;
//     dimensions on M for PV).  E4M3 codes are decoded to f16 in registers (exact) and
//     fed straight into the MMA fragments; the K scale is applied to the fp32 logits,
//     the V scale is folded into P.  bf16 P is split in two bf16 terms (hi + lo) so the
//     PV product keeps ~16 bits.
//   * Two passes per segment: all K blocks first (logits to shared memory, exact local
//     max), then the weights p = exp2(s - m) in place with the block sums and l, and
//     the CTA's (m, l) words are published; then all V blocks (PV) - no rescaling of
//     accumulators.
//   * The tenth warp (whole-CTA plan) stores the fused append's decode token while the
//     consumers run the K pass, then combines the sequence's normaliser from every
//     CTA's (m, l) words while they run the V pass.  Consumers hand their words and
//     partial output rows over with non-blocking named-barrier arrivals; this warp and
//     the producer publish them with one release-add per CTA on the sequence's counters.
//   * Epilogue: four consumer warps turn the CTA's own on-chip p into the final weights
//     and reduce them to the entry and block masses; the other four wait (bounded) for
//     every CTA's partial rows and share the output combine.  The last CTA to leave
//     resets the counters (and, for the fused append, advances the next position).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "append_store.cuh"
#include "kvs_internal.cuh"

namespace kvs {

namespace {

constexpr int kD = 128;
constexpr int kG = 8;
constexpr int kNCW = 8;                 // consumer warps
// A ring stage: every stage completion costs a few hundred ns of barrier traffic, so
// stages are large (48 KB: 6 E4M3 or 3 bf16 blocks of 4 KV heads); two or more stages.
constexpr int kStageBytes = 48 * 1024;
constexpr int kProducer = kNCW;         // warp that issues the copies
constexpr int kNormWarp = kNCW + 1;     // warp that combines the normaliser (whole plan)
constexpr int kThreads = (kNCW + 2) * 32;
// Named barriers: 1 all consumers, 2 + h the two consumer warps of KV head h, and in the
// whole plan: consumers -> normaliser warp for the statistics words (kBarMl) and for
// the partial output rows (kBarOut, producer warp), output warps among themselves
// (kBarOutWarps).
constexpr int kBarOut = 13, kBarMl = 14, kBarOutWarps = 15;
constexpr int kPubThreads = (kNCW + 1) * 32;   // consumers arrive, one publishing warp waits
constexpr int kMbarLimit = 1 << 22;     // polls of an mbarrier before giving up
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kVFold = 256.0f;        // E4M3: p * v_scale * 256 keeps P off f16 subnormals

template <int HKV, bool FP8>
struct Cfg {
  static constexpr int HQ = HKV * kG;
  static constexpr int WPK = kNCW / HKV;                   // consumer warps per KV head
  static constexpr int ESZ = FP8 ? 1 : 2;
  static constexpr int BLK = HKV * kBlock * kD * ESZ;       // one block of K or V, all heads
  static constexpr int SB = kStageBytes / BLK >= 1 ? kStageBytes / BLK : 1;   // blocks per ring stage
  static constexpr int STAGE = SB * BLK;
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
// Named barrier over n threads.  Every call site follows code that one thread or one
// lane runs alone (a wait, an atomic), so the warp is first reconverged and the
// non-aligned form is used: nothing here relies on the compiler having reconverged a
// warp before an inline-asm barrier.
__device__ __forceinline__ void named_sync(int id, int n) {
  __syncwarp();
  asm volatile("barrier.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}
// Named barrier that also returns the AND of every participant's v.
__device__ __forceinline__ bool named_sync_and(int id, int n, bool v) {
  __syncwarp();
  uint32_t r;
  asm volatile("{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.red.and.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
               : "=r"(r) : "r"((uint32_t)v), "r"(id), "r"(n) : "memory");
  return r != 0;
}
// Arrive on a named barrier of n threads without waiting (the waiters use named_sync).
__device__ __forceinline__ void named_arrive(int id, int n) {
  __syncwarp();
  asm volatile("barrier.arrive %0, %1;" :: "r"(id), "r"(n) : "memory");
}
// Add with release semantics: what this thread wrote or saw before is visible GPU-wide
// to whoever acquires the new value.
__device__ __forceinline__ void red_release_add(int32_t* p, int32_t v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void red_add(int32_t* p, int32_t v) {
  asm volatile("red.relaxed.gpu.global.add.s32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
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

// Logit / weight store: per local block i, [HQ][16] floats then 16 floats of padding
// (kLgPad: consecutive blocks start 64 bytes apart modulo 128, so reads of two blocks
// in one quarter-warp fall in different banks); the 4-float chunk index of a position
// is XOR-ed with bits of the head so both access patterns spread over banks.
constexpr int kLgPad = 16;
template <int HQ>
__host__ __device__ constexpr int lg_block() { return HQ * kBlock + kLgPad; }
template <int HQ>
__device__ __forceinline__ int lidx(int i, int h, int pos) {
  return i * lg_block<HQ>() + h * kBlock + ((((pos >> 2) ^ (h >> 1)) & 3) << 2) + (pos & 3);
}

// CTA holding global block x when CTA c holds q + (c < r) blocks.
__device__ __forceinline__ int cta_of(int x, int q, int r) {
  const int big = r * (q + 1);
  return x < big ? x / (q + 1) : r + (x - big) / q;
}

// QK^T of NB (1 or 2) blocks of one ring stage for one KV head, interleaved for ILP:
// logits (log2 domain, masked to -inf outside [lo, nxt)) go to the store, the running
// per-head max is updated.  Block b sits in stage slot j0 + b*WPK, CTA-local block
// index i_first + b*WPK.
template <int HKV, bool FP8, int NB>
__device__ __forceinline__ void qk_blocks(const uint8_t* stage, const float* sscale_st, int j0, int i_first,
                                          const int32_t* blk_id, const uint32_t (&qf)[8][2], float* lg, int kvh,
                                          int lane, int64_t lo, int64_t nxt, float qk_scale, float& mx0, float& mx1) {
  using C = Cfg<HKV, FP8>;
  constexpr int HQ = C::HQ, WPK = C::WPK;
  const int g = lane >> 2, t = lane & 3;
  float acc[NB][2][4];
#pragma unroll
  for (int b = 0; b < NB; ++b)
#pragma unroll
    for (int c2 = 0; c2 < 2; ++c2) acc[b][c2][0] = acc[b][c2][1] = acc[b][c2][2] = acc[b][c2][3] = 0.f;
  if constexpr (FP8) {
    uint32_t w0[NB][8], w1[NB][8];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const uint8_t* kb = stage + (size_t)(j0 + b * WPK) * C::BLK + kvh * kBlock * kD;
      const uint4 r0a = lds128(kb + g * kD + (((2 * t) ^ g) << 4));
      const uint4 r0b = lds128(kb + g * kD + (((2 * t + 1) ^ g) << 4));
      const uint4 r1a = lds128(kb + (g + 8) * kD + (((2 * t) ^ g) << 4));
      const uint4 r1b = lds128(kb + (g + 8) * kD + (((2 * t + 1) ^ g) << 4));
      w0[b][0] = r0a.x; w0[b][1] = r0a.y; w0[b][2] = r0a.z; w0[b][3] = r0a.w;
      w0[b][4] = r0b.x; w0[b][5] = r0b.y; w0[b][6] = r0b.z; w0[b][7] = r0b.w;
      w1[b][0] = r1a.x; w1[b][1] = r1a.y; w1[b][2] = r1a.z; w1[b][3] = r1a.w;
      w1[b][4] = r1b.x; w1[b][5] = r1b.y; w1[b][6] = r1b.z; w1[b][7] = r1b.w;
    }
#pragma unroll
    for (int ks = 0; ks < 8; ++ks)
#pragma unroll
      for (int b = 0; b < NB; ++b)
        mma_f16(acc[b][ks & 1], e4m3x2_to_f16x2(w0[b][ks] & 0xffffu), e4m3x2_to_f16x2(w1[b][ks] & 0xffffu),
                e4m3x2_to_f16x2(w0[b][ks] >> 16), e4m3x2_to_f16x2(w1[b][ks] >> 16), qf[ks][0], qf[ks][1]);
  } else {
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const int half = ks >> 2, c0 = (2 * ks) & 7;
      const int m = lane >> 3, row = ((m & 1) << 3) + (lane & 7), chunk = c0 + (m >> 1);
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const uint8_t* base = stage + (size_t)(j0 + b * WPK) * C::BLK + half * C::HALF + kvh * kBlock * 128;
        uint32_t a0, a1, a2, a3;
        ldsm_x4(smem_u32(base + row * 128 + ((chunk ^ (row & 7)) << 4)), a0, a1, a2, a3);
        mma_bf16(acc[b][ks & 1], a0, a1, a2, a3, qf[ks][0], qf[ks][1]);
      }
    }
  }
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const int i = i_first + b * WPK;
    const int64_t p0 = (int64_t)blk_id[i] * kBlock;
    float sc0 = qk_scale, sc1 = qk_scale;
    if constexpr (FP8) {
      const float* sk = sscale_st + (j0 + b * WPK) * kBlock;
      sc0 *= sk[g];
      sc1 *= sk[g + 8];
    }
    float s00 = (acc[b][0][0] + acc[b][1][0]) * sc0, s01 = (acc[b][0][1] + acc[b][1][1]) * sc0;
    float s10 = (acc[b][0][2] + acc[b][1][2]) * sc1, s11 = (acc[b][0][3] + acc[b][1][3]) * sc1;
    if (p0 < lo || p0 + kBlock > nxt) {                 // a block the window or the end cuts
      if (!(p0 + g >= lo && p0 + g < nxt)) s00 = s01 = -INFINITY;
      if (!(p0 + g + 8 >= lo && p0 + g + 8 < nxt)) s10 = s11 = -INFINITY;
    }
    const int h0 = kvh * kG + 2 * t;
    lg[lidx<HQ>(i, h0, g)] = s00;
    lg[lidx<HQ>(i, h0 + 1, g)] = s01;
    lg[lidx<HQ>(i, h0, g + 8)] = s10;
    lg[lidx<HQ>(i, h0 + 1, g + 8)] = s11;
    mx0 = fmaxf(mx0, fmaxf(s00, s10));
    mx1 = fmaxf(mx1, fmaxf(s01, s11));
  }
}

// PV of NB (1 or 2) blocks of one ring stage for one KV head: p = exp2(s - m) written
// back over the logits, per-head in-block sums to bsum, the running l, and the MMAs
// into the shared accumulators o (dimensions on M, heads on N).
template <int HKV, bool FP8, int NB>
__device__ __forceinline__ void pv_blocks(const uint8_t* stage, const float* sscale_st, int j0, int i_first,
                                          const float* lg, int kvh, int lane, float (&o)[8][4]) {
  using C = Cfg<HKV, FP8>;
  constexpr int HQ = C::HQ, WPK = C::WPK;
  const int g = lane >> 2, t = lane & 3;
  const int hg = kvh * kG + g;
  float p[NB][4];                                       // weights exp2(s - m), from the sweep
#pragma unroll
  for (int b = 0; b < NB; ++b) {
    const int i = i_first + b * WPK;
    const float2 pa = *reinterpret_cast<const float2*>(lg + lidx<HQ>(i, hg, 2 * t));
    const float2 pb = *reinterpret_cast<const float2*>(lg + lidx<HQ>(i, hg, 2 * t + 8));
    p[b][0] = pa.x;
    p[b][1] = pa.y;
    p[b][2] = pb.x;
    p[b][3] = pb.y;
  }
  if constexpr (FP8) {
    uint32_t b0[NB], b1[NB];
    uint32_t x0[NB][4], y0[NB][4], x2[NB][4], y2[NB][4];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float* sv = sscale_st + (j0 + b * WPK) * kBlock;
      b0[b] = pack_f16(p[b][0] * sv[2 * t] * kVFold, p[b][1] * sv[2 * t + 1] * kVFold);
      b1[b] = pack_f16(p[b][2] * sv[2 * t + 8] * kVFold, p[b][3] * sv[2 * t + 9] * kVFold);
      const uint8_t* vb = stage + (size_t)(j0 + b * WPK) * C::BLK + kvh * kBlock * kD;
      const uint4 L0 = lds128(vb + (2 * t) * kD + ((g ^ (2 * t)) << 4));
      const uint4 L1 = lds128(vb + (2 * t + 1) * kD + ((g ^ (2 * t + 1)) << 4));
      const uint4 L2 = lds128(vb + (2 * t + 8) * kD + ((g ^ (2 * t)) << 4));
      const uint4 L3 = lds128(vb + (2 * t + 9) * kD + ((g ^ (2 * t + 1)) << 4));
      x0[b][0] = L0.x; x0[b][1] = L0.y; x0[b][2] = L0.z; x0[b][3] = L0.w;
      y0[b][0] = L1.x; y0[b][1] = L1.y; y0[b][2] = L1.z; y0[b][3] = L1.w;
      x2[b][0] = L2.x; x2[b][1] = L2.y; x2[b][2] = L2.z; x2[b][3] = L2.w;
      y2[b][0] = L3.x; y2[b][1] = L3.y; y2[b][2] = L3.z; y2[b][3] = L3.w;
    }
#pragma unroll
    for (int w = 0; w < 4; ++w)
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const uint32_t lo = prmt(x0[b][w], y0[b][w], 0x5140), hi = prmt(x0[b][w], y0[b][w], 0x7362);
        const uint32_t lo2 = prmt(x2[b][w], y2[b][w], 0x5140), hi2 = prmt(x2[b][w], y2[b][w], 0x7362);
        mma_f16(o[2 * w], e4m3x2_to_f16x2(lo & 0xffffu), e4m3x2_to_f16x2(lo >> 16),
                e4m3x2_to_f16x2(lo2 & 0xffffu), e4m3x2_to_f16x2(lo2 >> 16), b0[b], b1[b]);
        mma_f16(o[2 * w + 1], e4m3x2_to_f16x2(hi & 0xffffu), e4m3x2_to_f16x2(hi >> 16),
                e4m3x2_to_f16x2(hi2 & 0xffffu), e4m3x2_to_f16x2(hi2 >> 16), b0[b], b1[b]);
      }
  } else {
    uint32_t bh0[NB], bh1[NB], bl0[NB], bl1[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      const float h0 = __bfloat162float(__float2bfloat16_rn(p[b][0])), h1 = __bfloat162float(__float2bfloat16_rn(p[b][1]));
      const float h8 = __bfloat162float(__float2bfloat16_rn(p[b][2])), h9 = __bfloat162float(__float2bfloat16_rn(p[b][3]));
      bh0[b] = pack_bf16(h0, h1);
      bh1[b] = pack_bf16(h8, h9);
      bl0[b] = pack_bf16(p[b][0] - h0, p[b][1] - h1);
      bl1[b] = pack_bf16(p[b][2] - h8, p[b][3] - h9);
    }
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) {
      const int half = mb >> 2, c0 = (2 * mb) & 7;
      const int m = lane >> 3, pos = ((m >> 1) << 3) + (lane & 7), chunk = c0 + (m & 1);
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const uint8_t* base = stage + (size_t)(j0 + b * WPK) * C::BLK + half * C::HALF + kvh * kBlock * 128;
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(smem_u32(base + pos * 128 + ((chunk ^ (pos & 7)) << 4)), a0, a1, a2, a3);
        mma_bf16(o[mb], a0, a1, a2, a3, bh0[b], bh1[b]);
        mma_bf16(o[mb], a0, a1, a2, a3, bl0[b], bl1[b]);
      }
    }
  }
}

// Between the passes: every logit of the CTA's blocks [i0, i1) becomes its weight
// p = exp2(s - m_h) in place (masked logits are -inf and give 0), each (block, head)
// row's sum goes to bsum, and each thread's sum over its rows to lred.  Thread tid
// keeps head tid % HQ, so the HQ-strided partials of lred add up to the head's l.
template <int HQ>
__device__ __forceinline__ void weights_sweep(float* lg, float* bsum, float* lred, const float* mseg, int i0,
                                              int i1, int tid) {
  constexpr int NT = kNCW * 32;
  static_assert(NT % HQ == 0, "a thread keeps one head");
  const int h = tid % HQ;
  const float m = mseg[h];
  float l = 0.f;
  for (int i = i0 + tid / HQ; i < i1; i += NT / HQ) {
    float4* row = reinterpret_cast<float4*>(lg + (size_t)i * lg_block<HQ>() + h * kBlock);
    // chunk u ^ (h >> 1): the lanes of a quarter-warp then read eight different bank groups
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = row[(u ^ (h >> 1)) & 3];
    float rs = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      v[u].x = exp2f(v[u].x - m);
      v[u].y = exp2f(v[u].y - m);
      v[u].z = exp2f(v[u].z - m);
      v[u].w = exp2f(v[u].w - m);
      rs += (v[u].x + v[u].y) + (v[u].z + v[u].w);
      row[(u ^ (h >> 1)) & 3] = v[u];
    }
    bsum[i * (HQ + 1) + h] = rs;                      // rows padded by one float
    l += rs;
  }
  lred[tid] = l;
}

constexpr int kSC = 32;                 // partial records per round of the normaliser
constexpr int kRingBytes = 144 * 1024;  // shared memory given to the TMA ring at most
constexpr int kMinStages = 2;

struct Params {
  int layer, n_seqs, cap;             // cap: blocks per CTA the buffers hold
  SeqSel sel;                          // the launch's sequences: b-th is sel.at(b)
  int ns;                              // ring stages
  const void* q;                       // [n_seqs][HQ][D] bf16
  float* out;                          // [n_seqs][HQ][D]
  float qk_scale;                      // log2(e) / sqrt(D)
  // Whole-CTA plan made on the host from the per-sequence block bounds (whole > 0):
  // sequence b owns CTAs [cst[b], cst[b+1]) and splits its blocks evenly over them.
  // The bounds hold for every later state the launch can see (a graph replays it), so
  // the plan stays valid; whole == 0 leaves the split to the device.
  int whole;
  int cst[kGridMax + 1];
  uint8_t cta_seq[kGridMax];           // whole plan: the b with cst[b] <= c < cst[b + 1]
  // Fused append (whole plan only): before attending, store one new token per sequence,
  // K and V rows [n_seqs][Hkv][D] in the input dtype, at position next_position.
  int fuse;
  const void* k_new;
  const void* v_new;
  // Block list (list_ids non-null): attend over the resident entries of the listed
  // blocks only, list_ids[b * list_stride + i] for i < list_count[b]; no masses.
  const int32_t* list_ids;
  const int32_t* list_count;
  int list_stride;
  float* tok_out;                      // optional: entry masses at [b][position] too
};

// Page of block k of sequence s for a block list: the slot rule of the mode, or the
// block table (H2O).  A block id out of range or not resident (H2O) is reported, and
// the block then reads page 0 with every position masked (k = -1).
__device__ __forceinline__ int32_t list_block(const Dev& d, int s, int32_t* k) {
  int32_t page = -1, slot;
  if (*k >= 0 && *k < d.max_blocks)
    page = d.mode == KVS_MODE_H2O ? d.block_table[(size_t)s * d.max_blocks + *k]
                                  : page_of(d, s, (int64_t)*k * kBlock, &slot);
  if (page < 0 || page >= d.num_pages) {
    set_error(d, kErrState);
    *k = -1;
    page = 0;
  }
  return page;
}

// Shared-memory carve-up (byte offsets from a 1024-aligned base); the ring comes first
// so every stage keeps the 1024-byte alignment the 128-byte swizzle needs.
struct SmemPlan {
  size_t ring, sscale, bars, seqb, blk, prefix, mbuf, lred, hv, flag, pm, bsum, obuf, lg, total;
};

__host__ __device__ inline size_t up16(size_t x) { return (x + 15) & ~size_t(15); }

// whole: the whole-CTA plan, whose output reduction buffer reuses the ring (nothing is
// in flight there once every consumer has finished the V pass of its one segment).
__host__ __device__ inline SmemPlan plan_smem(int hkv, bool fp8, bool lsmem, int cap, int n_seqs, int ns,
                                             bool whole) {
  const int HQ = hkv * kG, WPK = kNCW / hkv;
  const size_t blk = (size_t)hkv * kBlock * kD * (fp8 ? 1 : 2);
  const size_t sb = kStageBytes / blk;
  SmemPlan p;
  size_t o = 0;
  p.ring = o;   o += (size_t)ns * sb * blk;
  p.sscale = o; o += (size_t)ns * sb * kBlock * 4;
  p.bars = o;   o += (size_t)(2 * ns + 2) * 8;                   // full, empty, append done, normaliser
  p.seqb = o;   o = up16(o + (size_t)n_seqs * sizeof(SeqBlocks));
  p.blk = o;    o = up16(o + (size_t)5 * cap * 4);
  p.prefix = o; o = up16(o + (size_t)(n_seqs + 1) * 4);
  p.mbuf = o;   o += (size_t)WPK * HQ * 4;
  p.lred = o;   o += (size_t)kNCW * 32 * 4;
  p.hv = o;     o += (size_t)4 * HQ * 4;
  p.flag = o;   o += 16;
  p.pm = o;     o += (size_t)kSC * HQ * 4;
  p.bsum = o;   o = up16(o + (size_t)cap * (HQ + 1) * 4);
  p.obuf = whole ? p.ring : o;
  o += (WPK == 2 && !whole ? (size_t)hkv * 32 * 32 * 4 : 0);
  p.lg = o;     o += lsmem ? (size_t)cap * (HQ * kBlock + kLgPad) * 4 : 0;
  p.total = o + 1024;                       // alignment slack
  return p;
}

template <int HKV, bool FP8, bool LSMEM>
// 10 warps: two of the 4 schedulers hold 3 of them, and each scheduler has 16K
// registers, so 168 per thread is the most one CTA per SM can have
__global__ void __maxnreg__(168)
attend_tc_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                 const Dev d, const Params P) {
  using C = Cfg<HKV, FP8>;
  constexpr int HQ = C::HQ, WPK = C::WPK;
  const int NS = P.ns;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const SmemPlan sp = plan_smem(HKV, FP8, LSMEM, P.cap, P.n_seqs, NS, P.whole != 0);
  uint8_t* ring = smem + sp.ring;
  float* sscale = reinterpret_cast<float*>(smem + sp.sscale);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + sp.bars);          // full[NS], empty[NS], app
  SeqBlocks* seqb = reinterpret_cast<SeqBlocks*>(smem + sp.seqb);        // [n_seqs]
  int32_t* blk_id = reinterpret_cast<int32_t*>(smem + sp.blk);
  int32_t* blk_page = blk_id + P.cap;
  int32_t* blk_seq = blk_page + P.cap;
  int32_t* ticket = blk_seq + P.cap;                                   // arrival order, by segment start
  int32_t* ppage = ticket + P.cap;                                     // whole plan: the producer's pages
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + sp.prefix);       // [n_seqs + 1]
  float* mbuf = reinterpret_cast<float*>(smem + sp.mbuf);              // [WPK][HQ]
  float* lred = reinterpret_cast<float*>(smem + sp.lred);              // [consumer threads]
  float* mseg = reinterpret_cast<float*>(smem + sp.hv);                // [HQ]
  float* cfac = mseg + HQ;                                             // [HQ]
  float* gmax = cfac + HQ;                                             // [HQ]
  float* ginv = gmax + HQ;                                             // [HQ]
  int32_t* flag = reinterpret_cast<int32_t*>(smem + sp.flag);
  float* pm = reinterpret_cast<float*>(smem + sp.pm);                  // [kSC][HQ]
  float* bsum = reinterpret_cast<float*>(smem + sp.bsum);              // [cap][HQ]
  float* obuf = reinterpret_cast<float*>(smem + sp.obuf);              // WPK==2: [HKV][32][32]
  float* lg_smem = reinterpret_cast<float*>(smem + sp.lg);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, G = gridDim.x;
  const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + NS), app_bar = smem_u32(bars + 2 * NS);
  const uint32_t norm_bar = smem_u32(bars + 2 * NS + 1);
  // Whole plan with waits: the CTA holds one segment, publishes its softmax statistics
  // (m, l) before the V pass, and the normaliser warp combines the sequence's
  // statistics into the global normaliser while the consumers run the V pass.
  const bool early = P.whole && d.spin_limit >= 0;

  if (warp == kProducer && lane == 0) {     // fetch the two tensor maps before the first copy
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
    asm volatile("prefetch.tensormap [%0];" :: "l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
  }
  // barriers touch shared memory only: set them up while the previous kernel finishes
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(full0 + 8 * s, 1);
      mbar_init(empty0 + 8 * s, kNCW);      // every consumer warp releases every stage
    }
    mbar_init(app_bar, 1);
    mbar_init(norm_bar, 32);                // every lane of the normaliser warp
    flag[1] = 0;                            // normaliser valid (set by the normaliser warp)
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  // everything below may read what the previous kernel of the stream wrote; let the next
  // kernel's launch begin now (it too waits for this one before reading anything)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

#ifdef KVS_DEBUG
  // every sequence id of a device list in range, or nobody touches anything
  {
    bool ids_ok = true;
    for (int b = 0; b < P.n_seqs; ++b) {
      const int s = P.sel.at(b);
      ids_ok = ids_ok && s >= 0 && s < d.max_seqs;
    }
    if (!ids_ok) {
      if (tid == 0) set_error(d, kErrBounds);
      return;
    }
  }
#endif
  // Fused append: the normaliser warp of the CTA that will hold the newest block (the
  // sequence's last CTA when every CTA has blocks) reads the new K and V rows now,
  // before this SM's copies queue up ahead of any load.
  constexpr int kNch = HKV * kD / 8 / 32;   // 8-value chunks per lane of one position
  uint4 knew[kNch], vnew[kNch];
  bool preloaded = false;
  if (P.fuse && warp == kNormWarp && c < P.cst[P.n_seqs]) {
    const int b = P.cta_seq[c];
    if (c == P.cst[b + 1] - 1) {
      const size_t src_elem = (size_t)b * HKV * kD;
      load_position_bf16(P.k_new, src_elem, lane, knew);
      load_position_bf16(P.v_new, src_elem, lane, vnew);
      preloaded = true;
    }
  }

  // ---------------------------------------------------------------- partition
  int x0 = 0;                               // whole plan: block index within the sequence
  int nblk = 0, cseq = -1;                  // cseq: the CTA's one sequence (whole plan)
  int q = 0, r = 0;                         // device split: T = q * G + r
  SeqBlocks sbw = {};                       // whole plan: the CTA's sequence
  int wseq = -1;                            // whole plan: the sequence whose CTAs include c
  bool appends = false;                     // fused append: this CTA stores the new token
  if (P.whole) {
    if (c < P.cst[P.n_seqs]) {
      const int lo = P.cta_seq[c];          // one lookup (a search costs a chain of loads)
      wseq = lo;
      int64_t nxt = d.next_pos[(size_t)P.layer * d.max_seqs + P.sel.at(lo)];
      // fused append: attend over the state after the new position (the host checked the
      // capacity; a state that disagrees skips the append and reports it)
      const bool grow = P.fuse && nxt < d.max_positions;
      if (P.fuse && !grow && tid == 0) set_error(d, kErrCapacity);
      sbw = seq_blocks_at(d, P.sel.at(lo), grow ? nxt + 1 : nxt);
      if (P.list_ids) sbw.n = min(max(P.list_count[lo], 0), P.list_stride);
      const int cb = P.cst[lo + 1] - P.cst[lo], rk = c - P.cst[lo];
      const int qb = sbw.n / cb, rb = sbw.n % cb;
      x0 = rk * qb + (rk < rb ? rk : rb);
      nblk = qb + (rk < rb ? 1 : 0);
      if (nblk > 0) cseq = lo;
      appends = grow && nblk > 0 && x0 + nblk == sbw.n;   // holds the newest block
      if (tid == 0) seqb[lo] = sbw;
    }
  } else {
    if (warp == 0) {
      int run = 0;
      for (int b0 = 0; b0 < P.n_seqs; b0 += 32) {
        const int b = b0 + lane;
        int nb = 0;
        if (b < P.n_seqs) {
          SeqBlocks sb = seq_blocks(d, P.layer, P.sel.at(b));
          if (P.list_ids) sb.n = min(max(P.list_count[b], 0), P.list_stride);
          seqb[b] = sb;
          nb = sb.n;
        }
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
    const int T = prefix[P.n_seqs];
    q = T / G;
    r = T % G;
    x0 = c * q + (c < r ? c : r);
    nblk = q + (c < r ? 1 : 0);
  }
  if (nblk > P.cap) {                       // the host's bound was too small
    if (tid == 0) set_error(d, kErrCapacity);
    return;
  }
  if (cseq >= 0) {
    for (int i = warp < kNCW ? tid : nblk; i < nblk; i += kNCW * 32) {
      int32_t page, k;
      if (P.list_ids) {
        k = P.list_ids[(size_t)cseq * P.list_stride + x0 + i];
        page = list_block(d, P.sel.at(cseq), &k);
      } else {
        k = block_at(d, P.sel.at(cseq), sbw, x0 + i, &page);
      }
      blk_id[i] = k;
      blk_page[i] = page;
      blk_seq[i] = cseq;
    }
  } else {
    for (int i = tid; i < nblk; i += kThreads) {
      const int x = x0 + i;
      int lo = 0, hi = P.n_seqs - 1;        // last b with prefix[b] <= x
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= x) lo = mid; else hi = mid - 1;
      }
      int32_t page, k;
      if (P.list_ids) {
        k = P.list_ids[(size_t)lo * P.list_stride + x - prefix[lo]];
        page = list_block(d, P.sel.at(lo), &k);
      } else {
        k = block_at(d, P.sel.at(lo), seqb[lo], x - prefix[lo], &page);
      }
      blk_id[i] = k;
      blk_page[i] = page;
      blk_seq[i] = lo;
    }
  }
  // the split plan's lists are everybody's; the whole plan's are the consumers' (they
  // meet at their own barrier) and the producer builds its page list itself
  if (!P.whole) __syncthreads();
  int32_t* const ctr_base = d.counters;     // sequence s: arrivals [s * kCounterInts], departures + kDepartAt
  if (nblk == 0) {
    // A CTA of the whole plan with no block still read its sequence's next position:
    // it departs too, so that the last CTA to leave knows every reader is done.
    if (wseq >= 0 && tid == 0) {
      const int s = P.sel.at(wseq), cb = P.cst[wseq + 1] - P.cst[wseq];
      if (atomicAdd(ctr_base + (size_t)s * kCounterInts + kDepartAt, 1) == cb - 1) {
        ctr_base[(size_t)s * kCounterInts] = 0;
        ctr_base[(size_t)s * kCounterInts + kDepartAt] = 0;
        ctr_base[(size_t)s * kCounterInts + kMlAt] = 0;
        if (P.fuse && sbw.next > 0) d.next_pos[(size_t)P.layer * d.max_seqs + s] = sbw.next;
      }
    }
    return;
  }

  float* lgbase = LSMEM ? lg_smem : d.logit_scratch + (size_t)c * P.cap * lg_block<HQ>();
  const size_t lay_slot = (size_t)P.layer * d.slot_layer_elems;
  float* partials = d.partials;

  // ================================================================ producer warp
  if (warp == kProducer) {
    if (P.whole) {
      // its own page list, so the first copies go out without waiting for the consumers
      for (int i = lane; i < nblk; i += 32) {
        int32_t page;
        if (P.list_ids) {
          int32_t k = P.list_ids[(size_t)cseq * P.list_stride + x0 + i];
          page = list_block(d, P.sel.at(cseq), &k);
        } else {
          block_at(d, P.sel.at(cseq), sbw, x0 + i, &page);
        }
        ppage[i] = page;
      }
      __syncwarp();
    }
    if (lane == 0) {
      const uint64_t pol = evict_first_policy();
      const int32_t* pages = P.whole ? ppage : blk_page;
      uint32_t ctr = 0;
      int i0 = 0;
      while (i0 < nblk) {
        int i1 = i0 + 1;
        if (P.whole) i1 = nblk;                 // one segment
        else while (i1 < nblk && blk_seq[i1] == blk_seq[i0]) ++i1;
        for (int ph = 0; ph < 2; ++ph) {
          const CUtensorMap* map = ph == 0 ? &tmk : &tmv;
          const float* scales = ph == 0 ? d.k_scales : d.v_scales;
          for (int g0 = i0; g0 < i1; g0 += C::SB, ++ctr) {      // one stage = up to SB blocks
            const int nb = min(C::SB, i1 - g0);
            const uint32_t st = ctr % NS, round = ctr / NS;
            if (round > 0 && !mbar_wait(empty0 + 8 * st, (round - 1) & 1)) set_error(d, kErrTimeout);
            // the newest block (the CTA's last) is copied only once the fused append is stored
            if (appends && g0 + nb == nblk && !mbar_wait(app_bar, 0)) set_error(d, kErrTimeout);
            const uint32_t fb = full0 + 8 * st;
            mbar_expect_tx(fb, nb * (C::BLK + (FP8 ? kBlock * 4 : 0)));
            for (int j = 0; j < nb; ++j) {
              int page = pages[g0 + j];
              if (!KVS_DCHECK(d, page >= 0 && page < d.num_pages)) page = 0;
              const uint32_t dst = smem_u32(ring + (size_t)st * C::STAGE + (size_t)j * C::BLK);
              tma_load_4d(dst, map, 0, 0, 0, page, fb, pol);
              if constexpr (FP8) {
                bulk_load(smem_u32(sscale + (st * C::SB + j) * kBlock), scales + lay_slot + (size_t)page * kBlock,
                          kBlock * 4, fb);
              } else {
                tma_load_4d(dst + C::HALF, map, 64, 0, 0, page, fb, pol);
              }
            }
          }
        }
        i0 = i1;
      }
    }
    __syncwarp();                               // lanes 1..31 wait for the issuing lane
    if (early) {
      // publish the partial output rows once this CTA's consumers have written them
      named_sync(kBarOut, kPubThreads);
      if (lane == 0) red_release_add(ctr_base + (size_t)(P.sel.at(cseq)) * kCounterInts, 1);
    }
  } else if (warp == kNormWarp) {
    // ============================================================== normaliser warp
    if (appends) {
      // fused append of position next (the state attended is next + 1), stored exactly
      // as the append kernel does while the consumers already run the K pass; the
      // producer copies the newest block only after app_bar.  Every storing lane orders
      // its generic-proxy stores before those copies.
      const int s = P.sel.at(cseq);
      const int64_t pnew = sbw.next - 1;
      int32_t slot;
      int32_t page = page_of(d, s, pnew, &slot);
      const bool have_page = page >= 0 && page < d.num_pages;   // (H2O: allocated before the launch)
      if (!have_page) {                         // the pool ran dry: reported, nothing stored
        if (lane == 0) set_error(d, kErrCapacity);
        page = 0;
      }
      const size_t src_elem = (size_t)cseq * HKV * kD;
      const size_t lay_slot0 = (size_t)P.layer * d.slot_layer_elems + (size_t)page * kBlock;
      if (!preloaded) {                         // (a sequence with fewer blocks than CTAs)
        load_position_bf16(P.k_new, src_elem, lane, knew);
        load_position_bf16(P.v_new, src_elem, lane, vnew);
      }
      for (int kv = 0; kv < 2 && have_page; ++kv) {
        uint8_t* base = (kv == 0 ? d.k_pages : d.v_pages) + P.layer * d.page_layer_bytes + (size_t)page * d.page_bytes;
        float* scales = kv == 0 ? d.k_scales : d.v_scales;
        store_position_regs<FP8 ? KVS_E4M3 : KVS_BF16>(d, kv == 0 ? knew : vnew, base,
                                                        scales ? scales + lay_slot0 + slot : nullptr, slot, lane);
      }
      if (lane == 0 && have_page) d.pos[lay_slot0 + slot] = pnew;
      asm volatile("fence.proxy.async.global;" ::: "memory");
      __syncwarp();
      if (lane == 0) {
        __threadfence();
        mbar_arrive(app_bar);
      }
    }
    if (early) {
      // Global normaliser of the CTA's sequence, while the consumers run the V pass:
      // wait (bounded) until every CTA of the sequence has published its statistics,
      // then lane h merges head h's records in record order.  Record k is the
      // sequence's k-th CTA: per head the running max m and l = sum exp2(s - m).
      const int b = cseq, s = P.sel.at(b);
      const int cb = P.cst[b + 1] - P.cst[b], cf = P.cst[b];
      const int S = sbw.n >= cb ? cb : sbw.n;
      int ok = 1;
      named_sync(kBarMl, kPubThreads);          // this CTA's consumers wrote its words
      if (lane == 0) {
        red_release_add(ctr_base + (size_t)s * kCounterInts + kMlAt, 1);
        ok = wait_at_least(ctr_base + (size_t)s * kCounterInts + kMlAt, S, d.spin_limit) ? 1 : 0;
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (ok) {
        const unsigned long long* rec0 = d.part_ml + (size_t)(cf + b) * HQ;   // record k, head h: [k * HQ + h]
        const int own = c - cf;
#pragma unroll 1
        for (int u = 0; u < HQ / 32; ++u) {
          const int h = lane + 32 * u;
          if (S <= kSC) {
            // every record in registers: one round of loads
            unsigned long long w[kSC];
#pragma unroll
            for (int k = 0; k < kSC; ++k) w[k] = k < S ? __ldcg(rec0 + (size_t)k * HQ + h) : 0ull;
            float M = -INFINITY;
#pragma unroll
            for (int k = 0; k < kSC; ++k)
              if (k < S) M = fmaxf(M, __uint_as_float((uint32_t)w[k]));
            float Ls = 0.f;
#pragma unroll
            for (int k = 0; k < kSC; ++k)
              if (k < S) Ls += __uint_as_float((uint32_t)(w[k] >> 32)) * exp2f(__uint_as_float((uint32_t)w[k]) - M);
            const float inv = 1.0f / Ls;
#pragma unroll
            for (int k = 0; k < kSC; ++k) {
              if (k < S) {
                const float f = exp2f(__uint_as_float((uint32_t)w[k]) - M) * inv;
                pm[k * HQ + h] = f;
                if (k == own) cfac[h] = f;
              }
            }
            gmax[h] = M;
            ginv[h] = inv;
          } else {
            float M = -INFINITY, Ls = 0.f;
            for (int k0 = 0; k0 < S; k0 += 8) {
              unsigned long long w[8];
#pragma unroll
              for (int j = 0; j < 8; ++j) w[j] = __ldcg(rec0 + (size_t)min(k0 + j, S - 1) * HQ + h);
              float cm = -INFINITY;
#pragma unroll
              for (int j = 0; j < 8; ++j)
                if (k0 + j < S) cm = fmaxf(cm, __uint_as_float((uint32_t)w[j]));
              const float nm = fmaxf(M, cm);
              float part = 0.f;
#pragma unroll
              for (int j = 0; j < 8; ++j)
                if (k0 + j < S) part += __uint_as_float((uint32_t)(w[j] >> 32)) * exp2f(__uint_as_float((uint32_t)w[j]) - nm);
              Ls = Ls * exp2f(M - nm) + part;
              M = nm;
            }
            const float inv = 1.0f / Ls;
            cfac[h] = exp2f(__uint_as_float((uint32_t)__ldcg(rec0 + (size_t)own * HQ + h)) - M) * inv;
            gmax[h] = M;
            ginv[h] = inv;
          }
        }
      } else if (lane == 0) {
        set_error(d, kErrTimeout);
      }
      if (lane == 0) flag[1] = ok;
      __syncwarp();
      mbar_arrive(norm_bar);                    // every lane, after its own writes
    }
  } else {
    // ============================================================== consumer warps
    const int kvh = warp % HKV, sub = warp / HKV;
    const int g = lane >> 2, t = lane & 3;
    if (P.whole) named_sync(1, kNCW * 32);      // the block lists are written
    uint32_t ctr = 0;
    int i0 = 0;
    while (i0 < nblk) {
      int i1 = i0 + 1;
      while (i1 < nblk && blk_seq[i1] == blk_seq[i0]) ++i1;
      const int b = blk_seq[i0], s = P.sel.at(b);
      const SeqBlocks sb = seqb[b];

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
      for (int g0 = i0; g0 < i1; g0 += C::SB, ++ctr) {     // one ring stage: up to SB blocks
        const int nb = min(C::SB, i1 - g0);
        const uint32_t st = ctr % NS, round = ctr / NS;
        if (!mbar_wait(full0 + 8 * st, round & 1)) set_error(d, kErrTimeout);
        const uint8_t* stage = ring + (size_t)st * C::STAGE;
        const float* sst = sscale + st * C::SB * kBlock;
        int j = sub;
        for (; j + WPK < nb; j += 2 * WPK)
          qk_blocks<HKV, FP8, 2>(stage, sst, j, g0 + j, blk_id, qf, lgbase, kvh, lane, sb.lo, sb.next, P.qk_scale, mx0, mx1);
        if (j < nb)
          qk_blocks<HKV, FP8, 1>(stage, sst, j, g0 + j, blk_id, qf, lgbase, kvh, lane, sb.lo, sb.next, P.qk_scale, mx0, mx1);
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

      // ------------------------------------------------------------ weights
      // p = exp2(s - m) in place, block sums, and this segment's (m, l) per head as one
      // 64-bit word in a compact array of its own, published before the V pass
      weights_sweep<HQ>(lgbase, bsum, lred, mseg, i0, i1, tid);
      named_sync(1, kNCW * 32);
      if (tid < HQ) {
        float l = 0.f;
        for (int k = tid; k < kNCW * 32; k += HQ) l += lred[k];
        d.part_ml[(size_t)(c + b) * HQ + tid] = ((unsigned long long)__float_as_uint(l) << 32) | __float_as_uint(mseg[tid]);
      }
      // whole plan: hand the words to the normaliser warp, which publishes them (no
      // consumer waits on a fence; the producer warp does the same for the output rows)
      if (early) named_arrive(kBarMl, kPubThreads);

      // ------------------------------------------------------------ pass 2: V
      float o[8][4];
#pragma unroll
      for (int mb = 0; mb < 8; ++mb) o[mb][0] = o[mb][1] = o[mb][2] = o[mb][3] = 0.f;
      for (int g0 = i0; g0 < i1; g0 += C::SB, ++ctr) {
        const int nb = min(C::SB, i1 - g0);
        const uint32_t st = ctr % NS, round = ctr / NS;
        if (!mbar_wait(full0 + 8 * st, round & 1)) set_error(d, kErrTimeout);
        const uint8_t* stage = ring + (size_t)st * C::STAGE;
        const float* sst = sscale + st * C::SB * kBlock;
        int j = sub;
        for (; j + WPK < nb; j += 2 * WPK)
          pv_blocks<HKV, FP8, 2>(stage, sst, j, g0 + j, lgbase, kvh, lane, o);
        if (j < nb)
          pv_blocks<HKV, FP8, 1>(stage, sst, j, g0 + j, lgbase, kvh, lane, o);
        __syncwarp();
        if (lane == 0) mbar_arrive(empty0 + 8 * st);
      }
      if (WPK == 2 && P.whole) named_sync(1, kNCW * 32);   // the ring is free: obuf lives there
      if (WPK == 2 && sub == 1) {
#pragma unroll
        for (int mb = 0; mb < 8; ++mb)
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) obuf[(kvh * 32 + mb * 4 + rr) * 32 + lane] = o[mb][rr];
      }
      if (WPK == 2) named_sync(2 + kvh, 64);       // the two warps of KV head kvh
      if (sub == 0) {
        if (WPK == 2) {
#pragma unroll
          for (int mb = 0; mb < 8; ++mb)
#pragma unroll
            for (int rr = 0; rr < 4; ++rr) o[mb][rr] += obuf[(kvh * 32 + mb * 4 + rr) * 32 + lane];
        }
        const float ofold = FP8 ? 1.0f / kVFold : 1.0f;
        float* rec = partials + (size_t)(c + b) * HQ * kD;
        const int ha = kvh * kG + 2 * t;
        if constexpr (FP8) {
          // accumulator rows g, g+8 of tile mb hold dims 16g + 2mb and 16g + 2mb + 1:
          // this thread owns dims 16g .. 16g+15 of heads ha and ha+1 (four 16-byte rows)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float* ra = rec + (size_t)ha * kD + 16 * g + 4 * j;
            *reinterpret_cast<float4*>(ra) = make_float4(o[2 * j][0] * ofold, o[2 * j][2] * ofold,
                                                         o[2 * j + 1][0] * ofold, o[2 * j + 1][2] * ofold);
            *reinterpret_cast<float4*>(ra + kD) = make_float4(o[2 * j][1] * ofold, o[2 * j][3] * ofold,
                                                              o[2 * j + 1][1] * ofold, o[2 * j + 1][3] * ofold);
          }
        } else {
#pragma unroll
          for (int mb = 0; mb < 8; ++mb) {
            const int da = 16 * mb + g, db = da + 8;   // dims of accumulator rows g and g+8
            rec[(size_t)ha * kD + da] = o[mb][0];
            rec[(size_t)(ha + 1) * kD + da] = o[mb][1];
            rec[(size_t)ha * kD + db] = o[mb][2];
            rec[(size_t)(ha + 1) * kD + db] = o[mb][3];
          }
        }
        // Each writer warp releases its own rows and arrives (HKV arrivals per
        // CTA), without a return value: no CTA barrier on the way.  One poller per CTA
        // reads the counter (every thread polling the records themselves floods their
        // few L2 lines).
        if (d.spin_limit >= 0 && !early) {
          __syncwarp();
          if (lane == 0) {
            __threadfence();
            red_add(ctr_base + (size_t)s * kCounterInts, 1);
          }
        }
      }
      if (early) named_arrive(kBarOut, kPubThreads);   // the producer warp publishes the rows
      if (d.spin_limit < 0) {
        // nobody waits: one arrival per CTA, with its order, after a CTA barrier; only
        // the last CTA to arrive goes on
        named_sync(1, kNCW * 32);
        if (tid == 0) {
          __threadfence();
          ticket[i0] = atomicAdd(ctr_base + (size_t)s * kCounterInts, 1);
        }
      }
      i0 = i1;
    }

    // ================================================================ epilogue
    i0 = 0;
    while (i0 < nblk) {
      int i1 = i0 + 1;
      while (i1 < nblk && blk_seq[i1] == blk_seq[i0]) ++i1;
      const int b = blk_seq[i0], s = P.sel.at(b);
      const SeqBlocks sb = seqb[b];
      int cf, S;                                   // the sequence's CTAs: cf .. cf + S - 1
      if (P.whole) {
        const int cb = P.cst[b + 1] - P.cst[b];
        cf = P.cst[b];
        S = sb.n >= cb ? cb : sb.n;                // fewer blocks than CTAs: one block each
      } else {
        cf = cta_of(prefix[b], q, r);
        S = cta_of(prefix[b + 1] - 1, q, r) - cf + 1;
      }
      if (early) {
        // the normaliser warp has combined the normaliser during the V pass: wait for it
        // (bounded), and let every consumer thread take the same decision
        const bool w = mbar_wait(norm_bar, 0);
        if (!w) set_error(d, kErrTimeout);
        if (!named_sync_and(1, kNCW * 32, w && flag[1] != 0)) break;
      } else {
        if (tid == 0) {
          // spin_limit < 0: no wait at all, only the last CTA to arrive goes on
          const bool ok = d.spin_limit < 0 ? ticket[i0] == S - 1
                                           : wait_at_least(ctr_base + (size_t)s * kCounterInts, S * HKV, d.spin_limit);
          flag[0] = ok ? 1 : 0;
          if (!ok) set_error(d, kErrTimeout);
        }
        named_sync(1, kNCW * 32);
        if (!flag[0]) break;

        // global normaliser: warp w takes heads w, w + 8, ...; lane k reads the (m, l)
        // word of record k (rounds of 32 records when S > 32); with S <= kSC the
        // per-record output factors stay in pm
        {
          constexpr int HPW = HQ / kNCW;
          float M[HPW], Ls[HPW], mk[HPW], mo[HPW];
  #pragma unroll
          for (int u = 0; u < HPW; ++u) { M[u] = -INFINITY; Ls[u] = 0.f; mk[u] = -INFINITY; mo[u] = -INFINITY; }
          for (int k0 = 0; k0 < S; k0 += 32) {
            const int k = k0 + lane;
            // every lane loads (lanes past S re-read record S-1 and ignore it), all loads
            // issued before any is used
            const unsigned long long* wp = d.part_ml + (size_t)(cf + min(k, S - 1) + b) * HQ + warp;
            unsigned long long w[HPW];
  #pragma unroll
            for (int u = 0; u < HPW; ++u) w[u] = __ldcg(wp + u * kNCW);
            const int own = c - cf - k0;
  #pragma unroll
            for (int u = 0; u < HPW; ++u) {
              const float m = k < S ? __uint_as_float((uint32_t)w[u]) : -INFINITY;
              const float l = k < S ? __uint_as_float((uint32_t)(w[u] >> 32)) : 0.f;
              float cm = m;
  #pragma unroll
              for (int o2 = 16; o2 > 0; o2 >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xffffffffu, cm, o2));
              const float nm = fmaxf(M[u], cm);
              float part = l * exp2f(m - nm);              // 0 for lanes past S
  #pragma unroll
              for (int o2 = 16; o2 > 0; o2 >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o2);
              Ls[u] = Ls[u] * exp2f(M[u] - nm) + part;
              M[u] = nm;
              mk[u] = m;
              if (own >= 0 && own < 32) mo[u] = __shfl_sync(0xffffffffu, m, own);
            }
          }
  #pragma unroll
          for (int u = 0; u < HPW; ++u) {
            const int h = warp + u * kNCW;
            const float inv = 1.0f / Ls[u];
            if (S <= kSC && lane < S) pm[lane * HQ + h] = exp2f(mk[u] - M[u]) * inv;
            if (lane == 0) {
              cfac[h] = exp2f(mo[u] - M[u]) * inv;
              gmax[h] = M[u];
              ginv[h] = inv;
            }
          }
        }
        named_sync(1, kNCW * 32);
      }
      const bool fac_in_smem = S <= kSC;

      if (warp < kNCW / 2) {
        if (!P.list_ids) {                         // (a block-list attend records no mass)
        // masses: lane = (block bi = lane >> 2 of 8 per warp round, position chunk
        // c4 = lane & 3); each lane walks all heads for its 4 positions (no shuffles),
        // the head factors read 8 at a time; the padded block strides keep the 16-byte
        // weight reads and the bsum reads free of bank conflicts
        const int bi = lane >> 2, c4 = lane & 3;
        for (int ib = i0 + warp * 8; ib < i1; ib += (kNCW / 2) * 8) {
          const int i = ib + bi;
          if (i < i1) {
            const float* lgi = lgbase + (size_t)i * lg_block<HQ>();
            const float* bsi = bsum + i * (HQ + 1);
            float4 tau = make_float4(0.f, 0.f, 0.f, 0.f);   // entry: sum over heads
            float bm = 0.f;                                 // block: max over heads
#pragma unroll
            for (int u0 = 0; u0 < HQ; u0 += 8) {
              const float4 fa = *reinterpret_cast<const float4*>(cfac + u0);
              const float4 fb = *reinterpret_cast<const float4*>(cfac + u0 + 4);
              const float f[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                const int h = u0 + u;
                const float4 v = *reinterpret_cast<const float4*>(lgi + h * kBlock + (((c4 ^ (h >> 1)) & 3) << 2));
                tau.x += v.x * f[u];
                tau.y += v.y * f[u];
                tau.z += v.z * f[u];
                tau.w += v.w * f[u];
                bm = fmaxf(bm, bsi[h] * f[u]);
              }
            }
            const int64_t p0 = (int64_t)blk_id[i] * kBlock + 4 * c4;   // slots p % 16
            float* dst = d.tok_mass + lay_slot + (size_t)blk_page[i] * kBlock + 4 * c4;
            if (p0 >= sb.lo && p0 + 3 < sb.next) {
              *reinterpret_cast<float4*>(dst) = tau;
            } else {
              if (p0 >= sb.lo && p0 < sb.next) dst[0] = tau.x;
              if (p0 + 1 >= sb.lo && p0 + 1 < sb.next) dst[1] = tau.y;
              if (p0 + 2 >= sb.lo && p0 + 2 < sb.next) dst[2] = tau.z;
              if (p0 + 3 >= sb.lo && p0 + 3 < sb.next) dst[3] = tau.w;
            }
            if (P.tok_out) {                     // the caller's copy, by absolute position
              float* to = P.tok_out + (size_t)b * d.max_positions + p0;
              if (p0 >= sb.lo && p0 < sb.next) to[0] = tau.x;
              if (p0 + 1 >= sb.lo && p0 + 1 < sb.next) to[1] = tau.y;
              if (p0 + 2 >= sb.lo && p0 + 2 < sb.next) to[2] = tau.z;
              if (p0 + 3 >= sb.lo && p0 + 3 < sb.next) to[3] = tau.w;
            }
            if (c4 == 0)
              d.blk_mass[(size_t)P.layer * d.blk_layer_elems + (size_t)s * d.max_blocks + blk_id[i]] = bm;
            if (c4 == 1)                          // per-head profiles: the head's in-block weight
              for (int jh = 0; jh < d.n_hprof; ++jh)
                if (d.hprof_layer[jh] == P.layer)
                  record_head(d, P.layer, s, blk_id[i], d.hprof_head[jh], bsi[d.hprof_head[jh]] * cfac[d.hprof_head[jh]]);
          }
        }
        }
      } else {
        bool out_ready = true;
        if (early) {
          // only the output combine needs the other CTAs' partial rows: wait for them here
          if (warp == kNCW / 2 && lane == 0) {
            const bool ok = wait_at_least(ctr_base + (size_t)s * kCounterInts, S, d.spin_limit);
            flag[2] = ok ? 1 : 0;
            if (!ok) set_error(d, kErrTimeout);
          }
          named_sync(kBarOutWarps, (kNCW / 2) * 32);
          out_ready = flag[2] != 0;
        }
        // output: this CTA combines heads h with h % S == its rank among the sequence's
        // CTAs, 4 dimensions per thread
        constexpr int D4 = kD / 4;
        constexpr size_t kRec4 = (size_t)HQ * kD / 4;      // float4 between a head's records
        const int rank = c - cf;
        const int nh = rank < HQ && out_ready ? (HQ - rank + S - 1) / S : 0;
        const int ot = tid - (kNCW / 2) * 32;
        for (int idx = ot; idx < nh * D4; idx += (kNCW / 2) * 32) {
          const int h = rank + (idx / D4) * S, d4 = idx % D4;
          const float4* r0 = reinterpret_cast<const float4*>(partials + ((size_t)(cf + b) * HQ + h) * kD) + d4;
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
          if (fac_in_smem) {
            for (int k0 = 0; k0 < S; k0 += 16) {
              // 16 unconditional loads in flight (indices past S re-read record S-1,
              // which then gets factor 0)
              float4 ov[16];
#pragma unroll
              for (int u = 0; u < 16; ++u) ov[u] = __ldcg(r0 + (size_t)min(k0 + u, S - 1) * kRec4);
#pragma unroll
              for (int u = 0; u < 16; ++u) {
                const float f = (k0 + u < S) ? pm[min(k0 + u, S - 1) * HQ + h] : 0.f;
                acc.x += ov[u].x * f;
                acc.y += ov[u].y * f;
                acc.z += ov[u].z * f;
                acc.w += ov[u].w * f;
              }
            }
          } else {
            const float M = gmax[h], inv = ginv[h];
            for (int k = 0; k < S; ++k) {
              const float f = exp2f(__uint_as_float((uint32_t)__ldcg(d.part_ml + (size_t)(cf + k + b) * HQ + h)) - M);
              const float4 v = __ldcg(r0 + (size_t)k * kRec4);
              acc.x += v.x * f;
              acc.y += v.y * f;
              acc.z += v.z * f;
              acc.w += v.w * f;
            }
            acc.x *= inv;
            acc.y *= inv;
            acc.z *= inv;
            acc.w *= inv;
          }
          reinterpret_cast<float4*>(P.out + ((size_t)b * HQ + h) * kD)[d4] = acc;
        }
      }
      // Departure: once all S CTAs have departed, all have passed the wait and the last
      // one resets the counters.  (Issuing the departure right after the normaliser and
      // looking at its ticket only here measured 50% slower in graphs of launches.)
      named_sync(1, kNCW * 32);                    // also: the next segment reuses pm, cfac, flag
      if (early && !flag[2]) break;                // the output wait ran out (reported)
      const int departs = P.whole ? P.cst[b + 1] - P.cst[b] : S;   // whole plan: empty CTAs depart too
      if (tid == 0 && atomicAdd(ctr_base + (size_t)s * kCounterInts + kDepartAt, 1) == departs - 1) {
        ctr_base[(size_t)s * kCounterInts] = 0;    // last CTA of the sequence to leave
        ctr_base[(size_t)s * kCounterInts + kDepartAt] = 0;
        ctr_base[(size_t)s * kCounterInts + kMlAt] = 0;
        if (P.fuse) d.next_pos[(size_t)P.layer * d.max_seqs + s] = sb.next;   // every reader is done
      }
      i0 = i1;
    }
  }
  __syncthreads();
}

size_t tc_smem_limit() { return 227 * 1024; }

// Ring stages that fit next to the rest of the carve-up (0 if fewer than kMinStages).
int ring_stages(int hkv, bool fp8, bool lsmem, int cap, int n_seqs, bool whole) {
  const size_t blk = (size_t)hkv * kBlock * kD * (fp8 ? 1 : 2);
  const size_t sb = kStageBytes / blk;
  const size_t stage = sb * blk;
  const size_t rest = plan_smem(hkv, fp8, lsmem, cap, n_seqs, 0, whole).total;
  if (rest >= tc_smem_limit()) return 0;
  size_t ns = (tc_smem_limit() - rest) / (stage + sb * kBlock * 4 + 16);
  ns = ns < (size_t)(kRingBytes / stage) ? ns : (size_t)(kRingBytes / stage);
  return ns >= (size_t)kMinStages ? (int)ns : 0;
}

template <int HKV, bool FP8, bool LSMEM>
cudaError_t launch_one(const CUtensorMap& tk, const CUtensorMap& tv, const Dev& d, const Params& P, int grid,
                       cudaStream_t st) {
  auto fn = attend_tc_kernel<HKV, FP8, LSMEM>;
  const size_t smem = plan_smem(HKV, FP8, LSMEM, P.cap, P.n_seqs, P.ns, P.whole != 0).total;
  static std::atomic<unsigned long long> optin{0};   // per device: opt-in to the full limit
  const cudaError_t oe = smem_optin_once(optin, fn, (int)tc_smem_limit());
  if (oe != cudaSuccess) return oe;
  if (smem > tc_smem_limit()) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  // cooperative: every CTA resident at once (the cross-CTA waits rely on it);
  // programmatic serialisation: the launch may begin while the previous kernel of the
  // stream finishes; the kernel waits for it (griddepcontrol.wait) before reading state
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, fn, tk, tv, d, P);
}

// Per-CTA block capacity a whole-CTA plan may use: up to a quarter more blocks than an
// even split, plus two.  (A batch of many sequences that each need a little more than
// two even shares, such as 64 sequences of 130 blocks on 152 CTAs, then gets two CTAs
// per sequence in a whole-CTA plan instead of the device split: measured 9 % faster per
// attend, and the append joins the launch.)
int wide_cap(int base) { return base + base / 4 + 2; }

// Whole CTAs per sequence, planned on the host from the per-sequence block bounds: the
// fewest blocks per CTA X <= cap_limit such that ceil(bound_b / X) CTAs for every
// sequence b take at most `grid` CTAs.  Fills P.cst, sets P.whole and P.cap = X; false
// (P unchanged) when no such X exists or the launch has more sequences than CTAs.
bool plan_whole(Params& P, const int32_t* bounds, int grid, int cap_limit) {
  if (P.n_seqs > grid || P.n_seqs > kGridMax) return false;
  int64_t T = 0;
  for (int b = 0; b < P.n_seqs; ++b) T += bounds[b] > 0 ? bounds[b] : 0;
  if (T <= 0) return false;
  auto ctas = [&](int x) {
    int64_t n = 0;
    for (int b = 0; b < P.n_seqs; ++b) n += (bounds[b] + x - 1) / x;
    return n;
  };
  int lo = (int)((T + grid - 1) / grid), hi = cap_limit;
  if (lo < 1) lo = 1;
  if (lo > hi || ctas(hi) > grid) return false;
  while (lo < hi) {
    const int mid = (lo + hi) / 2;
    if (ctas(mid) <= grid) hi = mid; else lo = mid + 1;
  }
  int run = 0;
  for (int b = 0; b < P.n_seqs; ++b) {
    P.cst[b] = run;
    for (int x = run; x < run + (bounds[b] + lo - 1) / lo && x < kGridMax; ++x) P.cta_seq[x] = (uint8_t)b;
    run += (bounds[b] + lo - 1) / lo;
  }
  P.cst[P.n_seqs] = run;
  P.whole = 1;
  P.cap = lo;
  return true;
}

template <int HKV, bool FP8>
cudaError_t launch_pick(const CUtensorMap& tk, const CUtensorMap& tv, const Dev& d, Params P, int grid,
                        cudaStream_t st) {
  P.ns = ring_stages(HKV, FP8, true, P.cap, P.n_seqs, P.whole != 0);
  if (P.ns > 0) return launch_one<HKV, FP8, true>(tk, tv, d, P, grid, st);
  P.ns = ring_stages(HKV, FP8, false, P.cap, P.n_seqs, P.whole != 0);
  if (P.ns == 0) return cudaErrorInvalidConfiguration;
  if ((size_t)grid * P.cap * lg_block<Cfg<HKV, FP8>::HQ>() > d.logit_scratch_elems) return cudaErrorInvalidConfiguration;
  return launch_one<HKV, FP8, false>(tk, tv, d, P, grid, st);
}

}  // namespace

bool tc_supported(int Hq, int Hkv, int D, int kv_dtype, int in_dtype, int window, int mode) {
  if (D != kD || Hq != Hkv * kG || (Hkv != 4 && Hkv != 8)) return false;
  if (in_dtype != KVS_BF16 || (kv_dtype != KVS_BF16 && kv_dtype != KVS_E4M3)) return false;
  if (mode == KVS_MODE_WINDOW && window % kBlock != 0) return false;
  return true;
}

// The driver's cuTensorMapEncodeTiled, looked up once (threads racing on the first
// lookup store the same pointer); null when the driver does not provide it.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static std::atomic<PFN_cuTensorMapEncodeTiled_v12000> encode_fn{nullptr};
  PFN_cuTensorMapEncodeTiled_v12000 encode = encode_fn.load(std::memory_order_acquire);
  if (!encode) {
    cudaDriverEntryPointQueryResult qr;
    void* fn = nullptr;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &qr);
    if (e != cudaSuccess || qr != cudaDriverEntryPointSuccess || !fn) return nullptr;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    encode_fn.store(encode, std::memory_order_release);
  }
  return encode;
}

// Tensor map over one layer's pages viewed as [num_pages][Hkv][16][D] elements; a box is
// one 16-token block of box_heads KV heads (128 bytes of each row).
cudaError_t make_page_map(CUtensorMap* map, const void* base, int num_pages, int Hkv, int kv_dtype, int box_heads) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  const bool fp8 = kv_dtype == KVS_E4M3;
  const int esz = fp8 ? 1 : 2;
  cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)kBlock, (cuuint64_t)Hkv, (cuuint64_t)num_pages};
  cuuint64_t strides[3] = {(cuuint64_t)kD * esz, (cuuint64_t)kBlock * kD * esz, (cuuint64_t)Hkv * kBlock * kD * esz};
  cuuint32_t box[4] = {(cuuint32_t)(fp8 ? 128 : 64), (cuuint32_t)kBlock, (cuuint32_t)box_heads, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult res = encode(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Blocks one CTA must hold for a launch whose resident blocks number at most T_bound.
int tc_cap(int64_t T_bound, int grid) { return (int)((T_bound + grid - 1) / grid); }

// opt.k_new / v_new non-null: append one token per sequence in the same launch (NONE
// and WINDOW modes, whole-CTA plan); cudaErrorNotSupported when that plan is not
// possible or its buffers do not fit.  opt.list_ids non-null: attend over the listed
// blocks only (bounds then bound the list lengths).
cudaError_t launch_attend_tc(const CUtensorMap& tk, const CUtensorMap& tv, const Dev& d, int layer,
                             SeqSel sel, int n_seqs, const void* q, float* out, const int32_t* bounds,
                             int grid, const AttendOpts& opt, cudaStream_t st) {
  const void* k_new = opt.k_new;
  const void* v_new = opt.v_new;
  Params P;
  P.layer = layer;
  P.sel = sel;
  P.n_seqs = n_seqs;
  P.tok_out = opt.tok_out;
  int64_t T_bound = 0;
  for (int b = 0; b < n_seqs; ++b) T_bound += bounds[b];
  const int cap0 = tc_cap(T_bound, grid) < 1 ? 1 : tc_cap(T_bound, grid);
  P.cap = cap0;
  P.ns = 0;
  P.q = q;
  P.out = out;
  P.qk_scale = kLog2e / sqrtf((float)kD);
  P.whole = 0;
  P.fuse = 0;
  P.k_new = P.v_new = nullptr;
  P.list_ids = opt.list_ids;
  P.list_count = opt.list_count;
  P.list_stride = opt.list_stride;
  const bool fp8 = d.kv_dtype == KVS_E4M3;
  auto pick = [&](const Params& PP) {
    if (d.Hkv == 4) return fp8 ? launch_pick<4, true>(tk, tv, d, PP, grid, st) : launch_pick<4, false>(tk, tv, d, PP, grid, st);
    return fp8 ? launch_pick<8, true>(tk, tv, d, PP, grid, st) : launch_pick<8, false>(tk, tv, d, PP, grid, st);
  };
  if (plan_whole(P, bounds, grid, wide_cap(cap0))) {
    if (k_new) {                            // fused append: whole plan only
      P.fuse = 1;
      P.k_new = k_new;
      P.v_new = v_new;
      const cudaError_t e = pick(P);
      return e == cudaErrorInvalidConfiguration ? cudaErrorNotSupported : e;
    }
    const cudaError_t e = pick(P);
    if (e != cudaErrorInvalidConfiguration) return e;
    P.whole = 0;                            // the plan's buffers do not fit: split on the device
    P.cap = cap0;
  }
  if (k_new) return cudaErrorNotSupported;
  return pick(P);
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
// and three counters per sequence (output arrivals, statistics arrivals, departures).  kvs_decode_attend takes it from the caller's
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
// Device address of the array per device: filled under the mutex on a device's first
// call, read without it afterwards.
std::atomic<void*> g_scratch_addr[kMaxDevices];
std::mutex g_scratch_mu;
}  // namespace

size_t static_scratch_limit() { return kStaticScratchBytes; }

// Bytes of the array one launch uses: output rows for records (CTA + sequence index)
// < grid + n_seqs, then their (m, l) words (from *ml_offset), then the counters of all
// max_seqs sequences (indexed by absolute sequence), each 256-byte aligned.
size_t static_scratch_need(const Dev& d, int n_seqs, int grid, size_t* ml_offset) {
  const size_t records = (size_t)(grid + n_seqs);
  const size_t off = (records * d.Hq * kD * sizeof(float) + 255) & ~size_t(255);
  *ml_offset = off;
  const size_t ctr = (off + records * d.Hq * sizeof(unsigned long long) + 255) & ~size_t(255);
  return ctr + (size_t)kCounterInts * d.max_seqs * sizeof(int32_t);
}

// Device address of the array on the current device, looked up once per device (the
// host-side symbol is only a stand-in, never a device address).
cudaError_t static_scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  void* p = g_scratch_addr[dev].load(std::memory_order_acquire);
  if (!p) {
    // one lookup per device even when several host threads make their first call at
    // once; a failed lookup is not kept, so a later call tries again
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    p = g_scratch_addr[dev].load(std::memory_order_relaxed);
    if (!p) {
      e = cudaGetSymbolAddress(&p, g_attend_scratch);
      if (e != cudaSuccess) return e;
      g_scratch_addr[dev].store(p, std::memory_order_release);
    }
  }
  *out = p;
  return cudaSuccess;
}

// Returns cudaErrorInvalidValue if the launch needs more than the array holds and
// cudaErrorNotSupported if its logits do not fit in shared memory (that case needs the
// workspace's logit scratch).
cudaError_t launch_attend_tc_static(const CUtensorMap& tk, const CUtensorMap& tv, const Dev& d, int layer,
                                    SeqSel sel, int n_seqs, const void* q, float* out, float* tok_out,
                                    const int32_t* bounds, int grid, cudaStream_t st) {
  size_t ml_off = 0;
  const size_t need = static_scratch_need(d, n_seqs, grid, &ml_off);
  if (need > kStaticScratchBytes) return cudaErrorInvalidValue;
  Params P;
  P.layer = layer;
  P.sel = sel;
  P.n_seqs = n_seqs;
  P.tok_out = tok_out;
  int64_t T_bound = 0;
  for (int b = 0; b < n_seqs; ++b) T_bound += bounds[b];
  const int cap0 = tc_cap(T_bound, grid) < 1 ? 1 : tc_cap(T_bound, grid);
  P.cap = cap0;
  P.q = q;
  P.out = out;
  P.qk_scale = kLog2e / sqrtf((float)kD);
  P.whole = 0;
  P.fuse = 0;
  P.k_new = P.v_new = nullptr;
  P.list_ids = P.list_count = nullptr;
  P.list_stride = 0;
  const bool fp8 = d.kv_dtype == KVS_E4M3;
  P.ns = 0;
  if (plan_whole(P, bounds, grid, wide_cap(cap0))) {
    P.ns = ring_stages(d.Hkv, fp8, true, P.cap, n_seqs, true);
    if (P.ns == 0) {
      P.whole = 0;
      P.cap = cap0;
    }
  }
  if (P.ns == 0) P.ns = ring_stages(d.Hkv, fp8, true, P.cap, n_seqs, P.whole != 0);
  if (P.ns == 0) return cudaErrorNotSupported;
  void* base = nullptr;
  cudaError_t e = static_scratch_address(&base);
  if (e != cudaSuccess) return e;
  Dev dd = d;
  dd.partials = static_cast<float*>(base);
  dd.part_ml = reinterpret_cast<unsigned long long*>(static_cast<unsigned char*>(base) + ml_off);
  dd.counters = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(base) + need -
                                           (size_t)kCounterInts * d.max_seqs * sizeof(int32_t));
  e = cudaMemsetAsync(dd.counters, 0, (size_t)kCounterInts * d.max_seqs * sizeof(int32_t), st);
  if (e != cudaSuccess) return e;
  if (d.Hkv == 4) return fp8 ? launch_one<4, true, true>(tk, tv, dd, P, grid, st) : launch_one<4, false, true>(tk, tv, dd, P, grid, st);
  return fp8 ? launch_one<8, true, true>(tk, tv, dd, P, grid, st) : launch_one<8, false, true>(tk, tv, dd, P, grid, st);
}

}  // namespace kvs
