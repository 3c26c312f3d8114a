// SnapKV prefill scoring on the tensor cores (head_dim 128, 8 query heads per KV head,
// bf16 queries, bf16 or E4M3 storage).
//
// What it computes ("Context views at marginal cost", the per-system reductions,
// SnapKV): when prefill ends, the prompt's last n_obs queries (the observation window,
// at most 32) attend causally over the resident entries.  Query i, at position
// next - n_obs + i, sees the entries at positions <= its own.  Logits are q.k/sqrt(D),
// with E4M3 keys decoded as code * scale, and the softmax is per head.  Each entry's
// vote for head h is the sum of the weights the window's queries of head h give it.
// The votes are max-pooled along the positions (kernel 7: at each resident position,
// the largest vote within 3 positions), and the pooled votes become the layer's step
// masses.  The entry mass sums over heads, and the block mass is the max over heads
// of the in-block sum ("Per-Head Attention as a Scoring Signal", Fix: score per head,
// place per block).  kvs_accumulate_scores then folds them into the tables.
//
// How (three launches per layer):
//   1. stats: CTA = (sequence, KV head, chunk of resident blocks), one warp per query
//      head of the group and one lane row per observation query.  QK^T runs on
//      mma.sync m16n8k16: queries on M (two row tiles = the 32 observation rows), keys
//      on N.  The query fragments stay in registers, and K blocks stream through a
//      three-slot cp.async ring shared by the 8 warps.  The result is each row's
//      partial max and sum of exp2 over the chunk.
//   2. combine: one thread per (sequence, head, row) merges the chunks' partials into
//      the row's max and 1/sum.
//   3. votes: the same CTAs recompute the logits of their chunk plus one block on each
//      side (the pool's halo) and sum p = exp2(s - m) / l over the 32 rows with warp
//      shuffles.  They pool in shared memory and reduce over the group's 8 heads: the
//      group's entry sums and its per-block maxima of in-block sums.  The last of a
//      chunk's KV-head CTAs (a ticket) adds the groups' entry sums and takes the max of
//      their block values, in KV-head order, and writes the masses.
//
// The k index of every MMA is permuted the same way on both sides: lane (g, t) holds
// dimensions 32t + 4ks .. 32t + 4ks + 3 in k-step ks.  A dot product does not depend
// on the order of its terms, and each lane then reads 32 or 64 contiguous bytes of a
// key row.  E4M3 keys are decoded to f16 in registers (exact), so for them the bf16
// queries are rounded to f16, as the decode attend does.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "kvs_internal.cuh"

namespace kvs {

namespace {

constexpr int kD = 128;
constexpr int kObs = 32;            // observation rows per head: one lane each
constexpr int kGq = 8;              // query heads per KV head = warps per CTA
constexpr int kThreads = kGq * 32;
constexpr int kSlotBlocks = 2;      // K blocks per ring slot
constexpr int kRing = 3;
constexpr int kPool = 3;            // max-pool radius (kernel 7)
constexpr float kLog2e = 1.4426950408889634f;

template <bool FP8>
struct PS {
  static constexpr int ESZ = FP8 ? 1 : 2;
  static constexpr int ROW = kD * ESZ + 16;                 // padded key row in shared memory
  static constexpr int SLOT = kSlotBlocks * kBlock * ROW;
  static constexpr int CHUNKS16 = kD * ESZ / 16;            // 16-byte pieces of a key row
};

struct PSArgs {
  Dev d;
  int layer, seq_begin, n_obs, chunk_blocks, n_chunks;
  const __nv_bfloat16* q;     // [n_seqs][n_obs][Hq][D]
};

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t two) {
  uint32_t r;
  const uint16_t a = (uint16_t)two;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(a));
  return r;
}
__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}
template <bool FP8>
__device__ __forceinline__ void mma16816(float c[4], const uint32_t a[4], uint32_t b0, uint32_t b1) {
  if constexpr (FP8)
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Shared state of one CTA: the K ring, the E4M3 scales, and the chunk's block list
// (with halos).
template <bool FP8>
struct Smem {
  uint8_t ring[kRing][PS<FP8>::SLOT];
  float scale[kRing][kSlotBlocks * kBlock];
  int32_t blk[kPrefillChunkMax + 2];  // block ids of the listed blocks
  int32_t page[kPrefillChunkMax + 2];
};

// Query fragments of head h for the rows g, g+8 (tile 0) and g+16, g+24 (tile 1):
// a[rt][ks] = {row lo k-lo, row hi k-lo, row lo k-hi, row hi k-hi} under the permuted k.
template <bool FP8>
__device__ __forceinline__ void load_q(const PSArgs& A, int sl, int h, int lane, uint32_t (&a)[2][8][4]) {
  const int g = lane >> 2, t = lane & 3, Hq = A.d.Hq;
#pragma unroll
  for (int rt = 0; rt < 2; ++rt)
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int row = 16 * rt + g + 8 * half;
      uint32_t w[16];
      if (row < A.n_obs) {
        const uint4* src = reinterpret_cast<const uint4*>(A.q + (((size_t)sl * A.n_obs + row) * Hq + h) * kD + 32 * t);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 v = src[i];
          w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) w[i] = 0u;
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t lo = w[2 * ks], hi = w[2 * ks + 1];     // dims 32t+4ks+{0,1} and +{2,3}
        if constexpr (FP8) {
          const float2 f0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&lo));
          const float2 f1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&hi));
          lo = f16x2_of(f0.x, f0.y);
          hi = f16x2_of(f1.x, f1.y);
        }
        a[rt][ks][half] = lo;
        a[rt][ks][2 + half] = hi;
      }
    }
}

// Issue the copies of ring slot `slot`: listed blocks [b0, b0 + nb) of KV head kvh.
template <bool FP8>
__device__ __forceinline__ void issue_slot(Smem<FP8>& sm, const PSArgs& A, int kvh, int slot, int b0, int nb) {
  using C = PS<FP8>;
  const Dev& d = A.d;
  const uint8_t* kbase = d.k_pages + (size_t)A.layer * d.page_layer_bytes;
  const int per_block = kBlock * C::CHUNKS16;
  for (int i = threadIdx.x; i < nb * per_block; i += kThreads) {
    const int b = i / per_block, r = i % per_block, key = r / C::CHUNKS16, c16 = r % C::CHUNKS16;
    const uint8_t* src = kbase + (size_t)sm.page[b0 + b] * d.page_bytes + ((size_t)kvh * kBlock + key) * kD * C::ESZ + c16 * 16;
    cp_async16(smem_u32(&sm.ring[slot][(b * kBlock + key) * C::ROW + c16 * 16]), src);
  }
  if constexpr (FP8) {
    const float* sbase = d.k_scales + (size_t)A.layer * d.slot_layer_elems;
    for (int i = threadIdx.x; i < nb * 4; i += kThreads) {
      const int b = i / 4, c4 = i % 4;
      cp_async16(smem_u32(&sm.scale[slot][b * kBlock + 4 * c4]), sbase + (size_t)sm.page[b0 + b] * kBlock + 4 * c4);
    }
  }
}

// QK^T of one 16-key block (ring slot `slot`, position `bi` in it) for the warp's 32
// rows: c[rt][nt][e] holds (row 16rt + g + 8(e>>1), key 8nt + 2t + (e&1)), scaled to
// the log2 domain.
template <bool FP8>
__device__ __forceinline__ void block_logits(const Smem<FP8>& sm, int slot, int bi, int lane, const uint32_t (&a)[2][8][4],
                                             float qk_scale, float (&c)[2][2][4]) {
  using C = PS<FP8>;
  const int g = lane >> 2, t = lane & 3;
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
    for (int rt = 0; rt < 2; ++rt) c[rt][nt][0] = c[rt][nt][1] = c[rt][nt][2] = c[rt][nt][3] = 0.f;
    const uint8_t* row = &sm.ring[slot][(bi * kBlock + 8 * nt + g) * C::ROW];
    if constexpr (FP8) {
      const uint4 r0 = *reinterpret_cast<const uint4*>(row + 32 * t);
      const uint4 r1 = *reinterpret_cast<const uint4*>(row + 32 * t + 16);
      const uint32_t w[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t b0 = e4m3x2_f16x2(w[ks] & 0xffffu), b1 = e4m3x2_f16x2(w[ks] >> 16);
        mma16816<true>(c[0][nt], a[0][ks], b0, b1);
        mma16816<true>(c[1][nt], a[1][ks], b0, b1);
      }
    } else {
      uint32_t w[16];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + 64 * t + 16 * i);
        w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
      }
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        mma16816<false>(c[0][nt], a[0][ks], w[2 * ks], w[2 * ks + 1]);
        mma16816<false>(c[1][nt], a[1][ks], w[2 * ks], w[2 * ks + 1]);
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float sc = qk_scale;
      if constexpr (FP8) sc *= sm.scale[slot][bi * kBlock + 8 * nt + 2 * t + j];
#pragma unroll
      for (int rt = 0; rt < 2; ++rt) {
        c[rt][nt][j] *= sc;
        c[rt][nt][2 + j] *= sc;
      }
    }
  }
}

// The CTA's listed blocks: resident indices [i0 - lo_halo, i1 + hi_halo) of sequence s.
struct Chunk {
  int i0, i1, first, count;   // chunk proper [i0, i1); list = [first, first + count)
};

__device__ __forceinline__ Chunk chunk_of(const SeqBlocks& sb, int chunk, int cb, bool halo) {
  Chunk c;
  c.i0 = chunk * cb;
  c.i1 = min(c.i0 + cb, sb.n);
  c.first = (halo && c.i0 > 0) ? c.i0 - 1 : c.i0;
  const int last = (halo && c.i1 < sb.n) ? c.i1 + 1 : c.i1;
  c.count = last - c.first;
  return c;
}

// Stream the listed blocks through the ring and call f(list index, slot, position in slot)
// for each, in order.  Every thread of the CTA calls it.
template <bool FP8, class F>
__device__ __forceinline__ void stream_blocks(Smem<FP8>& sm, const PSArgs& A, int kvh, int count, F&& f) {
  const int nslots = (count + kSlotBlocks - 1) / kSlotBlocks;
  for (int p = 0; p < kRing - 1; ++p) {
    if (p < nslots) issue_slot<FP8>(sm, A, kvh, p % kRing, p * kSlotBlocks, min(kSlotBlocks, count - p * kSlotBlocks));
    cp_commit();
  }
  for (int st = 0; st < nslots; ++st) {
    cp_wait1();
    __syncthreads();
    const int nx = st + kRing - 1;
    if (nx < nslots) issue_slot<FP8>(sm, A, kvh, nx % kRing, nx * kSlotBlocks, min(kSlotBlocks, count - nx * kSlotBlocks));
    cp_commit();
    const int nb = min(kSlotBlocks, count - st * kSlotBlocks);
    for (int bi = 0; bi < nb; ++bi) f(st * kSlotBlocks + bi, st % kRing, bi);
  }
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  __syncthreads();
}

// ------------------------------------------------------------------ 1. stats
template <bool FP8>
__global__ void __launch_bounds__(kThreads) ps_stats_kernel(PSArgs A) {
  extern __shared__ __align__(128) uint8_t dyn[];
  Smem<FP8>& sm = *reinterpret_cast<Smem<FP8>*>(dyn);
  const Dev& d = A.d;
  const int chunk = blockIdx.x, kvh = blockIdx.y, sl = blockIdx.z, s = A.seq_begin + sl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int h = kvh * kGq + warp;
  const SeqBlocks sb = seq_blocks(d, A.layer, s);
  const Chunk ck = chunk_of(sb, chunk, A.chunk_blocks, false);
  if (ck.count <= 0) return;
  for (int i = threadIdx.x; i < ck.count; i += kThreads) {
    int32_t page;
    sm.blk[i] = block_at(d, s, sb, ck.first + i, &page);
    sm.page[i] = page;
  }
  __syncthreads();
  uint32_t a[2][8][4];
  load_q<FP8>(A, sl, h, lane, a);
  const float qk_scale = kLog2e / sqrtf((float)kD);
  const int64_t obs0 = sb.next - A.n_obs;
  float m[4], l[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) { m[r] = -INFINITY; l[r] = 0.f; }
  stream_blocks<FP8>(sm, A, kvh, ck.count, [&](int li, int slot, int bi) {
    float c[2][2][4];
    block_logits<FP8>(sm, slot, bi, lane, a, qk_scale, c);
    const int64_t p0 = (int64_t)sm.blk[li] * kBlock;
#pragma unroll
    for (int r = 0; r < 4; ++r) {                 // rows g, g+8, g+16, g+24
      const int rt = r >> 1, e2 = (r & 1) * 2, row = 16 * rt + g + 8 * (r & 1);
      float v[4];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          const int64_t p = p0 + 8 * nt + 2 * t + j;
          const bool ok = row < A.n_obs && p >= sb.lo && p < sb.next && p <= obs0 + row;
          v[2 * nt + j] = ok ? c[rt][nt][e2 + j] : -INFINITY;
        }
      const float bm = fmaxf(fmaxf(v[0], v[1]), fmaxf(v[2], v[3]));
      if (bm == -INFINITY) continue;
      const float mn = fmaxf(m[r], bm);
      l[r] = l[r] * exp2f(m[r] - mn) + exp2f(v[0] - mn) + exp2f(v[1] - mn) + exp2f(v[2] - mn) + exp2f(v[3] - mn);
      m[r] = mn;
    }
  });
  // merge the 4 lanes of a row (t = 0..3)
#pragma unroll
  for (int r = 0; r < 4; ++r) {
#pragma unroll
    for (int o = 1; o < 4; o <<= 1) {
      const float mo = __shfl_xor_sync(0xffffffffu, m[r], o), lo = __shfl_xor_sync(0xffffffffu, l[r], o);
      const float mn = fmaxf(m[r], mo);
      if (mn != -INFINITY) {
        l[r] = l[r] * exp2f(m[r] - mn) + lo * exp2f(mo - mn);
        m[r] = mn;
      }
    }
  }
  if (t == 0) {
    float2* part = d.ps_part + (((size_t)sl * A.n_chunks + chunk) * d.Hq + h) * kObs;
#pragma unroll
    for (int r = 0; r < 4; ++r) part[16 * (r >> 1) + g + 8 * (r & 1)] = make_float2(m[r], l[r]);
  }
}

// ------------------------------------------------------------------ 2. combine
__global__ void ps_combine_kernel(PSArgs A, int n_seqs) {
  const Dev& d = A.d;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_seqs * d.Hq * kObs) return;
  const int sl = idx / (d.Hq * kObs), hr = idx % (d.Hq * kObs);
  const SeqBlocks sb = seq_blocks(d, A.layer, A.seq_begin + sl);
  const int used = min((sb.n + A.chunk_blocks - 1) / A.chunk_blocks, A.n_chunks);
  float M = -INFINITY, L = 0.f;
  for (int c = 0; c < used; ++c) {
    const float2 p = d.ps_part[((size_t)sl * A.n_chunks + c) * d.Hq * kObs + hr];
    const float mn = fmaxf(M, p.x);
    if (mn == -INFINITY) continue;
    L = L * exp2f(M - mn) + p.y * exp2f(p.x - mn);
    M = mn;
  }
  d.ps_stat[(size_t)sl * d.Hq * kObs + hr] = make_float2(M, L > 0.f ? 1.f / L : 0.f);
}

// ------------------------------------------------------------------ 3. votes
template <bool FP8>
__global__ void __launch_bounds__(kThreads) ps_votes_kernel(PSArgs A) {
  extern __shared__ __align__(128) uint8_t dyn[];
  Smem<FP8>& sm = *reinterpret_cast<Smem<FP8>*>(dyn);
  const Dev& d = A.d;
  const int chunk = blockIdx.x, kvh = blockIdx.y, sl = blockIdx.z, s = A.seq_begin + sl;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int h = kvh * kGq + warp;
  const SeqBlocks sb = seq_blocks(d, A.layer, s);
  const Chunk ck = chunk_of(sb, chunk, A.chunk_blocks, true);
  if (ck.i1 <= ck.i0) return;
  const int nkeys = ck.count * kBlock;
  float* votes = reinterpret_cast<float*>(dyn + sizeof(Smem<FP8>));   // [8 heads][nkeys]
  float* bsum = votes + kGq * nkeys;                                    // [8 heads][chunk blocks]
  __shared__ int32_t is_last;
  for (int i = threadIdx.x; i < ck.count; i += kThreads) {
    int32_t page;
    sm.blk[i] = block_at(d, s, sb, ck.first + i, &page);
    sm.page[i] = page;
  }
  __syncthreads();
  uint32_t a[2][8][4];
  load_q<FP8>(A, sl, h, lane, a);
  const float qk_scale = kLog2e / sqrtf((float)kD);
  const int64_t obs0 = sb.next - A.n_obs;
  // the row statistics of this thread's rows g, g+8, g+16, g+24 (lane r holds row r)
  const float2 my = d.ps_stat[((size_t)sl * d.Hq + h) * kObs + lane];
  float m[4], il[4];
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int row = 16 * (r >> 1) + g + 8 * (r & 1);
    m[r] = __shfl_sync(0xffffffffu, my.x, row);
    il[r] = __shfl_sync(0xffffffffu, my.y, row);
  }
  stream_blocks<FP8>(sm, A, kvh, ck.count, [&](int li, int slot, int bi) {
    float c[2][2][4];
    block_logits<FP8>(sm, slot, bi, lane, a, qk_scale, c);
    const int64_t p0 = (int64_t)sm.blk[li] * kBlock;
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        const int64_t p = p0 + 8 * nt + 2 * t + j;
        const bool key_ok = p >= sb.lo && p < sb.next;
        float v = 0.f;
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int rt = r >> 1, row = 16 * rt + g + 8 * (r & 1);
          if (key_ok && row < A.n_obs && p <= obs0 + row) v += exp2f(c[rt][nt][(r & 1) * 2 + j] - m[r]) * il[r];
        }
        v += __shfl_xor_sync(0xffffffffu, v, 4);
        v += __shfl_xor_sync(0xffffffffu, v, 8);
        v += __shfl_xor_sync(0xffffffffu, v, 16);
        if (g == 0) votes[warp * nkeys + li * kBlock + 8 * nt + 2 * t + j] = v;
      }
  });
  // (stream_blocks ends with a barrier: every vote is in shared memory)
  const int lo_halo = ck.i0 - ck.first, nblk = ck.i1 - ck.i0;
  auto pooled = [&](int hl, int j) -> float {      // j: list key index of a chunk key
    const int64_t pj = (int64_t)sm.blk[j / kBlock] * kBlock + (j % kBlock);
    if (pj < sb.lo || pj >= sb.next) return 0.f;   // not resident: no mass
    float v = votes[hl * nkeys + j];
#pragma unroll
    for (int o = -kPool; o <= kPool; ++o) {
      const int jj = j + o;
      if (o == 0 || jj < 0 || jj >= nkeys) continue;
      const int64_t pjj = (int64_t)sm.blk[jj / kBlock] * kBlock + (jj % kBlock);
      if (pjj == pj + o) v = fmaxf(v, votes[hl * nkeys + jj]);
    }
    return v;
  };
  const size_t base = ((size_t)sl * d.Hkv + kvh) * d.ps_bound;
  // the group's entry sums over its 8 heads, in head order
  for (int i = threadIdx.x; i < nblk * kBlock; i += kThreads) {
    const int j = lo_halo * kBlock + i;
    float tsum = 0.f;
    for (int hl = 0; hl < kGq; ++hl) tsum += pooled(hl, j);
    d.ps_tok[(base + ck.i0) * kBlock + i] = tsum;
  }
  // per head and block the in-block sum, then the max over the group's heads
  for (int i = threadIdx.x; i < nblk * kGq; i += kThreads) {
    const int hl = i / nblk, b = i % nblk;
    float acc = 0.f;
    for (int c = 0; c < kBlock; ++c) acc += pooled(hl, (lo_halo + b) * kBlock + c);
    bsum[hl * nblk + b] = acc;
  }
  __syncthreads();
  for (int b = threadIdx.x; b < nblk; b += kThreads) {
    float mx = 0.f;
    for (int hl = 0; hl < kGq; ++hl) mx = fmaxf(mx, bsum[hl * nblk + b]);
    d.ps_blk[base + ck.i0 + b] = mx;
  }
  // the last KV-head CTA of this chunk combines the groups
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    int32_t* tk = &d.ps_tickets[(size_t)sl * A.n_chunks + chunk];
    const int arrived = atomicAdd(tk, 1);
    is_last = arrived == d.Hkv - 1;
    if (is_last) *tk = 0;
  }
  __syncthreads();
  if (!is_last) return;
  __threadfence();
  const size_t sbase = (size_t)sl * d.Hkv * d.ps_bound, stride = d.ps_bound;
  float* tok = d.tok_mass + (size_t)A.layer * d.slot_layer_elems;
  for (int i = threadIdx.x; i < nblk * kBlock; i += kThreads) {
    const int b = i / kBlock, c = i % kBlock;
    const int64_t p = (int64_t)sm.blk[lo_halo + b] * kBlock + c;
    if (p < sb.lo || p >= sb.next) continue;
    float tsum = 0.f;
    for (int g2 = 0; g2 < d.Hkv; ++g2) tsum += __ldcg(d.ps_tok + (sbase + g2 * stride + ck.i0) * kBlock + i);
    int32_t slot;
    const int32_t page = page_of(d, s, p, &slot);
    tok[(size_t)page * kBlock + slot] = tsum;
  }
  float* bm = d.blk_mass + (size_t)A.layer * d.blk_layer_elems + (size_t)s * d.max_blocks;
  for (int b = threadIdx.x; b < nblk; b += kThreads) {
    float mx = 0.f;
    for (int g2 = 0; g2 < d.Hkv; ++g2) mx = fmaxf(mx, __ldcg(d.ps_blk + sbase + g2 * stride + ck.i0 + b));
    bm[sm.blk[lo_halo + b]] = mx;
  }
}

template <bool FP8>
size_t votes_smem(int chunk_blocks) {
  return sizeof(Smem<FP8>) + (size_t)kGq * (chunk_blocks + 2) * kBlock * 4 + (size_t)kGq * chunk_blocks * 4;
}

template <bool FP8>
cudaError_t launch_ps(const PSArgs& A, int n_seqs, cudaStream_t st) {
  static bool attr = false;
  const size_t s1 = sizeof(Smem<FP8>), s3 = votes_smem<FP8>(kPrefillChunkMax);
  if (!attr) {
    cudaError_t e = cudaFuncSetAttribute(ps_stats_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s1);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(ps_votes_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)s3);
    if (e != cudaSuccess) return e;
    attr = true;
  }
  const dim3 grid(A.n_chunks, A.d.Hkv, n_seqs);
  ps_stats_kernel<FP8><<<grid, kThreads, s1, st>>>(A);
  const int rows = n_seqs * A.d.Hq * kObs;
  ps_combine_kernel<<<(rows + 255) / 256, 256, 0, st>>>(A, n_seqs);
  ps_votes_kernel<FP8><<<grid, kThreads, votes_smem<FP8>(A.chunk_blocks), st>>>(A);
  return cudaGetLastError();
}

}  // namespace

int prefill_obs_max() { return kObs; }

cudaError_t launch_prefill_score(const Dev& d, int layer, int seq_begin, int n_seqs, const void* q_obs, int n_obs,
                                 int chunk_blocks, int n_chunks, cudaStream_t st) {
  PSArgs A;
  A.d = d;
  A.layer = layer;
  A.seq_begin = seq_begin;
  A.n_obs = n_obs;
  A.chunk_blocks = chunk_blocks;
  A.n_chunks = n_chunks;
  A.q = static_cast<const __nv_bfloat16*>(q_obs);
  return d.kv_dtype == KVS_E4M3 ? launch_ps<true>(A, n_seqs, st) : launch_ps<false>(A, n_seqs, st);
}

}  // namespace kvs
