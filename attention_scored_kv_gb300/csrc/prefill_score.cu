// SnapKV prefill scoring on the 5th-generation tensor cores (head_dim 128, 8 query heads
// per KV head, bf16 queries, bf16 or E4M3 storage).
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
//   * A CTA takes one sequence, one KV head and a chunk of its resident blocks.  The
//     group's 8 heads x 32 observation rows (256 rows) are the MMA's A operand, staged
//     once in shared memory.  Keys stream through as the B operand, 64 per stage: each
//     stage is one tcgen05.mma chain per 128-row half (M 128, N 64, K 128), issued by
//     one thread.  The 128 x 64 fp32 logits of each half land in TMEM, which holds two
//     stages so the MMA of stage s + 1 overlaps the epilogue of stage s.  Four epilogue
//     warps, one TMEM lane each per row, also stage the keys: bf16 as is, E4M3 decoded
//     to f16 (exact), with the bf16 queries converted to f16 as the decode attend does
//     (exact in f16's normal range).  Each
//     stage's global loads are issued one stage ahead, into registers.
//   * pass 1 (stats): each row keeps its running max and sum of exp2 over the chunk.
//   * combine: one thread per (sequence, head, row) merges the chunks into max, 1/sum.
//   * pass 2 (votes): the same MMAs over the chunk plus one block on each side (the
//     pool's halo).  p = exp2(s - m) / l is summed over a head's 32 rows by a warp
//     reduce-scatter, which leaves lane j with key j.  The votes are pooled in shared
//     memory and reduced over the group's heads: entry sums and per-block maxima of the
//     in-block sums.  The last of a chunk's KV-head CTAs (a ticket) adds the groups'
//     entry sums and takes the max of their block values, in KV-head order, and
//     writes the masses.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "umma.cuh"

namespace kvs {

namespace {

constexpr int kD = 128;
constexpr int kObs = 32;                  // observation rows per head: one TMEM lane or column each
constexpr int kGq = 8;                    // query heads per KV head
constexpr int kQRows = kGq * kObs;        // 256 query rows
constexpr uint32_t kQBytes = kQRows * kD * 2;        // 64 KB
constexpr int kPool = 3;                  // max-pool radius (kernel 7)
constexpr int kMbarLimit = 1 << 20;       // polls of an mbarrier before giving up
constexpr float kLog2e = 1.4426950408889634f;

// Per pass: epilogue warps, keys per stage, TMEM columns (two stages), CTAs per SM.
//   pass 1: D = Q K^T, rows (head, observation) on M (two 128-row halves), keys on N 64;
//           two warpgroups take 32 keys each.
//   pass 2: D = K Q^T, keys on M 128, (head, observation) on N 256; four warpgroups
//           take two heads each.
// A warp reads the TMEM lanes of its warpgroup quarter (warp % 4).
template <int PASS>
struct PT {
  static constexpr int EPI = PASS == 1 ? 8 : 16;
  static constexpr int THREADS = (EPI + 1) * 32;
  static constexpr int KEYS = PASS == 1 ? 64 : 128;
  static constexpr int STAGE_BLOCKS = KEYS / kBlock;
  static constexpr uint32_t KBYTES = KEYS * kD * 2;
  static constexpr uint32_t TMEM = PASS == 1 ? 256 : 512;
  static constexpr uint32_t STAGE_COLS = TMEM / 2;
  static constexpr int MINB = PASS == 1 ? 2 : 1;
};

struct PSArgs {
  Dev d;
  int layer, n_obs, chunk_blocks, n_chunks;
  SeqSel sel;                 // the call's sequences (row sl is sequence sel.at(sl))
  const __nv_bfloat16* q;     // [n_seqs][n_obs][Hq][D]
};

struct TcSmem {
  uint64_t ready;             // epilogue -> MMA: the stage's keys are in shared memory
  uint64_t done[2];           // MMA -> epilogue: TMEM stage buffer written
  uint64_t freeb[2];          // epilogue -> MMA: TMEM stage buffer read
  uint32_t tmem;
  int32_t is_last;
  float scale[2][128];        // per stage key: E4M3 scale x log2(e) / sqrt(D)
  float mprime[kQRows];       // pass 2: per (head, observation) max + log2(sum); +inf = no row
  float merge[2][2][128];     // pass 1: the second warpgroup's (max, sum) per half and row
  int32_t blk[kPrefillChunkMax + 2];
  int32_t page[kPrefillChunkMax + 2];
};

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (int it = 0; it < kMbarLimit; ++it) {
    uint32_t ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    if (ok) return true;
  }
  return false;
}
__device__ __forceinline__ void named_sync(int id, int n) {
  __syncwarp();
  asm volatile("barrier.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t two) {
  uint32_t r;
  const uint16_t a = (uint16_t)two;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(a));
  return r;
}
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  const __half2 h = __floats2half2_rn(f.x, f.y);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ void sts128(uint8_t* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" :: "r"(dst), "l"(src) : "memory");
}

// The CTA's listed blocks: resident indices [first, first + count) of the sequence, the
// chunk proper [i0, i1) plus (pass 2) one block on each side.
struct Chunk {
  int i0, i1, first, count;
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

// One stage's keys of KV head kvh, held in registers between the global load and the
// shared-memory store: thread t takes 16-byte pieces t, t + NT, ... of the stage.
template <bool FP8, int KEYS, int NT>
struct StageRegs {
  static constexpr int PER_KEY = FP8 ? kD / 16 : kD * 2 / 16;   // 8 or 16 pieces per key
  static constexpr int N = KEYS * PER_KEY / NT;
  uint4 v[N];
  float scale;
};

template <bool FP8, int KEYS, int NT>
__device__ __forceinline__ void load_stage(const PSArgs& A, const TcSmem& sm, int count, int kvh, int st, int tid,
                                           StageRegs<FP8, KEYS, NT>& r) {
  using R = StageRegs<FP8, KEYS, NT>;
  const Dev& d = A.d;
  const uint8_t* kbase = d.k_pages + (size_t)A.layer * d.page_layer_bytes;
  constexpr int SB = KEYS / kBlock;
#pragma unroll
  for (int j = 0; j < R::N; ++j) {
    const int idx = tid + NT * j, key = idx / R::PER_KEY, c16 = idx % R::PER_KEY;
    const int li = st * SB + key / kBlock;
    if (li < count) {
      const uint8_t* src = kbase + (size_t)sm.page[li] * d.page_bytes +
                           ((size_t)kvh * kBlock + key % kBlock) * kD * (FP8 ? 1 : 2) + c16 * 16;
      r.v[j] = __ldcs(reinterpret_cast<const uint4*>(src));
    } else {
      r.v[j] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
  if constexpr (FP8) {
    r.scale = 0.f;
    if (tid < KEYS) {
      const int li = st * SB + tid / kBlock;
      if (li < count)
        r.scale = d.k_scales[(size_t)A.layer * d.slot_layer_elems + (size_t)sm.page[li] * kBlock + tid % kBlock];
    }
  }
}

template <bool FP8, int KEYS, int NT>
__device__ __forceinline__ void store_stage(uint8_t* kt, TcSmem& sm, int st, int tid, const StageRegs<FP8, KEYS, NT>& r,
                                            float qk_scale) {
  using R = StageRegs<FP8, KEYS, NT>;
#pragma unroll
  for (int j = 0; j < R::N; ++j) {
    const int idx = tid + NT * j, key = idx / R::PER_KEY, c16 = idx % R::PER_KEY;
    if constexpr (FP8) {                     // 16 codes -> 16 f16 (two 16-byte pieces)
      const uint4 c = r.v[j];
      const uint4 lo = make_uint4(e4m3x2_f16x2(c.x & 0xffffu), e4m3x2_f16x2(c.x >> 16), e4m3x2_f16x2(c.y & 0xffffu),
                                  e4m3x2_f16x2(c.y >> 16));
      const uint4 hi = make_uint4(e4m3x2_f16x2(c.z & 0xffffu), e4m3x2_f16x2(c.z >> 16), e4m3x2_f16x2(c.w & 0xffffu),
                                  e4m3x2_f16x2(c.w >> 16));
      sts128(kt + umma::sw128_offset(KEYS, key, 16 * c16), lo);
      sts128(kt + umma::sw128_offset(KEYS, key, 16 * c16 + 8), hi);
    } else {
      sts128(kt + umma::sw128_offset(KEYS, key, 8 * c16), r.v[j]);
    }
  }
  if constexpr (FP8)
    if (tid < KEYS) sm.scale[st & 1][tid] = r.scale * qk_scale;
}

// Positions [a, b) of a block (first position p0) that row i sees: resident and not
// after the row's own position.
struct RowWin {
  int a, b;
};
__device__ __forceinline__ RowWin row_window(const SeqBlocks& sb, int64_t p0, int64_t obs_i, bool row_ok) {
  RowWin w;
  const int64_t lo = sb.lo - p0, hi = (sb.next < obs_i + 1 ? sb.next : obs_i + 1) - p0;
  w.a = lo <= 0 ? 0 : (lo >= kBlock ? kBlock : (int)lo);
  w.b = !row_ok || hi <= 0 ? 0 : (hi >= kBlock ? kBlock : (int)hi);
  return w;
}

template <bool FP8, int PASS>
__global__ void __launch_bounds__(PT<PASS>::THREADS, PT<PASS>::MINB) ps_tc_kernel(PSArgs A) {
  using P = PT<PASS>;
  constexpr int NT = P::EPI * 32;           // epilogue threads
  extern __shared__ __align__(1024) uint8_t dyn_raw[];
  const uint32_t raw = smem_u32(dyn_raw);
  uint8_t* base = dyn_raw + (((raw + 1023u) & ~1023u) - raw);
  uint8_t* qt = base;
  uint8_t* kt = base + kQBytes;
  TcSmem& sm = *reinterpret_cast<TcSmem*>(base + kQBytes + P::KBYTES);
  float* votes = reinterpret_cast<float*>(base + kQBytes + P::KBYTES + sizeof(TcSmem));   // [8][nkeys]
  const Dev& d = A.d;
  const int chunk = blockIdx.x, kvh = blockIdx.y, sl = blockIdx.z, s = A.sel.at(sl);
  if (!KVS_DCHECK(d, s >= 0 && s < d.max_seqs)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const SeqBlocks sb = seq_blocks(d, A.layer, s);
  const Chunk ck = chunk_of(sb, chunk, A.chunk_blocks, PASS == 2);
  if (ck.i1 <= ck.i0) return;
  const int nst = (ck.count + P::STAGE_BLOCKS - 1) / P::STAGE_BLOCKS;
  const int nkeys = ck.count * kBlock;
  const float qk_scale = kLog2e / sqrtf((float)kD);
  const int64_t obs0 = sb.next - A.n_obs;        // position of observation row 0
  for (int i = tid; i < ck.count; i += P::THREADS) {
    int32_t page;
    sm.blk[i] = block_at(d, s, sb, ck.first + i, &page);
    sm.page[i] = page;
  }
  if constexpr (PASS == 2) {
    for (int c = tid; c < kQRows; c += P::THREADS) {   // column c = head (c / 32) x row (c % 32)
      const float2 st2 = d.ps_stat[((size_t)sl * d.Hq + kvh * kGq + c / kObs) * kObs + c % kObs];
      sm.mprime[c] = (c % kObs < A.n_obs && st2.y > 0.f) ? st2.x - __log2f(st2.y) : INFINITY;
    }
  }
  if (tid == 0) {
    mbar_init(smem_u32(&sm.ready), 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(smem_u32(&sm.done[b]), 1);
      mbar_init(smem_u32(&sm.freeb[b]), 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == P::EPI) {
    umma::alloc(smem_u32(&sm.tmem), P::TMEM);
    umma::relinquish();
  }
  umma::fence_before();
  __syncthreads();
  umma::fence_after();
  const uint32_t tmem = sm.tmem;

  if (warp == P::EPI) {
    // ------------------------------------------------------------ the MMA thread
    if (lane == 0) {
      const uint32_t qs = smem_u32(qt), ks = smem_u32(kt);
      int issued = 0;
      for (int st = 0; st < nst; ++st) {
        bool ok = mbar_wait(smem_u32(&sm.ready), st & 1);
        if (ok && st >= 2) ok = mbar_wait(smem_u32(&sm.freeb[st & 1]), ((st - 2) >> 1) & 1);
        if (!ok) {
          set_error(d, kErrTimeout);
          break;
        }
        umma::fence_after();
        const uint32_t dt = tmem + (st & 1) * P::STAGE_COLS;
        if constexpr (PASS == 1) {
          constexpr uint32_t idesc = umma::idesc_f16(!FP8, 128, P::KEYS);
          for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const uint64_t ad = umma::sw128_desc(qs + (kk / 4) * (kQRows * 128) + m * (128 * 128) + (kk % 4) * 32);
              const uint64_t bd = umma::sw128_desc(ks + (kk / 4) * (P::KEYS * 128) + (kk % 4) * 32);
              umma::mma_f16(dt + m * P::KEYS, ad, bd, idesc, kk > 0);
            }
        } else {
          constexpr uint32_t idesc = umma::idesc_f16(!FP8, 128, kQRows);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint64_t ad = umma::sw128_desc(ks + (kk / 4) * (P::KEYS * 128) + (kk % 4) * 32);
            const uint64_t bd = umma::sw128_desc(qs + (kk / 4) * (kQRows * 128) + (kk % 4) * 32);
            umma::mma_f16(dt, ad, bd, idesc, kk > 0);
          }
        }
        umma::commit(smem_u32(&sm.done[st & 1]));
        issued = st + 1;
      }
      // every MMA issued has completed before TMEM is freed
      if (issued > 0 && !mbar_wait(smem_u32(&sm.done[(issued - 1) & 1]), ((issued - 1) >> 1) & 1))
        set_error(d, kErrTimeout);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ the epilogue warps
    // the queries of the group: row r = head (r / 32) x observation (r % 32), all copies
    // in flight at once; E4M3 caches then round them to f16 in place
    constexpr int kQPieces = kQRows * 16 / NT;
#pragma unroll
    for (int j = 0; j < kQPieces; ++j) {
      const int idx = tid + NT * j, r = idx / 16, c = idx % 16, i = r % kObs, hl = r / kObs;
      uint8_t* dst = qt + umma::sw128_offset(kQRows, r, 8 * c);
      if (i < A.n_obs)
        cp_async16(smem_u32(dst), A.q + (((size_t)sl * A.n_obs + i) * d.Hq + kvh * kGq + hl) * kD + 8 * c);
      else
        sts128(dst, make_uint4(0u, 0u, 0u, 0u));
    }
    asm volatile("cp.async.commit_group;\n cp.async.wait_group 0;" ::: "memory");
    if constexpr (FP8) {
#pragma unroll 4
      for (int j = 0; j < kQPieces; ++j) {
        const int idx = tid + NT * j;
        uint8_t* dst = qt + umma::sw128_offset(kQRows, idx / 16, 8 * (idx % 16));
        const uint4 v = *reinterpret_cast<const uint4*>(dst);
        sts128(dst, make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z),
                               bf16x2_to_f16x2(v.w)));
      }
    }
    StageRegs<FP8, P::KEYS, NT> regs;
    load_stage<FP8, P::KEYS, NT>(A, sm, ck.count, kvh, 0, tid, regs);
    store_stage<FP8, P::KEYS, NT>(kt, sm, 0, tid, regs, qk_scale);
    umma::fence_async_smem();
    named_sync(1, NT);
    if (tid == 0) mbar_arrive(smem_u32(&sm.ready));
    if (nst > 1) load_stage<FP8, P::KEYS, NT>(A, sm, ck.count, kvh, 1, tid, regs);

    const uint32_t lane_base = (uint32_t)(32 * (warp % 4)) << 16;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};      // pass 1 rows
    // every epilogue thread runs every iteration (a wait that runs out only flags the
    // error), so the named barriers and the warp-wide TMEM loads stay uniform
    for (int st = 0; st < nst; ++st) {
      if (!mbar_wait(smem_u32(&sm.done[st & 1]), (st >> 1) & 1)) set_error(d, kErrTimeout);
      umma::fence_after();
      if (st + 1 < nst) {                       // the key tile is free: stage st + 1 goes in
        store_stage<FP8, P::KEYS, NT>(kt, sm, st + 1, tid, regs, qk_scale);
        umma::fence_async_smem();
        named_sync(1, NT);
        if (tid == 0) mbar_arrive(smem_u32(&sm.ready));
      }
      if (st + 2 < nst) load_stage<FP8, P::KEYS, NT>(A, sm, ck.count, kvh, st + 2, tid, regs);
      const uint32_t tcol = tmem + lane_base + (st & 1) * P::STAGE_COLS;
      if constexpr (PASS == 1) {
        // rows: lane = observation i of heads warp % 4 (half 0) and warp % 4 + 4 (half 1);
        // warpgroup `half` = warp / 4 takes keys 32 half .. 32 half + 31 (blocks 2 half,
        // 2 half + 1), whose row windows are the same for both row halves
        const bool row_ok = lane < A.n_obs;
        const int half = warp / 4;
        RowWin w[2];
#pragma unroll
        for (int bb = 0; bb < 2; ++bb) {
          const int li = st * P::STAGE_BLOCKS + 2 * half + bb;
          w[bb] = li < ck.count ? row_window(sb, (int64_t)sm.blk[li] * kBlock, obs0 + lane, row_ok) : RowWin{0, 0};
        }
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          {
            float v[32];
            umma::ld32(tcol + t * P::KEYS + 32 * half, v);
#pragma unroll
            for (int bb = 0; bb < 2; ++bb) {
              const RowWin ww = w[bb];
              if constexpr (FP8) {
                const float4* sc4 = reinterpret_cast<const float4*>(&sm.scale[st & 1][32 * half + 16 * bb]);
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                  const float4 sc = sc4[q4];
                  v[16 * bb + 4 * q4] *= sc.x;
                  v[16 * bb + 4 * q4 + 1] *= sc.y;
                  v[16 * bb + 4 * q4 + 2] *= sc.z;
                  v[16 * bb + 4 * q4 + 3] *= sc.w;
                }
              } else {
#pragma unroll
                for (int c = 0; c < kBlock; ++c) v[16 * bb + c] *= qk_scale;
              }
              if (ww.a != 0 || ww.b != kBlock) {
#pragma unroll
                for (int c = 0; c < kBlock; ++c)
                  if (c < ww.a || c >= ww.b) v[16 * bb + c] = -INFINITY;
              }
            }
            float bm = v[0];
#pragma unroll
            for (int j = 1; j < 32; ++j) bm = fmaxf(bm, v[j]);
            if (bm != -INFINITY) {
              const float mn = fmaxf(m_run[t], bm);
              float acc = 0.f;
#pragma unroll
              for (int j = 0; j < 32; ++j) acc += exp2f(v[j] - mn);
              l_run[t] = l_run[t] * exp2f(m_run[t] - mn) + acc;
              m_run[t] = mn;
            }
          }
        }
      } else {
        // thread = key (32 * (warp % 4) + lane of the stage); warpgroup g = warp / 4
        // takes heads 2g, 2g + 1; a head's 32 observation rows are 32 TMEM columns
        const int key = 32 * (warp % 4) + lane, li = st * P::STAGE_BLOCKS + key / kBlock;
        bool kv_ok = li < ck.count;
        int64_t pk = 0;
        if (kv_ok) {
          pk = (int64_t)sm.blk[li] * kBlock + key % kBlock;
          kv_ok = pk >= sb.lo && pk < sb.next;
        }
        const int64_t rel = pk - obs0;                                   // rows i < rel do not see it
        const int lim = rel <= 0 ? 0 : (rel >= kObs ? kObs : (int)rel);
        const float sck = FP8 ? sm.scale[st & 1][key] : qk_scale;
        const int g = warp / 4;
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const int h = 2 * g + hh;
          float v[32];
          umma::ld32(tcol + 32 * h, v);
          const float4* mp4 = reinterpret_cast<const float4*>(&sm.mprime[h * kObs]);
          float sum = 0.f;
          if (lim <= 0) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              const float4 mp = mp4[q4];
              sum += exp2f(fmaf(v[4 * q4], sck, -mp.x)) + exp2f(fmaf(v[4 * q4 + 1], sck, -mp.y)) +
                     exp2f(fmaf(v[4 * q4 + 2], sck, -mp.z)) + exp2f(fmaf(v[4 * q4 + 3], sck, -mp.w));
            }
          } else {
#pragma unroll
            for (int i = 0; i < kObs; ++i)
              if (i >= lim) sum += exp2f(fmaf(v[i], sck, -sm.mprime[h * kObs + i]));
          }
          const int lk = st * P::KEYS + key;
          if (lk < nkeys) votes[h * nkeys + lk] = kv_ok ? sum : 0.f;
        }
      }
      umma::fence_before();
      named_sync(1, NT);
      if (tid == 0) mbar_arrive(smem_u32(&sm.freeb[st & 1]));
    }
    if constexpr (PASS == 1) {
      // the two warpgroups' (max, sum) of a row merge; lane = row, so no shuffles
      const int row = 32 * (warp % 4) + lane;
      if (warp >= 4) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          sm.merge[t][0][row] = m_run[t];
          sm.merge[t][1][row] = l_run[t];
        }
      }
      named_sync(1, NT);
      if (warp < 4) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const float mo = sm.merge[t][0][row], lo = sm.merge[t][1][row], mn = fmaxf(m_run[t], mo);
          const float l = mn == -INFINITY ? 0.f : l_run[t] * exp2f(m_run[t] - mn) + lo * exp2f(mo - mn);
          d.ps_part[(((size_t)sl * A.n_chunks + chunk) * d.Hq + kvh * kGq + warp + 4 * t) * kObs + lane] =
              make_float2(mn, l);
        }
      }
    }
    umma::fence_before();
  }
  __syncthreads();
  if (warp == P::EPI) {
    umma::fence_after();
    umma::dealloc(tmem, P::TMEM);
  }
  if constexpr (PASS == 1) return;

  // ------------------------------------------------------------ pool and reduce (pass 2)
  // Positions inside a block are consecutive; across blocks they are when the next
  // listed block is the next block id.  A key that is not resident has vote 0, so it
  // can sit in a max without changing it, but its own pooled value is 0.
  const int lo_halo = ck.i0 - ck.first, nblk = ck.i1 - ck.i0, nck = nblk * kBlock;
  float* pool = votes + kGq * nkeys;                        // [8 heads][chunk keys]
  float* bsum = pool + kGq * nck;                           // [8 heads][chunk blocks]
  for (int i = tid; i < kGq * nck; i += P::THREADS) {
    const int hl = i / nck, ic = i % nck, j = lo_halo * kBlock + ic, b = j / kBlock, c = j % kBlock;
    const int64_t pj = (int64_t)sm.blk[b] * kBlock + c;
    float v = 0.f;
    if (pj >= sb.lo && pj < sb.next) {
      const bool prev = b > 0 && sm.blk[b - 1] == sm.blk[b] - 1, next = b + 1 < ck.count && sm.blk[b + 1] == sm.blk[b] + 1;
      const int lo = c >= kPool || prev ? j - kPool : j - c, hi = c + kPool < kBlock || next ? j + kPool : j - c + kBlock - 1;
      const float* vr = votes + hl * nkeys;
      v = vr[j];
      for (int jj = max(lo, 0); jj <= min(hi, nkeys - 1); ++jj) v = fmaxf(v, vr[jj]);
    }
    pool[hl * nck + ic] = v;
  }
  __syncthreads();
  const size_t gbase = ((size_t)sl * d.Hkv + kvh) * d.ps_bound;
  for (int i = tid; i < nck; i += P::THREADS) {             // the group's entry sums, head order
    float tsum = 0.f;
#pragma unroll
    for (int hl = 0; hl < kGq; ++hl) tsum += pool[hl * nck + i];
    d.ps_tok[(gbase + ck.i0) * kBlock + i] = tsum;
  }
  for (int i = tid; i < nblk * kGq; i += P::THREADS) {      // per head and block the in-block sum
    const int hl = i / nblk, b = i % nblk;
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < kBlock; ++c) acc += pool[hl * nck + b * kBlock + c];
    bsum[hl * nblk + b] = acc;
  }
  __syncthreads();
  for (int b = tid; b < nblk; b += P::THREADS) {            // ... and its max over the heads
    float mx = 0.f;
    for (int hl = 0; hl < kGq; ++hl) {
      mx = fmaxf(mx, bsum[hl * nblk + b]);
      record_head(d, A.layer, s, sm.blk[lo_halo + b], kvh * kGq + hl, bsum[hl * nblk + b]);   // head profiles
    }
    d.ps_blk[gbase + ck.i0 + b] = mx;
  }
  __syncthreads();
  if (tid == 0) {                                           // the last KV head of the chunk combines
    __threadfence();
    int32_t* tk = &d.ps_tickets[(size_t)sl * A.n_chunks + chunk];
    const int arrived = atomicAdd(tk, 1);
    sm.is_last = arrived == d.Hkv - 1;
    if (sm.is_last) *tk = 0;
  }
  __syncthreads();
  if (!sm.is_last) return;
  __threadfence();
  const size_t sbase = (size_t)sl * d.Hkv * d.ps_bound, stride = d.ps_bound;
  float* tok = d.tok_mass + (size_t)A.layer * d.slot_layer_elems;
  for (int i = tid; i < nblk * kBlock; i += P::THREADS) {
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
  for (int b = tid; b < nblk; b += P::THREADS) {
    float mx = 0.f;
    for (int g2 = 0; g2 < d.Hkv; ++g2) mx = fmaxf(mx, __ldcg(d.ps_blk + sbase + g2 * stride + ck.i0 + b));
    bm[sm.blk[lo_halo + b]] = mx;
  }
}

// ------------------------------------------------------------------ combine
__global__ void ps_combine_kernel(PSArgs A, int n_seqs) {
  const Dev& d = A.d;
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= n_seqs * d.Hq * kObs) return;
  const int sl = idx / (d.Hq * kObs), hr = idx % (d.Hq * kObs);
  const int s = A.sel.at(sl);
  if (!KVS_DCHECK(d, s >= 0 && s < d.max_seqs)) return;
  const SeqBlocks sb = seq_blocks(d, A.layer, s);
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

size_t tc_smem(int pass, int chunk_blocks) {
  size_t b = 1024 + kQBytes + (pass == 1 ? PT<1>::KBYTES : PT<2>::KBYTES) + sizeof(TcSmem);
  if (pass == 2)   // votes (chunk + halo), pooled votes (chunk), block sums
    b += (size_t)kGq * (chunk_blocks + 2) * kBlock * 4 + (size_t)kGq * chunk_blocks * kBlock * 4 +
         (size_t)kGq * chunk_blocks * 4;
  return b;
}

template <bool FP8>
cudaError_t launch_ps(const PSArgs& A, int n_seqs, cudaStream_t st) {
  static std::atomic<unsigned long long> optin1{0}, optin2{0};   // per device
  cudaError_t e = smem_optin_once(optin1, ps_tc_kernel<FP8, 1>, (int)tc_smem(1, kPrefillChunkMax));
  if (e == cudaSuccess) e = smem_optin_once(optin2, ps_tc_kernel<FP8, 2>, (int)tc_smem(2, kPrefillChunkMax));
  if (e != cudaSuccess) return e;
  const dim3 grid(A.n_chunks, A.d.Hkv, n_seqs);
  ps_tc_kernel<FP8, 1><<<grid, PT<1>::THREADS, tc_smem(1, A.chunk_blocks), st>>>(A);
  const int rows = n_seqs * A.d.Hq * kObs;
  ps_combine_kernel<<<(rows + 255) / 256, 256, 0, st>>>(A, n_seqs);
  ps_tc_kernel<FP8, 2><<<grid, PT<2>::THREADS, tc_smem(2, A.chunk_blocks), st>>>(A);
  return cudaGetLastError();
}

}  // namespace

int prefill_obs_max() { return kObs; }

cudaError_t launch_prefill_score(const Dev& d, int layer, SeqSel sel, int n_seqs, const void* q_obs, int n_obs,
                                 int chunk_blocks, int n_chunks, cudaStream_t st) {
  PSArgs A;
  A.d = d;
  A.layer = layer;
  A.sel = sel;
  A.n_obs = n_obs;
  A.chunk_blocks = chunk_blocks;
  A.n_chunks = n_chunks;
  A.q = static_cast<const __nv_bfloat16*>(q_obs);
  return d.kv_dtype == KVS_E4M3 ? launch_ps<true>(A, n_seqs, st) : launch_ps<false>(A, n_seqs, st);
}

}  // namespace kvs
