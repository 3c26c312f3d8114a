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
// How (one cooperative launch per layer, one CTA per SM):
//   * The launch's (sequence, KV head, resident block) triples are laid end to end,
//     sequence-major, each group led by a fixed charge for its per-run costs, and CTA c
//     takes the contiguous share [c T / G, (c + 1) T / G) of that weighted order.  A share
//     cuts into runs, one per (sequence, KV head) group whose blocks it touches.  Each run sees
//     the group's 8 heads x 32 observation rows (256 rows), staged once per group by TMA,
//     and its keys 128 (8 blocks) per stage.
//   * Phase 1 (row statistics): D = Q K^T, two M-128 halves of rows by N 128 keys, into
//     TMEM.  Sixteen epilogue warps read the logits back, one TMEM lane per row, and keep
//     each row's running max and sum of exp2.  At the end of a run the row partials go
//     to global memory and one release-add counts the CTA's arrival for the group.
//   * Phase 2 (votes): the same runs, cut into pieces of at most 62 blocks plus one halo
//     block on each side for the pool.  D = K Q^T, keys on M 128 and rows on N 256, so a
//     thread holds one key and sums exp2(s - M_row) over a head's 32 rows (TMEM columns)
//     without shuffles.  M_row = max + log2(sum) over the whole row is merged from the
//     partials of every CTA that shares the group, by a statistics warp that waits for
//     the group's arrivals one run ahead of the epilogue.  The pool and the reductions
//     over the group's heads run at the end of each piece.
//   * The KV heads of a block meet last: each group's entry sums and block values go to
//     global memory, a per-block ticket counts the KV heads, and the last arrival sums
//     the entries in KV-head order and takes the block maximum.
//   * Roles: a producer warp (key copies, block lists), an MMA warp (one thread issues
//     tcgen05.mma, commits to mbarriers, and copies a new group's queries once the old
//     ones' MMAs are done), a statistics warp and sixteen epilogue warps.  For E4M3 caches the epilogue warps also decode stage s + 1's codes to f16
//     (exact) into the swizzled operand tile while stage s's MMAs run, and round a new
//     group's queries to f16 (exact in f16's normal range).  Both phases stream the
//     keys, so the layer's keys are read from HBM once and from L2 the second time.
//     Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cudaTypedefs.h>

#include "umma.cuh"

namespace kvs {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();   // attend_tc.cu

namespace {

constexpr int kD = 128;
constexpr int kObs = 32;                               // observation rows per head
constexpr int kGq = 8;                                 // query heads per KV head
constexpr int kRows = kGq * kObs;                      // 256 rows: head (r / 32), observation (r % 32)
constexpr uint32_t kQBytes = kRows * kD * 2;           // 64 KB query tile
constexpr uint32_t kQHalf = kRows * 128;               // one 64-element half of it
constexpr int kSB = 8;                                 // blocks per stage
constexpr int kSK = kSB * kBlock;                      // 128 keys per stage
constexpr uint32_t kTileBytes = kSK * kD * 2;          // 32 KB f16 / bf16 key tile
constexpr uint32_t kTileHalf = kSK * 128;
constexpr uint32_t kRawBytes = kSK * kD;               // 16 KB of E4M3 codes
constexpr int kPieceMax = 62;                          // phase-2 piece: + 2 halo blocks = 8 stages
constexpr int kVoteKeys = (kPieceMax + 2) * kBlock;    // votes kept per head
constexpr int kPool = 3;                               // max-pool radius (kernel 7)
constexpr int kInfo = 8;                               // stage-info ring
constexpr int kScRing = 4;                             // E4M3 key-scale ring
constexpr int kPieceList = 64;                         // pieces whose tickets wait for the end
// A run costs about this many blocks on top of its blocks (the group's query copy, the
// halo, the pool and the wait for the group's statistics), so the shares are cut in a
// flattened order where each group carries kRunCost blocks before its own.
constexpr int kRunCost = 12;
static_assert(2 * kPieceList * kPieceMax <= kGq * kVoteKeys, "the winner list lives in the votes buffer");
// An mbarrier poll suspends the thread until the phase completes or kSuspendNs pass, so
// a waiting warp takes no issue slots; kMbarLimit polls (about a second) bound a wait.
constexpr uint32_t kSuspendNs = 2000;
constexpr int kMbarLimit = 1 << 19;
constexpr float kLog2e = 1.4426950408889634f;

constexpr int kEpiWarps = 16, kEpiThreads = kEpiWarps * 32;
constexpr int kProdWarp = 16, kMmaWarp = 17, kStatWarp = 18;
constexpr int kBarEpi = 1;                             // named barrier of the epilogue warps

template <bool FP8>
struct PC {
  static constexpr int THREADS = (kStatWarp + 1) * 32;
  static constexpr int NK = FP8 ? 2 : 3;               // operand tiles
  static constexpr int NR = 3;                         // copy slots (E4M3: raw codes; bf16: the tiles)
};

// A stage as the producer describes it to the epilogue (the stage-info ring).
struct StageInfo {
  int32_t blk[kSB];                                    // block ids (-1: none)
  int32_t nb, flags, sl, kvh, b0, v0, c0, c1;          // as in Stage
};
enum : int32_t { kFPhase2 = 1, kFRunFirst = 2, kFRunLast = 4, kFPieceLast = 8, kFNewQ = 16, kFLast = 32 };

struct PsShared {
  uint64_t qfull, qready, qfree;
  uint64_t kfull[3], kempty[3], kready[2], kfree[2];
  uint64_t done[2], tfree[2];
  uint64_t info_full[kInfo];
  uint64_t mp_full[2], mp_empty[2];
  uint32_t tmem;
  int32_t abort;
  int32_t n_pieces;
  StageInfo info[kInfo];                               // the stage-info ring
  int32_t n_win;                                       // KV-head tickets won (the final combine)
  __align__(16) float sc[kScRing][kSK];                // E4M3: key scale x log2(e) / sqrt(D)
  __align__(16) float sc_raw[3][kSK];                  // E4M3: key scales as copied
  __align__(16) float mprime[2][kRows];                // phase 2: -M_row of a run, -inf = no row
  float merge[2][2][128];                              // phase 1: (max, sum) of the second key half
  int32_t pblk[kPieceMax + 2];                         // block ids of the piece's streamed blocks
  int32_t piece[kPieceList][3];                        // (group, first own block, end)
  int32_t seq_off[kPsSeqMax + 1];                      // weighted blocks before each sequence
};

struct PsArgs {
  Dev d;
  SeqSel sel;                 // the launch's sequences (slot sl is sequence sel.at(sl))
  int layer, n_seqs, n_obs;
};

// ------------------------------------------------------------------ PTX helpers
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n"
               " selp.u32 %0, 1, 0, p;\n}\n"
               : "=r"(ok) : "r"(bar), "r"(parity), "n"(kSuspendNs) : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity.  A wait that runs out records
// kErrTimeout and raises the CTA's abort flag, after which every wait of the CTA gives
// up at once: the roles then run out their loops without blocking.
__device__ __forceinline__ bool mbar_wait(const Dev& d, PsShared& sm, const uint64_t& b, uint32_t parity) {
  const uint32_t bar = smem_u32(&b);
  for (int it = 0; it < kMbarLimit; ++it) {
    if (mbar_test(bar, parity)) return true;
    if ((it & 15) == 15 && *reinterpret_cast<volatile int32_t*>(&sm.abort)) return false;
  }
  *reinterpret_cast<volatile int32_t*>(&sm.abort) = 1;
  set_error(d, kErrTimeout);
  return false;
}
// The same without the abort shortcut (the final drain of the MMA commits).
__device__ __forceinline__ void mbar_drain(const Dev& d, const uint64_t& b, uint32_t parity) {
  const uint32_t bar = smem_u32(&b);
  for (int it = 0; it < kMbarLimit; ++it)
    if (mbar_test(bar, parity)) return;
  set_error(d, kErrTimeout);
}
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int x, int y, int z, int w,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5}], [%6];"
      :: "r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
__device__ __forceinline__ void named_sync(int id, int n) {
  __syncwarp();
  asm volatile("barrier.sync %0, %1;" :: "r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void red_release_add(int32_t* p, int32_t v) {
  asm volatile("red.release.gpu.global.add.s32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
// 2^x with the hardware's approximate exponential (relative error about 2^-22).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Paired f32 arithmetic (one instruction for two lanes, each rounded as the scalar op).
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n mov.b64 rc, {%6, %7};\n"
      " fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " add.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  float2 d;
  asm("{\n .reg .b64 ra, rb, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %5};\n"
      " mul.rn.f32x2 rd, ra, rb;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d.x), "=f"(d.y) : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Maximum of 32 values as a tree of three-input maxima.
__device__ __forceinline__ float max32(const float (&v)[32]) {
  float a[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) a[i] = max3(v[3 * i], v[3 * i + 1], v[3 * i + 2]);
  a[10] = fmaxf(v[30], v[31]);
  const float b0 = max3(a[0], a[1], a[2]), b1 = max3(a[3], a[4], a[5]), b2 = max3(a[6], a[7], a[8]);
  return max3(max3(b0, b1, b2), a[9], a[10]);
}
// Sum over 32 values of 2^(v * c + o) (two lanes per instruction, four partial sums).
__device__ __forceinline__ float sum_ex2(const float (&v)[32], float c, float o) {
  const float2 c2 = make_float2(c, c), o2 = make_float2(o, o);
  float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const float2 x = fma2(make_float2(v[2 * i], v[2 * i + 1]), c2, o2);
    acc[i & 1] = add2(acc[i & 1], make_float2(ex2(x.x), ex2(x.y)));
  }
  return (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
}
// Four E4M3 codes (one 32-bit word) to four f16 (two words), exact.
__device__ __forceinline__ uint2 e4m3x4_f16x4(uint32_t w) {
  uint2 r;
  asm("{\n .reg .b16 lo, hi;\n mov.b32 {lo, hi}, %2;\n cvt.rn.f16x2.e4m3x2 %0, lo;\n cvt.rn.f16x2.e4m3x2 %1, hi;\n}"
      : "=r"(r.x), "=r"(r.y) : "r"(w));
  return r;
}
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w));
  const __half2 h = __floats2half2_rn(f.x, f.y);
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ void sts128(uint8_t* p, uint4 v) { *reinterpret_cast<uint4*>(p) = v; }

// Positions [a, b) of a block (first position p0) that a row sees: resident and not
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

// ------------------------------------------------------------------ the stage schedule
// Every role walks the same schedule: phase 1 over the CTA's runs in stages of 8 blocks,
// then phase 2 over the same runs, each cut into pieces whose streamed blocks include one
// halo block on each side.
struct Stage {
  int phase;            // 0: phase 1 (row statistics), 1: phase 2 (votes)
  int sl, kvh, n;       // group (launch slot, KV head) and the sequence's resident blocks
  int64_t gs;           // weighted flattened index of the group's first block
  int b0, nb;           // streamed blocks [b0, b0 + nb), group-local
  int v0, c0, c1;       // the piece's first streamed block and its own blocks [c0, c1)
  bool run_first, run_last, piece_last, new_q;
};

struct Sched {
  const int32_t* off;
  int n_seqs, hkv;
  int64_t x0, x1, gs;
  int phase, sl, kvh, n, i1, p0, p1, v0, e, b, prev_g;
  bool live, first;

  __device__ void init(const int32_t* off_, int n_seqs_, int hkv_, int64_t x0_, int64_t x1_) {
    off = off_;
    n_seqs = n_seqs_;
    hkv = hkv_;
    x0 = x0_;
    x1 = x1_;
    phase = 0;
    prev_g = -1;
    live = x0 < x1 && start_run(x0);
  }
  // the first run at or after weighted index x, false if the share holds no block there.
  // x's sequence is the last slot that starts at or before x (an empty sequence carries
  // no weight, so that slot is not empty); x lies in a group's charge or in its blocks,
  // and when the share ends inside the charge, no later group meets the share either.
  __device__ bool start_run(int64_t x) {
    int lo = 0, hi = n_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if ((int64_t)hkv * off[mid] <= x) lo = mid;
      else hi = mid - 1;
    }
    sl = lo;
    const int w = off[sl + 1] - off[sl];
    n = w - kRunCost;
    const int64_t base = (int64_t)hkv * off[sl];
    kvh = (int)((x - base) / w);
    gs = base + (int64_t)kvh * w + kRunCost;
    i1 = (int)(x1 - gs < n ? x1 - gs : n);
    p0 = (int)(x > gs ? x - gs : 0);
    if (i1 <= p0) return false;
    first = true;
    start_piece();
    return true;
  }
  __device__ void start_piece() {
    if (phase == 0) {
      p1 = i1;
      v0 = p0;
      e = i1;
    } else {
      p1 = min(p0 + kPieceMax, i1);
      v0 = max(p0 - 1, 0);
      e = min(p1 + 1, n);
    }
    b = v0;
  }
  __device__ bool next(Stage& s) {
    if (!live) return false;
    s.phase = phase;
    s.sl = sl;
    s.kvh = kvh;
    s.n = n;
    s.gs = gs;
    s.b0 = b;
    s.nb = min(kSB, e - b);
    s.v0 = v0;
    s.c0 = p0;
    s.c1 = p1;
    const int g = sl * hkv + kvh;
    s.new_q = g != prev_g;
    prev_g = g;
    s.run_first = first;
    first = false;
    b += s.nb;
    s.piece_last = b >= e;
    s.run_last = false;
    if (s.piece_last) {
      if (phase == 1 && p1 < i1) {
        p0 = p1;
        start_piece();
      } else {
        s.run_last = true;
        const int64_t x = gs + i1;
        if (x < x1 && start_run(x)) {
        } else if (phase == 0) {
          phase = 1;
          start_run(x0);
        } else {
          live = false;
        }
      }
    }
    return true;
  }
};

// ------------------------------------------------------------------ the kernel
template <bool FP8>
__global__ void __launch_bounds__(PC<FP8>::THREADS, 1)
    ps_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk, const PsArgs A) {
  using C = PC<FP8>;
  extern __shared__ __align__(1024) uint8_t dyn_raw[];
  const uint32_t raw_addr = smem_u32(dyn_raw);
  uint8_t* qt = dyn_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
  uint8_t* tiles = qt + kQBytes;
  uint8_t* raws = tiles + C::NK * kTileBytes;
  float* votes = reinterpret_cast<float*>(raws + (FP8 ? C::NR * kRawBytes : 0));   // [8 heads][kVoteKeys]
  PsShared& sm = *reinterpret_cast<PsShared*>(votes + kGq * kVoteKeys);
  const Dev& d = A.d;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- the launch's layout: seq_off[i] = weighted blocks of slots 0 .. i-1 (a sequence
  // with n > 0 resident blocks weighs n + kRunCost per KV head)
  for (int i = tid; i < A.n_seqs; i += C::THREADS) {
    const int s = A.sel.at(i);
    int n = 0;
    if (KVS_DCHECK(d, s >= 0 && s < d.max_seqs)) n = min(seq_blocks(d, A.layer, s).n, d.ps_bound);
    sm.seq_off[i + 1] = n > 0 ? n + kRunCost : 0;
  }
  __syncthreads();
  if (warp == 0) {
    const int per = (A.n_seqs + 31) / 32, a = lane * per, end = min(a + per, A.n_seqs);
    int tot = 0;
    for (int i = a; i < end; ++i) tot += sm.seq_off[i + 1];
    int incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int run = incl - tot;
    for (int i = a; i < end; ++i) {
      run += sm.seq_off[i + 1];
      sm.seq_off[i + 1] = run;
    }
    if (lane == 0) sm.seq_off[0] = 0;
  }
  __syncthreads();
  const int64_t T = (int64_t)d.Hkv * sm.seq_off[A.n_seqs];
  if (T == 0) return;
  // CTAs with work: shares of at least kRunCost + 4, so every share holds a block (between
  // two groups' charges lies at least one block)
  const int64_t Ge = min((int64_t)gridDim.x, max((int64_t)1, T / (kRunCost + 4)));
  const int c = blockIdx.x;
  if (c >= Ge) return;
  const int64_t x0 = c * T / Ge, x1 = (c + 1) * T / Ge;

  if (tid == 0) {
    mbar_init(smem_u32(&sm.qfull), 1);
    mbar_init(smem_u32(&sm.qready), kEpiWarps);
    mbar_init(smem_u32(&sm.qfree), 1);
    for (int i = 0; i < 3; ++i) {
      mbar_init(smem_u32(&sm.kfull[i]), 1);
      mbar_init(smem_u32(&sm.kempty[i]), FP8 ? kEpiWarps : 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(smem_u32(&sm.kready[i]), kEpiWarps);
      mbar_init(smem_u32(&sm.kfree[i]), 1);
      mbar_init(smem_u32(&sm.done[i]), 1);
      mbar_init(smem_u32(&sm.tfree[i]), kEpiWarps);
      mbar_init(smem_u32(&sm.mp_full[i]), 1);
      mbar_init(smem_u32(&sm.mp_empty[i]), 1);
    }
    for (int i = 0; i < kInfo; ++i) mbar_init(smem_u32(&sm.info_full[i]), 1);
    sm.abort = 0;
    sm.n_pieces = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  // query rows n_obs .. 31 of every head stay zero: the copies fill rows < n_obs only
  if (A.n_obs < kObs) {
    const int zrows = kObs - A.n_obs, nz = 2 * kGq * zrows * 8;
    for (int i = tid; i < nz; i += C::THREADS) {
      const int kh = i / (kGq * zrows * 8), rem = i % (kGq * zrows * 8), hl = rem / (zrows * 8);
      const int r = A.n_obs + (rem % (zrows * 8)) / 8, ch = i % 8;
      sts128(qt + kh * kQHalf + (hl * kObs + r) * 128 + ch * 16, make_uint4(0u, 0u, 0u, 0u));
    }
    umma::fence_async_smem();
  }
  if (warp == kMmaWarp) {
    umma::alloc(smem_u32(&sm.tmem), 512);
    umma::relinquish();
  }
  umma::fence_before();
  __syncthreads();
  umma::fence_after();
  const uint32_t tmem = sm.tmem;
  const float qk_scale = kLog2e / sqrtf((float)kD);

  if (warp == kProdWarp) {
    // ============================================================ producer
    Sched S;
    S.init(sm.seq_off, A.n_seqs, d.Hkv, x0, x1);
    Stage st;
    int s = 0, cur = -1, sid = 0;
    SeqBlocks sb{};
    const uint8_t* kl = d.k_pages + (size_t)A.layer * d.page_layer_bytes;
    const float* kscl = FP8 ? d.k_scales + (size_t)A.layer * d.slot_layer_elems : nullptr;
    while (S.next(st)) {
      if (st.sl != cur) {
        cur = st.sl;
        sid = A.sel.at(st.sl);
        sb = seq_blocks(d, A.layer, sid);
      }
      // the stage's keys first: they do not wait for the query tile to be free
      const int slot = s % C::NR;
      if (lane == 0 && s >= C::NR) mbar_wait(d, sm, sm.kempty[slot], ((s / C::NR) - 1) & 1);
      __syncwarp();
      int32_t blk = -1, page = 0;
      if (lane < st.nb) {
        blk = block_at(d, sid, sb, st.b0 + lane, &page);
        if (!KVS_DCHECK(d, page >= 0 && page < d.num_pages)) page = 0;
      }
      StageInfo& info = sm.info[s % kInfo];
      if (lane < kSB) info.blk[lane] = blk;
      if (lane == 0) {
        info.nb = st.nb;
        info.flags = (st.phase ? kFPhase2 : 0) | (st.run_first ? kFRunFirst : 0) | (st.run_last ? kFRunLast : 0) |
                     (st.piece_last ? kFPieceLast : 0) | (st.new_q ? kFNewQ : 0) | (S.live ? 0 : kFLast);
        info.sl = st.sl;
        info.kvh = st.kvh;
        info.b0 = st.b0;
        info.v0 = st.v0;
        info.c0 = st.c0;
        info.c1 = st.c1;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sm.info_full[s % kInfo]));
        mbar_expect_tx(smem_u32(&sm.kfull[slot]),
                       (uint32_t)st.nb * (FP8 ? kBlock * kD + kBlock * 4 : kBlock * kD * 2));
      }
      __syncwarp();
      if (lane < st.nb) {
        const uint32_t bar = smem_u32(&sm.kfull[slot]);
        if constexpr (FP8) {
          bulk_load(smem_u32(raws + slot * kRawBytes + lane * kBlock * kD),
                    kl + (size_t)page * d.page_bytes + (size_t)st.kvh * kBlock * kD, kBlock * kD, bar);
          bulk_load(smem_u32(&sm.sc_raw[slot][lane * kBlock]), kscl + (size_t)page * kBlock, kBlock * 4, bar);
        } else {
#pragma unroll
          for (int kh = 0; kh < 2; ++kh)
            tma_load_4d(smem_u32(tiles + slot * kTileBytes + kh * kTileHalf + lane * kBlock * 128), &tk, 64 * kh, 0,
                        st.kvh, page, bar);
        }
      }
      ++s;
    }
  } else if (warp == kMmaWarp) {
    // ============================================================ MMA issue
    if (lane == 0) {
      Sched S;
      S.init(sm.seq_off, A.n_seqs, d.Hkv, x0, x1);
      Stage st;
      int s = 0, qn = 0;
      const uint32_t qs = smem_u32(qt), ts = smem_u32(tiles);
      while (S.next(st)) {
        if (st.new_q) {
          // a new group's queries: once the old ones' MMAs are done, this thread copies
          // them (the producer keeps streaming keys meanwhile)
          if (qn > 0) {
            umma::commit(smem_u32(&sm.qfree));
            mbar_wait(d, sm, sm.qfree, (qn - 1) & 1);
          }
          mbar_expect_tx(smem_u32(&sm.qfull), 2u * kGq * A.n_obs * 128u);
          for (int kh = 0; kh < 2; ++kh)
            for (int hl = 0; hl < kGq; ++hl)
              tma_load_4d(smem_u32(qt + kh * kQHalf + hl * kObs * 128), &tq, 64 * kh, st.kvh * kGq + hl, 0, st.sl,
                          smem_u32(&sm.qfull));
          mbar_wait(d, sm, FP8 ? sm.qready : sm.qfull, qn & 1);
          ++qn;
        }
        const int t = s % C::NK;
        mbar_wait(d, sm, FP8 ? sm.kready[t] : sm.kfull[t], (s / C::NK) & 1);
        const int buf = s & 1;
        if (s >= 2) mbar_wait(d, sm, sm.tfree[buf], ((s >> 1) - 1) & 1);
        umma::fence_after();
        const uint32_t dt = tmem + buf * 256, ks = ts + t * kTileBytes;
        if (st.phase == 0) {
          constexpr uint32_t idesc = umma::idesc_f16(!FP8, 128, kSK);
          for (int m = 0; m < 2; ++m)
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk) {
              const uint64_t ad = umma::sw128_desc(qs + (kk / 4) * kQHalf + m * (128 * 128) + (kk % 4) * 32);
              const uint64_t bd = umma::sw128_desc(ks + (kk / 4) * kTileHalf + (kk % 4) * 32);
              umma::mma_f16(dt + m * kSK, ad, bd, idesc, kk > 0);
            }
        } else {
          constexpr uint32_t idesc = umma::idesc_f16(!FP8, 128, kRows);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            const uint64_t ad = umma::sw128_desc(ks + (kk / 4) * kTileHalf + (kk % 4) * 32);
            const uint64_t bd = umma::sw128_desc(qs + (kk / 4) * kQHalf + (kk % 4) * 32);
            umma::mma_f16(dt, ad, bd, idesc, kk > 0);
          }
        }
        umma::commit(smem_u32(&sm.done[buf]));
        umma::commit(smem_u32(FP8 ? &sm.kfree[t] : &sm.kempty[t]));
        ++s;
      }
      // every slot's last commit has landed before TMEM and the barriers go away
      for (int j = max(0, s - C::NK); j < s; ++j) mbar_drain(d, FP8 ? sm.kfree[j % C::NK] : sm.kempty[j % C::NK], (j / C::NK) & 1);
    }
    __syncwarp();
  } else if (warp == kStatWarp) {
    // ============================================================ statistics (phase 2)
    // Per phase-2 run: wait for every CTA that shares the group to publish its row
    // partials, merge them into M_row = max + log2(sum), hand them to the epilogue.
    Sched S;
    S.init(sm.seq_off, A.n_seqs, d.Hkv, x0, x1);
    Stage st;
    int r = 0;
    while (S.next(st)) {
      if (st.phase != 1 || !st.run_first) continue;
      const int slot = r & 1;
      if (r >= 2) mbar_wait(d, sm, sm.mp_empty[slot], ((r >> 1) - 1) & 1);
      const int g = st.sl * d.Hkv + st.kvh;
      // the CTAs whose shares meet the group's blocks: CTA of weighted index x = ((x + 1) Ge - 1) / T
      const int cf = (int)(((st.gs + 1) * Ge - 1) / T), cl = (int)(((st.gs + st.n) * Ge - 1) / T);
      const int need = cl - cf + 1;
      if (lane == 0 && !wait_at_least(&d.ps_ready[g], need, d.spin_limit)) set_error(d, kErrTimeout);
      __syncwarp();
#pragma unroll 1
      for (int j = 0; j < kGq; ++j) {
        const int row = j * kObs + lane;
        float M = -INFINITY, Ls = 0.f;
        for (int cc = cf; cc <= cl; ++cc) {
          const float2 pp = __ldcg(&d.ps_part[(size_t)(cc + g) * kRows + row]);
          const float mn = fmaxf(M, pp.x);
          if (mn == -INFINITY) continue;
          Ls = Ls * ex2(M - mn) + pp.y * ex2(pp.x - mn);
          M = mn;
        }
        sm.mprime[slot][row] = (lane < A.n_obs && Ls > 0.f) ? -(M + __log2f(Ls)) : -INFINITY;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sm.mp_full[slot]));
        // the last CTA of the group to pass its wait resets the group's counters
        if (atomicAdd(&d.ps_done[g], 1) == need - 1) {
          d.ps_ready[g] = 0;
          d.ps_done[g] = 0;
        }
      }
      ++r;
    }
  } else if (warp < kEpiWarps) {
    // ============================================================ epilogue
    const int q = warp >> 2, wl = warp & 3;
    const uint32_t lane_base = (uint32_t)(32 * wl) << 16;
    int s = 0, r = 0, qn = 0, cur = -1, sid = 0;
    SeqBlocks sb{};
    int64_t obs0 = 0;
    float m_run = -INFINITY, l_run = 0.f;
    const float cs = FP8 ? 1.f : qk_scale;   // bf16: the logits stay raw until the exponent
    // E4M3: the thread decodes codes 16 c16 .. 16 c16 + 15 of keys dk_key and dk_key + 64
    // (c16 = tid % 8); their places in the raw copy and in the swizzled tile are the same
    // every stage
    const int dk_key = tid >> 3, dk_c16 = tid & 7;
    const int dk_src = dk_key * kD + dk_c16 * 16;
    const int dk_dst = (int)umma::sw128_offset(kSK, dk_key, 16 * dk_c16);
    const int dk_dst8 = (int)umma::sw128_offset(kSK, dk_key, 16 * dk_c16 + 8);
    // E4M3: this thread's share of stage j's decode (codes to f16 in the swizzled tile
    // j % 2, scales x log2(e)/sqrt(D) to the ring); returns whether stage j starts a
    // group.  Tile j % 2 is free: this warp waited for stage j - 2's MMAs one stage ago.
    auto decode_keys = [&](int j) -> bool {
      mbar_wait(d, sm, sm.info_full[j % kInfo], (j / kInfo) & 1);
      const int nb = sm.info[j % kInfo].nb;
      const bool nq = (sm.info[j % kInfo].flags & kFNewQ) != 0;
      const int slot = j % C::NR;
      mbar_wait(d, sm, sm.kfull[slot], (j / C::NR) & 1);
      const uint8_t* rw = raws + slot * kRawBytes;
      uint8_t* kt = tiles + (j % C::NK) * kTileBytes;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {                // keys dk_key and dk_key + 64
        if (dk_key + 64 * h2 >= nb * kBlock) break;
        const uint4 cw = *reinterpret_cast<const uint4*>(rw + dk_src + h2 * 64 * kD);
        const uint2 a = e4m3x4_f16x4(cw.x), b = e4m3x4_f16x4(cw.y), c2 = e4m3x4_f16x4(cw.z), e = e4m3x4_f16x4(cw.w);
        sts128(kt + dk_dst + h2 * 64 * 128, make_uint4(a.x, a.y, b.x, b.y));
        sts128(kt + dk_dst8 + h2 * 64 * 128, make_uint4(c2.x, c2.y, e.x, e.y));
      }
      if (tid < kSK) sm.sc[j % kScRing][tid] = tid < nb * kBlock ? sm.sc_raw[slot][tid] * qk_scale : 0.f;
      umma::fence_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(smem_u32(&sm.kready[j % C::NK]));
        mbar_arrive(smem_u32(&sm.kempty[slot]));
      }
      return nq;
    };
    // E4M3: this thread's share of a new group's queries, rounded to f16 in place
    auto round_queries = [&]() {
      mbar_wait(d, sm, sm.qfull, qn & 1);
      for (int i = tid; i < (int)(kQBytes / 16); i += kEpiThreads) {
        uint4* p = reinterpret_cast<uint4*>(qt + 16 * i);
        const uint4 v = *p;
        *p = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
      }
      umma::fence_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.qready));
      ++qn;
    };
    if constexpr (FP8) {          // the first stage starts a group
      round_queries();
      decode_keys(0);
    }
    for (;; ++s) {
      const int slot8 = s % kInfo, buf = s & 1;
      mbar_wait(d, sm, sm.info_full[slot8], (s / kInfo) & 1);
      // the stage's description stays in its ring slot until this stage is done here
      const StageInfo& I = sm.info[slot8];
      const int fl = I.flags;
      const bool more = !(fl & kFLast);   // a stage s + 1 follows
      bool next_new_q = false;
      if constexpr (FP8)
        if (more) next_new_q = decode_keys(s + 1);
      if (I.sl != cur) {
        cur = I.sl;
        sid = A.sel.at(cur);
        sb = seq_blocks(d, A.layer, sid);
        obs0 = sb.next - A.n_obs;
      }
      // E4M3: every warp's share of the stage's decode, scales included, is in
      if constexpr (FP8) mbar_wait(d, sm, sm.kready[s % C::NK], (s / C::NK) & 1);
      mbar_wait(d, sm, sm.done[buf], (s >> 1) & 1);
      umma::fence_after();
      const float* scs = sm.sc[s % kScRing];
      const uint32_t tcol = tmem + lane_base + buf * 256;
      if (!(fl & kFPhase2)) {
        // row = 128 t + 32 wl + lane: head 4 t + wl, observation lane; warpgroup q takes
        // row half t = q & 1 and the stage's key half kh = q >> 1 (blocks 4 kh .. 4 kh + 3)
        if (fl & kFRunFirst) {
          m_run = -INFINITY;
          l_run = 0.f;
        }
        const int t = q & 1, kh = q >> 1;
        const int64_t obs_i = obs0 + lane;
        const bool row_ok = lane < A.n_obs;
        // 32-key chunks u with a block in the stage (first block 4 kh + 2 u < nb)
        const int nb = I.nb;
        const int nu = nb > 4 * kh + 2 ? 2 : (nb > 4 * kh ? 1 : 0);
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          if (u >= nu) break;
          float v[32];
          umma::ld32(tcol + t * kSK + 64 * kh + 32 * u, v);
          const int j0 = 4 * kh + 2 * u;
          if constexpr (FP8) {
            const float4* s4 = reinterpret_cast<const float4*>(scs + 16 * j0);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
              const float4 sc = s4[q4];
              const float2 a = mul2(make_float2(v[4 * q4], v[4 * q4 + 1]), make_float2(sc.x, sc.y));
              const float2 b = mul2(make_float2(v[4 * q4 + 2], v[4 * q4 + 3]), make_float2(sc.z, sc.w));
              v[4 * q4] = a.x;
              v[4 * q4 + 1] = a.y;
              v[4 * q4 + 2] = b.x;
              v[4 * q4 + 3] = b.y;
            }
          }
#pragma unroll
          for (int bb = 0; bb < 2; ++bb) {
            const int jb = j0 + bb;
            if (jb >= nb) {
#pragma unroll
              for (int cc = 0; cc < kBlock; ++cc) v[16 * bb + cc] = -INFINITY;
              continue;
            }
            const int64_t p0 = (int64_t)I.blk[jb] * kBlock;
            if (p0 < sb.lo || p0 + kBlock - 1 > obs0) {     // not every row sees every entry
              const RowWin w = row_window(sb, p0, obs_i, row_ok);
#pragma unroll
              for (int cc = 0; cc < kBlock; ++cc)
                if (cc < w.a || cc >= w.b) v[16 * bb + cc] = -INFINITY;
            }
          }
          const float bm = max32(v);
          if (bm != -INFINITY) {
            const float mn = fmaxf(m_run, bm);
            const float acc = sum_ex2(v, cs, -mn * cs);
            l_run = l_run * ex2((m_run - mn) * cs) + acc;
            m_run = mn;
          }
        }
        if (fl & kFRunLast) {
          // the two key halves of a row merge; lane = row, so no shuffles
          const int row = 32 * wl + lane;
          if (kh == 1) {
            sm.merge[t][0][row] = m_run;
            sm.merge[t][1][row] = l_run;
          }
          named_sync(kBarEpi, kEpiThreads);
          if (kh == 0) {
            const float mo = sm.merge[t][0][row], lo = sm.merge[t][1][row], mn = fmaxf(m_run, mo);
            const float l = mn == -INFINITY ? 0.f : l_run * ex2((m_run - mn) * cs) + lo * ex2((mo - mn) * cs);
            const int g = I.sl * d.Hkv + I.kvh;
            d.ps_part[(size_t)(c + g) * kRows + 128 * t + row] = make_float2(mn * cs, l);
          }
          named_sync(kBarEpi, kEpiThreads);
          if (tid == 0) red_release_add(&d.ps_ready[I.sl * d.Hkv + I.kvh], 1);
        }
      } else {
        // thread = key L of the stage; warpgroup q takes heads 2 q, 2 q + 1, whose 32
        // observation rows are 32 TMEM columns each
        if (fl & kFRunFirst) mbar_wait(d, sm, sm.mp_full[r & 1], (r >> 1) & 1);
        const float* nmp = sm.mprime[r & 1];                // -M_row
        const int L = 32 * wl + lane, jb = L >> 4, vb = I.b0 - I.v0, nb = I.nb;
        if (warp == 0 && lane < nb) sm.pblk[vb + lane] = I.blk[lane];
        if (2 * wl < nb) {
          const bool key_ok = jb < nb;
          int64_t p = 0;
          bool res = false;
          if (key_ok) {
            p = (int64_t)I.blk[jb] * kBlock + (L & 15);
            res = p >= sb.lo && p < sb.next;
          }
          const int64_t rel = p - obs0;                    // rows i < rel do not see it
          const int lim = !key_ok || rel <= 0 ? 0 : (rel >= kObs ? kObs : (int)rel);
          const float sck = FP8 ? scs[L] : qk_scale;
          const float2 s2 = make_float2(sck, sck);
          const bool all_rows = __all_sync(0xffffffffu, lim == 0);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            const int h = 2 * q + hh;
            float v[32];
            umma::ld32(tcol + 32 * h, v);
            float sum = 0.f;
            if (all_rows) {
              const float4* nm4 = reinterpret_cast<const float4*>(nmp + h * kObs);
              float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
              for (int q4 = 0; q4 < 8; ++q4) {
                const float4 m4 = nm4[q4];
                const float2 x = fma2(make_float2(v[4 * q4], v[4 * q4 + 1]), s2, make_float2(m4.x, m4.y));
                const float2 y = fma2(make_float2(v[4 * q4 + 2], v[4 * q4 + 3]), s2, make_float2(m4.z, m4.w));
                acc[0] = add2(acc[0], make_float2(ex2(x.x), ex2(x.y)));
                acc[1] = add2(acc[1], make_float2(ex2(y.x), ex2(y.y)));
              }
              sum = (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
            } else {
#pragma unroll
              for (int i = 0; i < kObs; ++i)
                if (i >= lim) sum += ex2(fmaf(v[i], sck, nmp[h * kObs + i]));
            }
            if (key_ok) votes[h * kVoteKeys + vb * kBlock + L] = res ? sum : 0.f;
          }
        }
        if (fl & kFPieceLast) {
          named_sync(kBarEpi, kEpiThreads);
          // ---- pool and reduce the piece's own blocks [c0, c1).  Positions inside a
          // block are consecutive; across blocks they are when the next streamed block is
          // the next block id.  A key that is not resident has vote 0, so it can sit in a
          // max without changing it, but its own pooled value is 0.
          const int c0 = I.c0, c1 = I.c1, nstream = I.b0 + nb - I.v0, lo_halo = c0 - I.v0, nblk = c1 - c0;
          const int g = I.sl * d.Hkv + I.kvh;
          const size_t gbase = (size_t)g * d.ps_bound + c0;
          // thread = (own block b = tid / 8, head hl = tid % 8): the block's 16 votes and 3
          // on each side (0 where the neighbouring block is not the adjacent block id)
          // in registers, the 16 pooled values, their sum; the 8 heads of a block are 8
          // consecutive lanes, which reduce the block value (max) and the entry sums
          static_assert(kEpiThreads >= kGq * kPieceMax, "one thread per (head, block) of a piece");
          const int hl = tid & 7, b = tid >> 3;
          const bool live = b < nblk;
          const int sb_i = lo_halo + b;                    // streamed block index
          float pooled[kBlock];
#pragma unroll
          for (int cc = 0; cc < kBlock; ++cc) pooled[cc] = 0.f;
          float bsum = 0.f;
          int32_t blk = 0;
          if (live) {
            blk = sm.pblk[sb_i];
            const bool prev = sb_i > 0 && sm.pblk[sb_i - 1] == blk - 1;
            const bool next = sb_i + 1 < nstream && sm.pblk[sb_i + 1] == blk + 1;
            const float* vr = votes + hl * kVoteKeys + sb_i * kBlock;
            float w[kBlock + 2 * kPool];
#pragma unroll
            for (int k = 0; k < kPool; ++k) {
              w[k] = prev ? vr[k - kPool] : 0.f;
              w[kBlock + kPool + k] = next ? vr[kBlock + k] : 0.f;
            }
#pragma unroll
            for (int cc = 0; cc < kBlock; ++cc) w[kPool + cc] = vr[cc];
            const int64_t p0 = (int64_t)blk * kBlock;
#pragma unroll
            for (int cc = 0; cc < kBlock; ++cc) {
              const bool res = p0 + cc >= sb.lo && p0 + cc < sb.next;
              const float m = max3(max3(w[cc], w[cc + 1], w[cc + 2]), max3(w[cc + 3], w[cc + 4], w[cc + 5]), w[cc + 6]);
              pooled[cc] = res ? m : 0.f;
              bsum += pooled[cc];
            }
          }
          float mx = bsum;
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          // entry sums over the 8 heads: a reduce-scatter over the block's 8 lanes leaves
          // lane hl with entries e0 = 8 bit2(hl) + 4 bit1(hl) + 2 bit0(hl) and e0 + 1
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const bool up = (hl & 4) != 0;
            const float give = up ? pooled[k] : pooled[k + 8];
            const float got = __shfl_xor_sync(0xffffffffu, give, 4);
            pooled[k] = (up ? pooled[k + 8] : pooled[k]) + got;
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const bool up = (hl & 2) != 0;
            const float give = up ? pooled[k] : pooled[k + 4];
            const float got = __shfl_xor_sync(0xffffffffu, give, 2);
            pooled[k] = (up ? pooled[k + 4] : pooled[k]) + got;
          }
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const bool up = (hl & 1) != 0;
            const float give = up ? pooled[k] : pooled[k + 2];
            const float got = __shfl_xor_sync(0xffffffffu, give, 1);
            pooled[k] = (up ? pooled[k + 2] : pooled[k]) + got;
          }
          if (live) {
            const int e0 = 8 * ((hl >> 2) & 1) + 4 * ((hl >> 1) & 1) + 2 * (hl & 1);
            d.ps_tok[(gbase + b) * kBlock + e0] = pooled[0];
            d.ps_tok[(gbase + b) * kBlock + e0 + 1] = pooled[1];
            record_head(d, A.layer, sid, blk, I.kvh * kGq + hl, bsum);   // head profiles
            if (hl == 0) d.ps_blk[gbase + b] = mx;
          }
          if (tid == 0) {
            const int k = sm.n_pieces;
            sm.piece[k][0] = g;
            sm.piece[k][1] = c0;
            sm.piece[k][2] = c1;
            sm.n_pieces = k + 1;
          }
          named_sync(kBarEpi, kEpiThreads);
          if (fl & kFRunLast) {
            if (tid == 0) mbar_arrive(smem_u32(&sm.mp_empty[r & 1]));
            ++r;
          }
        }
      }
      umma::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&sm.tfree[buf]));
      // E4M3: stage s + 1 starts a group whose queries land once stage s's MMAs are done
      if constexpr (FP8)
        if (next_new_q) round_queries();

      // ---- the KV heads of a block meet: per (sequence, block) a ticket counts the
      // groups that wrote it; the last one sums the entries (KV-head order) and takes the
      // block maximum.  Run at the end, or when the piece list is full.
      const bool flush = !more || ((fl & kFPieceLast) && (fl & kFPhase2) && sm.n_pieces == kPieceList);
      if (flush && sm.n_pieces > 0) {
        // (1) one thread per owned block takes its ticket; the winners are listed as
        // (piece, block) pairs in the votes buffer, free between pieces (the pieces own at
        // most kPieceList * kPieceMax blocks, fewer than the buffer's pairs)
        const int np = sm.n_pieces;
        int32_t* win = reinterpret_cast<int32_t*>(votes);
        if (tid == 0) sm.n_win = 0;
        named_sync(kBarEpi, kEpiThreads);
        for (int k = 0; k < np; ++k) {
          const int g = sm.piece[k][0], c0 = sm.piece[k][1], c1 = sm.piece[k][2];
          for (int i = c0 + tid; i < c1; i += kEpiThreads) {
            __threadfence();
            int32_t* tk2 = &d.ps_tickets[(size_t)(g / d.Hkv) * d.ps_bound + i];
            if (atomicAdd(tk2, 1) == d.Hkv - 1) {
              *tk2 = 0;
              const int at = atomicAdd(&sm.n_win, 1);
              win[2 * at] = k;
              win[2 * at + 1] = i;
            }
          }
        }
        named_sync(kBarEpi, kEpiThreads);
        // (2) per won block its 16 entries (sum over KV heads, in order) and its block value
        // (max over KV heads), one (block, item) per thread
        __threadfence();
        const int nw = sm.n_win;
        float* tok = d.tok_mass + (size_t)A.layer * d.slot_layer_elems;
        for (int it = tid; it < nw * (kBlock + 1); it += kEpiThreads) {
          const int w = it / (kBlock + 1), cc = it % (kBlock + 1);
          const int k = win[2 * w], i = win[2 * w + 1];
          const int sl = sm.piece[k][0] / d.Hkv, sq = A.sel.at(sl);
          const SeqBlocks sbk = seq_blocks(d, A.layer, sq);
          int32_t page;
          const int32_t blk = block_at(d, sq, sbk, i, &page);
          const size_t sbase = (size_t)sl * d.Hkv * d.ps_bound + i;
          if (cc < kBlock) {
            const int64_t p = (int64_t)blk * kBlock + cc;
            if (p < sbk.lo || p >= sbk.next) continue;
            float v8[8];
#pragma unroll
            for (int g2 = 0; g2 < 8; ++g2)
              v8[g2] = g2 < d.Hkv ? __ldcg(d.ps_tok + (sbase + (size_t)g2 * d.ps_bound) * kBlock + cc) : 0.f;
            float tsum = 0.f;
#pragma unroll
            for (int g2 = 0; g2 < 8; ++g2) tsum += v8[g2];
            int32_t slot;
            const int32_t pg = page_of(d, sq, p, &slot);
            tok[(size_t)pg * kBlock + slot] = tsum;
          } else {
            float v8[8];
#pragma unroll
            for (int g2 = 0; g2 < 8; ++g2) v8[g2] = g2 < d.Hkv ? __ldcg(d.ps_blk + sbase + (size_t)g2 * d.ps_bound) : 0.f;
            float mx = 0.f;
#pragma unroll
            for (int g2 = 0; g2 < 8; ++g2) mx = fmaxf(mx, v8[g2]);
            d.blk_mass[(size_t)A.layer * d.blk_layer_elems + (size_t)sq * d.max_blocks + blk] = mx;
          }
        }
        named_sync(kBarEpi, kEpiThreads);
        if (tid == 0) sm.n_pieces = 0;
        named_sync(kBarEpi, kEpiThreads);
      }
      if (!more) break;
    }
  }
  __syncthreads();
  if (warp == kMmaWarp) {
    umma::fence_after();
    umma::dealloc(tmem, 512);
  }
}

size_t ps_smem(bool fp8) {
  const size_t tiles = (size_t)(fp8 ? PC<true>::NK : PC<false>::NK) * kTileBytes;
  const size_t raws = fp8 ? (size_t)PC<true>::NR * kRawBytes : 0;
  return 1024 + kQBytes + tiles + raws + (size_t)kGq * kVoteKeys * 4 + sizeof(PsShared);
}

template <bool FP8>
cudaError_t launch_ps(const CUtensorMap& tq, const CUtensorMap& tk, const PsArgs& A, int grid, cudaStream_t st) {
  auto fn = ps_kernel<FP8>;
  const size_t smem = ps_smem(FP8);
  static std::atomic<unsigned long long> optin{0};   // per device
  const cudaError_t e = smem_optin_once(optin, fn, (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(PC<FP8>::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  // cooperative: every CTA resident at once (a CTA waits for the others' row partials)
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, fn, tq, tk, A);
}

// Tensor map over the observation queries [n_seqs][n_obs][Hq][D] bf16, viewed with the
// head before the observation so that one box (64 elements x 1 head x n_obs rows) is a
// head's rows of one 64-element half, landing as consecutive 128-byte rows.
cudaError_t make_q_map(CUtensorMap* map, const void* q, int Hq, int n_obs, int n_seqs) {
  PFN_cuTensorMapEncodeTiled_v12000 encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)Hq, (cuuint64_t)n_obs, (cuuint64_t)n_seqs};
  cuuint64_t strides[3] = {(cuuint64_t)kD * 2, (cuuint64_t)Hq * kD * 2, (cuuint64_t)n_obs * Hq * kD * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)n_obs, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUresult res = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(q), dims, strides, box, estr,
                              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

}  // namespace

int prefill_obs_max() { return kObs; }

cudaError_t launch_prefill_score(const Dev& d, const CUtensorMap* k_map, int layer, SeqSel sel, int n_seqs,
                                 const void* q_obs, int n_obs, int grid, cudaStream_t st) {
  const bool fp8 = d.kv_dtype == KVS_E4M3;
  if (!fp8 && !k_map) return cudaErrorInvalidValue;
  CUtensorMap none;
  memset(&none, 0, sizeof(none));
  for (int off = 0; off < n_seqs; off += kPsSeqMax) {
    const int cnt = n_seqs - off < kPsSeqMax ? n_seqs - off : kPsSeqMax;
    PsArgs A;
    A.d = d;
    A.sel = sel;
    if (A.sel.ids) A.sel.ids += off;
    else A.sel.begin += off;
    A.layer = layer;
    A.n_seqs = cnt;
    A.n_obs = n_obs;
    CUtensorMap tq;
    const uint8_t* qb = static_cast<const uint8_t*>(q_obs) + (size_t)off * n_obs * d.Hq * kD * 2;
    cudaError_t e = make_q_map(&tq, qb, d.Hq, n_obs, cnt);
    if (e == cudaSuccess) e = fp8 ? launch_ps<true>(tq, none, A, grid, st) : launch_ps<false>(tq, *k_map, A, grid, st);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace kvs
