// kvs_append_kv: quantise (E4M3) or copy the new tokens' K and V into their slots.
//
// Flash-MoE "Context Optimization", FP8 KV Cache > How It Works: one scale per
// position (all KV heads of K, and separately of V) = absmax / 240, values divided by
// the scale and rounded to E4M3, the scale stored beside the codes.  The divisions
// are IEEE round-to-nearest (__fdiv_rn) and the code is the hardware's
// round-to-nearest-even, saturating conversion.  Sliding Window Attention > Design:
// window mode writes position p to slot p % window.  "LLM mechanics III", section 5:
// the absolute position is recorded per slot and next_position only ever advances.
#include "append_store.cuh"

namespace kvs {

namespace {

constexpr int kWarps = 8;

// grid (ceil(n_new / (kWarps/2)), n_seqs): two warps per new token, one for K, one for V.
template <int KV, int IN>
__global__ void __launch_bounds__(kWarps * 32) append_kernel(Dev d, int layer, SeqSel sel, int n_new,
                                                               const void* k_in, const void* v_in) {
  const int s_local = blockIdx.y;
  const int s = sel.at(s_local);
  if (!KVS_DCHECK(d, s >= 0 && s < d.max_seqs)) return;
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
__global__ void alloc_pages_kernel(Dev d, int layer, SeqSel sel, int n_seqs, int n_new) {
  const int sl = blockIdx.x * blockDim.x + threadIdx.x;
  if (sl >= n_seqs) return;
  const int s = sel.at(sl);
  if (!KVS_DCHECK(d, s >= 0 && s < d.max_seqs)) return;
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

cudaError_t launch_alloc_pages(const Dev& d, int layer, SeqSel sel, int n_seqs, int n_new,
                               cudaStream_t st) {
  alloc_pages_kernel<<<(n_seqs + 127) / 128, 128, 0, st>>>(d, layer, sel, n_seqs, n_new);
  return cudaGetLastError();
}

cudaError_t launch_append(const Dev& d, int layer, SeqSel sel, int n_seqs, int n_new,
                          const void* k, const void* v, cudaStream_t st) {
  dim3 grid((n_new + kWarps / 2 - 1) / (kWarps / 2), n_seqs);
  const int KV = d.kv_dtype, IN = d.in_dtype;
  if (KV == KVS_E4M3 && IN == KVS_BF16) append_kernel<KVS_E4M3, KVS_BF16><<<grid, kWarps * 32, 0, st>>>(d, layer, sel, n_new, k, v);
  else if (KV == KVS_E4M3 && IN == KVS_F32) append_kernel<KVS_E4M3, KVS_F32><<<grid, kWarps * 32, 0, st>>>(d, layer, sel, n_new, k, v);
  else if (KV == KVS_BF16) append_kernel<KVS_BF16, KVS_BF16><<<grid, kWarps * 32, 0, st>>>(d, layer, sel, n_new, k, v);
  else if (KV == KVS_F32 && IN == KVS_BF16) append_kernel<KVS_F32, KVS_BF16><<<grid, kWarps * 32, 0, st>>>(d, layer, sel, n_new, k, v);
  else append_kernel<KVS_F32, KVS_F32><<<grid, kWarps * 32, 0, st>>>(d, layer, sel, n_new, k, v);
  return cudaGetLastError();
}

}  // namespace kvs
