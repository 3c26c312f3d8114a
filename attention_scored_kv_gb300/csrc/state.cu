// Workspace initialisation, sequence reset, error clearing and EMA read-back.
#include "kvs_internal.cuh"

namespace kvs {

namespace {

__global__ void fill_i64(int64_t* p, size_t n, int64_t v) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    p[i] = v;
}

__global__ void fill_i32(int32_t* p, size_t n, int32_t v) {
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    p[i] = v;
}

__global__ void init_free_stack(Dev d) {
  // pops return pages 0, 1, 2, ... in order
  for (int32_t i = blockIdx.x * blockDim.x + threadIdx.x; i < d.num_pages; i += gridDim.x * blockDim.x)
    d.free_pages[i] = d.num_pages - 1 - i;
  if (blockIdx.x == 0 && threadIdx.x == 0) *d.free_top = d.num_pages;
}

// One CTA per sequence: empty it in every layer.
__global__ void reset_kernel(Dev d, SeqSel sel) {
  const int s = sel.at(blockIdx.x);
  if (!KVS_DCHECK(d, s >= 0 && s < d.max_seqs)) return;
  const size_t pos_base = (size_t)s * d.max_positions;
  const size_t blk_base = (size_t)s * d.max_blocks;
  for (int64_t p = threadIdx.x; p < d.max_positions; p += blockDim.x) {
    d.c_tok[pos_base + p] = 0.0;
    d.e_tok[pos_base + p] = 0.0;
    d.last_tok[pos_base + p] = -1;
  }
  for (int k = threadIdx.x; k < d.max_blocks; k += blockDim.x) {
    d.c_blk[blk_base + k] = 0.0;
    d.e_blk[blk_base + k] = 0.0;
    d.s_blk[blk_base + k] = 0.0;
    d.t_blk[blk_base + k] = 0.0;
    d.last_blk[blk_base + k] = -1;
  }
  for (size_t i = threadIdx.x; i < (size_t)d.max_blocks * d.traj_len; i += blockDim.x)
    d.traj[blk_base * d.traj_len + i] = 0.f;
  for (size_t i = threadIdx.x; i < (size_t)d.max_blocks * d.n_prof; i += blockDim.x)
    d.prof[blk_base * d.n_prof + i] = 0.0;
  for (size_t i = threadIdx.x; i < (size_t)d.max_blocks * d.n_hprof; i += blockDim.x)
    d.hprof[blk_base * d.n_hprof + i] = 0.0;
  if (d.mode == KVS_MODE_H2O) {
    // return every page of the sequence to the pool and clear its slots
    const int n = d.res_count[s];
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const int32_t page = d.res_pages[blk_base + i];
      const int32_t k = d.res_blocks[blk_base + i];
      d.block_table[blk_base + k] = -1;
      const int32_t top = atomicAdd(d.free_top, 1);
      d.free_pages[top] = page;
      for (int l = 0; l < d.L; ++l)
        for (int j = 0; j < kBlock; ++j) d.pos[(size_t)l * d.slot_layer_elems + (size_t)page * kBlock + j] = -1;
    }
  } else {
    for (int l = 0; l < d.L; ++l)
      for (int64_t i = threadIdx.x; i < (int64_t)d.pages_per_seq * kBlock; i += blockDim.x)
        d.pos[(size_t)l * d.slot_layer_elems + (size_t)s * d.pages_per_seq * kBlock + i] = -1;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    if (d.mode == KVS_MODE_H2O) d.res_count[s] = 0;
    for (int l = 0; l < d.L; ++l) {
      d.next_pos[(size_t)l * d.max_seqs + s] = 0;
      d.append_tickets[(size_t)l * d.max_seqs + s] = 0;
    }
    d.steps[s] = 0;
    d.acc_tickets[s] = 0;
  }
}

__global__ void clear_kernel(Dev d) {
  for (int i = threadIdx.x; i < kCounterInts * d.max_seqs; i += blockDim.x) d.counters[i] = 0;
  for (int i = threadIdx.x; i < d.max_seqs; i += blockDim.x) d.acc_tickets[i] = 0;
  for (int i = threadIdx.x; i < d.L * d.max_seqs; i += blockDim.x) d.append_tickets[i] = 0;
  if (threadIdx.x == 0) *d.err = 0;
}

// EMA as of the last accumulate step: stored value decayed by d^(steps-1-last).
__global__ void read_ema_kernel(const double* e, const int32_t* last, const int32_t* steps,
                                int per_seq, int max_seqs, double decay, double* dst) {
  const size_t n = (size_t)per_seq * max_seqs;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int s = (int)(i / per_seq);
    const int32_t l = last[i];
    dst[i] = (l < 0) ? 0.0 : e[i] * pow(decay, (double)(steps[s] - 1 - l));
  }
}

// Trajectory ring, oldest step first: column j of block k is step tau = steps - T + j,
// kept where the block was updated at tau.  A block is updated at every step of one
// stretch of residency (it never returns once it leaves), so its slot tau % T holds
// step tau exactly when 0 <= tau <= last; otherwise the column is 0.
__global__ void read_trajectory_kernel(Dev d, float* dst) {
  const int T = d.traj_len;
  const size_t n = (size_t)d.max_seqs * d.max_blocks * T;
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const size_t kb = i / T;                 // s * max_blocks + k
    const int j = (int)(i % T);
    const int s = (int)(kb / d.max_blocks);
    const int32_t tau = d.steps[s] - T + j, last = d.last_blk[kb];
    dst[i] = (tau >= 0 && tau <= last) ? d.traj[kb * T + tau % T] : 0.f;
  }
}

int grid_for(size_t n) {
  size_t g = (n + 255) / 256;
  if (g > 4096) g = 4096;
  if (g < 1) g = 1;
  return (int)g;
}

}  // namespace

cudaError_t launch_init(const Dev& d, cudaStream_t st) {
  const size_t slots = (size_t)d.L * d.slot_layer_elems;
  fill_i64<<<grid_for(slots), 256, 0, st>>>(d.pos, slots, -1);
  const size_t bt = (size_t)d.max_seqs * d.max_blocks;
  fill_i32<<<grid_for(bt), 256, 0, st>>>(d.block_table, bt, -1);
  fill_i32<<<grid_for(bt), 256, 0, st>>>(d.last_blk, bt, -1);
  const size_t tk = (size_t)d.max_seqs * d.max_positions;
  fill_i32<<<grid_for(tk), 256, 0, st>>>(d.last_tok, tk, -1);
  init_free_stack<<<grid_for(d.num_pages), 256, 0, st>>>(d);
  return cudaGetLastError();
}

cudaError_t launch_reset(const Dev& d, SeqSel sel, int n_seqs, cudaStream_t st) {
  reset_kernel<<<n_seqs, 256, 0, st>>>(d, sel);
  return cudaGetLastError();
}

cudaError_t launch_read_trajectory(const Dev& d, float* dst, cudaStream_t st) {
  const size_t n = (size_t)d.max_seqs * d.max_blocks * d.traj_len;
  read_trajectory_kernel<<<grid_for(n), 256, 0, st>>>(d, dst);
  return cudaGetLastError();
}

cudaError_t launch_clear(const Dev& d, cudaStream_t st) {
  clear_kernel<<<1, 256, 0, st>>>(d);
  return cudaGetLastError();
}

cudaError_t launch_read_ema(const Dev& d, int what, double* dst, cudaStream_t st) {
  if (what == KVS_STATE_E_TOKEN) {
    const size_t n = (size_t)d.max_seqs * d.max_positions;
    read_ema_kernel<<<grid_for(n), 256, 0, st>>>(d.e_tok, d.last_tok, d.steps, d.max_positions,
                                                 d.max_seqs, d.ema_decay, dst);
  } else if (what == KVS_STATE_T_BLOCK) {
    // the latest step's score: the stored value where the block was updated in the last
    // step, else 0 (decay 0: 0^0 = 1, 0^gap = 0)
    const size_t n = (size_t)d.max_seqs * d.max_blocks;
    read_ema_kernel<<<grid_for(n), 256, 0, st>>>(d.t_blk, d.last_blk, d.steps, d.max_blocks, d.max_seqs, 0.0, dst);
  } else {
    const size_t n = (size_t)d.max_seqs * d.max_blocks;
    read_ema_kernel<<<grid_for(n), 256, 0, st>>>(d.e_blk, d.last_blk, d.steps, d.max_blocks,
                                                 d.max_seqs, d.ema_decay, dst);
  }
  return cudaGetLastError();
}

}  // namespace kvs
