// KV append and rollback over the paged cache.
//
// The block manager of "LLM serving: speculative decoding and PagedAttention
// memory management" (PagedAttention section): a per-sequence block table maps
// logical blocks to physical ones, and a physical block is taken only when the
// current one is full. Rollback follows "Speculative decoding principles and a
// vLLM production setup", sec. 3.1: rejected positions are given back a whole
// block at a time, accepted entries stay where they are.
//
// Allocation and release order is deterministic. The free list is a stack
// (entry top-1 is popped first). Append pops in (sequence, logical block)
// order, so sequence b's j-th new block is free_list[top - 1 - (off_b + j)]
// with off_b an exclusive prefix sum of the per-sequence needs. Rollback pushes
// in sequence order, highest logical block first, at free_list[top + off_b + j].
//
// The bookkeeping runs in one CTA (a block-wide scan over the batch); the row
// scatter and the tree-path compaction run one CTA per row / per sequence.
#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr int kBookThreads = 1024;

// Block-wide exclusive scan of one int per thread; returns the thread's
// exclusive prefix and writes the block total to *total (all threads).
__device__ int block_excl_scan(int v, int *total) {
  __shared__ int warp_sums[32];
  __shared__ int s_total;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    const int nw = blockDim.x >> 5;
    int w = lane < nw ? warp_sums[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int y = __shfl_up_sync(0xffffffffu, w, o);
      if (lane >= o) w += y;
    }
    if (lane < nw) warp_sums[lane] = w;  // inclusive
    if (lane == nw - 1) s_total = w;
  }
  __syncthreads();
  int excl = x - v + (warp > 0 ? warp_sums[warp - 1] : 0);
  *total = s_total;
  __syncthreads();
  return excl;
}

__device__ __forceinline__ int blocks_for(int tokens, int bs) { return (tokens + bs - 1) / bs; }

// -------------------------------------------------------------------------
// append, step 1: block allocation (one CTA)
// -------------------------------------------------------------------------
// The kernel is a chain of dependent memory round trips, so it issues every
// load that does not depend on an earlier one at once: the status word, the
// free-list top and the first batch of sequence lengths. The ids about to be
// popped are read once into shared memory, checked, then popped from there.
constexpr int kIdCache = 4096;

__global__ void __launch_bounds__(kBookThreads) kv_alloc_kernel(KV kv, const int32_t *cu_q, int32_t *status) {
  grid_dependency_wait();  // the earlier kernel on the stream is complete and visible
  grid_dependents_launch();
  __shared__ int s_ids[kIdCache];
  const int B = kv.batch, bs = kv.block_size;
  const bool failed = status_set(status);
  const int top = *kv.free_top;
  int c0 = 0, n0 = 0;  // the thread's sequence of the first batch
  if ((int)threadIdx.x < B) {
    c0 = kv.seq_lens[threadIdx.x];
    n0 = cu_q[threadIdx.x + 1] - cu_q[threadIdx.x];
  }
  if (failed) return;  // every thread read the same word: the whole CTA leaves

  // pass 1: validate lengths, count blocks (the first batch's offsets are kept)
  int bad_len = 0;
  int total = 0, off0 = 0, need0 = 0, tot0 = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int need = 0;
    if (b < B) {
      const int c = base == 0 ? c0 : kv.seq_lens[b];
      const int n = base == 0 ? n0 : cu_q[b + 1] - cu_q[b];
      if (c < 0 || n < 0 || blocks_for(c + n, bs) > kv.max_blocks) bad_len = 1;
      else need = blocks_for(c + n, bs) - blocks_for(c, bs);
    }
    int chunk_total;
    const int off = block_excl_scan(need, &chunk_total);
    if (base == 0) {
      off0 = off;
      need0 = need;
      tot0 = chunk_total;
    }
    total += chunk_total;
  }
  if (__syncthreads_or(bad_len)) {
    if (threadIdx.x == 0) record(status, SV_ERR_BAD_LENGTH);
    return;
  }
  if (total > top || top > kv.num_blocks) {
    if (threadIdx.x == 0) record(status, SV_ERR_OUT_OF_BLOCKS);
    return;
  }
  // pass 2: every id about to be popped must be a valid block
  int bad_id = 0;
  for (int k = threadIdx.x; k < total; k += blockDim.x) {
    const int id = kv.free_list[top - 1 - k];
    if (k < kIdCache) s_ids[k] = id;
    if (id < 0 || id >= kv.num_blocks) bad_id = 1;
  }
  if (__syncthreads_or(bad_id)) {
    if (threadIdx.x == 0) record(status, SV_ERR_BAD_BLOCK_ID);
    return;
  }
  // pass 3: pop into the block tables
  auto popped = [&](int k) { return k < kIdCache ? s_ids[k] : kv.free_list[top - 1 - k]; };
  if ((int)threadIdx.x < B)
    for (int j = 0; j < need0; ++j)
      kv.block_table[(size_t)threadIdx.x * kv.max_blocks + blocks_for(c0, bs) + j] = popped(off0 + j);
  int carry = tot0;  // batches past the first (more sequences than threads)
  for (int base = blockDim.x; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int need = 0, first = 0;
    if (b < B) {
      const int c = kv.seq_lens[b], n = cu_q[b + 1] - cu_q[b];
      first = blocks_for(c, bs);
      need = blocks_for(c + n, bs) - first;
    }
    int chunk_total;
    const int off = carry + block_excl_scan(need, &chunk_total);
    for (int j = 0; j < need; ++j) kv.block_table[(size_t)b * kv.max_blocks + first + j] = popped(off + j);
    carry += chunk_total;
  }
  __syncthreads();
  for (int k = threadIdx.x; k < total; k += blockDim.x) kv.free_list[top - 1 - k] = -1;
  if (threadIdx.x == 0) *kv.free_top = top - total;
}

// -------------------------------------------------------------------------
// append, step 2: scatter the new rows (one CTA per query row)
// -------------------------------------------------------------------------
// The row's source vectors do not depend on where they go: they are loaded
// first, while cu_q is staged in shared memory for the search of the row's
// sequence; then the sequence length and the block id, then the stores.
constexpr int kScatterThreads = 128;
constexpr int kCuCache = 2048;

__global__ void __launch_bounds__(kScatterThreads) kv_scatter_kernel(KV kv, const uint8_t *new_k,
                                                                     const uint8_t *new_v, const int32_t *cu_q,
                                                                     int32_t *status) {
  grid_dependency_wait();  // the earlier kernel on the stream is complete and visible
  grid_dependents_launch();
  __shared__ int s_cu[kCuCache];
  const int row = blockIdx.x;
  const int B = kv.batch;
  const bool failed = status_set(status);
  const int row_bytes = kv.head_dim * kv.elem_bytes;  // a multiple of 16
  const int vec_per_row = row_bytes / 16;
  const int total = kv.num_kv_heads * vec_per_row;
  const size_t src_row = (size_t)row * kv.num_kv_heads * row_bytes;
  uint4 kk0 = make_uint4(0, 0, 0, 0), vv0 = kk0;  // the thread's first vector
  if ((int)threadIdx.x < total) {
    kk0 = *reinterpret_cast<const uint4 *>(new_k + src_row + (size_t)threadIdx.x * 16);
    vv0 = *reinterpret_cast<const uint4 *>(new_v + src_row + (size_t)threadIdx.x * 16);
  }
  const bool staged = B + 1 <= kCuCache;
  if (staged)
    for (int k = threadIdx.x; k <= B; k += blockDim.x) s_cu[k] = cu_q[k];
  __syncthreads();
  if (failed) return;
  auto cu = [&](int k) { return staged ? s_cu[k] : cu_q[k]; };
  int lo = 0, hi = B;  // the last b with cu_q[b] <= row owns the row
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (cu(mid) <= row) lo = mid;
    else hi = mid;
  }
  const int b = lo, row0 = cu(b), i = row - row0;
  if (i >= cu(b + 1) - row0) return;  // rows past cu_q[batch]: nothing to write
  const int pos = kv.seq_lens[b] + i;
  const int blk = kv.block_table[(size_t)b * kv.max_blocks + pos / kv.block_size];
  if (blk < 0 || blk >= kv.num_blocks) {
    if (threadIdx.x == 0) record(status, SV_ERR_BAD_BLOCK_ID);
    return;
  }
  const int slot = pos % kv.block_size;
  for (int x = threadIdx.x; x < total; x += blockDim.x) {
    const int h = x / vec_per_row, v = x % vec_per_row;
    uint4 kk = kk0, vv = vv0;
    if (x >= (int)blockDim.x) {
      kk = *reinterpret_cast<const uint4 *>(new_k + src_row + (size_t)x * 16);
      vv = *reinterpret_cast<const uint4 *>(new_v + src_row + (size_t)x * 16);
    }
    const size_t dst = (((size_t)blk * kv.num_kv_heads + h) * kv.block_size + slot) * row_bytes + (size_t)v * 16;
    *reinterpret_cast<uint4 *>((uint8_t *)kv.k_pool + dst) = kk;
    *reinterpret_cast<uint4 *>((uint8_t *)kv.v_pool + dst) = vv;
  }
}

// -------------------------------------------------------------------------
// rollback, tree drafts: move the accepted path's rows to c+1 .. c+a
// (one CTA per sequence, rows copied in path order)
// -------------------------------------------------------------------------
__global__ void kv_tree_compact_kernel(KV kv, const int32_t *cu_q, const int32_t *accept, const int32_t *path,
                                       int max_q, int32_t *status) {
  grid_dependency_wait();  // the earlier kernel on the stream is complete and visible
  grid_dependents_launch();
  if (status_set(status)) return;
  const int b = blockIdx.x;
  const int n = cu_q[b + 1] - cu_q[b];
  const int a = accept[b];
  if (a < 0 || a > n - 1) {
    if (threadIdx.x == 0) record(status, SV_ERR_BAD_LENGTH);
    return;
  }
  for (int j = 0; j < a; ++j) {
    const int p = path[(size_t)b * max_q + j];
    if (p < 1 || p >= n) {
      if (threadIdx.x == 0) record(status, SV_ERR_BAD_LENGTH);
      return;
    }
  }
  const int c = kv.seq_lens[b];
  if (c < 0 || blocks_for(c + n, kv.block_size) > kv.max_blocks) {
    if (threadIdx.x == 0) record(status, SV_ERR_BAD_LENGTH);
    return;
  }
  const int row_bytes = kv.head_dim * kv.elem_bytes;
  const int vec_per_row = row_bytes / 16;
  const int total = kv.num_kv_heads * vec_per_row;
  for (int j = 1; j <= a; ++j) {
    const int src_pos = c + path[(size_t)b * max_q + j - 1], dst_pos = c + j;
    if (src_pos != dst_pos) {
      const int sblk = kv.block_table[(size_t)b * kv.max_blocks + src_pos / kv.block_size];
      const int dblk = kv.block_table[(size_t)b * kv.max_blocks + dst_pos / kv.block_size];
      if (sblk < 0 || sblk >= kv.num_blocks || dblk < 0 || dblk >= kv.num_blocks) {
        if (threadIdx.x == 0) record(status, SV_ERR_BAD_BLOCK_ID);
        return;
      }
      const int ss = src_pos % kv.block_size, ds = dst_pos % kv.block_size;
      for (int x = threadIdx.x; x < total; x += blockDim.x) {
        const int h = x / vec_per_row, v = x % vec_per_row;
        const size_t so = (((size_t)sblk * kv.num_kv_heads + h) * kv.block_size + ss) * row_bytes + (size_t)v * 16;
        const size_t d_o = (((size_t)dblk * kv.num_kv_heads + h) * kv.block_size + ds) * row_bytes + (size_t)v * 16;
        const uint4 kk = *reinterpret_cast<const uint4 *>((const uint8_t *)kv.k_pool + so);
        const uint4 vv = *reinterpret_cast<const uint4 *>((const uint8_t *)kv.v_pool + so);
        *reinterpret_cast<uint4 *>((uint8_t *)kv.k_pool + d_o) = kk;
        *reinterpret_cast<uint4 *>((uint8_t *)kv.v_pool + d_o) = vv;
      }
    }
    __syncthreads();  // the next copy may read this one's destination
  }
}

// -------------------------------------------------------------------------
// rollback: truncate and give blocks back (one CTA)
// -------------------------------------------------------------------------
__global__ void __launch_bounds__(kBookThreads) kv_truncate_kernel(KV kv, const int32_t *cu_q,
                                                                   const int32_t *accept, int32_t *status) {
  grid_dependency_wait();  // the earlier kernel on the stream is complete and visible
  grid_dependents_launch();
  const int B = kv.batch, bs = kv.block_size;
  // every load that depends on no other at once (see kv_alloc_kernel)
  const bool failed = status_set(status);
  const int top = *kv.free_top;
  int c0 = 0, n0 = 0, a0 = 0;
  if ((int)threadIdx.x < B) {
    c0 = kv.seq_lens[threadIdx.x];
    n0 = cu_q[threadIdx.x + 1] - cu_q[threadIdx.x];
    a0 = accept[threadIdx.x];
  }
  if (failed) return;  // every thread read the same word: the whole CTA leaves
  int bad_len = 0, bad_id = 0;
  int total = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int freed = 0;
    if (b < B) {
      const int c = base == 0 ? c0 : kv.seq_lens[b];
      const int n = base == 0 ? n0 : cu_q[b + 1] - cu_q[b];
      const int a = base == 0 ? a0 : accept[b];
      if (c < 0 || n < 1 || a < 0 || a > n - 1 || blocks_for(c + n, bs) > kv.max_blocks) {
        bad_len = 1;
      } else {
        const int old_blocks = blocks_for(c + n, bs), keep = blocks_for(c + a + 1, bs);
        freed = old_blocks - keep;
        for (int lb = keep; lb < old_blocks; ++lb) {
          const int id = kv.block_table[(size_t)b * kv.max_blocks + lb];
          if (id < 0 || id >= kv.num_blocks) bad_id = 1;
        }
      }
    }
    int chunk_total;
    block_excl_scan(freed, &chunk_total);
    total += chunk_total;
  }
  if (__syncthreads_or(bad_len)) {
    if (threadIdx.x == 0) record(status, SV_ERR_BAD_LENGTH);
    return;
  }
  if (__syncthreads_or(bad_id)) {
    if (threadIdx.x == 0) record(status, SV_ERR_BAD_BLOCK_ID);
    return;
  }
  if (top < 0 || top + total > kv.num_blocks) {
    if (threadIdx.x == 0) record(status, SV_ERR_OUT_OF_BLOCKS);
    return;
  }
  int carry = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int freed = 0, old_blocks = 0, c = 0, a = 0;
    if (b < B) {
      c = base == 0 ? c0 : kv.seq_lens[b];
      const int n = base == 0 ? n0 : cu_q[b + 1] - cu_q[b];
      a = base == 0 ? a0 : accept[b];
      old_blocks = blocks_for(c + n, bs);
      freed = old_blocks - blocks_for(c + a + 1, bs);
    }
    int chunk_total;
    const int off = carry + block_excl_scan(freed, &chunk_total);
    for (int j = 0; j < freed; ++j) {
      int32_t *e = &kv.block_table[(size_t)b * kv.max_blocks + old_blocks - 1 - j];
      kv.free_list[top + off + j] = *e;
      *e = -1;
    }
    if (b < B) kv.seq_lens[b] = c + a + 1;
    carry += chunk_total;
  }
  __syncthreads();
  if (threadIdx.x == 0) *kv.free_top = top + total;
}

}  // namespace

cudaError_t launch_kv_append(const KV &kv, const void *new_k, const void *new_v, const int32_t *cu_q,
                             int total_q, int32_t *status, cudaStream_t st) {
  cudaError_t e = launch_pdl(kv_alloc_kernel, dim3(1), dim3(kBookThreads), 0, st, kv, cu_q, status);
  if (e != cudaSuccess || total_q == 0) return e;
  return launch_pdl(kv_scatter_kernel, dim3((unsigned)total_q), dim3(kScatterThreads), 0, st, kv, (const uint8_t *)new_k,
                    (const uint8_t *)new_v, cu_q, status);
}

cudaError_t launch_kv_rollback(const KV &kv, const int32_t *cu_q, const int32_t *accept, const int32_t *path,
                               int max_q, int32_t *status, cudaStream_t st) {
  if (path != nullptr) {
    cudaError_t e = launch_pdl(kv_tree_compact_kernel, dim3(kv.batch), dim3(256), 0, st, kv, cu_q, accept, path,
                               max_q, status);
    if (e != cudaSuccess) return e;
  }
  return launch_pdl(kv_truncate_kernel, dim3(1), dim3(kBookThreads), 0, st, kv, cu_q, accept, status);
}

}  // namespace sv
