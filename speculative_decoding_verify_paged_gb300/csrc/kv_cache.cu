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
#include <cuda_fp8.h>

#include "sv_internal.cuh"

namespace sv {
namespace {

// 16 bf16 values (two 16-byte vectors) -> 16 E4M3 codes of x / scale (fp32
// division; nearest, ties to even; saturating), element j in byte j.
__device__ __forceinline__ uint4 quantize16(const uint4 &a, const uint4 &b, float scale) {
  const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
  uint32_t out[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint32_t word = 0;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t v = w[2 * q + h];
      const float x0 = __fdiv_rn(__uint_as_float(v << 16), scale);
      const float x1 = __fdiv_rn(__uint_as_float(v & 0xffff0000u), scale);
      const __nv_fp8x2_storage_t c = __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3);
      word |= (uint32_t)c << (16 * h);
    }
    out[q] = word;
  }
  return make_uint4(out[0], out[1], out[2], out[3]);
}

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
//
// With reference counts, a sequence whose first new row lands in a partly
// filled shared block takes a private copy when the block is still shared at
// its turn: writer k (in sequence order) of a block held by r sequences copies
// iff k < r - 1. Its copy is popped just before its new blocks; the new block's
// count is set to -(old id + 1), which tells the scatter kernel to copy the
// old block's rows, and the scatter kernel then sets it to 1.
constexpr int kIdCache = 2048;
constexpr int kCowMaxBatch = 4096;  // sequences the sharing path handles (one per shared-memory slot)

__global__ void __launch_bounds__(kBookThreads) kv_alloc_kernel(KV kv, const int32_t *cu_q, int32_t *status) {
  grid_dependency_wait();  // the earlier kernel on the stream is complete and visible
  grid_dependents_launch();
  __shared__ int s_ids[kIdCache];
  __shared__ int s_cand[kCowMaxBatch];  // sharing: the shared partial block a sequence writes into, else -1
  __shared__ int s_copy[kCowMaxBatch];  // sharing: the block a sequence copies, else -1
  const int B = kv.batch, bs = kv.block_size;
  const bool sharing = kv.ref_count != nullptr;
  const bool failed = status_set(status);
  const int top = *kv.free_top;
  int c0 = 0, n0 = 0;  // the thread's sequence of the first batch
  if ((int)threadIdx.x < B) {
    c0 = kv.seq_lens[threadIdx.x];
    n0 = cu_q[threadIdx.x + 1] - cu_q[threadIdx.x];
  }
  if (failed) return;  // every thread read the same word: the whole CTA leaves
  auto len_of = [&](int base, int b, int &c, int &n) {
    c = base == 0 ? c0 : kv.seq_lens[b];
    n = base == 0 ? n0 : cu_q[b + 1] - cu_q[b];
  };

  // pass 1: validate lengths; with sharing, find the writers into shared partial blocks
  int bad_len = 0, bad_id = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    if (b >= B) continue;
    int c, n;
    len_of(base, b, c, n);
    if (c < 0 || n < 0 || blocks_for(c + n, bs) > kv.max_blocks) {
      bad_len = 1;
      continue;
    }
    if (sharing) {
      int cand = -1;
      if (n > 0 && c % bs != 0) {
        const int x = kv.block_table[(size_t)b * kv.max_blocks + c / bs];
        if (x < 0 || x >= kv.num_blocks) bad_id = 1;
        else if (kv.ref_count[x] < 1) bad_id = 1;
        else if (kv.ref_count[x] > 1) cand = x;
      }
      s_cand[b] = cand;
    }
  }
  if (__syncthreads_or(bad_len)) {
    if (threadIdx.x == 0) record(status, SV_ERR_BAD_LENGTH);
    return;
  }
  if (__syncthreads_or(bad_id)) {
    if (threadIdx.x == 0) record(status, SV_ERR_BAD_BLOCK_ID);
    return;
  }
  if (sharing) {  // writer k of a block held by r copies iff k < r - 1
    for (int b = threadIdx.x; b < B; b += blockDim.x) {
      const int x = s_cand[b];
      int copy = -1;
      if (x >= 0) {
        int k = 0;
        for (int e = 0; e < b; ++e) k += s_cand[e] == x;
        if (k < kv.ref_count[x] - 1) copy = x;
      }
      s_copy[b] = copy;
    }
    __syncthreads();
  }
  // blocks each sequence pops: its copy (if any), then its new blocks
  auto pops_of = [&](int base, int b, int &first, int &need, int &copy) {
    int c, n;
    len_of(base, b, c, n);
    first = blocks_for(c, bs);
    need = blocks_for(c + n, bs) - first;
    copy = sharing ? s_copy[b] : -1;
  };

  // pass 2: count the pops (the first batch's offsets are kept)
  int total = 0, off0 = 0, tot0 = 0;
  for (int base = 0; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int k = 0;
    if (b < B) {
      int first, need, copy;
      pops_of(base, b, first, need, copy);
      k = need + (copy >= 0);
    }
    int chunk_total;
    const int off = block_excl_scan(k, &chunk_total);
    if (base == 0) {
      off0 = off;
      tot0 = chunk_total;
    }
    total += chunk_total;
  }
  if (total > top || top > kv.num_blocks) {
    if (threadIdx.x == 0) record(status, SV_ERR_OUT_OF_BLOCKS);
    return;
  }
  // pass 3: every id about to be popped must be a valid block
  for (int k = threadIdx.x; k < total; k += blockDim.x) {
    const int id = kv.free_list[top - 1 - k];
    if (k < kIdCache) s_ids[k] = id;
    if (id < 0 || id >= kv.num_blocks) bad_id = 1;
  }
  if (__syncthreads_or(bad_id)) {
    if (threadIdx.x == 0) record(status, SV_ERR_BAD_BLOCK_ID);
    return;
  }
  // pass 4: pop into the block tables
  auto popped = [&](int k) { return k < kIdCache ? s_ids[k] : kv.free_list[top - 1 - k]; };
  auto pop_seq = [&](int base, int b, int off) {
    int first, need, copy;
    pops_of(base, b, first, need, copy);
    int32_t *row = kv.block_table + (size_t)b * kv.max_blocks;
    if (copy >= 0) {
      const int id = popped(off++);
      row[first - 1] = id;
      kv.ref_count[id] = -(copy + 1);  // the scatter kernel copies the rows, then sets 1
      atomicSub(&kv.ref_count[copy], 1);
    }
    for (int j = 0; j < need; ++j) {
      const int id = popped(off + j);
      row[first + j] = id;
      if (sharing) kv.ref_count[id] = 1;
    }
  };
  if ((int)threadIdx.x < B) pop_seq(0, threadIdx.x, off0);
  int carry = tot0;  // batches past the first (more sequences than threads)
  for (int base = blockDim.x; base < B; base += blockDim.x) {
    const int b = base + threadIdx.x;
    int k = 0;
    if (b < B) {
      int first, need, copy;
      pops_of(base, b, first, need, copy);
      k = need + (copy >= 0);
    }
    int chunk_total;
    const int off = carry + block_excl_scan(k, &chunk_total);
    if (b < B) pop_seq(base, b, off);
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
  __shared__ int s_cu[kCuCache];
  const int row = blockIdx.x;
  const int B = kv.batch;
  const int row_bytes = kv.head_dim * kv.elem_bytes;  // a multiple of 16
  const int vec_per_row = row_bytes / 16;
  const int total = kv.num_kv_heads * vec_per_row;
  // an fp8 pool's 16-byte vector (16 codes) comes from 32 bytes of bf16 input
  const int src_vec = kv.fp8 ? 32 : 16;
  const size_t src_row = (size_t)row * total * src_vec;
  uint4 kk0 = make_uint4(0, 0, 0, 0), vv0 = kk0, kk1 = kk0, vv1 = kk0;  // the thread's first vector
  if ((int)threadIdx.x < total) {
    kk0 = *reinterpret_cast<const uint4 *>(new_k + src_row + (size_t)threadIdx.x * src_vec);
    vv0 = *reinterpret_cast<const uint4 *>(new_v + src_row + (size_t)threadIdx.x * src_vec);
    if (kv.fp8) {
      kk1 = *reinterpret_cast<const uint4 *>(new_k + src_row + (size_t)threadIdx.x * src_vec + 16);
      vv1 = *reinterpret_cast<const uint4 *>(new_v + src_row + (size_t)threadIdx.x * src_vec + 16);
    }
  }
  const bool staged = B + 1 <= kCuCache;
  if (staged)
    for (int k = threadIdx.x; k <= B; k += blockDim.x) s_cu[k] = cu_q[k];
  __syncthreads();
  // the row's vectors and cu_q are the call's own inputs, read above before the wait; the status,
  // the lengths, the block table and the pool come after it
  grid_dependency_wait();  // the earlier kernel on the stream is complete and visible
  grid_dependents_launch();
  if (status_set(status)) return;
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
  if (i == 0 && slot > 0 && kv.ref_count != nullptr) {
    // the sequence's first row lands in its private copy of a shared block (see
    // kv_alloc_kernel): bring over the rows written before, every head, K and V
    const int m = kv.ref_count[blk];
    if (m < 0) {
      const int src = -m - 1;
      const int per_head = slot * vec_per_row;  // the rows before `slot` are contiguous in a (block, head)
      const size_t head_bytes = (size_t)kv.block_size * row_bytes;
      if (src >= 0 && src < kv.num_blocks) {
        for (int x = threadIdx.x; x < kv.num_kv_heads * per_head; x += blockDim.x) {
          const int h = x / per_head, v = x - h * per_head;
          const size_t so = ((size_t)src * kv.num_kv_heads + h) * head_bytes + (size_t)v * 16;
          const size_t d_o = ((size_t)blk * kv.num_kv_heads + h) * head_bytes + (size_t)v * 16;
          *reinterpret_cast<uint4 *>((uint8_t *)kv.k_pool + d_o) = *reinterpret_cast<const uint4 *>((const uint8_t *)kv.k_pool + so);
          *reinterpret_cast<uint4 *>((uint8_t *)kv.v_pool + d_o) = *reinterpret_cast<const uint4 *>((const uint8_t *)kv.v_pool + so);
        }
      } else if (threadIdx.x == 0) {
        record(status, SV_ERR_BAD_BLOCK_ID);
      }
      __syncthreads();  // every thread has read the marker
      if (threadIdx.x == 0) kv.ref_count[blk] = 1;
    }
  }
  for (int x = threadIdx.x; x < total; x += blockDim.x) {
    const int h = x / vec_per_row, v = x % vec_per_row;
    uint4 kk = kk0, vv = vv0, kb = kk1, vb = vv1;
    if (x >= (int)blockDim.x) {
      kk = *reinterpret_cast<const uint4 *>(new_k + src_row + (size_t)x * src_vec);
      vv = *reinterpret_cast<const uint4 *>(new_v + src_row + (size_t)x * src_vec);
      if (kv.fp8) {
        kb = *reinterpret_cast<const uint4 *>(new_k + src_row + (size_t)x * src_vec + 16);
        vb = *reinterpret_cast<const uint4 *>(new_v + src_row + (size_t)x * src_vec + 16);
      }
    }
    if (kv.fp8) {
      kk = quantize16(kk, kb, kv.k_scale);
      vv = quantize16(vv, vb, kv.v_scale);
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
        for (int lb = keep; lb < old_blocks; ++lb) {  // pushed: every block, or (sharing) the last reference
          const int id = kv.block_table[(size_t)b * kv.max_blocks + lb];
          if (id < 0 || id >= kv.num_blocks) bad_id = 1;
          else if (kv.ref_count == nullptr) ++freed;
          else if (kv.ref_count[id] < 1) bad_id = 1;
          else freed += kv.ref_count[id] == 1;
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
    int pushed = 0, old_blocks = 0, keep = 0, c = 0, a = 0;
    if (b < B) {
      c = base == 0 ? c0 : kv.seq_lens[b];
      const int n = base == 0 ? n0 : cu_q[b + 1] - cu_q[b];
      a = base == 0 ? a0 : accept[b];
      old_blocks = blocks_for(c + n, bs);
      keep = blocks_for(c + a + 1, bs);
      for (int lb = keep; lb < old_blocks; ++lb)
        pushed += kv.ref_count == nullptr || kv.ref_count[kv.block_table[(size_t)b * kv.max_blocks + lb]] == 1;
    }
    int chunk_total;
    int off = carry + block_excl_scan(pushed, &chunk_total);
    for (int lb = old_blocks - 1; lb >= keep; --lb) {  // highest logical block first
      int32_t *e = &kv.block_table[(size_t)b * kv.max_blocks + lb];
      const int id = *e;
      if (kv.ref_count == nullptr) {
        kv.free_list[top + off++] = id;
      } else if (kv.ref_count[id] == 1) {
        kv.ref_count[id] = 0;
        kv.free_list[top + off++] = id;
      } else {
        atomicSub(&kv.ref_count[id], 1);
      }
      *e = -1;
    }
    if (b < B) kv.seq_lens[b] = c + a + 1;
    carry += chunk_total;
  }
  __syncthreads();
  if (threadIdx.x == 0) *kv.free_top = top + total;
}

// -------------------------------------------------------------------------
// fork and release (one CTA each; bitmaps over the sequence ids)
// -------------------------------------------------------------------------
constexpr int kMaxSeqBits = 65536;  // sequences the fork and release kernels handle

// Marks bit `i`; true if it was already set.
__device__ __forceinline__ bool mark(unsigned *bits, int i) {
  const unsigned m = 1u << (i & 31);
  return (atomicOr(&bits[i >> 5], m) & m) != 0;
}
__device__ __forceinline__ bool marked(const unsigned *bits, int i) { return (bits[i >> 5] >> (i & 31)) & 1u; }

__global__ void __launch_bounds__(kBookThreads) kv_fork_kernel(KV kv, const int32_t *parents, const int32_t *children,
                                                               int n, int32_t *status) {
  grid_dependency_wait();  // the earlier kernel on the stream is complete and visible
  grid_dependents_launch();
  __shared__ unsigned s_child[kMaxSeqBits / 32], s_parent[kMaxSeqBits / 32];
  const int B = kv.batch, bs = kv.block_size;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  if (status_set(status)) return;
  for (int w = threadIdx.x; w < kMaxSeqBits / 32; w += blockDim.x) s_child[w] = s_parent[w] = 0u;
  __syncthreads();
  int bad_len = 0, bad_id = 0;
  for (int k = threadIdx.x; k < n; k += blockDim.x) {
    const int p = parents[k], c = children[k];
    if (p < 0 || p >= B || c < 0 || c >= B) {
      bad_len = 1;
      continue;
    }
    if (mark(s_child, c)) bad_len = 1;  // the same child twice
    mark(s_parent, p);
  }
  if (__syncthreads_or(bad_len)) {
    if (threadIdx.x == 0) record(status, SV_ERR_BAD_LENGTH);
    return;
  }
  // one warp per pair, lanes over the table entries
  for (int k = warp; k < n; k += nwarps) {
    const int p = parents[k], c = children[k];
    const int len = kv.seq_lens[p];
    if (marked(s_parent, c) || kv.seq_lens[c] != 0 || len < 0 || blocks_for(len, bs) > kv.max_blocks) {
      bad_len = 1;  // a child that is a parent, or not empty; a parent too long
      continue;
    }
    const int32_t *crow = kv.block_table + (size_t)c * kv.max_blocks;
    const int32_t *prow = kv.block_table + (size_t)p * kv.max_blocks;
    for (int lb = lane; lb < kv.max_blocks; lb += 32) bad_len |= crow[lb] != -1;
    for (int lb = lane; lb < blocks_for(len, bs); lb += 32) {
      const int id = prow[lb];
      if (id < 0 || id >= kv.num_blocks || kv.ref_count[id] < 1) bad_id = 1;
    }
  }
  if (__syncthreads_or(bad_len)) {
    if (threadIdx.x == 0) record(status, SV_ERR_BAD_LENGTH);
    return;
  }
  if (__syncthreads_or(bad_id)) {
    if (threadIdx.x == 0) record(status, SV_ERR_BAD_BLOCK_ID);
    return;
  }
  for (int k = warp; k < n; k += nwarps) {
    const int p = parents[k], c = children[k];
    const int len = kv.seq_lens[p];
    const int32_t *prow = kv.block_table + (size_t)p * kv.max_blocks;
    int32_t *crow = kv.block_table + (size_t)c * kv.max_blocks;
    for (int lb = lane; lb < blocks_for(len, bs); lb += 32) {
      crow[lb] = prow[lb];
      atomicAdd(&kv.ref_count[prow[lb]], 1);
    }
    if (lane == 0) kv.seq_lens[c] = len;  // children are not parents: no parent length changes under another warp
  }
}

// A block held only by listed sequences goes back at the last listed sequence
// that holds it. With counts: every listed reference is dropped (atomics); the
// blocks that reach zero are marked -1, then take the minimum over their
// holders of -(list index + 2), so the last holder finds its own mark; each
// sequence then pushes its marked blocks, highest logical block first, at an
// offset from a scan over the list. One warp per listed sequence, lanes over
// its blocks; the list goes through in batches of one sequence per thread for
// the scan.
__global__ void __launch_bounds__(kBookThreads) kv_release_kernel(KV kv, const int32_t *seqs, int n,
                                                                  int32_t *status) {
  grid_dependency_wait();  // the earlier kernel on the stream is complete and visible
  grid_dependents_launch();
  __shared__ unsigned s_seen[kMaxSeqBits / 32];
  __shared__ int s_cnt[kBookThreads];  // pushes of each sequence of the batch, then its offset
  const int B = kv.batch, bs = kv.block_size;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const bool sharing = kv.ref_count != nullptr;
  if (status_set(status)) return;
  const int top = *kv.free_top;
  for (int w = threadIdx.x; w < kMaxSeqBits / 32; w += blockDim.x) s_seen[w] = 0u;
  __syncthreads();
  int bad_len = 0, bad_id = 0;
  for (int j = threadIdx.x; j < n; j += blockDim.x) {
    const int b = seqs[j];
    if (b < 0 || b >= B || mark(s_seen, b)) {
      bad_len = 1;
      continue;
    }
    const int len = kv.seq_lens[b];
    if (len < 0 || blocks_for(len, bs) > kv.max_blocks) bad_len = 1;
  }
  if (__syncthreads_or(bad_len)) {
    if (threadIdx.x == 0) record(status, SV_ERR_BAD_LENGTH);
    return;
  }
  auto each_ref = [&](auto f) {  // f(list index, block id) over every listed reference, a warp per sequence
    for (int j = warp; j < n; j += nwarps) {
      const int b = seqs[j];
      const int32_t *row = kv.block_table + (size_t)b * kv.max_blocks;
      for (int lb = lane; lb < blocks_for(kv.seq_lens[b], bs); lb += 32) f(j, row[lb]);
    }
  };
  each_ref([&](int, int id) { bad_id |= id < 0 || id >= kv.num_blocks; });
  if (__syncthreads_or(bad_id)) {
    if (threadIdx.x == 0) record(status, SV_ERR_BAD_BLOCK_ID);
    return;
  }
  if (sharing) {
    each_ref([&](int, int id) { atomicSub(&kv.ref_count[id], 1); });
    __syncthreads();
    each_ref([&](int, int id) { bad_id |= kv.ref_count[id] < 0; });
    if (__syncthreads_or(bad_id)) {  // more references dropped than counted: put the counts back
      each_ref([&](int, int id) { atomicAdd(&kv.ref_count[id], 1); });
      if (threadIdx.x == 0) record(status, SV_ERR_BAD_BLOCK_ID);
      return;
    }
    each_ref([&](int, int id) {
      if (kv.ref_count[id] == 0) kv.ref_count[id] = -1;  // every writer stores the same value
    });
    __syncthreads();
    each_ref([&](int j, int id) {
      if (kv.ref_count[id] < 0) atomicMin(&kv.ref_count[id], -(j + 2));
    });
    __syncthreads();
  }
  auto pushed = [&](int j, int id) { return !sharing || kv.ref_count[id] == -(j + 2); };
  // total pushes, to check the free list's room before anything moves
  int mine = 0;
  each_ref([&](int j, int id) { mine += pushed(j, id); });
  __shared__ int s_total;
  if (threadIdx.x == 0) s_total = 0;
  __syncthreads();
  if (mine) atomicAdd(&s_total, mine);
  __syncthreads();
  const int all = s_total;
  if (top < 0 || top + all > kv.num_blocks) {
    // a free list that would overflow: nothing has moved but the counts, which go back
    if (sharing) {
      each_ref([&](int, int id) {
        if (kv.ref_count[id] < 0) kv.ref_count[id] = 0;
      });
      __syncthreads();
      each_ref([&](int, int id) { atomicAdd(&kv.ref_count[id], 1); });
    }
    if (threadIdx.x == 0) record(status, SV_ERR_OUT_OF_BLOCKS);
    return;
  }
  // pushes in list order: batches of blockDim.x sequences; warps count, threads scan, warps push
  int carry = 0;
  for (int base = 0; base < n; base += blockDim.x) {
    const int cnt_n = min((int)blockDim.x, n - base);
    for (int jj = warp; jj < cnt_n; jj += nwarps) {
      const int j = base + jj, b = seqs[j];
      const int32_t *row = kv.block_table + (size_t)b * kv.max_blocks;
      int c = 0;
      for (int lb = lane; lb < blocks_for(kv.seq_lens[b], bs); lb += 32) c += pushed(j, row[lb]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
      if (lane == 0) s_cnt[jj] = c;
    }
    __syncthreads();
    int chunk_total;
    const int v = (int)threadIdx.x < cnt_n ? s_cnt[threadIdx.x] : 0;
    const int off = carry + block_excl_scan(v, &chunk_total);
    if ((int)threadIdx.x < cnt_n) s_cnt[threadIdx.x] = off;
    __syncthreads();
    for (int jj = warp; jj < cnt_n; jj += nwarps) {
      const int j = base + jj, b = seqs[j];
      const int32_t *row = kv.block_table + (size_t)b * kv.max_blocks;
      const int nb = blocks_for(kv.seq_lens[b], bs);
      int pos = top + s_cnt[jj];
      for (int c0 = 0; c0 < nb; c0 += 32) {  // highest logical block first
        const int lb = nb - 1 - (c0 + lane);
        const int id = lb >= 0 ? row[lb] : -1;
        const bool push = lb >= 0 && pushed(j, id);
        const unsigned m = __ballot_sync(0xffffffffu, push);
        if (push) kv.free_list[pos + __popc(m & ((1u << lane) - 1u))] = id;
        pos += __popc(m);
      }
    }
    carry += chunk_total;
    __syncthreads();  // s_cnt is reused by the next batch
  }
  __syncthreads();  // every mark has been read
  each_ref([&](int, int id) {
    if (sharing && kv.ref_count[id] < 0) kv.ref_count[id] = 0;
  });
  __syncthreads();  // the rows are still read above
  for (int j = warp; j < n; j += nwarps) {
    const int b = seqs[j];
    int32_t *row = kv.block_table + (size_t)b * kv.max_blocks;
    for (int lb = lane; lb < blocks_for(kv.seq_lens[b], bs); lb += 32) row[lb] = -1;
  }
  __syncthreads();  // lengths are read above until every row is cleared
  for (int j = threadIdx.x; j < n; j += blockDim.x) kv.seq_lens[seqs[j]] = 0;
  if (threadIdx.x == 0) *kv.free_top = top + all;
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

cudaError_t launch_kv_fork(const KV &kv, const int32_t *parents, const int32_t *children, int n_pairs,
                           int32_t *status, cudaStream_t st) {
  return launch_pdl(kv_fork_kernel, dim3(1), dim3(kBookThreads), 0, st, kv, parents, children, n_pairs, status);
}

cudaError_t launch_kv_release(const KV &kv, const int32_t *seqs, int n, int32_t *status, cudaStream_t st) {
  return launch_pdl(kv_release_kernel, dim3(1), dim3(kBookThreads), 0, st, kv, seqs, n, status);
}

int kv_cow_max_batch() { return kCowMaxBatch; }
int kv_max_seq_bits() { return kMaxSeqBits; }

}  // namespace sv
