// Split-KV paged attention on CUDA cores, and the split combine.
//
// Computes, for each sequence b, query row i and query head h (KV head
// h / (Hq / Hkv)):  o = sum_t softmax_t(scale * <q, k_t>) v_t over the visible
// keys t < c_b + n_b (committed keys always; new row j when j <= i, or when bit
// j of the row's tree mask is set). The keys of position t are read through
// the block table (physical block block_table[b][t / bs], slot t % bs), as in
// the PagedAttention section of "LLM serving: speculative decoding and
// PagedAttention memory management". Tree masks follow "Speculative decoding
// principles and a vLLM production setup", sec. 3.2 and 5.2.
//
// This path serves fp32 caches and shapes the tensor-core kernel does not
// cover. A CTA owns (sequence, KV head, split of the key range) and all
// G * n_b query rows of that KV head, 16 at a time; keys go through shared
// memory 32 at a time; a warp keeps four rows' online-softmax state (base-2
// exponent, running max m, running sum l, accumulator) with a lane per key for
// the scores and a lane per output column for the weighted sum.
//
// A sequence whose keys span several splits writes per-split partial results
// (O normalised by its own l, plus log2-sum-exp m + log2 l); the combine kernel
// merges them: o = sum_s 2^(lse_s - M) O_s / sum_s 2^(lse_s - M).
#include <cuda_fp8.h>

#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr int kThreads = 128;
constexpr int kKeys = 32;      // keys per shared-memory tile
constexpr int kRowsPerPass = 16;  // query rows per pass (4 per warp)

__device__ __forceinline__ bool key_visible(int t, int c, int i, int mask_kind, uint64_t tmask) {
  if (t < c) return true;
  const int j = t - c;
  if (mask_kind == SV_MASK_CAUSAL) return j <= i;
  return j < 64 && ((tmask >> j) & 1ull);
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

// A pool element as fp32: bf16 or fp32 as is, an E4M3 code (uint8_t) times the pool's scale.
__device__ __forceinline__ float kv_f32(__nv_bfloat16 x, float) { return __bfloat162float(x); }
__device__ __forceinline__ float kv_f32(float x, float) { return x; }
__device__ __forceinline__ float kv_f32(uint8_t x, float scale) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(x, __NV_E4M3);
  return __half2float(__half(h)) * scale;
}

template <typename T, typename KT /* pool element */, int NK /* head_dim / 32 */>
__global__ void __launch_bounds__(kThreads) attn_simt_kernel(AttnArgs a) {
  grid_dependency_wait();  // the earlier kernel on the stream is complete and visible
  grid_dependents_launch();
  constexpr int D = NK * 32;
  __shared__ float q_s[kRowsPerPass][D];
  __shared__ float k_s[kKeys][D + 1];
  __shared__ float v_s[kKeys][D];
  __shared__ int s_bad;

  const int split = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const KV &kv = a.kv;
  const int c = kv.seq_lens[b];
  const int row0 = a.cu_q[b];
  const int n = a.cu_q[b + 1] - row0;
  const int L = c + n;
  if (L > a.max_seq_len || c < 0 || n < 0 || row0 + n > a.total_q || L > kv.max_blocks * kv.block_size) {
    if (split == 0 && kvh == 0 && tid == 0) record(a.status, SV_ERR_BAD_LENGTH);
    return;
  }
  const int nsplit = (L + a.chunk - 1) / a.chunk;
  if (split >= nsplit) return;
  const int kb = split * a.chunk, ke = min(L, kb + a.chunk);
  const int G = a.num_q_heads / kv.num_kv_heads;
  const int R = G * n;
  const T *qp = reinterpret_cast<const T *>(a.q);
  const KT *kp = reinterpret_cast<const KT *>(kv.k_pool);
  const KT *vp = reinterpret_cast<const KT *>(kv.v_pool);
  if (tid == 0) s_bad = 0;

  for (int rg = 0; rg < R; rg += kRowsPerPass) {
    __syncthreads();
    for (int x = tid; x < kRowsPerPass * D; x += kThreads) {
      const int rr = x / D, d = x % D, r = rg + rr;
      float val = 0.f;
      if (r < R) {
        const int i = r / G, g = r % G;
        val = to_f32(qp[((size_t)(row0 + i) * a.num_q_heads + kvh * G + g) * D + d]);
      }
      q_s[rr][d] = val;
    }
    float m[4], l[4], acc[4][NK];
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      m[w] = -INFINITY;
      l[w] = 0.f;
#pragma unroll
      for (int k = 0; k < NK; ++k) acc[w][k] = 0.f;
    }
    for (int kt = kb; kt < ke; kt += kKeys) {
      __syncthreads();
      for (int x = tid; x < kKeys * D; x += kThreads) {
        const int j = x / D, d = x % D, t = kt + j;
        float kk = 0.f, vv = 0.f;
        if (t < ke) {
          const int blk = kv.block_table[(size_t)b * kv.max_blocks + t / kv.block_size];
          if (blk >= 0 && blk < kv.num_blocks) {
            const size_t off = (((size_t)blk * kv.num_kv_heads + kvh) * kv.block_size + t % kv.block_size) * D + d;
            kk = kv_f32(kp[off], kv.k_scale);
            vv = kv_f32(vp[off], kv.v_scale);
          } else {
            s_bad = 1;
          }
        }
        k_s[j][d] = kk;
        v_s[j][d] = vv;
      }
      __syncthreads();
      const int t = kt + lane;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const int rr = warp * 4 + w, r = rg + rr;
        if (r >= R) continue;
        const int i = r / G;
        const uint64_t tm = (a.mask_kind == SV_MASK_TREE) ? a.tree_mask[row0 + i] : 0ull;
        const bool vis = t < ke && key_visible(t, c, i, a.mask_kind, tm);
        float s = -INFINITY;
        if (vis) {
          float dot = 0.f;
#pragma unroll 8
          for (int d = 0; d < D; ++d) dot = fmaf(q_s[rr][d], k_s[lane][d], dot);
          s = dot * a.scale_log2;
        }
        const float mn = fmaxf(m[w], warp_max(s));
        if (mn == -INFINITY) continue;
        const float p = vis ? exp2f(s - mn) : 0.f;
        const float alpha = exp2f(m[w] - mn);
        l[w] = l[w] * alpha + warp_sum(p);
#pragma unroll
        for (int k = 0; k < NK; ++k) acc[w][k] *= alpha;
        const int nk = min(kKeys, ke - kt);
        for (int j = 0; j < nk; ++j) {
          const float pj = __shfl_sync(0xffffffffu, p, j);
#pragma unroll
          for (int k = 0; k < NK; ++k) acc[w][k] = fmaf(pj, v_s[j][lane + 32 * k], acc[w][k]);
        }
        m[w] = mn;
      }
    }
    // write this pass's rows
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const int r = rg + warp * 4 + w;
      if (r >= R) continue;
      const int i = r / G, g = r % G, h = kvh * G + g;
      const size_t qrow = (size_t)(row0 + i) * a.num_q_heads + h;
      const float inv = l[w] > 0.f ? 1.f / l[w] : 0.f;
      if (nsplit == 1) {
        T *op = reinterpret_cast<T *>(a.out);
#pragma unroll
        for (int k = 0; k < NK; ++k) op[qrow * D + lane + 32 * k] = from_f32<T>(acc[w][k] * inv);
      } else {
        const size_t prow = (size_t)split * a.total_q * a.num_q_heads + qrow;
#pragma unroll
        for (int k = 0; k < NK; ++k) a.ws_o[prow * D + lane + 32 * k] = acc[w][k] * inv;
        if (lane == 0) a.ws_lse[prow] = l[w] > 0.f ? m[w] + log2f(l[w]) : -INFINITY;
      }
    }
  }
  __syncthreads();
  if (tid == 0 && s_bad) record(a.status, SV_ERR_BAD_BLOCK_ID);
}

// One warp per (query row, query head): merge the split partials.
template <typename T>
__global__ void __launch_bounds__(128) attn_combine_kernel(AttnArgs a) {
  grid_dependency_wait();  // the earlier kernel on the stream is complete and visible
  grid_dependents_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long idx = (long long)blockIdx.x * 4 + warp;
  if (idx >= (long long)a.total_q * a.num_q_heads) return;
  const int row = (int)(idx / a.num_q_heads);
  // sequence of this row: the last b with cu_q[b] <= row
  int lo = 0, hi = a.kv.batch;  // invariant: cu_q[lo] <= row < cu_q[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a.cu_q[mid] <= row) lo = mid;
    else hi = mid;
  }
  const int b = lo;
  const int L = a.kv.seq_lens[b] + a.cu_q[b + 1] - a.cu_q[b];
  if (L > a.max_seq_len || a.cu_q[b + 1] > a.total_q || L > a.kv.max_blocks * a.kv.block_size) return;
  const int nsplit = (L + a.chunk - 1) / a.chunk;
  if (nsplit <= 1) return;
  const int D = a.kv.head_dim;
  const size_t stride = (size_t)a.total_q * a.num_q_heads;
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, a.ws_lse[s * stride + idx]);
  T *op = reinterpret_cast<T *>(a.out);
  for (int d = lane; d < D; d += 32) {
    float num = 0.f, den = 0.f;
    if (M != -INFINITY) {
      for (int s = 0; s < nsplit; ++s) {
        const float w = exp2f(a.ws_lse[s * stride + idx] - M);
        den += w;
        num = fmaf(w, a.ws_o[(s * stride + idx) * D + d], num);
      }
    }
    op[(size_t)idx * D + d] = from_f32<T>(den > 0.f ? num / den : 0.f);
  }
}

template <typename T, typename KT, int NK>
cudaError_t launch_nk(const AttnArgs &a, cudaStream_t st) {
  dim3 grid(a.max_splits, a.kv.num_kv_heads, a.kv.batch);
  return launch_pdl(attn_simt_kernel<T, KT, NK>, grid, dim3(kThreads), 0, st, a);
}

template <typename T, typename KT>
cudaError_t launch_t(const AttnArgs &a, cudaStream_t st) {
  switch (a.kv.head_dim / 32) {
    case 1: return launch_nk<T, KT, 1>(a, st);
    case 2: return launch_nk<T, KT, 2>(a, st);
    case 3: return launch_nk<T, KT, 3>(a, st);
    case 4: return launch_nk<T, KT, 4>(a, st);
    case 5: return launch_nk<T, KT, 5>(a, st);
    case 6: return launch_nk<T, KT, 6>(a, st);
    case 7: return launch_nk<T, KT, 7>(a, st);
    default: return launch_nk<T, KT, 8>(a, st);
  }
}

}  // namespace

cudaError_t launch_attn_simt(const AttnArgs &a, int dtype, cudaStream_t st) {
  if (a.kv.batch == 0) return cudaSuccess;
  if (dtype == SV_DTYPE_E4M3) return launch_t<__nv_bfloat16, uint8_t>(a, st);  // bf16 queries and outputs
  return dtype == SV_DTYPE_BF16 ? launch_t<__nv_bfloat16, __nv_bfloat16>(a, st) : launch_t<float, float>(a, st);
}

cudaError_t launch_attn_combine(const AttnArgs &a, int dtype, cudaStream_t st) {
  if (a.max_splits <= 1 || a.total_q == 0) return cudaSuccess;
  const long long warps = (long long)a.total_q * a.num_q_heads;
  const unsigned blocks = (unsigned)((warps + 3) / 4);
  if (dtype == SV_DTYPE_BF16 || dtype == SV_DTYPE_E4M3)
    return launch_pdl(attn_combine_kernel<__nv_bfloat16>, dim3(blocks), dim3(128), 0, st, a);
  return launch_pdl(attn_combine_kernel<float>, dim3(blocks), dim3(128), 0, st, a);
}

}  // namespace sv
