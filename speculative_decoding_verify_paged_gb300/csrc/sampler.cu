// Fused verification sampler: one thread-block cluster per sequence.
//
// What it computes ("Speculative decoding and continuous batching in
// practice", sec. 1.2; "Speculative decoding principles and a vLLM production
// setup", sec. 2.1-2.2; greedy form: "LLM inference optimisation: speculative
// decoding and dynamic batching", engineering section):
//   p_i = softmax(l_target,i / T), q_i = softmax(l_draft,i / T);
//   accept x_i iff u_i < min(1, p_i(x_i) / q_i(x_i)), scanning i in order;
//   at the first rejection a, draw y from norm(max(0, p_a - q_a)) by inverse
//   CDF with u'; if all K drafts pass, draw y from p_K.
//   Greedy: accept while x_i == argmax p_i; y = argmax p_a.
//   Tree greedy: walk from the root to the child whose token is the argmax of
//   the current node's row; y = argmax of the last node's row.
//
// How: the vocabulary is cut into C equal chunks, one per CTA of the cluster.
//   phase 1  every CTA streams its chunk of every row of the sequence (target
//            rows and draft rows) once; a work item is 2 KB of one row for one
//            warp, and each warp has its next item's loads in flight while it
//            reduces the current one to a (max, sum of 2^((l - max) log2(e)/T))
//            pair, or to an argmax.
//   phase 2  cluster barrier; every CTA combines the C partial results of
//            every row through distributed shared memory with a fixed shuffle
//            tree (one lane per rank), so all CTAs hold identical row
//            statistics and take identical decisions.
//   phase 3  (T > 0) the row pair of the draw (target and draft row a, or the
//            bonus row) is copied once into shared memory. With a 128K
//            vocabulary the residual CDF has intervals of ~1e-5, so this phase
//            is exact where fp32 would not be: exponents carry log2(e)/T as a
//            hi+lo pair, the weights are summed in 64-bit fixed point (2^-40
//            units, order-free and exact), the draft normaliser enters as the
//            ratio Z_t/Z_d in hi+lo form, and the target is the integer
//            floor(u' * S). Pass A sums the two normalisers, pass B each
//            8-element group's residual mass (kept in shared memory) and each
//            CTA's total; after a cluster barrier the prefix over ranks picks
//            the CTA holding the crossing, which scans its group masses and
//            recomputes the one group that holds it.
// All reductions run in a fixed order, so results are deterministic.
#include <cooperative_groups.h>

#include <algorithm>
#include <cfloat>
#include <climits>

#include "sv_internal.cuh"

namespace cg = cooperative_groups;

namespace sv {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxQ = 64;
constexpr int kMaxRows = 2 * kMaxQ;  // target + draft rows of one sequence
constexpr int kMaxChunk = 16384;     // vocabulary elements per CTA
constexpr int kGroup = 8;            // consecutive elements of a group

// Phase 1 work item: one warp, LOADS loads of N elements per lane (2 KB).
template <typename T, bool VEC> struct ItemCfg;
template <> struct ItemCfg<__nv_bfloat16, true> { static constexpr int N = 8, LOADS = 4; };
template <> struct ItemCfg<float, true> { static constexpr int N = 4, LOADS = 4; };
template <typename T> struct ItemCfg<T, false> { static constexpr int N = 1, LOADS = 16; };
template <typename T, bool VEC> __host__ __device__ constexpr int item_elems() {
  return 32 * ItemCfg<T, VEC>::N * ItemCfg<T, VEC>::LOADS;
}

template <typename T, bool VEC> struct Raw;
template <typename T> struct Raw<T, true> { uint4 v; };
template <typename T> struct Raw<T, false> { T v; };

template <typename T, bool VEC>
__device__ __forceinline__ float elem(const Raw<T, VEC> &r, int k) {
  if constexpr (VEC) return to_f32(reinterpret_cast<const T *>(&r.v)[k]);
  else return to_f32(r.v);
}

// The lane's loads of one item: load u covers e0 + (u*32 + lane)*N .. +N.
// Chunks are multiples of N, so a load is wholly inside or outside [e0, e1).
template <typename T, bool VEC>
__device__ __forceinline__ void load_item(const T *__restrict__ row, int e0, int e1, int lane,
                                          Raw<T, VEC> (&raw)[ItemCfg<T, VEC>::LOADS], int &nvalid) {
  constexpr int N = ItemCfg<T, VEC>::N, LOADS = ItemCfg<T, VEC>::LOADS;
  nvalid = 0;
#pragma unroll
  for (int u = 0; u < LOADS; ++u) {
    const int e = e0 + (u * 32 + lane) * N;
    if (e < e1) {
      if constexpr (VEC) raw[u].v = __ldg(reinterpret_cast<const uint4 *>(row + e));
      else raw[u].v = row[e];
      nvalid = u + 1;
    }
  }
}

// 2^x by the MUFU approximation (flush-to-zero; relative error about 2^-22)
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (max, sum) pair combine: m is a raw logit maximum, s = sum 2^((l - m) * coef);
// m == -inf means "empty".
__device__ __forceinline__ void ms_combine(float &m, float &s, float m2, float s2, float coef) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) {
    m = mn;
    s = 0.f;
    return;
  }
  s = s * fast_exp2((m - mn) * coef) + s2 * fast_exp2((m2 - mn) * coef);
  m = mn;
}

// argmax combine: larger value wins, lower index on ties; idx -1 = empty.
__device__ __forceinline__ void am_combine(float &v, int &i, float v2, int i2) {
  if (i2 < 0) return;
  if (i < 0 || v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

// 2^(d * c) for d <= 0 with c = c_hi + c_lo: the product is carried to about
// 2^-40 before exp2f, so no rounding of c or of d*c shifts all weights alike.
__device__ __forceinline__ float exp2_acc(float d, float c_hi, float c_lo) {
  d = fmaxf(d, -200.f);  // -inf logits: 2^(d c) flushes to zero below 2^-126 either way
  const float xh = d * c_hi;
  const float xe = fmaf(d, c_hi, -xh) + d * c_lo;
  return fast_exp2(xh) * fmaf(xe, 0.69314718055994531f, 1.0f);
}

// Weights in [0, 1] as 64-bit fixed point with 40 fractional bits: sums of up
// to 2^23 of them are exact and independent of the order of addition.
__device__ __forceinline__ long long to_fix(float w) { return __float2ll_rn(w * 1099511627776.0f); }

__device__ long long block_sum_ll(long long x, long long *buf) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  if (lane == 0) buf[warp] = x;
  __syncthreads();
  long long t = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) t += buf[w];
  __syncthreads();
  return t;
}

__device__ long long block_excl_scan_ll(long long x, long long *buf, long long *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  long long inc = x;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  if (lane == 31) buf[warp] = inc;
  __syncthreads();
  long long before = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) {
    before += (w < warp) ? buf[w] : 0;
    tot += buf[w];
  }
  __syncthreads();
  *total = tot;
  return before + inc - x;
}

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// The eight elements of group g of a shared-memory copy of a chunk, as floats;
// -inf at and past element n (only the chunk's last group can reach it).
template <typename T>
__device__ __forceinline__ void group8(const T *buf, int g, int n, float (&x)[kGroup]) {
  const int e = g * kGroup;
  if constexpr (sizeof(T) == 2) {
    const uint4 r = *reinterpret_cast<const uint4 *>(buf + e);
    const uint32_t *w = reinterpret_cast<const uint32_t *>(&r);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[2 * k] = __uint_as_float(w[k] << 16);
      x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
    }
  } else {
    const uint4 r0 = *reinterpret_cast<const uint4 *>(buf + e);
    const uint4 r1 = *reinterpret_cast<const uint4 *>(buf + e + 4);
    const float *f0 = reinterpret_cast<const float *>(&r0), *f1 = reinterpret_cast<const float *>(&r1);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      x[k] = f0[k];
      x[k + 4] = f1[k];
    }
  }
  if (e + kGroup > n) {
#pragma unroll
    for (int k = 0; k < kGroup; ++k)
      if (e + k >= n) x[k] = -INFINITY;
  }
}

struct Smem {
  uint64_t pair;  // phase 3 row pair
  float rm[kMaxRows];  // per row, this CTA's chunk (cluster-visible)
  float rs[kMaxRows];
  int ri[kMaxRows];
  float tl[kMaxQ];  // target logit of the draft token, if this CTA owns it (cluster-visible)
  float dl[kMaxQ];
  float M[kMaxRows];  // per row, whole vocabulary (after phase 2)
  float Z[kMaxRows];
  int am[kMaxRows];
  float gtl[kMaxQ], gdl[kMaxQ];
  long long zt, zd;  // phase 3: this CTA's fixed-point normalisers (cluster-visible)
  long long S[2];    // phase 3: this CTA's fixed-point weight sum per pass (cluster-visible)
  long long ll_buf[kWarps];
  long long P_owner, target;
  float rho_hi, rho_lo;
  int a;
  int bad;
  int owner, fallback;
  int y_hit, y_last;
};

template <typename T, bool VEC, int MODE>
__global__ void __launch_bounds__(kThreads) sampler_kernel(SamplerArgs args, int ring_bytes) {
  grid_dependency_wait();  // the earlier kernel on the stream is complete and visible
  grid_dependents_launch();
  constexpr int IE = item_elems<T, VEC>();
  constexpr int LOADS = ItemCfg<T, VEC>::LOADS, N = ItemCfg<T, VEC>::N;
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ Smem sm;
  extern __shared__ __align__(128) uint8_t dyn[];
  // phase 1: per-row partials [kMaxRows][kWarps] x 2; phase 3: the row pair (same bytes)
  uint8_t *ring = dyn;
  float *pm = reinterpret_cast<float *>(dyn);
  float *ps = pm + kMaxRows * kWarps;
  long long *gmass = reinterpret_cast<long long *>(dyn + ring_bytes);  // phase 3: per-group mass

  const int V = args.vocab;
  const int t0 = args.cu_q[b];
  const int n = args.cu_q[b + 1] - t0;
  const int K = n - 1;
  const int d0 = t0 - b;
  const int lo = min(V, rank * args.chunk), hi = min(V, lo + args.chunk);
  const int len = hi - lo;
  const int rows = (MODE == kStochastic) ? n + K : n;
  const T *tgt = reinterpret_cast<const T *>(args.tgt);
  const T *drf = reinterpret_cast<const T *>(args.drf);
  const float coef = args.coef;

  // rows outside [0, total_q) or more than max_q rows: nothing is read or written.
  // Every CTA of the cluster takes this exit together (same b), before any barrier.
  if (n < 1 || n > args.max_q || t0 < 0 || t0 + n > args.total_q) {
    if (rank == 0 && tid == 0) record(args.status, SV_ERR_BAD_LENGTH);
    return;
  }
  if (tid == 0) {
    sm.bad = 0;
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm.pair)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  bool ok = true;  // false after a bounded wait gave up: the remaining work is skipped, barriers are kept

  // ---------------- phase 1: per-row statistics of this CTA's chunk ----------------
  // The items (2 KB of one row, row-major) are cut into kWarps contiguous runs, one
  // per warp. A lane accumulates its share of the current row online; the warp
  // reduces only where its run leaves a row, into slot [row][warp]. The next
  // item's loads are in flight while the current one is reduced.
  const int nsub = (len + IE - 1) / IE;
  const int items = rows * nsub;
  const int it_begin = (int)((long long)items * warp / kWarps);
  const int it_end = (int)((long long)items * (warp + 1) / kWarps);
  for (int x = tid; x < rows * kWarps; x += kThreads) {
    pm[x] = (MODE == kStochastic) ? -INFINITY : 0.f;
    ps[x] = (MODE == kStochastic) ? 0.f : __int_as_float(-1);
  }
  __syncthreads();
  int bad = 0;
  float lm = -INFINITY, ls = 0.f;  // stochastic: this lane's running max and sum of 2^((x - lm) c)
  float lb = 0.f;                  // greedy: this lane's best value and its index
  int lbi = -1;
  int cur_row = -1;
  auto flush = [&]() {  // warp-uniform: the lanes' state of cur_row into slot [cur_row][warp]
    if constexpr (MODE == kStochastic) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, lm, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, ls, o);
        ms_combine(lm, ls, m2, s2, coef);
      }
      if (lane == 0) {
        pm[cur_row * kWarps + warp] = lm;
        ps[cur_row * kWarps + warp] = ls;
      }
      lm = -INFINITY;
      ls = 0.f;
    } else {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, lb, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, lbi, o);
        am_combine(lb, lbi, v2, i2);
      }
      if (lane == 0) {
        pm[cur_row * kWarps + warp] = lb;
        ps[cur_row * kWarps + warp] = __int_as_float(lbi);
      }
      lb = 0.f;
      lbi = -1;
    }
  };
  // this lane's elements of item it into the running state
  auto reduce_item = [&](int it, const Raw<T, VEC> (&raw)[LOADS], int nv) {
    const int r = it / nsub, sub = it % nsub;
    if (r != cur_row) {
      if (cur_row >= 0) flush();
      cur_row = r;
    }
    const int e0 = lo + sub * IE;
    if constexpr (MODE == kStochastic) {
      float mi;
      if constexpr (VEC && sizeof(T) == 2) {
        // bf16 pairs: the maximum on packed pairs, NaN propagating
        __nv_bfloat162 mx2 = __floats2bfloat162_rn(-INFINITY, -INFINITY);
#pragma unroll
        for (int u = 0; u < LOADS; ++u)
          if (u < nv) {
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&raw[u].v);
#pragma unroll
            for (int k = 0; k < 4; ++k) mx2 = __hmax2_nan(mx2, h[k]);
          }
        const float l2 = __low2float(mx2), h2 = __high2float(mx2);
        mi = (l2 != l2 || h2 != h2) ? NAN : fmaxf(l2, h2);
      } else {
        mi = -INFINITY;
#pragma unroll
        for (int u = 0; u < LOADS; ++u)
          if (u < nv)
#pragma unroll
            for (int k = 0; k < N; ++k) {
              const float x = elem<T, VEC>(raw[u], k);
              mi = (x != x || mi != mi) ? NAN : fmaxf(mi, x);
            }
      }
      bad |= (mi != mi) | (mi == INFINITY);
      if (!(mi == mi) || mi == -INFINITY) return;  // nothing to add (or the row is reported)
      if (mi > lm) {
        ls = (lm == -INFINITY) ? 0.f : ls * fast_exp2((lm - mi) * coef);
        lm = mi;
      }
      const float nmc = -lm * coef;
      float acc = 0.f;
      if constexpr (VEC && sizeof(T) == 2) {
#pragma unroll
        for (int u = 0; u < LOADS; ++u)
          if (u < nv) {
            const uint32_t *w = reinterpret_cast<const uint32_t *>(&raw[u].v);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              acc += fast_exp2(fmaf(__uint_as_float(w[k] << 16), coef, nmc));
              acc += fast_exp2(fmaf(__uint_as_float(w[k] & 0xffff0000u), coef, nmc));
            }
          }
      } else {
#pragma unroll
        for (int u = 0; u < LOADS; ++u)
          if (u < nv)
#pragma unroll
            for (int k = 0; k < N; ++k) acc += fast_exp2(fmaf(elem<T, VEC>(raw[u], k), coef, nmc));
      }
      ls += acc;
    } else {
#pragma unroll
      for (int u = 0; u < LOADS; ++u)
        if (u < nv)
#pragma unroll
          for (int k = 0; k < N; ++k) {
            const float x = elem<T, VEC>(raw[u], k);
            bad |= (x != x);
            am_combine(lb, lbi, x, e0 + (u * 32 + lane) * N + k);
          }
    }
  };
  auto fetch = [&](int it, Raw<T, VEC> (&raw)[LOADS], int &nv) {
    const int r = it / nsub, sub = it % nsub;
    const T *row = (r < n) ? tgt + (size_t)(t0 + r) * V : drf + (size_t)(d0 + (r - n)) * V;
    const int e0 = lo + sub * IE;
    load_item<T, VEC>(row, e0, min(hi, e0 + IE), lane, raw, nv);
  };
  {
    Raw<T, VEC> ra[LOADS], rb[LOADS];
    int na = 0, nb = 0;
    int it = it_begin;
    if (it < it_end) fetch(it, ra, na);
    while (it < it_end) {
      if (it + 1 < it_end) fetch(it + 1, rb, nb);
      reduce_item(it, ra, na);
      if (++it >= it_end) break;
      if (it + 1 < it_end) fetch(it + 1, ra, na);
      reduce_item(it, rb, nb);
      ++it;
    }
    if (cur_row >= 0) flush();
  }
  __syncthreads();
  for (int r = tid; r < rows; r += kThreads) {
    if constexpr (MODE == kStochastic) {
      float m = -INFINITY, sum = 0.f;
      for (int w = 0; w < kWarps; ++w) ms_combine(m, sum, pm[r * kWarps + w], ps[r * kWarps + w], coef);
      sm.rm[r] = m;
      sm.rs[r] = sum;
    } else {
      float best = 0.f;
      int bi = -1;
      for (int w = 0; w < kWarps; ++w) am_combine(best, bi, pm[r * kWarps + w], __float_as_int(ps[r * kWarps + w]));
      sm.rm[r] = best;
      sm.ri[r] = bi;
    }
  }
  // token logits of the draft tokens this CTA owns
  if constexpr (MODE == kStochastic) {
    if (tid < K) {
      const int x = args.draft_tok[d0 + tid];
      if (x < 0 || x >= V) {
        record(args.status, SV_ERR_BAD_TOKEN);
      } else if (x >= lo && x < hi) {
        sm.tl[tid] = to_f32(tgt[(size_t)(t0 + tid) * V + x]);
        sm.dl[tid] = to_f32(drf[(size_t)(d0 + tid) * V + x]);
      }
    }
  }
  if (bad) atomicOr(&sm.bad, 1);
  __syncthreads();
  if (tid == 0 && sm.bad) record(args.status, SV_ERR_NONFINITE);
  cluster.sync();

  // ---------------- phase 2: combine across the cluster, one lane per rank ----------------
  for (int base = 0; base < rows * 16; base += kThreads) {
    const int x = base + tid, r = x >> 4, q = x & 15;
    const bool valid = x < rows * 16 && q < C;
    if constexpr (MODE == kStochastic) {
      float m = -INFINITY, s = 0.f;
      if (valid) {
        m = *cluster.map_shared_rank(&sm.rm[r], q);
        s = *cluster.map_shared_rank(&sm.rs[r], q);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        ms_combine(m, s, m2, s2, coef);
      }
      if (x < rows * 16 && q == 0) {
        sm.M[r] = m;
        sm.Z[r] = s;
      }
    } else {
      float best = 0.f;
      int bi = -1;
      if (valid) {
        best = *cluster.map_shared_rank(&sm.rm[r], q);
        bi = *cluster.map_shared_rank(&sm.ri[r], q);
      }
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, best, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
        am_combine(best, bi, v2, i2);
      }
      if (x < rows * 16 && q == 0) sm.am[r] = bi;
    }
  }
  if constexpr (MODE == kStochastic) {
    if (tid < K) {
      const int x = args.draft_tok[d0 + tid];
      const int owner = (x >= 0 && x < V) ? min(x / args.chunk, C - 1) : 0;
      sm.gtl[tid] = *cluster.map_shared_rank(&sm.tl[tid], owner);
      sm.gdl[tid] = *cluster.map_shared_rank(&sm.dl[tid], owner);
    }
  }
  __syncthreads();

  if constexpr (MODE == kGreedy) {
    if (rank == 0 && tid == 0) {
      int a = K;
      for (int i = 0; i < K; ++i)
        if (args.draft_tok[d0 + i] != sm.am[i]) {
          a = i;
          break;
        }
      int32_t *o = args.out_tok + (size_t)b * args.max_q;
      for (int j = 0; j < args.max_q; ++j) o[j] = j < a ? args.draft_tok[d0 + j] : -1;
      o[a] = sm.am[a];
      args.accept[b] = a;
      args.num_out[b] = a + 1;
    }
  } else if constexpr (MODE == kTree) {
    if (rank == 0 && tid == 0) {
      int32_t *o = args.out_tok + (size_t)b * args.max_q;
      int32_t *path = args.path + (size_t)b * args.max_q;
      for (int j = 0; j < args.max_q; ++j) {
        o[j] = -1;
        path[j] = -1;
      }
      int cur = 0, a = 0, am = sm.am[0];
      bool good = true;
      for (int j = 1; j < n; ++j) {
        const int p = args.parent[t0 + j];
        good &= (p >= 0 && p < n && p != j);
      }
      if (!good) record(args.status, SV_ERR_BAD_LENGTH);
      while (good && a < n - 1) {
        am = sm.am[cur];
        int next = -1;
        for (int j = 1; j < n; ++j)
          if (args.parent[t0 + j] == cur && args.draft_tok[d0 + j - 1] == am) {
            next = j;
            break;
          }
        if (next < 0) break;
        path[a] = next;
        o[a] = am;
        ++a;
        cur = next;
      }
      am = sm.am[cur];
      o[a] = am;
      args.accept[b] = a;
      args.num_out[b] = a + 1;
    }
  } else {
    // ---------------- accept scan (identical in every CTA) ----------------
    if (tid == 0) {
      int a = K;
      for (int i = 0; i < K; ++i) {
        const float Zt = sm.Z[i], Zd = sm.Z[n + i];
        const float p = exp2f((sm.gtl[i] - sm.M[i]) * coef) / Zt;
        const float q = exp2f((sm.gdl[i] - sm.M[n + i]) * coef) / Zd;
        const float thr = q > 0.f ? fminf(1.f, p / q) : 1.f;
        if (!(args.u_acc[d0 + i] < thr)) {
          a = i;
          break;
        }
      }
      sm.a = a;
      for (int r = 0; r < rows; ++r)
        if (!(sm.Z[r] > 0.f)) sm.bad = 1;
      if (sm.bad && rank == 0) record(args.status, SV_ERR_NONFINITE);
    }
    __syncthreads();
    const int a = sm.a;
    const bool resid = a < K;
    const T *trow = tgt + (size_t)(t0 + a) * V;
    const T *drow = resid ? drf + (size_t)(d0 + a) * V : nullptr;
    const float Mt = sm.M[a], Md = resid ? sm.M[n + a] : 0.f;
    const float chi = args.coef, clo = args.coef_lo;
    const float ur = args.u_res[b];
    const int pair_off = ((len * (int)sizeof(T) + 127) / 128) * 128;
    const T *bt = reinterpret_cast<const T *>(ring);
    const T *bd = reinterpret_cast<const T *>(ring + pair_off);
    const int ngroups = (len + kGroup - 1) / kGroup;

    // ---- the row pair of the draw into shared memory ----
    if (len > 0) {
      if (VEC) {
        if (tid == 0) {
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          const uint32_t bytes = static_cast<uint32_t>(len * sizeof(T));
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&sm.pair)),
                       "r"(resid ? 2 * bytes : bytes)
                       : "memory");
          asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                           smem_addr(ring)),
                       "l"(trow + lo), "r"(bytes), "r"(smem_addr(&sm.pair))
                       : "memory");
          if (resid)
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_addr(ring + pair_off)),
                "l"(drow + lo), "r"(bytes), "r"(smem_addr(&sm.pair))
                : "memory");
        }
        if (ok && !mbar_wait_bounded(smem_addr(&sm.pair), 0)) {
          ok = false;
          record(args.status, SV_ERR_TIMEOUT);
        }
      } else {
        T *wt = reinterpret_cast<T *>(ring);
        T *wd = reinterpret_cast<T *>(ring + pair_off);
        for (int k = tid; k < len; k += kThreads) {
          wt[k] = trow[lo + k];
          if (resid) wd[k] = drow[lo + k];
        }
      }
    }
    __syncthreads();

    // ---- pass A: fixed-point normalisers of the row pair (residual draws) ----
    if (resid) {
      long long zt = 0, zd = 0;
      if (ok) {
        for (int g = tid; g < ngroups; g += kThreads) {
          float xt[kGroup], xd[kGroup];
          group8<T>(bt, g, len, xt);
          group8<T>(bd, g, len, xd);
#pragma unroll
          for (int k = 0; k < kGroup; ++k) {
            zt += to_fix(exp2_acc(xt[k] - Mt, chi, clo));
            zd += to_fix(exp2_acc(xd[k] - Md, chi, clo));
          }
        }
      }
      zt = block_sum_ll(zt, sm.ll_buf);
      zd = block_sum_ll(zd, sm.ll_buf);
      if (tid == 0) {
        sm.zt = zt;
        sm.zd = zd;
      }
    }
    cluster.sync();
    if (resid && warp == 0) {
      long long Zt = 0, Zd = 0;
      if (lane < C) {
        Zt = *cluster.map_shared_rank(&sm.zt, lane);
        Zd = *cluster.map_shared_rank(&sm.zd, lane);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        Zt += __shfl_xor_sync(0xffffffffu, Zt, o);
        Zd += __shfl_xor_sync(0xffffffffu, Zd, o);
      }
      if (lane == 0) {
        // q_v enters as e_d * (Z_t / Z_d), carried as hi + lo
        const double rho = Zd > 0 ? (double)Zt / (double)Zd : 0.0;
        sm.rho_hi = (float)rho;
        sm.rho_lo = (float)(rho - (double)sm.rho_hi);
      }
    }
    __syncthreads();
    const float rho_hi = sm.rho_hi, rho_lo = sm.rho_lo;

    for (int pass = 0; pass < 2; ++pass) {
      const bool res_pass = resid && pass == 0;
      // the eight weights of group g, in [0, 1]: proportional to max(0, p_v - q_v)
      // (scaled by Z_t), or to p_v
      auto weights8 = [&](int g, long long (&w)[kGroup]) {
        float xt[kGroup];
        group8<T>(bt, g, len, xt);
        if (res_pass) {
          float xd[kGroup];
          group8<T>(bd, g, len, xd);
#pragma unroll
          for (int k = 0; k < kGroup; ++k) {
            const float et = exp2_acc(xt[k] - Mt, chi, clo);
            const float ed = exp2_acc(xd[k] - Md, chi, clo);
            w[k] = to_fix(fmaxf(et - fmaf(ed, rho_hi, ed * rho_lo), 0.f));
          }
        } else {
#pragma unroll
          for (int k = 0; k < kGroup; ++k) w[k] = to_fix(exp2_acc(xt[k] - Mt, chi, clo));
        }
      };
      // ---- pass B: each group's mass and this CTA's total ----
      long long mass = 0;
      if (ok) {
        for (int g = tid; g < ngroups; g += kThreads) {
          long long w[kGroup];
          weights8(g, w);
          long long m8 = 0;
#pragma unroll
          for (int k = 0; k < kGroup; ++k) m8 += w[k];
          gmass[g] = m8;
          mass += m8;
        }
      }
      mass = block_sum_ll(mass, sm.ll_buf);
      if (tid == 0) sm.S[pass] = mass;
      cluster.sync();
      if (warp == 0) {
        // the draw: the smallest v whose inclusive prefix exceeds u' * S
        const long long Sq = lane < C ? *cluster.map_shared_rank(&sm.S[pass], lane) : 0;
        long long inc = Sq;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long y = __shfl_up_sync(0xffffffffu, inc, o);
          if (lane >= o) inc += y;
        }
        const long long S = __shfl_sync(0xffffffffu, inc, 31);
        const long long target = (long long)floor((double)ur * (double)S);
        const unsigned hit = __ballot_sync(0xffffffffu, lane < C && inc > target);
        const unsigned has = __ballot_sync(0xffffffffu, Sq > 0);
        const int owner_l = hit ? __ffs(hit) - 1 : -1;
        const long long P_l = __shfl_sync(0xffffffffu, inc - Sq, owner_l < 0 ? 0 : owner_l);
        if (lane == 0) {
          sm.fallback = (res_pass && S == 0) ? 1 : 0;
          if (owner_l >= 0) {
            sm.owner = owner_l;
            sm.P_owner = P_l;
          } else {  // u' outside [0, 1): the last token with mass
            sm.owner = has ? 31 - __clz(has) : -1;
            sm.P_owner = -1;
          }
          sm.target = target;
          sm.y_hit = INT_MAX;
          sm.y_last = -1;
        }
      }
      __syncthreads();
      if (sm.fallback) continue;  // residual without mass: draw from p_a instead
      if (rank == sm.owner) {
        // ---- the owner: scan the group masses in order, then the group of the crossing ----
        const long long P = sm.P_owner, target = sm.target;
        const int per = (ngroups + kThreads - 1) / kThreads;  // consecutive groups of this thread
        const int g0 = min(ngroups, tid * per), g1 = min(ngroups, g0 + per);
        long long local = 0;
        int last_g = -1;
        for (int g = g0; g < g1; ++g) {
          local += gmass[g];
          if (gmass[g] > 0) last_g = g;
        }
        long long seg_total;
        long long cum = P + block_excl_scan_ll(local, sm.ll_buf, &seg_total);
        if (last_g >= 0) atomicMax(&sm.y_last, last_g);
        if (P >= 0) {
          for (int g = g0; g < g1 && cum <= target; ++g) {
            if (cum + gmass[g] > target) {  // the group whose prefix range holds the target
              long long w[kGroup];
              weights8(g, w);
              long long c2 = cum;
              int y = g * kGroup + kGroup - 1;
#pragma unroll
              for (int k = 0; k < kGroup; ++k) {
                c2 += w[k];
                if (c2 > target) {
                  y = g * kGroup + k;
                  break;
                }
              }
              atomicMin(&sm.y_hit, lo + y);
              break;
            }
            cum += gmass[g];
          }
        }
        __syncthreads();
        if (tid == 0) {
          int y = sm.y_hit;
          if (y == INT_MAX) {  // u' at or past the end: the last token with mass
            const int g = sm.y_last;
            y = lo + max(0, g) * kGroup;
            if (g >= 0) {
              long long w[kGroup];
              weights8(g, w);
              for (int k = 0; k < kGroup; ++k)
                if (w[k] > 0) y = lo + g * kGroup + k;
            }
          }
          int32_t *o = args.out_tok + (size_t)b * args.max_q;
          for (int j = 0; j < args.max_q; ++j) o[j] = j < a ? args.draft_tok[d0 + j] : -1;
          o[a] = y;
          args.accept[b] = a;
          args.num_out[b] = a + 1;
        }
      }
      break;
    }
  }
  cluster.sync();  // keep this CTA's shared memory alive until every peer is done reading it
}

// Cluster size: enough CTAs to cover the SMs a few times over, and chunks of at
// most kMaxChunk elements.
int pick_cluster(int batch, int vocab) {
  const int sms = num_sms();
  int C = (batch * 8 < 3 * sms) ? 16 : 8;
  while (C < 16 && (vocab + C - 1) / C > kMaxChunk) C *= 2;
  return C;
}

template <typename T, bool VEC, int MODE>
cudaError_t launch_t(const SamplerArgs &a, int C, cudaStream_t st) {
  auto kern = sampler_kernel<T, VEC, MODE>;
  const int pair = ((a.chunk * (int)sizeof(T) + 127) / 128) * 128;
  const int ring = std::max(2 * kMaxRows * kWarps * (int)sizeof(float), 2 * pair);
  const int groups = (a.chunk + kGroup - 1) / kGroup;
  const int dyn = ring + groups * (int)sizeof(long long);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  if (e != cudaSuccess) return e;
  if (C > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, a.batch, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = dyn;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see launch_pdl
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, a, ring);
}

// rows 16-byte aligned: vector loads and 1-D bulk copies (every chunk then starts on
// 16 bytes and is a multiple of 16 bytes long); otherwise scalar loads and copies
template <typename T, int MODE>
cudaError_t launch_m(const SamplerArgs &a, int C, cudaStream_t st) {
  const bool vec = ((size_t)a.vocab * sizeof(T)) % 16 == 0 && ((uintptr_t)a.tgt % 16 == 0) &&
                   (a.drf == nullptr || (uintptr_t)a.drf % 16 == 0);
  return vec ? launch_t<T, true, MODE>(a, C, st) : launch_t<T, false, MODE>(a, C, st);
}

template <typename T>
cudaError_t launch_d(const SamplerArgs &a, int mode, int C, cudaStream_t st) {
  switch (mode) {
    case kStochastic: return launch_m<T, kStochastic>(a, C, st);
    case kGreedy: return launch_m<T, kGreedy>(a, C, st);
    default: return launch_m<T, kTree>(a, C, st);
  }
}

}  // namespace

cudaError_t launch_sampler(const SamplerArgs &a0, int dtype, int mode, cudaStream_t st) {
  SamplerArgs a = a0;
  if (a.batch == 0) return cudaSuccess;
  const int C = pick_cluster(a.batch, a.vocab);
  a.chunk = ((a.vocab + C - 1) / C + 7) / 8 * 8;
  return dtype == SV_DTYPE_BF16 ? launch_d<__nv_bfloat16>(a, mode, C, st) : launch_d<float>(a, mode, C, st);
}

// Largest vocabulary: 16 chunks of kMaxChunk elements.
bool sampler_supports(int vocab) { return vocab <= 16 * kMaxChunk; }

}  // namespace sv
