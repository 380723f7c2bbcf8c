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
//            rows and draft rows) once; a work item is 4 KB of one row for
//            one warp (eight 16-byte loads in flight per lane), reduced to a
//            (max, sum of 2^((l - max) log2(e)/T)) pair, or to an argmax.
//   phase 2  cluster barrier; every CTA combines the C partial results of
//            every row through distributed shared memory in rank order, so all
//            CTAs hold identical row statistics and take identical decisions.
//   phase 3  (T > 0) the row pair of the draw (target and draft row a, or the
//            bonus row) is re-read. With a 128K vocabulary the residual CDF
//            has intervals of ~1e-5, so this phase is exact where fp32 would
//            not be: exponents carry log2(e)/T as a hi+lo pair, the weights
//            are summed in 64-bit fixed point (2^-40 units, order-free and
//            exact), the draft normaliser enters as the ratio Z_t/Z_d in
//            hi+lo form, and the target is the integer floor(u' * S). Pass A
//            sums the two normalisers, pass B each CTA's residual mass, and
//            after a cluster barrier the prefix over ranks picks the CTA
//            holding the crossing, which rescans its chunk (pass C).
// All reductions run in a fixed order, so results are deterministic.
#include <cooperative_groups.h>

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
constexpr int kMaxSub = 16;          // work items per row per CTA
constexpr int kMaxChunk = 16384;     // vocabulary elements per CTA
constexpr int kGroup = 8;            // phase 3: consecutive elements per thread
constexpr int kSeg = kThreads * kGroup;

// Work-item geometry: LOADS loads of N elements per lane.
template <typename T, bool VEC> struct ItemCfg;
template <> struct ItemCfg<__nv_bfloat16, true> { static constexpr int N = 8, LOADS = 8; };
template <> struct ItemCfg<float, true> { static constexpr int N = 4, LOADS = 8; };
template <typename T> struct ItemCfg<T, false> { static constexpr int N = 1, LOADS = 32; };
template <typename T, bool VEC> __host__ __device__ constexpr int item_elems() { return 32 * ItemCfg<T, VEC>::N * ItemCfg<T, VEC>::LOADS; }

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

// (max, sum) pair combine: m is a raw logit maximum, s = sum 2^((l - m) * coef);
// m == -inf means "empty".
__device__ __forceinline__ void ms_combine(float &m, float &s, float m2, float s2, float coef) {
  const float mn = fmaxf(m, m2);
  if (mn == -INFINITY) {
    m = mn;
    s = 0.f;
    return;
  }
  s = s * exp2f((m - mn) * coef) + s2 * exp2f((m2 - mn) * coef);
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
  const float xh = d * c_hi;
  if (!(xh > -160.f)) return 0.f;  // -inf logits and underflow
  const float xe = fmaf(d, c_hi, -xh) + d * c_lo;
  return exp2f(xh) * fmaf(xe, 0.69314718055994531f, 1.0f);
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

// Eight consecutive logits e .. e+7 of a row as floats; -inf past `hi`.
template <typename T, bool VEC>
__device__ __forceinline__ void load8(const T *__restrict__ row, int e, int hi, float (&x)[kGroup]) {
  if (VEC && e + kGroup <= hi) {
    if constexpr (sizeof(T) == 2) {
      const uint4 r = __ldg(reinterpret_cast<const uint4 *>(row + e));
      const T *t = reinterpret_cast<const T *>(&r);
#pragma unroll
      for (int k = 0; k < 8; ++k) x[k] = to_f32(t[k]);
    } else {
      const uint4 r0 = __ldg(reinterpret_cast<const uint4 *>(row + e));
      const uint4 r1 = __ldg(reinterpret_cast<const uint4 *>(row + e + 4));
      const float *f0 = reinterpret_cast<const float *>(&r0), *f1 = reinterpret_cast<const float *>(&r1);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[k] = f0[k];
        x[k + 4] = f1[k];
      }
    }
  } else {
#pragma unroll
    for (int k = 0; k < kGroup; ++k) x[k] = (e + k < hi) ? to_f32(row[e + k]) : -INFINITY;
  }
}

struct Smem {
  float pm[kMaxRows][kMaxSub];  // per item: raw max, or best value
  float ps[kMaxRows][kMaxSub];  // per item: sum of exp2, or best index (as int bits)
  float rm[kMaxRows];           // per row, this CTA's chunk (cluster-visible)
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
  int y_min, y_last;
  int owner, fallback;
};

template <typename T, bool VEC, int MODE>
__global__ void __launch_bounds__(kThreads) sampler_kernel(SamplerArgs args) {
  constexpr int IE = item_elems<T, VEC>();
  constexpr int LOADS = ItemCfg<T, VEC>::LOADS, N = ItemCfg<T, VEC>::N;
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ Smem sm;

  const int V = args.vocab;
  const int t0 = args.cu_q[b];
  const int n = args.cu_q[b + 1] - t0;
  const int K = n - 1;
  const int d0 = t0 - b;
  const int lo = min(V, rank * args.chunk), hi = min(V, lo + args.chunk);
  const int len = hi - lo;
  const int nsub = (len + IE - 1) / IE;
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
  if (tid == 0) sm.bad = 0;
  __syncthreads();

  // ---------------- phase 1: per-item partial statistics ----------------
  int bad = 0;
  const int items = rows * nsub;
  for (int it = warp; it < items; it += kWarps) {
    const int r = it / nsub, s = it % nsub;
    const T *row = (r < n) ? tgt + (size_t)(t0 + r) * V : drf + (size_t)(d0 + (r - n)) * V;
    const int e0 = lo + s * IE, e1 = min(hi, e0 + IE);
    Raw<T, VEC> raw[LOADS];
    int nv;
    load_item<T, VEC>(row, e0, e1, lane, raw, nv);
    if constexpr (MODE == kStochastic) {
      float m = -INFINITY;  // raw logit maximum (exact)
#pragma unroll
      for (int u = 0; u < LOADS; ++u)
        if (u < nv)
#pragma unroll
          for (int k = 0; k < N; ++k) {
            const float x = elem<T, VEC>(raw[u], k);
            bad |= (x != x) | (x == INFINITY);
            m = fmaxf(m, x);
          }
      float sum = 0.f;
      if (m != -INFINITY) {
#pragma unroll
        for (int u = 0; u < LOADS; ++u)
          if (u < nv)
#pragma unroll
            for (int k = 0; k < N; ++k) sum += exp2f((elem<T, VEC>(raw[u], k) - m) * coef);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
        const float s2 = __shfl_xor_sync(0xffffffffu, sum, o);
        ms_combine(m, sum, m2, s2, coef);
      }
      if (lane == 0) {
        sm.pm[r][s] = m;
        sm.ps[r][s] = sum;
      }
    } else {
      float best = 0.f;
      int bi = -1;
#pragma unroll
      for (int u = 0; u < LOADS; ++u)
        if (u < nv)
#pragma unroll
          for (int k = 0; k < N; ++k) {
            const float x = elem<T, VEC>(raw[u], k);
            bad |= (x != x);
            am_combine(best, bi, x, e0 + (u * 32 + lane) * N + k);
          }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, best, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
        am_combine(best, bi, v2, i2);
      }
      if (lane == 0) {
        sm.pm[r][s] = best;
        sm.ps[r][s] = __int_as_float(bi);
      }
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
  if (tid < rows) {
    if constexpr (MODE == kStochastic) {
      float m = -INFINITY, s = 0.f;
      for (int k = 0; k < nsub; ++k) ms_combine(m, s, sm.pm[tid][k], sm.ps[tid][k], coef);
      sm.rm[tid] = m;
      sm.rs[tid] = s;
    } else {
      float best = 0.f;
      int bi = -1;
      for (int k = 0; k < nsub; ++k) am_combine(best, bi, sm.pm[tid][k], __float_as_int(sm.ps[tid][k]));
      sm.rm[tid] = best;
      sm.ri[tid] = bi;
    }
  }
  if (tid == 0 && sm.bad) record(args.status, SV_ERR_NONFINITE);
  cluster.sync();

  // ---------------- phase 2: combine across the cluster ----------------
  if (tid < rows) {
    if constexpr (MODE == kStochastic) {
      float m = -INFINITY, s = 0.f;
      for (int q = 0; q < C; ++q) {
        const float m2 = *cluster.map_shared_rank(&sm.rm[tid], q);
        const float s2 = *cluster.map_shared_rank(&sm.rs[tid], q);
        ms_combine(m, s, m2, s2, coef);
      }
      sm.M[tid] = m;
      sm.Z[tid] = s;
    } else {
      float best = 0.f;
      int bi = -1;
      for (int q = 0; q < C; ++q)
        am_combine(best, bi, *cluster.map_shared_rank(&sm.rm[tid], q), *cluster.map_shared_rank(&sm.ri[tid], q));
      sm.am[tid] = bi;
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
      bool ok = true;
      for (int j = 1; j < n; ++j) {
        const int p = args.parent[t0 + j];
        ok &= (p >= 0 && p < n && p != j);
      }
      if (!ok) record(args.status, SV_ERR_BAD_LENGTH);
      while (ok && a < n - 1) {
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

    // ---- pass A: fixed-point normalisers of the row pair (residual draws) ----
    if (resid) {
      long long zt = 0, zd = 0;
      for (int e = lo + tid * kGroup; e < hi; e += kSeg) {
        float xt[kGroup], xd[kGroup];
        load8<T, VEC>(trow, e, hi, xt);
        load8<T, VEC>(drow, e, hi, xd);
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
          zt += to_fix(exp2_acc(xt[k] - Mt, chi, clo));
          zd += to_fix(exp2_acc(xd[k] - Md, chi, clo));
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
    if (resid && tid == 0) {
      long long Zt = 0, Zd = 0;
      for (int q = 0; q < C; ++q) {
        Zt += *cluster.map_shared_rank(&sm.zt, q);
        Zd += *cluster.map_shared_rank(&sm.zd, q);
      }
      // q_v enters as e_d * (Z_t / Z_d), carried as hi + lo
      const double rho = Zd > 0 ? (double)Zt / (double)Zd : 0.0;
      sm.rho_hi = (float)rho;
      sm.rho_lo = (float)(rho - (double)sm.rho_hi);
    }
    __syncthreads();
    const float rho_hi = sm.rho_hi, rho_lo = sm.rho_lo;

    for (int pass = 0; pass < 2; ++pass) {
      const bool res_pass = resid && pass == 0;
      // the eight weights of elements e .. e+7, in [0, 1]: proportional to
      // max(0, p_v - q_v) (scaled by Z_t), or to p_v
      auto weights8 = [&](int e, long long (&w)[kGroup]) {
        float xt[kGroup];
        load8<T, VEC>(trow, e, hi, xt);
        if (res_pass) {
          float xd[kGroup];
          load8<T, VEC>(drow, e, hi, xd);
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
      // ---- pass B: this CTA's fixed-point mass ----
      long long mass = 0;
      for (int e = lo + tid * kGroup; e < hi; e += kSeg) {
        long long w[kGroup];
        weights8(e, w);
#pragma unroll
        for (int k = 0; k < kGroup; ++k) mass += w[k];
      }
      mass = block_sum_ll(mass, sm.ll_buf);
      if (tid == 0) sm.S[pass] = mass;
      cluster.sync();
      if (tid == 0) {
        long long S = 0;
        for (int q = 0; q < C; ++q) S += *cluster.map_shared_rank(&sm.S[pass], q);
        // the draw: the smallest v whose inclusive prefix exceeds u' * S
        const long long target = (long long)floor((double)ur * (double)S);
        long long cum = 0, P = 0;
        int owner = -1, last_pos = -1;
        for (int q = 0; q < C; ++q) {
          const long long Sq = *cluster.map_shared_rank(&sm.S[pass], q);
          if (Sq > 0) last_pos = q;
          if (owner < 0 && cum + Sq > target) {
            owner = q;
            P = cum;
          }
          cum += Sq;
        }
        sm.fallback = (res_pass && S == 0) ? 1 : 0;
        sm.y_min = INT_MAX;
        sm.y_last = -1;
        if (owner < 0) {  // u' outside [0, 1): the last token with mass
          owner = last_pos;
          P = -1;
        }
        sm.owner = owner;
        sm.P_owner = P;
        sm.target = target;
      }
      __syncthreads();
      if (sm.fallback) continue;  // residual without mass: draw from p_a instead
      if (rank == sm.owner) {
        // ---- pass C: exact prefix sums over this chunk, segment by segment ----
        const long long P = sm.P_owner, target = sm.target;
        long long carry = 0;
        for (int s0 = lo; s0 < hi; s0 += kSeg) {
          const int e = s0 + tid * kGroup;
          long long w[kGroup];
          if (e < hi) {
            weights8(e, w);
          } else {
#pragma unroll
            for (int k = 0; k < kGroup; ++k) w[k] = 0;
          }
          long long local = 0;
#pragma unroll
          for (int k = 0; k < kGroup; ++k) local += w[k];
          long long seg_total;
          const long long excl = block_excl_scan_ll(local, sm.ll_buf, &seg_total);
          long long inc = P + carry + excl;
#pragma unroll
          for (int k = 0; k < kGroup; ++k) {
            inc += w[k];
            if (w[k] > 0) {
              if (P >= 0 && inc > target) atomicMin(&sm.y_min, e + k);
              atomicMax(&sm.y_last, e + k);
            }
          }
          carry += seg_total;
        }
        __syncthreads();
        if (tid == 0) {
          const int y = (sm.y_min != INT_MAX) ? sm.y_min : sm.y_last;
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
  if (C > 8) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(C, a.batch, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a);
}

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

// Largest vocabulary: 16 chunks of kMaxChunk elements (a chunk is at most
// kMaxSub work items of 1024 or 2048 elements).
bool sampler_supports(int vocab) { return vocab <= 16 * kMaxChunk; }

}  // namespace sv
