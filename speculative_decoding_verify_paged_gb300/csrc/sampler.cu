// Verification sampler: a row-statistics kernel, then one decision cluster
// per sequence.
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
//   Tree at T > 0: children are point-mass proposals, accepted with p'(x) (p
//   without the siblings rejected before, renormalised); y drawn from p'.
//   Optional margin: the smallest |uniform - threshold| of a sequence's
//   decisions, the draw's included (near-ties below 1e-4).
//
// How:
//   statistics  every row of the batch (target rows, then draft rows) is cut
//               into 32 KB items; the launch's items are cut into contiguous
//               ranges (one item apart at most), one per persistent CTA, so the whole batch
//               streams through every SM at once whatever the number of
//               sequences. A producer warp keeps three items in flight with 1-D
//               bulk copies; eight consumer warps reduce each item to a
//               (max, sum of 2^((l - max) log2(e)/T)) pair, or to an argmax,
//               per warp, into a workspace of per-(item, warp) partials.
//   decisions   one cluster per sequence (4, 8 or 16 CTAs; one for greedy and
//               greedy tree). The tree walks run on one warp. Every
//               CTA combines its sequence's partials in the same fixed order,
//               so all CTAs hold identical row statistics and take identical
//               accept decisions. For T > 0 the row pair of the draw (target
//               and draft row a, or the bonus row) is then read once, cut into
//               one chunk per CTA. With a 128K vocabulary the residual CDF has
//               intervals of ~1e-5, so the draw is exact where fp32 would not
//               be: exponents carry log2(e)/T as a hi+lo pair, the weights are
//               summed in 64-bit fixed point (2^-40 units, order-free and
//               exact), and the draft side enters as e_d Z_t/Z_d with the
//               normaliser ratio (from the row statistics, relative error about
//               1e-6) in hi+lo form; the target is the integer floor(u' * S).
//               One pass sums each 8-element group's residual mass (kept in
//               shared memory) and each CTA's total; after a cluster barrier
//               the prefix over ranks picks the CTA holding the crossing, which
//               scans its group masses and recomputes the one group that holds
//               it.
// All reductions run in a fixed order for a given device, so results are
// deterministic.
#include <cooperative_groups.h>

#include <algorithm>
#include <cfloat>
#include <climits>

#include "sv_internal.cuh"

namespace cg = cooperative_groups;

namespace sv {
namespace {

constexpr int kThreads = 256;  // decision kernel
constexpr int kWarps = kThreads / 32;
constexpr int kStatWarps = 8;                          // statistics kernel: consumer warps
constexpr int kStatThreads = (kStatWarps + 1) * 32;   // + one producer warp
constexpr int kStatStages = 3;
constexpr int kMaxRuns = 64;                           // statistics kernel: runs a CTA keeps until its wait
constexpr int kPartBytes = 32768;                      // one statistics item: 32 KB of one row
constexpr int kMaxQ = 64;
constexpr int kMaxRows = 2 * kMaxQ;  // target + draft rows of one sequence
constexpr int kMaxChunk = 32768;     // vocabulary elements per CTA
constexpr int kGroup = 8;            // consecutive elements of a group
// The decisions keep one fixed-point mass per unit of one group (8-CTA and larger clusters) or
// two groups (4-CTA clusters, whose chunks are twice as long), in shared memory with one spare
// slot every eight, so that the threads summing consecutive units read different bank pairs
__host__ __device__ constexpr int upad(int u) { return u + (u >> 3); }
constexpr int kSub = 4096;           // decisions: elements of a sub-chunk of the row pair (two groups a thread)
constexpr int kRingBytes = 65536;    // decisions: the sub-chunk ring (target and draft halves), 8-CTA and
                                     // larger clusters; half that at 4 CTAs, so that four fit an SM
constexpr int kMaxSubStages = 4;

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
// A weight below 2^-200 is returned as exactly zero; so is the weight of a
// -inf logit (and of the -inf padding past a chunk's end) at any temperature,
// as the statistics kernel gives it (to_fix rounds anything below 2^-41 to 0).
__device__ __forceinline__ float exp2_acc(float d, float c_hi, float c_lo) {
  const float xh = d * c_hi;  // -inf for d = -inf
  const float xe = fmaf(d, c_hi, -xh) + d * c_lo;
  const float w = fast_exp2(xh) * fmaf(xe, 0.69314718055994531f, 1.0f);  // NaN for d = -inf
  return xh > -200.f ? w : 0.f;
}

// Weights in [0, 1] as 64-bit fixed point with 40 fractional bits: sums of up
// to 2^23 of them are exact and independent of the order of addition. The
// value is round-to-nearest-even of w 2^40, formed from two 20-bit halves with
// single-precision adds (a float in [2^23, 2^24) has unit spacing, so adding
// 2^23 rounds to an integer that its low mantissa bits hold): float-to-64-bit
// conversions run on a slow unit, these adds on the fast one.
__device__ __forceinline__ long long to_fix(float w) {
  const float t = w * 1048576.0f;                      // w 2^20, exact, in [0, 2^20]
  const float h = __fadd_rd(t, 8388608.0f);            // 2^23 + floor(t)
  const float r = (t - (h - 8388608.0f)) * 1048576.0f;  // frac(t) 2^20, exact, in [0, 2^20)
  const float l = __fadd_rn(r, 8388608.0f);            // 2^23 + rint(r)
  return ((long long)(__float_as_int(h) - 0x4B000000) << 20) + (__float_as_int(l) - 0x4B000000);
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
// Group g (elements 8 g .. 8 g + 7) of a span of n elements, from global memory (GLOBAL) or
// shared memory; elements past n read as -inf.
template <typename T, bool VEC, bool GLOBAL>
__device__ __forceinline__ void group8(const T *row, int g, int n, float (&x)[kGroup]) {
  const int e = g * kGroup;
  auto ld16 = [](const void *q) -> uint4 {
    return GLOBAL ? __ldg(reinterpret_cast<const uint4 *>(q)) : *reinterpret_cast<const uint4 *>(q);
  };
  if (VEC && e + kGroup <= n) {  // 16-byte aligned: the span starts at a multiple of 8 elements
    if constexpr (sizeof(T) == 2) {
      const uint4 r = ld16(row + e);
      const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        x[2 * k] = __uint_as_float(w[k] << 16);
        x[2 * k + 1] = __uint_as_float(w[k] & 0xffff0000u);
      }
    } else {
      const uint4 r0 = ld16(row + e), r1 = ld16(row + e + 4);
      x[0] = __uint_as_float(r0.x), x[1] = __uint_as_float(r0.y), x[2] = __uint_as_float(r0.z);
      x[3] = __uint_as_float(r0.w), x[4] = __uint_as_float(r1.x), x[5] = __uint_as_float(r1.y);
      x[6] = __uint_as_float(r1.z), x[7] = __uint_as_float(r1.w);
    }
  } else {  // the chunk's ragged end (elements past it read as -inf), or rows without alignment
#pragma unroll
    for (int k = 0; k < kGroup; ++k) x[k] = e + k < n ? to_f32(row[e + k]) : -INFINITY;
  }
}


// ===========================================================================
// Row statistics: every target row (and, for T > 0, every draft row) cut into
// items of 32 KB, the items of the launch cut into contiguous ranges that
// differ by one item at most, one per CTA. A producer warp streams a CTA's items through a 3-stage ring of
// 1-D bulk copies; eight consumer warps each reduce an eighth of every item.
// A lane keeps a running (max, sum of 2^(x c - max c)) or argmax of the
// current row; where a warp's run of items leaves a row the warp reduces it and
// writes it as the partial of (the run's first item, warp); every other
// (item, warp) partial is written as the identity, so each launch writes all
// of them and nothing needs to start at zero.
// ===========================================================================
struct StatsArgs {
  const void *tgt, *drf;
  float *pm, *ps;  // [items][kStatWarps]: max (or best value), sum (or best index bits)
  int32_t *status;
  int vocab, total_q, rows, nchunk, items, per, extra;  // CTA c: per items, one more when c < extra
  float coef;
  unsigned long long wait_ns;  // budget of the pipeline waits
  int stall;                   // SV_STALL_SAMPLER: the producer waits on nothing (failure-path test)
};

template <typename T, bool VEC, int MODE>
__global__ void __launch_bounds__(kStatThreads) stats_kernel(const StatsArgs A) {
  // This kernel reads only the call's logits, which no kernel of the library writes: it streams
  // them without waiting for the kernel before it (the end of the attention call), and waits
  // only before its first write to global memory, which goes to a workspace another call may
  // share. Its partials wait in shared memory until then (kMaxRuns runs; more are written after
  // an early wait).
  grid_dependents_launch();
  constexpr int CH = kPartBytes / (int)sizeof(T);  // elements of an item
  constexpr int SL = CH / kStatWarps;              // elements of a warp's slice
  extern __shared__ __align__(128) uint8_t ring[];  // kStatStages x kPartBytes
  __shared__ uint64_t full[kStatStages], empty[kStatStages];
  __shared__ uint64_t stall_bar;  // failure-path test: a barrier nothing arrives on
  __shared__ float2 runbuf[kMaxRuns][kStatWarps];  // consumers: each run's per-warp statistics
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i0 = blockIdx.x * A.per + min((int)blockIdx.x, A.extra);
  const int i1 = min(A.items, i0 + A.per + ((int)blockIdx.x < A.extra ? 1 : 0));
  const int V = A.vocab;
  const T *tgt = reinterpret_cast<const T *>(A.tgt);
  const T *drf = reinterpret_cast<const T *>(A.drf);
  auto row_ptr = [&](int r) -> const T * {
    return r < A.total_q ? tgt + (size_t)r * V : drf + (size_t)(r - A.total_q) * V;
  };
  if (tid == 0) {
    for (int s = 0; s < kStatStages; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&full[s])) : "memory");
      asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(&empty[s])), "r"(kStatWarps)
                   : "memory");
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&stall_bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  bool ok = true;
  int issued = 0;  // producer: items whose copies were issued

  if (warp == kStatWarps) {
    // ---------------- producer ----------------
    if (VEC && lane == 0) {
      if (A.stall == SV_STALL_SAMPLER) ok = wait_on_nothing(smem_addr(&stall_bar), A.wait_ns);
      for (int it = i0, j = 0; ok && it < i1; ++it, ++j) {
        const int s = j % kStatStages;
        // a stage is refilled only after all eight consumer warps read its last item (they stop
        // arriving once one of their waits gave up, so nothing is copied over a stage in flight)
        if (j >= kStatStages && !mbar_wait_bounded(smem_addr(&empty[s]), ((j / kStatStages) - 1) & 1, A.wait_ns)) {
          ok = false;
          break;
        }
        const int r = it / A.nchunk, k = it - r * A.nchunk;
        const int e0 = k * CH, cnt = min(CH, V - e0);
        const uint32_t bytes = static_cast<uint32_t>(cnt * sizeof(T));
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&full[s])), "r"(bytes)
                     : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         smem_addr(ring + s * kPartBytes)),
                     "l"(row_ptr(r) + e0), "r"(bytes), "r"(smem_addr(&full[s]))
                     : "memory");
        ++issued;
      }
    }
    grid_dependency_wait();
  } else {
    // ---------------- consumers: warp w reduces elements [w SL, (w + 1) SL) of each item ----------------
    int bad = 0;
    float lm = -INFINITY, ls = 0.f;  // stochastic: running max, sum of 2^(x c - lm c)
    float lb = 0.f;                  // greedy: best value and index
    int lbi = -1;
    int cur_row = -1, run_start = -1, nrun = 0;
    bool waited = false;
    auto wait_once = [&]() {
      if (!waited) grid_dependency_wait();
      waited = true;
    };
    // the run's (max, sum) or (value, index bits) for item run_start: kept in shared memory, or
    // (past kMaxRuns runs) written after the wait
    auto put = [&](float a, float b) {
      if (nrun < kMaxRuns) {
        runbuf[nrun][warp] = make_float2(a, b);
      } else {
        wait_once();
        A.pm[(size_t)run_start * kStatWarps + warp] = a;
        A.ps[(size_t)run_start * kStatWarps + warp] = b;
      }
    };
    auto flush = [&]() {  // warp-uniform: the run's statistics into (run_start, warp)
      if constexpr (MODE == kStochastic) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float m2 = __shfl_xor_sync(0xffffffffu, lm, o);
          const float s2 = __shfl_xor_sync(0xffffffffu, ls, o);
          ms_combine(lm, ls, m2, s2, A.coef);
        }
        if (lane == 0) put(lm, ls);
        lm = -INFINITY;
        ls = 0.f;
      } else {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float v2 = __shfl_xor_sync(0xffffffffu, lb, o);
          const int i2 = __shfl_xor_sync(0xffffffffu, lbi, o);
          am_combine(lb, lbi, v2, i2);
        }
        if (lane == 0) put(lb, __int_as_float(lbi));
        lb = 0.f;
        lbi = -1;
      }
      ++nrun;
    };
    for (int it = i0, j = 0; it < i1; ++it, ++j) {
      const int s = j % kStatStages;
      const int r = it / A.nchunk, k = it - r * A.nchunk;
      const int e0 = k * CH, cnt = min(CH, V - e0);
      if (r != cur_row) {
        if (cur_row >= 0) flush();
        cur_row = r;
        run_start = it;
      }
      const T *src;
      if constexpr (VEC) {
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_addr(&full[s]), (j / kStatStages) & 1, A.wait_ns));
        src = reinterpret_cast<const T *>(ring + s * kPartBytes);
      } else {
        src = row_ptr(r) + e0;  // rows not 16-byte aligned: scalar loads straight from memory
      }
      // this lane's elements: groups of 8 at slice offset 8 * (lane + 32 u); -inf past the item
      const int s0 = warp * SL;
      if (ok && s0 < cnt) {
        if constexpr (VEC && sizeof(T) == 2 && MODE == kStochastic) {
          // bf16 pairs: the maximum on packed pairs (NaN-propagating), the sum on floats
          uint32_t w[SL / 64];
#pragma unroll
          for (int u = 0; u < SL / 256; ++u) {
            const int e = s0 + 8 * (lane + 32 * u);
            const uint4 q = *reinterpret_cast<const uint4 *>(src + e);
            w[4 * u] = q.x;
            w[4 * u + 1] = q.y;
            w[4 * u + 2] = q.z;
            w[4 * u + 3] = q.w;
            if (e + 8 > cnt) {
#pragma unroll
              for (int p = 0; p < 4; ++p) {
                if (e + 2 * p >= cnt) w[4 * u + p] = (w[4 * u + p] & 0xffff0000u) | 0xff80u;
                if (e + 2 * p + 1 >= cnt) w[4 * u + p] = (w[4 * u + p] & 0xffffu) | 0xff800000u;
              }
            }
          }
          __nv_bfloat162 m2 = __halves2bfloat162(__ushort_as_bfloat16(0xff80), __ushort_as_bfloat16(0xff80));
#pragma unroll
          for (int q = 0; q < SL / 64; ++q) m2 = __hmax2_nan(m2, *reinterpret_cast<const __nv_bfloat162 *>(&w[q]));
          const float ma = __low2float(m2), mb = __high2float(m2);
          const float mi = (ma != ma || mb != mb) ? NAN : fmaxf(ma, mb);
          bad |= (mi != mi) | (mi == INFINITY);
          if (mi == mi && mi != -INFINITY) {
            if (mi > lm) {
              ls = (lm == -INFINITY) ? 0.f : ls * fast_exp2((lm - mi) * A.coef);
              lm = mi;
            }
            const float nmc = -lm * A.coef;
            float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
            for (int q = 0; q < SL / 64; ++q) {
              acc0 += fast_exp2(fmaf(__uint_as_float(w[q] << 16), A.coef, nmc));
              acc1 += fast_exp2(fmaf(__uint_as_float(w[q] & 0xffff0000u), A.coef, nmc));
            }
            ls += acc0 + acc1;
          }
        } else if constexpr (VEC && sizeof(T) == 2) {
          // argmax on bf16 pairs: a group of 8 is looked into only when its packed
          // maximum beats the lane's best (ties keep the lower index seen first)
#pragma unroll
          for (int u = 0; u < SL / 256; ++u) {
            const int e = s0 + 8 * (lane + 32 * u);
            const uint4 q = *reinterpret_cast<const uint4 *>(src + e);
            uint32_t w[4] = {q.x, q.y, q.z, q.w};
            if (e + 8 > cnt) {
#pragma unroll
              for (int p = 0; p < 4; ++p) {
                if (e + 2 * p >= cnt) w[p] = (w[p] & 0xffff0000u) | 0xff80u;
                if (e + 2 * p + 1 >= cnt) w[p] = (w[p] & 0xffffu) | 0xff800000u;
              }
            }
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(w);
            const __nv_bfloat162 m2 = __hmax2_nan(__hmax2_nan(h[0], h[1]), __hmax2_nan(h[2], h[3]));
            const float ga = __low2float(m2), gb = __high2float(m2);
            if (ga != ga || gb != gb) {
              bad = 1;
            } else if (e < cnt) {
              const float gm = fmaxf(ga, gb);
              if (lbi < 0 || gm > lb) {
                int p = 0;
                for (; p < 7; ++p) {
                  const uint32_t wp = w[p >> 1];
                  if (__uint_as_float((p & 1) ? (wp & 0xffff0000u) : (wp << 16)) == gm) break;
                }
                lb = gm;
                lbi = e0 + e + p;
              }
            }
          }
        } else {
        float x[SL / 32];
#pragma unroll
        for (int u = 0; u < SL / 256; ++u) {
          const int e = s0 + 8 * (lane + 32 * u);
          if constexpr (VEC && sizeof(T) == 2) {
            const uint4 q = *reinterpret_cast<const uint4 *>(src + e);
            const uint32_t *w = reinterpret_cast<const uint32_t *>(&q);
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              x[8 * u + 2 * p] = __uint_as_float(w[p] << 16);
              x[8 * u + 2 * p + 1] = __uint_as_float(w[p] & 0xffff0000u);
            }
          } else if constexpr (VEC) {
            const uint4 q0 = *reinterpret_cast<const uint4 *>(src + e);
            const uint4 q1 = *reinterpret_cast<const uint4 *>(src + e + 4);
            const float *f0 = reinterpret_cast<const float *>(&q0), *f1 = reinterpret_cast<const float *>(&q1);
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              x[8 * u + p] = f0[p];
              x[8 * u + 4 + p] = f1[p];
            }
          } else {
#pragma unroll
            for (int p = 0; p < 8; ++p) x[8 * u + p] = (e + p < cnt) ? to_f32(src[e + p]) : -INFINITY;
          }
          if (e + 8 > cnt) {
#pragma unroll
            for (int p = 0; p < 8; ++p)
              if (e + p >= cnt) x[8 * u + p] = -INFINITY;
          }
        }
        if constexpr (MODE == kStochastic) {
          float mi = -INFINITY;
#pragma unroll
          for (int q = 0; q < SL / 32; ++q) mi = (x[q] != x[q] || mi != mi) ? NAN : fmaxf(mi, x[q]);
          bad |= (mi != mi) | (mi == INFINITY);
          if (mi == mi && mi != -INFINITY) {
            if (mi > lm) {
              ls = (lm == -INFINITY) ? 0.f : ls * fast_exp2((lm - mi) * A.coef);
              lm = mi;
            }
            const float nmc = -lm * A.coef;
            float acc = 0.f;
#pragma unroll
            for (int q = 0; q < SL / 32; ++q) acc += fast_exp2(fmaf(x[q], A.coef, nmc));
            ls += acc;
          }
        } else {
#pragma unroll
          for (int u = 0; u < SL / 256; ++u) {
            const int e = s0 + 8 * (lane + 32 * u);
#pragma unroll
            for (int p = 0; p < 8; ++p) {
              const float v = x[8 * u + p];
              bad |= (v != v);
              if (e + p < cnt) am_combine(lb, lbi, v, e0 + e + p);
            }
          }
        }
        }
      }
      if constexpr (VEC) {
        __syncwarp();
        if (lane == 0 && ok)
          asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(&empty[s])) : "memory");
      }
    }
    if (cur_row >= 0) flush();
    // the writes: each run's first item gets the run's statistics (those kept here), every other
    // item the identity
    wait_once();
    if (lane == 0) {
      int run = -1, prev = -1;
      for (int it = i0; it < i1; ++it) {
        const int r = it / A.nchunk;
        const size_t at = (size_t)it * kStatWarps + warp;
        if (r != prev) {
          prev = r;
          if (++run < kMaxRuns) {
            A.pm[at] = runbuf[run][warp].x;
            A.ps[at] = runbuf[run][warp].y;
          }
        } else {
          A.pm[at] = (MODE == kStochastic) ? -INFINITY : 0.f;
          A.ps[at] = (MODE == kStochastic) ? 0.f : __int_as_float(-1);
        }
      }
    }
    if (bad) record(A.status, SV_ERR_NONFINITE);
    if (!ok) record(A.status, SV_ERR_TIMEOUT);
  }
  // after a failed wait, let the producer's copies in flight land before shared memory is released:
  // a copy older than the last kStatStages issued was read by every consumer before its stage
  // was refilled, so only those can still be in flight
  const bool any_fail = __syncthreads_or(!ok);
  if (VEC && any_fail && tid == kStatWarps * 32) {
    for (int j = max(0, issued - kStatStages); j < issued; ++j)
      mbar_wait_bounded(smem_addr(&full[j % kStatStages]), (j / kStatStages) & 1, kDrainBudgetNs);
  }
}


// ===========================================================================
// Decisions: one cluster per sequence (C CTAs for T > 0, one CTA for greedy
// and tree). Every CTA combines its sequence's row partials in the same fixed
// order (one warp per row), so all CTAs hold identical row statistics and take
// identical decisions; for T > 0 the draw runs over the C vocabulary chunks.
// ===========================================================================
struct Smem {
  float M[kMaxRows];  // per row, whole vocabulary
  float Z[kMaxRows];
  int am[kMaxRows];
  float gtl[kMaxQ], gdl[kMaxQ];  // target and draft logits of the draft tokens
  float uacc[kMaxQ];             // accept uniforms
  int tok[kMaxQ];                // draft tokens (chain) or node tokens (tree)
  int par[kMaxQ];                // tree: parent row of each row
  int path[kMaxQ];               // tree at T > 0: rows of the accepted nodes
  int excl[kMaxQ];               // tree at T > 0: tokens rejected at the final node
  int nexcl;
  int cur;                       // tree at T > 0: the final node's row
  uint64_t sub_full[kMaxSubStages];  // phase 3: ring of row-pair sub-chunks
  long long S[2];    // phase 3: this CTA's fixed-point weight sum per pass (cluster-visible)
  long long ll_buf[kWarps];
  long long P_owner, target;
  float rho_hi, rho_lo;
  float m1, m2;       // margins: of the accept tests, and of the draw's CDF crossing
  long long Stot;     // the draw's total fixed-point mass
  int a;
  int owner, fallback;
  int y_hit, y_last;
};

// UG: groups of a mass unit (1, or 2 with the half ring of 4-CTA clusters)
template <typename T, bool VEC, int MODE, int UG>
__global__ void __launch_bounds__(kThreads) decide_kernel(SamplerArgs args, const float *__restrict__ pm,
                                                          const float *__restrict__ ps, int nchunk) {
  cg::cluster_group cluster = cg::this_cluster();
  const int C = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int b = blockIdx.y;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  __shared__ Smem sm;
  extern __shared__ __align__(128) uint8_t dyn[];
  // phase 3: a ring of sub-chunk stages (target, then draft: kSub elements each), then the
  // per-unit masses
  static_assert(UG == 1 || UG == 2, "one or two groups a mass unit");
  constexpr int kRing = kRingBytes / UG;
  constexpr int kSubStages = kRing / (2 * kSub * (int)sizeof(T));  // bf16: 4 or 2, fp32: 2 or 1
  static_assert(kSubStages >= 1 && kSubStages <= kMaxSubStages, "sub-chunk stages");
  constexpr int ug = UG;
  uint8_t *sring = dyn;
  long long *gmass = reinterpret_cast<long long *>(dyn + kRing);

  // Before the grid-dependency wait this kernel reads only the call's own inputs (cu_q, draft
  // tokens, uniforms, parents and logits), which no kernel of the library writes, so their
  // latency overlaps the statistics kernel's tail. The status word, the partials and every
  // output are touched only after the wait.
  const int V = args.vocab;
  const int t0 = args.cu_q[b];
  const int n = args.cu_q[b + 1] - t0;
  const int K = n - 1;
  const int d0 = t0 - b;
  const int lo = min(V, rank * args.chunk), hi = min(V, lo + args.chunk);
  const int len = hi - lo;
  constexpr bool STOCH = MODE == kStochastic || MODE == kTreeStochastic;  // (max, sum) statistics
  const int rows = (MODE == kStochastic) ? n + K : n;
  const T *tgt = reinterpret_cast<const T *>(args.tgt);
  const T *drf = reinterpret_cast<const T *>(args.drf);
  const float coef = args.coef;
  // rows outside [0, total_q) or more than max_q rows: nothing is read or written
  const bool valid = !(n < 1 || n > args.max_q || t0 < 0 || t0 + n > args.total_q);
  bool bad_token = false;
  if (valid) {
    if (tid == 0) {
      for (int st = 0; st < kSubStages; ++st)
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_addr(&sm.sub_full[st])) : "memory");
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    // the sequence's small inputs into shared memory, so the serial scans below read no global memory
    if (tid < K) sm.tok[tid] = args.draft_tok[d0 + tid];
    if ((MODE == kTree || MODE == kTreeStochastic) && tid < n) sm.par[tid] = args.parent[t0 + tid];
    if constexpr (MODE == kTreeStochastic) {
      if (tid < K) {  // node tid + 1: its accept uniform and its token's target logit in its parent's row
        sm.uacc[tid] = args.u_acc[d0 + tid];
        const int x = args.draft_tok[d0 + tid], pr = args.parent[t0 + tid + 1];
        sm.gtl[tid] = 0.f;
        if (x < 0 || x >= V) {
          bad_token = true;
        } else if (pr >= 0 && pr < n) {
          sm.gtl[tid] = to_f32(tgt[(size_t)(t0 + pr) * V + x]);
        }
      }
    }
    if constexpr (MODE == kStochastic) {
      if (tid < K) {  // the accept uniform and the target and draft logits of each draft token
        sm.uacc[tid] = args.u_acc[d0 + tid];
        const int x = args.draft_tok[d0 + tid];
        if (x < 0 || x >= V) {
          bad_token = true;
          sm.gtl[tid] = 0.f;
          sm.gdl[tid] = 0.f;
        } else {
          sm.gtl[tid] = to_f32(tgt[(size_t)(t0 + tid) * V + x]);
          sm.gdl[tid] = to_f32(drf[(size_t)(d0 + tid) * V + x]);
        }
      }
    }
  }
  grid_dependency_wait();  // the statistics kernel is complete and its partials visible
  grid_dependents_launch();
  // Every CTA of the cluster takes this exit together (same b), before any barrier.
  if (!valid) {
    if (rank == 0 && tid == 0) record(args.status, SV_ERR_BAD_LENGTH);
    return;
  }
  if (bad_token && rank == 0) record(args.status, SV_ERR_BAD_TOKEN);
  bool ok = true;  // false after a bounded wait gave up: the remaining work is skipped, barriers are kept

  // ---------------- row statistics from the partials: one warp per row ----------------
  const int np = nchunk * kStatWarps;
  if constexpr (STOCH) {
    // four rows per warp at a time, every load of them in flight before any is used
    constexpr int kRB = 4;
    for (int r0 = warp; r0 < rows; r0 += kRB * kWarps) {
      size_t p0[kRB];
#pragma unroll
      for (int h = 0; h < kRB; ++h) {
        const int r = r0 + h * kWarps;
        const int gr = r < n ? t0 + r : args.total_q + d0 + (r - n);  // row of the statistics kernel
        p0[h] = (size_t)gr * np;
      }
      float m[kRB], sum[kRB];
#pragma unroll
      for (int h = 0; h < kRB; ++h) {
        m[h] = -INFINITY;
        sum[h] = 0.f;
      }
      for (int q0 = 0; q0 < np; q0 += 64) {  // two loads of each array per row in flight per lane
        float lm[kRB][2], lsum[kRB][2];
#pragma unroll
        for (int h = 0; h < kRB; ++h)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int q = q0 + 32 * j + lane;
            const bool in = q < np && r0 + h * kWarps < rows;
            lm[h][j] = in ? pm[p0[h] + q] : -INFINITY;
            lsum[h][j] = in ? ps[p0[h] + q] : 0.f;
          }
#pragma unroll
        for (int h = 0; h < kRB; ++h)
#pragma unroll
          for (int j = 0; j < 2; ++j) ms_combine(m[h], sum[h], lm[h][j], lsum[h][j], coef);
      }
#pragma unroll
      for (int h = 0; h < kRB; ++h) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float m2 = __shfl_xor_sync(0xffffffffu, m[h], o);
          const float s2 = __shfl_xor_sync(0xffffffffu, sum[h], o);
          ms_combine(m[h], sum[h], m2, s2, coef);
        }
        const int r = r0 + h * kWarps;
        if (lane == 0 && r < rows) {
          sm.M[r] = m[h];
          sm.Z[r] = sum[h];
        }
      }
    }
  } else {
    // argmax rows, four per warp at a time (tree rows are many), every load in flight first
    constexpr int kRB = 4;
    for (int r0 = warp; r0 < rows; r0 += kRB * kWarps) {
      size_t p0[kRB];
#pragma unroll
      for (int h = 0; h < kRB; ++h) p0[h] = (size_t)(t0 + r0 + h * kWarps) * np;  // rows < n: target rows
      float best[kRB];
      int bi[kRB];
#pragma unroll
      for (int h = 0; h < kRB; ++h) {
        best[h] = 0.f;
        bi[h] = -1;
      }
      for (int q0 = 0; q0 < np; q0 += 64) {  // two loads of each array per row in flight per lane
        float lv[kRB][2];
        int li[kRB][2];
#pragma unroll
        for (int h = 0; h < kRB; ++h)
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const int q = q0 + 32 * j + lane;
            const bool in = q < np && r0 + h * kWarps < rows;
            lv[h][j] = in ? pm[p0[h] + q] : 0.f;
            li[h][j] = in ? __float_as_int(ps[p0[h] + q]) : -1;
          }
#pragma unroll
        for (int h = 0; h < kRB; ++h)
#pragma unroll
          for (int j = 0; j < 2; ++j) am_combine(best[h], bi[h], lv[h][j], li[h][j]);
      }
#pragma unroll
      for (int h = 0; h < kRB; ++h) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float v2 = __shfl_xor_sync(0xffffffffu, best[h], o);
          const int i2 = __shfl_xor_sync(0xffffffffu, bi[h], o);
          am_combine(best[h], bi[h], v2, i2);
        }
        const int r = r0 + h * kWarps;
        if (lane == 0 && r < rows) sm.am[r] = bi[h];
      }
    }
  }
  __syncthreads();

  if constexpr (MODE == kGreedy) {
    if (rank == 0 && tid == 0) {
      int a = K;
      for (int i = 0; i < K; ++i)
        if (sm.tok[i] != sm.am[i]) {
          a = i;
          break;
        }
      int32_t *o = args.out_tok + (size_t)b * args.max_q;
      for (int j = 0; j < args.max_q; ++j) o[j] = j < a ? sm.tok[j] : -1;
      o[a] = sm.am[a];
      args.accept[b] = a;
      args.num_out[b] = a + 1;
      if (args.margin) args.margin[b] = INFINITY;
    }
  } else if constexpr (MODE == kTree) {
    // the walk with one warp: at each node the lanes look for the first child (in row
    // order) whose token is the node's argmax
    if (rank == 0 && warp == 0) {
      int32_t *o = args.out_tok + (size_t)b * args.max_q;
      int32_t *path = args.path + (size_t)b * args.max_q;
      for (int j = lane; j < args.max_q; j += 32) {
        o[j] = -1;
        path[j] = -1;
      }
      bool g_l = true;
      for (int j = 1 + lane; j < n; j += 32) {
        const int p = sm.par[j];
        g_l &= (p >= 0 && p < n && p != j);
      }
      const bool good = __all_sync(0xffffffffu, g_l);
      if (!good && lane == 0) record(args.status, SV_ERR_BAD_LENGTH);
      __syncwarp();  // the -1 fill lands before the path entries below
      int cur = 0, a = 0;
      while (good && a < n - 1) {
        const int am = sm.am[cur];
        int next = -1;
        for (int j0 = 1; j0 < n && next < 0; j0 += 32) {
          const int j = j0 + lane;
          const unsigned m = __ballot_sync(0xffffffffu, j < n && sm.par[j] == cur && sm.tok[j - 1] == am);
          if (m) next = j0 + __ffs(m) - 1;
        }
        if (next < 0) break;
        if (lane == 0) {
          path[a] = next;
          o[a] = am;
        }
        ++a;
        cur = next;
      }
      if (lane == 0) {
        o[a] = sm.am[cur];
        args.accept[b] = a;
        args.num_out[b] = a + 1;
        if (args.margin) args.margin[b] = INFINITY;
      }
    }
  } else {
    if constexpr (MODE == kTreeStochastic) {
      // ---------------- the tree walk (identical in every CTA, one warp) ----------------
      // at the current node, children in row order: child x is accepted iff u < p'(x), p'
      // the node's p without the tokens of the siblings rejected before, renormalised. The
      // lanes find the node's children and their p(x) (a child whose token an earlier
      // sibling had weighs 0: that sibling was rejected); lane order then adds the rejected
      // mass one child at a time, as a single thread would.
      if (warp == 0) {
        bool g_l = true, nz_l = false;
        for (int j = 1 + lane; j < n; j += 32) g_l &= sm.par[j] >= 0 && sm.par[j] < j;
        for (int r = lane; r < n; r += 32) nz_l |= !(sm.Z[r] > 0.f);
        const bool good = __all_sync(0xffffffffu, g_l);
        if (__any_sync(0xffffffffu, nz_l) && rank == 0 && lane == 0) record(args.status, SV_ERR_NONFINITE);
        if (!good && rank == 0 && lane == 0) record(args.status, SV_ERR_BAD_LENGTH);
        int cur = 0, a = 0;
        float mmin = INFINITY;  // the accept tests' margin
        bool moved = good;
        while (moved) {  // one node per pass; children of cur lie after cur (checked above)
          moved = false;
          float removed = 0.f;
          for (int j0 = cur + 1; j0 < n && !moved; j0 += 32) {
            const int j = j0 + lane;
            const bool child = j < n && sm.par[j] == cur;
            unsigned m = __ballot_sync(0xffffffffu, child);
            float px = 0.f;
            if (child) {
              const int x = sm.tok[j - 1];
              bool dup = false;
              for (int k = cur + 1; k < j; ++k) dup |= sm.par[k] == cur && sm.tok[k - 1] == x;
              px = dup ? 0.f : exp2f((sm.gtl[j - 1] - sm.M[cur]) * coef) / sm.Z[cur];
            }
            while (m) {  // warp-uniform: the children of this chunk in row order
              const int k = __ffs(m) - 1;
              m &= m - 1;
              const float pk = __shfl_sync(0xffffffffu, px, k);
              const float thr = removed < 1.f ? pk / (1.f - removed) : 0.f;
              mmin = fminf(mmin, fabsf(sm.uacc[j0 + k - 1] - thr));
              if (sm.uacc[j0 + k - 1] < thr) {  // accepted: the walk goes on from this child
                if (lane == 0) sm.path[a] = j0 + k;
                ++a;
                cur = j0 + k;
                moved = true;
                break;
              }
              removed += pk;
            }
          }
        }
        // the final node's children were all rejected: their distinct tokens, in row order
        int nexcl = 0;
        for (int j0 = cur + 1; good && j0 < n; j0 += 32) {
          const int j = j0 + lane;
          bool keep = j < n && sm.par[j] == cur;
          if (keep) {
            const int x = sm.tok[j - 1];
            for (int k = cur + 1; k < j; ++k) keep &= !(sm.par[k] == cur && sm.tok[k - 1] == x);
          }
          const unsigned m = __ballot_sync(0xffffffffu, keep);
          if (keep) sm.excl[nexcl + __popc(m & ((1u << lane) - 1u))] = sm.tok[j - 1];
          nexcl += __popc(m);
        }
        if (lane == 0) {
          sm.a = a;
          sm.cur = cur;
          sm.nexcl = nexcl;
          sm.m1 = mmin;
        }
      }
    } else {
    // ---------------- accept scan (identical in every CTA): one lane per draft, first rejection by ballot ----------------
    if (warp == 0) {
      unsigned rej[2];
      float dist[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int i = lane + 32 * h;
        bool r = false;
        dist[h] = INFINITY;
        if (i < K) {
          const float p = exp2f((sm.gtl[i] - sm.M[i]) * coef) / sm.Z[i];
          const float q = exp2f((sm.gdl[i] - sm.M[n + i]) * coef) / sm.Z[n + i];
          const float thr = q > 0.f ? fminf(1.f, p / q) : 1.f;
          r = !(sm.uacc[i] < thr);
          dist[h] = fabsf(sm.uacc[i] - thr);
        }
        rej[h] = __ballot_sync(0xffffffffu, r);
      }
      {  // the accept tests' margin: the drafts up to the first rejection
        const int a_all = rej[0] ? __ffs(rej[0]) - 1 : rej[1] ? 31 + __ffs(rej[1]) : K;
        float m = fminf(lane <= a_all ? dist[0] : INFINITY, lane + 32 <= a_all ? dist[1] : INFINITY);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fminf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) sm.m1 = m;
      }
      bool nz = false;
      for (int r = lane; r < rows; r += 32) nz |= !(sm.Z[r] > 0.f);
      const bool bad = __any_sync(0xffffffffu, nz);
      if (lane == 0) {
        const int a = rej[0] ? __ffs(rej[0]) - 1 : rej[1] ? 31 + __ffs(rej[1]) : K;
        sm.a = a;
        if (bad && rank == 0) record(args.status, SV_ERR_NONFINITE);
        // a residual draw weighs q_v as e_d (Z_t / Z_d) against e_t, the ratio carried as hi + lo
        const double rho = a < K && sm.Z[n + a] > 0.f ? (double)sm.Z[a] / (double)sm.Z[n + a] : 0.0;
        sm.rho_hi = (float)rho;
        sm.rho_lo = (float)(rho - (double)sm.rho_hi);
      }
    }
    }
    __syncthreads();
    const int a = sm.a;
    // the row of the draw: the first rejected position (chain) or the walk's last node (tree)
    const int dr = MODE == kTreeStochastic ? sm.cur : a;
    const bool resid = MODE == kStochastic && a < K;         // residual max(0, p - q) of a chain
    const int nexcl = MODE == kTreeStochastic ? sm.nexcl : 0;  // tokens left out of p (tree)
    const T *trow = tgt + (size_t)(t0 + dr) * V;
    const T *drow = resid ? drf + (size_t)(d0 + a) * V : nullptr;
    const float Mt = sm.M[dr], Md = resid ? sm.M[n + a] : 0.f;
    const float chi = args.coef, clo = args.coef_lo;
    const float ur = args.u_res[b];
    // this CTA's chunk of the row (pair) of the draw
    const T *bt = trow + lo;
    const T *bd = resid ? drow + lo : nullptr;
    const int ngroups = (len + kGroup - 1) / kGroup;
    const int nsub = (len + kSub - 1) / kSub;
    const uint32_t sub_bytes = kSub * sizeof(T);
    int subs_done = 0;  // sub-chunks consumed so far (over both passes): ring stage and phase

    const float rho_hi = sm.rho_hi, rho_lo = sm.rho_lo;

    for (int pass = 0; pass < 2; ++pass) {
      const bool res_pass = resid && pass == 0;
      const bool excl_pass = nexcl > 0 && pass == 0;
      // the eight weights of group g, in [0, 1]: proportional to max(0, p_v - q_v)
      // (scaled by Z_t), or to p_v
      auto weights_of = [&](int g, const float (&xt)[kGroup], const float (&xd)[kGroup], float (&w)[kGroup]) {
        if (res_pass) {
#pragma unroll
          for (int k = 0; k < kGroup; ++k) {
            const float et = exp2_acc(xt[k] - Mt, chi, clo);
            const float ed = exp2_acc(xd[k] - Md, chi, clo);
            w[k] = fmaxf(et - fmaf(ed, rho_hi, ed * rho_lo), 0.f);
          }
        } else {
#pragma unroll
          for (int k = 0; k < kGroup; ++k) w[k] = exp2_acc(xt[k] - Mt, chi, clo);
          if (excl_pass) {  // the rejected children's tokens carry no mass
            const int v0 = lo + g * kGroup;
            for (int e = 0; e < nexcl; ++e) {
              const int d = sm.excl[e] - v0;
              if (d >= 0 && d < kGroup) w[d] = 0.f;
            }
          }
        }
      };
      // ... read from global memory (the owner's one group)
      // ... for the owner's one group: from the ring while the whole chunk stays in it (no stage
      // was refilled), else from global memory
      const int pass_base = subs_done;
      auto weightsf8 = [&](int g, float (&w)[kGroup]) {
        float xt[kGroup], xd[kGroup];
        if (VEC && nsub <= kSubStages) {
          const int i = g / (kSub / kGroup), gl = g - i * (kSub / kGroup);
          const int n_i = min(kSub, len - i * kSub);
          const uint8_t *stage = sring + ((pass_base + i) % kSubStages) * 2 * sub_bytes;
          group8<T, true, false>(reinterpret_cast<const T *>(stage), gl, n_i, xt);
          if (res_pass) group8<T, true, false>(reinterpret_cast<const T *>(stage + sub_bytes), gl, n_i, xd);
        } else {
          group8<T, VEC, true>(bt, g, len, xt);
          if (res_pass) group8<T, VEC, true>(bd, g, len, xd);
        }
        weights_of(g, xt, xd, w);
      };
      // ... as fixed point, one by one
      auto weights8 = [&](int g, long long (&w)[kGroup]) {
        float f[kGroup];
        weightsf8(g, f);
#pragma unroll
        for (int k = 0; k < kGroup; ++k) w[k] = to_fix(f[k]);
      };
      // ... and their fixed-point sum, equal to the sum of the values above: the 20-bit
      // halves of to_fix summed as float bit patterns (2^23 + integer, eight of them:
      // no carry leaves 32 bits), the offsets taken off once
      auto mass8 = [&](int g, const float (&xt)[kGroup], const float (&xd)[kGroup]) -> long long {
        float f[kGroup];
        weights_of(g, xt, xd, f);
        uint32_t sh = 0u, sl = 0u;
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
          const float t = f[k] * 1048576.0f;
          const float h = __fadd_rd(t, 8388608.0f);
          const float r = (t - (h - 8388608.0f)) * 1048576.0f;
          const float l = __fadd_rn(r, 8388608.0f);
          sh += __float_as_uint(h);
          sl += __float_as_uint(l);
        }
        sh -= static_cast<uint32_t>(kGroup) * 0x4B000000u;
        sl -= static_cast<uint32_t>(kGroup) * 0x4B000000u;
        return (static_cast<long long>(sh) << 20) + static_cast<long long>(sl);
      };
      // ---- pass B: each group's mass and this CTA's total. The chunk streams through the
      // ring in sub-chunks of kSub elements (two groups a thread): thread 0 keeps kSubStages of
      // them in flight with bulk copies, refilling a stage once every thread has read it ----
      auto issue_sub = [&](int i) {  // sub-chunk i of this pass into its stage (thread 0, VEC)
        const int st = (subs_done + i) % kSubStages;
        const int e0 = i * kSub;
        const uint32_t bytes = static_cast<uint32_t>(min(kSub, len - e0)) * sizeof(T);
        uint8_t *dst = sring + st * 2 * sub_bytes;
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the stage's earlier reads are done
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&sm.sub_full[st])),
                     "r"(res_pass ? 2 * bytes : bytes)
                     : "memory");
        asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                         smem_addr(dst)),
                     "l"(bt + e0), "r"(bytes), "r"(smem_addr(&sm.sub_full[st]))
                     : "memory");
        if (res_pass)
          asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                           smem_addr(dst + sub_bytes)),
                       "l"(bd + e0), "r"(bytes), "r"(smem_addr(&sm.sub_full[st]))
                       : "memory");
      };
      if (ok && VEC && tid == 0)
        for (int i = 0; i < min(nsub, kSubStages); ++i) issue_sub(i);
      for (int i = 0; ok && i < nsub; ++i) {
        const int st = (subs_done + i) % kSubStages;
        const T *sbt = reinterpret_cast<const T *>(sring + st * 2 * sub_bytes);
        const T *sbd = reinterpret_cast<const T *>(sring + st * 2 * sub_bytes + sub_bytes);
        const int n_i = min(kSub, len - i * kSub);
        if (VEC) {
          if (!mbar_wait_bounded(smem_addr(&sm.sub_full[st]), ((subs_done + i) / kSubStages) & 1)) {
            ok = false;
            record(args.status, SV_ERR_TIMEOUT);
          }
        } else {
          T *wt = const_cast<T *>(sbt), *wd = const_cast<T *>(sbd);
          for (int k = tid; k < n_i; k += kThreads) {
            wt[k] = bt[i * kSub + k];
            if (res_pass) wd[k] = bd[i * kSub + k];
          }
          __syncthreads();
        }
        // groups tid and tid + kThreads of the sub-chunk (consecutive threads read consecutive
        // 16-byte pieces of the stage); the two groups of a unit are on adjacent lanes
        static_assert(kSub == 2 * kGroup * kThreads, "two groups a thread and sub-chunk");
        if constexpr (UG == 1) {
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int gl = tid + h * kThreads, g = i * (kSub / kGroup) + gl;
            if (ok && gl * kGroup < n_i) {
              float xt[kGroup], xd[kGroup];
              group8<T, true, false>(sbt, gl, n_i, xt);
              if (res_pass) group8<T, true, false>(sbd, gl, n_i, xd);
              gmass[upad(g)] = mass8(g, xt, xd);
            }
          }
        } else {
          long long mh[2];  // both groups' masses first (independent chains), then the pair sums
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int gl = tid + h * kThreads, g = i * (kSub / kGroup) + gl;
            mh[h] = 0;
            if (ok && gl * kGroup < n_i) {
              float xt[kGroup], xd[kGroup];
              group8<T, true, false>(sbt, gl, n_i, xt);
              if (res_pass) group8<T, true, false>(sbd, gl, n_i, xd);
              mh[h] = mass8(g, xt, xd);
            }
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int gl = tid + h * kThreads, g = i * (kSub / kGroup) + gl;
            const long long pair = mh[h] + __shfl_down_sync(0xffffffffu, mh[h], 1);
            if (ok && gl * kGroup < n_i && (lane & 1) == 0) gmass[upad(g >> 1)] = pair;
          }
        }
        __syncthreads();  // every thread is done with the stage
        if (ok && VEC && tid == 0 && i + kSubStages < nsub) issue_sub(i + kSubStages);
      }
      subs_done += nsub;
      // every CTA, before the cluster barrier: each thread's consecutive units, their mass, its
      // exclusive prefix within the CTA and the CTA's total, and the last unit with mass, so
      // that the owner needs no scan after the barrier
      const int nunits = (ngroups + ug - 1) / ug;
      const int per = (nunits + kThreads - 1) / kThreads;  // consecutive units of this thread
      const int u0 = min(nunits, tid * per), u1 = min(nunits, u0 + per);
      long long local = 0;
      int last_g = -1;  // the last unit with mass
      for (int u = u0; u < u1; ++u) {
        local += gmass[upad(u)];
        if (gmass[upad(u)] > 0) last_g = u;
      }
      if (tid == 0) sm.y_last = -1;
      long long cta_total;
      const long long excl = block_excl_scan_ll(local, sm.ll_buf, &cta_total);
      if (last_g >= 0) atomicMax(&sm.y_last, last_g);
      if (tid == 0) sm.S[pass] = cta_total;
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
          sm.fallback = ((res_pass || excl_pass) && S == 0) ? 1 : 0;
          if (owner_l >= 0) {
            sm.owner = owner_l;
            sm.P_owner = P_l;
          } else {  // u' outside [0, 1): the last token with mass
            sm.owner = has ? 31 - __clz(has) : -1;
            sm.P_owner = -1;
          }
          sm.target = target;
          sm.Stot = S;
          sm.m2 = 0.f;  // stays 0 when rounding leaves no crossing
          sm.y_hit = INT_MAX;
        }
      }
      __syncthreads();
      if (sm.fallback) continue;  // residual without mass: draw from p_a instead
      if (rank == sm.owner) {
        // ---- the owner: the thread whose groups hold the crossing finds it ----
        const long long P = sm.P_owner, target = sm.target;
        long long cum = P + excl;
        if (P >= 0) {
          for (int u = u0; u < u1 && cum <= target; ++u) {
            if (cum + gmass[upad(u)] > target) {  // the unit whose prefix range holds the target
              long long c2 = cum;
              int y = -1;
              for (int g = ug * u; g < min(ug * u + ug, ngroups) && y < 0; ++g) {  // its groups in order
                long long w[kGroup];
                weights8(g, w);
#pragma unroll
                for (int k = 0; k < kGroup; ++k) {
                  c2 += w[k];
                  if (y < 0 && c2 > target) {
                    y = g * kGroup + k;
                    // distance of u' S from the chosen interval's edges, on the normalised CDF
                    const long long below = target - (c2 - w[k]), above = c2 - target;
                    sm.m2 = (float)((double)(below < above ? below : above) / (double)sm.Stot);
                  }
                }
              }
              if (y < 0) y = min(ug * u + ug, ngroups) * kGroup - 1;
              atomicMin(&sm.y_hit, lo + y);
              break;
            }
            cum += gmass[upad(u)];
          }
        }
        __syncthreads();
        if (tid == 0) {
          int y = sm.y_hit;
          if (y == INT_MAX) {  // u' at or past the end: the last token with mass
            const int u = sm.y_last;
            y = lo + max(0, ug * u) * kGroup;
            if (u >= 0)
              for (int g = ug * u; g < min(ug * u + ug, ngroups); ++g) {
                long long w[kGroup];
                weights8(g, w);
                for (int k = 0; k < kGroup; ++k)
                  if (w[k] > 0) y = lo + g * kGroup + k;
              }
          }
          int32_t *o = args.out_tok + (size_t)b * args.max_q;
          if constexpr (MODE == kTreeStochastic) {
            int32_t *path = args.path + (size_t)b * args.max_q;
            for (int j = 0; j < args.max_q; ++j) {
              o[j] = j < a ? sm.tok[sm.path[j] - 1] : -1;
              path[j] = j < a ? sm.path[j] : -1;
            }
          } else {
            for (int j = 0; j < args.max_q; ++j) o[j] = j < a ? sm.tok[j] : -1;
          }
          o[a] = y;
          args.accept[b] = a;
          args.num_out[b] = a + 1;
          if (args.margin) args.margin[b] = fminf(sm.m1, sm.m2);
        }
      }
      break;
    }
  }
  cluster.sync();  // keep this CTA's shared memory alive until every peer is done reading it
}


// Decision cluster size for T > 0: 16 CTAs while 8 a sequence would leave SMs
// idle, 8 while the batch's clusters fit about four CTAs an SM at once, 4 beyond
// (so that large batches run in one wave); chunks of at most kMaxChunk elements.
int pick_cluster(int batch, int vocab) {
  const int sms = num_sms();
  int C = (batch * 8 < sms) ? 16 : (batch * 8 <= 4 * sms ? 8 : 4);
  while (C < 16 && (vocab + C - 1) / C > kMaxChunk) C *= 2;
  return C;
}

template <typename T, bool VEC, int MODE, int UG>
cudaError_t launch_decide(const SamplerArgs &a, float *pm, float *ps, int nchunk, int C, cudaStream_t st) {
  constexpr bool STOCH = MODE == kStochastic || MODE == kTreeStochastic;
  SamplerArgs da = a;
  da.chunk = ((a.vocab + C - 1) / C + 7) / 8 * 8;
  auto dkern = decide_kernel<T, VEC, MODE, UG>;
  const int units = ((da.chunk + kGroup - 1) / kGroup + UG - 1) / UG;
  const int dyn = STOCH ? kRingBytes / UG + upad(units) * (int)sizeof(long long) : 0;
  cudaError_t e = cudaFuncSetAttribute(dkern, cudaFuncAttributeMaxDynamicSharedMemorySize, dyn);
  if (e != cudaSuccess) return e;
  if (C > 8) {
    e = cudaFuncSetAttribute(dkern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
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
  return cudaLaunchKernelEx(&cfg, dkern, da, static_cast<const float *>(pm), static_cast<const float *>(ps), nchunk);
}

template <typename T, bool VEC, int MODE>
cudaError_t launch_t(const SamplerArgs &a, float *pm, float *ps, int nchunk, int rows, cudaStream_t st) {
  // ---- statistics ----
  const int items = rows * nchunk;
  // every CTA of the launch takes floor(items / grid) items, the first (items mod grid) one
  // more: the CTAs of one SM (c and c + SMs when the blocks go round the SMs) differ by one
  // item at most
  const int grid = std::max(1, std::min(items, 2 * num_sms()));
  const int per = items / grid, extra = items - per * grid;
  StatsArgs sa;
  sa.tgt = a.tgt;
  sa.drf = a.drf;
  sa.pm = pm;
  sa.ps = ps;
  sa.status = a.status;
  sa.vocab = a.vocab;
  sa.total_q = a.total_q;
  sa.rows = rows;
  sa.nchunk = nchunk;
  sa.items = items;
  sa.per = per;
  sa.extra = extra;
  sa.coef = a.coef;
  sa.wait_ns = a.wait_ns;
  sa.stall = a.stall;
  constexpr int SMODE = MODE == kTreeStochastic ? kStochastic : MODE;  // statistics of the target rows
  auto skern = stats_kernel<T, VEC, SMODE>;
  const int sdyn = VEC ? kStatStages * kPartBytes : 0;
  cudaError_t e = cudaFuncSetAttribute(skern, cudaFuncAttributeMaxDynamicSharedMemorySize, sdyn);
  if (e != cudaSuccess) return e;
  e = launch_pdl(skern, dim3(grid), dim3(kStatThreads), sdyn, st, sa);
  if (e != cudaSuccess) return e;

  // ---- decisions ----
  constexpr bool STOCH = MODE == kStochastic || MODE == kTreeStochastic;
  const int C = STOCH ? pick_cluster(a.batch, a.vocab) : 1;
  if constexpr (STOCH) {
    if (C < 8) return launch_decide<T, VEC, MODE, 2>(a, pm, ps, nchunk, C, st);
  }
  return launch_decide<T, VEC, MODE, 1>(a, pm, ps, nchunk, C, st);
}

// rows 16-byte aligned: 1-D bulk copies (every item and chunk then starts on 16
// bytes and is a multiple of 16 bytes long); otherwise scalar loads
template <typename T, int MODE>
cudaError_t launch_m(const SamplerArgs &a, float *pm, float *ps, int nchunk, int rows, cudaStream_t st) {
  const bool vec = ((size_t)a.vocab * sizeof(T)) % 16 == 0 && ((uintptr_t)a.tgt % 16 == 0) &&
                   (a.drf == nullptr || (uintptr_t)a.drf % 16 == 0);
  return vec ? launch_t<T, true, MODE>(a, pm, ps, nchunk, rows, st)
             : launch_t<T, false, MODE>(a, pm, ps, nchunk, rows, st);
}

template <typename T>
cudaError_t launch_d(const SamplerArgs &a, int mode, float *pm, float *ps, int nchunk, int rows, cudaStream_t st) {
  switch (mode) {
    case kStochastic: return launch_m<T, kStochastic>(a, pm, ps, nchunk, rows, st);
    case kGreedy: return launch_m<T, kGreedy>(a, pm, ps, nchunk, rows, st);
    case kTreeStochastic: return launch_m<T, kTreeStochastic>(a, pm, ps, nchunk, rows, st);
    default: return launch_m<T, kTree>(a, pm, ps, nchunk, rows, st);
  }
}

long long stat_rows(int total_q, int batch, int mode) {
  return mode == kStochastic ? 2LL * total_q - batch : (long long)total_q;
}

long long stat_chunks(int vocab, int dtype) {
  const long long es = dtype == SV_DTYPE_BF16 ? 2 : 4;
  return ((long long)vocab * es + kPartBytes - 1) / kPartBytes;
}

}  // namespace

size_t sampler_workspace_bytes(int vocab, int dtype, int total_q, int batch, int mode) {
  if (vocab < 1 || total_q < 0 || batch < 0 || batch > total_q) return 0;
  const long long parts = stat_rows(total_q, batch, mode) * stat_chunks(vocab, dtype) * kStatWarps;
  if (parts >= (1LL << 31)) return 0;
  return (size_t)parts * 2 * sizeof(float);
}

cudaError_t launch_sampler(const SamplerArgs &a, int dtype, int mode, void *workspace, cudaStream_t st) {
  if (a.batch == 0) return cudaSuccess;
  const int nchunk = (int)stat_chunks(a.vocab, dtype);
  const int rows = (int)stat_rows(a.total_q, a.batch, mode);
  float *pm = static_cast<float *>(workspace);
  float *ps = pm + (size_t)rows * nchunk * kStatWarps;
  return dtype == SV_DTYPE_BF16 ? launch_d<__nv_bfloat16>(a, mode, pm, ps, nchunk, rows, st)
                                : launch_d<float>(a, mode, pm, ps, nchunk, rows, st);
}

// Largest vocabulary: 16 decision chunks of kMaxChunk elements.
bool sampler_supports(int vocab) { return vocab <= 16 * kMaxChunk; }

}  // namespace sv
