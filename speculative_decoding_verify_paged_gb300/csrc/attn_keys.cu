// Keys-major paged attention on the 5th-generation tensor cores for units of
// at most 32 query rows (bf16 caches, head_dim 128).
//
// What it computes is the same as attn_umma.cu (the verify-pass attention of
// "Speculative decoding and continuous batching in practice", sec. 1.2, over
// the paged cache of "LLM serving: speculative decoding and PagedAttention
// memory management", causal or tree mask of "Speculative decoding principles
// and a vLLM production setup", sec. 3.2 and 5.2).
//
// A verify step has few query rows per (sequence, KV head) unit: the G query
// heads of the KV head times K+1 positions (24 for 32/8 heads and K=5). With
// query rows on the MMA's M dimension (128) most of the tensor work and all
// but one softmax warp are idle, and the S product costs 8 MMA issues per 32
// keys. Here the keys take the M dimension instead: S^T = K Q^T with M = 128
// keys, N = 32 query rows, K = head_dim (8 MMAs per 128 keys; A = K and B = Q,
// both K-major in shared memory), written to TMEM with one key per lane. The
// four softmax warps hold 32 keys each: a thread has one key's scores for all
// 32 rows. The tile maximum of each row is reduced over the lanes by a
// transpose-reduction (lane l ends with row l's maximum) and over the warps
// through shared memory (one barrier of the four softmax warps per tile);
// every thread then weights its key for all rows, P^T goes to shared memory
// (one 64-byte key row per thread, the MN-major layout of an A operand), and
// O += P V runs with A = P (MN-major), B = V (MN-major), M = 128 (rows past 32
// unused), N = 128, 16 keys per MMA. O holds one query row per TMEM lane in
// the lanes of the first softmax warp, which rescales it when a row's running
// maximum moves (by more than 2^8) and writes it at the end of a piece.
//
// Work, pieces, workspace slots and their merge are those of attn_umma.cu with
// 128-key tiles and one persistent CTA per SM: 2 K slots and 3 V slots of 32 KB
// (a K tile is free once S^T has read it, a V tile once P V has).
// All mbarrier waits are bounded; a wait that gives up records SV_ERR_TIMEOUT.
#include <cuda.h>

#include <algorithm>

#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr int kD = 128;
constexpr int kTileK = 128;                    // keys per tile (MMA M)
constexpr int kRowsK = 32;                     // query rows per unit (MMA N)
constexpr int kKSlots = 2, kVSlots = 3;
constexpr int kSoftWarps = 4;
constexpr int kThreads = (2 + kSoftWarps) * 32;
constexpr int kTileBytes = kTileK * kD * 2;    // 32 KB: 16 groups of 8 keys x [half 0 | half 1]
constexpr int kQBytes = kRowsK * kD * 2;       // 8 KB, the same layout
constexpr int kPBytes = kTileK / 8 * 1024;     // 16 KB: 16 groups of 8 keys x 128 B (rows 0-63 of P^T)
constexpr int kTmemCols = 256;                 // S^T 0 [0,32) S^T 1 [32,64) O [64,192)
constexpr int kColO = 64;
constexpr float kRescaleThreshold = 8.f;       // log2 units

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
// budget: the launch's pipeline budget, or kDrainBudgetNs for copies and MMAs already issued
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned long long budget) {
  return mbar_wait_bounded(bar, parity, budget);
}
// One box of the (64 elements, 8 rows, 2 halves, row groups) view of a pool.
__device__ __forceinline__ void tma_load_rows(uint32_t dst, const CUtensorMap *map, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, %5}], [%6];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(0), "r"(0), "r"(y >> 3), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Shared-memory matrix descriptor: start, leading and stride byte offsets (16-byte
// units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// Instruction descriptor of kind::f16: fp32 accumulate, bf16 A and B, A and B
// K-major (0) or MN-major (1), N / 8 and M / 16.
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)a_mn << 15) | ((uint32_t)b_mn << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, int accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accum));
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

#define SV_R8(r, o) "=r"(r[o + 0]), "=r"(r[o + 1]), "=r"(r[o + 2]), "=r"(r[o + 3]), "=r"(r[o + 4]), "=r"(r[o + 5]), \
                    "=r"(r[o + 6]), "=r"(r[o + 7])
#define SV_W8(r, o) "r"(r[o + 0]), "r"(r[o + 1]), "r"(r[o + 2]), "r"(r[o + 3]), "r"(r[o + 4]), "r"(r[o + 5]), \
                    "r"(r[o + 6]), "r"(r[o + 7])
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,"
      "%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : SV_R8(r, 0), SV_R8(r, 8), SV_R8(r, 16), SV_R8(r, 24)
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      SV_W8(r, 0), SV_W8(r, 8), SV_W8(r, 16), SV_W8(r, 24)
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// 2^x by the MUFU approximation (flush-to-zero): softmax weights only, rounded to bf16 next
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
// Named barrier 1 over the softmax warps, AND of `v` over their threads.
__device__ __forceinline__ bool soft_bar_and(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred pi, po;\n setp.ne.u32 pi, %1, 0;\n bar.red.and.pred po, 1, %2, pi;\n selp.u32 %0, 1, 0, po;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kSoftWarps * 32)
      : "memory");
  return r != 0;
}

struct KeysParams {
  AttnArgs a;
  int box_rows;     // rows per TMA box: min(block_size, 32)
  int G;            // query heads per KV head
  int rows_cap;     // rows of a workspace slot: G * max_q (<= 32)
  int ctas;         // CTAs of the launch
  float *part_o;    // [ctas][2][rows_cap][128] normalised partial outputs
  float *part_lse;  // [ctas][2][rows_cap] their log-sum-exp (base 2)
  int *prefix;      // [batch + 1]: first tile of each sequence's units; [batch] = all tiles
};

// One sequence as the work decomposition sees it; tiles == 0: nothing to do.
struct Seq {
  int c, row0, n, L;
  int tiles;  // key tiles of each of its units: ceil(L / 128)
};

__device__ __forceinline__ Seq load_seq(const KeysParams &P, int b, bool *bad) {
  const AttnArgs &a = P.a;
  const KV &kv = a.kv;
  Seq s;
  s.c = kv.seq_lens[b];
  s.row0 = a.cu_q[b];
  s.n = a.cu_q[b + 1] - s.row0;
  const long long L = (long long)s.c + s.n;
  const bool ok = s.c >= 0 && s.n >= 0 && s.n <= a.max_q && s.row0 >= 0 &&
                  (long long)s.row0 + s.n <= a.total_q && L <= a.max_seq_len &&
                  L <= (long long)kv.max_blocks * kv.block_size && P.G * s.n <= kRowsK;
  *bad = !ok;
  s.L = ok ? (int)L : 0;
  s.tiles = (ok && s.n > 0) ? (s.L + kTileK - 1) / kTileK : 0;
  return s;
}
__device__ __forceinline__ int seq_work(const KeysParams &P, const Seq &s) { return P.a.kv.num_kv_heads * s.tiles; }

// Inclusive sum over the CTA's threads; *total gets the sum over all of them.
__device__ __forceinline__ int block_scan(int v, int *sh, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += y;
  }
  if (lane == 31) sh[warp] = x;
  __syncthreads();
  int before = 0, all = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const int t = sh[w];
    before += w < warp ? t : 0;
    all += t;
  }
  __syncthreads();
  *total = all;
  return x + before;
}

// The part of one unit (sequence, KV head) that lies in a CTA's tile range.
struct Piece {
  int b, kvh, c, row0, n, L;
  int kt0, kt1;  // key tiles [kt0, kt1) of the unit
  bool whole;    // the piece is the whole unit
};

// Walks the tile range [g, end) piece by piece, sequence b starting at global tile `base`.
struct Walker {
  int b, base, g, end;
  Seq s;
  __device__ __forceinline__ bool next(const KeysParams &P, Piece &p) {
    if (g >= end) return false;
    int work = seq_work(P, s);
    while (g - base >= work) {
      if (b + 1 >= P.a.kv.batch) {  // cannot happen while the lengths stay put; never read past the batch
        g = end;
        return false;
      }
      base += work;
      ++b;
      bool bad;
      s = load_seq(P, b, &bad);
      work = seq_work(P, s);
    }
    const int local = g - base;
    const int j = local / s.tiles, off = local - j * s.tiles;
    const int len = min(s.tiles - off, end - g);
    p.b = b;
    p.kvh = j;
    p.c = s.c;
    p.row0 = s.row0;
    p.n = s.n;
    p.L = s.L;
    p.kt0 = off;
    p.kt1 = off + len;
    p.whole = off == 0 && len == s.tiles;
    g += len;
    return true;
  }
};

// Shared memory (1024-aligned): K slots, V slots, the Q tile, two P^T tiles and
// 1 KB read past the last one by the P V MMAs (rows 64-127, unused).
constexpr size_t kSmemBytes = 1024 + (size_t)(kKSlots + kVSlots) * kTileBytes + kQBytes + 2 * kPBytes + 1024;

__global__ void __launch_bounds__(kThreads, 1) attn_keys_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                                                const __grid_constant__ CUtensorMap tmap_v,
                                                                const KeysParams P) {
  grid_dependency_wait();  // the earlier kernel on the stream is complete and visible
  grid_dependents_launch();
  const AttnArgs &a = P.a;
  const KV &kv = a.kv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = kv.batch;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *kring = base;                               // kKSlots x 32 KB
  uint8_t *vring = kring + kKSlots * kTileBytes;       // kVSlots x 32 KB
  uint8_t *qbuf = vring + kVSlots * kTileBytes;        // 8 KB
  uint8_t *pbuf = qbuf + kQBytes;                      // 2 x 16 KB
  __shared__ uint64_t k_full[kKSlots], k_empty[kKSlots], v_full[kVSlots], v_empty[kVSlots];
  __shared__ uint64_t s_full[2], p_ready[2], o_bar, q_ready, mma_done;
  __shared__ uint32_t tmem_slot;
  __shared__ int sh_scan[kThreads / 32];
  __shared__ int sh_first_b, sh_first_base, sh_err;
  __shared__ float xm[2][kSoftWarps][32];  // per tile parity: each warp's column maxima
  __shared__ float xl[kSoftWarps][32];     // each warp's column sums at the end of a piece
  __shared__ int s_i[kSoftWarps][kRowsK];  // each softmax warp's copy: the piece's position of each row
  __shared__ unsigned long long s_tm[kSoftWarps][kRowsK];  // and its tree mask

  if (tid == 0) {
    for (int s = 0; s < kKSlots; ++s) {
      mbar_init(smem_u32(&k_full[s]), 1);
      mbar_init(smem_u32(&k_empty[s]), 1);
    }
    for (int s = 0; s < kVSlots; ++s) {
      mbar_init(smem_u32(&v_full[s]), 1);
      mbar_init(smem_u32(&v_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&s_full[s]), 1);
      mbar_init(smem_u32(&p_ready[s]), kSoftWarps);
    }
    mbar_init(smem_u32(&o_bar), 1);
    mbar_init(smem_u32(&q_ready), kSoftWarps);
    mbar_init(smem_u32(&mma_done), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    sh_first_b = 0;
    sh_first_base = 0;
    sh_err = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }

  // ---- this CTA's tile range [g0, g1) of the W tiles of the launch ----
  int mine = 0;
  for (int b = tid; b < B; b += kThreads) {
    bool bad;
    const Seq s = load_seq(P, b, &bad);
    if (bad && blockIdx.x == 0) record(a.status, SV_ERR_BAD_LENGTH);
    mine += seq_work(P, s);
  }
  int W;
  block_scan(mine, sh_scan, &W);
  const int per = max(1, (W + P.ctas - 1) / P.ctas);
  const int g0 = min(W, (int)blockIdx.x * per), g1 = min(W, g0 + per);
  int run = 0;
  for (int b0 = 0; b0 < B; b0 += kThreads) {  // the sequence holding tile g0; CTA 0 also stores the prefix
    const int b = b0 + tid;
    int v = 0;
    if (b < B) {
      bool bad;
      v = seq_work(P, load_seq(P, b, &bad));
    }
    int tot;
    const int excl = run + block_scan(v, sh_scan, &tot) - v;
    if (blockIdx.x == 0 && b < B) P.prefix[b] = excl;
    if (v > 0 && excl <= g0 && g0 < excl + v) {
      sh_first_b = b;
      sh_first_base = excl;
    }
    run += tot;
    if (blockIdx.x != 0 && run > g0) break;  // uniform: run and g0 are the same in every thread
  }
  if (blockIdx.x == 0 && tid == 0) P.prefix[B] = W;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  Walker walker;
  walker.b = sh_first_b;
  walker.base = sh_first_base;
  walker.g = g0;
  walker.end = g1;
  {
    bool bad;
    walker.s = load_seq(P, walker.b, &bad);
  }
  bool ok = true;
  int issued = 0;  // producer: tiles whose loads were issued

  if (warp == 0) {
    // ================= producer: K then V of each 128-key tile =================
    const int bs = kv.block_size, box = P.box_rows;
    const int bs_shift = __ffs(bs) - 1;
    const uint32_t box_bytes = static_cast<uint32_t>(box) * 256;
    Piece p;
    while (ok && walker.next(P, p)) {
      const int kb = p.kt0 * kTileK, ke = min(p.L, p.kt1 * kTileK);
      const int lb_last = (ke - 1) >> bs_shift;
      const int32_t *bt = kv.block_table + (size_t)p.b * kv.max_blocks;
      // first pool row of logical block lb for this KV head; -1 past the piece or for a bad id
      auto load_y = [&](int lb) -> int {
        if (lb > lb_last) return -1;
        const int id = bt[lb];
        if (id < 0 || id >= kv.num_blocks) {
          record(a.status, SV_ERR_BAD_BLOCK_ID);
          return -1;
        }
        return (id * kv.num_kv_heads + p.kvh) << bs_shift;
      };
      int wbase = kb >> bs_shift;  // lane l holds logical block wbase + l (cur) and wbase + 32 + l (nxt)
      int cur = load_y(wbase + lane);
      int nxt = load_y(wbase + 32 + lane);
      for (int kt = p.kt0; kt < p.kt1; ++kt, ++issued) {
        const int k0 = kt * kTileK;
        int ys[kTileK / 16];
        int nbox = 0;
#pragma unroll
        for (int j = 0; j < kTileK / 16; ++j) {
          const int tok = k0 + j * box;
          int y = -1;
          if (j * box < kTileK && tok < ke) {
            const int lb = tok >> bs_shift;
            while (lb >= wbase + 32) {  // warp-uniform
              wbase += 32;
              cur = nxt;
              nxt = load_y(wbase + 32 + lane);
            }
            const int yb = __shfl_sync(0xffffffffu, cur, lb - wbase);
            y = yb < 0 ? -1 : yb + (tok & (bs - 1));
          }
          ys[j] = y;
          nbox += y >= 0;
        }
        const int ks = issued % kKSlots, vs = issued % kVSlots;
        if (issued >= kKSlots)
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&k_empty[ks]), ((issued / kKSlots) - 1) & 1, a.wait_ns));
        if (!ok) break;
        if (lane == 0) {
          const uint32_t fb = smem_u32(&k_full[ks]);
          mbar_expect_tx(fb, static_cast<uint32_t>(nbox) * box_bytes);
#pragma unroll
          for (int j = 0; j < kTileK / 16; ++j)
            if (ys[j] >= 0) tma_load_rows(smem_u32(kring + ks * kTileBytes) + j * box_bytes, &tmap_k, ys[j], fb);
        }
        __syncwarp();
        if (issued >= kVSlots)
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&v_empty[vs]), ((issued / kVSlots) - 1) & 1, a.wait_ns));
        if (!ok) break;
        if (lane == 0) {
          const uint32_t fb = smem_u32(&v_full[vs]);
          mbar_expect_tx(fb, static_cast<uint32_t>(nbox) * box_bytes);
#pragma unroll
          for (int j = 0; j < kTileK / 16; ++j)
            if (ys[j] >= 0) tma_load_rows(smem_u32(vring + vs * kTileBytes) + j * box_bytes, &tmap_v, ys[j], fb);
        }
        __syncwarp();
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    constexpr uint32_t idesc_s = mma_idesc(128, kRowsK, 0, 0);  // S^T = K Q^T: A, B K-major
    constexpr uint32_t idesc_o = mma_idesc(128, kD, 1, 1);      // O += P V: A, B MN-major
    // O (+)= P(u) V(u), 16 keys per MMA: P^T groups of 8 keys 1 KB apart (rows 64-127 of the
    // A operand read the next group: unused), V groups 2 KB apart with the head_dim halves 1 KB apart
    auto issue_pv = [&](int u, bool accumulate) {
      const int vs = u % kVSlots;
      const uint32_t v_base = smem_u32(vring + vs * kTileBytes);
      const uint32_t p_base = smem_u32(pbuf + (u & 1) * kPBytes);
#pragma unroll
      for (int kk = 0; kk < kTileK / 16; ++kk)
        mma_ss(tmem + kColO, smem_desc(p_base + kk * 2048, 1024, 1024), smem_desc(v_base + kk * 4096, 1024, 2048),
               idesc_o, (accumulate || kk > 0) ? 1 : 0);
      mma_commit(smem_u32(&v_empty[vs]));
      mma_commit(smem_u32(&o_bar));
    };
    int t = 0, piece = 0;
    int pend = -1;  // P V of tile t - 1 still to issue: -1 none, 0 overwrite O, 1 accumulate
    Piece p;
    auto finish_pv = [&](int u, int mode) -> bool {  // P(u) written and V(u) landed, then P V(u)
      bool w = mbar_wait(smem_u32(&p_ready[u & 1]), (u >> 1) & 1, a.wait_ns);
      if (w) w = mbar_wait(smem_u32(&v_full[u % kVSlots]), (u / kVSlots) & 1, a.wait_ns);
      if (!__all_sync(0xffffffffu, w)) return false;
      tc_fence_after();
      if (lane == 0) issue_pv(u, mode == 1);
      __syncwarp();
      return true;
    };
    while (ok && walker.next(P, p)) {
      for (int kt = p.kt0; kt < p.kt1; ++kt, ++t) {
        const int ks = t % kKSlots;
        bool w = mbar_wait(smem_u32(&k_full[ks]), (t / kKSlots) & 1, a.wait_ns);
        if (w && kt == p.kt0) w = mbar_wait(smem_u32(&q_ready), piece & 1, a.wait_ns);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t k_base = smem_u32(kring + ks * kTileBytes), q_base = smem_u32(qbuf);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)  // 16 head_dim elements per MMA: half kk / 4 at +1 KB
            mma_ss(tmem + (t & 1) * kRowsK, smem_desc(k_base + (kk >> 2) * 1024 + (kk & 3) * 32, 16, 2048),
                   smem_desc(q_base + (kk >> 2) * 1024 + (kk & 3) * 32, 16, 2048), idesc_s, kk > 0 ? 1 : 0);
          mma_commit(smem_u32(&s_full[t & 1]));
          mma_commit(smem_u32(&k_empty[ks]));
        }
        __syncwarp();
        if (pend >= 0) {
          ok = finish_pv(t - 1, pend);
          if (!ok) break;
        }
        pend = kt != p.kt0 ? 1 : 0;
      }
      ++piece;
    }
    if (ok && pend >= 0) ok = finish_pv(t - 1, pend);
    // every MMA issued finishes before TMEM is released
    if (lane == 0) mma_commit(smem_u32(&mma_done));
    __syncwarp();
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&mma_done), 0, kDrainBudgetNs))) ok = false;
  } else {
    // ================= softmax: one key per thread, 32 query rows =================
    const int q4 = warp & 3;                           // TMEM lane quarter: keys 32 q4 .. 32 q4 + 31
    const int tsoft = q4 * 32 + lane;                  // 0..127
    const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
    const bool owner = q4 == 0;                        // its lanes hold O's rows
    const __nv_bfloat16 *qsrc = reinterpret_cast<const __nv_bfloat16 *>(a.q);
    // the piece's 32 query rows into the Q tile (K-major, 128-byte swizzle: row r's
    // 16-byte chunk c of head_dim half h at (r / 8) 2 KB + h 1 KB + (r % 8) 128 + (c ^ r % 8) 16);
    // rows past the unit's are zero. Also the rows' positions and tree masks.
    auto stage_q = [&](const Piece &p) {
      const int rows = P.G * p.n;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int x = tsoft + 128 * j;  // 512 chunks of 16 bytes
        const int r = x >> 4, c = x & 15, h = c >> 3, cc = c & 7;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (r < rows) {
          const int i = r / P.G, g = r - i * P.G;
          v = *reinterpret_cast<const uint4 *>(qsrc + ((size_t)(p.row0 + i) * a.num_q_heads + p.kvh * P.G + g) * kD +
                                               c * 8);
        }
        *reinterpret_cast<uint4 *>(qbuf + (r >> 3) * 2048 + h * 1024 + (r & 7) * 128 + ((cc ^ (r & 7)) * 16)) = v;
      }
      {  // this warp's own copy, read only by its lanes (a __syncwarp orders it)
        const int r = lane;
        const int i = r < rows ? r / P.G : 0;
        s_i[q4][r] = r < rows ? i : -1;
        s_tm[q4][r] = (r < rows && a.mask_kind == SV_MASK_TREE) ? a.tree_mask[p.row0 + i] : 0ull;
      }
      fence_proxy_async();  // visible to the tensor core's reads
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(&q_ready));
    };
    Piece cur, nxt;
    bool has_cur = walker.next(P, cur);
    bool has_nxt = has_cur && walker.next(P, nxt);
    if (has_cur) stage_q(cur);
    int t = 0;
    bool first_piece = true;
    while (has_cur && ok) {
      const int rows = P.G * cur.n;
      const int c = cur.c, ke = min(cur.L, cur.kt1 * kTileK);
      float m_run = -INFINITY;  // lane l: running maximum of row l
      float lsum[kRowsK];       // this key's share of each row's sum
#pragma unroll
      for (int r = 0; r < kRowsK; ++r) lsum[r] = 0.f;
      bool all_ok = true;
      for (int kt = cur.kt0; kt < cur.kt1; ++kt, ++t) {
        const bool handoff = kt == cur.kt1 - 1 && has_nxt;
        const int k0 = kt * kTileK;
        const int valid = min(kTileK, ke - k0);
        bool w = ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(&s_full[t & 1]), (t >> 1) & 1, a.wait_ns));
        tc_fence_after();
        uint32_t sr[kRowsK];
        if (w) {
          tmem_ld32(lane_addr + (t & 1) * kRowsK, sr);
          tmem_wait_ld();
        }
        if (w && kt == cur.kt1 - 1 && t >= 1)  // P V(t-1) done before P(t) goes out (o_bar phase, see attn_umma.cu)
          w = __all_sync(0xffffffffu, mbar_wait(smem_u32(&o_bar), (t - 1) & 1, a.wait_ns));
        if (w && valid < kTileK) {
          // zero this tile's V rows past the unit's end before P V reads them
          w = __all_sync(0xffffffffu, mbar_wait(smem_u32(&v_full[t % kVSlots]), (t / kVSlots) & 1, a.wait_ns));
          uint8_t *vst = vring + (t % kVSlots) * kTileBytes;
          for (int x = tsoft; w && x < (kTileK - valid) * 16; x += kSoftWarps * 32) {
            const int rr = valid + (x >> 4), ch = x & 15;
            *reinterpret_cast<uint4 *>(vst + (rr >> 3) * 2048 + (ch >> 3) * 1024 + (rr & 7) * 128 + (ch & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async();
        }
        // scores of this key for every row, in log2 units; edge tiles (new rows, ragged end) masked
        const int key = k0 + tsoft;
        float sv[kRowsK];
        const bool edge = (k0 + kTileK > c) || (valid < kTileK);  // uniform over the four warps
        if (!edge) {
#pragma unroll
          for (int r = 0; r < kRowsK; ++r) sv[r] = __uint_as_float(sr[r]) * a.scale_log2;
        } else {
#pragma unroll
          for (int r = 0; r < kRowsK; ++r) {
            bool vis = key < ke;
            if (vis && key >= c) {
              const int j = key - c;
              vis = (a.mask_kind == SV_MASK_CAUSAL) ? (j <= s_i[q4][r]) : (j < 64 && ((s_tm[q4][r] >> j) & 1ull));
            }
            sv[r] = vis ? __uint_as_float(sr[r]) * a.scale_log2 : -INFINITY;
          }
        }
        // the warp's maximum of each row over its 32 keys: lane l ends with row l's
        float v[kRowsK];
#pragma unroll
        for (int r = 0; r < kRowsK; ++r) v[r] = w ? sv[r] : -INFINITY;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const bool upper = (lane & o) != 0;
#pragma unroll
          for (int k = 0; k < o; ++k) {
            const float send = upper ? v[k] : v[k + o];
            const float keep = upper ? v[k + o] : v[k];
            v[k] = fmaxf(keep, __shfl_xor_sync(0xffffffffu, send, o));
          }
        }
        xm[t & 1][q4][lane] = v[0];
        if (!soft_bar_and(w)) {  // every softmax warp leaves here together
          all_ok = false;
          break;
        }
        // S^T(t) was this piece's last product with its Q, and every warp is past its reads of the
        // tile's masks: the next piece's rows can take their place
        if (handoff) stage_q(nxt);
        float mx = xm[t & 1][0][lane];
#pragma unroll
        for (int q = 1; q < kSoftWarps; ++q) mx = fmaxf(mx, xm[t & 1][q][lane]);
        // row `lane`: move the running maximum only when the tile's exceeds it by the threshold
        const bool move = mx > m_run + kRescaleThreshold || (m_run == -INFINITY && mx != -INFINITY);
        const float f = (move && m_run != -INFINITY) ? exp2f(m_run - mx) : 1.f;
        if (move) m_run = mx;
        if (__any_sync(0xffffffffu, f != 1.f)) {
          // rows whose sums and O must be rescaled: every thread its share of the sums
#pragma unroll
          for (int r = 0; r < kRowsK; ++r) lsum[r] *= __shfl_sync(0xffffffffu, f, r);
          if (owner) {
            // O row `lane`: wait for P(t-1) V(t-1) (S^T(t) done means P V up to t-2 is)
            if (!mbar_wait(smem_u32(&o_bar), (t - 1) & 1, a.wait_ns)) ok = false;
            tc_fence_after();
#pragma unroll
            for (int cb = 0; cb < kD / 32; ++cb) {
              uint32_t o[32];
              tmem_ld32(lane_addr + kColO + cb * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * f);
              tmem_st32(lane_addr + kColO + cb * 32, o);
            }
            tmem_wait_st();
          }
        }
        // P^T: this key's weights for every row, relative to the rows' running maxima
        uint32_t pr[kRowsK / 2];
#pragma unroll
        for (int r = 0; r < kRowsK; r += 2) {
          const float m0 = __shfl_sync(0xffffffffu, m_run, r), m1 = __shfl_sync(0xffffffffu, m_run, r + 1);
          const float p0 = fast_exp2(sv[r] - (m0 == -INFINITY ? 0.f : m0));
          const float p1 = fast_exp2(sv[r + 1] - (m1 == -INFINITY ? 0.f : m1));
          lsum[r] += p0;
          lsum[r + 1] += p1;
          pr[r >> 1] = pack_bf16(p0, p1);
        }
        // key row tsoft of the P^T tile (MN-major, 128-byte swizzle): group tsoft / 8 at 1 KB
        // steps, row tsoft % 8 at 128 B, 16-byte chunk cc (rows 8 cc .. 8 cc + 7) at (cc ^ tsoft % 8) 16
        uint8_t *prow = pbuf + (t & 1) * kPBytes + (tsoft >> 3) * 1024 + (tsoft & 7) * 128;
#pragma unroll
        for (int cc = 0; cc < kRowsK / 8; ++cc)
          *reinterpret_cast<uint4 *>(prow + ((cc ^ (tsoft & 7)) * 16)) =
              make_uint4(pr[4 * cc], pr[4 * cc + 1], pr[4 * cc + 2], pr[4 * cc + 3]);
        fence_proxy_async();  // visible to the tensor core's reads
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&p_ready[t & 1]));
      }
      if (!all_ok) {
        ok = false;
        break;
      }
      // ---- end of the piece: wait for its last P V, then write ----
      const int tl = t - 1;
      const bool w = ok && __all_sync(0xffffffffu, mbar_wait(smem_u32(&o_bar), tl & 1, a.wait_ns));
      tc_fence_after();
      // each row's sum over the warp's keys: lane l ends with row l's (transpose-reduction)
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const bool upper = (lane & o) != 0;
#pragma unroll
        for (int k = 0; k < o; ++k) {
          const float send = upper ? lsum[k] : lsum[k + o];
          const float keep = upper ? lsum[k + o] : lsum[k];
          lsum[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      xl[q4][lane] = lsum[0];
      if (!soft_bar_and(w)) {
        ok = false;
        break;
      }
      if (owner) {
        float L = 0.f;  // row `lane`'s sum, over the warps in a fixed order
#pragma unroll
        for (int q = 0; q < kSoftWarps; ++q) L += xl[q][lane];
        const int r = lane;
        const bool live = r < rows;
        const int i = live ? r / P.G : 0, g = live ? r - i * P.G : 0;
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const size_t qrow = (size_t)(cur.row0 + i) * a.num_q_heads + cur.kvh * P.G + g;
        const size_t slot = ((size_t)blockIdx.x * 2 + (first_piece ? 0 : 1)) * P.rows_cap + r;
#pragma unroll
        for (int cb = 0; cb < kD / 32; ++cb) {
          uint32_t o[32];
          tmem_ld32(lane_addr + kColO + cb * 32, o);
          tmem_wait_ld();
          if (!live) continue;
          if (cur.whole) {
            uint4 *op = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.out) + qrow * kD + cb * 32);
#pragma unroll
            for (int v4 = 0; v4 < 4; ++v4)
              op[v4] = make_uint4(pack_bf16(__uint_as_float(o[8 * v4 + 0]) * inv, __uint_as_float(o[8 * v4 + 1]) * inv),
                                  pack_bf16(__uint_as_float(o[8 * v4 + 2]) * inv, __uint_as_float(o[8 * v4 + 3]) * inv),
                                  pack_bf16(__uint_as_float(o[8 * v4 + 4]) * inv, __uint_as_float(o[8 * v4 + 5]) * inv),
                                  pack_bf16(__uint_as_float(o[8 * v4 + 6]) * inv, __uint_as_float(o[8 * v4 + 7]) * inv));
          } else {
            float4 *op = reinterpret_cast<float4 *>(P.part_o + slot * kD + cb * 32);
#pragma unroll
            for (int v4 = 0; v4 < 8; ++v4)
              op[v4] = make_float4(__uint_as_float(o[4 * v4]) * inv, __uint_as_float(o[4 * v4 + 1]) * inv,
                                   __uint_as_float(o[4 * v4 + 2]) * inv, __uint_as_float(o[4 * v4 + 3]) * inv);
            if (cb == 0) P.part_lse[slot] = L > 0.f ? m_run + log2f(L) : -INFINITY;
          }
        }
      }
      first_piece = false;
      cur = nxt;
      has_cur = has_nxt;
      has_nxt = has_cur && walker.next(P, nxt);
    }
  }
  if (!ok) {
    if (lane == 0) record(a.status, SV_ERR_TIMEOUT);
    sh_err = 1;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (sh_err != 0 && warp == 0 && lane == 0) {
    // after a failed wait, let this CTA's copies in flight land before its shared memory is released
    for (int k = max(0, issued - kKSlots); k < issued; ++k) mbar_wait(smem_u32(&k_full[k % kKSlots]), (k / kKSlots) & 1, kDrainBudgetNs);
    for (int k = max(0, issued - kVSlots); k < issued; ++k) mbar_wait(smem_u32(&v_full[k % kVSlots]), (k / kVSlots) & 1, kDrainBudgetNs);
  }
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

// Merges the partial results of every unit that two or more CTAs shared (as
// attn_umma.cu's combine, with 128-key tiles and one row block).
__global__ void __launch_bounds__(128) attn_keys_combine(const KeysParams P) {
  grid_dependency_wait();  // the earlier kernel on the stream is complete and visible
  grid_dependents_launch();
  const AttnArgs &a = P.a;
  const int b = blockIdx.x, kvh = blockIdx.y;
  const int tid = threadIdx.x;
  __shared__ float row_max[kRowsK], row_inv[kRowsK];
  const int W = P.prefix[a.kv.batch], base = P.prefix[b];
  bool bad;
  const Seq s = load_seq(P, b, &bad);
  if (s.tiles == 0) return;
  const int per = max(1, (W + P.ctas - 1) / P.ctas);
  const int T0 = base + kvh * s.tiles, T1 = T0 + s.tiles;
  const int c0 = T0 / per, c1 = (T1 - 1) / per;
  if (c0 == c1) return;  // one CTA held the whole unit and wrote its rows
  const int slot0 = T0 == c0 * per ? 0 : 1;
  auto slot_of = [&](int cc, int row) -> size_t {
    return ((size_t)cc * 2 + (cc == c0 ? slot0 : 0)) * P.rows_cap + row;
  };
  const int rows = P.G * s.n;
  for (int row = tid; row < rows; row += blockDim.x) {
    float M = -INFINITY;
    for (int cc = c0; cc <= c1; ++cc) M = fmaxf(M, P.part_lse[slot_of(cc, row)]);
    float den = 0.f;
    if (M != -INFINITY)
      for (int cc = c0; cc <= c1; ++cc) den += exp2f(P.part_lse[slot_of(cc, row)] - M);
    row_max[row] = M;
    row_inv[row] = den > 0.f ? 1.f / den : 0.f;
  }
  __syncthreads();
  constexpr int kUnroll = 4;
  const int outs = rows * (kD / 4);
  for (int x0 = tid; x0 < outs; x0 += blockDim.x * kUnroll) {
    float4 acc[kUnroll];
    int xr[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      xr[u] = x0 + u * blockDim.x;
    }
    for (int cc = c0; cc <= c1; ++cc) {
      float lse[kUnroll];
      float4 o[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        lse[u] = -INFINITY;
        o[u] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (xr[u] < outs) {
          const int row = xr[u] / (kD / 4), c4 = (xr[u] % (kD / 4)) * 4;
          const size_t sl = slot_of(cc, row);
          lse[u] = P.part_lse[sl];
          o[u] = *reinterpret_cast<const float4 *>(P.part_o + sl * kD + c4);
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        if (xr[u] >= outs) continue;
        const float M = row_max[xr[u] / (kD / 4)];
        const float wk = M == -INFINITY ? 0.f : exp2f(lse[u] - M);
        acc[u].x = fmaf(wk, o[u].x, acc[u].x);
        acc[u].y = fmaf(wk, o[u].y, acc[u].y);
        acc[u].z = fmaf(wk, o[u].z, acc[u].z);
        acc[u].w = fmaf(wk, o[u].w, acc[u].w);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (xr[u] >= outs) continue;
      const int row = xr[u] / (kD / 4), c4 = (xr[u] % (kD / 4)) * 4;
      const float inv = row_inv[row];
      const int i = row / P.G, g = row - i * P.G;
      const size_t qrow = (size_t)(s.row0 + i) * a.num_q_heads + kvh * P.G + g;
      *reinterpret_cast<uint2 *>(reinterpret_cast<__nv_bfloat16 *>(a.out) + qrow * kD + c4) =
          make_uint2(pack_bf16(acc[u].x * inv, acc[u].y * inv), pack_bf16(acc[u].z * inv, acc[u].w * inv));
    }
  }
}

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *q = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault, &r) ==
            cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(q);
    else
      cudaGetLastError();
  }
  return fn;
}

// The pool as a 4-D tensor (64 elements of a half row, 8 rows, 2 halves, groups
// of 8 rows), strides 256 B per row, 128 B per half, 2 KB per group: a box of R
// rows lands as R/8 groups of [half 0: 8 rows x 128 B][half 1], 128-byte swizzled.
bool pool_map(CUtensorMap *map, void *pool, const KV &kv, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t rows = (cuuint64_t)kv.num_blocks * kv.num_kv_heads * kv.block_size;
  const cuuint64_t gdim[4] = {64, 8, 2, rows / 8};
  const cuuint64_t gstride[3] = {(cuuint64_t)kD * 2, 128, (cuuint64_t)kD * 2 * 8};
  const cuuint32_t box[4] = {64, 8, 2, (cuuint32_t)box_rows / 8};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, pool, gdim, gstride, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct KeysLayout {
  int ctas, rows_cap;
  size_t lse_offset, prefix_offset, bytes;  // byte offsets in the workspace, and its size
};

KeysLayout keys_layout(const KV &kv, int num_q_heads, int max_q, int max_seq_len) {
  KeysLayout l;
  const int G = num_q_heads / kv.num_kv_heads;
  const long long max_tiles = (long long)kv.batch * kv.num_kv_heads * ((max_seq_len + kTileK - 1) / kTileK);
  l.ctas = (int)std::max(1LL, std::min<long long>(num_sms(), max_tiles));
  l.rows_cap = std::min(kRowsK, G * max_q);
  const size_t slots = (size_t)l.ctas * 2 * l.rows_cap;
  l.lse_offset = slots * kD * sizeof(float);
  l.prefix_offset = (l.lse_offset + slots * sizeof(float) + 255) / 256 * 256;
  l.bytes = l.prefix_offset + ((size_t)kv.batch + 1) * sizeof(int);
  return l;
}

}  // namespace

// Units of at most 32 rows (G * max_q); the rest as attn_umma_supported.
bool attn_keys_fits(const KV &kv, int num_q_heads, int max_q, int max_seq_len) {
  const int G = num_q_heads / kv.num_kv_heads;
  const long long max_tiles = (long long)kv.batch * kv.num_kv_heads * ((max_seq_len + kTileK - 1) / kTileK);
  return G * max_q <= kRowsK && max_tiles < (1LL << 30);
}

size_t attn_keys_workspace_bytes(const KV &kv, int num_q_heads, int max_q, int max_seq_len) {
  return keys_layout(kv, num_q_heads, max_q, max_seq_len).bytes;
}

cudaError_t launch_attn_keys(const AttnArgs &a, void *workspace, size_t workspace_bytes, cudaStream_t st) {
  if (a.kv.batch == 0) return cudaSuccess;
  const KeysLayout l = keys_layout(a.kv, a.num_q_heads, a.max_q, a.max_seq_len);
  if (workspace == nullptr || workspace_bytes < l.bytes || (uintptr_t)workspace % 256 != 0)
    return cudaErrorInvalidValue;
  KeysParams p;
  p.a = a;
  p.box_rows = a.kv.block_size < 32 ? a.kv.block_size : 32;
  p.G = a.num_q_heads / a.kv.num_kv_heads;
  p.rows_cap = l.rows_cap;
  p.ctas = l.ctas;
  p.part_o = reinterpret_cast<float *>(workspace);
  p.part_lse = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(workspace) + l.lse_offset);
  p.prefix = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(workspace) + l.prefix_offset);
  CUtensorMap mk, mv;
  if (!pool_map(&mk, a.kv.k_pool, a.kv, p.box_rows) || !pool_map(&mv, a.kv.v_pool, a.kv, p.box_rows))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_keys_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  e = launch_pdl(attn_keys_kernel, dim3(p.ctas), dim3(kThreads), kSmemBytes, st, mk, mv, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_keys_combine, dim3(a.kv.batch, a.kv.num_kv_heads), dim3(128), 0, st, p);
}

}  // namespace sv
