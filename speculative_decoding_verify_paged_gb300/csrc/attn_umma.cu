// Persistent split-KV paged attention on the 5th-generation tensor cores
// (tcgen05 + TMEM) for bf16 and E4M3 caches with head_dim 128.
//
// What it computes is the attention of the verify pass ("Speculative decoding
// and continuous batching in practice", sec. 1.2: the target scores all K+1
// positions in one pass) over the paged cache (PagedAttention section of "LLM
// serving: speculative decoding and PagedAttention memory management"), with a
// causal or a tree mask ("Speculative decoding principles and a vLLM
// production setup", sec. 3.2 and 5.2): for query row i of a sequence with c
// committed tokens, key t is visible if t < c, or if new row j = t - c is
// visible to row i (j <= i causal; bit j of the row's tree mask).
//
// Work. A unit is one sequence x one KV head x one block of up to 128 query
// rows (the G query heads of the KV head times the sequence's rows; one row
// per TMEM lane); its keys form ceil(L / 32) tiles. Two CTAs run per SM. The
// tiles of all units, laid end to end (sequence, KV head, row block order),
// are cut into equal contiguous ranges, one per CTA, so that every CTA
// streams the same number of tiles within one. A range holds whole units,
// whose rows the CTA writes itself, and at its two ends pieces of units it
// shares with its neighbours: such a piece leaves its normalised partial
// output and log-sum-exp in one of the CTA's two workspace slots (slot 0 for
// the range's first piece, slot 1 for its last), and attn_umma_combine merges
// them. Each CTA finds its range with a block scan over the sequences; CTA 0
// also stores the per-sequence tile prefix for the combine.
//
// Six warps per CTA, each walking the same pieces in the same order:
//  * warp 0, producer: TMA of 32-key K and V tiles into a 6-stage ring that
//    runs on across unit boundaries. The pool is viewed as a 4-D tensor (64
//    elements, 8 rows, 2 halves of head_dim, groups of 8 rows) so that one
//    128-byte-swizzled box brings both halves of R = min(block_size, 32) rows
//    as 1 KB atoms [8 rows of half 0][8 rows of half 1]...; block ids are
//    read 32 at a time and turned into pool rows by shift and mask;
//  * warp 1, MMA issuer (one lane) and TMEM owner: S(t) = Q K(t)^T with
//    tcgen05.mma kind::f16 (M = 128 rows, N = 32 keys, K = 128; A = Q in
//    TMEM, B = K K-major in shared memory) into one of two TMEM S buffers,
//    then O += P(t-1) V(t-1) (A = P in TMEM, B = V MN-major in shared memory,
//    N = 128; the first tile of a piece overwrites O); tcgen05.commit frees
//    the K/V stage and signals the softmax. Before the first S of a piece it
//    waits for that unit's Q;
//  * warps 2-5, softmax and epilogue: thread = query row = TMEM lane. They
//    store the unit's Q rows into TMEM (the next unit's as soon as the last S
//    of the current one has landed, prefetched into L2 one tile earlier), read
//    S(t) (tcgen05.ld), mask edge tiles, keep a running maximum that moves
//    only when the tile maximum exceeds it by more than 2^8 (then O is
//    rescaled in TMEM), write P = 2^(s - m) as bf16 over S (tcgen05.st), and
//    at the end of a piece read O, divide by the row sum and store the rows or
//    the partial result.
// An E4M3 cache (the kernel's F8 form) adds two warps: the producer's boxes
// bring rows of 128 one-byte codes into a ring of code stages, and the two
// converter warps widen each stage to fp16 (exactly, as the code's value times
// 2^-8) in the layout above, in a ring of operand stages that the MMA reads;
// Q and P are fp16, 2^8 k_scale joins the score scale and 2^8 v_scale the
// output's normalisation.
// All mbarrier waits are bounded; a wait that gives up records SV_ERR_TIMEOUT.
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <algorithm>

#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr int kD = 128;
constexpr int kTile = 32;                       // keys per tile
constexpr int kStages = 6;
constexpr int kRowsMax = 128;                   // query rows per unit (TMEM lanes)
constexpr int kSoftWarps = 4;
constexpr int kThreads = (2 + kSoftWarps) * 32;
constexpr int kHalfBytes = kTile * 128;         // 32 keys x 128 bytes (half of head_dim)
constexpr int kStageBytes = 4 * kHalfBytes;     // K and V, two halves each
constexpr int kTmemCols = 256;                  // S0 [0,32) S1 [32,64) O [64,192) Q [192,256)
constexpr int kColO = 64;
constexpr int kColQ = 192;
constexpr float kRescaleThreshold = 8.f;        // log2 units
constexpr int kCtasPerSm = 2;                   // TMEM: 2 x 256 columns; shared memory: 2 x ~100 KB
// E4M3 pools: a ring of code stages (K | V codes, 4 KB each) that the TMA fills, two converter
// warps that widen each stage to fp16 in the operand layout above, and a ring of operand stages
constexpr int kCodeStages = 6;
constexpr int kCodeHalf = kTile * 128;          // 32 keys x 128 one-byte codes
constexpr int kCodeStageBytes = 2 * kCodeHalf;  // K and V codes
constexpr int kConvStages = 3;
constexpr int kConvWarps = 2;                   // warps 6-7, after the softmax warps
// What starting and finishing a unit costs a CTA (the Q load, the pipeline refill, the last
// P V and the epilogue), in tiles: the work order gives each unit this many lead-in positions,
// so that ranges with more units hold fewer tiles.
constexpr int kUnitLeadIn = 4;

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
// One box of an E4M3 pool's (128 codes, rows) view: R rows starting at row y, 128 B each.
__device__ __forceinline__ void tma_load_codes(uint32_t dst, const CUtensorMap *map, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(y), "r"(bar)
      : "memory");
}
// One box of the (64 elements, 8 rows, 2 halves, row groups) view: R rows
// starting at row y (a multiple of 8), both halves, as R/8 groups of
// [half 0: 8 rows x 128 B][half 1: 8 rows x 128 B].
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

// Shared-memory matrix descriptor (sm_100 family): start address, leading and
// stride byte offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFF) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFF) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFF) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}
// Instruction descriptor of kind::f16: fp32 accumulate, bf16 (or fp16) A and B,
// A K-major, B K-major or MN-major, N / 8 and M / 16.
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N, int b_mn_major, bool f16 = false) {
  return (1u << 4) | (f16 ? 0u : (1u << 7) | (1u << 10)) | ((uint32_t)b_mn_major << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc, int accum) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accum));
}
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

#define SV_R8(r, o) "=r"(r[o + 0]), "=r"(r[o + 1]), "=r"(r[o + 2]), "=r"(r[o + 3]), "=r"(r[o + 4]), "=r"(r[o + 5]), \
                    "=r"(r[o + 6]), "=r"(r[o + 7])
#define SV_W8(r, o) "r"(r[o + 0]), "r"(r[o + 1]), "r"(r[o + 2]), "r"(r[o + 3]), "r"(r[o + 4]), "r"(r[o + 5]), \
                    "r"(r[o + 6]), "r"(r[o + 7])

// 32 consecutive TMEM columns of this thread's lane.
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
__device__ __forceinline__ void tmem_st64(uint32_t taddr, const uint32_t (&r)[64]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x64.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,"
      "%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,"
      "%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64};" ::"r"(taddr),
      SV_W8(r, 0), SV_W8(r, 8), SV_W8(r, 16), SV_W8(r, 24), SV_W8(r, 32), SV_W8(r, 40), SV_W8(r, 48), SV_W8(r, 56)
      : "memory");
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      SV_W8(r, 0), SV_W8(r, 8)
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
__device__ __forceinline__ uint32_t pack_f16(float lo, float hi) {
  __half2 v = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
// Two E4M3 codes of a word (bytes sel0 and sel1 of w) as an fp16 pair holding their
// values times 2^-8, exactly. Both formats put the sign on top and the exponent next,
// with biases 7 and 15 and subnormals at the lowest exponent field, so code bits
// s.eeee.mmm placed as fp16 bits s.0eeee.mmm0000000 read as the code's value times
// 2^(7-15), subnormals and zero included (the NaN codes are never stored: the append
// saturates). The byte goes to bits 8-15 of its half (prmt), the magnitude one bit down.
template <int SEL>
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2_scaled(uint32_t w) {
  const uint32_t y = __byte_perm(w, 0u, SEL);
  return (y & 0x80008000u) | ((y >> 1) & 0x3f803f80u);
}
constexpr float kF16CodeScale = 256.f;  // 2^8: what the fp16 operands above lack
// A bf16 pair as an fp16 pair (round to nearest); *over is set when a value leaves the fp16 range.
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t x, bool *over) {
  const uint32_t h = pack_f16(__uint_as_float(x << 16), __uint_as_float(x & 0xffff0000u));
  if ((h & 0x7c00u) == 0x7c00u || (h & 0x7c000000u) == 0x7c000000u) *over = true;  // inf or NaN
  return h;
}
struct UmmaParams {
  AttnArgs a;
  int box_rows;     // rows per TMA box (a group): min(block_size, 32), 16 or 32
  int G;            // query heads per KV head
  int rows_cap;     // rows of a workspace slot: min(128, G * max_q)
  int rb_max;       // row blocks of the longest sequence: ceil(G * max_q / 128)
  int ctas;         // CTAs of the launch
  int alpha;        // lead-in positions of a unit in the work order
  float *part_o;    // [ctas][2][rows_cap][128] normalised partial outputs
  float *part_lse;  // [ctas][2][rows_cap] their log-sum-exp (base 2)
  int *prefix;      // [batch + 1]: first tile of each sequence's units; [batch] = all tiles
};

// One sequence as the work decomposition sees it; tiles == 0: nothing to do.
struct Seq {
  int c, row0, n, L;
  int rbs;    // row blocks: ceil(G n / 128)
  int tiles;  // key tiles of each of its units: ceil(L / 32)
};

__device__ __forceinline__ Seq load_seq(const UmmaParams &P, int b, bool *bad) {
  const AttnArgs &a = P.a;
  const KV &kv = a.kv;
  Seq s;
  s.c = kv.seq_lens[b];
  s.row0 = a.cu_q[b];
  s.n = a.cu_q[b + 1] - s.row0;
  const long long L = (long long)s.c + s.n;
  const bool ok = s.c >= 0 && s.n >= 0 && s.n <= a.max_q && s.row0 >= 0 &&
                  (long long)s.row0 + s.n <= a.total_q && L <= a.max_seq_len &&
                  L <= (long long)kv.max_blocks * kv.block_size;
  *bad = !ok;
  s.L = ok ? (int)L : 0;
  s.rbs = ok ? (P.G * s.n + kRowsMax - 1) / kRowsMax : 0;
  s.tiles = (ok && s.rbs > 0) ? (s.L + kTile - 1) / kTile : 0;
  return s;
}
// Positions a sequence takes in the launch's work order: per unit, a lead-in of alpha
// positions (the cost of starting and finishing a unit, in tiles) and then its tiles.
__device__ __forceinline__ int seq_work(const UmmaParams &P, const Seq &s) {
  return s.tiles > 0 ? P.a.kv.num_kv_heads * s.rbs * (s.tiles + P.alpha) : 0;
}
// CTA c's positions start at range_start(c): the W positions cut as evenly as integers allow
__device__ __forceinline__ int range_start(int c, int W, int ctas) { return (int)(((long long)c * W) / ctas); }
// the CTA whose positions hold position x (0 <= x < W)
__device__ __forceinline__ int range_owner(int x, int W, int ctas) {
  return (int)((((long long)x + 1) * ctas + W - 1) / W) - 1;
}

// Inclusive sum over the CTA's threads; *total gets the sum over all of them.
template <int NT>
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
  for (int w = 0; w < NT / 32; ++w) {
    const int t = sh[w];
    before += w < warp ? t : 0;
    all += t;
  }
  __syncthreads();
  *total = all;
  return x + before;
}

// The part of one unit that lies in a CTA's tile range.
struct Piece {
  int b, kvh, rb, c, row0, n, L;
  int kt0, kt1;  // key tiles [kt0, kt1) of the unit
  bool whole;    // the piece is the whole unit
};

// Walks the tile range [g, end) piece by piece, sequence b starting at global tile `base`.
struct Walker {
  int b, base, g, end;
  Seq s;
  __device__ __forceinline__ bool next(const UmmaParams &P, Piece &p) {
    for (;;) {
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
      const int U = s.tiles + P.alpha;  // a unit's positions: lead-in, then tiles
      const int local = g - base;
      const int j = local / U, off = local - j * U;
      const int npos = min(U - off, end - g);
      g += npos;
      const int kt0 = max(0, off - P.alpha), kt1 = off + npos - P.alpha;
      if (kt1 <= 0) continue;  // only the unit's lead-in lies in this range
      p.b = b;
      p.kvh = j / s.rbs;
      p.rb = j - p.kvh * s.rbs;
      p.c = s.c;
      p.row0 = s.row0;
      p.n = s.n;
      p.L = s.L;
      p.kt0 = kt0;
      p.kt1 = kt1;
      p.whole = kt0 == 0 && kt1 == s.tiles;
      return true;
    }
  }
};

// F8: the pool holds E4M3 codes; the operands are fp16 (codes widened exactly, times 2^-8, by
// the converter warps; Q and P rounded to fp16); the scores carry 2^8 k_scale and the output
// 2^8 v_scale.
template <bool F8>
__global__ void __launch_bounds__(F8 ? kThreads + kConvWarps * 32 : kThreads, kCtasPerSm)
    attn_umma_kernel(const __grid_constant__ CUtensorMap tmap_k, const __grid_constant__ CUtensorMap tmap_v,
                     const UmmaParams P) {
  grid_dependency_wait();  // the earlier kernel on the stream is complete and visible
  grid_dependents_launch();
  constexpr int kNT = F8 ? kThreads + kConvWarps * 32 : kThreads;
  constexpr int kLS = F8 ? kCodeStages : kStages;  // stages of the ring the TMA fills
  constexpr int kLoadStageBytes = F8 ? kCodeStageBytes : kStageBytes;
  constexpr int kMS = F8 ? kConvStages : kStages;  // stages of the ring the MMA reads
  constexpr int kSoft0 = 2;                        // first softmax warp
  const AttnArgs &a = P.a;
  const KV &kv = a.kv;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = kv.batch;
  const unsigned long long wns = a.wait_ns;  // budget of the pipeline waits

  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *stages = base;  // kLS x (K | V): 16 KB of bf16 operands, or 8 KB of E4M3 codes
  uint8_t *mstages = F8 ? base + kLS * kLoadStageBytes : base;  // kMS x 16 KB operand stages
  uint64_t *full = reinterpret_cast<uint64_t *>(base + kLS * kLoadStageBytes + (F8 ? kMS * kStageBytes : 0));
  uint64_t *empty = full + kLS;
  uint64_t *s_full = empty + kLS;      // [2] S(t) in TMEM buffer t % 2
  uint64_t *p_ready = s_full + 2;      // [2] P(t) written over buffer t % 2
  uint64_t *o_bar = p_ready + 2;       // one phase per finished P V
  uint64_t *q_ready = o_bar + 1;       // one phase per unit whose Q rows are in TMEM
  uint64_t *mma_done = q_ready + 1;    // every MMA issued has finished
  uint64_t *cfull = mma_done + 1;      // [kConvStages] F8: operand stage converted
  uint64_t *cempty = cfull + kConvStages;  // [kConvStages] F8: operand stage read by its last MMA
  uint64_t *stall_bar = cempty + kConvStages;  // failure-path test: a barrier nothing arrives on
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(stall_bar + 1);
  uint64_t *mfull = F8 ? cfull : full;    // the MMA waits on these ...
  uint64_t *mempty = F8 ? cempty : empty;  // ... and frees its stages through these
  __shared__ int sh_scan[kNT / 32];
  __shared__ int sh_first_b, sh_first_base, sh_err;

  if (tid == 0) {
    for (int s = 0; s < kLS; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), F8 ? kConvWarps : 1);
    }
    if (F8)
      for (int s = 0; s < kConvStages; ++s) {
        mbar_init(smem_u32(&cfull[s]), kConvWarps);
        mbar_init(smem_u32(&cempty[s]), 1);
      }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&s_full[s]), 1);
      mbar_init(smem_u32(&p_ready[s]), kSoftWarps);
    }
    mbar_init(smem_u32(o_bar), 1);
    mbar_init(smem_u32(q_ready), kSoftWarps);
    mbar_init(smem_u32(mma_done), 1);
    mbar_init(smem_u32(stall_bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    sh_first_b = 0;
    sh_first_base = 0;
    sh_err = 0;
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }

  // ---- this CTA's tile range [g0, g1) of the W tiles of the launch ----
  int mine = 0;
  for (int b = tid; b < B; b += kNT) {
    bool bad;
    const Seq s = load_seq(P, b, &bad);
    if (bad && blockIdx.x == 0) record(a.status, SV_ERR_BAD_LENGTH);
    mine += seq_work(P, s);
  }
  int W;
  block_scan<kNT>(mine, sh_scan, &W);
  const int g0 = range_start(blockIdx.x, W, P.ctas), g1 = range_start(blockIdx.x + 1, W, P.ctas);
  int run = 0;
  for (int b0 = 0; b0 < B; b0 += kNT) {  // the sequence holding tile g0; CTA 0 also stores the prefix
    const int b = b0 + tid;
    int v = 0;
    if (b < B) {
      bool bad;
      v = seq_work(P, load_seq(P, b, &bad));
    }
    int tot;
    const int excl = run + block_scan<kNT>(v, sh_scan, &tot) - v;
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
  const uint32_t tmem = *tmem_slot;
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
    // ================= producer =================
    // Lane j copies box j of a tile (box rows of one block), K and V. The block ids come from
    // a 64-block window of the block table, two entries per lane, each loaded one window
    // before it is used and checked only then, so no load latency sits in the issue loop.
    // block_size is a power of two: logical blocks and row offsets by shift and mask
    const int bs = kv.block_size, box = P.box_rows;
    const int bs_shift = __ffs(bs) - 1;
    const uint32_t row_bytes = F8 ? 128u : 256u;  // one key's row of K (or V) as the TMA brings it
    const uint32_t box_bytes = static_cast<uint32_t>(box) * row_bytes;
    const int nboxes = kTile / box;  // 1 or 2
    if (a.stall == SV_STALL_ATTENTION) ok = __all_sync(0xffffffffu, wait_on_nothing(smem_u32(stall_bar), wns));
    Piece p;
    while (ok && walker.next(P, p)) {
      const int ke = min(p.L, p.kt1 * kTile);
      const int lb_last = (ke - 1) >> bs_shift;
      const int32_t *bt = kv.block_table + (size_t)p.b * kv.max_blocks;
      auto load_id = [&](int lb) -> int { return lb <= lb_last ? bt[lb] : -1; };
      int wbase = (p.kt0 * kTile) >> bs_shift;  // lane l holds blocks wbase + l (cur) and wbase + 32 + l (nxt)
      int cur = load_id(wbase + lane);
      int nxt = load_id(wbase + 32 + lane);
      for (int kt = p.kt0; kt < p.kt1; ++kt, ++issued) {
        const int s = issued % kLS;
        const int k0 = kt * kTile;
        while ((k0 >> bs_shift) >= wbase + 32) {  // warp-uniform
          wbase += 32;
          cur = nxt;
          nxt = load_id(wbase + 32 + lane);
        }
        const int tok = k0 + lane * box;
        const bool want = lane < nboxes && tok < ke;
        const int src = (tok >> bs_shift) - wbase;  // below 34 for a wanted box
        const int idc = __shfl_sync(0xffffffffu, cur, src & 31);
        const int idn = __shfl_sync(0xffffffffu, nxt, src & 31);
        const int id = src < 32 ? idc : idn;
        const bool bad = want && (id < 0 || id >= kv.num_blocks);
        if (bad) record(a.status, SV_ERR_BAD_BLOCK_ID);
        const bool go = want && !bad;
        const int y = ((id * kv.num_kv_heads + p.kvh) << bs_shift) + (tok & (bs - 1));
        const int nbox = __popc(__ballot_sync(0xffffffffu, go));
        if (issued >= kLS) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&empty[s]), ((issued / kLS) - 1) & 1, wns));
        if (!ok) break;
        const uint32_t fb = smem_u32(&full[s]);
        if (lane == 0) mbar_expect_tx(fb, static_cast<uint32_t>(nbox) * 2u * box_bytes);
        __syncwarp();
        const uint32_t kdst = smem_u32(stages + s * kLoadStageBytes);
        const uint32_t vdst = kdst + (F8 ? kCodeHalf : 2 * kHalfBytes);
        const uint32_t off = static_cast<uint32_t>(lane * box) * row_bytes;  // group of `box` rows
        if (go) {
          if (F8) {
            tma_load_codes(kdst + off, &tmap_k, y, fb);
            tma_load_codes(vdst + off, &tmap_v, y, fb);
          } else {
            tma_load_rows(kdst + off, &tmap_k, y, fb);
            tma_load_rows(vdst + off, &tmap_v, y, fb);
          }
        }
        __syncwarp();
      }
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    const int R = P.box_rows;  // rows per group: 16 or 32
    constexpr uint32_t idesc_s = mma_idesc(128, kTile, 0, F8);
    constexpr uint32_t idesc_o = mma_idesc(128, kD, 1, F8);
    (void)R;
    auto issue_pv = [&](int u, bool accumulate) {  // O (+)= P(u) V(u), 16 keys per MMA
      const int su = u % kMS;
      const uint32_t v_base = smem_u32(mstages + su * kStageBytes) + 2 * kHalfBytes;
      const uint32_t p_col = tmem + (u & 1) * kTile;
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)  // keys 16 kk .. 16 kk + 15: two 8-key groups of 2 KB
        mma_ts(tmem + kColO, p_col + kk * 8, smem_desc(v_base + kk * 4096, 1024, 2048), idesc_o,
               (accumulate || kk > 0) ? 1 : 0);
      mma_commit(smem_u32(&mempty[su]));
      mma_commit(smem_u32(o_bar));
    };
    int t = 0, piece = 0;
    int pend = -1;  // P V of tile t - 1 still to issue: -1 none, 0 overwrite O, 1 accumulate
    Piece p;
    while (ok && walker.next(P, p)) {
      for (int kt = p.kt0; kt < p.kt1; ++kt, ++t) {
        const int s = t % kMS;
        bool w = mbar_wait(smem_u32(&mfull[s]), (t / kMS) & 1, wns);
        if (w && kt == p.kt0) w = mbar_wait(smem_u32(q_ready), piece & 1, wns);
        ok = __all_sync(0xffffffffu, w);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t k_base = smem_u32(mstages + s * kStageBytes);
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk)  // 8-key groups 2 KB apart, half kk / 4 at +1 KB
            mma_ts(tmem + (t & 1) * kTile, tmem + kColQ + kk * 8,
                   smem_desc(k_base + (kk >> 2) * 1024 + (kk & 3) * 32, 16, 2048), idesc_s, kk > 0 ? 1 : 0);
          mma_commit(smem_u32(&s_full[t & 1]));
        }
        __syncwarp();
        if (pend >= 0) {
          const int u = t - 1;
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&p_ready[u & 1]), (u >> 1) & 1, wns));
          if (!ok) break;
          tc_fence_after();
          if (lane == 0) issue_pv(u, pend == 1);
          __syncwarp();
        }
        pend = kt != p.kt0 ? 1 : 0;
      }
      ++piece;
    }
    if (ok && pend >= 0) {
      const int u = t - 1;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&p_ready[u & 1]), (u >> 1) & 1, wns));
      if (ok) {
        tc_fence_after();
        if (lane == 0) issue_pv(u, pend == 1);
        __syncwarp();
      }
    }
    // every MMA issued finishes before TMEM is released
    if (lane == 0) mma_commit(smem_u32(mma_done));
    __syncwarp();
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(mma_done), 0, kDrainBudgetNs))) ok = false;
  } else if (warp >= kSoft0 && warp < kSoft0 + kSoftWarps) {
    // ================= softmax, one query row per thread =================
    const int q4 = warp & 3;                 // TMEM lane quarter this warp may access
    const int row = q4 * 32 + lane;          // row within the unit's row block = TMEM lane
    const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
    const __nv_bfloat16 *qsrc = reinterpret_cast<const __nv_bfloat16 *>(a.q);
    // query row (i, head g) of this lane in piece p; false for a padding lane
    auto row_of = [&](const Piece &p, int &i, int &g) -> bool {
      const int r = p.rb * kRowsMax + row;
      const bool live = r < P.G * p.n;
      i = live ? r / P.G : 0;
      g = live ? r - i * P.G : 0;
      return live;
    };
    // this lane's Q row of piece p into TMEM as bf16 pairs, fp16 pairs for F8 (zeros for a
    // padding lane); then q_ready. All 16 loads go out before the first store.
    auto load_store_q = [&](const Piece &p) {
      int i, g;
      const bool live = row_of(p, i, g);
      uint32_t qr[64];
      if (live) {
        const uint4 *qp =
            reinterpret_cast<const uint4 *>(qsrc + ((size_t)(p.row0 + i) * a.num_q_heads + p.kvh * P.G + g) * kD);
#pragma unroll
        for (int v = 0; v < 16; ++v) {
          const uint4 x = qp[v];
          qr[4 * v] = x.x;
          qr[4 * v + 1] = x.y;
          qr[4 * v + 2] = x.z;
          qr[4 * v + 3] = x.w;
        }
        if (F8) {
          bool over = false;
#pragma unroll
          for (int v = 0; v < 64; ++v) qr[v] = bf16x2_to_f16x2(qr[v], &over);
          if (over) record(a.status, SV_ERR_NONFINITE);  // a query element beyond the fp16 range
        }
      } else {
#pragma unroll
        for (int v = 0; v < 64; ++v) qr[v] = 0u;
      }
      if (__any_sync(0xffffffffu, live)) {
        tmem_st64(lane_addr + kColQ, qr);
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(q_ready));
    };
    // the next unit's Q row into L2 while this unit's last S is awaited
    auto prefetch_q = [&](const Piece &p) {
      int i, g;
      if (row_of(p, i, g)) {
        const char *qp = reinterpret_cast<const char *>(qsrc + ((size_t)(p.row0 + i) * a.num_q_heads + p.kvh * P.G + g) * kD);
        asm volatile("prefetch.global.L2 [%0];" ::"l"(qp));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(qp + 128));
      }
    };
    const float sl2 = F8 ? a.scale_log2 * (kv.k_scale * kF16CodeScale) : a.scale_log2;  // scores in log2 units
    Piece cur, nxt;
    bool has_cur = walker.next(P, cur);
    bool has_nxt = has_cur && walker.next(P, nxt);
    if (has_cur) load_store_q(cur);
    int t = 0;
    bool first_piece = true;
    while (has_cur && ok) {
      int i, g;
      const bool live = row_of(cur, i, g);
      const uint64_t tm = (live && a.mask_kind == SV_MASK_TREE) ? a.tree_mask[cur.row0 + i] : 0ull;
      const bool warp_live = __any_sync(0xffffffffu, live);
      const int c = cur.c, ke = min(cur.L, cur.kt1 * kTile);
      float m_run = -INFINITY, l_run = 0.f;
      for (int kt = cur.kt0; kt < cur.kt1; ++kt, ++t) {
        const bool handoff = kt == cur.kt1 - 1 && has_nxt;
        if (handoff) prefetch_q(nxt);
        const int k0 = kt * kTile;
        const int valid = min(kTile, ke - k0);
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&s_full[t & 1]), (t >> 1) & 1, wns));
        if (!ok) break;
        tc_fence_after();
        // S(t) was this unit's last product with its Q: the next unit's rows can take its place
        if (handoff) load_store_q(nxt);
        if (kt == cur.kt1 - 1 && t >= 1) {
          // last tile of the piece: P(t-1) V(t-1) must be done before P(t) goes out. Here
          // P V(t) cannot have started, so o_bar is in the phase of t-1 or t and the parity
          // wait is unambiguous; the end of the piece then waits for phase t alone.
          ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(o_bar), (t - 1) & 1, wns));
          if (!ok) break;
        }
        if (!F8 && valid < kTile) {
          // zero this tile's V rows past the unit's end before P V reads them (F8: the converters do)
          uint8_t *vst = stages + (t % kStages) * kStageBytes + 2 * kHalfBytes;
          for (int x = (warp - kSoft0) * 32 + lane; x < (kTile - valid) * 16; x += kSoftWarps * 32) {
            const int rr = valid + (x >> 4), ch = x & 15;
            *reinterpret_cast<uint4 *>(vst + (rr >> 3) * 2048 + (ch >> 3) * 1024 + (rr & 7) * 128 + (ch & 7) * 16) =
                make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async();
        }
        if (warp_live) {
          uint32_t sr[32];
          tmem_ld32(lane_addr + (t & 1) * kTile, sr);
          tmem_wait_ld();
          // scores in log2 units; only the last tiles of a unit (new rows, ragged end) need
          // the mask. Padding lanes (no query row) score against a zero Q row: finite values
          // whose P V rows are never stored.
          const bool edge = (k0 + kTile > c) || (valid < kTile);  // warp-uniform
          float sv[32];
          if (!edge) {
#pragma unroll
            for (int k = 0; k < kTile; ++k) sv[k] = __uint_as_float(sr[k]) * sl2;
          } else {
#pragma unroll
            for (int k = 0; k < kTile; ++k) {
              const int key = k0 + k;
              bool vis = key < ke;
              if (vis && key >= c) {
                const int j = key - c;
                vis = (a.mask_kind == SV_MASK_CAUSAL) ? (j <= i) : (j < 64 && ((tm >> j) & 1ull));
              }
              sv[k] = vis ? __uint_as_float(sr[k]) * sl2 : -INFINITY;
            }
          }
          float mx;
          {
            float t16[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) t16[k] = fmaxf(sv[k], sv[k + 16]);
#pragma unroll
            for (int w = 8; w > 0; w >>= 1)
#pragma unroll
              for (int k = 0; k < w; ++k) t16[k] = fmaxf(t16[k], t16[k + w]);
            mx = t16[0];
          }
          // move the running maximum only when the tile's exceeds it by the threshold
          const bool move = mx > m_run + kRescaleThreshold || (m_run == -INFINITY && mx != -INFINITY);
          if (__any_sync(0xffffffffu, move && l_run > 0.f)) {
            // O must be rescaled: wait for P(t-1) V(t-1) (S(t) done means P V up to t-2 is),
            // then scale this lane's row
            if (!mbar_wait(smem_u32(o_bar), (t - 1) & 1, wns)) ok = false;
            tc_fence_after();
            const float f = (move && l_run > 0.f) ? exp2f(m_run - mx) : 1.f;
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
          if (move) {
            l_run = (l_run > 0.f) ? l_run * exp2f(m_run - mx) : l_run;
            m_run = mx;
          }
          const float ref = (m_run == -INFINITY) ? 0.f : m_run;
          uint32_t pr[kTile / 2];
          float ps[kTile / 2];
#pragma unroll
          for (int k = 0; k < kTile / 2; ++k) {
            const float p0 = fast_exp2(sv[2 * k] - ref), p1 = fast_exp2(sv[2 * k + 1] - ref);
            ps[k] = p0 + p1;
            pr[k] = F8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
          }
#pragma unroll
          for (int w = 8; w > 0; w >>= 1)
#pragma unroll
            for (int k = 0; k < w; ++k) ps[k] += ps[k + w];
          l_run += ps[0];
          tmem_st16(lane_addr + (t & 1) * kTile, pr);
          tmem_wait_st();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&p_ready[t & 1]));
      }
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      // ---- end of the piece: wait for its last P V, then write ----
      // P V(tl-1) finished before P(tl) went out, and P V(tl+1) cannot start before
      // this warp's next p_ready: o_bar is in the phase of tl or tl+1.
      const int tl = t - 1;
      ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(o_bar), tl & 1, wns));
      if (!ok) break;
      tc_fence_after();
      if (warp_live) {
        const float inv = l_run > 0.f ? (F8 ? kv.v_scale * kF16CodeScale : 1.f) / l_run : 0.f;
        const size_t qrow = (size_t)(cur.row0 + i) * a.num_q_heads + cur.kvh * P.G + g;
        const size_t slot = ((size_t)blockIdx.x * 2 + (first_piece ? 0 : 1)) * P.rows_cap + row;
#pragma unroll
        for (int cb = 0; cb < kD / 32; ++cb) {
          uint32_t o[32];
          tmem_ld32(lane_addr + kColO + cb * 32, o);
          tmem_wait_ld();
          if (!live) continue;
          if (cur.whole) {
            uint4 *op = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.out) + qrow * kD + cb * 32);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              op[v] = make_uint4(pack_bf16(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv),
                                 pack_bf16(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv),
                                 pack_bf16(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv),
                                 pack_bf16(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv));
          } else {
            float4 *op = reinterpret_cast<float4 *>(P.part_o + slot * kD + cb * 32);
#pragma unroll
            for (int v = 0; v < 8; ++v)
              op[v] = make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                  __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv);
            if (cb == 0) P.part_lse[slot] = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
          }
        }
      }
      first_piece = false;
      cur = nxt;
      has_cur = has_nxt;
      has_nxt = has_cur && walker.next(P, nxt);
    }
  } else if (F8) {
    // ================= E4M3 codes -> fp16 operands =================
    // Each code stage holds K then V as rows of 128 one-byte codes; each operand stage
    // takes them in the layout the TMA gives bf16 rows (8-row groups of [half 0][half 1],
    // 16-byte chunks swizzled by the row within the group). Keys past the piece's end
    // become zero rows, so P V never reads stale values.
    constexpr int kCT = kConvWarps * 32;             // converter threads
    constexpr int kPer = (kTile * 8) / kCT;          // 16-code chunks of K (and of V) per thread and tile
    const int ct = tid - (kSoft0 + kSoftWarps) * 32;
    int t = 0;
    Piece p;
    while (ok && walker.next(P, p)) {
      const int ke = min(p.L, p.kt1 * kTile);
      for (int kt = p.kt0; kt < p.kt1; ++kt, ++t) {
        const int cs = t % kLS, ms = t % kMS;
        ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&full[cs]), (t / kLS) & 1, wns));
        if (!ok) break;
        const int valid = min(kTile, ke - kt * kTile);
        const uint8_t *src = stages + cs * kCodeStageBytes;
        uint4 x[2 * kPer];  // 16 codes each: K chunks, then V chunks
#pragma unroll
        for (int j = 0; j < 2 * kPer; ++j) {
          const int chunk = ct + kCT * (j % kPer), r = chunk >> 3, c = chunk & 7;
          x[j] = r < valid ? *reinterpret_cast<const uint4 *>(src + (j / kPer) * kCodeHalf + r * 128 + c * 16)
                           : make_uint4(0, 0, 0, 0);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[cs]));  // the codes are in registers: the stage can refill
        if (t >= kMS) ok = __all_sync(0xffffffffu, mbar_wait(smem_u32(&cempty[ms]), ((t / kMS) - 1) & 1, wns));
        if (!ok) break;
        tc_fence_after();
        uint8_t *dst = mstages + ms * kStageBytes;
#pragma unroll
        for (int j = 0; j < 2 * kPer; ++j) {
          const int half = j / kPer;               // 0: K, 1: V
          const int chunk = ct + kCT * (j % kPer);  // 16 codes: row chunk >> 3, columns 16 (chunk & 7) ..
          const int r = chunk >> 3, c = chunk & 7;
          // byte selectors: codes 0, 1 of a word -> 0x1404; codes 2, 3 -> 0x3424 (zero codes: zero rows)
          const uint4 lo = make_uint4(e4m3x2_to_f16x2_scaled<0x1404>(x[j].x), e4m3x2_to_f16x2_scaled<0x3424>(x[j].x),
                                      e4m3x2_to_f16x2_scaled<0x1404>(x[j].y), e4m3x2_to_f16x2_scaled<0x3424>(x[j].y));
          const uint4 hi = make_uint4(e4m3x2_to_f16x2_scaled<0x1404>(x[j].z), e4m3x2_to_f16x2_scaled<0x3424>(x[j].z),
                                      e4m3x2_to_f16x2_scaled<0x1404>(x[j].w), e4m3x2_to_f16x2_scaled<0x3424>(x[j].w));
          uint8_t *row = dst + half * 2 * kHalfBytes + (r >> 3) * 2048 + (c >> 2) * 1024 + (r & 7) * 128;
          const int j0 = (c & 3) * 2;  // the 16-byte chunk of columns 16 c .. 16 c + 7 within the half row
          *reinterpret_cast<uint4 *>(row + ((j0 ^ (r & 7)) << 4)) = lo;
          *reinterpret_cast<uint4 *>(row + (((j0 + 1) ^ (r & 7)) << 4)) = hi;
        }
        fence_proxy_async();  // the generic-proxy stores, visible to the tensor cores
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&cfull[ms]));
      }
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
    for (int k = max(0, issued - kLS); k < issued; ++k) mbar_wait(smem_u32(&full[k % kLS]), (k / kLS) & 1, kDrainBudgetNs);
  }
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

// Merges the partial results of every unit that two or more CTAs shared. A
// thread takes one (row, 32 head_dim elements) item and issues the loads of
// every piece's log-sum-exp and 32 partial outputs before it uses any (up to
// four pieces; more go four at a time), so a merge costs about one round trip.
__global__ void __launch_bounds__(128) attn_umma_combine(const UmmaParams P) {
  // the next kernel may launch at once (it reads before its own wait only what no kernel of the
  // library writes): the sampler's statistics can then start on the SMs the attention frees
  grid_dependents_launch();
  grid_dependency_wait();  // the earlier kernel on the stream is complete and visible
  const AttnArgs &a = P.a;
  const int b = blockIdx.x, kvh = blockIdx.y / P.rb_max, rb = blockIdx.y % P.rb_max;
  const int tid = threadIdx.x;
  const int W = P.prefix[a.kv.batch], base = P.prefix[b];  // loaded together with the sequence
  bool bad;
  const Seq s = load_seq(P, b, &bad);
  if (s.tiles == 0 || rb >= s.rbs) return;
  const int T0 = base + (kvh * s.rbs + rb) * (s.tiles + P.alpha) + P.alpha, T1 = T0 + s.tiles;  // its tiles
  const int c0 = range_owner(T0, W, P.ctas), c1 = range_owner(T1 - 1, W, P.ctas);
  if (c0 == c1) return;  // one CTA held the whole unit and wrote its rows
  // CTA c0 holds the unit as its first piece (slot 0) only when its range starts in the unit's
  // lead-in (before that come tiles of an earlier unit); every later CTA holds it as its first piece
  const int slot0 = range_start(c0, W, P.ctas) >= T0 - P.alpha ? 0 : 1;
  auto slot_of = [&](int cc, int row) -> size_t {
    return ((size_t)cc * 2 + (cc == c0 ? slot0 : 0)) * P.rows_cap + row;
  };
  constexpr int kPc = 4;  // pieces in flight
  const int rows = min(kRowsMax, P.G * s.n - rb * kRowsMax);
  for (int x = tid; x < rows * (kD / 32); x += blockDim.x) {
    const int row = x / (kD / 32), c32 = (x % (kD / 32)) * 32;
    float M = -INFINITY, den = 0.f;
    float acc[32];
#pragma unroll
    for (int k = 0; k < 32; ++k) acc[k] = 0.f;
    for (int cb = c0; cb <= c1; cb += kPc) {
      float lse[kPc];
      float4 v[kPc][8];
#pragma unroll
      for (int k = 0; k < kPc; ++k) {
        // a CTA between c0 and c1 whose range is empty (more CTAs than positions) holds nothing
        const bool in = cb + k <= c1 && range_start(cb + k, W, P.ctas) < range_start(cb + k + 1, W, P.ctas);
        const size_t sl = slot_of(in ? cb + k : cb, row);
        lse[k] = in ? __ldcg(P.part_lse + sl) : -INFINITY;
        const float4 *src = reinterpret_cast<const float4 *>(P.part_o + sl * kD + c32);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[k][j] = in ? __ldcg(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      float mn = M;
#pragma unroll
      for (int k = 0; k < kPc; ++k) mn = fmaxf(mn, lse[k]);
      if (mn == -INFINITY) continue;
      const float f = exp2f(M - mn);  // 0 while nothing was taken yet
      den *= f;
#pragma unroll
      for (int k = 0; k < 32; ++k) acc[k] *= f;
#pragma unroll
      for (int k = 0; k < kPc; ++k) {
        const float w = exp2f(lse[k] - mn);
        den += w;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          acc[4 * j] = fmaf(w, v[k][j].x, acc[4 * j]);
          acc[4 * j + 1] = fmaf(w, v[k][j].y, acc[4 * j + 1]);
          acc[4 * j + 2] = fmaf(w, v[k][j].z, acc[4 * j + 2]);
          acc[4 * j + 3] = fmaf(w, v[k][j].w, acc[4 * j + 3]);
        }
      }
      M = mn;
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    const int r = rb * kRowsMax + row, i = r / P.G, g = r - i * P.G;
    const size_t qrow = (size_t)(s.row0 + i) * a.num_q_heads + kvh * P.G + g;
    uint4 *op = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.out) + qrow * kD + c32);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      op[j] = make_uint4(pack_bf16(acc[8 * j] * inv, acc[8 * j + 1] * inv), pack_bf16(acc[8 * j + 2] * inv, acc[8 * j + 3] * inv),
                         pack_bf16(acc[8 * j + 4] * inv, acc[8 * j + 5] * inv),
                         pack_bf16(acc[8 * j + 6] * inv, acc[8 * j + 7] * inv));
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
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    else
      cudaGetLastError();
  }
  return fn;
}

// The pool as a 4-D tensor: (64 elements of a half row, 8 rows, 2 halves,
// groups of 8 rows) with strides (256 B per row, 128 B per half, 2 KB per
// group); a box of R rows lands as R/8 groups of [half 0: 8 rows x 128 B]
// [half 1: 8 rows x 128 B], 128-byte swizzled: every 1 KB is one swizzle
// atom, and the atoms of one half are 2 KB apart across the whole tile.
//
// An E4M3 pool is a 2-D tensor (128 one-byte codes, rows) read without swizzle: a
// box of R rows lands as R rows of 128 B.
bool make_map(CUtensorMap *map, void *pool, const KV &kv, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t rows = (cuuint64_t)kv.num_blocks * kv.num_kv_heads * kv.block_size;
  if (kv.fp8) {
    const cuuint64_t gdim[2] = {(cuuint64_t)kD, rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)kD};
    const cuuint32_t box[2] = {(cuuint32_t)kD, (cuuint32_t)box_rows};
    const cuuint32_t estride[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, pool, gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  }
  const cuuint64_t gdim[4] = {64, 8, 2, rows / 8};
  const cuuint64_t gstride[3] = {(cuuint64_t)kD * 2, 128, (cuuint64_t)kD * 2 * 8};
  const cuuint32_t box[4] = {64, 8, 2, (cuuint32_t)box_rows / 8};
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, pool, gdim, gstride, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 6 stages of 16 KB (E4M3: 4 code stages of 8 KB and 4 operand stages of 16 KB); at most two
// CTAs fit an SM, which is what TMEM allows (2 x 256 columns)
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + 32 * 8;
static_assert(kCodeStages * kCodeStageBytes + kConvStages * kStageBytes <= kStages * kStageBytes,
              "the E4M3 rings fit the bf16 ring's space");
static_assert(2 * (kStages > kCodeStages ? kStages : kCodeStages) + 2 * kConvStages + 8 <= 31,
              "barriers and the TMEM slot fit 256 B");
static_assert(3 * (kSmemBytes + 1024) > 228 * 1024, "a third CTA per SM would wait for TMEM");

struct UmmaLayout {
  int ctas, rows_cap, rb_max;
  size_t lse_offset, prefix_offset, bytes;  // byte offsets in the workspace, and its size
};

UmmaLayout umma_layout(const KV &kv, int num_q_heads, int max_q, int max_seq_len) {
  UmmaLayout l;
  const int G = num_q_heads / kv.num_kv_heads;
  const long long max_tiles =
      (long long)kv.batch * kv.num_kv_heads * ((G * max_q + kRowsMax - 1) / kRowsMax) * ((max_seq_len + kTile - 1) / kTile);
  l.ctas = (int)std::max(1LL, std::min<long long>((long long)kCtasPerSm * num_sms(), max_tiles));
  l.rows_cap = std::min(kRowsMax, G * max_q);
  l.rb_max = (G * max_q + kRowsMax - 1) / kRowsMax;
  const size_t slots = (size_t)l.ctas * 2 * l.rows_cap;
  l.lse_offset = slots * kD * sizeof(float);
  l.prefix_offset = (l.lse_offset + slots * sizeof(float) + 255) / 256 * 256;
  l.bytes = l.prefix_offset + ((size_t)kv.batch + 1) * sizeof(int);
  return l;
}

}  // namespace

bool attn_umma_supported(const KV &kv) {
  // TMA row coordinates are 32-bit: the pool's rows (blocks x KV heads x block_size) must fit
  const long long rows = (long long)kv.num_blocks * kv.num_kv_heads * kv.block_size;
  return (kv.elem_bytes == 2 || kv.fp8) && kv.head_dim == kD && kv.block_size >= 16 && kv.block_size <= 256 &&
         (kv.block_size & (kv.block_size - 1)) == 0 && rows < (1LL << 31) &&
         encode_fn() != nullptr && ((uintptr_t)kv.k_pool % 16 == 0) && ((uintptr_t)kv.v_pool % 16 == 0);
}

bool attn_umma_fits(const KV &kv, int num_q_heads, int max_q, int max_seq_len) {
  const int G = num_q_heads / kv.num_kv_heads;
  const long long units = (long long)kv.batch * kv.num_kv_heads * ((G * max_q + kRowsMax - 1) / kRowsMax);
  const long long positions = units * (((max_seq_len + kTile - 1) / kTile) + kUnitLeadIn);
  return positions < (1LL << 30);
}

size_t attn_umma_workspace_bytes(const KV &kv, int num_q_heads, int max_q, int max_seq_len) {
  return umma_layout(kv, num_q_heads, max_q, max_seq_len).bytes;
}

cudaError_t launch_attn_umma(const AttnArgs &a, void *workspace, size_t workspace_bytes, cudaStream_t st) {
  if (a.kv.batch == 0) return cudaSuccess;
  const UmmaLayout l = umma_layout(a.kv, a.num_q_heads, a.max_q, a.max_seq_len);
  if (workspace == nullptr || workspace_bytes < l.bytes || (uintptr_t)workspace % 256 != 0)
    return cudaErrorInvalidValue;
  UmmaParams p;
  p.a = a;
  p.box_rows = a.kv.block_size < kTile ? a.kv.block_size : kTile;
  p.G = a.num_q_heads / a.kv.num_kv_heads;
  p.rows_cap = l.rows_cap;
  p.rb_max = l.rb_max;
  p.ctas = l.ctas;
  p.alpha = kUnitLeadIn;
  p.part_o = reinterpret_cast<float *>(workspace);
  p.part_lse = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(workspace) + l.lse_offset);
  p.prefix = reinterpret_cast<int *>(reinterpret_cast<uint8_t *>(workspace) + l.prefix_offset);
  CUtensorMap mk, mv;
  if (!make_map(&mk, a.kv.k_pool, a.kv, p.box_rows) || !make_map(&mv, a.kv.v_pool, a.kv, p.box_rows))
    return cudaErrorInvalidValue;
  auto kernel = a.kv.fp8 ? attn_umma_kernel<true> : attn_umma_kernel<false>;
  const int threads = a.kv.fp8 ? kThreads + kConvWarps * 32 : kThreads;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  e = launch_pdl(kernel, dim3(p.ctas), dim3(threads), kSmemBytes, st, mk, mv, p);
  if (e != cudaSuccess) return e;
  return launch_pdl(attn_umma_combine, dim3(a.kv.batch, a.kv.num_kv_heads * p.rb_max), dim3(128), 0, st, p);
}

}  // namespace sv
