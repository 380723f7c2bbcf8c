// Split-KV paged attention on the 5th-generation tensor cores (tcgen05 + TMEM)
// for bf16 caches with head_dim 128.
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
// One CTA = one sequence x one KV head x one split of its keys x up to 128
// query rows (the G query heads of the KV head times the sequence's rows, one
// row per TMEM lane). Six warps:
//  * warp 0, producer: TMA of 32-key K and V tiles into a 6-stage ring. The
//    pool is viewed as a 3-D tensor (64 elements, rows, 2 halves of
//    head_dim) so that one 128-byte-swizzled box brings both halves of a
//    group of R = min(block_size, 32) rows: a tile is 32/R groups, each
//    stored [half 0 | half 1]; block ids are read 32 at a time;
//  * warp 1, MMA issuer (one lane) and TMEM owner: S(t) = Q K(t)^T with
//    tcgen05.mma kind::f16 (M = 128 rows, N = R keys per group, K = 128; A = Q
//    in TMEM, B = K K-major in shared memory) into one of two TMEM S buffers,
//    then
//    O += P(t-1) V(t-1) (A = P in TMEM, B = V MN-major in shared memory,
//    N = 128); tcgen05.commit frees the K/V stage and signals the softmax;
//  * warps 2-5, softmax and epilogue: thread = query row = TMEM lane. Each
//    first stores its row of Q into TMEM (the tensor core then reads Q from
//    TMEM instead of shared memory), reads its row of S(t) (tcgen05.ld),
//    masks edge tiles, keeps a running
//    maximum that moves only when the tile maximum exceeds it by more than
//    2^8 (then O is rescaled in TMEM), writes P = 2^(s - m) as bf16 over S
//    (tcgen05.st), and at the end reads O, divides by the row sum and stores
//    the row (or the split's partial result and log-sum-exp).
// All mbarrier waits are bounded; a wait that gives up records SV_ERR_TIMEOUT.
#include <cuda.h>

#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr int kD = 128;
constexpr int kTile = 32;                       // keys per tile
constexpr int kStages = 6;
constexpr int kRowsMax = 128;                   // query rows per CTA (TMEM lanes)
constexpr int kSoftWarps = 4;
constexpr int kThreads = (2 + kSoftWarps) * 32;
constexpr int kHalfBytes = kTile * 128;         // 32 keys x 128 bytes (half of head_dim)
constexpr int kStageBytes = 4 * kHalfBytes;     // K and V, two halves each
constexpr int kTmemCols = 256;                  // S0 [0,32) S1 [32,64) O [64,192) Q [192,256)
constexpr int kColO = 64;
constexpr int kColQ = 192;
constexpr float kRescaleThreshold = 8.f;        // log2 units
constexpr long long kSpinLimit = 1LL << 24;

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
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  for (long long i = 0; i < kSpinLimit; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    if (ok) return true;
  }
  return false;
}
// One box of the (64 elements, rows, 2 halves) view: R rows, both halves.
__device__ __forceinline__ void tma_load_rows(uint32_t dst, const CUtensorMap *map, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(y), "r"(0), "r"(bar)
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
// Instruction descriptor of kind::f16: fp32 accumulate, bf16 A and B, A K-major,
// B K-major or MN-major, N / 8 and M / 16.
__host__ __device__ constexpr uint32_t mma_idesc(int M, int N, int b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn_major << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
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

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}
struct UmmaParams {
  AttnArgs a;
  int box_rows;    // rows per TMA box (a group): min(block_size, 32), 16 or 32
  int row_blocks;  // CTAs per (sequence, KV head, split) along the query rows
};

__global__ void __launch_bounds__(kThreads, 2) attn_umma_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                                                const __grid_constant__ CUtensorMap tmap_v,
                                                                const UmmaParams P) {
  const AttnArgs &a = P.a;
  const KV &kv = a.kv;
  const int split = blockIdx.x;
  const int kvh = blockIdx.y / P.row_blocks, rb = blockIdx.y % P.row_blocks;
  const int b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  const int c = kv.seq_lens[b];
  const int row0 = a.cu_q[b];
  const int n = a.cu_q[b + 1] - row0;
  const int L = c + n;
  if (L > a.max_seq_len || c < 0 || n < 0 || row0 + n > a.total_q || L > kv.max_blocks * kv.block_size) {
    if (split == 0 && blockIdx.y == 0 && tid == 0) record(a.status, SV_ERR_BAD_LENGTH);
    return;
  }
  const int nsplit = (L + a.chunk - 1) / a.chunk;
  if (split >= nsplit) return;
  const int G = a.num_q_heads / kv.num_kv_heads;
  const int R = G * n;
  const int rbase = rb * kRowsMax;
  if (rbase >= R) return;
  const int kb = split * a.chunk, ke = min(L, kb + a.chunk);
  const int ntiles = (ke - kb + kTile - 1) / kTile;

  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *stages = base;  // kStages x (K 8 KB | V 8 KB)
  uint64_t *full = reinterpret_cast<uint64_t *>(stages + kStages * kStageBytes);
  uint64_t *empty = full + kStages;
  uint64_t *s_full = empty + kStages;  // [2] S(t) in TMEM buffer t % 2
  uint64_t *p_ready = s_full + 2;      // [2] P(t) written over buffer t % 2
  uint64_t *o_bar = p_ready + 2;       // one phase per finished P V
  uint64_t *q_ready = o_bar + 1;       // Q rows stored in TMEM
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(q_ready + 1);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_u32(&s_full[s]), 1);
      mbar_init(smem_u32(&p_ready[s]), kSoftWarps);
    }
    mbar_init(smem_u32(o_bar), 1);
    mbar_init(smem_u32(q_ready), kSoftWarps);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;

  if (warp == 0) {
    // ================= producer =================
    const int bs = kv.block_size, box = P.box_rows;
    const uint32_t box_bytes = static_cast<uint32_t>(box) * 256;
    const int lb_first = kb / bs, lb_last = (ke - 1) / bs;
    const int32_t *bt = kv.block_table + (size_t)b * kv.max_blocks;
    auto load_id = [&](int lb) -> int {
      if (lb > lb_last) return -1;
      const int id = bt[lb];
      if (id < 0 || id >= kv.num_blocks) {
        record(a.status, SV_ERR_BAD_BLOCK_ID);
        return -1;
      }
      return id;
    };
    int wbase = lb_first;
    int cur = load_id(wbase + lane);
    int nxt = load_id(wbase + 32 + lane);
    for (int t = 0; t < ntiles && ok; ++t) {
      const int s = t % kStages;
      if (t >= kStages && !mbar_wait(smem_u32(&empty[s]), ((t / kStages) - 1) & 1)) {
        ok = false;
        break;
      }
      const int kt = kb + t * kTile;
      int ids[kTile / 16];
      int nbox = 0;
      for (int r = 0; r < kTile; r += box) {
        const int tok = kt + r;
        int id = -1;
        if (tok < ke) {
          const int lb = tok / bs;
          while (lb >= wbase + 32) {  // warp-uniform
            wbase += 32;
            cur = nxt;
            nxt = load_id(wbase + 32 + lane);
          }
          id = __shfl_sync(0xffffffffu, cur, lb - wbase);
        }
        ids[r / box] = id;
        nbox += id >= 0;
      }
      if (lane == 0) {
        const uint32_t fb = smem_u32(&full[s]);
        mbar_expect_tx(fb, static_cast<uint32_t>(nbox) * 2u * box_bytes);
        const uint32_t kdst = smem_u32(stages + s * kStageBytes);
        const uint32_t vdst = kdst + 2 * kHalfBytes;
        for (int r = 0; r < kTile; r += box) {
          const int id = ids[r / box];
          if (id < 0) continue;
          const int tok = kt + r;
          const int y = (id * kv.num_kv_heads + kvh) * bs + (tok % bs);
          const uint32_t off = static_cast<uint32_t>(r) * 256;  // group of `box` rows, both halves
          tma_load_rows(kdst + off, &tmap_k, y, fb);
          tma_load_rows(vdst + off, &tmap_v, y, fb);
        }
      }
      __syncwarp();
    }
  } else if (warp == 1) {
    // ================= MMA issuer =================
    const int R = P.box_rows;            // rows per group: 16 or 32
    const uint32_t idesc_s = mma_idesc(128, R, 0);
    constexpr uint32_t idesc_o = mma_idesc(128, kD, 1);
    const uint32_t half_bytes = static_cast<uint32_t>(R) * 128;  // one half of a group
    auto issue_pv = [&](int u) {  // O += P(u) V(u), 16 keys per MMA
      const int su = u % kStages;
      const uint32_t v_base = smem_u32(stages + su * kStageBytes) + 2 * kHalfBytes;
      const uint32_t p_col = tmem + (u & 1) * kTile;
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) {
        const int grp = (kk * 16) / R, sub = ((kk * 16) % R) / 16;
        const uint32_t start = v_base + grp * 2 * half_bytes + sub * 2048;
        mma_ts(tmem + kColO, p_col + kk * 8, smem_desc(start, half_bytes, 1024), idesc_o, (u > 0 || kk > 0) ? 1 : 0);
      }
      mma_commit(smem_u32(&empty[su]));
      mma_commit(smem_u32(o_bar));
    };
    ok = mbar_wait(smem_u32(q_ready), 0);
    tc_fence_after();
    for (int t = 0; t <= ntiles && ok; ++t) {
      if (t < ntiles) {
        const int s = t % kStages;
        ok = mbar_wait(smem_u32(&full[s]), (t / kStages) & 1);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) {
          const uint32_t k_base = smem_u32(stages + s * kStageBytes);
          for (int grp = 0; grp < kTile / R; ++grp) {
            const uint32_t kg = k_base + grp * 2 * half_bytes;
#pragma unroll
            for (int kk = 0; kk < kD / 16; ++kk)
              mma_ts(tmem + (t & 1) * kTile + grp * R, tmem + kColQ + kk * 8,
                     smem_desc(kg + (kk >> 2) * half_bytes + (kk & 3) * 32, 16, 1024), idesc_s, kk > 0 ? 1 : 0);
          }
          mma_commit(smem_u32(&s_full[t & 1]));
        }
        __syncwarp();
      }
      if (t > 0) {
        const int u = t - 1;
        ok = mbar_wait(smem_u32(&p_ready[u & 1]), (u >> 1) & 1);
        if (!ok) break;
        tc_fence_after();
        if (lane == 0) issue_pv(u);
        __syncwarp();
      }
    }
  } else {
    // ================= softmax, one query row per thread =================
    const int q4 = warp & 3;                 // TMEM lane quarter this warp may access
    const int row = q4 * 32 + lane;          // row within the CTA = TMEM lane
    const int r = rbase + row;
    const bool live = r < R;
    const int i = live ? r / G : 0;
    const uint64_t tm = (live && a.mask_kind == SV_MASK_TREE) ? a.tree_mask[row0 + i] : 0ull;
    const uint32_t lane_addr = tmem + ((uint32_t)(q4 * 32) << 16);
    const bool warp_live = __any_sync(0xffffffffu, live);
    if (warp_live) {
      // this lane's query row into TMEM columns [kColQ, kColQ + 64): bf16 pairs, zeros for padding rows
      uint32_t qr[64];
      if (live) {
        const uint4 *qp = reinterpret_cast<const uint4 *>(reinterpret_cast<const __nv_bfloat16 *>(a.q) +
                                                          ((size_t)(row0 + i) * a.num_q_heads + kvh * G + r % G) * kD);
#pragma unroll
        for (int v = 0; v < 16; ++v) {
          const uint4 x = qp[v];
          qr[4 * v] = x.x;
          qr[4 * v + 1] = x.y;
          qr[4 * v + 2] = x.z;
          qr[4 * v + 3] = x.w;
        }
      } else {
#pragma unroll
        for (int v = 0; v < 64; ++v) qr[v] = 0u;
      }
      tmem_st64(lane_addr + kColQ, qr);
      tmem_wait_st();
    }
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(q_ready));
    float m_run = -INFINITY, l_run = 0.f;
    for (int t = 0; t < ntiles; ++t) {
      const int kt = kb + t * kTile;
      const int valid = min(kTile, ke - kt);
      ok = mbar_wait(smem_u32(&s_full[t & 1]), (t >> 1) & 1);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after();
      if (valid < kTile) {
        // zero this tile's V rows past the split's end before P V reads them
        uint8_t *vst = stages + (t % kStages) * kStageBytes + 2 * kHalfBytes;
        const int R = P.box_rows;
        for (int x = (warp - 2) * 32 + lane; x < (kTile - valid) * 16; x += kSoftWarps * 32) {
          const int rr = valid + (x >> 4), ch = x & 15;
          const int grp = rr / R, rin = rr % R;
          *reinterpret_cast<uint4 *>(vst + grp * 2 * R * 128 + (ch >> 3) * R * 128 + rin * 128 + (ch & 7) * 16) =
              make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async();
      }
      if (warp_live) {
        uint32_t sr[32];
        tmem_ld32(lane_addr + (t & 1) * kTile, sr);
        tmem_wait_ld();
        const bool edge = (kt + kTile > c) || (valid < kTile);
        float sv[32];
#pragma unroll
        for (int k = 0; k < kTile; ++k) {
          float v = __uint_as_float(sr[k]) * a.scale_log2;
          if (edge) {
            const int key = kt + k;
            bool vis = live && key < ke;
            if (vis && key >= c) {
              const int j = key - c;
              vis = (a.mask_kind == SV_MASK_CAUSAL) ? (j <= i) : (j < 64 && ((tm >> j) & 1ull));
            }
            if (!vis) v = -INFINITY;
          }
          if (!live) v = -INFINITY;
          sv[k] = v;
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
          // O must be rescaled: wait for P(t-1) V(t-1), then scale this lane's row
          if (t > 0 && !mbar_wait(smem_u32(o_bar), (t - 1) & 1)) ok = false;
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
          const float p0 = exp2f(sv[2 * k] - ref), p1 = exp2f(sv[2 * k + 1] - ref);
          ps[k] = p0 + p1;
          pr[k] = pack_bf16(p0, p1);
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
    // ---- epilogue: wait for the last P V, then write the row ----
    // S(t) is issued before P(t-1) V(t-1), so seeing S(ntiles-1) proves only
    // that P V up to ntiles-3 finished: o_bar may still be in the phase of
    // ntiles-2, and a parity wait for ntiles-1 alone would pass early there.
    if (ok && ntiles > 1) ok = mbar_wait(smem_u32(o_bar), (ntiles - 2) & 1);
    if (ok && ntiles > 0) ok = mbar_wait(smem_u32(o_bar), (ntiles - 1) & 1);
    ok = __all_sync(0xffffffffu, ok);
    tc_fence_after();
    if (ok && warp_live) {
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const int g = live ? r % G : 0;
      const size_t qrow = (size_t)(row0 + i) * a.num_q_heads + kvh * G + g;
#pragma unroll
      for (int cb = 0; cb < kD / 32; ++cb) {
        uint32_t o[32];
        tmem_ld32(lane_addr + kColO + cb * 32, o);
        tmem_wait_ld();
        if (!live) continue;
        if (nsplit == 1) {
          uint4 *op = reinterpret_cast<uint4 *>(reinterpret_cast<__nv_bfloat16 *>(a.out) + qrow * kD + cb * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            op[v] = make_uint4(pack_bf16(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv),
                               pack_bf16(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv),
                               pack_bf16(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv),
                               pack_bf16(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv));
        } else {
          const size_t prow = (size_t)split * a.total_q * a.num_q_heads + qrow;
          float4 *op = reinterpret_cast<float4 *>(a.ws_o + prow * kD + cb * 32);
#pragma unroll
          for (int v = 0; v < 8; ++v)
            op[v] = make_float4(__uint_as_float(o[4 * v]) * inv, __uint_as_float(o[4 * v + 1]) * inv,
                                __uint_as_float(o[4 * v + 2]) * inv, __uint_as_float(o[4 * v + 3]) * inv);
          if (cb == 0) a.ws_lse[prow] = l_run > 0.f ? m_run + log2f(l_run) : -INFINITY;
        }
      }
    }
  }
  if (!ok && lane == 0) record(a.status, SV_ERR_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
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

// The pool as a 3-D tensor: (64 elements of a half row, rows, 2 halves) with
// strides (256 B per row, 128 B per half); a box of R rows lands as
// [half 0: R rows x 128 B][half 1: R rows x 128 B], 128-byte swizzled.
bool make_map(CUtensorMap *map, void *pool, const KV &kv, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t rows = (cuuint64_t)kv.num_blocks * kv.num_kv_heads * kv.block_size;
  const cuuint64_t gdim[3] = {64, rows, 2};
  const cuuint64_t gstride[2] = {(cuuint64_t)kD * 2, 128};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 2};
  const cuuint32_t estride[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, pool, gdim, gstride, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 6 stages of 16 KB; at most two CTAs fit an SM, which is what TMEM allows (2 x 256 columns)
constexpr size_t kSmemBytes = 1024 + (size_t)kStages * kStageBytes + 32 * 8;
static_assert(3 * (kSmemBytes + 1024) > 228 * 1024, "a third CTA per SM would wait for TMEM");

}  // namespace

bool attn_umma_supported(const KV &kv) {
  return kv.elem_bytes == 2 && kv.head_dim == kD && kv.block_size >= 16 && kv.block_size <= 256 &&
         encode_fn() != nullptr && ((uintptr_t)kv.k_pool % 16 == 0) && ((uintptr_t)kv.v_pool % 16 == 0);
}

cudaError_t launch_attn_umma(const AttnArgs &a, cudaStream_t st) {
  if (a.kv.batch == 0) return cudaSuccess;
  UmmaParams p;
  p.a = a;
  p.box_rows = a.kv.block_size < kTile ? a.kv.block_size : kTile;
  const int G = a.num_q_heads / a.kv.num_kv_heads;
  p.row_blocks = (G * a.max_q + kRowsMax - 1) / kRowsMax;
  CUtensorMap mk, mv;
  if (!make_map(&mk, a.kv.k_pool, a.kv, p.box_rows) || !make_map(&mv, a.kv.v_pool, a.kv, p.box_rows))
    return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(attn_umma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
  if (e != cudaSuccess) return e;
  dim3 grid(a.max_splits, a.kv.num_kv_heads * p.row_blocks, a.kv.batch);
  attn_umma_kernel<<<grid, kThreads, kSmemBytes, st>>>(mk, mv, p);
  return cudaGetLastError();
}

}  // namespace sv
