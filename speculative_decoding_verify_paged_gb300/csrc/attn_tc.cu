// Split-KV paged attention on tensor cores for bf16 caches with head_dim 128.
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
// Design (one CTA = one sequence x one KV head x one split of its keys x up to
// 64 query rows, i.e. the G query heads sharing the KV head times the rows of
// the sequence):
//  * a producer warp streams 64-token K and V tiles into a 3-stage ring with
//    TMA (cp.async.bulk.tensor.2d over the pool viewed as [rows, 128] bf16,
//    128-byte swizzle, one box per (physical block, half of head_dim));
//    mbarriers with transaction counts signal "full", consumer arrivals
//    signal "empty"; every wait is bounded;
//  * consumer warps (4 by default): S = Q K^T with bf16 mma.sync m16n8k16
//    (warp w takes an equal slice of the tile's keys for all rows), online
//    softmax in base 2 with the running max shared through shared memory,
//    P (bf16) to shared memory, then O += P V with warp w taking an equal
//    slice of the output columns;
//  * the final tile of a split zeroes the V rows past the split's end before
//    P V (pool slots past a sequence's length hold arbitrary bytes).
// Partial results of multi-split sequences go to the workspace in the same
// layout as the CUDA-core path; the shared combine kernel merges them.
#include <cuda.h>

#include "sv_internal.cuh"

namespace sv {
namespace {

constexpr int kD = 128;
constexpr int kTile = 64;  // keys per tile
// Ring depth and consumer warps are build-time constants (defaults below).
#ifndef SV_ATTN_STAGES
#define SV_ATTN_STAGES 3
#endif
#ifndef SV_ATTN_CONSUMER_WARPS
#define SV_ATTN_CONSUMER_WARPS 4
#endif
constexpr int kStages = SV_ATTN_STAGES;
constexpr int kConsumerWarps = SV_ATTN_CONSUMER_WARPS;  // 4 or 8
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kKeysPerWarp = kTile / kConsumerWarps;  // S = Q K^T: keys per warp
constexpr int kNtS = kKeysPerWarp / 8;                // n8 tiles of keys per warp
constexpr int kColsPerWarp = kD / kConsumerWarps;      // O += P V: output columns per warp
constexpr int kNtO = kColsPerWarp / 8;                 // n8 tiles of columns per warp
static_assert(kConsumerWarps == 4 || kConsumerWarps == 8, "4 or 8 consumer warps");
constexpr int kStageBytes = 2 * kTile * kD * 2;  // K and V
constexpr int kHalfBytes = kTile * 128;          // 64 rows x 128 bytes (half of head_dim)

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
// Bounded wait for the phase with the given parity; false after the limit.
// This kernel's consumers leave without draining the copies still in flight when a wait gives
// up, so every wait keeps the long budget kDrainBudgetNs (the pipeline budget option does not
// apply here): a wait gives up only when a copy has not landed after half a second.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, unsigned long long budget) {
  return mbar_wait_bounded(bar, parity, budget);
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap *map, int x, int y, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory"); }
// Barrier of the consumer warps that also ORs a flag over them.
__device__ __forceinline__ bool consumers_sync_or(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 1, %2, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v), "n"(kConsumerWarps * 32)
      : "memory");
  return r != 0;
}
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t &r0, uint32_t &r1) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0, %1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
      "{%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` in a 128-byte-swizzled
// region of 128-byte rows (the layout TMA writes with SWIZZLE_128B).
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

struct TcParams {
  AttnArgs a;
  int box_rows;   // rows per TMA box: min(block_size, 64)
  int row_blocks; // CTAs per (sequence, KV head, split) along the query rows
};

template <int RG /* 16-row groups per CTA */>
__global__ void __launch_bounds__(kThreads) attn_tc_kernel(const __grid_constant__ CUtensorMap tmap_k,
                                                           const __grid_constant__ CUtensorMap tmap_v,
                                                           const TcParams P) {
  grid_dependency_wait();  // the earlier kernel on the stream is complete and visible
  grid_dependents_launch();
  constexpr int kRows = 16 * RG;
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
  const int rbase = rb * kRows;
  if (rbase >= R) return;
  const int kb = split * a.chunk, ke = min(L, kb + a.chunk);
  const int ntiles = (ke - kb + kTile - 1) / kTile;

  // ---- shared memory carve-up (1024-byte aligned for the 128B swizzle) ----
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t *stages = base;                                     // kStages x (K 16 KB | V 16 KB)
  uint8_t *q_s = stages + kStages * kStageBytes;              // 2 halves x kRows x 128 B
  uint8_t *p_s = q_s + 2 * kRows * 128;                       // kRows x 128 B (64 keys)
  float *red_max = reinterpret_cast<float *>(p_s + kRows * 128);  // [4][kRows]
  float *red_l = red_max + kConsumerWarps * kRows;                // [4][kRows]
  uint64_t *full = reinterpret_cast<uint64_t *>(red_l + kConsumerWarps * kRows);
  uint64_t *empty = full + kStages;

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(&full[s]), 1);
      mbar_init(smem_u32(&empty[s]), kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ================= producer: TMA K/V tiles into the ring =================
    // The split's physical block ids are read 32 at a time (one per lane) into
    // registers, with the next window in flight while the current one is used;
    // lane 0 picks ids by shuffle and issues the copies.
    const int bs = kv.block_size, box = P.box_rows;
    const uint32_t box_bytes = static_cast<uint32_t>(box) * 128;
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
    for (int t = 0; t < ntiles; ++t) {
      const int s = t % kStages;
      if (t >= kStages && !mbar_wait(smem_u32(&empty[s]), ((t / kStages) - 1) & 1, kDrainBudgetNs)) {
        if (lane == 0) record(a.status, SV_ERR_TIMEOUT);
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
        mbar_expect_tx(fb, static_cast<uint32_t>(nbox) * 4u * box_bytes);
        const uint32_t kdst = smem_u32(stages + s * kStageBytes);
        const uint32_t vdst = kdst + kStageBytes / 2;
        for (int r = 0; r < kTile; r += box) {
          const int id = ids[r / box];
          if (id < 0) continue;
          const int tok = kt + r;
          const int y = (id * kv.num_kv_heads + kvh) * bs + (tok % bs);
          const uint32_t off = static_cast<uint32_t>(r) * 128;
          tma_load_2d(kdst + off, &tmap_k, 0, y, fb);
          tma_load_2d(kdst + kHalfBytes + off, &tmap_k, 64, y, fb);
          tma_load_2d(vdst + off, &tmap_v, 0, y, fb);
          tma_load_2d(vdst + kHalfBytes + off, &tmap_v, 64, y, fb);
        }
      }
      __syncwarp();
    }
    return;
  }

  // ================= consumers =================
  // Q rows rbase .. rbase+kRows-1 of this (sequence, KV head): row r -> position
  // r / G, query head kvh*G + r % G. Rows past R are zero and never written.
  {
    const __nv_bfloat16 *qp = reinterpret_cast<const __nv_bfloat16 *>(a.q);
    for (int x = tid; x < kRows * 16; x += kConsumerWarps * 32) {
      const int rr = x >> 4, ch = x & 15, r = rbase + rr;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (r < R) {
        const int i = r / G, g = r % G;
        v = *reinterpret_cast<const uint4 *>(qp + ((size_t)(row0 + i) * a.num_q_heads + kvh * G + g) * kD + ch * 8);
      }
      *reinterpret_cast<uint4 *>(q_s + (ch >> 3) * (kRows * 128) + swz(rr, ch & 7)) = v;
    }
  }
  consumers_sync();

  // per-thread row bookkeeping: the thread holds rows (mt*16 + lane/4 + 8*h)
  const int qr = lane >> 2, qc = lane & 3;
  float m_run[RG][2], l_run[RG][2];
  int pos_of[RG][2];
  uint64_t tmask_of[RG][2];
#pragma unroll
  for (int mt = 0; mt < RG; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      m_run[mt][h] = -INFINITY;
      l_run[mt][h] = 0.f;
      const int r = rbase + mt * 16 + qr + 8 * h;
      pos_of[mt][h] = r < R ? r / G : -1;
      tmask_of[mt][h] = (r < R && a.mask_kind == SV_MASK_TREE) ? a.tree_mask[row0 + r / G] : 0ull;
    }
  float o_acc[RG][kNtO][4];
#pragma unroll
  for (int mt = 0; mt < RG; ++mt)
#pragma unroll
    for (int nt = 0; nt < kNtO; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o_acc[mt][nt][e] = 0.f;

  const uint32_t q_base = smem_u32(q_s), p_base = smem_u32(p_s);
  bool ok = true;
  for (int t = 0; t < ntiles; ++t) {
    const int s = t % kStages;
    const bool got = mbar_wait(smem_u32(&full[s]), (t / kStages) & 1, kDrainBudgetNs);
    const int kt = kb + t * kTile;
    const int valid = min(kTile, ke - kt);
    uint8_t *kst = stages + s * kStageBytes;
    uint8_t *vst = kst + kStageBytes / 2;
    if (valid < kTile) {
      // zero V rows past the split's end (both halves), before P V reads them
      for (int x = tid; x < (kTile - valid) * 16; x += kConsumerWarps * 32) {
        const int rr = valid + (x >> 4), ch = x & 15;
        *reinterpret_cast<uint4 *>(vst + (ch >> 3) * kHalfBytes + rr * 128 + (ch & 7) * 16) = make_uint4(0, 0, 0, 0);
      }
      fence_proxy_async();
    }
    const uint32_t k_base = smem_u32(kst), v_base = smem_u32(vst);

    // ---- S = Q K^T for keys kKeysPerWarp*w .. of the tile ----
    float sfr[RG][kNtS][4];
#pragma unroll
    for (int mt = 0; mt < RG; ++mt)
#pragma unroll
      for (int nt = 0; nt < kNtS; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) sfr[mt][nt][e] = 0.f;
#pragma unroll
    for (int kk = 0; kk < kD / 16; ++kk) {
      // B fragments: keys (kKeysPerWarp*w + 8*nt + lane%8), head_dim chunk 2kk + (lane/8)%2
      uint32_t b00, b01, b10 = 0, b11 = 0;
      {
        const int mi = lane >> 3;
        const int key = warp * kKeysPerWarp + (kNtS == 2 ? (mi >> 1) : 0) * 8 + (lane & 7);
        const int ch = 2 * kk + (mi & 1);
        if constexpr (kNtS == 2) ldsm_x4(k_base + (ch >> 3) * kHalfBytes + swz(key, ch & 7), b00, b01, b10, b11);
        else ldsm_x2(k_base + (ch >> 3) * kHalfBytes + swz(key, ch & 7), b00, b01);
      }
#pragma unroll
      for (int mt = 0; mt < RG; ++mt) {
        uint32_t a0, a1, a2, a3;
        const int mi = lane >> 3;
        const int row = mt * 16 + (lane & 7) + (mi & 1) * 8;
        const int ch = 2 * kk + (mi >> 1);
        ldsm_x4(q_base + (ch >> 3) * (kRows * 128) + swz(row, ch & 7), a0, a1, a2, a3);
        mma16816(sfr[mt][0], a0, a1, a2, a3, b00, b01);
        if constexpr (kNtS == 2) mma16816(sfr[mt][kNtS - 1], a0, a1, a2, a3, b10, b11);
      }
    }
    // ---- scale, mask, per-warp row max ----
#pragma unroll
    for (int mt = 0; mt < RG; ++mt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        float mx = -INFINITY;
        const int i = pos_of[mt][h];
#pragma unroll
        for (int nt = 0; nt < kNtS; ++nt)
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int key = kt + warp * kKeysPerWarp + nt * 8 + 2 * qc + e;
            bool vis = i >= 0 && key < ke;
            if (vis && key >= c) {
              const int j = key - c;
              vis = (a.mask_kind == SV_MASK_CAUSAL) ? (j <= i) : (j < 64 && ((tmask_of[mt][h] >> j) & 1ull));
            }
            float &v = sfr[mt][nt][2 * h + e];
            v = vis ? v * a.scale_log2 : -INFINITY;
            mx = fmaxf(mx, v);
          }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        if (qc == 0) red_max[warp * kRows + mt * 16 + qr + 8 * h] = mx;
      }
    // every consumer leaves together if any of them gave up waiting for the tile
    if (consumers_sync_or(!got)) {
      if (tid == 0) record(a.status, SV_ERR_TIMEOUT);
      ok = false;
      break;
    }
    // ---- new running max, P, partial row sums ----
    float alpha[RG][2];
#pragma unroll
    for (int mt = 0; mt < RG; ++mt)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        const int row = mt * 16 + qr + 8 * h;
        float tm = red_max[row];
#pragma unroll
        for (int w = 1; w < kConsumerWarps; ++w) tm = fmaxf(tm, red_max[w * kRows + row]);
        const float mn = fmaxf(m_run[mt][h], tm);
        const float ref = (mn == -INFINITY) ? 0.f : mn;
        alpha[mt][h] = exp2f(m_run[mt][h] - ref);  // 0 when nothing was seen yet
        m_run[mt][h] = mn;
        float ls = 0.f;
#pragma unroll
        for (int nt = 0; nt < kNtS; ++nt) {
          const float p0 = exp2f(sfr[mt][nt][2 * h] - ref);
          const float p1 = exp2f(sfr[mt][nt][2 * h + 1] - ref);
          ls += p0 + p1;
          const int chunk = warp * kNtS + nt;
          *reinterpret_cast<uint32_t *>(p_s + swz(row, chunk) + qc * 4) = pack_bf16(p0, p1);
        }
        l_run[mt][h] = l_run[mt][h] * alpha[mt][h] + ls;
      }
    consumers_sync();
    // ---- O = alpha * O + P V for output columns kColsPerWarp*w .. ----
#pragma unroll
    for (int mt = 0; mt < RG; ++mt)
#pragma unroll
      for (int nt = 0; nt < kNtO; ++nt) {
        o_acc[mt][nt][0] *= alpha[mt][0];
        o_acc[mt][nt][1] *= alpha[mt][0];
        o_acc[mt][nt][2] *= alpha[mt][1];
        o_acc[mt][nt][3] *= alpha[mt][1];
      }
#pragma unroll
    for (int kk = 0; kk < kTile / 16; ++kk) {
      uint32_t bv[kNtO][2];
#pragma unroll
      for (int np = 0; np < kNtO / 2; ++np) {
        const int mi = lane >> 3;
        const int key = kk * 16 + (mi & 1) * 8 + (lane & 7);
        const int ch = warp * kNtO + np * 2 + (mi >> 1);  // 16-byte chunk along head_dim (0..15)
        ldsm_x4_t(v_base + (ch >> 3) * kHalfBytes + swz(key, ch & 7), bv[2 * np][0], bv[2 * np][1], bv[2 * np + 1][0],
                  bv[2 * np + 1][1]);
      }
#pragma unroll
      for (int mt = 0; mt < RG; ++mt) {
        uint32_t a0, a1, a2, a3;
        const int mi = lane >> 3;
        const int row = mt * 16 + (lane & 7) + (mi & 1) * 8;
        const int ch = 2 * kk + (mi >> 1);
        ldsm_x4(p_base + swz(row, ch), a0, a1, a2, a3);
#pragma unroll
        for (int nt = 0; nt < kNtO; ++nt) mma16816(o_acc[mt][nt], a0, a1, a2, a3, bv[nt][0], bv[nt][1]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(&empty[s]));
  }

  // ---- reduce the per-warp row sums, write the rows ----
#pragma unroll
  for (int mt = 0; mt < RG; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float l = l_run[mt][h];
      l += __shfl_xor_sync(0xffffffffu, l, 1);
      l += __shfl_xor_sync(0xffffffffu, l, 2);
      if (qc == 0) red_l[warp * kRows + mt * 16 + qr + 8 * h] = l;
    }
  consumers_sync();
  if (!ok) return;
#pragma unroll
  for (int mt = 0; mt < RG; ++mt)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int row = mt * 16 + qr + 8 * h;
      const int r = rbase + row;
      if (r >= R) continue;
      float l = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) l += red_l[w * kRows + row];
      const float inv = l > 0.f ? 1.f / l : 0.f;
      const int i = r / G, g = r % G;
      const size_t qrow = (size_t)(row0 + i) * a.num_q_heads + kvh * G + g;
      if (nsplit == 1) {
        __nv_bfloat16 *op = reinterpret_cast<__nv_bfloat16 *>(a.out) + qrow * kD;
#pragma unroll
        for (int nt = 0; nt < kNtO; ++nt) {
          const int col = warp * kColsPerWarp + nt * 8 + 2 * qc;
          *reinterpret_cast<uint32_t *>(op + col) = pack_bf16(o_acc[mt][nt][2 * h] * inv, o_acc[mt][nt][2 * h + 1] * inv);
        }
      } else {
        const size_t prow = (size_t)split * a.total_q * a.num_q_heads + qrow;
#pragma unroll
        for (int nt = 0; nt < kNtO; ++nt) {
          const int col = warp * kColsPerWarp + nt * 8 + 2 * qc;
          *reinterpret_cast<float2 *>(a.ws_o + prow * kD + col) =
              make_float2(o_acc[mt][nt][2 * h] * inv, o_acc[mt][nt][2 * h + 1] * inv);
        }
        if (warp == 0 && qc == 0) a.ws_lse[prow] = l > 0.f ? m_run[mt][h] + log2f(l) : -INFINITY;
      }
    }
}

// ------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------
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

bool make_map(CUtensorMap *map, void *pool, const KV &kv, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t rows = (cuuint64_t)kv.num_blocks * kv.num_kv_heads * kv.block_size;
  const cuuint64_t gdim[2] = {(cuuint64_t)kD, rows};
  const cuuint64_t gstride[1] = {(cuuint64_t)kD * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
  const cuuint32_t estride[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, pool, gdim, gstride, box, estride,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int rows_groups(const AttnArgs &a) {
  const int G = a.num_q_heads / a.kv.num_kv_heads;
  const int rows = G * a.max_q;
  const int rg = (rows + 15) / 16;
  return rg < 4 ? rg : 4;
}

size_t smem_bytes(int rg) {
  const int rows = 16 * rg;
  return 1024 + (size_t)kStages * kStageBytes + 2 * rows * 128 + rows * 128 + 2 * kConsumerWarps * rows * 4 +
         2 * kStages * 8;
}

template <int RG>
cudaError_t launch_rg(const AttnArgs &a, const CUtensorMap &mk, const CUtensorMap &mv, cudaStream_t st) {
  TcParams p;
  p.a = a;
  p.box_rows = a.kv.block_size < kTile ? a.kv.block_size : kTile;
  const int G = a.num_q_heads / a.kv.num_kv_heads;
  p.row_blocks = (G * a.max_q + 16 * RG - 1) / (16 * RG);
  const size_t smem = smem_bytes(RG);
  cudaError_t e = cudaFuncSetAttribute(attn_tc_kernel<RG>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(a.max_splits, a.kv.num_kv_heads * p.row_blocks, a.kv.batch);
  return launch_pdl(attn_tc_kernel<RG>, grid, dim3(kThreads), smem, st, mk, mv, p);
}

}  // namespace

bool attn_tc_supported(const KV &kv, int num_q_heads, int max_q) {
  (void)num_q_heads;
  (void)max_q;
  return kv.elem_bytes == 2 && kv.head_dim == kD && kv.block_size >= 16 && kv.block_size <= 256 &&
         encode_fn() != nullptr && ((uintptr_t)kv.k_pool % 16 == 0) && ((uintptr_t)kv.v_pool % 16 == 0);
}

cudaError_t launch_attn_tc(const AttnArgs &a, cudaStream_t st) {
  if (a.kv.batch == 0) return cudaSuccess;
  const int box = a.kv.block_size < kTile ? a.kv.block_size : kTile;
  CUtensorMap mk, mv;
  if (!make_map(&mk, a.kv.k_pool, a.kv, box) || !make_map(&mv, a.kv.v_pool, a.kv, box)) return cudaErrorInvalidValue;
  switch (rows_groups(a)) {
    case 1: return launch_rg<1>(a, mk, mv, st);
    case 2: return launch_rg<2>(a, mk, mv, st);
    case 3: return launch_rg<3>(a, mk, mv, st);
    default: return launch_rg<4>(a, mk, mv, st);
  }
}

}  // namespace sv
