// Internal declarations shared by the translation units of libspecverify.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_verify.h"

namespace sv {

// ---------------------------------------------------------------------------
// device status word: the first recorded error wins
// ---------------------------------------------------------------------------
__device__ __forceinline__ void record(int32_t *status, int32_t code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

__device__ __forceinline__ bool status_set(const int32_t *status) {
  return status != nullptr && *((volatile const int32_t *)status) != 0;
}

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

__host__ __device__ __forceinline__ int ceil_div(int a, int b) { return (a + b - 1) / b; }

// ---------------------------------------------------------------------------
// programmatic dependent launch: every kernel of the library is launched with
// launch_pdl, so its launch and set-up may overlap the end of the kernel
// before it on the stream. Each kernel calls grid_dependency_wait() before it
// writes any memory, before it reads anything an earlier kernel of the library
// may write, and before any return: the earlier kernel has then completed and
// its writes are visible, and, since every kernel waits before it can
// complete, completion stays transitive along the stream. Before the wait a
// kernel may read what no kernel of the library writes (the call's own
// inputs: whatever produced them is not a kernel of the library, so it let
// the library's kernels start only once it had completed).
// grid_dependents_launch() lets the next kernel launch.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

// ---------------------------------------------------------------------------
// bounded mbarrier wait: gives up (returns false) once it has waited about
// `budget_ns` of wall-clock time (globaltimer), so that a kernel whose
// barrier phase never completes ends instead of spinning on. Two budgets:
//  - pipeline waits (a consumer waiting for its producer, a producer for a
//    free stage) take the launch's budget (sv_set_option SV_OPT_WAIT_BUDGET_US,
//    0.5 s unless set);
//  - drain waits (for copies or MMAs this CTA has already issued, before its
//    shared memory or TMEM is released) always take kDrainBudgetNs, so that
//    nothing lands in memory the CTA no longer owns, whatever the option says.
// ---------------------------------------------------------------------------
constexpr unsigned long long kDrainBudgetNs = 500ull * 1000 * 1000;
constexpr unsigned long long kDefaultWaitNs = 500ull * 1000 * 1000;

__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  unsigned long long budget_ns = kDrainBudgetNs) {
  unsigned long long deadline = 0;
  for (uint32_t i = 0; i < (1u << 30); ++i) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if ((i & 63u) == 63u) {
      const unsigned long long now = global_ns();
      if (deadline == 0) deadline = now + budget_ns;
      else if (now > deadline) return false;
    }
  }
  return false;
}

// The failure-path test hook (sv_set_option SV_OPT_STALL_FOR_TEST): a
// producer waits, with the pipeline budget, on a barrier of its own that no
// thread ever arrives on, as a producer would whose data never comes. The wait
// runs out, so the producer issues nothing and its consumers' waits run out in
// turn. Returns false (always). `bar` is an initialised mbarrier of count 1.
__device__ __forceinline__ bool wait_on_nothing(uint32_t bar, unsigned long long budget_ns) {
  return mbar_wait_bounded(bar, 0, budget_ns);
}

// ---------------------------------------------------------------------------
// plain-data views of the ABI struct, passed by value to kernels
// ---------------------------------------------------------------------------
struct KV {
  void *k_pool;
  void *v_pool;
  int32_t *block_table;
  int32_t *seq_lens;
  int32_t *free_list;
  int32_t *free_top;
  int32_t *ref_count;  // null: no sharing
  int num_blocks, block_size, max_blocks, num_kv_heads, head_dim, batch;
  int elem_bytes;
  bool fp8;                // E4M3 pool: 1-byte codes, bf16 rows in and out
  float k_scale, v_scale;  // E4M3 dequantisation scales
};

inline KV make_kv(const sv_paged_kv &p) {
  KV k;
  k.k_pool = p.k_pool;
  k.v_pool = p.v_pool;
  k.block_table = p.block_table;
  k.seq_lens = p.seq_lens;
  k.free_list = p.free_list;
  k.free_top = p.free_top;
  k.ref_count = p.ref_count;
  k.num_blocks = p.num_blocks;
  k.block_size = p.block_size;
  k.max_blocks = p.max_blocks_per_seq;
  k.num_kv_heads = p.num_kv_heads;
  k.head_dim = p.head_dim;
  k.batch = p.batch;
  k.elem_bytes = p.dtype == SV_DTYPE_BF16 ? 2 : (p.dtype == SV_DTYPE_E4M3 ? 1 : 4);
  k.fp8 = p.dtype == SV_DTYPE_E4M3;
  k.k_scale = p.k_scale;
  k.v_scale = p.v_scale;
  return k;
}

// Split-KV attention arguments.
struct AttnArgs {
  KV kv;
  const void *q;
  void *out;
  const int32_t *cu_q;
  const uint64_t *tree_mask;
  float *ws_o;    // [max_splits, total_q, num_q_heads, head_dim]
  float *ws_lse;  // [max_splits, total_q, num_q_heads]
  int32_t *status;
  int num_q_heads, total_q, max_q, max_seq_len, chunk, max_splits;
  int mask_kind;
  float scale_log2;  // scale * log2(e)
  unsigned long long wait_ns;  // budget of the pipeline waits
  int stall;                   // failure-path test: SV_STALL_ATTENTION makes the producer wait on nothing
};

// How the key range of every sequence is split across CTAs.
struct SplitPlan {
  int chunk;       // tokens per split, a multiple of `granule`
  int max_splits;  // ceil(max_seq_len / chunk)
};
SplitPlan plan_splits(int batch, int num_kv_heads, int max_seq_len, int granule);

// kernels' host-side launchers (return a cudaError_t from the launch)
cudaError_t launch_kv_append(const KV &kv, const void *new_k, const void *new_v, const int32_t *cu_q,
                             int total_q, int32_t *status, cudaStream_t st);
cudaError_t launch_kv_rollback(const KV &kv, const int32_t *cu_q, const int32_t *accept, const int32_t *path,
                               int max_q, int32_t *status, cudaStream_t st);
cudaError_t launch_kv_fork(const KV &kv, const int32_t *parents, const int32_t *children, int n_pairs,
                           int32_t *status, cudaStream_t st);
cudaError_t launch_kv_release(const KV &kv, const int32_t *seqs, int n, int32_t *status, cudaStream_t st);
int kv_cow_max_batch();  // batch limit of append and rollback with reference counts
int kv_max_seq_bits();   // batch limit of fork and release
cudaError_t launch_attn_simt(const AttnArgs &a, int dtype, cudaStream_t st);
cudaError_t launch_attn_combine(const AttnArgs &a, int dtype, cudaStream_t st);
bool attn_tc_supported(const KV &kv, int num_q_heads, int max_q);
cudaError_t launch_attn_tc(const AttnArgs &a, cudaStream_t st);
bool attn_umma_supported(const KV &kv);
bool attn_umma_fits(const KV &kv, int num_q_heads, int max_q, int max_seq_len);
size_t attn_umma_workspace_bytes(const KV &kv, int num_q_heads, int max_q, int max_seq_len);
// launches the persistent tcgen05 kernel and its combine (workspace: attn_umma_workspace_bytes, 256-aligned)
cudaError_t launch_attn_umma(const AttnArgs &a, void *workspace, size_t workspace_bytes, cudaStream_t st);
// The keys-major tcgen05 kernel (attn_keys.cu): units of at most 32 query rows.
bool attn_keys_fits(const KV &kv, int num_q_heads, int max_q, int max_seq_len);
size_t attn_keys_workspace_bytes(const KV &kv, int num_q_heads, int max_q, int max_seq_len);
cudaError_t launch_attn_keys(const AttnArgs &a, void *workspace, size_t workspace_bytes, cudaStream_t st);

struct SamplerArgs {
  const void *tgt;
  const void *drf;
  const int32_t *cu_q;
  const int32_t *draft_tok;  // chain drafts, or tree node tokens
  const float *u_acc;
  const float *u_res;
  const int32_t *parent;
  int32_t *accept;
  int32_t *out_tok;
  int32_t *num_out;
  int32_t *path;
  float *margin;  // nullable: per sequence, the smallest |uniform - threshold| of the decisions (+inf greedy)
  int32_t *status;
  int vocab, batch, max_q, chunk, total_q;
  float coef;     // log2(e) / temperature, rounded to fp32
  float coef_lo;  // log2(e) / temperature - coef
  unsigned long long wait_ns;  // budget of the pipeline waits
  int stall;                   // failure-path test: SV_STALL_SAMPLER makes the statistics producer wait on nothing
};
enum SamplerMode { kStochastic = 0, kGreedy = 1, kTree = 2, kTreeStochastic = 3 };
// Bytes of the partials workspace: rows (total_q target rows, plus total_q - batch
// draft rows for kStochastic) x 32 KB items x 8 warps x (max, sum); 0 if the sizes
// are invalid or too large.
size_t sampler_workspace_bytes(int vocab, int dtype, int total_q, int batch, int mode);
cudaError_t launch_sampler(const SamplerArgs &a, int dtype, int mode, void *workspace, cudaStream_t st);
int num_sms();

}  // namespace sv
