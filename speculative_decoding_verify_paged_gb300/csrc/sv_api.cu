// extern "C" entry points of libspecverify: argument checks, launch planning
// and dispatch. Nothing here allocates device memory or synchronises.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>

#include "sv_internal.cuh"

namespace sv {

int num_sms() {
  static int cached[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 152;
  }
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
      cudaGetLastError();
      n = 152;
    }
    cached[dev] = n;
  }
  return cached[dev];
}

// Keys per split: enough splits that (sequences x KV heads x splits) covers
// the SMs about four times over, each split a multiple of `granule` keys.
SplitPlan plan_splits(int batch, int num_kv_heads, int max_seq_len, int granule) {
  SplitPlan p;
  const long long units = (long long)batch * num_kv_heads;
  const long long target = 4LL * num_sms();
  int splits = units > 0 ? (int)((target + units - 1) / units) : 1;
  const int max_useful = (max_seq_len + granule - 1) / granule;
  if (splits > max_useful) splits = max_useful;
  if (splits < 1) splits = 1;
  int chunk = (max_seq_len + splits - 1) / splits;
  chunk = (chunk + granule - 1) / granule * granule;
  if (chunk < granule) chunk = granule;
  p.chunk = chunk;
  p.max_splits = (max_seq_len + chunk - 1) / chunk;
  return p;
}

bool sampler_supports(int vocab);

}  // namespace sv

using namespace sv;

namespace {

constexpr int kMaxQ = 64;
constexpr int kGranule = 64;
int g_attn_path = SV_ATTN_AUTO;
unsigned long long g_wait_ns = kDefaultWaitNs;  // budget of the kernels' pipeline waits
int g_stall = SV_STALL_NONE;                    // failure-path test hook

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }

sv_status check_kv(const sv_paged_kv *kv, bool need_free) {
  if (kv == nullptr) return SV_ERR_INVALID_ARG;
  if (kv->batch < 0 || kv->num_blocks <= 0 || kv->max_blocks_per_seq <= 0 || kv->num_kv_heads <= 0)
    return SV_ERR_INVALID_ARG;
  if (!pow2(kv->block_size) || kv->block_size > 256) return SV_ERR_INVALID_ARG;
  if (kv->head_dim < 8 || kv->head_dim > 256 || kv->head_dim % 8 != 0) return SV_ERR_INVALID_ARG;
  if (kv->dtype != SV_DTYPE_BF16 && kv->dtype != SV_DTYPE_F32 && kv->dtype != SV_DTYPE_E4M3) return SV_ERR_INVALID_ARG;
  if (kv->dtype == SV_DTYPE_E4M3 &&
      (kv->head_dim % 16 != 0 || !(kv->k_scale > 0.f) || !(kv->v_scale > 0.f) || kv->k_scale == INFINITY ||
       kv->v_scale == INFINITY))
    return SV_ERR_INVALID_ARG;
  if (kv->batch > 0 && (kv->block_table == nullptr || kv->seq_lens == nullptr)) return SV_ERR_INVALID_ARG;
  if (kv->k_pool == nullptr || kv->v_pool == nullptr) return SV_ERR_INVALID_ARG;
  if (!aligned16(kv->k_pool) || !aligned16(kv->v_pool)) return SV_ERR_INVALID_ARG;
  if (need_free && (kv->free_list == nullptr || kv->free_top == nullptr)) return SV_ERR_INVALID_ARG;
  return SV_OK;
}

sv_status cuda_status(cudaError_t e) { return e == cudaSuccess ? SV_OK : SV_ERR_CUDA; }

// Whether the tcgen05 kernel can take these sizes.
bool umma_usable(const sv_paged_kv *kv, int32_t num_q_heads, int32_t max_q, int32_t max_seq_len) {
  return (kv->dtype == SV_DTYPE_BF16 || kv->dtype == SV_DTYPE_E4M3) && attn_umma_supported(make_kv(*kv)) &&
         attn_umma_fits(make_kv(*kv), num_q_heads, max_q, max_seq_len);
}

// Whether the keys-major tcgen05 kernel can (units of at most 32 query rows).
bool keys_usable(const sv_paged_kv *kv, int32_t num_q_heads, int32_t max_q, int32_t max_seq_len) {
  return kv->dtype == SV_DTYPE_BF16 && umma_usable(kv, num_q_heads, max_q, max_seq_len) &&
         attn_keys_fits(make_kv(*kv), num_q_heads, max_q, max_seq_len);
}

// Workspace of whichever kernel a call may select: the split-KV partials of the
// CUDA-core and mma.sync kernels, or the tcgen05 kernel's slots and tile prefix.
size_t attn_workspace(const sv_paged_kv *kv, int32_t num_q_heads, int32_t total_q, int32_t max_q,
                      int32_t max_seq_len) {
  const SplitPlan p = plan_splits(kv->batch, kv->num_kv_heads, max_seq_len, kGranule);
  size_t need = 0;
  if (p.max_splits > 1) {
    const size_t rows = (size_t)p.max_splits * total_q * num_q_heads;
    need = rows * (size_t)kv->head_dim * sizeof(float) + rows * sizeof(float) + 256;
  }
  if (kv->batch > 0 && umma_usable(kv, num_q_heads, max_q, max_seq_len))
    need = std::max(need, attn_umma_workspace_bytes(make_kv(*kv), num_q_heads, max_q, max_seq_len));
  if (kv->batch > 0 && keys_usable(kv, num_q_heads, max_q, max_seq_len))
    need = std::max(need, attn_keys_workspace_bytes(make_kv(*kv), num_q_heads, max_q, max_seq_len));
  return need;
}

// The sampler's partials workspace: present, 256-byte aligned and large enough.
sv_status check_sampler_workspace(const void *workspace, size_t workspace_bytes, int dtype, int vocab, int batch,
                                  int total_q, int mode) {
  const size_t need = sampler_workspace_bytes(vocab, dtype, total_q, batch, mode);
  if (need == 0) return SV_ERR_UNSUPPORTED;
  if (workspace == nullptr || ((uintptr_t)workspace & 255u) != 0 || workspace_bytes < need) return SV_ERR_WORKSPACE;
  return SV_OK;
}

}  // namespace

extern "C" {

const char *sv_status_string(int32_t status) {
  switch (status) {
    case SV_OK: return "SV_OK";
    case SV_ERR_INVALID_ARG: return "SV_ERR_INVALID_ARG: a pointer, size or enum argument is invalid";
    case SV_ERR_UNSUPPORTED: return "SV_ERR_UNSUPPORTED: valid arguments outside what this build handles";
    case SV_ERR_CUDA: return "SV_ERR_CUDA: a CUDA launch failed";
    case SV_ERR_OUT_OF_BLOCKS: return "SV_ERR_OUT_OF_BLOCKS: the free list holds too few blocks";
    case SV_ERR_TIMEOUT: return "SV_ERR_TIMEOUT: a bounded wait inside a kernel gave up";
    case SV_ERR_BAD_BLOCK_ID: return "SV_ERR_BAD_BLOCK_ID: a block id outside [0, num_blocks)";
    case SV_ERR_BAD_LENGTH: return "SV_ERR_BAD_LENGTH: a length, accept count or path entry is out of range";
    case SV_ERR_BAD_TOKEN: return "SV_ERR_BAD_TOKEN: a token id outside [0, vocab)";
    case SV_ERR_NONFINITE: return "SV_ERR_NONFINITE: a NaN or +inf logit, or a row without finite logits";
    case SV_ERR_WORKSPACE: return "SV_ERR_WORKSPACE: workspace missing or too small";
    default: return "unknown sv_status";
  }
}

int32_t sv_version(void) { return 30100; }

sv_status sv_set_option(int32_t option, int32_t value) {
  if (option == SV_OPT_ATTN_PATH && value >= SV_ATTN_AUTO && value <= SV_ATTN_KEYS_MAJOR) {
    g_attn_path = value;
    return SV_OK;
  }
  if (option == SV_OPT_WAIT_BUDGET_US && value >= 1000 && value <= 2000000) {
    g_wait_ns = (unsigned long long)value * 1000ull;
    return SV_OK;
  }
  if (option == SV_OPT_STALL_FOR_TEST && value >= SV_STALL_NONE && value <= SV_STALL_SAMPLER) {
    g_stall = value;
    return SV_OK;
  }
  return SV_ERR_INVALID_ARG;
}

sv_status sv_kv_append(const sv_paged_kv *kv, const void *new_k, const void *new_v, const int32_t *cu_q,
                       int32_t total_q, int32_t *status_dev, void *stream) {
  sv_status s = check_kv(kv, true);
  if (s != SV_OK) return s;
  if (status_dev == nullptr || total_q < 0 || (kv->batch > 0 && cu_q == nullptr)) return SV_ERR_INVALID_ARG;
  if (total_q > 0 && (new_k == nullptr || new_v == nullptr || !aligned16(new_k) || !aligned16(new_v)))
    return SV_ERR_INVALID_ARG;
  if (kv->batch == 0) return SV_OK;
  if (kv->ref_count != nullptr && kv->batch > kv_cow_max_batch()) return SV_ERR_UNSUPPORTED;
  return cuda_status(
      launch_kv_append(make_kv(*kv), new_k, new_v, cu_q, total_q, status_dev, (cudaStream_t)stream));
}

size_t sv_spec_verify_attn_workspace_bytes(const sv_paged_kv *kv, int32_t num_q_heads, int32_t total_q,
                                           int32_t max_q_per_seq, int32_t max_seq_len) {
  if (kv == nullptr || num_q_heads <= 0 || kv->num_kv_heads <= 0 || num_q_heads % kv->num_kv_heads != 0 ||
      total_q < 0 || max_q_per_seq < 1 || max_q_per_seq > kMaxQ || max_seq_len <= 0)
    return 0;
  return attn_workspace(kv, num_q_heads, total_q, max_q_per_seq, max_seq_len);
}

sv_status sv_spec_verify_attn(const sv_paged_kv *kv, const void *q, void *out, const int32_t *cu_q,
                              int32_t num_q_heads, int32_t total_q, int32_t max_q_per_seq,
                              int32_t max_seq_len, float scale, int32_t mask_kind, const uint64_t *tree_mask,
                              void *workspace, size_t workspace_bytes, int32_t *status_dev, void *stream) {
  sv_status s = check_kv(kv, false);
  if (s != SV_OK) return s;
  if (num_q_heads <= 0 || num_q_heads % kv->num_kv_heads != 0) return SV_ERR_INVALID_ARG;
  if (total_q < 0 || max_q_per_seq < 1 || max_q_per_seq > kMaxQ || max_seq_len < 1) return SV_ERR_INVALID_ARG;
  if (mask_kind != SV_MASK_CAUSAL && mask_kind != SV_MASK_TREE) return SV_ERR_INVALID_ARG;
  if (mask_kind == SV_MASK_TREE && tree_mask == nullptr && total_q > 0) return SV_ERR_INVALID_ARG;
  if (!(scale == scale)) return SV_ERR_INVALID_ARG;
  if (kv->batch == 0 || total_q == 0) return SV_OK;
  if (q == nullptr || out == nullptr || cu_q == nullptr || !aligned16(q) || !aligned16(out))
    return SV_ERR_INVALID_ARG;
  if (kv->head_dim % 32 != 0) return SV_ERR_UNSUPPORTED;
  const size_t need = attn_workspace(kv, num_q_heads, total_q, max_q_per_seq, max_seq_len);
  if (need > 0 && (workspace == nullptr || workspace_bytes < need || ((uintptr_t)workspace & 255u) != 0))
    return SV_ERR_WORKSPACE;

  const SplitPlan p = plan_splits(kv->batch, kv->num_kv_heads, max_seq_len, kGranule);
  AttnArgs a;
  a.kv = make_kv(*kv);
  a.q = q;
  a.out = out;
  a.cu_q = cu_q;
  a.tree_mask = tree_mask;
  const size_t rows = (size_t)p.max_splits * total_q * num_q_heads;
  a.ws_o = p.max_splits > 1 ? (float *)workspace : nullptr;
  a.ws_lse = p.max_splits > 1 ? (float *)workspace + rows * (size_t)kv->head_dim : nullptr;
  a.status = status_dev;
  a.num_q_heads = num_q_heads;
  a.total_q = total_q;
  a.max_q = max_q_per_seq;
  a.max_seq_len = max_seq_len;
  a.chunk = p.chunk;
  a.max_splits = p.max_splits;
  a.mask_kind = mask_kind;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.wait_ns = g_wait_ns;
  a.stall = g_stall;
  cudaStream_t st = (cudaStream_t)stream;
  const bool umma_ok = umma_usable(kv, num_q_heads, max_q_per_seq, max_seq_len);
  const bool keys_ok = keys_usable(kv, num_q_heads, max_q_per_seq, max_seq_len);
  const bool mma_ok = kv->dtype == SV_DTYPE_BF16 && attn_tc_supported(a.kv, num_q_heads, max_q_per_seq);
  cudaError_t e;
  switch (g_attn_path) {
    case SV_ATTN_CUDA_CORES: e = launch_attn_simt(a, kv->dtype, st); break;
    case SV_ATTN_TENSOR_CORES:
      if (!umma_ok) return SV_ERR_UNSUPPORTED;
      return cuda_status(launch_attn_umma(a, workspace, workspace_bytes, st));
    case SV_ATTN_WARP_MMA:
      if (!mma_ok) return SV_ERR_UNSUPPORTED;
      e = launch_attn_tc(a, st);
      break;
    case SV_ATTN_KEYS_MAJOR:
      if (!keys_ok) return SV_ERR_UNSUPPORTED;
      return cuda_status(launch_attn_keys(a, workspace, workspace_bytes, st));
    default:
      if (umma_ok) return cuda_status(launch_attn_umma(a, workspace, workspace_bytes, st));
      e = launch_attn_simt(a, kv->dtype, st);
  }
  if (e != cudaSuccess) return SV_ERR_CUDA;
  return cuda_status(launch_attn_combine(a, kv->dtype, st));
}

size_t sv_spec_rejection_sample_workspace_bytes(int32_t logits_dtype, int32_t vocab, int32_t batch, int32_t total_q,
                                                float temperature) {
  if (logits_dtype != SV_DTYPE_BF16 && logits_dtype != SV_DTYPE_F32) return 0;
  if (!(temperature >= 0.f) || temperature == INFINITY) return 0;
  return sampler_workspace_bytes(vocab, logits_dtype, total_q, batch, temperature == 0.f ? kGreedy : kStochastic);
}

sv_status sv_spec_rejection_sample(const void *target_logits, const void *draft_logits, int32_t logits_dtype,
                                   int32_t vocab, int32_t batch, const int32_t *cu_q, int32_t total_q,
                                   int32_t max_q_per_seq, const int32_t *draft_tokens, const float *u_accept,
                                   const float *u_resample, float temperature, int32_t *accept_count,
                                   int32_t *out_tokens, int32_t *num_out, float *margin, void *workspace,
                                   size_t workspace_bytes, int32_t *status_dev, void *stream) {
  if (logits_dtype != SV_DTYPE_BF16 && logits_dtype != SV_DTYPE_F32) return SV_ERR_INVALID_ARG;
  if (vocab < 1 || batch < 0 || batch > 65535 || total_q < batch || max_q_per_seq < 1 || max_q_per_seq > kMaxQ)
    return SV_ERR_INVALID_ARG;
  if (!(temperature >= 0.f) || temperature == INFINITY) return SV_ERR_INVALID_ARG;
  if (!sampler_supports(vocab)) return SV_ERR_UNSUPPORTED;
  if (batch == 0) return SV_OK;
  const bool greedy = temperature == 0.f;
  if (target_logits == nullptr || cu_q == nullptr || accept_count == nullptr || out_tokens == nullptr ||
      num_out == nullptr)
    return SV_ERR_INVALID_ARG;
  if (total_q > batch && draft_tokens == nullptr) return SV_ERR_INVALID_ARG;
  if (!greedy && (u_resample == nullptr || (total_q > batch && (draft_logits == nullptr || u_accept == nullptr))))
    return SV_ERR_INVALID_ARG;
  const sv_status ws = check_sampler_workspace(workspace, workspace_bytes, logits_dtype, vocab, batch, total_q,
                                               greedy ? kGreedy : kStochastic);
  if (ws != SV_OK) return ws;
  SamplerArgs a;
  std::memset(&a, 0, sizeof a);
  a.tgt = target_logits;
  a.drf = greedy ? nullptr : draft_logits;
  a.cu_q = cu_q;
  a.draft_tok = draft_tokens;
  a.u_acc = u_accept;
  a.u_res = u_resample;
  a.accept = accept_count;
  a.out_tok = out_tokens;
  a.num_out = num_out;
  a.margin = margin;
  a.status = status_dev;
  a.vocab = vocab;
  a.batch = batch;
  a.max_q = max_q_per_seq;
  a.total_q = total_q;
  a.wait_ns = g_wait_ns;
  a.stall = g_stall;
  if (!greedy) {
    const double c = 1.4426950408889634 / (double)temperature;
    a.coef = (float)c;
    a.coef_lo = (float)(c - (double)a.coef);
  }
  return cuda_status(launch_sampler(a, logits_dtype, greedy ? kGreedy : kStochastic, workspace, (cudaStream_t)stream));
}

namespace {
sv_status tree_greedy(const void *target_logits, int32_t logits_dtype, int32_t vocab, int32_t batch,
                      const int32_t *cu_q, int32_t total_q, int32_t max_q_per_seq, const int32_t *node_tokens,
                      const int32_t *parent, int32_t *accept_count, int32_t *path_nodes, int32_t *out_tokens,
                      int32_t *num_out, float *margin, void *workspace, size_t workspace_bytes, int32_t *status_dev,
                      void *stream) {
  if (logits_dtype != SV_DTYPE_BF16 && logits_dtype != SV_DTYPE_F32) return SV_ERR_INVALID_ARG;
  if (vocab < 1 || batch < 0 || batch > 65535 || total_q < batch || max_q_per_seq < 1 || max_q_per_seq > kMaxQ)
    return SV_ERR_INVALID_ARG;
  if (!sampler_supports(vocab)) return SV_ERR_UNSUPPORTED;
  if (batch == 0) return SV_OK;
  if (target_logits == nullptr || cu_q == nullptr || parent == nullptr || accept_count == nullptr ||
      path_nodes == nullptr || out_tokens == nullptr || num_out == nullptr)
    return SV_ERR_INVALID_ARG;
  if (total_q > batch && node_tokens == nullptr) return SV_ERR_INVALID_ARG;
  const sv_status ws = check_sampler_workspace(workspace, workspace_bytes, logits_dtype, vocab, batch, total_q, kTree);
  if (ws != SV_OK) return ws;
  SamplerArgs a;
  std::memset(&a, 0, sizeof a);
  a.tgt = target_logits;
  a.cu_q = cu_q;
  a.draft_tok = node_tokens;
  a.parent = parent;
  a.accept = accept_count;
  a.out_tok = out_tokens;
  a.num_out = num_out;
  a.path = path_nodes;
  a.margin = margin;
  a.status = status_dev;
  a.vocab = vocab;
  a.batch = batch;
  a.max_q = max_q_per_seq;
  a.total_q = total_q;
  a.wait_ns = g_wait_ns;
  a.stall = g_stall;
  return cuda_status(launch_sampler(a, logits_dtype, kTree, workspace, (cudaStream_t)stream));
}
}  // namespace

sv_status sv_tree_greedy_accept(const void *target_logits, int32_t logits_dtype, int32_t vocab, int32_t batch,
                                const int32_t *cu_q, int32_t total_q, int32_t max_q_per_seq,
                                const int32_t *node_tokens, const int32_t *parent, int32_t *accept_count,
                                int32_t *path_nodes, int32_t *out_tokens, int32_t *num_out, void *workspace,
                                size_t workspace_bytes, int32_t *status_dev, void *stream) {
  return tree_greedy(target_logits, logits_dtype, vocab, batch, cu_q, total_q, max_q_per_seq, node_tokens, parent,
                     accept_count, path_nodes, out_tokens, num_out, nullptr, workspace, workspace_bytes, status_dev,
                     stream);
}

sv_status sv_tree_rejection_sample(const void *target_logits, int32_t logits_dtype, int32_t vocab, int32_t batch,
                                   const int32_t *cu_q, int32_t total_q, int32_t max_q_per_seq,
                                   const int32_t *node_tokens, const int32_t *parent, const float *u_accept,
                                   const float *u_resample, float temperature, int32_t *accept_count,
                                   int32_t *path_nodes, int32_t *out_tokens, int32_t *num_out, float *margin,
                                   void *workspace, size_t workspace_bytes, int32_t *status_dev, void *stream) {
  if (temperature == 0.f)
    return tree_greedy(target_logits, logits_dtype, vocab, batch, cu_q, total_q, max_q_per_seq, node_tokens, parent,
                       accept_count, path_nodes, out_tokens, num_out, margin, workspace, workspace_bytes,
                       status_dev, stream);
  if (logits_dtype != SV_DTYPE_BF16 && logits_dtype != SV_DTYPE_F32) return SV_ERR_INVALID_ARG;
  if (vocab < 1 || batch < 0 || batch > 65535 || total_q < batch || max_q_per_seq < 1 || max_q_per_seq > kMaxQ)
    return SV_ERR_INVALID_ARG;
  if (!(temperature > 0.f) || temperature == INFINITY) return SV_ERR_INVALID_ARG;
  if (!sampler_supports(vocab)) return SV_ERR_UNSUPPORTED;
  if (batch == 0) return SV_OK;
  if (target_logits == nullptr || cu_q == nullptr || parent == nullptr || accept_count == nullptr ||
      path_nodes == nullptr || out_tokens == nullptr || num_out == nullptr || u_resample == nullptr)
    return SV_ERR_INVALID_ARG;
  if (total_q > batch && (node_tokens == nullptr || u_accept == nullptr)) return SV_ERR_INVALID_ARG;
  const sv_status ws = check_sampler_workspace(workspace, workspace_bytes, logits_dtype, vocab, batch, total_q,
                                               kTreeStochastic);
  if (ws != SV_OK) return ws;
  SamplerArgs a;
  std::memset(&a, 0, sizeof a);
  a.tgt = target_logits;
  a.cu_q = cu_q;
  a.draft_tok = node_tokens;
  a.parent = parent;
  a.u_acc = u_accept;
  a.u_res = u_resample;
  a.accept = accept_count;
  a.out_tok = out_tokens;
  a.num_out = num_out;
  a.path = path_nodes;
  a.margin = margin;
  a.status = status_dev;
  a.vocab = vocab;
  a.batch = batch;
  a.max_q = max_q_per_seq;
  a.total_q = total_q;
  a.wait_ns = g_wait_ns;
  a.stall = g_stall;
  const double c = 1.4426950408889634 / (double)temperature;
  a.coef = (float)c;
  a.coef_lo = (float)(c - (double)a.coef);
  return cuda_status(launch_sampler(a, logits_dtype, kTreeStochastic, workspace, (cudaStream_t)stream));
}

sv_status sv_kv_rollback(const sv_paged_kv *kv, const int32_t *cu_q, const int32_t *accept_count,
                         const int32_t *path_nodes, int32_t max_q_per_seq, int32_t *status_dev, void *stream) {
  sv_status s = check_kv(kv, true);
  if (s != SV_OK) return s;
  if (status_dev == nullptr || max_q_per_seq < 1 || max_q_per_seq > kMaxQ) return SV_ERR_INVALID_ARG;
  if (kv->batch == 0) return SV_OK;
  if (cu_q == nullptr || accept_count == nullptr) return SV_ERR_INVALID_ARG;
  return cuda_status(launch_kv_rollback(make_kv(*kv), cu_q, accept_count, path_nodes, max_q_per_seq, status_dev,
                                        (cudaStream_t)stream));
}

sv_status sv_kv_fork(const sv_paged_kv *kv, const int32_t *parents, const int32_t *children, int32_t n_pairs,
                     int32_t *status_dev, void *stream) {
  sv_status s = check_kv(kv, false);
  if (s != SV_OK) return s;
  if (kv->ref_count == nullptr || status_dev == nullptr || n_pairs < 0) return SV_ERR_INVALID_ARG;
  if (n_pairs > 0 && (parents == nullptr || children == nullptr)) return SV_ERR_INVALID_ARG;
  if (kv->batch > kv_max_seq_bits()) return SV_ERR_UNSUPPORTED;
  if (n_pairs == 0 || kv->batch == 0) return SV_OK;
  return cuda_status(launch_kv_fork(make_kv(*kv), parents, children, n_pairs, status_dev, (cudaStream_t)stream));
}

sv_status sv_kv_release(const sv_paged_kv *kv, const int32_t *seqs, int32_t n, int32_t *status_dev, void *stream) {
  sv_status s = check_kv(kv, true);
  if (s != SV_OK) return s;
  if (status_dev == nullptr || n < 0 || (n > 0 && seqs == nullptr)) return SV_ERR_INVALID_ARG;
  if (kv->batch > kv_max_seq_bits()) return SV_ERR_UNSUPPORTED;
  if (n == 0 || kv->batch == 0) return SV_OK;
  return cuda_status(launch_kv_release(make_kv(*kv), seqs, n, status_dev, (cudaStream_t)stream));
}

}  // extern "C"
