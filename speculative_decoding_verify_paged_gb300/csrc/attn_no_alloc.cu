// sv_spec_verify_attn_no_alloc: the verify-pass attention for callers that
// cannot allocate device memory. It is sv_spec_verify_attn with the split-KV
// partial results placed in a file-scope device array instead of a workspace
// the caller allocates.
//
// The array is SV_ATTN_NO_ALLOC_SCRATCH_BYTES long and lives on every device
// that loads this library until the process exits. Its device address is
// looked up once per device, on the first call there that launches work, with
// the device current (host code cannot hand the array's name to a kernel: on
// the host it names a stand-in, not device memory). Sizes are checked before
// that look-up, so a refused call, or one with nothing to launch, makes no
// call into the CUDA runtime that could load the module or create a context.
#include <mutex>

#include "sv_internal.cuh"

namespace {

__device__ __align__(256) unsigned char g_attn_scratch[SV_ATTN_NO_ALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 256;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices];  // device address of g_attn_scratch, per device ordinal

// Device address of the scratch array on the current device, set up on first use.
sv_status scratch_address(void **addr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return SV_ERR_CUDA;
  }
  if (dev < 0 || dev >= kMaxDevices) return SV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_attn_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return SV_ERR_CUDA;
    }
    g_scratch_addr[dev] = p;
  }
  *addr = g_scratch_addr[dev];
  return SV_OK;
}

}  // namespace

extern "C" sv_status sv_spec_verify_attn_no_alloc(const sv_paged_kv *kv, const void *q, void *out,
                                                  const int32_t *cu_q, int32_t num_q_heads, int32_t total_q,
                                                  int32_t max_q_per_seq, int32_t max_seq_len, float scale,
                                                  int32_t mask_kind, const uint64_t *tree_mask, int32_t *status_dev,
                                                  void *stream) {
  if (kv == nullptr) return SV_ERR_INVALID_ARG;
  const size_t need = sv_spec_verify_attn_workspace_bytes(kv, num_q_heads, total_q, max_q_per_seq, max_seq_len);
  if (need > SV_ATTN_NO_ALLOC_SCRATCH_BYTES) return SV_ERR_WORKSPACE;
  // invalid sizes (need == 0 then), an empty batch or no scratch needed: the workspace
  // entry point decides, and launches nothing that would read a workspace
  if (need == 0 || kv->batch == 0 || total_q == 0)
    return sv_spec_verify_attn(kv, q, out, cu_q, num_q_heads, total_q, max_q_per_seq, max_seq_len, scale,
                               mask_kind, tree_mask, nullptr, 0, status_dev, stream);
  void *scratch = nullptr;
  const sv_status s = scratch_address(&scratch);
  if (s != SV_OK) return s;
  return sv_spec_verify_attn(kv, q, out, cu_q, num_q_heads, total_q, max_q_per_seq, max_seq_len, scale, mask_kind,
                             tree_mask, scratch, SV_ATTN_NO_ALLOC_SCRATCH_BYTES, status_dev, stream);
}
