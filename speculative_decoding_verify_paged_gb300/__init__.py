"""GB300-native batched speculative-decoding verification over a paged KV cache.

The work is done by libspecverify.so (hand-written CUDA for sm_103a behind the
C ABI in include/spec_verify.h). This package holds the ctypes binding
(`_lib`), the step orchestration (`step`), the nvcc build (`build`) and the
seeded synthetic workloads (`workloads`). Importing it loads nothing; the
library is loaded on the first call and its absence is an error.
"""
from ._lib import (AdaptiveK, PagedKV, SVError, SV_DTYPE_BF16, SV_DTYPE_F32, SV_MASK_CAUSAL, SV_MASK_TREE,
                   kv_append, kv_fork, kv_release, kv_rollback, load, spec_rejection_sample,
                   spec_rejection_sample_workspace_bytes, spec_verify_attn, spec_verify_attn_workspace_bytes,
                   status_string, tree_greedy_accept, tree_rejection_sample)

__all__ = [
    "AdaptiveK", "PagedKV", "SVError", "SV_DTYPE_BF16", "SV_DTYPE_F32", "SV_MASK_CAUSAL", "SV_MASK_TREE",
    "kv_append", "kv_fork", "kv_release", "kv_rollback", "load", "spec_rejection_sample",
    "spec_rejection_sample_workspace_bytes", "spec_verify_attn", "spec_verify_attn_workspace_bytes",
    "status_string", "tree_greedy_accept", "tree_rejection_sample",
]
