"""ctypes binding of libspecverify (include/spec_verify.h).

Argument marshalling only: every function takes torch CUDA tensors, passes
their device pointers and the current CUDA stream to the C ABI, and raises
SVError on a non-OK return. Nothing here computes any part of the verify
step, and nothing falls back to the CPU: a missing library or a CPU tensor is
an error.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libspecverify.so")

SV_OK = 0
SV_ERR_INVALID_ARG = 1
SV_ERR_NONFINITE = 9
SV_ERR_WORKSPACE = 10
SV_DTYPE_BF16, SV_DTYPE_F32, SV_DTYPE_E4M3 = 0, 1, 2
SV_MASK_CAUSAL, SV_MASK_TREE = 0, 1
STATUS_NAMES = {
    0: "SV_OK", 1: "SV_ERR_INVALID_ARG", 2: "SV_ERR_UNSUPPORTED", 3: "SV_ERR_CUDA",
    4: "SV_ERR_OUT_OF_BLOCKS", 5: "SV_ERR_TIMEOUT", 6: "SV_ERR_BAD_BLOCK_ID", 7: "SV_ERR_BAD_LENGTH",
    8: "SV_ERR_BAD_TOKEN", 9: "SV_ERR_NONFINITE", 10: "SV_ERR_WORKSPACE",
}

EXPORTS = ("sv_kv_append", "sv_spec_verify_attn_workspace_bytes", "sv_spec_verify_attn",
           "sv_spec_verify_attn_no_alloc", "sv_spec_rejection_sample_workspace_bytes", "sv_spec_rejection_sample",
           "sv_tree_greedy_accept", "sv_tree_rejection_sample", "sv_kv_rollback", "sv_kv_fork", "sv_kv_release", "sv_adaptive_k_state_bytes", "sv_adaptive_k_init",
           "sv_adaptive_k_update", "sv_adaptive_k_reset", "sv_adaptive_k_current",
           "sv_status_string", "sv_version", "sv_set_option")
SV_OPT_ATTN_PATH = 1
ATTN_PATHS = {"auto": 0, "cuda_cores": 1, "tensor_cores": 2, "warp_mma": 3, "keys_major": 4}


class SVError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)}")


class sv_adaptive_k_params(ctypes.Structure):
    _fields_ = [
        ("k_min", ctypes.c_int32), ("k_max", ctypes.c_int32), ("k_init", ctypes.c_int32),
        ("window", ctypes.c_int32), ("min_samples", ctypes.c_int32),
        ("up_threshold", ctypes.c_double), ("down_threshold", ctypes.c_double),
    ]


class sv_paged_kv(ctypes.Structure):
    _fields_ = [
        ("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
        ("block_table", ctypes.c_void_p), ("seq_lens", ctypes.c_void_p),
        ("free_list", ctypes.c_void_p), ("free_top", ctypes.c_void_p),
        ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
        ("max_blocks_per_seq", ctypes.c_int32), ("num_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32), ("batch", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("ref_count", ctypes.c_void_p), ("k_scale", ctypes.c_float), ("v_scale", ctypes.c_float),
    ]


_lib = None
_lock = threading.Lock()


def load(path: Optional[str] = None, build_if_missing: bool = True) -> ctypes.CDLL:
    """Load libspecverify.so (building it with nvcc first if it is absent)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            if not build_if_missing:
                raise RuntimeError(f"{p} is not built")
            from . import build as _build
            _build.build()
        lib = ctypes.CDLL(p)
        P, I, F, S = ctypes.c_void_p, ctypes.c_int32, ctypes.c_float, ctypes.c_size_t
        KVP = ctypes.POINTER(sv_paged_kv)
        sig = {
            "sv_kv_append": (I, [KVP, P, P, P, I, P, P]),
            "sv_spec_verify_attn_workspace_bytes": (S, [KVP, I, I, I, I]),
            "sv_spec_verify_attn": (I, [KVP, P, P, P, I, I, I, I, F, I, P, P, S, P, P]),
            "sv_spec_verify_attn_no_alloc": (I, [KVP, P, P, P, I, I, I, I, F, I, P, P, P]),
            "sv_spec_rejection_sample_workspace_bytes": (S, [I, I, I, I, F]),
            "sv_spec_rejection_sample": (I, [P, P, I, I, I, P, I, I, P, P, P, F, P, P, P, P, P, S, P, P]),
            "sv_tree_greedy_accept": (I, [P, I, I, I, P, I, I, P, P, P, P, P, P, P, S, P, P]),
            "sv_tree_rejection_sample": (I, [P, I, I, I, P, I, I, P, P, P, P, F, P, P, P, P, P, P, S, P, P]),
            "sv_kv_rollback": (I, [KVP, P, P, P, I, P, P]),
            "sv_kv_fork": (I, [KVP, P, P, I, P, P]),
            "sv_kv_release": (I, [KVP, P, I, P, P]),
            "sv_adaptive_k_state_bytes": (S, [I, I]),
            "sv_adaptive_k_init": (I, [P, S, I, ctypes.POINTER(sv_adaptive_k_params)]),
            "sv_adaptive_k_update": (I, [P, P, P, P]),
            "sv_adaptive_k_reset": (I, [P, I]),
            "sv_adaptive_k_current": (I, [P, P]),
            "sv_status_string": (ctypes.c_char_p, [I]),
            "sv_version": (I, []),
            "sv_set_option": (I, [I, I]),
        }
        for name, (res, args) in sig.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        if path is None:
            _lib = lib
        return lib


def set_attn_path(path: str) -> None:
    """Select the attention implementation: "auto", "cuda_cores", "tensor_cores"
    (tcgen05) or "warp_mma" (mma.sync)."""
    _check(load().sv_set_option(SV_OPT_ATTN_PATH, ATTN_PATHS[path]), "sv_set_option")


SV_OPT_WAIT_BUDGET_US = 2
SV_OPT_STALL_FOR_TEST = 3
SV_ERR_TIMEOUT = 5
STALLS = {"none": 0, "attention": 1, "sampler": 2}
DEFAULT_WAIT_BUDGET_US = 500_000


def set_wait_budget_us(us: int) -> None:
    """Budget of the kernels' pipeline waits, in microseconds (1000 .. 2000000)."""
    _check(load().sv_set_option(SV_OPT_WAIT_BUDGET_US, int(us)), "sv_set_option")


def set_stall_for_test(which: str) -> None:
    """Failure-path test hook: "attention" or "sampler" makes that kernel's
    producer wait on a barrier nothing completes; "none" turns it off."""
    _check(load().sv_set_option(SV_OPT_STALL_FOR_TEST, STALLS[which]), "sv_set_option")


def status_string(code: int) -> str:
    try:
        return load().sv_status_string(int(code)).decode()
    except Exception:  # the library may be what failed to load
        return STATUS_NAMES.get(int(code), f"status {code}")


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError("libspecverify takes CUDA tensors only")
    if not t.is_contiguous():
        raise ValueError("libspecverify takes contiguous tensors only")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _check(rc: int, what: str):
    if rc != SV_OK:
        raise SVError(rc, what)


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SV_DTYPE_BF16
    if t.dtype == torch.float32:
        return SV_DTYPE_F32
    raise TypeError(f"unsupported dtype {t.dtype}")


@dataclass
class PagedKV:
    """One layer's paged KV cache held in torch CUDA tensors (see sv_paged_kv)."""

    k_pool: torch.Tensor  # [num_blocks, num_kv_heads, block_size, head_dim]
    v_pool: torch.Tensor
    block_table: torch.Tensor  # int32 [batch, max_blocks_per_seq]
    seq_lens: torch.Tensor  # int32 [batch]
    free_list: torch.Tensor  # int32 [num_blocks]
    free_top: torch.Tensor  # int32 [1]
    ref_count: Optional[torch.Tensor] = None  # int32 [num_blocks]: copy-on-write sharing when given
    k_scale: float = 1.0  # E4M3 pools (uint8 codes): dequantisation scales
    v_scale: float = 1.0

    def struct(self) -> sv_paged_kv:
        nb, hkv, bs, d = self.k_pool.shape
        return sv_paged_kv(
            _ptr(self.k_pool), _ptr(self.v_pool), _ptr(self.block_table), _ptr(self.seq_lens),
            _ptr(self.free_list), _ptr(self.free_top), nb, bs, self.block_table.shape[1], hkv, d,
            self.seq_lens.shape[0], SV_DTYPE_E4M3 if self.k_pool.dtype == torch.uint8 else _dtype_code(self.k_pool),
            _ptr(self.ref_count), float(self.k_scale), float(self.v_scale))

    @property
    def batch(self) -> int:
        return int(self.seq_lens.shape[0])


def kv_append(kv: PagedKV, new_k: torch.Tensor, new_v: torch.Tensor, cu_q: torch.Tensor,
              status: torch.Tensor, stream=None) -> None:
    s = kv.struct()
    _check(load().sv_kv_append(ctypes.byref(s), _ptr(new_k), _ptr(new_v), _ptr(cu_q), int(new_k.shape[0]),
                               _ptr(status), _stream(stream)), "sv_kv_append")


def spec_verify_attn_workspace_bytes(kv: PagedKV, num_q_heads: int, total_q: int, max_q: int,
                                     max_seq_len: int) -> int:
    s = kv.struct()
    return int(load().sv_spec_verify_attn_workspace_bytes(ctypes.byref(s), num_q_heads, total_q, max_q,
                                                          max_seq_len))


def spec_verify_attn(kv: PagedKV, q: torch.Tensor, out: torch.Tensor, cu_q: torch.Tensor, *, max_q: int,
                     max_seq_len: int, scale: float, mask_kind: int = SV_MASK_CAUSAL,
                     tree_mask: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                     status: Optional[torch.Tensor] = None, stream=None) -> None:
    s = kv.struct()
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(load().sv_spec_verify_attn(ctypes.byref(s), _ptr(q), _ptr(out), _ptr(cu_q), int(q.shape[1]),
                                      int(q.shape[0]), int(max_q), int(max_seq_len), float(scale), int(mask_kind),
                                      _ptr(tree_mask), _ptr(workspace), ws_bytes, _ptr(status), _stream(stream)),
           "sv_spec_verify_attn")


# size of the static scratch behind spec_verify_attn_no_alloc (SV_ATTN_NO_ALLOC_SCRATCH_BYTES)
ATTN_NO_ALLOC_SCRATCH_BYTES = 16 << 20


def spec_verify_attn_no_alloc(kv: PagedKV, q: torch.Tensor, out: torch.Tensor, cu_q: torch.Tensor, *, max_q: int,
                              max_seq_len: int, scale: float, mask_kind: int = SV_MASK_CAUSAL,
                              tree_mask: Optional[torch.Tensor] = None, status: Optional[torch.Tensor] = None,
                              stream=None) -> None:
    """spec_verify_attn for callers that cannot allocate device memory: the
    split-KV scratch is a static array inside the library, shared by every
    call on a device (calls that overlap on the GPU race on it)."""
    s = kv.struct()
    _check(load().sv_spec_verify_attn_no_alloc(ctypes.byref(s), _ptr(q), _ptr(out), _ptr(cu_q), int(q.shape[1]),
                                               int(q.shape[0]), int(max_q), int(max_seq_len), float(scale),
                                               int(mask_kind), _ptr(tree_mask), _ptr(status), _stream(stream)),
           "sv_spec_verify_attn_no_alloc")


def spec_rejection_sample_workspace_bytes(logits_dtype: torch.dtype, vocab: int, batch: int, total_q: int,
                                          temperature: float) -> int:
    code = SV_DTYPE_BF16 if logits_dtype == torch.bfloat16 else SV_DTYPE_F32
    return int(load().sv_spec_rejection_sample_workspace_bytes(code, int(vocab), int(batch), int(total_q),
                                                               float(temperature)))


def _sampler_workspace(workspace: Optional[torch.Tensor], logits: torch.Tensor, batch: int,
                       temperature: float) -> tuple:
    """The caller's workspace, or a new one of the size the library asks for."""
    if workspace is None:
        need = spec_rejection_sample_workspace_bytes(logits.dtype, int(logits.shape[1]), batch,
                                                     int(logits.shape[0]), temperature)
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=logits.device)
    return workspace, workspace.numel() * workspace.element_size()


def spec_rejection_sample(target_logits: torch.Tensor, draft_logits: Optional[torch.Tensor], cu_q: torch.Tensor,
                          draft_tokens: Optional[torch.Tensor], u_accept: Optional[torch.Tensor],
                          u_resample: Optional[torch.Tensor], temperature: float, accept_count: torch.Tensor,
                          out_tokens: torch.Tensor, num_out: torch.Tensor, *, workspace: Optional[torch.Tensor] = None,
                          status: Optional[torch.Tensor] = None, margin: Optional[torch.Tensor] = None,
                          stream=None) -> None:
    batch = int(cu_q.shape[0]) - 1
    ws, ws_bytes = _sampler_workspace(workspace, target_logits, batch, temperature)
    _check(load().sv_spec_rejection_sample(
        _ptr(target_logits), _ptr(draft_logits), _dtype_code(target_logits), int(target_logits.shape[1]), batch,
        _ptr(cu_q), int(target_logits.shape[0]), int(out_tokens.shape[1]), _ptr(draft_tokens), _ptr(u_accept),
        _ptr(u_resample), float(temperature), _ptr(accept_count), _ptr(out_tokens), _ptr(num_out), _ptr(margin),
        _ptr(ws), ws_bytes, _ptr(status), _stream(stream)), "sv_spec_rejection_sample")


def tree_greedy_accept(target_logits: torch.Tensor, cu_q: torch.Tensor, node_tokens: torch.Tensor,
                       parent: torch.Tensor, accept_count: torch.Tensor, path_nodes: torch.Tensor,
                       out_tokens: torch.Tensor, num_out: torch.Tensor, *, workspace: Optional[torch.Tensor] = None,
                       status: Optional[torch.Tensor] = None, stream=None) -> None:
    batch = int(cu_q.shape[0]) - 1
    ws, ws_bytes = _sampler_workspace(workspace, target_logits, batch, 0.0)
    _check(load().sv_tree_greedy_accept(
        _ptr(target_logits), _dtype_code(target_logits), int(target_logits.shape[1]), batch, _ptr(cu_q),
        int(target_logits.shape[0]), int(out_tokens.shape[1]), _ptr(node_tokens), _ptr(parent),
        _ptr(accept_count), _ptr(path_nodes), _ptr(out_tokens), _ptr(num_out), _ptr(ws), ws_bytes, _ptr(status),
        _stream(stream)), "sv_tree_greedy_accept")


def tree_rejection_sample(target_logits: torch.Tensor, cu_q: torch.Tensor, node_tokens: torch.Tensor,
                          parent: torch.Tensor, u_accept: torch.Tensor, u_resample: torch.Tensor, temperature: float,
                          accept_count: torch.Tensor, path_nodes: torch.Tensor, out_tokens: torch.Tensor,
                          num_out: torch.Tensor, *, workspace: Optional[torch.Tensor] = None,
                          status: Optional[torch.Tensor] = None, margin: Optional[torch.Tensor] = None,
                          stream=None) -> None:
    """Lossless tree verification at T > 0 (children as point-mass proposals)."""
    batch = int(cu_q.shape[0]) - 1
    ws, ws_bytes = _sampler_workspace(workspace, target_logits, batch, 0.0)
    _check(load().sv_tree_rejection_sample(
        _ptr(target_logits), _dtype_code(target_logits), int(target_logits.shape[1]), batch, _ptr(cu_q),
        int(target_logits.shape[0]), int(out_tokens.shape[1]), _ptr(node_tokens), _ptr(parent), _ptr(u_accept),
        _ptr(u_resample), float(temperature), _ptr(accept_count), _ptr(path_nodes), _ptr(out_tokens), _ptr(num_out),
        _ptr(margin), _ptr(ws), ws_bytes, _ptr(status), _stream(stream)), "sv_tree_rejection_sample")


def kv_rollback(kv: PagedKV, cu_q: torch.Tensor, accept_count: torch.Tensor, status: torch.Tensor, *,
                max_q: int, path_nodes: Optional[torch.Tensor] = None, stream=None) -> None:
    s = kv.struct()
    _check(load().sv_kv_rollback(ctypes.byref(s), _ptr(cu_q), _ptr(accept_count), _ptr(path_nodes), int(max_q),
                                 _ptr(status), _stream(stream)), "sv_kv_rollback")


def kv_fork(kv: PagedKV, parents: torch.Tensor, children: torch.Tensor, status: torch.Tensor, stream=None) -> None:
    """Children (empty slots) share their parents' blocks copy-on-write; needs kv.ref_count."""
    s = kv.struct()
    _check(load().sv_kv_fork(ctypes.byref(s), _ptr(parents), _ptr(children), int(parents.numel()), _ptr(status),
                             _stream(stream)), "sv_kv_fork")


def kv_release(kv: PagedKV, seqs: torch.Tensor, status: torch.Tensor, stream=None) -> None:
    """Finished sequences give their blocks back (shared blocks at their last holder)."""
    s = kv.struct()
    _check(load().sv_kv_release(ctypes.byref(s), _ptr(seqs), int(seqs.numel()), _ptr(status), _stream(stream)),
           "sv_kv_release")


class AdaptiveK:
    """Per-sequence draft length from observed acceptance (host side; the
    sv_adaptive_k_* calls). The state lives in host memory owned here; the
    arrays passed in and out are host int32 arrays (numpy or CPU tensors)."""

    def __init__(self, batch: int, *, k_min: int = 2, k_max: int = 8, k_init: Optional[int] = None,
                 window: int = 50, min_samples: int = 10, up_threshold: float = 0.6 + 0.1,
                 down_threshold: float = 0.6 - 0.1):
        import numpy as np
        self._np = np
        self.batch = int(batch)
        self.params = sv_adaptive_k_params(int(k_min), int(k_max), int(k_min if k_init is None else k_init),
                                           int(window), int(min_samples), float(up_threshold),
                                           float(down_threshold))
        lib = load()
        n = int(lib.sv_adaptive_k_state_bytes(self.batch, self.params.window))
        if n == 0:
            raise SVError(SV_ERR_INVALID_ARG, "sv_adaptive_k_state_bytes")
        self._state = (ctypes.c_double * ((n + 7) // 8))()  # 8-byte aligned host memory
        _check(lib.sv_adaptive_k_init(self._state, n, self.batch, ctypes.byref(self.params)), "sv_adaptive_k_init")

    def _host_i32(self, x):
        a = self._np.ascontiguousarray(x.cpu().numpy() if isinstance(x, torch.Tensor) else x, dtype=self._np.int32)
        if a.shape != (self.batch,):
            raise ValueError(f"expected {self.batch} entries")
        return a

    def update(self, accepted, drafted):
        """Feed one step's accept counts and draft lengths; returns next K (int32 numpy array)."""
        a, d = self._host_i32(accepted), self._host_i32(drafted)
        out = self._np.empty(self.batch, dtype=self._np.int32)
        _check(load().sv_adaptive_k_update(self._state, a.ctypes.data, d.ctypes.data, out.ctypes.data),
               "sv_adaptive_k_update")
        return out

    def reset(self, seq: int) -> None:
        _check(load().sv_adaptive_k_reset(self._state, int(seq)), "sv_adaptive_k_reset")

    @property
    def k(self):
        out = self._np.empty(self.batch, dtype=self._np.int32)
        _check(load().sv_adaptive_k_current(self._state, out.ctypes.data), "sv_adaptive_k_current")
        return out
