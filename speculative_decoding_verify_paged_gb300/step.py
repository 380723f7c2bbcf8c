"""One verify step through the C ABI: device-side buffers and the call order.

`DeviceStep` holds one step's inputs on the GPU, `StepBuffers` its outputs
and scratch, and `run_step` issues the four library calls on one stream:

    kv_append -> spec_verify_attn -> spec_rejection_sample (or
    tree_greedy_accept) -> kv_rollback

Host arrays come in the layout of `workloads` (bf16 as uint16 bit patterns).
This module only moves data and orders calls; the arithmetic is in the CUDA
library.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional

import numpy as np
import torch

from . import _lib as L


def _dev(x: np.ndarray, device, dtype: Optional[str] = None) -> torch.Tensor:
    x = np.ascontiguousarray(x)
    if dtype == "bf16" or x.dtype == np.uint16:
        return torch.from_numpy(x.view(np.int16)).to(device).view(torch.bfloat16)
    return torch.from_numpy(x).to(device)


def _host(x: np.ndarray, dtype: Optional[str] = None, pin: bool = False) -> torch.Tensor:
    x = np.ascontiguousarray(x)
    t = torch.from_numpy(x.view(np.int16)).view(torch.bfloat16) if (dtype == "bf16" or x.dtype == np.uint16) \
        else torch.from_numpy(x)
    return t.pin_memory() if pin else t


def to_bits(t: torch.Tensor) -> np.ndarray:
    """Device/host tensor -> numpy (bf16 as uint16 bit patterns)."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def device_kv(state, device="cuda", ref_count=None) -> L.PagedKV:
    """The cache on the device; `ref_count` (int32 [num_blocks], host) turns on
    copy-on-write sharing."""
    return L.PagedKV(
        k_pool=_dev(state.k_pool, device, state.dtype), v_pool=_dev(state.v_pool, device, state.dtype),
        block_table=_dev(state.block_table.astype(np.int32), device),
        seq_lens=_dev(state.seq_lens.astype(np.int32), device),
        free_list=_dev(state.free_list.astype(np.int32), device),
        free_top=torch.tensor([state.free_top], dtype=torch.int32, device=device),
        ref_count=None if ref_count is None else _dev(np.asarray(ref_count, np.int32), device),
        k_scale=float(getattr(state, "k_scale", 1.0)), v_scale=float(getattr(state, "v_scale", 1.0)))


@dataclass
class DeviceStep:
    cu_q: torch.Tensor
    q: torch.Tensor
    new_k: torch.Tensor
    new_v: torch.Tensor
    target_logits: torch.Tensor
    draft_logits: torch.Tensor
    draft_tokens: torch.Tensor
    u_accept: torch.Tensor
    u_resample: torch.Tensor
    tree_mask: Optional[torch.Tensor]
    parent: Optional[torch.Tensor]
    temperature: float
    mask_kind: int
    max_q: int
    scale: float
    num_q_heads: int

    @property
    def batch(self) -> int:
        return int(self.cu_q.shape[0]) - 1

    @property
    def total_q(self) -> int:
        return int(self.q.shape[0])

    @staticmethod
    def tensors_of(step, make) -> dict:
        d = dict(
            cu_q=make(step.cu_q.astype(np.int32)),
            q=make(step.q), new_k=make(step.new_k), new_v=make(step.new_v),
            target_logits=make(step.target_logits), draft_logits=make(step.draft_logits),
            draft_tokens=make(step.draft_tokens.astype(np.int32)),
            u_accept=make(step.u_accept.astype(np.float32)), u_resample=make(step.u_resample.astype(np.float32)),
            tree_mask=make(step.tree_mask.view(np.int64)) if step.tree_mask is not None else None,
            parent=make(step.parent.astype(np.int32)) if step.parent is not None else None)
        return d

    @classmethod
    def from_host(cls, step, device="cuda") -> "DeviceStep":
        t = cls.tensors_of(step, lambda x: _dev(x, device))
        return cls(**t, temperature=float(step.temperature),
                   mask_kind=L.SV_MASK_TREE if step.mask_kind == "tree" else L.SV_MASK_CAUSAL,
                   max_q=step.max_q, scale=float(step.scale), num_q_heads=int(step.num_q_heads))


@dataclass
class StepBuffers:
    attn_out: torch.Tensor
    workspace: Optional[torch.Tensor]
    sampler_ws: torch.Tensor
    accept: torch.Tensor
    out_tok: torch.Tensor
    num_out: torch.Tensor
    path: torch.Tensor
    status: torch.Tensor
    margin: torch.Tensor  # per sequence: the decisions' smallest distance to a threshold (near-ties < 1e-4)

    @classmethod
    def make(cls, kv: L.PagedKV, dstep: DeviceStep, max_seq_len: int, device="cuda") -> "StepBuffers":
        ws = L.spec_verify_attn_workspace_bytes(kv, dstep.num_q_heads, dstep.total_q, dstep.max_q, max_seq_len)
        B = dstep.batch
        temp = 0.0 if dstep.mask_kind == L.SV_MASK_TREE else dstep.temperature
        sws = L.spec_rejection_sample_workspace_bytes(dstep.target_logits.dtype, int(dstep.target_logits.shape[1]),
                                                      B, dstep.total_q, temp)
        return cls(
            attn_out=torch.empty_like(dstep.q),
            workspace=torch.empty(max(ws, 16), dtype=torch.uint8, device=device) if ws > 0 else None,
            sampler_ws=torch.empty(max(sws, 16), dtype=torch.uint8, device=device),
            accept=torch.empty(B, dtype=torch.int32, device=device),
            out_tok=torch.empty((B, dstep.max_q), dtype=torch.int32, device=device),
            num_out=torch.empty(B, dtype=torch.int32, device=device),
            path=torch.empty((B, dstep.max_q), dtype=torch.int32, device=device),
            status=torch.zeros(1, dtype=torch.int32, device=device),
            margin=torch.empty(B, dtype=torch.float32, device=device))


def append(kv, d: DeviceStep, buf: StepBuffers, stream=None):
    L.kv_append(kv, d.new_k, d.new_v, d.cu_q, buf.status, stream=stream)


def attention(kv, d: DeviceStep, buf: StepBuffers, max_seq_len: int, stream=None):
    L.spec_verify_attn(kv, d.q, buf.attn_out, d.cu_q, max_q=d.max_q, max_seq_len=max_seq_len, scale=d.scale,
                       mask_kind=d.mask_kind, tree_mask=d.tree_mask, workspace=buf.workspace, status=buf.status,
                       stream=stream)


def sample(d: DeviceStep, buf: StepBuffers, stream=None):
    if d.mask_kind == L.SV_MASK_TREE and d.temperature > 0.0:
        L.tree_rejection_sample(d.target_logits, d.cu_q, d.draft_tokens, d.parent, d.u_accept, d.u_resample,
                                d.temperature, buf.accept, buf.path, buf.out_tok, buf.num_out,
                                workspace=buf.sampler_ws, status=buf.status, margin=buf.margin, stream=stream)
    elif d.mask_kind == L.SV_MASK_TREE:
        L.tree_greedy_accept(d.target_logits, d.cu_q, d.draft_tokens, d.parent, buf.accept, buf.path, buf.out_tok,
                             buf.num_out, workspace=buf.sampler_ws, status=buf.status, stream=stream)
    else:
        greedy = d.temperature == 0.0
        L.spec_rejection_sample(d.target_logits, None if greedy else d.draft_logits, d.cu_q, d.draft_tokens,
                                None if greedy else d.u_accept, None if greedy else d.u_resample, d.temperature,
                                buf.accept, buf.out_tok, buf.num_out, workspace=buf.sampler_ws, status=buf.status,
                                margin=buf.margin, stream=stream)


def rollback(kv, d: DeviceStep, buf: StepBuffers, stream=None):
    L.kv_rollback(kv, d.cu_q, buf.accept, buf.status, max_q=d.max_q,
                  path_nodes=buf.path if d.mask_kind == L.SV_MASK_TREE else None, stream=stream)


def run_step(kv: L.PagedKV, d: DeviceStep, buf: StepBuffers, max_seq_len: int, stream=None) -> None:
    """The whole verify step: four library calls on one stream, no host sync."""
    append(kv, d, buf, stream)
    attention(kv, d, buf, max_seq_len, stream)
    sample(d, buf, stream)
    rollback(kv, d, buf, stream)


def launches_per_step(d: DeviceStep, max_seq_len: int, kv: L.PagedKV) -> int:
    """Kernels the library launches for one run_step (append 2, attention 1 or
    2, sampler 2: statistics and decisions, rollback 1 or 2)."""
    ws = L.spec_verify_attn_workspace_bytes(kv, d.num_q_heads, d.total_q, d.max_q, max_seq_len)
    n = 2 + (2 if ws > 0 else 1) + 2 + (2 if d.mask_kind == L.SV_MASK_TREE else 1)
    return n
