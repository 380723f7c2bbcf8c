"""sv_spec_verify_attn_no_alloc, the attention entry point for callers that
cannot allocate device memory: an engine that handed all free HBM to its KV
block pool at start-up, or a host framework that owns the allocator and
forbids a plug-in from calling cudaMalloc. Its split-KV scratch is a static
array inside the library instead of a caller workspace.

Through the C ABI, on every attention path that uses scratch memory, two calls
in a row with different shapes (different query rows per KV head and key
splits, so the second call overwrites the first call's scratch with another
layout) must give exactly the output of sv_spec_verify_attn with a
caller-allocated workspace: the same deterministic kernels on the same inputs,
so bit-identical (torch.equal). The calls must leave the caching allocator's
statistics and, once the library's module is loaded on the device, the
device's free memory unchanged. Sizes that need more scratch than the array
holds are refused on the host.

The file name makes pytest collect it last, so that a run stopping at the
first failure has already run every other test.
"""
import ctypes

import pytest
import torch

from speculative_decoding_verify_paged_gb300 import _lib as L
from speculative_decoding_verify_paged_gb300 import step as S
from speculative_decoding_verify_paged_gb300 import workloads as W

from _helpers import max_seq_len, upload

pytestmark = pytest.mark.gpu


def _cases():
    return [
        W.llama8b(),  # 4 query heads per KV head x 6 rows: 24 rows per unit, 32 sequences
        W.custom(31, batch=5, ctx_lens=[3000, 1500, 40, 700, 2], n_q=[8, 4, 2, 8, 1], num_q_heads=16,
                 num_kv_heads=8, head_dim=128, block_size=16, vocab=16, use_bank=False),  # 2 x 8 rows per unit
    ]


def _prepared(case, path):
    kv, d, buf = upload(case)
    S.append(kv, d, buf)
    msl = max_seq_len(case.state, case.step)
    need = L.spec_verify_attn_workspace_bytes(kv, d.num_q_heads, d.total_q, d.max_q, msl)
    assert 0 < need <= L.ATTN_NO_ALLOC_SCRATCH_BYTES, need
    try:
        S.attention(kv, d, buf, msl)  # the entry point with a caller-allocated workspace
    except L.SVError as e:
        if e.code == 2:
            return None  # this path does not cover the shape
        raise
    return kv, d, buf, msl


def _no_alloc(kv, d, buf, msl, out):
    L.spec_verify_attn_no_alloc(kv, d.q, out, d.cu_q, max_q=d.max_q, max_seq_len=msl, scale=d.scale,
                                mask_kind=d.mask_kind, tree_mask=d.tree_mask, status=buf.status)


def _allocator():
    """The caching allocator's cumulative counts of allocations and of segments it
    took from the device (they only grow), and the bytes it holds (a garbage
    collection between two snapshots may lower them, never raise them)."""
    st = torch.cuda.memory_stats()
    return st.get("allocation.all.allocated", 0), st.get("segment.all.allocated", 0), torch.cuda.memory_reserved()


@pytest.mark.parametrize("path", ["auto", "tensor_cores", "cuda_cores", "warp_mma", "keys_major"])
def test_two_calls_match_the_workspace_entry_point(path):
    L.set_attn_path(path)
    try:
        prepared = [_prepared(c, path) for c in _cases()]
        if any(p is None for p in prepared):
            pytest.skip(f"the {path} path does not cover both shapes")
        outs = [torch.full_like(p[2].attn_out, float("nan")) for p in prepared]
        torch.cuda.synchronize()
        before = _allocator()
        for p, out in zip(prepared, outs):  # back to back on one stream
            _no_alloc(*p, out)
        torch.cuda.synchronize()
        after = _allocator()
        assert after[:2] == before[:2] and after[2] <= before[2], "the caching allocator was used"
        for (kv, d, buf, msl), out in zip(prepared, outs):
            assert int(buf.status.item()) == 0
            assert torch.equal(out, buf.attn_out)
        # the module holding the array is loaded now: two more calls leave the device's free memory as it was
        free0 = torch.cuda.mem_get_info()[0]
        for p, out in zip(prepared, outs):
            out.fill_(float("nan"))
            _no_alloc(*p, out)
        torch.cuda.synchronize()
        assert torch.cuda.mem_get_info()[0] == free0, "device memory was allocated"
        for (kv, d, buf, msl), out in zip(prepared, outs):
            assert torch.equal(out, buf.attn_out)
    finally:
        L.set_attn_path("auto")


def test_sizes_beyond_the_static_scratch_are_refused():
    lib = L.load()
    s = L.sv_paged_kv()  # sizes only: a refused call touches no pointer
    s.num_blocks, s.block_size, s.max_blocks_per_seq, s.num_kv_heads, s.head_dim, s.batch = 4096, 16, 256, 8, 128, 1
    hq, total_q, max_q, msl = 64, 64, 64, 4096
    need = lib.sv_spec_verify_attn_workspace_bytes(ctypes.byref(s), hq, total_q, max_q, msl)
    assert need > L.ATTN_NO_ALLOC_SCRATCH_BYTES
    rc = lib.sv_spec_verify_attn_no_alloc(ctypes.byref(s), None, None, None, hq, total_q, max_q, msl, 0.088,
                                          L.SV_MASK_CAUSAL, None, None, None)
    assert rc == L.SV_ERR_WORKSPACE
