"""sv_spec_verify_attn_no_alloc, the attention entry point for callers that
cannot allocate device memory: an engine that handed all free HBM to its KV
block pool at start-up, or a host framework that owns the allocator and
forbids a plug-in from calling cudaMalloc. Its split-KV scratch is a static
array inside the library instead of a caller workspace.

Through the C ABI, two calls in a row (different shapes, both split along the
keys so that the scratch is really used, the second overwriting what the
first left there) must give the output of sv_spec_verify_attn with a
caller-allocated workspace, within the attention tolerance of the other
tests (max-abs error <= 1e-2 * max|out| for bf16). Sizes that need more
scratch than the array holds are refused on the host.

The file name makes pytest collect it last, so that a run stopping at the
first failure has already run every other test.
"""
import ctypes

import pytest
import torch

from speculative_decoding_verify_paged_gb300 import _lib as L
from speculative_decoding_verify_paged_gb300 import step as S
from speculative_decoding_verify_paged_gb300 import workloads as W

from _helpers import assert_attn_close, attn_as_f64, max_seq_len, upload

pytestmark = pytest.mark.gpu


def _prepared(case):
    kv, d, buf = upload(case)
    S.append(kv, d, buf)
    msl = max_seq_len(case.state, case.step)
    need = L.spec_verify_attn_workspace_bytes(kv, d.num_q_heads, d.total_q, d.max_q, msl)
    assert 0 < need <= L.ATTN_NO_ALLOC_SCRATCH_BYTES, need
    S.attention(kv, d, buf, msl)  # the entry point with a caller-allocated workspace
    return kv, d, buf, msl


def test_two_calls_match_the_workspace_entry_point():
    L.set_attn_path("auto")
    cases = [W.llama8b(),
             W.custom(31, batch=3, ctx_lens=[3000, 1500, 40], n_q=[6, 4, 2], num_q_heads=32, num_kv_heads=8,
                      head_dim=128, block_size=16, vocab=16, use_bank=False)]
    prepared = [_prepared(c) for c in cases]
    torch.cuda.synchronize()
    outs = []
    for kv, d, buf, msl in prepared:  # back to back on one stream
        out = torch.full_like(buf.attn_out, float("nan"))
        L.spec_verify_attn_no_alloc(kv, d.q, out, d.cu_q, max_q=d.max_q, max_seq_len=msl, scale=d.scale,
                                    mask_kind=d.mask_kind, tree_mask=d.tree_mask, status=buf.status)
        outs.append(out)
    torch.cuda.synchronize()
    for (kv, d, buf, msl), out in zip(prepared, outs):
        assert int(buf.status.item()) == 0
        assert_attn_close(attn_as_f64(out), attn_as_f64(buf.attn_out), rel=1e-2)


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
