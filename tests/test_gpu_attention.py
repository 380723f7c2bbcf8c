"""GPU parity of sv_spec_verify_attn against the fp64 oracle.

Bar: max-abs error <= 1e-2 * max|out| for bf16 KV with fp32 accumulation
(the stated tolerance), 1e-4 for fp32 KV. Small cases are compared in full
(several key tiles, several splits, ragged tails, every block size); so are
the full-size workloads, every query row of every sequence, in the launch
configuration the benchmark uses: the persistent kernel's split of the key
tiles (and so which units two CTAs share and merge) depends on the whole
batch, so a sample of sequences could miss a wrong merge.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_paged_gb300 import _lib as L
from speculative_decoding_verify_paged_gb300 import step as S
from speculative_decoding_verify_paged_gb300 import workloads as W

from _helpers import assert_attn_close, attn_as_f64, max_seq_len, rows_of, status_of, upload

pytestmark = pytest.mark.gpu


def _run(case, seqs=None, rel=None, slack=0, path="auto"):
    L.set_attn_path(path)
    try:
        return _run_path(case, seqs, rel, slack)
    finally:
        L.set_attn_path("auto")


def _run_path(case, seqs, rel, slack):
    kv, d, buf = upload(case)
    okv = oracle.OracleKV(case.state)
    assert okv.append(case.step) is None
    S.append(kv, d, buf)
    msl = max_seq_len(case.state, case.step, slack)
    if slack:
        buf = S.StepBuffers.make(kv, d, msl)
    S.attention(kv, d, buf, msl)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    ref = oracle.paged_attention(okv.as_state(), case.step, seqs=seqs)
    got = attn_as_f64(buf.attn_out)
    rows = None if seqs is None else rows_of(case.step, seqs)
    if rel is None:
        rel = 1e-4 if case.state.dtype == "f32" else 1e-2
    return assert_attn_close(got, ref, rows, rel)


def test_tiny_fp32():
    _run(W.tiny())


SMALL = {
    # name: (seed, ctx, n_q, hq, hkv, d, bs, dtype)
    "bf16-g4-bs16": (11, [700, 65, 1, 300], [6, 6, 6, 6], 32, 8, 128, 16, "bf16"),
    "bf16-g8-bs16": (12, [513, 640, 100], [5, 5, 5], 64, 8, 128, 16, "bf16"),
    "bf16-ragged-bs128": (13, [16, 900, 255, 129, 1], [3, 9, 2, 5, 1], 32, 8, 128, 128, "bf16"),
    "bf16-bs64": (14, [191, 64, 63], [4, 4, 4], 16, 4, 128, 64, "bf16"),
    "bf16-bs256": (15, [700, 255], [6, 2], 16, 2, 128, 256, "bf16"),
    "bf16-d64": (16, [333, 47], [5, 3], 8, 2, 64, 16, "bf16"),
    "f32-d128": (17, [400, 3], [6, 4], 8, 2, 128, 32, "f32"),
    "bf16-empty-ctx": (18, [0, 0, 5], [1, 7, 2], 8, 2, 128, 16, "bf16"),
    "bf16-mqa": (19, [200, 90], [5, 5], 8, 1, 128, 16, "bf16"),
}


@pytest.mark.parametrize("path", ["auto", "cuda_cores", "warp_mma", "tensor_cores", "keys_major"])
@pytest.mark.parametrize("name", list(SMALL))
def test_small_cases(name, path):
    seed, ctx, nq, hq, hkv, d, bs, dt = SMALL[name]
    case = W.custom(seed, batch=len(ctx), ctx_lens=ctx, n_q=nq, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                    block_size=bs, vocab=16, dtype=dt, use_bank=False)
    if path in ("warp_mma", "tensor_cores", "keys_major") and (dt != "bf16" or d != 128):
        pytest.skip("the tensor-core kernels cover bf16 with head_dim 128")
    if path == "keys_major" and (hq // hkv) * max(nq) > 32:
        pytest.skip("the keys-major kernel covers units of at most 32 query rows")
    _run(case, path=path)


def test_keys_major_refuses_wide_units():
    """More than 32 query rows in a unit: the keys-major path is unsupported."""
    case = W.custom(27, batch=2, ctx_lens=[300, 40], n_q=[5, 5], num_q_heads=64, num_kv_heads=8, head_dim=128,
                    block_size=16, vocab=16, use_bank=False)
    kv, d, buf = upload(case)
    L.set_attn_path("keys_major")
    try:
        with pytest.raises(L.SVError) as e:
            S.attention(kv, d, buf, max_seq_len(case.state, case.step))
        assert e.value.code == 2
    finally:
        L.set_attn_path("auto")


def test_tensor_core_path_refuses_unsupported_shapes():
    case = W.custom(26, batch=2, ctx_lens=[30, 40], n_q=[3, 3], num_q_heads=8, num_kv_heads=2, head_dim=64,
                    block_size=16, vocab=16, use_bank=False)
    kv, d, buf = upload(case)
    L.set_attn_path("tensor_cores")
    try:
        with pytest.raises(L.SVError) as e:
            S.attention(kv, d, buf, max_seq_len(case.state, case.step))
        assert e.value.code == 2
    finally:
        L.set_attn_path("auto")


def test_small_case_with_loose_length_bound():
    """max_seq_len well above the real lengths: more (empty) splits, same answer."""
    case = W.custom(21, batch=3, ctx_lens=[100, 10, 250], n_q=[6, 6, 6], num_q_heads=32, num_kv_heads=8,
                    head_dim=128, block_size=16, vocab=16, use_bank=False)
    _run(case, slack=3000)


def test_chain_tree_mask_equals_causal():
    case = W.custom(22, batch=2, ctx_lens=[300, 70], n_q=[6, 4], num_q_heads=32, num_kv_heads=8, head_dim=128,
                    block_size=16, vocab=16, use_bank=False)
    kv, d, buf = upload(case)
    S.append(kv, d, buf)
    msl = max_seq_len(case.state, case.step)
    S.attention(kv, d, buf, msl)
    causal = buf.attn_out.clone()
    masks = np.concatenate([np.array([(1 << (i + 1)) - 1 for i in range(int(n))], np.uint64)
                            for n in case.step.n_q])
    d.tree_mask = torch.from_numpy(masks.view(np.int64)).cuda()
    d.mask_kind = L.SV_MASK_TREE
    S.attention(kv, d, buf, msl)
    torch.cuda.synchronize()
    assert torch.equal(causal, buf.attn_out)


@pytest.mark.parametrize("path", ["auto", "cuda_cores", "warp_mma"])
def test_tree_small(path):
    case = W.tree(batch=2, ctx=333, vocab=256)
    _run(case, path=path)


FULL_PATHS = {
    "llama8b": ["auto", "keys_major", "cuda_cores", "warp_mma"],
    "llama70b": ["auto", "warp_mma", "cuda_cores"],  # 8 query heads x 5 rows per KV head: too wide for keys-major
    "contbatch": ["auto"],
    "tree": ["auto", "warp_mma", "cuda_cores"],
}


@pytest.mark.parametrize("name", list(FULL_PATHS))
def test_full_size_every_sequence(name):
    """Every query row of every sequence of the full-size workload, on each
    attention path that covers it; the oracle's reference is computed once."""
    case = W.CONFIGS[name]()
    kv, d, buf = upload(case)
    okv = oracle.OracleKV(case.state)
    assert okv.append(case.step) is None
    S.append(kv, d, buf)
    msl = max_seq_len(case.state, case.step)
    ref = oracle.paged_attention(okv.as_state(), case.step)
    del okv
    for path in FULL_PATHS[name]:
        L.set_attn_path(path)
        try:
            buf.attn_out.fill_(float("nan"))
            S.attention(kv, d, buf, msl)
            torch.cuda.synchronize()
        finally:
            L.set_attn_path("auto")
        assert status_of(buf) == 0, path
        got = attn_as_f64(buf.attn_out)
        assert np.isfinite(got).all(), f"{path}: rows left unwritten"
        assert_attn_close(got, ref)


def test_bad_block_id_is_reported():
    case = W.custom(23, batch=2, ctx_lens=[100, 40], n_q=[3, 3], num_q_heads=8, num_kv_heads=2, head_dim=128,
                    block_size=16, vocab=16, use_bank=False)
    kv, d, buf = upload(case)
    S.append(kv, d, buf)
    torch.cuda.synchronize()
    kv.block_table[1, 0] = case.state.num_blocks + 5
    S.attention(kv, d, buf, max_seq_len(case.state, case.step))
    torch.cuda.synchronize()
    assert status_of(buf) == 6


def test_too_long_sequence_is_reported():
    case = W.custom(24, batch=2, ctx_lens=[100, 40], n_q=[3, 3], num_q_heads=8, num_kv_heads=2, head_dim=128,
                    block_size=16, vocab=16, use_bank=False)
    kv, d, buf = upload(case)
    S.append(kv, d, buf)
    S.attention(kv, d, buf, 50)  # sequence 0 has 103 tokens
    torch.cuda.synchronize()
    assert status_of(buf) == 7


def test_workspace_is_checked():
    case = W.custom(25, batch=1, ctx_lens=[2000], n_q=[6], num_q_heads=32, num_kv_heads=8, head_dim=128,
                    block_size=16, vocab=16, use_bank=False)
    kv, d, buf = upload(case)
    msl = max_seq_len(case.state, case.step)
    need = L.spec_verify_attn_workspace_bytes(kv, 32, d.total_q, d.max_q, msl)
    assert need > 0
    with pytest.raises(L.SVError) as e:
        L.spec_verify_attn(kv, d.q, buf.attn_out, d.cu_q, max_q=d.max_q, max_seq_len=msl, scale=d.scale,
                           workspace=None, status=buf.status)
    assert e.value.code == 10
