"""GPU parity of the fp8 (E4M3) KV pool against the oracle: the codes the
append stores are bit-exact, attention over the dequantised pool is within the
bf16 bar (1e-2 * max|out|; both sides read code * scale exactly), and whole
verify steps keep tables, lengths and pools equal to the oracle's."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_paged_gb300 import _lib as L
from speculative_decoding_verify_paged_gb300 import step as S
from speculative_decoding_verify_paged_gb300 import workloads as W

from _helpers import (assert_attn_close, assert_kv_equal, attn_as_f64, compare_samples, gpu_sample_result, max_seq_len,
                      rows_of, status_of, upload)

pytestmark = pytest.mark.gpu


def _case(seed=31, **kw):
    args = dict(batch=3, ctx_lens=[100, 17, 260], n_q=[4, 6, 2], num_q_heads=8, num_kv_heads=2, head_dim=128,
                block_size=16, vocab=64)
    args.update(kw)
    return W.custom(seed, dtype="e4m3", use_bank=False, **args)


def test_append_stores_the_oracles_codes():
    case = _case()
    kv, d, buf = upload(case)
    assert kv.k_pool.dtype == torch.uint8
    okv = oracle.OracleKV(case.state)
    assert okv.append(case.step) is None
    S.append(kv, d, buf)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    np.testing.assert_array_equal(kv.k_pool.cpu().numpy(), okv.k_pool)
    np.testing.assert_array_equal(kv.v_pool.cpu().numpy(), okv.v_pool)


FP8_CASES = {
    # name: keyword arguments of the e4m3 custom case
    "g4-bs16": {},
    "g4-bs64": {"block_size": 64, "ctx_lens": [700, 3, 129]},
    "g4-bs32-llama": {"num_q_heads": 32, "num_kv_heads": 8, "n_q": [6, 6, 6], "block_size": 32},
    "g8-bs256": {"num_q_heads": 16, "num_kv_heads": 2, "block_size": 256, "ctx_lens": [600, 255, 1]},
    "g16-wide-unit": {"num_q_heads": 32, "num_kv_heads": 2, "n_q": [9, 6, 2]},
    "empty-ctx": {"ctx_lens": [0, 0, 40], "n_q": [1, 7, 3]},
    "d64": {"head_dim": 64, "num_q_heads": 4, "num_kv_heads": 4},
}


def _attention(case, path):
    kv, d, buf = upload(case)
    okv = oracle.OracleKV(case.state)
    assert okv.append(case.step) is None
    S.append(kv, d, buf)
    msl = max_seq_len(case.state, case.step)
    L.set_attn_path(path)
    try:
        S.attention(kv, d, buf, msl)
        torch.cuda.synchronize()
    finally:
        L.set_attn_path("auto")
    assert status_of(buf) == 0
    return attn_as_f64(buf.attn_out), okv


@pytest.mark.parametrize("path", ["auto", "cuda_cores", "tensor_cores"])
@pytest.mark.parametrize("name", list(FP8_CASES))
def test_attention_over_fp8_pool(name, path):
    case = _case(32, **FP8_CASES[name])
    if path == "tensor_cores" and case.state.head_dim != 128:
        pytest.skip("the tensor-core kernel covers head_dim 128")
    got, okv = _attention(case, path)
    ref = oracle.paged_attention(okv.as_state(), case.step)
    assert_attn_close(got, ref, None, 1e-2)


def test_tree_mask_over_fp8_pool():
    case = W.tree(batch=2, ctx=700, block_size=64, kv_dtype="e4m3", vocab=512)
    got, okv = _attention(case, "auto")
    ref = oracle.paged_attention(okv.as_state(), case.step)
    assert_attn_close(got, ref, None, 1e-2)


def test_query_beyond_fp16_range_is_reported():
    """The tensor-core kernel rounds queries to fp16 for an fp8 pool: a query
    element past 65504 records SV_ERR_NONFINITE instead of scoring with inf."""
    case = _case(34, num_q_heads=32, num_kv_heads=8, n_q=[6, 6, 6])
    case.step.q[1, 3, 17] = 0x4880  # bf16 bits of 2^18
    kv, d, buf = upload(case)
    S.append(kv, d, buf)
    L.set_attn_path("tensor_cores")
    try:
        S.attention(kv, d, buf, max_seq_len(case.state, case.step))
        torch.cuda.synchronize()
    finally:
        L.set_attn_path("auto")
    assert status_of(buf) == L.SV_ERR_NONFINITE


def test_steps_with_fp8_pool():
    """Three greedy verify steps of a llama8b-shaped batch of 6 on an fp8 pool."""
    case = W.llama8b(batch=6, ctx_range=(100, 900), vocab=4096, growth_tokens=24, kv_dtype="e4m3",
                     temperature=0.0)
    kv = S.device_kv(case.state)
    okv = oracle.OracleKV(case.state)
    msl = int(case.state.seq_lens.max()) + 3 * 6 + 16
    for it in range(3):
        step = case.step if it == 0 else W.make_chain_step(
            case.seed, case.step.n_q, num_q_heads=32, num_kv_heads=8, head_dim=128, qkv_dtype="bf16", vocab=4096,
            logits_dtype="bf16", target_sigma=3.0, draft_coef=0.8, draft_sigma=1.5, temperature=0.0, stream=it)
        d = S.DeviceStep.from_host(step)
        buf = S.StepBuffers.make(kv, d, msl)
        S.append(kv, d, buf)
        S.attention(kv, d, buf, msl)
        S.sample(d, buf)
        assert okv.append(step) is None
        torch.cuda.synchronize()
        ref = oracle.paged_attention(okv.as_state(), step, seqs=[0, 5])
        assert_attn_close(attn_as_f64(buf.attn_out), ref, rows_of(step, [0, 5]))
        rs = oracle.rejection_sample(step)
        got = gpu_sample_result(buf)
        compare_samples(step, got, rs)  # bit-exact except at near-ties, which are bounded
        if not np.array_equal(got[0], rs.accept_cnt):
            buf.accept.copy_(torch.from_numpy(rs.accept_cnt))
        S.rollback(kv, d, buf)
        okv.rollback(step, rs.accept_cnt)
        torch.cuda.synchronize()
        assert status_of(buf) == 0
        assert_kv_equal(kv, okv, pools=False)
        np.testing.assert_array_equal(kv.k_pool.cpu().numpy(), okv.k_pool)
        np.testing.assert_array_equal(kv.v_pool.cpu().numpy(), okv.v_pool)


def test_fp8_pool_arguments_are_checked():
    case = _case(33)
    kv, d, buf = upload(case)
    kv.k_scale = 0.0
    with pytest.raises(L.SVError):
        S.append(kv, d, buf)
