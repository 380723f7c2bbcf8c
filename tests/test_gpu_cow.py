"""GPU parity of copy-on-write block sharing (sv_kv_fork, sv_kv_append and
sv_kv_rollback with reference counts, sv_kv_release) against the oracle.

Parallel sampling: 8 parent sequences are forked into 3 children each, then
every one of the 32 sequences runs verify steps of its own (greedy, so every
decision is exact); some finish and give their blocks back. Block tables,
lengths, the free list, the reference counts and both pools must equal the
oracle's after every call, and the attention over shared blocks must match.
"""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_paged_gb300 import _lib as L
from speculative_decoding_verify_paged_gb300 import step as S
from speculative_decoding_verify_paged_gb300 import workloads as W

from _helpers import assert_attn_close, assert_kv_equal, attn_as_f64, gpu_sample_result, rows_of, status_of

pytestmark = pytest.mark.gpu


def _assert_same(kv, okv):
    assert_kv_equal(kv, okv, pools=True)
    np.testing.assert_array_equal(kv.ref_count.cpu().numpy(), okv.ref_count())


def _step(seed, it, K, B):
    return W.make_chain_step(seed, K + 1, num_q_heads=32, num_kv_heads=8, head_dim=128, qkv_dtype="bf16",
                             vocab=4096, logits_dtype="bf16", target_sigma=3.0, draft_coef=0.8, draft_sigma=1.0,
                             temperature=0.0, stream=100 + it)


def _verify(kv, okv, step, msl, attn_seqs):
    d = S.DeviceStep.from_host(step)
    buf = S.StepBuffers.make(kv, d, msl)
    S.append(kv, d, buf)
    assert okv.append(step) is None
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    # mid-step: the new rows (and any private copies) are in place
    np.testing.assert_array_equal(kv.ref_count.cpu().numpy(), okv.ref_count())
    np.testing.assert_array_equal(kv.block_table.cpu().numpy(), okv.block_table())
    S.attention(kv, d, buf, msl)
    S.sample(d, buf)
    torch.cuda.synchronize()
    ref = oracle.paged_attention(okv.as_state(), step, seqs=attn_seqs)
    assert_attn_close(attn_as_f64(buf.attn_out), ref, rows_of(step, attn_seqs))
    acc = oracle.rejection_sample(step).accept_cnt
    np.testing.assert_array_equal(gpu_sample_result(buf)[0], acc)  # greedy: exact
    S.rollback(kv, d, buf)
    okv.rollback(step, acc)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    _assert_same(kv, okv)


@pytest.mark.parametrize("kv_dtype", ["bf16", "e4m3"])
def test_parallel_sampling_fork_step_release(kv_dtype):
    seed, P, C = 11, 8, 3
    B = P * (C + 1)
    rng = np.random.default_rng(seed)
    ctx = np.zeros(B, np.int32)
    ctx[:P] = rng.integers(40, 200, size=P)  # partial last blocks (block size 16) in most parents
    st = W.make_kv_state(seed, ctx, block_size=16, num_kv_heads=8, head_dim=128, dtype=kv_dtype,
                         growth_tokens=200 + 40, pool_factor=1.2)
    okv = oracle.OracleKV(st)
    okv.enable_sharing()
    kv = S.device_kv(st, ref_count=okv.ref_count())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    parents = np.repeat(np.arange(P), C).astype(np.int32)
    children = np.arange(P, B).astype(np.int32)
    L.kv_fork(kv, torch.from_numpy(parents).cuda(), torch.from_numpy(children).cuda(), status)
    assert okv.fork(parents, children) is None
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _assert_same(kv, okv)
    assert okv.ref_count().max() == C + 1
    msl = int(ctx.max()) + 5 * 9 + 16
    for it in range(3):
        K = rng.integers(2, 8, size=B).astype(np.int32)
        _verify(kv, okv, _step(seed, it, K, B), msl, [0, P, P + 1, B - 1])
    # finished sequences give their blocks back: a parent and one of its children,
    # then another parent with all of its children
    done = np.array([0, P, 1, P + 3, P + 4, P + 5], np.int32)
    L.kv_release(kv, torch.from_numpy(done).cuda(), status)
    assert okv.release(done) is None
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    _assert_same(kv, okv)
    # another step over every slot: the released ones start over from fresh blocks
    K = rng.integers(2, 8, size=B).astype(np.int32)
    _verify(kv, okv, _step(seed, 9, K, B), msl, [2, P + 6])


def test_fork_and_release_refusals_change_nothing():
    seed = 12
    ctx = np.array([30, 0, 17, 0], np.int32)
    st = W.make_kv_state(seed, ctx, block_size=16, num_kv_heads=8, head_dim=128, dtype="bf16", growth_tokens=32)
    okv = oracle.OracleKV(st)
    okv.enable_sharing()
    kv = S.device_kv(st, ref_count=okv.ref_count())
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t = lambda a: torch.tensor(a, dtype=torch.int32, device="cuda")
    bad_length = 7
    cases = [
        (lambda: L.kv_fork(kv, t([0]), t([2]), status), bad_length),  # child not empty
        (lambda: L.kv_fork(kv, t([0, 2]), t([1, 1]), status), bad_length),  # the same child twice
        (lambda: L.kv_fork(kv, t([0, 1]), t([1, 3]), status), bad_length),  # a child is also a parent
        (lambda: L.kv_fork(kv, t([0]), t([9]), status), bad_length),  # out of range
        (lambda: L.kv_release(kv, t([0, 0]), status), bad_length),  # the same sequence twice
    ]
    for call, code in cases:
        status.zero_()
        call()
        torch.cuda.synchronize()
        assert int(status.item()) == code
        _assert_same(kv, okv)
    # a call made while the status word holds an error does nothing
    status.fill_(5)
    L.kv_fork(kv, t([0]), t([1]), status)
    L.kv_release(kv, t([2]), status)
    torch.cuda.synchronize()
    _assert_same(kv, okv)
    # host-side refusal: fork without reference counts
    kv_plain = S.device_kv(st)
    with pytest.raises(L.SVError):
        L.kv_fork(kv_plain, t([0]), t([1]), status)
