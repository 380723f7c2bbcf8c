"""Failure detection on the GPU without a fault: a pipeline wait that never
completes must end the kernel with SV_ERR_TIMEOUT in the status word, within
the wait budget, and leave the context usable.

The failure is made on purpose by the library's test hook
(SV_OPT_STALL_FOR_TEST): the producer warp of the tensor-core attention kernel,
or of the sampler's statistics kernel, waits on a barrier that nothing ever
completes, as a producer whose data never arrives would. With the budget cut to
a few milliseconds (SV_OPT_WAIT_BUDGET_US), that wait runs out, the producer
issues no copy, and every consumer's wait runs out in turn; the kernels then
let the copies and matrix operations they issued finish and free their tensor
memory before they end. Nothing traps, faults or hangs. The next call on the
same stream, with the hook off, must pass parity with the oracle.
"""
import time

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_paged_gb300 import _lib as L
from speculative_decoding_verify_paged_gb300 import step as S
from speculative_decoding_verify_paged_gb300 import workloads as W

from _helpers import assert_attn_close, attn_as_f64, compare_samples, gpu_sample_result, max_seq_len, status_of, upload

pytestmark = pytest.mark.gpu

BUDGET_US = 2000


def _case():
    return W.custom(51, batch=4, ctx_lens=[700, 65, 1, 300], n_q=[6, 6, 6, 6], num_q_heads=32, num_kv_heads=8,
                    head_dim=128, block_size=16, vocab=4096, dtype="bf16", use_bank=False)


def _stalled(call, which):
    """Runs `call` with the stall hook on and a short budget; returns its wall time."""
    L.set_wait_budget_us(BUDGET_US)
    L.set_stall_for_test(which)
    try:
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        call()
        torch.cuda.synchronize()
        return time.perf_counter() - t0
    finally:
        L.set_stall_for_test("none")
        L.set_wait_budget_us(L.DEFAULT_WAIT_BUDGET_US)


def test_attention_wait_runs_out_then_recovers():
    case = _case()
    kv, d, buf = upload(case)
    S.append(kv, d, buf)
    msl = max_seq_len(case.state, case.step)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    secs = _stalled(lambda: S.attention(kv, d, buf, msl), "attention")
    assert status_of(buf) == L.SV_ERR_TIMEOUT
    assert secs < 1.0, f"the stalled call took {secs:.3f} s"
    # the same stream, the hook off: the context is usable and the result right
    buf.status.zero_()
    buf.attn_out.fill_(float("nan"))
    S.attention(kv, d, buf, msl)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    okv = oracle.OracleKV(case.state)
    assert okv.append(case.step) is None
    assert_attn_close(attn_as_f64(buf.attn_out), oracle.paged_attention(okv.as_state(), case.step))


def test_sampler_wait_runs_out_then_recovers():
    case = _case()
    kv, d, buf = upload(case)
    secs = _stalled(lambda: S.sample(d, buf), "sampler")
    assert status_of(buf) == L.SV_ERR_TIMEOUT
    assert secs < 1.0, f"the stalled call took {secs:.3f} s"
    buf.status.zero_()
    S.sample(d, buf)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    compare_samples(case.step, gpu_sample_result(buf), oracle.rejection_sample(case.step))
