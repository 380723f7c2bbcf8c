"""The benchmark's algorithmic byte and flop counts (the roofline numerators),
checked against hand counts of small cases: every visible K and V row once, Q
in and O out; every target row (and at T > 0 every draft row) once."""
import importlib.util
import os

import numpy as np

from speculative_decoding_verify_paged_gb300 import workloads as W

_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
_spec = importlib.util.spec_from_file_location("bench_module", os.path.join(_ROOT, "bench.py"))
bench = importlib.util.module_from_spec(_spec)
_spec.loader.exec_module(bench)


def _case(dtype, T=1.0):
    return W.custom(3, batch=2, ctx_lens=[10, 30], n_q=[3, 5], num_q_heads=8, num_kv_heads=2, head_dim=64,
                    block_size=16, vocab=100, dtype=dtype, temperature=T, use_bank=False)


def test_attention_bytes_by_pool_type():
    for dtype, kv_el, io_el in (("bf16", 2, 2), ("f32", 4, 4), ("e4m3", 1, 2)):
        c = _case(dtype)
        lens = c.state.seq_lens + c.step.n_q  # 13 and 35 visible keys
        want = (13 + 35) * 2 * 2 * 64 * kv_el + 2 * 8 * 8 * 64 * io_el  # K and V rows; Q in, O out (8 rows)
        assert bench.attn_bytes(lens, c.step, c.state) == want


def test_sampler_bytes():
    c = _case("bf16", T=1.0)
    assert bench.sampler_bytes(c.step) == (8 + 6) * 100 * 2  # 8 target rows, 6 draft rows
    g = _case("bf16", T=0.0)
    assert bench.sampler_bytes(g.step) == 8 * 100 * 2  # greedy reads the target rows only
    t = W.tree(batch=2, ctx=40, block_size=16, vocab=64)
    assert bench.sampler_bytes(t.step) == t.step.total_q * 64 * 2


def test_attention_flops():
    c = _case("bf16")
    ctx = c.state.seq_lens.astype(np.float64)
    # per query row i (0-based) of sequence b: c_b + i + 1 visible keys, 2 * D flops each for
    # q.k and 2 * D for p.v, per query head
    want = sum(4 * 8 * 64 * (ctx[b] + i + 1) for b in range(2) for i in range(int(c.step.n_q[b])))
    assert abs(bench.attn_flops(ctx, c.step, 4) - want) < 1e-6 * want
