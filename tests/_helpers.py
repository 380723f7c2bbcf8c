"""Shared helpers of the GPU parity tests (not collected as tests)."""
import numpy as np
import torch

import oracle
from speculative_decoding_verify_paged_gb300 import step as S
from speculative_decoding_verify_paged_gb300 import workloads as W

NEAR_TIE = 1e-4          # |u - min(1, p/q)| or CDF-crossing distance that counts as a near-tie
MAX_TIE_FRACTION = 1e-4  # divergent decisions allowed, as a fraction of verified positions


def max_seq_len(state, step, slack=0):
    return int((state.seq_lens + step.n_q).max()) + slack


def upload(case, device="cuda"):
    kv = S.device_kv(case.state, device)
    d = S.DeviceStep.from_host(case.step, device)
    buf = S.StepBuffers.make(kv, d, max_seq_len(case.state, case.step), device)
    return kv, d, buf


def status_of(buf):
    return int(buf.status.item())


def attn_as_f64(t):
    t = t.detach().float().cpu().numpy()
    return t.astype(np.float64)


def assert_attn_close(gpu, ref, rows=None, rel=1e-2):
    """max-abs error <= rel * max|ref| over the compared rows."""
    g = gpu if rows is None else gpu[rows]
    r = ref if rows is None else ref[rows]
    scale = np.abs(r).max()
    err = np.abs(g - r).max()
    assert err <= rel * scale, f"attention max-abs error {err:.3e} > {rel} * {scale:.3e}"
    return err, scale


def rows_of(step, seqs):
    return np.concatenate([np.arange(step.cu_q[b], step.cu_q[b + 1]) for b in seqs])


def compare_samples(step, gpu, ref, *, tree=False, max_fraction=MAX_TIE_FRACTION):
    """Bit-exact decisions except at oracle-flagged near-ties, whose count must stay
    below MAX_TIE_FRACTION of the verified positions. Returns the number of
    sequences that diverged at a near-tie."""
    acc, tok, num = gpu
    B = step.n_q.shape[0]
    diverged = 0
    details = []
    for b in range(B):
        same = (acc[b] == ref.accept_cnt[b] and num[b] == ref.num_out[b]
                and np.array_equal(tok[b], ref.out_tok[b]))
        if tree:
            assert same, f"tree sequence {b}: gpu {acc[b]} {tok[b]} vs oracle {ref.accept_cnt[b]} {ref.out_tok[b]}"
            continue
        if not same:
            m = ref.margin[b] if ref.margin is not None else np.inf
            assert m < NEAR_TIE, (f"sequence {b}: gpu a={acc[b]} tok={tok[b]} vs oracle a={ref.accept_cnt[b]} "
                                  f"tok={ref.out_tok[b]} with margin {m:.3e}")
            diverged += 1
            details.append(f"seq {b} (K={int(step.n_q[b]) - 1}): gpu a={acc[b]} y={tok[b][acc[b]]} vs oracle "
                           f"a={ref.accept_cnt[b]} y={ref.out_tok[b][ref.accept_cnt[b]]}, margin {m:.2e}")
    positions = int(step.n_q.sum())
    if max_fraction is not None:
        assert diverged <= max_fraction * positions, (f"{diverged} near-tie divergences in {positions} positions: "
                                                      + "; ".join(details))
    return diverged


def gpu_sample_result(buf):
    return (buf.accept.cpu().numpy(), buf.out_tok.cpu().numpy(), buf.num_out.cpu().numpy())


def kv_host(kv):
    return dict(block_table=kv.block_table.cpu().numpy(), seq_lens=kv.seq_lens.cpu().numpy(),
                free_list=kv.free_list.cpu().numpy(), free_top=int(kv.free_top.item()))


def assert_kv_equal(kv, okv, pools=True, rows=None):
    h = kv_host(kv)
    np.testing.assert_array_equal(h["block_table"], okv.block_table())
    np.testing.assert_array_equal(h["seq_lens"], np.array(okv.seq_lens, np.int32))
    assert h["free_top"] == len(okv.free)
    np.testing.assert_array_equal(h["free_list"], okv.free_list())
    if pools:
        kp, vp = S.to_bits(kv.k_pool), S.to_bits(kv.v_pool)
        if rows is None:
            np.testing.assert_array_equal(kp, okv.k_pool)
            np.testing.assert_array_equal(vp, okv.v_pool)
        else:
            for (blk, slot) in rows:
                np.testing.assert_array_equal(kp[blk, :, slot], okv.k_pool[blk, :, slot])
                np.testing.assert_array_equal(vp[blk, :, slot], okv.v_pool[blk, :, slot])


def appended_rows(okv, step, c0):
    """(physical block, slot) of every row the step appended, from the oracle's table."""
    out = []
    for b in range(len(c0)):
        for j in range(int(step.n_q[b])):
            pos = c0[b] + j
            out.append((okv.bt[b][pos // okv.bs], pos % okv.bs))
    return out
