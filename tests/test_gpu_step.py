"""The whole verify step through the C ABI, iterated: the continuous-batching
workload (256 sequences, lognormal contexts, K_b ~ U{2..8} redrawn every
iteration, 128-token blocks from a fragmented free list) runs 10 iterations of
append -> attention -> rejection sample -> rollback on the GPU and in the
oracle. Block tables, seq_lens, the free list and every emitted token must be
bit-exact at every iteration; attention is compared on every sequence at the
first and the last iteration.

A decision may differ from the oracle only at an oracle-flagged near-tie, and
such divergences, counted over the whole run, must stay below 0.01% of the
verified positions. After one, the GPU rollback is given the oracle's accept
counts for that step (oracle output into the GPU, never the reverse), so the
caches stay comparable in the iterations that follow."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verify_paged_gb300 import step as S
from speculative_decoding_verify_paged_gb300 import workloads as W

from _helpers import (MAX_TIE_FRACTION, assert_attn_close, assert_kv_equal, attn_as_f64, compare_samples,
                      gpu_sample_result, rows_of, status_of, upload)

pytestmark = pytest.mark.gpu


def _loop(case, iterations, steps_of, attn_check_iters, attn_seqs, with_pools, observe=None):
    st = case.state
    kv = S.device_kv(st)
    okv = oracle.OracleKV(st, with_pools=with_pools)
    msl = int(st.seq_lens.max()) + 9 * iterations + 16
    accepted = []
    diverged, positions = 0, 0
    for it in range(iterations):
        step = steps_of(it)
        d = S.DeviceStep.from_host(step)
        buf = S.StepBuffers.make(kv, d, msl)
        S.append(kv, d, buf)
        S.attention(kv, d, buf, msl)
        S.sample(d, buf)
        assert okv.append(step) is None
        if it in attn_check_iters:
            torch.cuda.synchronize()
            ref = oracle.paged_attention(okv.as_state(), step, seqs=attn_seqs)
            assert_attn_close(attn_as_f64(buf.attn_out), ref, None if attn_seqs is None else rows_of(step, attn_seqs))
        ref = oracle.rejection_sample(step)
        got = gpu_sample_result(buf)
        diverged += compare_samples(step, got, ref, max_fraction=None)
        positions += int(step.n_q.sum())
        if observe is not None:
            observe(step, got[0], ref.accept_cnt)
        if not np.array_equal(got[0], ref.accept_cnt):
            buf.accept.copy_(torch.from_numpy(ref.accept_cnt))
        S.rollback(kv, d, buf)
        okv.rollback(step, ref.accept_cnt)
        torch.cuda.synchronize()
        assert status_of(buf) == 0
        assert_kv_equal(kv, okv, pools=False)
        accepted.append(ref.accept_cnt)
    assert diverged <= MAX_TIE_FRACTION * positions, f"{diverged} near-tie divergences in {positions} positions"
    return kv, okv, accepted


def test_contbatch_ten_iterations():
    case = W.contbatch()
    sig = case.meta["sigma_b"]
    steps = lambda it: case.step if it == 0 else W.contbatch_step(case.seed, it, batch=case.state.batch,
                                                                   vocab=case.step.vocab, sigma_b=sig)
    kv, okv, accepted = _loop(case, W.CONTBATCH_ITERS, steps, {0, W.CONTBATCH_ITERS - 1}, None, with_pools=True)
    # acceptance spreads with the per-sequence draft noise
    rate = np.mean(np.stack(accepted), axis=0)
    assert rate[sig < 1.0].mean() > rate[sig > 2.5].mean()


def test_llama8b_three_steps_with_pools():
    """Pools bit-exact after three full steps (only the rows the steps wrote can differ)."""
    case = W.llama8b(batch=6, ctx_range=(100, 900), vocab=4096, growth_tokens=24)
    kv, okv, _ = _loop(case, 3, lambda it: case.step if it == 0 else W.make_chain_step(
        case.seed, case.step.n_q, num_q_heads=32, num_kv_heads=8, head_dim=128, qkv_dtype="bf16", vocab=4096,
        logits_dtype="bf16", target_sigma=3.0, draft_coef=0.8, draft_sigma=1.5, temperature=1.0, stream=it),
        {2}, [0, 5], with_pools=True)
    kp, vp = S.to_bits(kv.k_pool), S.to_bits(kv.v_pool)
    for b in range(case.state.batch):
        for pos in range(okv.seq_lens[b]):
            blk = okv.bt[b][pos // okv.bs]
            np.testing.assert_array_equal(kp[blk, :, pos % okv.bs], okv.k_pool[blk, :, pos % okv.bs])
            np.testing.assert_array_equal(vp[blk, :, pos % okv.bs], okv.v_pool[blk, :, pos % okv.bs])


def test_contbatch_adaptive_k():
    """The draft lengths come from the library's adaptive-K controller (sliding
    window of acceptance rates, page defaults but starting at K = 4), fed with
    the GPU's accept counts; the oracle's controller, fed with the oracle's, must
    choose the same K for every sequence at every iteration."""
    from oracle import adaptive_k as AK
    from speculative_decoding_verify_paged_gb300 import AdaptiveK
    iters = 14
    case = W.contbatch(batch=64, vocab=32000, iterations=iters)
    sig = case.meta["sigma_b"]
    B = case.state.batch
    p = AK.Params(**{**AK.vllm_params().__dict__, "k_init": 4})
    nat = AdaptiveK(B, k_min=p.k_min, k_max=p.k_max, k_init=p.k_init, window=p.window, min_samples=p.min_samples,
                    up_threshold=p.up_threshold, down_threshold=p.down_threshold)
    ora = AK.BatchController(B, p)
    ks = []

    def steps(it):
        k = nat.k
        np.testing.assert_array_equal(k, np.array(ora.k, dtype=np.int32))
        ks.append(k)
        return W.contbatch_step(case.seed, it, batch=B, vocab=32000, sigma_b=sig, K=k)

    def observe(step, gpu_acc, ref_acc):
        drafted = step.n_q - 1
        # a near-tie divergence: the GPU side takes the oracle's counts, as the rollback does
        nat.update(gpu_acc if np.array_equal(gpu_acc, ref_acc) else ref_acc, drafted)
        ora.update(ref_acc, drafted)

    _loop(case, iters, steps, {iters - 1}, [0, 7], with_pools=True, observe=observe)
    ks = np.stack(ks)
    assert (ks[:10] == 4).all()  # nothing moves before ten rates are held
    assert len(set(ks[-1].tolist())) > 1  # then low- and high-noise drafts part ways


@pytest.mark.parametrize("T", [0.0, 1.0])
def test_tree_full_size_step(T):
    """The draft-tree workload at full size (16 sequences of 8192 tokens in
    64-token blocks, 61 rows per sequence): append, tree attention on every row,
    the tree sampler (greedy walk, or the lossless tree rule at T = 1), and the
    rollback that moves the accepted path's rows into place. Block tables,
    lengths, the free list, the emitted tokens, the path and the compacted rows
    must equal the oracle's."""
    case = W.tree(temperature=T)
    st, sp = case.state, case.step
    kv, d, buf = upload(case)
    okv = oracle.OracleKV(st)
    c0 = list(okv.seq_lens)
    msl = int((st.seq_lens + sp.n_q).max())
    S.append(kv, d, buf)
    S.attention(kv, d, buf, msl)
    S.sample(d, buf)
    assert okv.append(sp) is None
    ref_attn = oracle.paged_attention(okv.as_state(), sp)
    ref = oracle.tree_sample(sp) if T > 0 else oracle.tree_greedy(sp)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    assert_attn_close(attn_as_f64(buf.attn_out), ref_attn)
    got = gpu_sample_result(buf)
    compare_samples(sp, got, ref, tree=T == 0.0)
    path = buf.path.cpu().numpy()
    same = got[0] == ref.accept_cnt
    np.testing.assert_array_equal(path[same], ref.path_nodes[same])
    if not same.all():  # a flagged near-tie (T > 0): the rollback takes the oracle's decisions
        buf.accept.copy_(torch.from_numpy(ref.accept_cnt))
        buf.path.copy_(torch.from_numpy(ref.path_nodes))
    assert ref.accept_cnt.max() >= 1
    S.rollback(kv, d, buf)
    okv.rollback(sp, ref.accept_cnt, path_nodes=ref.path_nodes)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    rows = [(okv.bt[b][(c0[b] + j) // okv.bs], (c0[b] + j) % okv.bs)
            for b in range(st.batch) for j in range(int(ref.accept_cnt[b]) + 1)]
    assert_kv_equal(kv, okv, rows=rows)
