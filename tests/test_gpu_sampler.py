"""GPU parity of sv_spec_rejection_sample / sv_tree_greedy_accept /
sv_tree_rejection_sample against the oracle: accept counts and emitted tokens bit-exact, except at oracle-flagged
near-ties (|u - min(1, p/q)| < 1e-4 or a CDF crossing within 1e-4), whose
divergences must stay below 0.01% of the verified positions. Greedy and tree
decisions are exact (argmax, lowest index on ties)."""
import numpy as np
import pytest
import torch
from scipy import stats

import oracle
from speculative_decoding_verify_paged_gb300 import _lib as L
from speculative_decoding_verify_paged_gb300 import step as S
from speculative_decoding_verify_paged_gb300 import workloads as W

from _helpers import compare_samples, gpu_sample_result, status_of, upload

pytestmark = pytest.mark.gpu


def _sample(case):
    kv, d, buf = upload(case)
    S.sample(d, buf)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    return gpu_sample_result(buf)


def _check(case):
    kv, d, buf = upload(case)
    buf.margin.fill_(-1.0)
    S.sample(d, buf)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    got = gpu_sample_result(buf)
    if case.step.mask_kind == "tree" and case.step.temperature > 0:
        ref = oracle.tree_sample(case.step)
        compare_samples(case.step, got, ref)  # near-ties as for chains
        _check_margins(got, ref, buf.margin.cpu().numpy())
    elif case.step.mask_kind == "tree":
        ref = oracle.tree_greedy(case.step)
        compare_samples(case.step, got, ref, tree=True)
    else:
        ref = oracle.rejection_sample(case.step)
        compare_samples(case.step, got, ref)
        _check_margins(got, ref, buf.margin.cpu().numpy())
    return got, ref


def _check_margins(got, ref, margin):
    """The kernel's per-sequence margin (smallest |uniform - threshold| of its
    decisions) against the oracle's fp64 one, where the decisions agree: +inf
    for greedy, else within 1e-5 (fp32 thresholds, fixed-point CDF)."""
    acc, tok, num = got
    same = (acc == ref.accept_cnt) & (num == ref.num_out) & np.all(tok == ref.out_tok, axis=1)
    assert same.sum() > 0
    m, r = margin[same].astype(np.float64), ref.margin[same]
    np.testing.assert_array_equal(np.isinf(m), np.isinf(r))
    fin = ~np.isinf(r)
    assert np.all(m[fin] >= 0.0)
    np.testing.assert_allclose(m[fin], r[fin], rtol=0, atol=1e-5)


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_tiny(T):
    _check(W.tiny(temperature=T))


@pytest.mark.parametrize("name,T", [("llama8b", 1.0), ("llama8b", 0.0), ("llama70b", 1.0), ("llama70b", 0.0)])
def test_full_size(name, T):
    _check(W.CONFIGS[name](temperature=T))


def test_contbatch_first_iteration():
    _check(W.contbatch())


def test_tree_full_size():
    got, ref = _check(W.tree())
    assert ref.accept_cnt.max() >= 2  # the trees do get walked


@pytest.mark.parametrize("T", [1.0, 0.6])
def test_tree_stochastic_full_size(T):
    """16 trees of 60 nodes at V = 32000: paths and tokens equal the oracle's."""
    case = W.tree(temperature=T)
    kv, d, buf = upload(case)
    S.sample(d, buf)
    torch.cuda.synchronize()
    assert status_of(buf) == 0
    got = gpu_sample_result(buf)
    ref = oracle.tree_sample(case.step)
    compare_samples(case.step, got, ref)
    path = buf.path.cpu().numpy()
    for b in range(case.state.batch):
        if got[0][b] == ref.accept_cnt[b]:
            np.testing.assert_array_equal(path[b], ref.path_nodes[b])
    assert ref.accept_cnt.max() >= 1


def test_tree_stochastic_many_small_trees():
    """3000 copies of a 7-node tree over 8 tokens with fresh uniforms: every
    decision and draw equals the oracle's (whose law is pinned by chi-square)."""
    rng = np.random.default_rng(45)
    V, trials = 8, 3000
    parent = [-1, 0, 0, 0, 1, 1, 2]
    n = len(parent)
    tgt = (rng.standard_normal((n, V)) * 1.5).astype(np.float32)
    tok = [-1, 3, 0, 6, 1, 2, 5]
    n_q = np.full(trials, n, np.int32)
    cu = np.zeros(trials + 1, np.int32)
    cu[1:] = np.cumsum(n_q)
    dummy = np.zeros((cu[-1], 1, 1), np.float32)
    step = W.StepInputs(n_q, cu, 1, dummy, dummy, dummy, V, "f32", np.tile(tgt, (trials, 1)),
                        np.zeros((trials * (n - 1), V), np.float32), np.tile(np.array(tok[1:], np.int32), trials),
                        rng.random(trials * (n - 1), dtype=np.float32), rng.random(trials, dtype=np.float32), 0.9,
                        mask_kind="tree", parent=np.tile(np.array(parent, np.int32), trials))
    dev = "cuda"
    t = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)
    acc = torch.empty(trials, dtype=torch.int32, device=dev)
    path = torch.empty((trials, n), dtype=torch.int32, device=dev)
    out = torch.empty((trials, n), dtype=torch.int32, device=dev)
    num = torch.empty(trials, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    L.tree_rejection_sample(t(step.target_logits), t(step.cu_q), t(step.draft_tokens), t(step.parent),
                            t(step.u_accept), t(step.u_resample), 0.9, acc, path, out, num, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.tree_sample(step)
    compare_samples(step, (acc.cpu().numpy(), out.cpu().numpy(), num.cpu().numpy()), ref)
    same = acc.cpu().numpy() == ref.accept_cnt
    np.testing.assert_array_equal(path.cpu().numpy()[same], ref.path_nodes[same])


@pytest.mark.parametrize("V,dtype", [(5, "f32"), (4099, "bf16"), (20000, "f32"), (131072, "bf16"),
                                     (200000, "bf16"), (200000, "f32")])
def test_vocab_sizes(V, dtype):
    """Odd vocabularies (scalar loads), cluster of 8 and of 16, chunks of many items; at
    200000 f32 the decision chunk passes through its sub-chunk ring more than once."""
    case = W.custom(31, batch=6, ctx_lens=[4] * 6, n_q=[1, 2, 3, 5, 7, 9], num_q_heads=1, num_kv_heads=1,
                    head_dim=8, block_size=16, vocab=V, dtype=dtype, target_sigma=2.0, draft_coef=0.8,
                    draft_sigma=1.0, use_bank=V > 50000)
    _check(case)
    case.step.temperature = 0.0
    _check(case)


@pytest.mark.parametrize("V,dtype", [(40001, "f32"), (40003, "bf16")])
def test_large_batch_clusters_of_four(V, dtype):
    """160 sequences take 4-CTA decision clusters; with an odd vocabulary the chunks are
    staged by scalar loads, and at f32 each chunk passes through the ring more than once.
    Decisions, emitted tokens and accept counts equal the oracle's (near-ties aside)."""
    case = W.custom(71, batch=160, ctx_lens=[4] * 160, n_q=[1, 2, 4, 6, 8] * 32, num_q_heads=1, num_kv_heads=1,
                    head_dim=8, block_size=16, vocab=V, dtype=dtype, target_sigma=2.0, draft_coef=0.8,
                    draft_sigma=1.0, use_bank=False)
    _check(case)


@pytest.mark.parametrize("V,dtype", [(1004, "f32"), (1001, "bf16"), (4099, "bf16"), (2052, "f32")])
def test_high_temperature_with_neg_inf_logits(V, dtype):
    """T = 10 with -inf logits scattered over target and draft rows and a
    vocabulary that is not a multiple of 8 (the last group of a chunk is padded
    with -inf): a -inf logit has p = 0 (or q = 0), so no emitted token may carry
    one, every token is < V, and the decisions equal the oracle's."""
    case = W.custom(61, batch=24, ctx_lens=[4] * 24, n_q=[1, 2, 3, 6] * 6, num_q_heads=1, num_kv_heads=1,
                    head_dim=8, block_size=16, vocab=V, dtype=dtype, temperature=10.0, target_sigma=2.0,
                    draft_coef=0.8, draft_sigma=1.0, use_bank=False)
    sp = case.step
    rng = np.random.default_rng(62)
    ninf = np.uint16(0xFF80) if dtype == "bf16" else np.float32(-np.inf)
    tgt, drf = sp.target_logits.copy(), sp.draft_logits.copy()
    for rows in (tgt, drf):
        hit = rng.random(rows.shape) < 0.3  # 30% of each row is -inf
        hit[:, 0] = False  # every row keeps a finite logit
        rows[hit] = ninf
    sp.target_logits, sp.draft_logits = tgt, drf
    # the draft model's tokens, drawn again from the draft rows that now hold -inf
    drf_f = W.bf16_bits_to_f32(drf) if dtype == "bf16" else drf
    sp.draft_tokens = W._draft_sample(np.random.default_rng(63), drf_f, sp.temperature)
    got, ref = _check(case)
    acc, tok, num = got
    tgt_f = W.bf16_bits_to_f32(tgt) if dtype == "bf16" else tgt
    for b in range(case.state.batch):
        y = int(tok[b][acc[b]])
        assert 0 <= y < V
        assert np.isfinite(tgt_f[sp.cu_q[b] + acc[b], y]), f"sequence {b} emitted token {y} with p = 0"


def test_temperature_half():
    case = W.custom(32, batch=16, ctx_lens=[4] * 16, n_q=[6] * 16, num_q_heads=1, num_kv_heads=1, head_dim=8,
                    block_size=16, vocab=32000, temperature=0.5, use_bank=True)
    _check(case)


def test_greedy_ties_take_lowest_index():
    V, B = 4096, 8
    rng = np.random.default_rng(33)
    tgt = np.zeros((B * 3, V), np.float32)
    for r in range(B * 3):
        pos = rng.choice(V, size=5, replace=False)
        tgt[r, pos] = 7.0  # five-way tie at the maximum
    case = W.custom(34, batch=B, ctx_lens=[1] * B, n_q=[3] * B, num_q_heads=1, num_kv_heads=1, head_dim=8,
                    block_size=16, vocab=V, dtype="bf16", temperature=0.0, use_bank=False)
    case.step.target_logits = W.to_bf16_bits(tgt)
    am = np.argmax(tgt, axis=1).reshape(B, 3)
    case.step.draft_tokens = am[:, :2].reshape(-1).astype(np.int32)
    acc, tok, num = _sample(case)
    assert (acc == 2).all()
    np.testing.assert_array_equal(tok[:, 2], am[:, 2])


def _chi2_ok(samples, p, min_p=1e-3):
    obs = np.bincount(samples, minlength=p.shape[0]).astype(np.float64)
    exp = p * samples.shape[0]
    assert obs[exp == 0].sum() == 0
    keep = exp > 0
    return stats.chisquare(obs[keep], exp[keep]).pvalue > min_p


@pytest.mark.parametrize("V", [4, 8, 16])
def test_lossless_chi_square_on_gpu(V):
    """Many sequences that share p and q: the first emitted token follows p,
    the second (when emitted) follows p_2."""
    rng = np.random.default_rng(200 + V)
    K, trials = 3, 400_000
    tgt_rows = (rng.standard_normal((K + 1, V)) * 1.5).astype(np.float32)
    drf_rows = (0.6 * tgt_rows[:K] + rng.standard_normal((K, V))).astype(np.float32)
    n_q = np.full(trials, K + 1, np.int32)
    cu = np.concatenate([[0], np.cumsum(n_q)]).astype(np.int32)

    def softmax(l):
        w = np.exp(l.astype(np.float64) - l.max())
        return w / w.sum()

    qs = [softmax(drf_rows[i]) for i in range(K)]
    x = np.stack([rng.choice(V, size=trials, p=qs[i]) for i in range(K)], 1).reshape(-1).astype(np.int32)
    dev = "cuda"
    tgt = torch.from_numpy(np.tile(tgt_rows, (trials, 1))).to(dev)
    drf = torch.from_numpy(np.tile(drf_rows, (trials, 1))).to(dev)
    ua = torch.from_numpy(rng.random(trials * K, dtype=np.float32)).to(dev)
    ur = torch.from_numpy(rng.random(trials, dtype=np.float32)).to(dev)
    acc = torch.empty(trials, dtype=torch.int32, device=dev)
    tok = torch.empty((trials, K + 1), dtype=torch.int32, device=dev)
    num = torch.empty(trials, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    # the sampler takes at most 65535 sequences per call
    for s in range(0, trials, 50_000):
        e = min(trials, s + 50_000)
        cu_s = torch.from_numpy((cu[s:e + 1] - cu[s]).astype(np.int32)).to(dev)
        L.spec_rejection_sample(tgt[cu[s]:cu[e]], drf[s * K:e * K], cu_s, torch.from_numpy(x[s * K:e * K]).to(dev),
                                ua[s * K:e * K], ur[s:e], 1.0, acc[s:e], tok[s:e], num[s:e], status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    tok = tok.cpu().numpy()
    acc = acc.cpu().numpy()
    assert _chi2_ok(tok[:, 0], softmax(tgt_rows[0]))
    assert _chi2_ok(tok[acc >= 1, 1], softmax(tgt_rows[1]))


def test_nan_logits_are_reported():
    case = W.custom(35, batch=3, ctx_lens=[4] * 3, n_q=[4] * 3, num_q_heads=1, num_kv_heads=1, head_dim=8,
                    block_size=16, vocab=1024, dtype="f32", use_bank=False)
    case.step.target_logits = case.step.target_logits.copy()
    case.step.target_logits[5, 17] = np.nan
    kv, d, buf = upload(case)
    S.sample(d, buf)
    torch.cuda.synchronize()
    assert status_of(buf) == 9


def test_bad_draft_token_is_reported():
    case = W.custom(36, batch=2, ctx_lens=[4] * 2, n_q=[4] * 2, num_q_heads=1, num_kv_heads=1, head_dim=8,
                    block_size=16, vocab=1024, dtype="f32", use_bank=False)
    case.step.draft_tokens = case.step.draft_tokens.copy()
    case.step.draft_tokens[2] = 5000
    kv, d, buf = upload(case)
    S.sample(d, buf)
    torch.cuda.synchronize()
    assert status_of(buf) == 8


def test_host_argument_errors():
    case = W.tiny()
    kv, d, buf = upload(case)
    with pytest.raises(L.SVError) as e:
        L.spec_rejection_sample(d.target_logits, d.draft_logits, d.cu_q, d.draft_tokens, d.u_accept, d.u_resample,
                                -1.0, buf.accept, buf.out_tok, buf.num_out)
    assert e.value.code == 1
    with pytest.raises(L.SVError) as e:
        L.spec_rejection_sample(d.target_logits, None, d.cu_q, d.draft_tokens, d.u_accept, d.u_resample,
                                1.0, buf.accept, buf.out_tok, buf.num_out)
    assert e.value.code == 1
