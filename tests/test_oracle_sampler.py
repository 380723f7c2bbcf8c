"""Pins of the oracle's sampler against what the pages and the mathematics fix.

* lossless: the emitted token at the first position follows p exactly, and
  so does the token at position 2 given that it is emitted ("Speculative
  decoding and continuous batching in practice", sec. 1.2; "Speculative
  decoding principles and a vLLM production setup", sec. 2.2) -- chi-square
  on tiny vocabularies;
* the closed form (1 - alpha^(K+1)) / (1 - alpha) tokens per step for i.i.d.
  positions ("LLM serving: speculative decoding and PagedAttention memory
  management", principle section), including the pages' worked example;
* q = p accepts everything; disjoint supports reject at once and draw from p;
* greedy: the accepted prefix is the longest prefix equal to the target
  argmax ("LLM inference optimisation: speculative decoding and dynamic
  batching", engineering section) -- brute force;
* tree greedy: the deepest root-to-node path whose tokens match the argmax of
  their parent's row -- brute force over all paths.
"""
import os

import numpy as np
import pytest
from scipy import stats

import oracle
from speculative_decoding_verify_paged_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _softmax(l, T=1.0):
    z = np.asarray(l, np.float64) / T
    w = np.exp(z - z.max())
    return w / w.sum()


def _make_step(tgt_rows, drf_rows, trials, rng, temperature=1.0, draft_tokens=None):
    """`trials` sequences that all share the same per-position target rows
    (K+1 of them) and draft rows (K); draft tokens x_i ~ q_i drawn per trial."""
    tgt_rows = np.asarray(tgt_rows, np.float32)
    drf_rows = np.asarray(drf_rows, np.float32).reshape(-1, tgt_rows.shape[1])
    K = drf_rows.shape[0]
    V = tgt_rows.shape[1]
    assert tgt_rows.shape[0] == K + 1
    n_q = np.full(trials, K + 1, np.int32)
    cu = np.zeros(trials + 1, np.int32)
    cu[1:] = np.cumsum(n_q)
    tgt = np.tile(tgt_rows, (trials, 1))
    drf = np.tile(drf_rows, (trials, 1))
    if draft_tokens is None:
        cols = []
        for i in range(K):
            qd = _softmax(drf_rows[i], temperature) if temperature > 0 else None
            if temperature > 0:
                cols.append(rng.choice(V, size=trials, p=qd))
            else:
                cols.append(np.full(trials, int(np.argmax(drf_rows[i]))))
        draft_tokens = (np.stack(cols, 1).reshape(-1) if K else np.zeros(0)).astype(np.int32)
    dummy = np.zeros((cu[-1], 1, 1), np.float32)
    return W.StepInputs(n_q, cu, 1, dummy, dummy, dummy, V, "f32", tgt, drf, draft_tokens,
                        rng.random(trials * K, dtype=np.float32), rng.random(trials, dtype=np.float32),
                        float(temperature))


def _chi2_ok(samples, p, min_p=1e-3):
    V = p.shape[0]
    obs = np.bincount(samples, minlength=V).astype(np.float64)
    exp = p * samples.shape[0]
    assert obs[exp == 0].sum() == 0, "a zero-probability token was emitted"
    keep = exp > 0
    return stats.chisquare(obs[keep], exp[keep]).pvalue > min_p


@pytest.mark.parametrize("V", [4, 8, 16])
def test_lossless_first_and_second_position(V):
    rng = np.random.default_rng(100 + V)
    K = 3
    tgt = rng.standard_normal((K + 1, V)) * 1.5
    drf = 0.6 * tgt[:K] + rng.standard_normal((K, V))
    first, second = [], []
    for _ in range(5):
        step = _make_step(tgt, drf, 200_000, rng)
        r = oracle.rejection_sample(step)
        first.append(r.out_tok[:, 0])
        second.append(r.out_tok[r.accept_cnt >= 1, 1])
    p1 = _softmax(np.float32(tgt[0]))
    p2 = _softmax(np.float32(tgt[1]))
    assert _chi2_ok(np.concatenate(first), p1)
    assert _chi2_ok(np.concatenate(second), p2)


def test_lossless_at_temperature():
    rng = np.random.default_rng(7)
    V, K, T = 8, 2, 0.6
    tgt = rng.standard_normal((K + 1, V))
    drf = rng.standard_normal((K, V))
    step = _make_step(tgt, drf, 400_000, rng, temperature=T)
    r = oracle.rejection_sample(step)
    assert _chi2_ok(r.out_tok[:, 0], _softmax(np.float32(tgt[0]), T))
    # and not the distribution at T = 1
    assert not _chi2_ok(r.out_tok[:, 0], _softmax(np.float32(tgt[0]), 1.0))


def test_bonus_only_when_no_drafts():
    rng = np.random.default_rng(8)
    V = 8
    tgt = rng.standard_normal((1, V))
    step = _make_step(tgt, np.zeros((0, V)), 300_000, rng)
    r = oracle.rejection_sample(step)
    assert (r.accept_cnt == 0).all() and (r.num_out == 1).all()
    assert _chi2_ok(r.out_tok[:, 0], _softmax(np.float32(tgt[0])))


def _closed_form(alpha, K):
    return (1 - alpha ** (K + 1)) / (1 - alpha)


def test_golden_closed_form_value():
    vals = {}
    with open(os.path.join(GOLDEN, "closed_form_alpha0.8_k5.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                k, v = line.split()
                vals[k] = float(v)
    assert abs(_closed_form(vals["alpha"], int(vals["K"])) - vals["tokens_per_step"]) < 1e-5


@pytest.mark.parametrize("p,q,K", [((0.9, 0.1), (0.7, 0.3), 5),
                                   ((0.5, 0.3, 0.2), (0.2, 0.3, 0.5), 4),
                                   ((0.25, 0.25, 0.25, 0.25), (0.7, 0.1, 0.1, 0.1), 7)])
def test_closed_form_mean_tokens_per_step(p, q, K):
    rng = np.random.default_rng(9)
    p, q = np.array(p), np.array(q)
    alpha = np.minimum(p, q).sum()
    tgt = np.tile(np.log(p), (K + 1, 1))
    drf = np.tile(np.log(q), (K, 1))
    N = 400_000
    step = _make_step(tgt, drf, N, rng)
    r = oracle.rejection_sample(step)
    got = r.num_out.astype(np.float64)
    want = _closed_form(alpha, K)
    assert abs(got.mean() - want) < 4 * got.std() / np.sqrt(N) + 1e-6
    # the acceptance count is geometric, truncated at K
    a = r.accept_cnt
    for k in range(K):
        frac = (a == k).mean()
        assert abs(frac - alpha ** k * (1 - alpha)) < 5 * np.sqrt(alpha ** k / N) + 1e-4


def test_q_equals_p_accepts_all():
    rng = np.random.default_rng(10)
    V, K = 32, 6
    tgt = rng.standard_normal((K + 1, V)) * 2
    step = _make_step(tgt, tgt[:K], 20_000, rng)
    r = oracle.rejection_sample(step)
    assert (r.accept_cnt == K).all()
    assert _chi2_ok(r.out_tok[:, K], _softmax(np.float32(tgt[K])))


def test_disjoint_supports_reject_first_and_draw_p():
    rng = np.random.default_rng(11)
    V, K = 12, 3
    tgt = rng.standard_normal((K + 1, V))
    drf = rng.standard_normal((K, V))
    tgt[:, V // 2:] = -np.inf
    drf[:, :V // 2] = -np.inf
    step = _make_step(tgt, drf, 200_000, rng)
    r = oracle.rejection_sample(step)
    assert (r.accept_cnt == 0).all()
    assert _chi2_ok(r.out_tok[:, 0], _softmax(np.float32(tgt[0])))


def test_greedy_longest_matching_prefix_bruteforce():
    rng = np.random.default_rng(12)
    V, K, trials = 5, 4, 3000
    # small integer logits so that ties at the maximum are common
    tgt = rng.integers(-2, 3, size=(trials * (K + 1), V)).astype(np.float32)
    am = np.argmax(tgt, axis=1).reshape(trials, K + 1)  # lowest index on ties
    x = np.where(rng.random((trials, K)) < 0.7, am[:, :K], rng.integers(0, V, (trials, K)))
    n_q = np.full(trials, K + 1, np.int32)
    cu = np.concatenate([[0], np.cumsum(n_q)]).astype(np.int32)
    dummy = np.zeros((cu[-1], 1, 1), np.float32)
    step = W.StepInputs(n_q, cu, 1, dummy, dummy, dummy, V, "f32", tgt, np.zeros((trials * K, V), np.float32),
                        x.reshape(-1).astype(np.int32), np.zeros(trials * K, np.float32),
                        np.zeros(trials, np.float32), 0.0)
    r = oracle.rejection_sample(step)
    for t in range(trials):
        a = 0
        while a < K and x[t, a] == am[t, a]:
            a += 1
        assert r.accept_cnt[t] == a
        assert list(r.out_tok[t, :a]) == list(x[t, :a])
        assert r.out_tok[t, a] == am[t, a]


def _random_tree(rng, n):
    parent = [-1]
    for j in range(1, n):
        parent.append(int(rng.integers(0, j)))
    return parent


def test_tree_greedy_bruteforce():
    rng = np.random.default_rng(13)
    V = 6
    for trial in range(300):
        n = int(rng.integers(1, 11))
        parent = _random_tree(rng, n)
        tgt = rng.integers(-3, 3, size=(n, V)).astype(np.float32)
        am = np.argmax(tgt, axis=1)
        tok = [-1]
        for j in range(1, n):
            sib = [tok[i] for i in range(1, j) if parent[i] == parent[j]]
            choices = [v for v in range(V) if v not in sib]
            if rng.random() < 0.6 and am[parent[j]] in choices:
                tok.append(int(am[parent[j]]))
            else:
                tok.append(int(rng.choice(choices)))
        # brute force: every node whose root path matches the argmax at each parent
        best = [0]
        for j in range(1, n):
            path, a, ok = [], j, True
            while a != 0:
                ok &= tok[a] == am[parent[a]]
                path.append(a)
                a = parent[a]
            if ok and len(path) > len(best) - 1:
                best = [0] + path[::-1]
        n_q = np.array([n], np.int32)
        cu = np.array([0, n], np.int32)
        dummy = np.zeros((n, 1, 1), np.float32)
        step = W.StepInputs(n_q, cu, 1, dummy, dummy, dummy, V, "f32", tgt, np.zeros((n - 1, V), np.float32),
                            np.array(tok[1:], np.int32), np.zeros(n - 1, np.float32), np.zeros(1, np.float32),
                            0.0, mask_kind="tree", parent=np.array(parent, np.int32))
        r = oracle.tree_greedy(step)
        a = len(best) - 1
        assert r.accept_cnt[0] == a
        assert list(r.path_nodes[0, :a]) == best[1:]
        assert r.out_tok[0, a] == am[best[-1]]
        assert list(r.out_tok[0, :a]) == [tok[j] for j in best[1:]]


def test_margins_flag_near_ties():
    """The reported margin is |u - min(1, p/q)| at the deciding comparison."""
    V = 2
    p = np.array([0.6, 0.4])
    q = np.array([0.8, 0.2])
    tgt = np.log(np.array([p, p]))
    drf = np.log(np.array([q]))
    n_q = np.array([2], np.int32)
    cu = np.array([0, 2], np.int32)
    dummy = np.zeros((2, 1, 1), np.float32)
    ratio = 0.6 / 0.8
    u = np.float32(ratio + 3e-5)
    step = W.StepInputs(n_q, cu, 1, dummy, dummy, dummy, V, "f32", tgt.astype(np.float32),
                        drf.astype(np.float32), np.array([0], np.int32), np.array([u], np.float32),
                        np.array([0.5], np.float32), 1.0)
    r = oracle.rejection_sample(step)
    assert r.accept_cnt[0] == 0  # u just above the ratio: rejected
    assert r.margin[0] < 1e-4
    # residual max(0, p - q) = (0, 0.2): the only token with mass is 1
    assert r.out_tok[0, 0] == 1


def test_nonfinite_logits_are_an_error():
    rng = np.random.default_rng(3)
    tgt = rng.standard_normal((3, 8)).astype(np.float32)
    tgt[1, 3] = np.nan
    step = _make_step(tgt, rng.standard_normal((2, 8)), 4, rng, draft_tokens=np.zeros(8, np.int32))
    step.u_accept[:] = 0.0  # accept position 0 so that row 1 is read
    with pytest.raises(oracle.OracleError):
        oracle.rejection_sample(step)


def test_margin_hand_worked():
    """The margin, worked by hand on four-token rows: the smallest of |u - min(1, p/q)| over the
    drafts tested and the draw's distance to its interval edges on the normalised CDF."""
    V = 4
    p0 = np.array([0.1, 0.2, 0.3, 0.4])
    q0 = np.array([0.4, 0.3, 0.2, 0.1])
    p1 = np.array([0.25, 0.25, 0.25, 0.25])
    dummy = np.zeros((2, 1, 1), np.float32)

    def run(u, ur):
        step = W.StepInputs(np.array([2], np.int32), np.array([0, 2], np.int32), 1, dummy, dummy, dummy, V, "f32",
                            np.log(np.array([p0, p1])).astype(np.float32), np.log(np.array([q0])).astype(np.float32),
                            np.array([0], np.int32), np.array([u], np.float32), np.array([ur], np.float32), 1.0)
        return oracle.rejection_sample(step)

    # rejected (u = 0.7 against 0.1 / 0.4 = 0.25): residual (0, 0, 0.1, 0.3), u' S = 0.2 falls in
    # token 3's interval [0.1, 0.4): edges 0.25 and 0.5 of the mass 0.4 away; margin min(0.45, 0.25)
    r = run(0.7, 0.5)
    assert r.accept_cnt[0] == 0 and r.out_tok[0, 0] == 3
    np.testing.assert_allclose(r.margin[0], 0.25, rtol=1e-6)
    # accepted (u = 0.1 < 0.25, distance 0.15); the bonus draw from p1 at 0.6 lands in token 2's
    # interval [0.5, 0.75): edges 0.1 and 0.15 away; margin 0.1
    r = run(0.1, 0.6)
    assert r.accept_cnt[0] == 1 and list(r.out_tok[0, :2]) == [0, 2]
    np.testing.assert_allclose(r.margin[0], 0.1, rtol=1e-6)
