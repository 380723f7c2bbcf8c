"""Pins of the oracle's tree verification at T > 0 (the reading: a node's
children are point-mass proposals on their tokens, tried in row order; see
so_tree_sample).

* lossless: over many trials, the first emitted token follows the root's p
  and, given that child c was accepted, the second follows p at c --
  chi-square on a tiny vocabulary;
* a chain-shaped tree is the chain rule with one-hot draft distributions:
  the tree oracle and the chain rejection sampler agree on every decision;
* a root without children draws from p by inverse CDF (numpy cumsum);
* a child whose token holds all of p is always accepted, and one whose token
  has probability zero never is.
"""
import numpy as np
import pytest
from scipy import stats

import oracle
from speculative_decoding_verify_paged_gb300 import workloads as W


def _softmax(l, T=1.0):
    z = np.asarray(l, np.float64) / T
    w = np.exp(z - z.max())
    return w / w.sum()


def _tree_step(tgt_rows, parent, tok, trials, rng, T=1.0):
    """`trials` copies of one tree (target rows, parents, node tokens), fresh uniforms."""
    tgt_rows = np.asarray(tgt_rows, np.float32)
    n, V = tgt_rows.shape
    n_q = np.full(trials, n, np.int32)
    cu = np.zeros(trials + 1, np.int32)
    cu[1:] = np.cumsum(n_q)
    dummy = np.zeros((cu[-1], 1, 1), np.float32)
    return W.StepInputs(n_q, cu, 1, dummy, dummy, dummy, V, "f32", np.tile(tgt_rows, (trials, 1)),
                        np.zeros((trials * (n - 1), V), np.float32), np.tile(np.asarray(tok[1:], np.int32), trials),
                        rng.random(trials * (n - 1), dtype=np.float32), rng.random(trials, dtype=np.float32), T,
                        mask_kind="tree", parent=np.tile(np.asarray(parent, np.int32), trials))


def _chi2_ok(samples, p, min_p=1e-3):
    obs = np.bincount(samples, minlength=p.shape[0]).astype(np.float64)
    exp = p * samples.shape[0]
    assert obs[exp == 0].sum() == 0, "a zero-probability token was emitted"
    keep = exp > 0
    return stats.chisquare(obs[keep], exp[keep]).pvalue > min_p


@pytest.mark.parametrize("T", [1.0, 0.7])
def test_lossless_first_and_second_token(T):
    rng = np.random.default_rng(41)
    V = 8
    # root -> children 1, 2, 3; node 1 -> 4, 5; node 2 -> 6. Children carry the
    # top tokens of a draft made from the target plus noise.
    parent = [-1, 0, 0, 0, 1, 1, 2]
    n = len(parent)
    tgt = rng.standard_normal((n, V)) * 1.5
    tok = [-1]
    for j in range(1, n):
        drf = 0.7 * tgt[parent[j]] + rng.standard_normal(V)
        order = [int(v) for v in np.argsort(-drf)]
        sib = [tok[i] for i in range(1, j) if parent[i] == parent[j]]
        tok.append(next(v for v in order if v not in sib))
    first, second = [], {1: [], 2: []}
    for _ in range(4):
        trials = 50000
        step = _tree_step(tgt, parent, tok, trials, rng, T)
        r = oracle.tree_sample(step)
        first.append(r.out_tok[:, 0])
        for c in (1, 2):
            hit = (r.accept_cnt >= 1) & (r.path_nodes[:, 0] == c)
            second[c].append(r.out_tok[hit, 1])
        # the first token is a child's token exactly when that child was accepted
        acc1 = r.accept_cnt >= 1
        assert np.array_equal(r.out_tok[acc1, 0], np.array(tok)[r.path_nodes[acc1, 0]])
        assert not np.isin(r.out_tok[~acc1, 0], [tok[1], tok[2], tok[3]]).any()
    assert _chi2_ok(np.concatenate(first), _softmax(tgt[0], T))
    for c in (1, 2):
        assert _chi2_ok(np.concatenate(second[c]), _softmax(tgt[c], T))


def test_chain_tree_is_the_chain_rule_with_one_hot_drafts():
    rng = np.random.default_rng(42)
    V, K, trials = 16, 4, 3000
    parent = [-1] + list(range(K))
    tgt = rng.standard_normal((K + 1, V)) * 2.0
    for _ in range(3):
        tok = [-1] + [int(x) for x in rng.integers(0, V, size=K)]
        step = _tree_step(tgt, parent, tok, trials, rng)
        r = oracle.tree_sample(step)
        # the same uniforms through the chain rule with q = one-hot at each draft token
        drf = np.full((trials * K, V), -1e4, np.float32)
        drf[np.arange(trials * K), step.draft_tokens] = 0.0
        chain = W.StepInputs(step.n_q, step.cu_q, 1, step.q, step.new_k, step.new_v, V, "f32", step.target_logits,
                             drf, step.draft_tokens, step.u_accept, step.u_resample, 1.0)
        c = oracle.rejection_sample(chain)
        np.testing.assert_array_equal(r.accept_cnt, c.accept_cnt)
        np.testing.assert_array_equal(r.out_tok, c.out_tok)
        np.testing.assert_allclose(r.margin, c.margin, rtol=1e-12, atol=1e-15)
        a = r.accept_cnt
        for t in range(0, trials, 97):
            assert list(r.path_nodes[t, :a[t]]) == list(range(1, a[t] + 1))


def test_root_alone_draws_by_inverse_cdf():
    rng = np.random.default_rng(43)
    V, trials = 32, 500
    tgt = rng.standard_normal((1, V)) * 2.0
    step = _tree_step(tgt, [-1], [-1], trials, rng, T=0.8)
    r = oracle.tree_sample(step)
    cdf = np.cumsum(_softmax(tgt[0], 0.8))
    want = np.searchsorted(cdf, step.u_resample.astype(np.float64), side="right")
    np.testing.assert_array_equal(r.out_tok[:, 0], want)
    assert (r.accept_cnt == 0).all() and (r.num_out == 1).all()


def test_certain_and_impossible_children():
    rng = np.random.default_rng(44)
    V = 8
    tgt = np.full((3, V), -1e4, np.float32)
    tgt[0, 5] = 0.0  # the root's p is all on token 5
    tgt[1] = rng.standard_normal(V)
    tgt[2] = rng.standard_normal(V)
    # child 1 carries token 2 (probability 0), child 2 carries token 5 (probability 1)
    step = _tree_step(tgt, [-1, 0, 0], [-1, 2, 5], 2000, rng)
    r = oracle.tree_sample(step)
    assert (r.accept_cnt >= 1).all()
    assert (r.path_nodes[:, 0] == 2).all() and (r.out_tok[:, 0] == 5).all()


def test_margin_hand_worked():
    """Root p = (0.1, 0.2, 0.3, 0.4); child 1 carries token 3 (p' = 0.4, u = 0.5: rejected, 0.1
    away), child 2 token 2 (p' = 0.3 / 0.6 = 0.5, u = 0.42: accepted, 0.08 away); child 2 is a
    leaf with a uniform row, and u' = 0.3 lands in token 1's interval [0.25, 0.5): 0.05 from its
    edge. The margin is the smallest of the three, 0.05."""
    dummy = np.zeros((3, 1, 1), np.float32)
    tgt = np.log(np.array([[0.1, 0.2, 0.3, 0.4], [0.25] * 4, [0.25] * 4])).astype(np.float32)
    step = W.StepInputs(np.array([3], np.int32), np.array([0, 3], np.int32), 1, dummy, dummy, dummy, 4, "f32", tgt,
                        np.zeros((2, 4), np.float32), np.array([3, 2], np.int32), np.array([0.5, 0.42], np.float32),
                        np.array([0.3], np.float32), 1.0, mask_kind="tree", parent=np.array([-1, 0, 0], np.int32))
    r = oracle.tree_sample(step)
    assert r.accept_cnt[0] == 1 and r.path_nodes[0, 0] == 2 and list(r.out_tok[0, :2]) == [2, 1]
    np.testing.assert_allclose(r.margin[0], 0.05, rtol=1e-6)
