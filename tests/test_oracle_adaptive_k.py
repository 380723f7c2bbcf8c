"""The adaptive draft-length oracle pinned to step counts derived by hand from
the rule ("Speculative decoding principles and a vLLM production setup",
sec. 4.3; "LLM inference optimisation: speculative decoding and dynamic
batching", engineering parameters), then the library's host controller
compared with it on random traces (host code only: no GPU)."""
import ctypes

import numpy as np
import pytest

from oracle import adaptive_k as AK
from speculative_decoding_verify_paged_gb300 import _lib as L


def _run(p, rates, k_init=None):
    """Feed (accepted, drafted) pairs; return K after each update."""
    if k_init is not None:
        p = AK.Params(**{**p.__dict__, "k_init": k_init})
    c = AK.SequenceController(p)
    return [c.observe(a, d) for a, d in rates]


def test_all_accepted_climbs_one_per_step_after_ten_samples():
    # page defaults: K starts at k_min = 2, nothing moves before 10 rates, mean 1 > 0.7
    ks = _run(AK.vllm_params(), [(5, 5)] * 20)
    assert ks == [min(8, 2 + max(0, n - 9)) for n in range(1, 21)]


def test_all_rejected_sinks_to_k_min():
    ks = _run(AK.vllm_params(), [(0, 6)] * 15, k_init=5)
    assert ks == [max(2, 5 - max(0, n - 9)) for n in range(1, 16)]


def test_mean_at_target_holds():
    # alpha = 3/5 = 0.6 sits between 0.5 and 0.7
    assert set(_run(AK.vllm_params(), [(3, 5)] * 30, k_init=4)) == {4}


def test_window_of_fifty():
    # 50 full acceptances (K at 8), then z rejections: the mean is (50 - z) / 50.
    # It drops below 0.6 - 0.1 (a double just under 0.5) first at z = 26
    # (z = 25 gives exactly 0.5: no move), and K then falls one per step to 2.
    ks = _run(AK.vllm_params(), [(4, 4)] * 50 + [(0, 4)] * 35)
    assert ks[49] == 8
    tail = ks[50:]
    assert tail == [8 if z <= 25 else max(2, 8 - (z - 25)) for z in range(1, 36)]


def test_mean_is_over_the_rates_held_not_the_window():
    # 10 rates, six of 1 and four of 0: the mean of what is held is 0.6 (no move);
    # dividing by the window (50) would give 0.12 and a step down.
    ks = _run(AK.vllm_params(), [(2, 2)] * 6 + [(0, 2)] * 4, k_init=5)
    assert ks[-1] == 5


def test_oldest_rate_leaves_first():
    # window 3, min 3: rates 1, 1, 0 (mean 2/3, no move at target 0.6 +- 0.1),
    # then 0 replaces the oldest 1: mean 1/3 < 0.5, one step down
    p = AK.Params(k_min=1, k_max=8, k_init=4, window=3, min_samples=3, up_threshold=0.7, down_threshold=0.5)
    assert _run(p, [(1, 1), (1, 1), (0, 1), (0, 1)]) == [4, 4, 4, 3]


def test_no_drafts_counts_as_rate_zero():
    # alpha = 0 / max(0, 1) = 0
    assert _run(AK.vllm_params(), [(0, 0)] * 10, k_init=6)[-1] == 5


def test_min_samples_above_window_never_moves():
    p = AK.Params(k_init=4, window=5, min_samples=10)
    assert set(_run(p, [(5, 5)] * 40)) == {4}


def test_engineering_rule():
    # start 4, last 10 rounds: above 80% -> +1, below 50% -> -1
    p = AK.engineering_params()
    ks = _run(p, [(7, 8)] * 14)  # 0.875 > 0.8
    assert ks == [4] * 9 + [5, 6, 7, 8, 8]
    ks = _run(p, [(3, 8)] * 12)  # 0.375 < 0.5
    assert ks == [4] * 9 + [3, 2, 2]


def test_invalid_counts_rejected():
    c = AK.BatchController(2, AK.vllm_params())
    with pytest.raises(ValueError):
        c.update([3, 1], [2, 4])


# ---------------------------------------------------------------------------
# the library's host controller against the oracle (no GPU is touched)
# ---------------------------------------------------------------------------
def _native(batch, p):
    return L.AdaptiveK(batch, k_min=p.k_min, k_max=p.k_max, k_init=p.k_init, window=p.window,
                       min_samples=p.min_samples, up_threshold=p.up_threshold, down_threshold=p.down_threshold)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_native_controller_matches_oracle(seed):
    rng = np.random.default_rng(seed)
    batch = 64
    p = [AK.vllm_params(), AK.engineering_params(),
         AK.Params(k_min=1, k_max=12, k_init=3, window=7, min_samples=4, up_threshold=0.55, down_threshold=0.45)][seed]
    nat, ora = _native(batch, p), AK.BatchController(batch, p)
    acc_p = rng.uniform(0.2, 0.95, size=batch)  # per-sequence acceptance probability
    k = np.array(ora.k, dtype=np.int32)
    for step in range(150):
        drafted = k.copy()
        accepted = np.zeros(batch, dtype=np.int32)
        for b in range(batch):  # drafts pass in order until the first rejection
            while accepted[b] < drafted[b] and rng.random() < acc_p[b]:
                accepted[b] += 1
        if step == 60:  # a new request takes slot 5
            nat.reset(5)
            ora.reset(5)
        got = nat.update(accepted, drafted)
        want = ora.update(accepted, drafted)
        np.testing.assert_array_equal(got, np.array(want, dtype=np.int32))
        np.testing.assert_array_equal(nat.k, got)
        k = got
    assert len(set(k.tolist())) > 1  # acceptance spreads the K's


def test_native_controller_all_or_nothing():
    p = AK.vllm_params()
    nat = _native(3, p)
    for _ in range(12):
        nat.update([4, 4, 4], [4, 4, 4])
    before = nat.k.copy()
    with pytest.raises(L.SVError):
        nat.update([4, 5, 0], [4, 4, 4])  # accepted > drafted in one sequence
    np.testing.assert_array_equal(nat.k, before)
    with pytest.raises(L.SVError):
        nat.reset(3)


def test_native_state_and_params_validation():
    lib = L.load()
    assert lib.sv_adaptive_k_state_bytes(4, 50) > 4 * 50 * 8
    assert lib.sv_adaptive_k_state_bytes(4, 0) == 0
    assert lib.sv_adaptive_k_state_bytes(-1, 5) == 0
    buf = (ctypes.c_double * 4096)()
    bad = [dict(k_min=3, k_init=2), dict(k_max=64, k_init=2), dict(window=0), dict(min_samples=0),
           dict(up_threshold=float("nan"))]
    for kw in bad:
        base = dict(k_min=2, k_max=8, k_init=2, window=5, min_samples=3, up_threshold=0.7, down_threshold=0.5)
        base.update(kw)
        prm = L.sv_adaptive_k_params(base["k_min"], base["k_max"], base["k_init"], base["window"],
                                     base["min_samples"], base["up_threshold"], base["down_threshold"])
        assert lib.sv_adaptive_k_init(buf, ctypes.sizeof(buf), 4, ctypes.byref(prm)) == 1, kw
    prm = L.sv_adaptive_k_params(2, 8, 2, 5, 3, 0.7, 0.5)
    assert lib.sv_adaptive_k_init(buf, 16, 4, ctypes.byref(prm)) == 1  # too small
    # an uninitialised block is refused
    blank = (ctypes.c_double * 64)()
    assert lib.sv_adaptive_k_update(blank, None, None, None) == 1


def test_thresholds_are_strict():
    # a mean exactly at both thresholds moves nothing (strict comparisons)
    p = AK.Params(k_min=1, k_max=8, k_init=4, window=4, min_samples=2, up_threshold=0.5, down_threshold=0.5)
    assert set(_run(p, [(1, 2)] * 8)) == {4}
    nat = _native(1, p)
    assert {int(nat.update([1], [2])[0]) for _ in range(8)} == {4}
