"""Pins of the DSpark prefix-scheduler oracle against values fixed by the
pages' description and by mathematics, not by the oracle itself: a hand
worked case, closed forms for flat and 1/B throughput curves, brute force
over every length vector on tiny pools, the strict-rise stop, clamping and
the SPS-table bound."""

import itertools
import json
import os

import numpy as np
import pytest

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden", "schedule_hand_case.json")


def test_hand_worked_case():
    case = json.load(open(GOLD))
    res = oracle.schedule_prefix(np.array(case["conf"]), np.array(case["sps"]))
    assert res["lens"].tolist() == case["lens"]
    assert res["added"] == case["added"]
    assert res["theta"] == pytest.approx(case["theta"], rel=1e-12)


def test_flat_throughput_adds_every_positive_candidate():
    # Theta = tau * const rises with every S > 0: every position with a
    # positive prefix survival is verified, nothing after a zero
    rng = np.random.default_rng(0)
    conf = rng.uniform(0.05, 1.0, (7, 5))
    conf[2, 3] = 0.0  # request 2 survives only three positions
    res = oracle.schedule_prefix(conf, np.full(100, 3.0))
    want = np.full(7, 6)
    want[2] = 4
    assert res["lens"].tolist() == want.tolist()


def test_inverse_batch_curve_matches_brute_force():
    # SPS(b) = 1/b: Theta = tau / B, the mean expected tokens per verified
    # row; adding candidates best-first raises it while the next S beats the
    # running mean, so the greedy stop is the optimum over all length vectors
    rng = np.random.default_rng(1)
    for trial in range(40):
        B, K = rng.integers(1, 4), rng.integers(1, 4)
        conf = rng.uniform(0.0, 1.0, (B, K))
        sps = np.array([0.0] + [1.0 / b for b in range(1, B * (K + 1) + 2)])
        res = oracle.schedule_prefix(conf, sps)
        S = np.cumprod(conf, axis=1)
        best = max(
            (B + sum(S[r, :lr - 1].sum() for r, lr in enumerate(ls))) / sum(ls)
            for ls in itertools.product(range(1, K + 2), repeat=B))
        assert res["theta"] == pytest.approx(best, rel=1e-12)


def test_stop_requires_a_strict_rise():
    # one request, c = 1: tau 1 -> 2 and B 1 -> 2 leave tau / B at 1: no rise
    res = oracle.schedule_prefix(np.array([[1.0, 1.0]]), np.array([0.0, 1.0, 0.5, 1 / 3]))
    assert res["lens"].tolist() == [1] and res["added"] == 0
    # the same with a slightly better curve at B = 2 adds
    res = oracle.schedule_prefix(np.array([[1.0, 1.0]]), np.array([0.0, 1.0, 0.5001, 0.1]))
    assert res["lens"].tolist() == [2]


def test_result_invariants_and_early_stop():
    rng = np.random.default_rng(2)
    for trial in range(30):
        B, K = rng.integers(1, 9), rng.integers(0, 8)
        conf = rng.uniform(0.0, 1.0, (B, K))
        b = np.arange(B * (K + 1) + 2, dtype=np.float64)
        sps = 1000.0 / (1.0 + 0.05 * b + 0.002 * b * b)  # a decreasing, convex-ish curve
        res = oracle.schedule_prefix(conf, sps)
        lens = res["lens"]
        assert (lens >= 1).all() and (lens <= K + 1).all()
        assert res["added"] == lens.sum() - B
        tau = oracle.expected_tokens(conf, lens)
        assert res["theta"] == pytest.approx(tau * sps[lens.sum()], rel=1e-12)
        # the best remaining candidate (one more position of some request)
        # would not raise Theta
        S = np.cumprod(conf, axis=1)
        nxt = [S[r, lens[r] - 1] for r in range(B) if lens[r] <= K]
        if nxt and lens.sum() + 1 < len(sps):
            assert (tau + max(nxt)) * sps[lens.sum() + 1] <= res["theta"] * (1 + 1e-12)


def test_clamping_and_nan():
    # c > 1 counts as 1, NaN and negatives as 0: request 0 then survives
    # one position at S = 1, request 1 none
    conf = np.array([[1.7, np.nan], [-0.2, 0.9]])
    res = oracle.schedule_prefix(conf, np.full(10, 2.0))
    assert res["lens"].tolist() == [2, 1]


def test_sps_table_bounds_the_batch():
    conf = np.ones((3, 4)) * 0.9
    res = oracle.schedule_prefix(conf, np.full(6, 1.0))  # B may grow to 5 at most
    assert res["lens"].sum() == 5
    with pytest.raises(ValueError):
        oracle.schedule_prefix(conf, np.full(3, 1.0))  # no entry for B = 3


@pytest.mark.parametrize("sign,lens,added", [(+1, [2], 1), (-1, [1], 0)])
def test_near_tied_theta_margin(sign, lens, added):
    """Hand case: one request, c = 1/2, SPS = [0, 3/2, 1 + s 2^-36].  Start:
    tau = 1, Theta = 3/2.  The candidate S = 1/2 gives tau = 3/2 and
    Theta_next = 3/2 (1 + s 2^-36), exact in float64: it is added only when
    s = +1, and the recorded margin is the relative gap 2^-36 (about 1.5e-11)
    either way."""
    sps = np.array([0.0, 1.5, 1.0 + sign * 2.0 ** -36])
    res = oracle.schedule_prefix(np.array([[0.5]]), sps)
    assert res["lens"].tolist() == lens and res["added"] == added
    assert res["margin"] == 2.0 ** -36
    assert res["theta"] == (1.5 * (1.0 + 2.0 ** -36) if sign > 0 else 1.5)
