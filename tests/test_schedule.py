"""Prefix scheduler (DSpark summary, "Confidence-Scheduled Verification"): CPU only.

The library's greedy global sort must reach the throughput of an exhaustive
search over every vector of verify lengths on small cases, with any cost
table (the sort is exact for every M: the M - B largest survival
probabilities form prefixes). Early stopping reaches it when the throughput
is unimodal in M, and never exceeds it.
"""
import itertools

import numpy as np
import pytest

import verify_step_02_b300 as vs


def brute_force(conf, step_us):
    """max over L in [0, gamma]^B of tau(L) / T(M(L)), the textbook definition."""
    b, g = conf.shape
    surv = np.cumprod(conf.astype(np.float64), axis=1)
    best, best_l = -1.0, None
    for lens in itertools.product(range(g + 1), repeat=b):
        m = b + sum(lens)
        if m > len(step_us):
            continue
        tau = b + sum(surv[r, :lens[r]].sum() for r in range(b))
        th = tau / float(step_us[m - 1])
        if th > best:
            best, best_l = th, lens
    return best, best_l


def theta_of(conf, step_us, lens):
    surv = np.cumprod(conf.astype(np.float64), axis=1)
    tau = conf.shape[0] + sum(surv[r, :l].sum() for r, l in enumerate(lens))
    return tau / float(step_us[conf.shape[0] + int(sum(lens)) - 1])


@pytest.mark.parametrize("case", range(40))
def test_global_search_matches_exhaustive(case):
    rng = np.random.default_rng(case)
    b, g = int(rng.integers(1, 5)), int(rng.integers(1, 5))
    conf = rng.beta(8, 2, size=(b, g)).astype(np.float32)
    if case % 3 == 0:
        conf[:, rng.integers(0, g)] = rng.random(b)  # some low-confidence positions
    n_cost = b * (g + 1) - int(rng.integers(0, b * g // 2 + 1))
    # costs: a base plus a per-row slope, with steps (the measured tables fall in steps)
    m = np.arange(1, n_cost + 1)
    cost = (100.0 + rng.uniform(0, 20) * m + 30.0 * (m > rng.integers(1, n_cost + 1))).astype(np.float32)
    lens, tau, th = vs.schedule_prefix(conf, cost, early_stop=False)
    want, _ = brute_force(conf, cost)
    assert lens.min() >= 0 and lens.max() <= g and b + lens.sum() <= n_cost
    assert th / 1e6 == pytest.approx(want, rel=1e-9)
    assert theta_of(conf, cost, lens) == pytest.approx(want, rel=1e-9)
    surv = np.cumprod(conf.astype(np.float64), axis=1)
    assert tau == pytest.approx(b + sum(surv[r, :l].sum() for r, l in enumerate(lens)), rel=1e-9)


def test_early_stop_on_unimodal_and_stepped_costs():
    rng = np.random.default_rng(7)
    for _ in range(30):
        b, g = 3, 4
        conf = rng.beta(8, 2, size=(b, g)).astype(np.float32)
        m = np.arange(1, b * (g + 1) + 1)
        smooth = (50.0 + 9.0 * m).astype(np.float32)  # affine cost: tau / T(M) rises then falls
        l1, _, t1 = vs.schedule_prefix(conf, smooth, early_stop=True)
        l2, _, t2 = vs.schedule_prefix(conf, smooth, early_stop=False)
        assert t1 == pytest.approx(t2, rel=1e-9)
        stepped = (50.0 + 100.0 * (m > b + 1) + 0.1 * m).astype(np.float32)  # a cliff after one draft
        l3, _, t3 = vs.schedule_prefix(conf, stepped, early_stop=True)
        l4, _, t4 = vs.schedule_prefix(conf, stepped, early_stop=False)
        assert t3 <= t4 * (1 + 1e-12)
        assert t4 / 1e6 == pytest.approx(brute_force(conf, stepped)[0], rel=1e-9)


def test_special_cases():
    # certain drafts and a flat cost: verify everything
    lens, tau, _ = vs.schedule_prefix(np.ones((2, 5), np.float32), np.full(12, 7.0, np.float32))
    assert list(lens) == [5, 5] and tau == pytest.approx(12.0)
    # hopeless drafts: anchors only
    lens, tau, _ = vs.schedule_prefix(np.zeros((3, 4), np.float32), np.arange(1, 16, dtype=np.float32) * 10)
    assert list(lens) == [0, 0, 0] and tau == pytest.approx(3.0)
    # a confidence outside [0, 1] and a table that cannot hold the anchors are refused
    with pytest.raises(vs.SvError):
        vs.schedule_prefix(np.full((1, 2), 1.5, np.float32), np.ones(3, np.float32))
    with pytest.raises(vs.SvError):
        vs.schedule_prefix(np.full((4, 2), 0.5, np.float32), np.ones(3, np.float32))
