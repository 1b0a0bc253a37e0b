"""Pins for the oracle's acceptance rules and the speculative loop (CPU only)."""
import itertools
import os

import numpy as np
import pytest
from scipy import stats

import synth
from oracle import accept, spec
from oracle.decoder import Config, DenseWeights


# ---------------------------------------------------------------- greedy
def test_greedy_brute_force_all_draft_sequences():
    """V = 4, gamma = 3: all 64 draft blocks against a table of target argmaxes."""
    rng = np.random.default_rng(0)
    for _ in range(5):
        target = rng.integers(0, 4, size=4)               # argmax at rows 0..3
        logits = np.full((4, 4), -1.0)
        logits[np.arange(4), target] = 2.0
        for drafts in itertools.product(range(4), repeat=3):
            k, nxt = accept.greedy_accept(logits, drafts)
            # independent rule: the common prefix of the draft string and the target string
            a = "".join(map(str, drafts))
            b = "".join(map(str, target[:3]))
            want_k = len(os.path.commonprefix([a, b]))
            assert k == want_k
            assert nxt == target[want_k]


def test_greedy_ties_take_lowest_index():
    z = np.array([[0.0, 3.0, 3.0, 1.0]])
    assert accept.greedy_accept(z, []) == (0, 1)


# ---------------------------------------------------------------- sampling helpers
def test_inverse_cdf_boundaries():
    w = np.array([0.0, 0.25, 0.0, 0.75])
    assert accept.inverse_cdf(w, 0.0) == 1
    assert accept.inverse_cdf(w, 0.2499999) == 1
    assert accept.inverse_cdf(w, 0.25) == 3
    assert accept.inverse_cdf(w, 0.9999999) == 3


def test_uniform_positions_and_streams():
    u_acc, u_res = accept.uniforms(11, 3, 100, 4)
    from oracle import philox
    assert np.array_equal(u_acc, philox.uniform(11, 3, np.arange(101, 105), 0))
    assert np.array_equal(u_res, philox.uniform(11, 3, np.arange(101, 106), 1))


def _dists(v, rng, zeros_p=False, zeros_q=False):
    p = rng.random(v) ** 2
    q = rng.random(v) ** 2
    if zeros_p:
        p[: v // 4] = 0.0
    if zeros_q:
        q[v // 2: v // 2 + v // 4] = 0.0
    return p / p.sum(), q / q.sum()


def _logits_for(p, T):
    with np.errstate(divide="ignore"):
        return np.where(p > 0, np.log(np.where(p > 0, p, 1.0)) * T, -np.inf)


def test_q_equal_p_always_accepts():
    rng = np.random.default_rng(1)
    p, _ = _dists(8, rng)
    z = np.tile(_logits_for(p, 1.0), (4, 1))
    qq = np.tile(p, (3, 1))
    for s in range(200):
        drafts = rng.choice(8, size=3, p=p)
        u_acc, u_res = accept.uniforms(s, 0, 50, 3)
        k, _ = accept.sampled_accept(z, drafts, qq, 1.0, u_acc, u_res)
        assert k == 3


N_STAT = 100_000


@pytest.mark.parametrize("zeros_p,zeros_q", [(False, False), (True, False), (False, True), (True, True)])
def test_acceptance_rate_is_one_minus_tv_and_output_is_target(zeros_p, zeros_q):
    """One draft per step; closed form P(accept) = sum_v min(p, q) = 1 - TV(p, q)
    (DSpark summary, confidence head: c* = 1 - 0.5 ||p_d - p_t||_1), and the emitted
    token is distributed as p (chi-square)."""
    v, T = 8, 0.7
    rng = np.random.default_rng(2 + 2 * zeros_p + zeros_q)
    p, q = _dists(v, rng, zeros_p, zeros_q)
    z = np.tile(_logits_for(p, T), (2, 1))
    drafts = rng.choice(v, size=N_STAT, p=q)
    pos = np.arange(N_STAT) * 4
    from oracle import philox
    u0 = philox.uniform(99, 1, pos + 1, 0)
    u1 = philox.uniform(99, 1, pos + 1, 1)
    u2 = philox.uniform(99, 1, pos + 2, 1)
    acc = 0
    first = np.zeros(v, np.int64)
    for n in range(N_STAT):
        k, nxt = accept.sampled_accept(z, [drafts[n]], q[None, :], T, [u0[n]], [u1[n], u2[n]])
        acc += k
        first[drafts[n] if k == 1 else nxt] += 1
    want = np.minimum(p, q).sum()
    assert abs(want - (1 - 0.5 * np.abs(p - q).sum())) < 1e-12
    assert stats.binomtest(acc, N_STAT, want).pvalue > 1e-3
    mask = p > 0
    assert first[~mask].sum() == 0
    chi = stats.chisquare(first[mask], N_STAT * p[mask])
    assert chi.pvalue > 1e-3


N_BIG = 1_000_000


@pytest.mark.parametrize("v", [8, 16])
@pytest.mark.parametrize("zeros_p,zeros_q", [(False, False), (True, False), (False, True), (True, True)])
def test_acceptance_rate_and_output_law_at_one_million(v, zeros_p, zeros_q):
    """The same closed form and chi-square as above at N = 10^6 single-draft blocks and
    V in {8, 16}, on the oracle's batched one-draft rule; that rule equals the per-block
    sampled_accept exactly on the first 20 000 blocks."""
    T = 0.7
    rng = np.random.default_rng(100 + 10 * v + 2 * zeros_p + zeros_q)
    p, q = _dists(v, rng, zeros_p, zeros_q)
    z = np.tile(_logits_for(p, T), (2, 1))
    drafts = rng.choice(v, size=N_BIG, p=q)
    from oracle import philox
    pos = np.arange(N_BIG) * 4
    u0 = philox.uniform(77, 3, pos + 1, 0)
    u1 = philox.uniform(77, 3, pos + 1, 1)
    u2 = philox.uniform(77, 3, pos + 2, 1)
    acc, nxt = accept.sampled_accept_one_draft_batch(z, drafts, q, T, u0, u1, u2)
    for n in range(20_000):
        k, t = accept.sampled_accept(z, [drafts[n]], q[None, :], T, [u0[n]], [u1[n], u2[n]])
        assert (k, t) == (acc[n], nxt[n])
    want = np.minimum(p, q).sum()
    assert stats.binomtest(int(acc.sum()), N_BIG, want).pvalue > 1e-3
    first = np.bincount(np.where(acc == 1, drafts, nxt), minlength=v)
    mask = p > 0
    assert first[~mask].sum() == 0
    assert stats.chisquare(first[mask], N_BIG * p[mask]).pvalue > 1e-3


def test_two_position_chain_joint_distribution():
    """Joint law of the first two emitted tokens equals p0(x1) p1(x2 | x1).

    The target is a table: row 0 of the block has p0; the row after token x has p1(.|x).
    Drafts come from q0 and q1(.|d1). A step that emits only one token is followed by a
    second step with that token as the anchor.
    """
    v, T = 4, 1.0
    rng = np.random.default_rng(7)
    p0, q0 = _dists(v, rng)
    p1 = np.stack([_dists(v, rng)[0] for _ in range(v)])
    q1 = np.stack([_dists(v, rng)[1] for _ in range(v)])
    p_next = np.stack([p1[x] for x in range(v)])           # distribution after token x
    counts = np.zeros((v, v), np.int64)
    n_runs = 60_000
    from oracle import philox
    for n in range(n_runs):
        d1 = rng.choice(v, p=q0)
        d2 = rng.choice(v, p=q1[d1])
        z = np.stack([_logits_for(p0, T), _logits_for(p_next[d1], T), _logits_for(p_next[d2], T)])
        c = 3 * n
        u_acc, u_res = accept.uniforms(5, 2, 10 * n, 2)
        k, nxt = accept.sampled_accept(z, [d1, d2], np.stack([q0, q1[d1]]), T, u_acc, u_res)
        if k >= 1:
            x1 = d1
            x2 = d2 if k == 2 else nxt
        else:
            x1 = nxt
            dd = rng.choice(v, p=q1[x1])
            z2 = np.stack([_logits_for(p_next[x1], T), _logits_for(p_next[dd], T)])
            u_acc, u_res = accept.uniforms(5, 3, 10 * n, 1)
            k2, nxt2 = accept.sampled_accept(z2, [dd], q1[x1][None, :], T, u_acc, u_res)
            x2 = dd if k2 == 1 else nxt2
        counts[x1, x2] += 1
    want = p0[:, None] * p1
    chi = stats.chisquare(counts.ravel(), n_runs * want.ravel())
    assert chi.pvalue > 1e-3


# ---------------------------------------------------------------- speculative loop
def _tiny():
    shape = synth.SHAPES["tiny"]
    cfg = Config(**shape)
    w = synth.host_weights(shape, "f32")
    return cfg, DenseWeights(cfg, w["layers"], w["embed"], w["final_norm"], w["lm_head"])


def test_token_forcing_spec_greedy_equals_ar_greedy():
    """The speculative greedy output equals plain AR greedy token for token
    (LFM2.5-DSpark post, "Quality parity"; SpecPilot digest, token forcing)."""
    cfg, W = _tiny()
    prompt = synth.uniform_tokens(64, cfg.vocab, 1, 0)
    st, logits, nk, nv = spec.prefill(cfg, W, prompt)
    spec.commit(st, [], [a[-1:] for a in nk], [a[-1:] for a in nv], 0, int(np.argmax(logits[-1])))
    ar = spec.ar_greedy(cfg, W, st, 120)
    g_all = ar.emitted

    def drafter(s):
        off = len(s.emitted) - 1             # emitted includes the anchor itself
        return synth.greedy_mix_drafts(g_all[off + 1: off + 5], 4, 0.8, cfg.vocab, 2, off)

    sp, lens = spec.spec_greedy(cfg, W, st, drafter, 32)
    n = len(sp.emitted)
    assert n >= 32 and sum(lens) > 0
    assert sp.emitted == g_all[:n]
    # the committed cache equals the one AR decoding built for the same positions
    c = sp.length
    for l in range(cfg.n_layers):
        assert np.array_equal(sp.k[l], ar.k[l][:c])
        assert np.array_equal(sp.v[l], ar.v[l][:c])
