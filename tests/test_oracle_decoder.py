"""Pins for the oracle's decoder forward (CPU only).

The pages print no worked example of a forward pass, so the logits are
pinned by special cases that reduce to closed forms and by invariants.
"""
import cmath

import numpy as np
import pytest

import synth
from oracle import decoder, spec
from oracle.decoder import Config, DenseWeights


def tiny_cfg(**kw):
    base = dict(synth.SHAPES["tiny"])
    base.update(kw)
    return Config(**base)


def tiny_weights(cfg):
    w = synth.host_weights(synth.SHAPES["tiny"], "f32")
    return w, DenseWeights(cfg, w["layers"], w["embed"], w["final_norm"], w["lm_head"])


def test_rope_identity_at_zero_and_complex_rotation():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((3, 2, 8))
    assert np.array_equal(decoder.rope(x, np.zeros(3), 1e4), x)
    pos = np.array([1, 17, 4095])
    got = decoder.rope(x, pos, 1e4)
    # independent statement: pair (x_i, x_{i+4}) as the complex number x_i + j x_{i+4},
    # multiplied by exp(j * p * theta^(-2i/8))
    for m, p in enumerate(pos):
        for h in range(2):
            for i in range(4):
                z = complex(x[m, h, i], x[m, h, i + 4]) * cmath.exp(1j * p * 1e4 ** (-2 * i / 8))
                assert abs(got[m, h, i] - z.real) < 1e-12
                assert abs(got[m, h, i + 4] - z.imag) < 1e-12


def test_rope_scores_depend_on_offset_only():
    rng = np.random.default_rng(1)
    q, k = rng.standard_normal((1, 1, 64)), rng.standard_normal((1, 1, 64))
    s1 = (decoder.rope(q, [10], 1e6) * decoder.rope(k, [3], 1e6)).sum()
    s2 = (decoder.rope(q, [1007], 1e6) * decoder.rope(k, [1000], 1e6)).sum()
    assert abs(s1 - s2) < 1e-9


def test_attention_single_key_returns_value_per_kv_head():
    rng = np.random.default_rng(2)
    q = rng.standard_normal((8, 16))
    keys = rng.standard_normal((1, 2, 16))
    vals = rng.standard_normal((1, 2, 16))
    out = decoder.attention_row(q, keys, vals)
    for i in range(8):
        assert np.array_equal(out[i], vals[0, i // 4])     # query head i reads kv head i // 4


def test_attention_equal_keys_average_values():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((2, 16))
    keys = np.repeat(rng.standard_normal((1, 1, 16)), 7, axis=0)
    vals = rng.standard_normal((7, 1, 16))
    out = decoder.attention_row(q, keys, vals)
    assert np.allclose(out, vals[:, 0].mean(axis=0)[None, :], atol=1e-13)


def test_attention_two_keys_logistic_weight():
    q = np.array([[1.0, 0.0, 0.0, 0.0]])
    keys = np.array([[[2.0, 0, 0, 0]], [[0.0, 0, 0, 0]]])
    vals = np.array([[[1.0, 0, 0, 0]], [[0.0, 0, 0, 0]]])
    w = 1.0 / (1.0 + np.exp(-2.0 / 2.0))               # scores 2/sqrt(4) and 0
    assert abs(decoder.attention_row(q, keys, vals)[0, 0] - w) < 1e-15


def test_rmsnorm_constant_and_scale():
    x = np.full((1, 256), -3.0)
    g = np.linspace(0.5, 2.0, 256)
    got = decoder.rmsnorm(x, g, 1e-6)
    assert np.allclose(got, -g / np.sqrt(1 + 1e-6 / 9.0), rtol=0, atol=1e-15)
    y = np.random.default_rng(4).standard_normal((2, 256))
    assert np.allclose(decoder.rmsnorm(y, 1.0, 0.0), decoder.rmsnorm(1000 * y, 1.0, 0.0))


def test_silu_closed_forms():
    assert decoder.silu(0.0) == 0.0
    assert abs(decoder.silu(1.0) - 1.0 / (1.0 + np.exp(-1.0))) < 1e-16
    assert abs(decoder.silu(-40.0)) < 1e-15


def test_round_to_bf16_matches_float32_route_and_ties_to_even():
    import torch
    x = np.random.default_rng(5).standard_normal(20000).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).to(torch.float64).numpy()   # RNE from float32
    assert np.array_equal(decoder.round_to_bf16(x.astype(np.float64)), want)
    # exact ties: 1 + 2^-8 lies halfway between 1 and 1 + 2^-7 -> even mantissa (1.0)
    assert decoder.round_to_bf16(1.0 + 2**-8) == 1.0
    assert decoder.round_to_bf16(1.0 + 3 * 2**-8) == 1.0 + 2**-6
    assert decoder.round_to_bf16(-(1.0 + 2**-8 + 2**-30)) == -(1.0 + 2**-7)


def test_rowwise_and_blocked_linear_agree():
    rng = np.random.default_rng(6)
    x, w = rng.standard_normal((5, 64)), rng.standard_normal((33, 64))
    assert np.allclose(decoder.linear(x, w, True), x @ w.T, atol=1e-12)
    assert np.allclose(decoder.linear(x, w, False), np.einsum("mk,nk->mn", x, w), atol=1e-12)


def _zeroed(w, names):
    out = {k: v for k, v in w.items() if k != "layers"}
    out["layers"] = []
    for lay in w["layers"]:
        d = dict(lay)
        for n in names:
            d[n] = np.zeros_like(d[n])
        out["layers"].append(d)
    return out


def test_zero_sublayers_reduce_to_embedding_logits():
    cfg = tiny_cfg()
    w, _ = tiny_weights(cfg)
    wz = _zeroed(w, ["wo", "wd"])
    W = DenseWeights(cfg, wz["layers"], wz["embed"], wz["final_norm"], wz["lm_head"])
    st = spec.empty_state(cfg, 0)
    toks = [3, 900, 17]
    logits, _, _ = decoder.forward_block(cfg, W, st.k, st.v, toks, 0)
    e = w["embed"][toks].astype(np.float64)
    want = (e / np.sqrt((e * e).mean(axis=1, keepdims=True) + 1e-6)) @ w["lm_head"].astype(np.float64).T
    assert np.allclose(logits, want, atol=1e-12)


def test_zero_query_key_weights_give_causal_mean_of_values():
    """With Wq = Wk = 0 every score is 0, so row j averages the values of keys 0 .. C+j."""
    cfg = tiny_cfg(n_layers=1)
    w, _ = tiny_weights(cfg)
    lay = dict(w["layers"][0])
    nq = cfg.n_heads * cfg.head_dim
    wqkv = lay["wqkv"].copy()
    wqkv[: 2 * nq] = 0.0                           # q rows and k rows (n_kv == n_heads here)
    lay["wqkv"] = wqkv
    lay["wd"] = np.zeros_like(lay["wd"])
    W = DenseWeights(cfg, [lay], w["embed"], w["final_norm"], w["lm_head"])
    rng = np.random.default_rng(7)
    c = 5
    ctx_k = [rng.standard_normal((c, 4, 64))]
    ctx_v = [rng.standard_normal((c, 4, 64))]
    toks = [1, 2, 3, 4]
    out = []
    decoder.forward_block(cfg, W, ctx_k, ctx_v, toks, c, layers_out=out)
    e = w["embed"][toks].astype(np.float64)
    u = e / np.sqrt((e * e).mean(axis=1, keepdims=True) + 1e-6)
    v_new = (u @ wqkv[2 * nq:].astype(np.float64).T).astype(np.float32).astype(np.float64)
    allv = np.concatenate([ctx_v[0].reshape(c, -1), v_new], axis=0)
    for j in range(4):
        o = allv[: c + j + 1].mean(axis=0)
        want = e[j] + lay["wo"].astype(np.float64) @ o
        assert np.allclose(out[0][j], want, atol=1e-12)


def test_block_rows_do_not_see_later_rows_and_match_ar():
    cfg = tiny_cfg()
    _, W = tiny_weights(cfg)
    st, _, _, _ = spec.prefill(cfg, W, synth.uniform_tokens(12, cfg.vocab, 9, 9))
    toks = [st.anchor, 5, 6, 7]
    l1, _, _ = decoder.forward_block(cfg, W, st.k, st.v, toks, st.length)
    l2, _, _ = decoder.forward_block(cfg, W, st.k, st.v, toks[:3] + [1000], st.length)
    assert np.array_equal(l1[:3], l2[:3])
    assert not np.array_equal(l1[3], l2[3])
    # a row computed alone (AR) is bit-identical to the same row inside the block
    one, _, _ = decoder.forward_block(cfg, W, st.k, st.v, toks[:1], st.length)
    assert np.array_equal(one[0], l1[0])


@pytest.mark.parametrize("kv_dtype", ["f32", "bf16"])
def test_cache_rounding(kv_dtype):
    cfg = tiny_cfg(kv_dtype=kv_dtype, n_layers=1)
    _, W = tiny_weights(cfg)
    st = spec.empty_state(cfg, 0)
    _, nk, nv = decoder.forward_block(cfg, W, st.k, st.v, [4, 5], 0)
    r = decoder.round_to_cache(nk[0], kv_dtype)
    assert np.array_equal(r, nk[0])
    if kv_dtype == "bf16":
        assert np.array_equal(decoder.bf16_bits_to_f64(decoder.f64_to_bf16_bits(nv[0])), nv[0])


def test_swiglu_gate_and_up_closed_form():
    """One gate row reading coordinate 3 (times 2), one up row reading coordinate 7,
    one down column writing coordinate 5: h += e_5 * SiLU(2 u_3) * u_7."""
    from scipy.special import expit
    cfg = tiny_cfg(n_layers=1)
    w, _ = tiny_weights(cfg)
    lay = dict(w["layers"][0])
    lay["wo"] = np.zeros_like(lay["wo"])
    wgu = np.zeros_like(lay["wgu"])
    wgu[0, 3] = 2.0                       # gate row 0
    wgu[cfg.ffn + 0, 7] = 1.0             # up row 0
    wd = np.zeros_like(lay["wd"])
    wd[5, 0] = 1.0
    lay["wgu"], lay["wd"] = wgu, wd
    W = DenseWeights(cfg, [lay], w["embed"], w["final_norm"], w["lm_head"])
    st = spec.empty_state(cfg, 0)
    out = []
    toks = [11, 12]
    decoder.forward_block(cfg, W, st.k, st.v, toks, 0, layers_out=out)
    e = w["embed"][toks].astype(np.float64)
    u = e / np.sqrt((e * e).mean(axis=1, keepdims=True) + 1e-6)
    want = e.copy()
    want[:, 5] += (2 * u[:, 3]) * expit(2 * u[:, 3]) * u[:, 7]
    assert np.allclose(out[0], want, atol=1e-13)
