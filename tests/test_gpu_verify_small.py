"""GPU verify step against the oracle on the small workloads (through the C ABI).

- tiny fp32 greedy: 2 layers, d 256, 4 heads x 64, ffn 688, vocab 1024; 64-token
  prompt prefilled by the oracle; gamma 4 drafts (greedy token w.p. 0.8^(i+1)).
  One step compared row by row, then a 32-step token-forcing run.
- W12: the same shapes with 16-binade-window weights packed to W12, gamma 16.
- bf16 GQA ragged batch on shuffled pages (GQA group 4, ragged L_r incl. 0).
- tiny fp32 sampled: batch 64, context 2048, gamma 8 chain drafts, T = 1.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import synth  # noqa: E402
import synth.device as sd  # noqa: E402
import verify_step_02_b300 as vs  # noqa: E402
from oracle import accept, decoder, spec  # noqa: E402

from helpers import (LOGIT_TOL, build_kv, classify_greedy, classify_sampled, oracle_weights,  # noqa: E402
                     torch_dtype)

PAGE = 16


def gpu_weights(hw, kind):
    if kind == "f32":
        return sd.host_to_device_weights(hw, "f32")
    w = sd.host_to_device_weights(hw, "bf16")
    if kind == "w12":
        for lay in w["layers"]:
            for name in ("wqkv", "wo", "wgu", "wd"):
                lay[name] = vs.pack_w12(lay[name])
        w["lm_head"] = vs.pack_w12(w["lm_head"])
    return w


def make_model(shape, kind, wdev, max_batch, max_gamma, max_seq_len, keep=True):
    wd = {"f32": vs.SV_F32, "bf16": vs.SV_BF16, "w12": vs.SV_W12}[kind]
    cfg = vs.make_config(shape, wd, max_batch, max_gamma, max_seq_len, PAGE,
                         flags=vs.SV_FLAG_KEEP_LOGITS if keep else 0)
    return vs.Model(cfg, wdev)


def prompt_state(cfg, W, n_prompt, stream):
    prompt = synth.uniform_tokens(n_prompt, cfg.vocab, *stream)
    st, logits, nk, nv = spec.prefill(cfg, W, prompt)
    spec.commit(st, [], [a[-1:] for a in nk], [a[-1:] for a in nv], 0, int(np.argmax(logits[-1])))
    return st


def run_step(model, states, drafts, max_gamma, kv, temperature=0.0, probs=None, seed=0, req_ids=None):
    b = len(states)
    tok = np.zeros((b, max_gamma + 1), np.int32)
    for r, st in enumerate(states):
        tok[r, 0] = st.anchor
        tok[r, 1:1 + len(drafts[r])] = drafts[r]
    tok_d = torch.from_numpy(tok).cuda()
    acc = torch.zeros(b, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(b, dtype=torch.int32, device="cuda")
    pd = None if probs is None else torch.from_numpy(np.ascontiguousarray(probs, dtype=np.float32)).cuda()
    rid = None if req_ids is None else torch.tensor(req_ids, dtype=torch.int64, device="cuda")
    model.verify(tok_d, [len(d) for d in drafts], kv, acc, nxt, draft_probs=pd, temperature=temperature,
                 seed=seed, request_ids=rid)
    m = sum(len(d) + 1 for d in drafts)
    logits = model.logits(m).cpu().numpy().astype(np.float64)
    model.sync_status()
    return acc.cpu().numpy(), nxt.cpu().numpy(), logits


@pytest.mark.parametrize("kind", ["f32", "w12"])
def test_tiny_single_step_rows_kv_and_commit(kind):
    shape = synth.SHAPES["tiny"]
    hw = synth.host_weights(shape, "f32" if kind == "f32" else "w12window")
    cfg, W = oracle_weights(shape, hw, kind)
    gamma = 4 if kind == "f32" else 16
    st = prompt_state(cfg, W, 64, (1, 0))
    g = spec.ar_greedy(cfg, W, st, gamma + 1).emitted[1:]
    drafts = [int(x) for x in synth.greedy_mix_drafts(g, gamma, 0.8, cfg.vocab, 2, 0)]
    k_o, n_o, lo, nk, nv = spec.verify(cfg, W, st, drafts)
    model = make_model(shape, kind, gpu_weights(hw, kind), 1, gamma, 256)
    ks, vs_, table, seq = build_kv(shape, [st], PAGE, gamma, kind)
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    acc, nxt, lg = run_step(model, [st], [drafts], gamma, kv)
    tol = LOGIT_TOL["f32" if kind == "f32" else "bf16"]
    assert np.abs(lg - lo).max() <= tol, np.abs(lg - lo).max()
    assert classify_greedy(lo, drafts, acc[0], nxt[0]) in ("match", "near_tie")
    assert seq.cpu().numpy()[0] == st.length + int(acc[0]) + 1
    pos = st.length + np.arange(gamma + 1)
    for l in range(shape["n_layers"]):
        gk = sd.read_positions(ks[l], table[0], pos, PAGE).float().cpu().numpy()
        gv = sd.read_positions(vs_[l], table[0], pos, PAGE).float().cpu().numpy()
        kv_tol = 1e-5 if kind == "f32" else 2 ** -7
        assert np.allclose(gk, nk[l], rtol=kv_tol, atol=kv_tol)
        assert np.allclose(gv, nv[l], rtol=kv_tol, atol=kv_tol)


def test_tiny_token_forcing_32_steps():
    """Spec greedy on the GPU reproduces the oracle's AR greedy sequence token for token."""
    shape = synth.SHAPES["tiny"]
    hw = synth.host_weights(shape, "f32")
    cfg, W = oracle_weights(shape, hw, "f32")
    gamma = 4
    st = prompt_state(cfg, W, 64, (1, 0))
    g_all = spec.ar_greedy(cfg, W, st, 32 * (gamma + 1) + gamma + 2).emitted   # g_all[0] is the anchor
    model = make_model(shape, "f32", gpu_weights(hw, "f32"), 1, gamma, 64 + 32 * (gamma + 1) + 32)
    ks, vs_, table, seq = build_kv(shape, [st], PAGE, 32 * (gamma + 1) + gamma, "f32")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    emitted = [st.anchor]
    anchor = st.anchor
    tok_d = torch.zeros((1, gamma + 1), dtype=torch.int32, device="cuda")
    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    accepted = 0
    for step in range(32):
        off = len(emitted) - 1
        drafts = synth.greedy_mix_drafts(g_all[off + 1: off + 1 + gamma], gamma, 0.8, cfg.vocab, 3, step)
        tok_d.copy_(torch.tensor([[anchor] + [int(d) for d in drafts]], dtype=torch.int32))
        model.verify(tok_d, [gamma], kv, acc, nxt)
        k, n = int(acc.item()), int(nxt.item())
        accepted += k
        emitted += [int(d) for d in drafts[:k]] + [n]
        anchor = n
    model.sync_status()
    assert accepted > 0
    assert emitted == g_all[:len(emitted)]
    assert int(seq.item()) == st.length + len(emitted) - 1


@pytest.mark.parametrize("kind", ["bf16", "w12"])
def test_bf16_gqa_ragged_batch_shuffled_pages(kind):
    """bf16 or W12 weights (both on the tensor-core GEMM: ffn is a multiple of 64)."""
    shape = dict(n_layers=2, d_model=512, n_heads=8, n_kv_heads=2, head_dim=128, ffn=1024, vocab=4096,
                 rope_theta=1e6)
    hw = synth.host_weights(shape, "w12window")
    # keep activations moderate: scale the window weights down by 2^-4 (still exact bf16)
    for lay in hw["layers"]:
        for name in ("wqkv", "wo", "wgu", "wd"):
            lay[name] = (lay[name].astype(np.int64) - (4 << 7)).astype(np.uint16)
    cfg, W = oracle_weights(shape, hw, "bf16")
    gamma = 8
    lens = [8, 0, 3, 8, 1]
    ctx = [40, 7, 0, 129, 16]
    rng = np.random.default_rng(11)
    states = []
    for r, c in enumerate(ctx):
        stt = spec.empty_state(cfg, int(rng.integers(0, cfg.vocab)), request_id=r)
        stt.k = [decoder.round_to_bf16(rng.standard_normal((c, 2, 128))) for _ in range(2)]
        stt.v = [decoder.round_to_bf16(rng.standard_normal((c, 2, 128))) for _ in range(2)]
        states.append(stt)
    drafts = [[int(x) for x in rng.integers(0, cfg.vocab, size=n)] for n in lens]
    model = make_model(shape, kind, gpu_weights(hw, kind), 8, gamma, 512)
    ks, vs_, table, seq = build_kv(shape, states, PAGE, gamma, "bf16")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    acc, nxt, lg = run_step(model, states, drafts, gamma, kv)
    row = 0
    for r, stt in enumerate(states):
        k_o, n_o, lo, _, _ = spec.verify(cfg, W, stt, drafts[r])
        rows = lens[r] + 1
        assert np.abs(lg[row:row + rows] - lo).max() <= LOGIT_TOL["bf16"], (r, np.abs(lg[row:row + rows] - lo).max())
        assert classify_greedy(lo, drafts[r], acc[r], nxt[r]) in ("match", "near_tie")
        row += rows
    assert np.array_equal(seq.cpu().numpy(), np.array(ctx) + acc + 1)


def test_tiny_sampled_batch64_ctx2048():
    """T = 1 rejection sampling; chain drafts q_i = softmax(z_{i-1} + N(0,1)), d_i ~ q_i."""
    shape = synth.SHAPES["tiny"]
    hw = synth.host_weights(shape, "f32")
    cfg, W = oracle_weights(shape, hw, "f32")
    B, C, gamma, T, seed = 64, 2048, 8, 1.0, 20261202
    rng = np.random.default_rng(5)
    states, drafts, probs, logits_o = [], [], [], []
    for r in range(B):
        stt = spec.empty_state(cfg, int(rng.integers(0, cfg.vocab)), request_id=1000 + r)
        stt.k = [rng.standard_normal((C, 4, 64)).astype(np.float32).astype(np.float64) for _ in range(2)]
        stt.v = [rng.standard_normal((C, 4, 64)).astype(np.float32).astype(np.float64) for _ in range(2)]
        # chain: row j's logits need the drafts before it; rows are computed one at a time
        work = stt.copy()
        block, zs, qs = [stt.anchor], [], []
        for i in range(gamma + 1):
            z, nk, nv = decoder.forward_block(cfg, W, work.k, work.v, [block[-1]], work.length)
            zs.append(z[0])
            work.k = [np.concatenate([a, b]) for a, b in zip(work.k, nk)]
            work.v = [np.concatenate([a, b]) for a, b in zip(work.v, nv)]
            if i == gamma:
                break
            ql = accept.softmax(z[0] + rng.standard_normal(cfg.vocab), T).astype(np.float32)
            ql = ql / ql.sum(dtype=np.float64)
            d = int(rng.choice(cfg.vocab, p=ql.astype(np.float64) / ql.astype(np.float64).sum()))
            qs.append(ql.astype(np.float32))
            block.append(d)
        states.append(stt)
        drafts.append(block[1:])
        probs.append(np.stack(qs))
        logits_o.append(np.stack(zs))
    model = make_model(shape, "f32", gpu_weights(hw, "f32"), B, gamma, C + gamma + 2, keep=False)
    ks, vs_, table, seq = build_kv(shape, states, PAGE, gamma, "f32")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    acc, nxt, lg = run_step(model, states, drafts, gamma, kv, temperature=T, probs=np.stack(probs), seed=seed,
                            req_ids=[1000 + r for r in range(B)])
    verdicts = []
    for r in range(B):
        lo = logits_o[r]
        assert np.abs(lg[r * (gamma + 1):(r + 1) * (gamma + 1)] - lo).max() <= LOGIT_TOL["f32"]
        verdicts.append(classify_sampled(lo, drafts[r], probs[r], T, seed, 1000 + r, C, acc[r], nxt[r]))
    assert "mismatch" not in verdicts, verdicts
    assert verdicts.count("near_tie") <= 2
    assert acc.sum() > 0


def test_bf16_gqa_sampled_batch():
    """T = 0.8 rejection sampling on the tensor-core path (bf16 GQA model, ragged contexts): chain
    drafts q_i = softmax((z_{i-1} + N(0, 1)) / T) from the oracle's target logits, d_i ~ q_i."""
    from helpers import report_decisions
    shape = dict(n_layers=2, d_model=512, n_heads=8, n_kv_heads=2, head_dim=128, ffn=1024, vocab=4096,
                 rope_theta=1e6)
    hw = synth.host_weights(shape, "w12window")
    for lay in hw["layers"]:
        for name in ("wqkv", "wo", "wgu", "wd"):
            lay[name] = (lay[name].astype(np.int64) - (4 << 7)).astype(np.uint16)
    cfg, W = oracle_weights(shape, hw, "bf16")
    B, gamma, T, seed = 6, 5, 0.8, 777
    rng = np.random.default_rng(29)
    ctx = [int(c) for c in rng.integers(1, 200, size=B)]
    states, drafts, probs, logits_o = [], [], [], []
    for r, c in enumerate(ctx):
        stt = spec.empty_state(cfg, int(rng.integers(0, cfg.vocab)), request_id=500 + r)
        stt.k = [decoder.round_to_bf16(rng.standard_normal((c, 2, 128))) for _ in range(2)]
        stt.v = [decoder.round_to_bf16(rng.standard_normal((c, 2, 128))) for _ in range(2)]
        work = stt.copy()
        block, zs, qs = [stt.anchor], [], []
        for i in range(gamma + 1):
            z, nk, nv = decoder.forward_block(cfg, W, work.k, work.v, [block[-1]], work.length)
            zs.append(z[0])
            work.k = [np.concatenate([a, b]) for a, b in zip(work.k, nk)]
            work.v = [np.concatenate([a, b]) for a, b in zip(work.v, nv)]
            if i == gamma:
                break
            ql = accept.softmax(z[0] + rng.standard_normal(cfg.vocab), T).astype(np.float32)
            ql = ql / ql.sum(dtype=np.float64)
            block.append(int(rng.choice(cfg.vocab, p=ql.astype(np.float64) / ql.astype(np.float64).sum())))
            qs.append(ql.astype(np.float32))
        states.append(stt)
        drafts.append(block[1:])
        probs.append(np.stack(qs))
        logits_o.append(np.stack(zs))
    model = make_model(shape, "bf16", gpu_weights(hw, "bf16"), B, gamma, 512)
    ks, vs_, table, seq = build_kv(shape, states, PAGE, gamma, "bf16")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    acc, nxt, lg = run_step(model, states, drafts, gamma, kv, temperature=T, probs=np.stack(probs), seed=seed,
                            req_ids=[500 + r for r in range(B)])
    verdicts = []
    for r in range(B):
        lo = logits_o[r]
        err = np.abs(lg[r * (gamma + 1):(r + 1) * (gamma + 1)] - lo).max()
        assert err <= LOGIT_TOL["bf16"], (r, err)
        verdicts.append(classify_sampled(lo, drafts[r], probs[r], T, seed, 500 + r, ctx[r], acc[r], nxt[r]))
    report_decisions("bf16 GQA sampled, T 0.8", verdicts, 1)
    assert np.array_equal(seq.cpu().numpy(), np.array(ctx) + acc + 1)
