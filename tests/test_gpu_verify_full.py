"""GPU verify step against the oracle at the full 8B-class and 27B-class sizes.

8B-class: 36 layers, d 4096, 32 q / 8 kv heads x 128, ffn 12288, vocab 151936,
bf16 N(0, 0.02); random bf16 N(0, 1) context of 4096; one request with 16
drafts (M = 17), temperature 0. Every logit of the block is compared. The
drafts follow the workload's rule (draft i is the target's greedy token with
probability 0.9^(i+1), else uniform; the greedy tokens come from the engine's
own one-row steps), so long accepted prefixes are compared with the oracle.

27B-class: 64 layers, d 5120, 40 q / 8 kv heads x 128, ffn 17408, vocab
151936; 32 requests with contexts uniform in 512..8192 on a shuffled pool of
16-token pages; verify lengths from the cumulative-confidence rule
(c_i ~ Beta(8, 2), keep while prod c >= 0.3); drafts by the same greedy-mix
rule. The oracle recomputes requests 0, 7 and 31 through all layers (the
others are checked through the commit).

W12 at the 8B-class shapes: 4 decoder layers and the LM head with weights in
a 16-binade window (random sign and mantissa, exponents 108..123, so the
magnitudes resemble N(0, 0.02)), packed to W12 and rebuilt inside the GEMM.
"""
import numpy as np
import pytest

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

torch = pytest.importorskip("torch")
import synth  # noqa: E402
import synth.device as sd  # noqa: E402
import verify_step_02_b300 as vs  # noqa: E402
from oracle import decoder  # noqa: E402

from helpers import (LOGIT_TOL, DeviceContext, classify_greedy, device_oracle_weights,  # noqa: E402
                     engine_greedy_chain, report_decisions)

PAGE = 16


def _verify(model, tokens, lens, kv, gamma):
    b = len(lens)
    tok = np.zeros((b, gamma + 1), np.int32)
    for r, t in enumerate(tokens):
        tok[r, :len(t)] = t
    acc = torch.zeros(b, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(b, dtype=torch.int32, device="cuda")
    model.verify(torch.from_numpy(tok).cuda(), lens, kv, acc, nxt)
    m = int(sum(l + 1 for l in lens))
    logits = model.logits(m)
    model.sync_status()
    return acc.cpu().numpy(), nxt.cpu().numpy(), logits


def test_8b_gamma16_block_matches_oracle():
    shape = synth.SHAPES["8b"]
    C, gamma = 4096, 16
    wdev = sd.random_bf16_model(shape)
    table, n_pages = synth.contiguous_page_table([C + gamma + 1], PAGE, (C + gamma + 1) // PAGE + 2)
    ks, vs_ = sd.kv_pools(shape, n_pages, PAGE, torch.bfloat16, fill="normal")
    seq = torch.tensor([C], dtype=torch.int32, device="cuda")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    rng = np.random.default_rng(2)
    anchor = int(rng.integers(0, shape["vocab"]))
    model = vs.Model(vs.make_config(shape, vs.SV_BF16, 1, gamma, C + 64, PAGE, flags=vs.SV_FLAG_KEEP_LOGITS), wdev)
    chain = engine_greedy_chain(model, kv, [anchor], gamma, gamma)[0]
    block = [anchor] + [int(x) for x in synth.greedy_mix_drafts(chain, gamma, 0.9, shape["vocab"], 40, 0)]
    ctx = DeviceContext(ks, table[0], C, PAGE), DeviceContext(vs_, table[0], C, PAGE)
    cfg, W = device_oracle_weights(shape, wdev)
    lo, nk, nv = decoder.forward_block(cfg, W, ctx[0], ctx[1], block, C, rowwise=False)
    acc, nxt, lg = _verify(model, [block], [gamma], kv, gamma)
    lg = lg.cpu().numpy().astype(np.float64)
    err = np.abs(lg - lo).max()
    print(f"[8b] max |dlogit| {err:.4f}, accepted {int(acc[0])} of {gamma}")
    assert err <= LOGIT_TOL["bf16"], err
    report_decisions("8b gamma 16", [classify_greedy(lo, block[1:], acc[0], nxt[0])], 1)
    assert int(seq.item()) == C + int(acc[0]) + 1
    pos = C + np.arange(gamma + 1)
    for l in (0, shape["n_layers"] - 1):
        gk = sd.read_positions(ks[l], table[0], pos, PAGE).float().cpu().numpy()
        gv = sd.read_positions(vs_[l], table[0], pos, PAGE).float().cpu().numpy()
        assert np.allclose(gk, nk[l], rtol=2 ** -7, atol=1e-2)
        assert np.allclose(gv, nv[l], rtol=2 ** -7, atol=1e-2)
    model.close()


def test_27b_ragged_batch32_shuffled_pages():
    shape = synth.SHAPES["27b"]
    B, gamma = 32, 16
    rng = np.random.default_rng(3)
    ctx_len = rng.integers(512, 8193, size=B)
    lens = synth.truncated_verify_lens(B, gamma, 0.3, 3, 1)
    wdev = sd.random_bf16_model(shape)
    need = [int(c) + gamma + 1 for c in ctx_len]
    max_pages = max((n + PAGE - 1) // PAGE for n in need) + 1
    table, n_pages = synth.shuffled_page_table(need, PAGE, max_pages, 3, 2)
    ks, vs_ = sd.kv_pools(shape, n_pages, PAGE, torch.bfloat16, fill="normal")
    seq = torch.tensor(ctx_len, dtype=torch.int32, device="cuda")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    anchors = [int(x) for x in rng.integers(0, shape["vocab"], size=B)]
    model = vs.Model(vs.make_config(shape, vs.SV_BF16, B, gamma, 8192 + gamma + 16, PAGE,
                                    flags=vs.SV_FLAG_KEEP_LOGITS), wdev)
    chains = engine_greedy_chain(model, kv, anchors, gamma, gamma)
    blocks = [[anchors[r]] + [int(x) for x in synth.greedy_mix_drafts(chains[r], int(lens[r]), 0.9, shape["vocab"],
                                                                        41, r)] for r in range(B)]
    acc, nxt, lg = _verify(model, blocks, [int(l) for l in lens], kv, gamma)
    assert np.array_equal(seq.cpu().numpy(), ctx_len + acc + 1)
    row0 = np.r_[0, np.cumsum(np.asarray(lens) + 1)]
    picks = [0, 7, 31]
    cfg, W = device_oracle_weights(shape, wdev)
    reqs = [(DeviceContext(ks, table[r], int(ctx_len[r]), PAGE), DeviceContext(vs_, table[r], int(ctx_len[r]), PAGE),
             blocks[r], int(ctx_len[r])) for r in picks]
    outs = decoder.forward_blocks(cfg, W, reqs, rowwise=False)
    verdicts = []
    for r, (lo, _, _) in zip(picks, outs):
        g = lg[row0[r]:row0[r + 1]].cpu().numpy().astype(np.float64)
        err = np.abs(g - lo).max()
        print(f"[27b] request {r}: max |dlogit| {err:.4f}, accepted {int(acc[r])} of {int(lens[r])}")
        assert err <= LOGIT_TOL["bf16"], (r, err)
        verdicts.append(classify_greedy(lo, blocks[r][1:], acc[r], nxt[r]))
    report_decisions("27b ragged batch 32 (requests 0, 7, 31)", verdicts, 1)
    print(f"[27b] accepted lengths of all 32 requests: {acc.tolist()}")
    model.close()


def window_bits_device(shp, seed):
    """bf16 patterns: random sign and mantissa, exponent uniform in 108..123 (a 16-binade window)."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    bits = (torch.randint(0, 2, shp, device="cuda", generator=g, dtype=torch.int32) << 15) | \
        (torch.randint(108, 124, shp, device="cuda", generator=g, dtype=torch.int32) << 7) | \
        torch.randint(0, 128, shp, device="cuda", generator=g, dtype=torch.int32)
    return bits.to(torch.int16).view(torch.bfloat16)


def test_w12_8b_shapes_four_layers_and_lm_head():
    shape = dict(synth.SHAPES["8b"], n_layers=4)
    C, gamma = 1024, 16
    ms = synth.matrix_shapes(shape)
    d = shape["d_model"]
    ones = torch.ones(d, dtype=torch.bfloat16, device="cuda")
    wbf = {"layers": [], "final_norm": ones,
           "embed": synth.device_bf16_normal((shape["vocab"], d), 0.02, (0, synth.T_EMBED), "cuda"),
           "lm_head": window_bits_device((shape["vocab"], d), 9100)}
    for l in range(shape["n_layers"]):
        wbf["layers"].append(dict(attn_norm=ones, mlp_norm=ones,
                                  **{n: window_bits_device(ms[n], 9000 + 10 * l + i)
                                     for i, n in enumerate(("wqkv", "wo", "wgu", "wd"))}))
    w12 = {"embed": wbf["embed"], "final_norm": ones, "lm_head": vs.pack_w12(wbf["lm_head"]),
           "layers": [dict(attn_norm=ones, mlp_norm=ones, **{n: vs.pack_w12(lay[n])
                                                             for n in ("wqkv", "wo", "wgu", "wd")})
                      for lay in wbf["layers"]]}
    for lay, lay12 in zip(wbf["layers"], w12["layers"]):  # the planes rebuild the same bits
        got = vs.unpack_w12(*lay12["wo"], *ms["wo"])
        assert torch.equal(got.view(torch.int16), lay["wo"].view(torch.int16))
    table, n_pages = synth.contiguous_page_table([C + gamma + 1], PAGE, (C + gamma + 1) // PAGE + 2)
    ks, vs_ = sd.kv_pools(shape, n_pages, PAGE, torch.bfloat16, fill="normal")
    seq = torch.tensor([C], dtype=torch.int32, device="cuda")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    model = vs.Model(vs.make_config(shape, vs.SV_W12, 1, gamma, C + 64, PAGE, flags=vs.SV_FLAG_KEEP_LOGITS), w12)
    rng = np.random.default_rng(12)
    anchor = int(rng.integers(0, shape["vocab"]))
    chain = engine_greedy_chain(model, kv, [anchor], gamma, gamma)[0]
    block = [anchor] + [int(x) for x in synth.greedy_mix_drafts(chain, gamma, 0.9, shape["vocab"], 42, 0)]
    acc, nxt, lg = _verify(model, [block], [gamma], kv, gamma)
    lg = lg.cpu().numpy().astype(np.float64)
    cfg, W = device_oracle_weights(shape, wbf)
    ctx = DeviceContext(ks, table[0], C, PAGE), DeviceContext(vs_, table[0], C, PAGE)
    lo, _, _ = decoder.forward_block(cfg, W, ctx[0], ctx[1], block, C, rowwise=False)
    err = np.abs(lg - lo).max()
    print(f"[w12 8b shapes] max |dlogit| {err:.4f} (logit scale {np.abs(lo).max():.2f}), accepted {int(acc[0])}")
    assert err <= LOGIT_TOL["bf16"], err
    report_decisions("w12 8b shapes", [classify_greedy(lo, block[1:], acc[0], nxt[0])], 1)
    model.close()


def test_8b_token_tree_matches_oracle():
    """A 32-node token tree at the 8B-class shapes (context 4096): every node's logits, the accepted
    path and the committed keys/values against the oracle's tree forward."""
    from oracle import accept
    from helpers import classify_tree
    shape = synth.SHAPES["8b"]
    C, n = 4096, 32
    wdev = sd.random_bf16_model(shape)
    table, n_pages = synth.contiguous_page_table([C + n], PAGE, (C + n) // PAGE + 2)
    ks, vs_ = sd.kv_pools(shape, n_pages, PAGE, torch.bfloat16, fill="normal")
    seq = torch.tensor([C], dtype=torch.int32, device="cuda")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    rng = np.random.default_rng(6)
    anchor = int(rng.integers(0, shape["vocab"]))
    model = vs.Model(vs.make_config(shape, vs.SV_BF16, 1, n - 1, C + 64, PAGE, flags=vs.SV_FLAG_KEEP_LOGITS), wdev)
    chain = engine_greedy_chain(model, kv, [anchor], 8, n - 1)[0]
    parents = synth.random_tree(n, 3, 90, 0)
    tokens = synth.tree_drafts(parents, anchor, chain, 0.9, shape["vocab"], 91, 0)
    ctx = DeviceContext(ks, table[0], C, PAGE), DeviceContext(vs_, table[0], C, PAGE)
    cfg, W = device_oracle_weights(shape, wdev)
    lo, nk, nv = decoder.forward_tree(cfg, W, ctx[0], ctx[1], tokens, parents, C, rowwise=False)
    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    nodes = torch.zeros((1, n), dtype=torch.int32, device="cuda")
    model.verify_tree(torch.from_numpy(np.asarray([tokens], np.int32)).cuda(),
                      torch.from_numpy(np.asarray([parents], np.int32)).cuda(), [n - 1], kv, acc, nxt, nodes)
    lg = model.logits(n).cpu().numpy().astype(np.float64)
    model.sync_status()
    err = np.abs(lg - lo).max()
    k = int(acc.item())
    k_o, _, _ = accept.greedy_accept_tree(lo, tokens, parents)
    print(f"[8b tree] {n} nodes: max |dlogit| {err:.4f}, accepted {k} (oracle {k_o})")
    assert err <= LOGIT_TOL["bf16"], err
    report_decisions("8b token tree", [classify_tree(lo, tokens, parents, k, int(nxt.item()),
                                                     nodes.cpu().numpy()[0])], 1)
    assert int(seq.item()) == C + k + 1
    path = [int(x) for x in nodes.cpu().numpy()[0, :k + 1]]
    pos = C + np.arange(k + 1)
    for l in (0, shape["n_layers"] - 1):
        gk = sd.read_positions(ks[l], table[0], pos, PAGE).float().cpu().numpy()
        assert np.allclose(gk, nk[l][path], rtol=2 ** -7, atol=1e-2)
    model.close()
