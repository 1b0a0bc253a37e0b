"""GPU token-tree verification against the oracle (through the C ABI).

Trees of every shape in one batch (a chain, a star, random trees up to the
64-node limit) with drafts that follow the target's greedy continuation, so
that accepted paths run deep and through side branches:
  * float32 tiny model (CUDA-core GEMM and attention) and a bf16 GQA model
    (tensor-core GEMM and attention, 64 nodes x group 4 = two row tiles);
  * every node's logits against the oracle's tree forward, the decision
    (accepted length, next token, path) exactly, and the committed cache:
    positions C .. C + k hold the path's keys/values;
  * a chain-shaped tree gives bit-identical logits to the block verify;
  * token forcing: twelve tree steps emit the oracle's AR greedy sequence;
  * a parent that does not precede its node is a device check.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import synth  # noqa: E402
import synth.device as sd  # noqa: E402
import verify_step_02_b300 as vs  # noqa: E402
from oracle import decoder, spec  # noqa: E402

from helpers import LOGIT_TOL, build_kv, classify_tree, oracle_weights  # noqa: E402

PAGE = 16
GQA = dict(n_layers=2, d_model=512, n_heads=8, n_kv_heads=2, head_dim=128, ffn=1024, vocab=4096, rope_theta=1e6)


def setup(kind):
    shape = synth.SHAPES["tiny"] if kind == "f32" else GQA
    hw = synth.host_weights(shape, "f32" if kind == "f32" else "w12window")
    if kind == "bf16":  # moderate activations: scale the window weights by 2^-4 (exact in bf16)
        for lay in hw["layers"]:
            for name in ("wqkv", "wo", "wgu", "wd"):
                lay[name] = (lay[name].astype(np.int64) - (4 << 7)).astype(np.uint16)
    cfg, W = oracle_weights(shape, hw, kind)
    wdev = sd.host_to_device_weights(hw, "f32" if kind == "f32" else "bf16")
    return shape, cfg, W, wdev


def states_for(kind, cfg, W, ctx):
    rng = np.random.default_rng(21)
    out = []
    for r, c in enumerate(ctx):
        if kind == "f32":
            prompt = synth.uniform_tokens(c + 1, cfg.vocab, 60, r)
            st, logits, nk, nv = spec.prefill(cfg, W, prompt)
        else:
            st = spec.empty_state(cfg, int(rng.integers(0, cfg.vocab)), request_id=r)
            st.k = [decoder.round_to_bf16(rng.standard_normal((c, cfg.n_kv_heads, cfg.head_dim)))
                    for _ in range(cfg.n_layers)]
            st.v = [decoder.round_to_bf16(rng.standard_normal((c, cfg.n_kv_heads, cfg.head_dim)))
                    for _ in range(cfg.n_layers)]
        out.append(st)
    return out


def run_tree(model, trees, max_gamma, kv):
    b = len(trees)
    tok = np.zeros((b, max_gamma + 1), np.int32)
    par = np.full((b, max_gamma + 1), -1, np.int32)
    for r, (t, p) in enumerate(trees):
        tok[r, :len(t)] = t
        par[r, :len(p)] = p
    acc = torch.zeros(b, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(b, dtype=torch.int32, device="cuda")
    nodes = torch.full((b, max_gamma + 1), -1, dtype=torch.int32, device="cuda")
    model.verify_tree(torch.from_numpy(tok).cuda(), torch.from_numpy(par).cuda(), [len(t) - 1 for t, _ in trees],
                      kv, acc, nxt, nodes)
    m = sum(len(t) for t, _ in trees)
    logits = model.logits(m).cpu().numpy().astype(np.float64)
    model.sync_status()
    return acc.cpu().numpy(), nxt.cpu().numpy(), nodes.cpu().numpy(), logits


@pytest.mark.parametrize("kind", ["f32", "bf16"])
def test_tree_batch_matches_oracle(kind):
    shape, cfg, W, wdev = setup(kind)
    ctx = [40, 0, 129, 63] if kind == "bf16" else [40, 21, 70, 33]
    sizes = [(9, 1), (13, 12), (64, 3), (30, 2)]  # (nodes, max children): a chain, a star, random trees
    states = states_for(kind, cfg, W, ctx)
    max_gamma = 63
    trees = []
    for r, (st, (n, mc)) in enumerate(zip(states, sizes)):
        greedy = spec.ar_greedy(cfg, W, st, 12).emitted[len(st.emitted):]
        parents = synth.random_tree(n, mc, 70, r) if mc < n - 1 else np.r_[-1, np.zeros(n - 1, np.int32)]
        trees.append((synth.tree_drafts(parents, st.anchor, greedy, 0.85, cfg.vocab, 71, r), parents))
    model = vs.Model(vs.make_config(shape, vs.SV_F32 if kind == "f32" else vs.SV_BF16, len(ctx), max_gamma, 512, PAGE,
                                    flags=vs.SV_FLAG_KEEP_LOGITS), wdev)
    ks, vs_, table, seq = build_kv(shape, states, PAGE, max_gamma, kind)
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    acc, nxt, nodes, lg = run_tree(model, trees, max_gamma, kv)
    tol = LOGIT_TOL[kind]
    row = 0
    verdicts = []
    for r, (st, (tokens, parents)) in enumerate(zip(states, trees)):
        k_o, n_o, path_o, lo, nk, nv = spec.verify_tree(cfg, W, st, tokens, parents)
        n = len(tokens)
        err = np.abs(lg[row:row + n] - lo).max()
        assert err <= tol, (r, err)
        verdicts.append(classify_tree(lo, tokens, parents, acc[r], nxt[r], nodes[r]))
        k = int(acc[r])
        assert int(seq[r].item()) == st.length + k + 1
        path = [int(x) for x in nodes[r, :k + 1]]
        assert path[0] == 0 and all(parents[path[i]] == path[i - 1] for i in range(1, k + 1))
        pos = st.length + np.arange(k + 1)
        kv_tol = 1e-5 if kind == "f32" else 2 ** -7
        for l in range(shape["n_layers"]):
            gk = sd.read_positions(ks[l], table[r], pos, PAGE).float().cpu().numpy()
            gv = sd.read_positions(vs_[l], table[r], pos, PAGE).float().cpu().numpy()
            assert np.allclose(gk, nk[l][path], rtol=kv_tol, atol=kv_tol), (r, l)
            assert np.allclose(gv, nv[l][path], rtol=kv_tol, atol=kv_tol), (r, l)
        print(f"[tree {kind}] request {r}: {n} nodes, accepted {k} (oracle {k_o}), max |dlogit| {err:.2e}")
        row += n
    assert "mismatch" not in verdicts, verdicts
    assert verdicts.count("near_tie") <= 1
    assert acc.sum() >= 4
    model.close()


@pytest.mark.parametrize("kind", ["f32", "bf16"])
def test_chain_tree_equals_block_verify(kind):
    shape, cfg, W, wdev = setup(kind)
    states = states_for(kind, cfg, W, [50, 17])
    gamma = 10
    rng = np.random.default_rng(4)
    blocks = [[st.anchor] + [int(x) for x in rng.integers(0, cfg.vocab, size=gamma)] for st in states]
    cfgm = vs.make_config(shape, vs.SV_F32 if kind == "f32" else vs.SV_BF16, 2, gamma, 256, PAGE,
                          flags=vs.SV_FLAG_KEEP_LOGITS)
    outs = []
    for mode in ("block", "tree"):
        model = vs.Model(cfgm, wdev)
        ks, vs_, table, seq = build_kv(shape, states, PAGE, gamma, kind)
        kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
        tok = torch.tensor(blocks, dtype=torch.int32, device="cuda")
        acc = torch.zeros(2, dtype=torch.int32, device="cuda")
        nxt = torch.zeros(2, dtype=torch.int32, device="cuda")
        if mode == "block":
            model.verify(tok, [gamma, gamma], kv, acc, nxt)
        else:
            par = torch.tensor([[-1] + list(range(gamma))] * 2, dtype=torch.int32, device="cuda")
            nodes = torch.zeros((2, gamma + 1), dtype=torch.int32, device="cuda")
            model.verify_tree(tok, par, [gamma, gamma], kv, acc, nxt, nodes)
        outs.append((model.logits(2 * (gamma + 1)).cpu().numpy(), acc.cpu().numpy(), nxt.cpu().numpy(),
                     seq.cpu().numpy()))
        model.sync_status()
        model.close()
    assert np.array_equal(outs[0][0], outs[1][0])
    for a, b in zip(outs[0][1:], outs[1][1:]):
        assert np.array_equal(a, b)


def test_tree_token_forcing_12_steps():
    shape, cfg, W, wdev = setup("f32")
    (st,) = states_for("f32", cfg, W, [48])
    n_steps, n_nodes = 12, 16
    g_all = spec.ar_greedy(cfg, W, st, n_steps * n_nodes + 2).emitted[len(st.emitted):]
    model = vs.Model(vs.make_config(shape, vs.SV_F32, 1, n_nodes - 1, 48 + n_steps * n_nodes + 32, PAGE), wdev)
    ks, vs_, table, seq = build_kv(shape, [st], PAGE, n_steps * n_nodes, "f32")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    emitted, anchor = [], st.anchor
    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    nodes = torch.zeros((1, n_nodes), dtype=torch.int32, device="cuda")
    accepted = 0
    for step in range(n_steps):
        greedy = g_all[len(emitted):len(emitted) + 8]
        parents = synth.random_tree(n_nodes, 3, 80, step)
        tokens = synth.tree_drafts(parents, anchor, greedy, 0.8, cfg.vocab, 81, step)
        model.verify_tree(torch.from_numpy(np.asarray([tokens], np.int32)).cuda(),
                          torch.from_numpy(np.asarray([parents], np.int32)).cuda(), [n_nodes - 1], kv, acc, nxt,
                          nodes)
        k, n = int(acc.item()), int(nxt.item())
        path = nodes.cpu().numpy()[0, :k + 1]
        emitted += [int(tokens[i]) for i in path[1:]] + [n]
        accepted += k
        anchor = n
    model.sync_status()
    assert accepted > n_steps
    assert emitted == g_all[:len(emitted)]
    assert int(seq.item()) == st.length + len(emitted)
    model.close()


@pytest.mark.parametrize("kind", ["f32", "bf16"])
def test_bad_parent_is_a_device_check(kind):
    shape, cfg, W, wdev = setup(kind)
    states = states_for(kind, cfg, W, [20])
    model = vs.Model(vs.make_config(shape, vs.SV_F32 if kind == "f32" else vs.SV_BF16, 1, 7, 128, PAGE), wdev)
    ks, vs_, table, seq = build_kv(shape, states, PAGE, 7, kind)
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    tok = torch.tensor([[states[0].anchor, 1, 2, 3, 4, 5, 6, 7]], dtype=torch.int32, device="cuda")
    par = torch.tensor([[-1, 0, 0, 1, 5, 2, 3, 4]], dtype=torch.int32, device="cuda")   # node 4's parent is 5
    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    nodes = torch.zeros((1, 8), dtype=torch.int32, device="cuda")
    model.verify_tree(tok, par, [7], kv, acc, nxt, nodes)
    with pytest.raises(vs.SvError) as e:
        model.sync_status()
    assert e.value.status == vs.SV_ERR_DEVICE_CHECK
    with pytest.raises(vs.SvError):   # more than 64 nodes is refused on the host
        big = vs.Model(vs.make_config(shape, vs.SV_F32 if kind == "f32" else vs.SV_BF16, 1, 100, 256, PAGE), wdev)
        try:
            big.verify_tree(torch.zeros((1, 101), dtype=torch.int32, device="cuda"),
                            torch.zeros((1, 101), dtype=torch.int32, device="cuda"), [64], kv, acc, nxt,
                            torch.zeros((1, 101), dtype=torch.int32, device="cuda"))
        finally:
            big.close()
    model.close()
