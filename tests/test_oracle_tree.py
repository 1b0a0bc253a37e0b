"""Pins for the oracle's token-tree verification (CPU only).

Tree verification (SpecPilot digest, "Reasons") runs the target once over a
tree of drafts rooted at the anchor: node i sits at position C + depth(i)
and sees the cached positions and its own ancestors. The pins:
  * every node's logits and keys/values are bit-identical to the last row of
    a block forward over its root-to-node path (the chain forward is pinned
    elsewhere by closed forms and the AR invariant);
  * leakage: changing a node that is not an ancestor leaves a node unchanged;
  * the acceptance rule on a chain is the chain rule;
  * brute force over every small tree and draft assignment against a
    lookup-table target: the accepted tokens are the longest prefix of the
    target's greedy continuation that some root path spells;
  * token forcing: the speculative tree loop emits exactly the tokens of
    plain autoregressive greedy decoding (LFM2.5-DSpark post, "Quality parity").
"""
import itertools

import numpy as np
import pytest

import synth
from oracle import accept, decoder, spec
from oracle.decoder import Config, DenseWeights


def tiny():
    cfg = Config(**synth.SHAPES["tiny"])
    w = synth.host_weights(synth.SHAPES["tiny"], "f32")
    return cfg, DenseWeights(cfg, w["layers"], w["embed"], w["final_norm"], w["lm_head"])


@pytest.fixture(scope="module")
def model():
    cfg, W = tiny()
    st, _, _, _ = spec.prefill(cfg, W, synth.uniform_tokens(20, cfg.vocab, 31, 0))
    return cfg, W, st


def test_depths_and_paths():
    parents = [-1, 0, 0, 1, 3, 2, 0]
    assert decoder.tree_depths(parents) == [0, 1, 1, 2, 3, 2, 1]
    assert decoder.tree_path(parents, 4) == [0, 1, 3, 4]
    assert decoder.tree_path(parents, 0) == [0]
    with pytest.raises(ValueError):
        decoder.tree_depths([-1, 0, 2])


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_node_equals_last_row_of_its_path(model, seed):
    cfg, W, st = model
    parents = synth.random_tree(11, 3, 40, seed)
    tokens = synth.uniform_tokens(11, cfg.vocab, 41, seed)
    tokens[0] = st.anchor
    lt, kt, vt = decoder.forward_tree(cfg, W, st.k, st.v, tokens, parents, st.length)
    for i in range(len(parents)):
        path = decoder.tree_path(parents, i)
        lb, kb, vb = decoder.forward_block(cfg, W, st.k, st.v, [tokens[j] for j in path], st.length)
        assert np.array_equal(lt[i], lb[-1]), i
        for l in range(cfg.n_layers):
            assert np.array_equal(kt[l][i], kb[l][-1]) and np.array_equal(vt[l][i], vb[l][-1])


def test_chain_tree_is_the_block(model):
    cfg, W, st = model
    tokens = [st.anchor, 5, 6, 7, 8]
    lt, _, _ = decoder.forward_tree(cfg, W, st.k, st.v, tokens, [-1, 0, 1, 2, 3], st.length)
    lb, _, _ = decoder.forward_block(cfg, W, st.k, st.v, tokens, st.length)
    assert np.array_equal(lt, lb)


def test_leakage_only_ancestors_matter(model):
    cfg, W, st = model
    parents = [-1, 0, 0, 1, 2, 3, 1]
    tokens = [st.anchor, 10, 11, 12, 13, 14, 15]
    base, _, _ = decoder.forward_tree(cfg, W, st.k, st.v, tokens, parents, st.length)
    for j in range(1, len(tokens)):
        t2 = list(tokens)
        t2[j] = 900 + j
        got, _, _ = decoder.forward_tree(cfg, W, st.k, st.v, t2, parents, st.length)
        for i in range(len(tokens)):
            if j in decoder.tree_path(parents, i):
                assert not np.array_equal(got[i], base[i]), (i, j)
            else:
                assert np.array_equal(got[i], base[i]), (i, j)


def test_accept_on_a_chain_is_the_chain_rule():
    g = np.random.default_rng(5)
    for _ in range(300):
        L = int(g.integers(0, 8))
        z = g.standard_normal((L + 1, 6))
        t = np.argmax(z, axis=1)
        drafts = [int(t[i]) if g.random() < 0.7 else int(g.integers(0, 6)) for i in range(L)]
        k, nxt = accept.greedy_accept(z, drafts)
        kt, nt, path = accept.greedy_accept_tree(z, [0] + drafts, [-1] + list(range(L)))
        assert (kt, nt, path) == (k, nxt, list(range(k + 1)))


def _target(V):
    """A deterministic lookup-table target: next token = f(prefix)."""
    def f(prefix):
        h = 7
        for x in prefix:
            h = (h * 31 + int(x) + 3) % 1009
        return h % V
    return f


def _all_parent_arrays(n):
    return [[-1] + list(ch) for ch in itertools.product(*[range(i) for i in range(1, n)])]


def test_accept_brute_force_small_trees():
    V = 3
    f = _target(V)
    anchor = 1
    cont = [anchor]
    for _ in range(6):
        cont.append(f(cont))
    g_cont = cont[1:]                         # the target's greedy continuation after the anchor
    cases = 0
    for n in range(1, 6):
        for parents in _all_parent_arrays(n):
            for drafts in itertools.product(range(V), repeat=n - 1):
                tokens = [anchor] + list(drafts)
                paths = [decoder.tree_path(parents, i) for i in range(n)]
                # logits of node i: one-hot on the target's next token after its path
                z = np.zeros((n, V))
                for i in range(n):
                    z[i, f([tokens[j] for j in paths[i]])] = 1.0
                k, nxt, path = accept.greedy_accept_tree(z, tokens, parents)
                # brute force: the deepest node whose path spells a prefix of the continuation
                match = [i for i in range(n) if [tokens[j] for j in paths[i][1:]] == g_cont[:len(paths[i]) - 1]]
                best = max(len(paths[i]) - 1 for i in match)
                end = min(i for i in match if len(paths[i]) - 1 == best)
                assert k == best and path == paths[end]
                assert [tokens[j] for j in path[1:]] + [nxt] == g_cont[:k + 1]
                cases += 1
    assert cases == 1 + 3 + 2 * 9 + 6 * 27 + 24 * 81


def test_spec_tree_loop_equals_ar_greedy(model):
    cfg, W, st0 = model
    n_steps = 5
    ar = spec.ar_greedy(cfg, W, st0, 40)

    def drafter(st):
        step = len(st.emitted)
        greedy = ar.emitted[step:step + 6]
        parents = synth.random_tree(9, 3, 50, step)
        return synth.tree_drafts(parents, st.anchor, greedy, 0.8, cfg.vocab, 51, step), parents

    out, lens = spec.spec_greedy_tree(cfg, W, st0, drafter, n_steps)
    n = len(out.emitted)
    assert n == n_steps + sum(lens) and sum(lens) > 0
    assert out.emitted == ar.emitted[:n]
    # the committed cache is the AR cache of the same tokens
    for l in range(cfg.n_layers):
        assert np.array_equal(out.k[l], ar.k[l][:out.length])
        assert np.array_equal(out.v[l], ar.v[l][:out.length])
