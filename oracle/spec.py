"""Verify, commit, autoregressive greedy and the speculative loop (test infrastructure).

A request's state is its cache (per layer, [C, hkv, hd] keys and values), its
committed length C and its anchor, the last emitted token, whose KV is not
yet cached (DSpark summary, "Architecture": the target emits D, the anchor,
then verifies the drafts that follow it).

Verify runs the block [anchor, d_1 .. d_L], applies the acceptance rule and
commits the anchor plus the k accepted drafts: C grows by k + 1 and the
emitted token becomes the next anchor. Rows past the accepted prefix are
discarded.

Token forcing (SpecPilot digest, intro): the speculative loop's emitted
tokens are compared, one by one, with plain autoregressive greedy decoding.
"""
from dataclasses import dataclass, field

import numpy as np

from . import accept, decoder


@dataclass
class RequestState:
    k: list                      # per layer [C, hkv, hd]
    v: list
    anchor: int
    request_id: int = 0
    emitted: list = field(default_factory=list)

    @property
    def length(self):
        return self.k[0].shape[0]

    def copy(self):
        return RequestState([a.copy() for a in self.k], [a.copy() for a in self.v],
                            self.anchor, self.request_id, list(self.emitted))


def empty_state(cfg, anchor, request_id=0):
    z = np.zeros((0, cfg.n_kv_heads, cfg.head_dim))
    return RequestState([z.copy() for _ in range(cfg.n_layers)], [z.copy() for _ in range(cfg.n_layers)],
                        anchor, request_id)


def prefill(cfg, weights, tokens, rowwise=True):
    """Cache every token of a prompt but the last, which becomes the anchor.

    Returns the state and the greedy token after the prompt (the prompt's
    last row's argmax) — callers that want that token as the anchor call
    commit() with it.
    """
    st = empty_state(cfg, int(tokens[-1]))
    logits, nk, nv = decoder.forward_block(cfg, weights, st.k, st.v, tokens, 0, rowwise)
    st.k = [a[:-1] for a in nk]
    st.v = [a[:-1] for a in nv]
    return st, logits, nk, nv


def verify(cfg, weights, st, drafts, temperature=0.0, seed=0, q=None, rowwise=True):
    """One verify of one request. Returns (accepted_len, next_token, logits, new_k, new_v)."""
    drafts = [int(d) for d in drafts]
    block = [st.anchor] + drafts
    logits, nk, nv = decoder.forward_block(cfg, weights, st.k, st.v, block, st.length, rowwise)
    if temperature == 0.0:
        k, nxt = accept.greedy_accept(logits, drafts)
    else:
        u_acc, u_res = accept.uniforms(seed, st.request_id, st.length, len(drafts))
        k, nxt = accept.sampled_accept(logits, drafts, q, temperature, u_acc, u_res)
    return k, nxt, logits, nk, nv


def commit(st, drafts, new_k, new_v, accepted_len, next_token):
    """Append the anchor and the accepted drafts to the cache; the emitted token becomes the anchor."""
    n = accepted_len + 1
    st.k = [np.concatenate([a, b[:n]], axis=0) for a, b in zip(st.k, new_k)]
    st.v = [np.concatenate([a, b[:n]], axis=0) for a, b in zip(st.v, new_v)]
    st.emitted.extend([int(d) for d in drafts[:accepted_len]] + [int(next_token)])
    st.anchor = int(next_token)
    return st


def verify_tree(cfg, weights, st, tokens, parents, rowwise=True):
    """One greedy tree verify of one request: tokens[0] must be the anchor.

    Returns (accepted_len, next_token, path, logits, new_k, new_v) with the
    nodes' keys/values indexed by node.
    """
    if int(tokens[0]) != st.anchor:
        raise ValueError("node 0 must hold the anchor")
    logits, nk, nv = decoder.forward_tree(cfg, weights, st.k, st.v, tokens, parents, st.length, rowwise)
    k, nxt, path = accept.greedy_accept_tree(logits, tokens, parents)
    return k, nxt, path, logits, nk, nv


def commit_tree(st, tokens, path, new_k, new_v, next_token):
    """Append the accepted path's keys/values (root first: positions C .. C + k)."""
    st.k = [np.concatenate([a, b[path]], axis=0) for a, b in zip(st.k, new_k)]
    st.v = [np.concatenate([a, b[path]], axis=0) for a, b in zip(st.v, new_v)]
    st.emitted.extend([int(tokens[i]) for i in path[1:]] + [int(next_token)])
    st.anchor = int(next_token)
    return st


def spec_greedy_tree(cfg, weights, st, drafter, n_steps, rowwise=True):
    """Speculative greedy loop over token trees; drafter(state) returns (tokens, parents)."""
    st = st.copy()
    lens = []
    for _ in range(n_steps):
        tokens, parents = drafter(st)
        k, nxt, path, _, nk, nv = verify_tree(cfg, weights, st, tokens, parents, rowwise)
        commit_tree(st, tokens, path, nk, nv, nxt)
        lens.append(k)
    return st, lens


def ar_greedy(cfg, weights, st, n_tokens, rowwise=True):
    """Plain autoregressive greedy decoding: one row per step."""
    st = st.copy()
    for _ in range(n_tokens):
        k, nxt, _, nk, nv = verify(cfg, weights, st, [], 0.0, rowwise=rowwise)
        commit(st, [], nk, nv, k, nxt)
    return st


def spec_greedy(cfg, weights, st, drafter, n_steps, rowwise=True):
    """Speculative greedy loop; drafter(state) returns the draft list for a step."""
    st = st.copy()
    lens = []
    for _ in range(n_steps):
        drafts = list(drafter(st))
        k, nxt, _, nk, nv = verify(cfg, weights, st, drafts, 0.0, rowwise=rowwise)
        commit(st, drafts, nk, nv, k, nxt)
        lens.append(k)
    return st, lens
