"""Acceptance rules of the verify step (test infrastructure; see the package docstring).

Block row j's logits z_j give the target's distribution for the token after
row j. With drafts d_1 .. d_L (d_i sits at row i):

Greedy (temperature 0; LFM2.5-DSpark post, "Quality parity" and "Usage";
DSpark summary, "Architecture", the E F accepted / G rejected / G* example):
  t_j = argmax_v z_j[v] (lowest index on ties); the accepted length k is the
  largest k <= L with d_i = t_{i-1} for all i <= k; the emitted token is t_k,
  the correction when k < L and the bonus when k = L.

Rejection sampling (temperature T > 0; DSpark summary, "Problem": the
longest prefix consistent with the target distribution is accepted, so the
output is distributed as the target's). The pages only name the scheme; this
is the standard rule (Leviathan et al., 2023):
  p_j = softmax(z_j / T); q_i is the distribution d_i was drawn from.
  for i = 1 .. L: accept d_i iff u_i * q_i(d_i) < p_{i-1}(d_i)
                  (u_i < min(1, p/q) for q > 0);
                  at the first rejection, emit a draw from
                  r = max(0, p_{i-1} - q_i) / sum(...) and stop.
  if all L are accepted, emit a draw from p_L.
  Draws use the inverse CDF in token-index order: the first v with
  cumsum(w)[v] > u' * sum(w).
Uniforms: u_i = U(seed, request, C+i, stream 0), u'_i = U(seed, request, C+i, stream 1),
where C+i is the absolute position of the emitted token (philox.uniform).
If r sums to zero (p_{i-1} = q_i, where rejection has probability zero) the
draw falls back to p_{i-1}.
"""
import numpy as np

from . import philox


def greedy_accept(logits, drafts):
    """logits [L+1, V], drafts [L] -> (accepted_len, next_token)."""
    t = np.argmax(np.asarray(logits), axis=-1)
    drafts = list(drafts)
    k = 0
    while k < len(drafts) and drafts[k] == t[k]:
        k += 1
    return k, int(t[k])


def greedy_accept_tree(logits, tokens, parents):
    """Greedy acceptance over a token tree (SpecPilot digest, "Reasons", names tree
    verification; the rule is the chain rule above applied along every root path).

    logits [n, V] per node, tokens [n] (node 0 = the anchor), parents [n]
    (parents[0] ignored, 0 <= parents[i] < i). With t_i = argmax z_i (lowest
    index on ties), node i's draft is correct when tokens[i] = t_{parent(i)};
    a node is accepted when it and every non-root ancestor are correct. The
    accepted path ends at the deepest accepted node (the lowest index among
    equally deep ones). Returns (accepted_len = its depth, next_token = t at
    its end, path = its nodes, root first).
    """
    z = np.asarray(logits)
    n = len(tokens)
    t = [int(np.argmax(z[i])) for i in range(n)]
    depth = [0] * n
    ok = [True] + [False] * (n - 1)
    for i in range(1, n):
        p = int(parents[i])
        depth[i] = depth[p] + 1
        ok[i] = ok[p] and int(tokens[i]) == t[p]
    end = 0
    for i in range(1, n):
        if ok[i] and depth[i] > depth[end]:
            end = i
    path = [end]
    while path[-1] != 0:
        path.append(int(parents[path[-1]]))
    return depth[end], t[end], path[::-1]


def softmax(z, temperature):
    s = np.asarray(z, dtype=np.float64) / temperature
    s = s - s.max(axis=-1, keepdims=True)
    e = np.exp(s)
    return e / e.sum(axis=-1, keepdims=True)


def inverse_cdf(w, u):
    """First index v with cumsum(w)[v] > u * sum(w); w >= 0, u in [0, 1)."""
    w = np.asarray(w, dtype=np.float64)
    cdf = np.cumsum(w)
    hit = np.nonzero(cdf > u * cdf[-1])[0]
    if hit.size:
        return int(hit[0])
    return int(np.nonzero(w > 0)[0][-1])


def sampled_accept(logits, drafts, q, temperature, u_acc, u_res):
    """logits [L+1, V]; drafts [L]; q [L, V]; u_acc [L]; u_res [L+1].

    Returns (accepted_len, next_token).
    """
    p = softmax(logits, temperature)
    q = np.asarray(q, dtype=np.float64)
    drafts = list(drafts)
    for i in range(1, len(drafts) + 1):
        d = drafts[i - 1]
        if u_acc[i - 1] * q[i - 1, d] < p[i - 1, d]:
            continue
        r = np.maximum(0.0, p[i - 1] - q[i - 1])
        if r.sum() <= 0.0:
            r = p[i - 1]
        return i - 1, inverse_cdf(r, u_res[i - 1])
    return len(drafts), inverse_cdf(p[len(drafts)], u_res[len(drafts)])


def sampled_accept_one_draft_batch(logits, drafts, q, temperature, u_acc, u_res0, u_res1):
    """sampled_accept for N independent one-draft blocks that share their target rows and q.

    logits [2, V] (rows 0 and 1 of every block); drafts [N]; q [V]; u_acc, u_res0,
    u_res1 [N] (the accept uniform, the residual draw's and the bonus draw's).
    The same rule as sampled_accept, applied to every block at once. Returns
    (accepted [N] in {0, 1}, next_token [N]).
    """
    p = softmax(logits, temperature)
    q = np.asarray(q, dtype=np.float64)
    d = np.asarray(drafts, dtype=np.int64)
    acc = np.asarray(u_acc) * q[d] < p[0, d]
    r = np.maximum(0.0, p[0] - q)
    if r.sum() <= 0.0:
        r = p[0]

    def draw(w, u):  # inverse_cdf for every u at once
        cdf = np.cumsum(w)
        v = np.searchsorted(cdf, np.asarray(u) * cdf[-1], side="right")
        return np.minimum(v, np.nonzero(w > 0)[0][-1])
    nxt = np.where(acc, draw(p[1], u_res1), draw(r, u_res0))
    return acc.astype(np.int64), nxt


def uniforms(seed, request_id, start_pos, n_drafts):
    """u_acc [L] and u_res [L+1] for a request whose anchor sits at start_pos."""
    pos = start_pos + np.arange(1, n_drafts + 2)
    u_acc = philox.uniform(seed, request_id, pos[:-1], 0)
    u_res = philox.uniform(seed, request_id, pos, 1)
    return u_acc, u_res
