"""Decoder forward over one request's verify block, in float64.

Test infrastructure (see the package docstring).

What it computes (DSpark summary, "Architecture", the decode round with an
anchor): the target runs one forward over the block [anchor, d_1 .. d_L] at
absolute positions C .. C+L against the C cached positions; the logits of
block row j give the target's distribution for the token at row j+1.
The target is a Llama-style pre-norm decoder; the pages name no formulas, so
the plain textbook definitions are written out:

  h   = E[token]
  per layer:  u = RMSNorm(h) * g_attn
              q, k, v = u Wq^T, u Wk^T, u Wv^T       (W stored [out, in])
              q, k rotated by RoPE (rotate-half pairing i <-> i + hd/2)
              k, v rounded to the cache's storage type and appended
              o_j = softmax(q_j K^T / sqrt(hd)) V over keys 0 .. C+j
                    (query head i reads kv head i // (n_heads / n_kv_heads))
              h  += o Wo^T
              u   = RMSNorm(h) * g_mlp
              h  += (SiLU(u Wg^T) * (u Wu^T)) Wd^T
  z = (RMSNorm(h) * g_final) W_lm^T

RMSNorm(x) = x / sqrt(mean(x^2) + eps). SiLU(x) = x / (1 + e^-x).
RoPE at position p rotates the pair (x_i, x_{i+hd/2}) by p * theta^(-2i/hd).

A bf16 target (the pages' targets run in BF16, LFM2.5-DSpark post, "CPU &
GPU speed") has bf16 weights and a bf16 KV cache: every key and value is
rounded to the cache's storage type (ties to even) when it is stored. The
pages fix no activation precision; activations are not rounded here, so this
is the exact forward of the stored weights and cache.

With rowwise=True every block row goes through its own matrix-vector
products in a fixed order, so a row's logits are bit-identical whether it is
computed alone (autoregressive decoding) or inside a block: this is what
makes the oracle's speculative greedy output equal its AR greedy output
exactly (LFM2.5-DSpark post, "Quality parity").
"""
from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Config:
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    head_dim: int
    ffn: int
    vocab: int
    rope_theta: float
    rms_eps: float = 1e-6
    kv_dtype: str = "f32"      # storage type of the KV cache: "f32" or "bf16"


def bf16_bits_to_f64(bits):
    """Interpret uint16 bf16 patterns as numbers (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(np.float64)


def round_to_bf16(x):
    """Round float64 values to the nearest bf16 value, ties to even (normal range)."""
    x = np.asarray(x, dtype=np.float64)
    mant, expo = np.frexp(x)                 # x = mant * 2**expo, 0.5 <= |mant| < 1
    return np.ldexp(np.rint(np.ldexp(mant, 8)), expo - 8)


def f64_to_bf16_bits(x):
    """bf16 patterns of already-bf16-valued float64 numbers."""
    f = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def round_to_cache(x, kv_dtype):
    if kv_dtype == "bf16":
        return round_to_bf16(x)
    if kv_dtype == "f32":
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
    raise ValueError(kv_dtype)


def rmsnorm(x, g, eps):
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * g


def silu(x):
    return x / (1.0 + np.exp(-x))


def rope(x, positions, theta):
    """Rotate-half RoPE. x: [M, heads, hd]; positions: [M]."""
    hd = x.shape[-1]
    half = hd // 2
    inv_freq = theta ** (-2.0 * np.arange(half, dtype=np.float64) / hd)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * inv_freq[None, :]
    cos = np.cos(ang)[:, None, :]
    sin = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    return np.concatenate([x1 * cos - x2 * sin, x2 * cos + x1 * sin], axis=-1)


def attention_row(q, keys, vals):
    """Softmax attention of one query row. q [hq, hd]; keys, vals [T, hkv, hd]."""
    hq, hd = q.shape
    hkv = keys.shape[1]
    group = hq // hkv
    out = np.empty((hq, hd))
    for i in range(hq):
        kh = i // group
        s = keys[:, kh, :] @ q[i] / np.sqrt(hd)
        w = np.exp(s - s.max())
        out[i] = (w / w.sum()) @ vals[:, kh, :]
    return out


def linear(x, w, rowwise):
    """x [M, in] times w [out, in] transposed."""
    if rowwise:
        return np.stack([w @ x[m] for m in range(x.shape[0])]) if x.shape[0] else np.zeros((0, w.shape[0]))
    return x @ w.T


class DenseWeights:
    """Weights held in host memory (any float dtype, or bf16 as uint16 patterns).

    Matrices use the [out, in] layout. Per layer: attn_norm, wqkv (q rows, then
    k rows, then v rows), wo, mlp_norm, wgu (gate rows, then up rows), wd.
    Global: embed [V, d], final_norm [d], lm_head [V, d].
    """

    def __init__(self, cfg, layers, embed, final_norm, lm_head, bf16=False):
        self.cfg, self._layers, self._embed = cfg, layers, embed
        self._final_norm, self._lm_head, self._bf16 = final_norm, lm_head, bf16

    def _f64(self, a):
        return bf16_bits_to_f64(a) if self._bf16 else np.asarray(a, dtype=np.float64)

    def embed(self, tokens):
        return self._f64(self._embed[np.asarray(tokens, dtype=np.int64)])

    def layer(self, l):
        c = self.cfg
        raw = self._layers[l]
        nq, nkv = c.n_heads * c.head_dim, c.n_kv_heads * c.head_dim
        wqkv = self._f64(raw["wqkv"])
        wgu = self._f64(raw["wgu"])
        return {
            "attn_norm": self._f64(raw["attn_norm"]),
            "wq": wqkv[:nq], "wk": wqkv[nq:nq + nkv], "wv": wqkv[nq + nkv:nq + 2 * nkv],
            "wo": self._f64(raw["wo"]),
            "mlp_norm": self._f64(raw["mlp_norm"]),
            "wg": wgu[:c.ffn], "wu": wgu[c.ffn:2 * c.ffn],
            "wd": self._f64(raw["wd"]),
        }

    def final_norm(self):
        return self._f64(self._final_norm)

    def logits(self, x, rowwise, chunk=16384):
        out = np.empty((x.shape[0], self.cfg.vocab))
        for v0 in range(0, self.cfg.vocab, chunk):
            w = self._f64(self._lm_head[v0:v0 + chunk])
            out[:, v0:v0 + w.shape[0]] = linear(x, w, rowwise)
        return out


def forward_block(cfg, weights, ctx_k, ctx_v, tokens, start_pos, rowwise=True, layers_out=None):
    """Forward one request's block.

    ctx_k, ctx_v: per layer, the cached values [C, hkv, hd] (float64 holding
    values of the cache's storage type). tokens: the block, anchor first.
    Returns (logits [M, V], new_k, new_v) where new_k[l], new_v[l] are the
    block's keys/values [M, hkv, hd] as the cache stores them. If layers_out
    is a list, the residual stream after each layer is appended to it.
    """
    (out,) = forward_blocks(cfg, weights, [(ctx_k, ctx_v, tokens, start_pos)], rowwise, layers_out)
    return out


def tree_depths(parents):
    """Depth of every node of a token tree (node 0, the anchor, is the root at depth 0).

    parents[0] is ignored; every other node's parent precedes it (0 <= parents[i] < i).
    """
    depth = [0] * len(parents)
    for i in range(1, len(parents)):
        p = int(parents[i])
        if not 0 <= p < i:
            raise ValueError(f"node {i}: parent {p} must precede it")
        depth[i] = depth[p] + 1
    return depth


def tree_path(parents, i):
    """Nodes from the root to node i, root first."""
    path = [i]
    while path[-1] != 0:
        path.append(int(parents[path[-1]]))
    return path[::-1]


def forward_tree(cfg, weights, ctx_k, ctx_v, tokens, parents, start_pos, rowwise=True):
    """Forward one request's token tree (tree verification; SpecPilot digest, "Reasons").

    The pages name tree verification without spelling it out; this is the
    plain generalisation of the block forward: node i sits at position
    C + depth(i) and attends to the cached positions and to its own ancestors
    (root first, itself last), so each node computes exactly what the last
    row of a block forward over its root-to-node path computes. Returns
    (logits [n, V], new_k, new_v) indexed by node.
    """
    (out,) = forward_blocks(cfg, weights, [(ctx_k, ctx_v, tokens, start_pos, parents)], rowwise)
    return out


def forward_blocks(cfg, weights, requests, rowwise=True, layers_out=None):
    """forward_block for several independent requests, sharing each layer's weights.

    requests: list of (ctx_k, ctx_v, tokens, start_pos) or (ctx_k, ctx_v,
    tokens, start_pos, parents) for a token tree (see forward_tree); ctx_k /
    ctx_v only need to support indexing by layer. The layer loop is outermost
    so a layer's weights are fetched once; each request's arithmetic is
    exactly that of forward_block (requests never mix). Returns a list of
    (logits, new_k, new_v).
    """
    c = cfg
    state = []
    for req in requests:
        ctx_k, ctx_v, tokens, start_pos = req[:4]
        tokens = np.asarray(tokens, dtype=np.int64)
        m = tokens.shape[0]
        parents = req[4] if len(req) > 4 and req[4] is not None else [-1] + list(range(m - 1))
        depth = np.asarray(tree_depths(parents))
        # block rows row j attends to after the cached keys: its root-to-node path
        # (for a chain, rows 0 .. j)
        vis = [tree_path(parents, j) for j in range(m)]
        state.append({"m": m, "pos": start_pos + depth, "vis": vis, "h": weights.embed(tokens), "k": [], "v": [],
                      "ctx_k": ctx_k, "ctx_v": ctx_v})
    for l in range(c.n_layers):
        p = weights.layer(l)
        for st in state:
            m, pos, h = st["m"], st["pos"], st["h"]
            u = rmsnorm(h, p["attn_norm"], c.rms_eps)
            q = linear(u, p["wq"], rowwise).reshape(m, c.n_heads, c.head_dim)
            k = linear(u, p["wk"], rowwise).reshape(m, c.n_kv_heads, c.head_dim)
            v = linear(u, p["wv"], rowwise).reshape(m, c.n_kv_heads, c.head_dim)
            q = rope(q, pos, c.rope_theta)
            k = round_to_cache(rope(k, pos, c.rope_theta), c.kv_dtype)
            v = round_to_cache(v, c.kv_dtype)
            ck, cv = st["ctx_k"][l], st["ctx_v"][l]
            keys = np.concatenate([ck, k], axis=0)
            vals = np.concatenate([cv, v], axis=0)
            n_ctx = ck.shape[0]
            rows = [np.concatenate([np.arange(n_ctx), n_ctx + np.asarray(st["vis"][j])]) for j in range(m)]
            o = np.stack([attention_row(q[j], keys[rows[j]], vals[rows[j]]) for j in range(m)])
            o = o.reshape(m, c.n_heads * c.head_dim)
            h = h + linear(o, p["wo"], rowwise)
            u = rmsnorm(h, p["mlp_norm"], c.rms_eps)
            a = silu(linear(u, p["wg"], rowwise)) * linear(u, p["wu"], rowwise)
            h = h + linear(a, p["wd"], rowwise)
            st["h"] = h
            st["k"].append(k)
            st["v"].append(v)
        if layers_out is not None and len(state) == 1:
            layers_out.append(state[0]["h"].copy())
        del p
    out = []
    for st in state:
        hf = rmsnorm(st["h"], weights.final_norm(), c.rms_eps)
        out.append((weights.logits(hf, rowwise), st["k"], st["v"]))
    return out
