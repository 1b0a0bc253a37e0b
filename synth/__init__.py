"""Seeded synthetic inputs for the verify step (shared by the tests and the benchmark).

This module draws inputs only: model weights, KV contents, prompts, drafts,
confidences and page tables. It holds none of the verify step's arithmetic,
so the oracle and the CUDA path can both consume it without sharing code.
No checkpoint or benchmark dataset is used or imitated; every tensor is
random with the shapes of the pages' targets (an 8B-class and a 27B-class
dense decoder, SpecPilot digest "Reasons" and DSpark summary "Experiments").

Seeding: global seed 20261202; tensor t of layer l draws from the stream
(seed, l, t), so any one layer can be regenerated alone.
"""
import numpy as np

SEED = 20261202

# Model shapes of the five workloads. kv = n_kv_heads; theta = RoPE base.
SHAPES = {
    # tiny decoder: 2 layers, d 256, 4 heads x 64 (MHA), ffn 688, vocab 1024
    "tiny": dict(n_layers=2, d_model=256, n_heads=4, n_kv_heads=4, head_dim=64, ffn=688,
                 vocab=1024, rope_theta=1e4),
    # 8B-class: 36 layers, d 4096, 32 q / 8 kv heads x 128, ffn 12288, vocab 151936
    "8b": dict(n_layers=36, d_model=4096, n_heads=32, n_kv_heads=8, head_dim=128, ffn=12288,
               vocab=151936, rope_theta=1e6),
    # 27B-class: 64 layers, d 5120, 40 q / 8 kv heads x 128, ffn 17408, vocab 151936
    "27b": dict(n_layers=64, d_model=5120, n_heads=40, n_kv_heads=8, head_dim=128, ffn=17408,
                vocab=151936, rope_theta=1e6),
}

# tensor ids for the per-tensor seed streams
T_ATTN_NORM, T_WQKV, T_WO, T_MLP_NORM, T_WGU, T_WD = range(6)
T_EMBED, T_FINAL_NORM, T_LM_HEAD = 100, 101, 102
T_KV_K, T_KV_V = 200, 201


def rng(*stream):
    return np.random.default_rng([SEED, *[int(s) for s in stream]])


def torch_seed(*stream):
    """A 63-bit seed for torch generators, derived from a stream tuple."""
    ss = np.random.SeedSequence([SEED, *[int(s) for s in stream]])
    return int(ss.generate_state(2, dtype=np.uint64)[0] >> np.uint64(1))


def matrix_shapes(shape):
    s = shape
    nqkv = (s["n_heads"] + 2 * s["n_kv_heads"]) * s["head_dim"]
    return {
        "wqkv": (nqkv, s["d_model"]),
        "wo": (s["d_model"], s["n_heads"] * s["head_dim"]),
        "wgu": (2 * s["ffn"], s["d_model"]),
        "wd": (s["d_model"], s["ffn"]),
    }


def _tensor(kind, gen, shp, std):
    if kind == "f32":
        return (gen.standard_normal(shp) * std).astype(np.float32)
    if kind == "w12window":
        return w12_window_bits(gen, shp)
    raise ValueError(kind)


def w12_window_bits(gen, shp):
    """bf16 patterns with random sign, uniform 7-bit mantissa and exponent in [111, 126].

    Magnitudes lie in [2^-16, 1): a 16-binade window (the W12 workload).
    """
    s = gen.integers(0, 2, size=shp, dtype=np.int64)
    e = gen.integers(111, 127, size=shp, dtype=np.int64)
    m = gen.integers(0, 128, size=shp, dtype=np.int64)
    return ((s << 15) | (e << 7) | m).astype(np.uint16)


def host_weights(shape, kind="f32", std=0.02):
    """Host weights for small models.

    kind "f32": float32 N(0, std) matrices and embeddings, unit norm gains.
    kind "w12window": bf16 patterns (uint16) from w12_window_bits for every
    matrix and the embedding; unit gains (0x3f80).
    Returns dict(layers=[...], embed, final_norm, lm_head).
    """
    s = shape
    d = s["d_model"]
    ones = np.ones(d, np.float32) if kind == "f32" else np.full(d, 0x3F80, np.uint16)
    layers = []
    for l in range(s["n_layers"]):
        ms = matrix_shapes(s)
        layers.append({
            "attn_norm": ones.copy(),
            "wqkv": _tensor(kind, rng(l, T_WQKV), ms["wqkv"], std),
            "wo": _tensor(kind, rng(l, T_WO), ms["wo"], std),
            "mlp_norm": ones.copy(),
            "wgu": _tensor(kind, rng(l, T_WGU), ms["wgu"], std),
            "wd": _tensor(kind, rng(l, T_WD), ms["wd"], std),
        })
    return {
        "layers": layers,
        "embed": _tensor(kind, rng(0, T_EMBED), (s["vocab"], d), std),
        "final_norm": ones.copy(),
        "lm_head": _tensor(kind, rng(0, T_LM_HEAD), (s["vocab"], d), std),
    }


def device_bf16_normal(shp, std, stream, device):
    """bf16 N(0, std) tensor drawn on the device by torch's generator (large models)."""
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(torch_seed(*stream))
    t = torch.empty(shp, dtype=torch.bfloat16, device=device)
    t.normal_(0.0, std, generator=g)
    return t


def uniform_tokens(n, vocab, *stream):
    return rng(*stream).integers(0, vocab, size=n, dtype=np.int64)


def greedy_mix_drafts(greedy, gamma, p, vocab, *stream):
    """Draft i (0-based) is greedy[i] with probability p**(i+1), else a uniform token.

    greedy: the target's greedy continuation after the anchor (>= gamma tokens).
    """
    g = rng(*stream)
    keep = g.random(gamma) < p ** (np.arange(gamma) + 1)
    unif = g.integers(0, vocab, size=gamma)
    return np.where(keep, np.asarray(greedy[:gamma], dtype=np.int64), unif)


def random_tree(n_nodes, max_children, *stream):
    """Parents of a random token tree in topological order.

    Node 0 is the root (parent -1); node i > 0 picks its parent uniformly among
    the earlier nodes that have fewer than max_children children (1: a chain).
    """
    g = rng(*stream)
    parents, kids = [-1], [0]
    for i in range(1, n_nodes):
        open_ = [j for j in range(i) if kids[j] < max_children]
        p = int(open_[int(g.integers(0, len(open_)))])
        parents.append(p)
        kids[p] += 1
        kids.append(0)
    return np.asarray(parents, dtype=np.int32)


def tree_drafts(parents, anchor, greedy, p, vocab, *stream):
    """Node tokens for a tree: node 0 is the anchor; a node at depth d whose
    parent's path follows the greedy continuation takes greedy[d-1] with
    probability p, every other node a uniform token."""
    g = rng(*stream)
    tok, on, depth = [int(anchor)], [True], [0]
    for i in range(1, len(parents)):
        par = int(parents[i])
        d = depth[par] + 1
        depth.append(d)
        if on[par] and d <= len(greedy) and g.random() < p:
            t = int(greedy[d - 1])
        else:
            t = int(g.integers(0, vocab))
        tok.append(t)
        on.append(on[par] and d <= len(greedy) and t == int(greedy[d - 1]))
    return np.asarray(tok, dtype=np.int64)


def truncated_verify_lens(batch, gamma, threshold, *stream):
    """Per request: c_i ~ Beta(8, 2) i.i.d.; keep the drafts while prod_{j<=i} c_j >= threshold.

    L_r = max(1, #{i <= gamma : prod_{j <= i} c_j >= threshold}).
    """
    g = rng(*stream)
    c = g.beta(8.0, 2.0, size=(batch, gamma))
    surv = np.cumprod(c, axis=1)
    return np.maximum(1, (surv >= threshold).sum(axis=1)).astype(np.int32)


def shuffled_page_table(lengths, page_size, max_pages, *stream):
    """Pages for each request from one shuffled pool.

    lengths[r]: positions request r must be able to hold. Returns
    (page_table int32 [B, max_pages] padded with -1, n_pages).
    """
    need = [(int(n) + page_size - 1) // page_size for n in lengths]
    total = sum(need)
    perm = rng(*stream).permutation(total).astype(np.int32)
    table = np.full((len(lengths), max_pages), -1, np.int32)
    o = 0
    for r, n in enumerate(need):
        if n > max_pages:
            raise ValueError("request needs more pages than max_pages")
        table[r, :n] = perm[o:o + n]
        o += n
    return table, total


def contiguous_page_table(lengths, page_size, max_pages):
    need = [(int(n) + page_size - 1) // page_size for n in lengths]
    table = np.full((len(lengths), max_pages), -1, np.int32)
    o = 0
    for r, n in enumerate(need):
        table[r, :n] = np.arange(o, o + n, dtype=np.int32)
        o += n
    return table, o
