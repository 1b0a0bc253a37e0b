"""Test glue: oracle-side references and GPU setup from the same seeded inputs."""
import numpy as np

import synth
import synth.device as sd
from oracle import accept, decoder, spec
from oracle.decoder import Config, DenseWeights

MARGIN = 0.1        # greedy: a decision may differ only where the oracle's top-1/top-2 gap is <= this
RATIO_TOL = 1e-3    # sampled: ... or where |u - p/q| <= this
CDF_TOL = 1e-5      # sampled draws: ... or where u * S lies within this fraction of S of a CDF step
LOGIT_TOL = {"f32": 1e-4, "bf16": 5e-2}


def oracle_config(shape, kind):
    return Config(**shape, kv_dtype="f32" if kind == "f32" else "bf16")


def oracle_weights(shape, hw, kind):
    cfg = oracle_config(shape, kind)
    return cfg, DenseWeights(cfg, hw["layers"], hw["embed"], hw["final_norm"], hw["lm_head"], bf16=(kind != "f32"))


def torch_dtype(kind):
    import torch
    return torch.float32 if kind == "f32" else torch.bfloat16


def build_kv(shape, states, page_size, max_gamma, kind, shuffled=True, extra_pages=0, stream_id=(7, 7)):
    """Device KV pools holding each oracle state's cache; returns (pools_k, pools_v, table, seq_len)."""
    import torch
    lengths = [st.length + max_gamma + 1 for st in states]
    max_pages = max((n + page_size - 1) // page_size for n in lengths) + 1
    if shuffled:
        table, n_pages = synth.shuffled_page_table(lengths, page_size, max_pages, *stream_id)
    else:
        table, n_pages = synth.contiguous_page_table(lengths, page_size, max_pages)
    ks, vs = sd.kv_pools(shape, n_pages + extra_pages, page_size, torch_dtype(kind), fill="zeros")
    for r, st in enumerate(states):
        if st.length == 0:
            continue
        pos = np.arange(st.length)
        for l in range(shape["n_layers"]):
            sd.write_positions(ks[l], table[r], pos, torch.from_numpy(st.k[l]), page_size)
            sd.write_positions(vs[l], table[r], pos, torch.from_numpy(st.v[l]), page_size)
    seq = torch.tensor([st.length for st in states], dtype=torch.int32, device="cuda")
    return ks, vs, table, seq


def top2_gap(z):
    t = np.partition(np.asarray(z), -2)[-2:]
    return float(t[1] - t[0])


def classify_greedy(logits, drafts, k_gpu, next_gpu):
    """'match', 'near_tie' or 'mismatch' for one request's greedy decision."""
    k_o, n_o = accept.greedy_accept(logits, drafts)
    if (k_o, n_o) == (int(k_gpu), int(next_gpu)):
        return "match"
    last = min(len(drafts), max(k_o, int(k_gpu)))
    if any(top2_gap(logits[j]) <= MARGIN for j in range(last + 1)):
        return "near_tie"
    return "mismatch"


def classify_tree(logits, tokens, parents, k_gpu, next_gpu, path_gpu):
    """'match', 'near_tie' or 'mismatch' for one request's greedy tree decision."""
    k_o, n_o, path_o = accept.greedy_accept_tree(logits, tokens, parents)
    if (k_o, n_o, path_o) == (int(k_gpu), int(next_gpu), [int(x) for x in path_gpu[:int(k_gpu) + 1]]):
        return "match"
    if any(top2_gap(logits[j]) <= MARGIN for j in range(len(tokens))):
        return "near_tie"
    return "mismatch"


def classify_sampled(logits, drafts, q, temperature, seed, req, start, k_gpu, next_gpu):
    u_acc, u_res = accept.uniforms(seed, req, start, len(drafts))
    k_o, n_o = accept.sampled_accept(logits, drafts, q, temperature, u_acc, u_res)
    if (k_o, n_o) == (int(k_gpu), int(next_gpu)):
        return "match"
    p = accept.softmax(logits, temperature)
    q = np.asarray(q, dtype=np.float64)
    for i in range(1, min(len(drafts), max(k_o, int(k_gpu)) + 1) + 1):
        d = drafts[i - 1]
        ratio = p[i - 1, d] / q[i - 1, d] if q[i - 1, d] > 0 else np.inf
        if abs(u_acc[i - 1] - ratio) <= RATIO_TOL:
            return "near_tie"
    if k_o == int(k_gpu):
        if k_o < len(drafts):
            w = np.maximum(0.0, p[k_o] - q[k_o])
            if w.sum() <= 0:
                w = p[k_o]
        else:
            w = p[k_o]
        cdf = np.cumsum(w)
        if np.min(np.abs(cdf - u_res[k_o] * cdf[-1])) <= CDF_TOL * cdf[-1]:
            return "near_tie"
    return "mismatch"


def report_decisions(name, verdicts, max_near_ties):
    """Print how many decisions matched the oracle and how many were near-ties; fail on any
    mismatch (a decision that differs where the oracle's margins were clear) or on more
    near-ties than `max_near_ties`."""
    n_match, n_tie = verdicts.count("match"), verdicts.count("near_tie")
    n_bad = len(verdicts) - n_match - n_tie
    print(f"[decisions] {name}: {len(verdicts)} compared, {n_match} identical, {n_tie} near-tie, {n_bad} mismatch")
    assert n_bad == 0, verdicts
    assert n_tie <= max_near_ties, verdicts


def engine_greedy_chain(model, kv, anchors, n, gamma):
    """n greedy tokens per request from the engine itself (one row per request per step), to
    build drafts that agree with the target for long prefixes; seq_len is restored after."""
    import torch
    b = len(anchors)
    seq0 = kv.seq_len.clone()
    tok = torch.zeros((b, gamma + 1), dtype=torch.int32, device="cuda")
    tok[:, 0] = torch.as_tensor(np.asarray(anchors, dtype=np.int32), device="cuda")
    acc = torch.zeros(b, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(b, dtype=torch.int32, device="cuda")
    out = []
    for _ in range(n):
        model.verify(tok, [0] * b, kv, acc, nxt)
        out.append(nxt.clone())
        tok[:, 0] = nxt
    model.sync_status()
    kv.seq_len.copy_(seq0)
    return torch.stack(out, 1).cpu().numpy()


class DeviceLayers:
    """Per-layer host copies (bf16 patterns) of device weights, fetched when the oracle asks."""

    def __init__(self, wdev):
        self.w = wdev

    def __getitem__(self, l):
        return {k: sd.bf16_to_bits(v) for k, v in self.w["layers"][l].items()}

    def __len__(self):
        return len(self.w["layers"])


class DeviceRows:
    """Row access (index array or slice) to a device bf16 matrix, as host bf16 patterns."""

    def __init__(self, t):
        self.t = t

    def __getitem__(self, idx):
        import torch
        if isinstance(idx, slice):
            return sd.bf16_to_bits(self.t[idx])
        return sd.bf16_to_bits(self.t[torch.as_tensor(np.asarray(idx), device=self.t.device)])


class DeviceContext:
    """ctx[l] = the first C cached positions of one request, layer l, as float64 [C, n_kv, hd]."""

    def __init__(self, pools, table_row, length, page_size):
        self.pools, self.row, self.n, self.page = pools, table_row, length, page_size

    def __getitem__(self, l):
        return sd.read_positions(self.pools[l], self.row, np.arange(self.n), self.page).float().cpu().numpy() \
            .astype(np.float64)


def device_oracle_weights(shape, wdev):
    cfg = oracle_config(shape, "bf16")
    return cfg, DenseWeights(cfg, DeviceLayers(wdev), DeviceRows(wdev["embed"]), sd.bf16_to_bits(wdev["final_norm"]),
                             DeviceRows(wdev["lm_head"]), bf16=True)
