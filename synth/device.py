"""Synthetic inputs as device tensors (torch), for the tests and the benchmark.

Like the rest of synth, this draws and places inputs only: weights, KV pool
contents and page tables. Nothing here computes any part of the verify step.
"""
import numpy as np

from . import (SHAPES, T_EMBED, T_FINAL_NORM, T_KV_K, T_KV_V, T_LM_HEAD, T_WD, T_WGU, T_WO, T_WQKV,
               device_bf16_normal, matrix_shapes, torch_seed)


def _torch():
    import torch
    return torch


def host_to_device_weights(hw, kind, device="cuda"):
    """Host weights from synth.host_weights -> dict of device tensors.

    kind "f32": float32 tensors. kind "bf16": the uint16 patterns viewed as bfloat16.
    """
    torch = _torch()

    def dev(a):
        a = np.ascontiguousarray(a)
        if kind == "bf16":
            return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)
        return torch.from_numpy(a).to(device)

    out = {k: dev(hw[k]) for k in ("embed", "final_norm", "lm_head")}
    out["layers"] = [{k: dev(v) for k, v in lay.items()} for lay in hw["layers"]]
    return out


def bits_to_bf16(bits, device="cuda"):
    """uint16 numpy bf16 patterns -> device bfloat16 tensor with the same bits."""
    torch = _torch()
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).to(device)


def bf16_to_bits(t):
    """device/host bfloat16 tensor -> uint16 numpy patterns."""
    torch = _torch()
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def random_bf16_model(shape, device="cuda", std=0.02):
    """bf16 N(0, std) matrices and embeddings drawn on the device; unit norm gains."""
    torch = _torch()
    d = shape["d_model"]
    ms = matrix_shapes(shape)
    ones = torch.ones(d, dtype=torch.bfloat16, device=device)
    layers = []
    for l in range(shape["n_layers"]):
        layers.append({
            "attn_norm": ones.clone(),
            "wqkv": device_bf16_normal(ms["wqkv"], std, (l, T_WQKV), device),
            "wo": device_bf16_normal(ms["wo"], std, (l, T_WO), device),
            "mlp_norm": ones.clone(),
            "wgu": device_bf16_normal(ms["wgu"], std, (l, T_WGU), device),
            "wd": device_bf16_normal(ms["wd"], std, (l, T_WD), device),
        })
    return {
        "layers": layers,
        "embed": device_bf16_normal((shape["vocab"], d), std, (0, T_EMBED), device),
        "final_norm": ones.clone(),
        "lm_head": device_bf16_normal((shape["vocab"], d), std, (0, T_LM_HEAD), device),
    }


def kv_pools(shape, n_pages, page_size, dtype, device="cuda", fill="zeros", std=1.0):
    """Per-layer K and V pools [n_pages, n_kv, page_size, head_dim].

    fill "zeros" or "normal" (N(0, std), drawn per layer from streams (l, T_KV_K/V)).
    """
    torch = _torch()
    shp = (n_pages, shape["n_kv_heads"], page_size, shape["head_dim"])
    ks, vs = [], []
    for l in range(shape["n_layers"]):
        if fill == "zeros":
            ks.append(torch.zeros(shp, dtype=dtype, device=device))
            vs.append(torch.zeros(shp, dtype=dtype, device=device))
        else:
            for lst, tid in ((ks, T_KV_K), (vs, T_KV_V)):
                g = torch.Generator(device=device)
                g.manual_seed(torch_seed(l, tid))
                t = torch.empty(shp, dtype=dtype, device=device)
                t.normal_(0.0, std, generator=g)
                lst.append(t)
    return ks, vs


def write_positions(pool, page_table_row, positions, values, page_size):
    """Place values [n, n_kv, head_dim] at absolute positions of one request."""
    torch = _torch()
    pos = np.asarray(positions)
    pages = np.asarray(page_table_row)[pos // page_size]
    slots = pos % page_size
    v = values if hasattr(values, "device") else torch.from_numpy(np.ascontiguousarray(values))
    pool[torch.as_tensor(pages, device=pool.device), :, torch.as_tensor(slots, device=pool.device), :] = \
        v.to(pool.device, pool.dtype)


def read_positions(pool, page_table_row, positions, page_size):
    """Values [n, n_kv, head_dim] at absolute positions of one request (a device tensor)."""
    torch = _torch()
    pos = np.asarray(positions)
    pages = np.asarray(page_table_row)[pos // page_size]
    slots = pos % page_size
    return pool[torch.as_tensor(pages, device=pool.device), :, torch.as_tensor(slots, device=pool.device), :]
