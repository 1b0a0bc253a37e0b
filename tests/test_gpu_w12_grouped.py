"""Grouped W12 on the GPU (per-64-row-block bases plus escapes), through the C ABI.

  * device packing equals the oracle's format byte for byte (planes, bases,
    escape offsets and entries) on ragged tensors with zeros, subnormals,
    infinities and wide tails; every one of the 65536 patterns round-trips;
  * N(0, 0.02) weights at the 8B-class projection size round-trip exactly;
  * the matrix product with grouped W12 weights (tensor path, and the CUDA-core
    path at float32 activations) against float64 over the exact weights;
  * an 8B-shape model (2 layers, N(0, 0.02) weights with exact zeros) with
    grouped W12 matrices against the oracle's forward.
"""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import synth  # noqa: E402
import synth.device as sd  # noqa: E402
import verify_step_02_b300 as vs  # noqa: E402
from oracle import decoder, w12  # noqa: E402
from oracle.decoder import bf16_bits_to_f64  # noqa: E402

from helpers import LOGIT_TOL, DeviceContext, classify_greedy, device_oracle_weights, report_decisions  # noqa: E402

PAGE = 16


def normal_bits(shape, std, seed, zeros=0.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(shape, generator=g) * std).to(torch.bfloat16)
    bits = x.view(torch.int16).numpy().view(np.uint16).copy()
    if zeros:
        rng = np.random.default_rng(seed)
        bits[rng.random(shape) < zeros] = 0
    return bits


def gpu_pack(bits):
    return vs.pack_w12_grouped(sd.bits_to_bf16(bits))


@pytest.mark.parametrize("rows,cols,seed", [(150, 300, 1), (64, 128, 2), (1, 17, 3), (300, 1000, 4)])
def test_format_equals_oracle(rows, cols, seed):
    bits = normal_bits((rows, cols), 0.02, seed, zeros=0.01)
    bits[0, 0] = 0x7F80      # +inf
    bits[-1, -1] = 0x0003    # subnormal
    bits[rows // 2, cols // 3] = 0x3F80   # 1.0: widens its block's window
    planes, bases, off, esc = gpu_pack(bits)
    wp, wb, wo, we = w12.pack_grouped(bits)
    assert np.array_equal(planes.cpu().numpy().reshape(3, -1), wp)
    assert np.array_equal(bases.cpu().numpy(), wb)
    assert np.array_equal(off.cpu().numpy(), wo)
    assert np.array_equal(esc.cpu().numpy().view(np.uint32), we)
    back = vs.unpack_w12_grouped(planes, bases, off, esc, rows, cols)
    assert np.array_equal(sd.bf16_to_bits(back), bits)


def test_every_pattern_round_trips():
    rng = np.random.default_rng(0)
    bits = rng.permutation(np.arange(65536, dtype=np.uint32)).astype(np.uint16).reshape(256, 256)
    planes, bases, off, esc = gpu_pack(bits)
    assert np.array_equal(sd.bf16_to_bits(vs.unpack_w12_grouped(planes, bases, off, esc, 256, 256)), bits)


def test_normal_weights_at_projection_size():
    w = synth.device_bf16_normal((6144, 4096), 0.02, (5, 1), "cuda")
    planes, bases, off, esc = vs.pack_w12_grouped(w)
    back = vs.unpack_w12_grouped(planes, bases, off, esc, 6144, 4096)
    assert torch.equal(back.view(torch.int16), w.view(torch.int16))
    print(f"[w12 grouped] 6144 x 4096 N(0, 0.02): {esc.numel()} escapes ({esc.numel() / w.numel():.2e})")
    assert esc.numel() < 1e-3 * w.numel()


@pytest.mark.parametrize("m,n,k", [(17, 6144, 4096), (1, 4096, 4096), (187, 1280, 5120), (17, 24576, 4096)])
def test_linear_grouped_against_float64(m, n, k):
    rng = np.random.default_rng(m + n)
    bits = normal_bits((n, k), 0.02, n + k, zeros=0.002)
    w64 = bf16_bits_to_f64(bits)
    g = gpu_pack(bits)
    xf = torch.from_numpy(rng.standard_normal((m, k)).astype(np.float32)).cuda()
    hi = xf.to(torch.bfloat16)
    lo = (xf - hi.float()).to(torch.bfloat16)
    y, _ = vs.linear(vs.SV_W12, g, torch.stack([hi, lo]), n, k)
    x2 = (hi.double() + lo.double()).cpu().numpy()
    want = x2 @ w64.T
    scale = np.sqrt((np.abs(x2) ** 2) @ (np.abs(w64) ** 2).T) + 1e-30
    err = np.abs(y.cpu().numpy() - want) / scale
    assert err.max() < 1e-4, err.max()
    # the same product with the bf16 weights themselves
    yb, _ = vs.linear(vs.SV_BF16, sd.bits_to_bf16(bits), torch.stack([hi, lo]), n, k)
    assert (torch.abs(y - yb) / torch.from_numpy(scale).cuda()).max().item() < 1e-4


def test_model_8b_shapes_grouped_w12():
    shape = dict(synth.SHAPES["8b"], n_layers=2)
    C, gamma = 512, 16
    ms = synth.matrix_shapes(shape)
    d = shape["d_model"]
    ones = torch.ones(d, dtype=torch.bfloat16, device="cuda")

    def normal_dev(shp, seed):
        w = synth.device_bf16_normal(shp, 0.02, (seed, 0), "cuda")
        z = torch.rand(shp, generator=torch.Generator(device="cuda").manual_seed(seed), device="cuda") < 0.001
        return torch.where(z, torch.zeros_like(w), w)

    wbf = {"layers": [], "final_norm": ones,
           "embed": synth.device_bf16_normal((shape["vocab"], d), 0.02, (0, synth.T_EMBED), "cuda"),
           "lm_head": normal_dev((shape["vocab"], d), 9300)}
    for l in range(shape["n_layers"]):
        wbf["layers"].append(dict(attn_norm=ones, mlp_norm=ones,
                                  **{nm: normal_dev(ms[nm], 9200 + 10 * l + i)
                                     for i, nm in enumerate(("wqkv", "wo", "wgu", "wd"))}))
    wg = {"embed": wbf["embed"], "final_norm": ones, "lm_head": vs.pack_w12_grouped(wbf["lm_head"]),
          "layers": [dict(attn_norm=ones, mlp_norm=ones, **{nm: vs.pack_w12_grouped(lay[nm])
                                                            for nm in ("wqkv", "wo", "wgu", "wd")})
                     for lay in wbf["layers"]]}
    table, n_pages = synth.contiguous_page_table([C + gamma + 1], PAGE, (C + gamma + 1) // PAGE + 2)
    ks, vs_ = sd.kv_pools(shape, n_pages, PAGE, torch.bfloat16, fill="normal")
    seq = torch.tensor([C], dtype=torch.int32, device="cuda")
    kv = vs.KVCache(ks, vs_, torch.from_numpy(table).cuda(), seq)
    model = vs.Model(vs.make_config(shape, vs.SV_W12, 1, gamma, C + 64, PAGE, flags=vs.SV_FLAG_KEEP_LOGITS), wg)
    rng = np.random.default_rng(13)
    block = [int(x) for x in rng.integers(0, shape["vocab"], size=gamma + 1)]
    tok = torch.tensor([block], dtype=torch.int32, device="cuda")
    acc = torch.zeros(1, dtype=torch.int32, device="cuda")
    nxt = torch.zeros(1, dtype=torch.int32, device="cuda")
    model.verify(tok, [gamma], kv, acc, nxt)
    lg = model.logits(gamma + 1).cpu().numpy().astype(np.float64)
    model.sync_status()
    cfg, W = device_oracle_weights(shape, wbf)
    ctx = DeviceContext(ks, table[0], C, PAGE), DeviceContext(vs_, table[0], C, PAGE)
    lo, _, _ = decoder.forward_block(cfg, W, ctx[0], ctx[1], block, C, rowwise=False)
    err = np.abs(lg - lo).max()
    print(f"[w12 grouped 8b shapes] max |dlogit| {err:.4f}")
    assert err <= LOGIT_TOL["bf16"], err
    report_decisions("w12 grouped 8b shapes", [classify_greedy(lo, block[1:], acc[0], nxt[0])], 1)
    model.close()
