"""GPU parity of the W12 codec, the Philox uniforms and the skinny GEMM (through the C ABI)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import synth  # noqa: E402
import synth.device as sd  # noqa: E402
import verify_step_02_b300 as vs  # noqa: E402
from oracle import philox, w12  # noqa: E402
from oracle.decoder import bf16_bits_to_f64  # noqa: E402


def test_w12_every_window_bit_exact():
    """All 2^16 patterns, grouped into every representable 16-binade window, pack to the
    oracle's planes and round-trip bit-exactly; tensors spanning more fail with the oracle's count."""
    allbits = np.arange(65536, dtype=np.uint16)
    e = (allbits.astype(np.int64) >> 7) & 0xFF
    for base in range(1, 240):
        sel = allbits[(e >= base) & (e <= base + 15)].reshape(64, 64)
        planes, b = vs.pack_w12(sd.bits_to_bf16(sel))
        want_planes, want_base = w12.pack(sel)
        assert b == want_base == base
        assert np.array_equal(planes.cpu().numpy(), want_planes)
        back = vs.unpack_w12(planes, b, 64, 64)
        assert np.array_equal(sd.bf16_to_bits(back), sel)
    full = allbits.reshape(256, 256)
    with pytest.raises(w12.NotRepresentable) as want:
        w12.pack(full)
    with pytest.raises(vs.SvError) as got:
        vs.pack_w12(sd.bits_to_bf16(full))
    assert got.value.status == vs.SV_ERR_NOT_REPRESENTABLE
    assert got.value.n_unrepresentable == want.value.args[0]


def test_w12_ragged_shapes_round_trip():
    for rows, cols in [(1, 16), (3, 40), (67, 688), (128, 1024), (5, 4097)]:
        bits = synth.w12_window_bits(np.random.default_rng(rows * cols), (rows, cols))
        planes, b = vs.pack_w12(sd.bits_to_bf16(bits))
        wp, wb = w12.pack(bits)
        assert b == wb and np.array_equal(planes.cpu().numpy(), wp)
        assert np.array_equal(sd.bf16_to_bits(vs.unpack_w12(planes, b, rows, cols)), bits)


@pytest.mark.parametrize("seed,req,pos,stream", [(0, 0, 0, 0), (20261202, 7, 4096, 1),
                                                  (0xFFFFFFFFFFFFFFFF, (1 << 40) + 3, (1 << 31) - 5, 0),
                                                  (12345, -1, 100, 1)])
def test_philox_bit_exact(seed, req, pos, stream):
    n = 4099
    got = vs.philox_uniform(seed, req, pos, stream, n).cpu().numpy().astype(np.float64)
    want = philox.uniform(seed, np.int64(req), np.arange(pos, pos + n) & 0xFFFFFFFF, stream)
    assert np.array_equal(got, want)


# (N, K) of the tiny decoder's projections: q/k/v (in one QKV matrix), o, gate, up, down, lm_head
TINY_SHAPES = [(256, 256), (256, 256), (256, 256), (256, 256), (688, 256), (688, 256), (256, 688), (1024, 256)]


def _weights(kind, n, k, rng):
    if kind == "f32":
        w = (rng.standard_normal((n, k)) * 0.02).astype(np.float32)
        return torch.from_numpy(w).cuda(), w.astype(np.float64), 0
    bits = synth.w12_window_bits(rng, (n, k))
    if kind == "bf16":
        return sd.bits_to_bf16(bits), bf16_bits_to_f64(bits), 0
    planes, base = vs.pack_w12(sd.bits_to_bf16(bits))
    return planes, bf16_bits_to_f64(bits), base


@pytest.mark.parametrize("kind", ["f32", "bf16", "w12"])
@pytest.mark.parametrize("m", [1, 4, 16, 17, 64, 256])
def test_linear_matches_float64(kind, m):
    rng = np.random.default_rng(m)
    wdtype = {"f32": vs.SV_F32, "bf16": vs.SV_BF16, "w12": vs.SV_W12}[kind]
    for n, k in sorted(set(TINY_SHAPES)):
        w_dev, w64, base = _weights(kind, n, k, rng)
        x = rng.standard_normal((m, k))
        if kind == "f32":
            x_dev = torch.from_numpy(x.astype(np.float32)).cuda()
            x64 = x.astype(np.float32).astype(np.float64)
        else:
            x_dev = torch.from_numpy(x).to(torch.bfloat16).cuda()
            x64 = x_dev.float().cpu().numpy().astype(np.float64)
        y, _ = vs.linear(wdtype, w_dev, x_dev, n, k, base=base)
        want = x64 @ w64.T
        scale = np.sqrt((np.abs(x64) ** 2) @ (np.abs(w64) ** 2).T) + 1e-30
        err = np.abs(y.cpu().numpy() - want) / scale
        assert err.max() < 1e-5, (n, k, err.max())
        if kind != "f32":   # activations as a hi/lo bf16 pair: the product uses hi + lo
            xf = torch.from_numpy(x.astype(np.float32)).cuda()
            hi = xf.to(torch.bfloat16)
            lo = (xf - hi.float()).to(torch.bfloat16)
            y2, _ = vs.linear(wdtype, w_dev, torch.stack([hi, lo]), n, k, base=base)
            x2 = (hi.double() + lo.double()).cpu().numpy()
            err2 = np.abs(y2.cpu().numpy() - x2 @ w64.T) / scale
            assert err2.max() < 1e-5, (n, k, err2.max())


@pytest.mark.parametrize("kind", ["bf16", "w12"])
@pytest.mark.parametrize("m,n,k", [(17, 6144, 4096), (17, 4096, 12288), (17, 24576, 4096), (64, 4096, 4096), (1, 4096, 4096), (33, 1000, 4096),
                                   (64, 1000, 4112), (187, 1280, 5120), (256, 512, 1024), (300, 384, 512)])
def test_linear_projection_shapes(kind, m, n, k):
    """The skinny product at the decoder's projection sizes: many tiles, K shared by several CTAs,
    ragged N and K, M beyond one 256-column accumulator; hi/lo pair activations as the verify
    step passes them; bf16 weights or W12 planes rebuilt in the kernel; against float64."""
    rng = np.random.default_rng(m * 131 + n)
    bits = synth.w12_window_bits(rng, (n, k))
    w_dev, w64 = sd.bits_to_bf16(bits), bf16_bits_to_f64(bits)
    wdtype, base = vs.SV_BF16, 0
    if kind == "w12":
        (w_dev, base), wdtype = vs.pack_w12(w_dev), vs.SV_W12
    xf = torch.from_numpy(rng.standard_normal((m, k)).astype(np.float32)).cuda()
    hi = xf.to(torch.bfloat16)
    lo = (xf - hi.float()).to(torch.bfloat16)
    y, ws = vs.linear(wdtype, w_dev, torch.stack([hi, lo]), n, k, base=base)
    x2 = (hi.double() + lo.double()).cpu().numpy()
    want = x2 @ w64.T
    scale = np.sqrt((np.abs(x2) ** 2) @ (np.abs(w64) ** 2).T) + 1e-30
    err = np.abs(y.cpu().numpy() - want) / scale
    # the tensor cores accumulate the 2K products (hi and lo) in float32 inside the MMA;
    # its rounding error grows with K, about 1e-5 of the scale at K = 4096. A wrong
    # operand offset, a dropped K block or a lost lo plane gives errors of order 1e-3 .. 1.
    assert err.max() < 1e-4, err.max()
    # a second call on the same workspace gives the same bits (fixed-order split-K sums)
    y2, _ = vs.linear(wdtype, w_dev, torch.stack([hi, lo]), n, k, base=base, workspace=ws)
    assert torch.equal(y, y2)


@pytest.mark.parametrize("splits", range(1, 9))
@pytest.mark.parametrize("m", [1, 5, 33])
def test_fma_linear_cluster_splits(splits, m):
    # one 128-row tile and K = 32 x splits: the CUDA-core product splits K into exactly
    # `splits` CTAs of one cluster (1: no cluster), whose partials meet in distributed
    # shared memory; against float64
    rng = np.random.default_rng(100 * splits + m)
    n, k = 128, 32 * splits
    w = rng.standard_normal((n, k)).astype(np.float32)
    x = rng.standard_normal((m, k)).astype(np.float32)
    y, _ = vs.linear(vs.SV_F32, torch.from_numpy(w).cuda(), torch.from_numpy(x).cuda(), n, k)
    want = x.astype(np.float64) @ w.astype(np.float64).T
    scale = np.sqrt((x.astype(np.float64) ** 2) @ (w.astype(np.float64) ** 2).T) + 1e-30
    err = np.abs(y.cpu().numpy() - want) / scale
    assert err.max() < 1e-5, err.max()
