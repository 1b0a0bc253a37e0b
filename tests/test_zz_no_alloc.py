"""sv_linear_noalloc, the allocation-free skinny product, against sv_linear (GPU, through the C ABI).

Callers that must not allocate device memory while they run (cudaMalloc can
synchronize the device; some hosts own every allocation) use this entry
point. Its K splits meet in distributed shared memory within one cluster, so
it keeps no state between calls; each case below still calls it twice in a row
to check that the second call gives the same result.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import synth  # noqa: E402
import synth.device as sd  # noqa: E402
import verify_step_02_b300 as vs  # noqa: E402

def noalloc(wdtype, w, base, x, n, k):
    planes = 2 if x.dim() == 3 else 1
    m = int(x.shape[-2])
    y = torch.full((m, n), float("nan"), dtype=torch.float32, device="cuda")
    mat = vs.matrix(w) if isinstance(w, tuple) else vs.Matrix(w.data_ptr(), int(base))
    st = vs.lib.sv_linear_noalloc(int(wdtype), ctypes.byref(mat), n, k, ctypes.c_void_p(x.data_ptr()), planes, m,
                                  ctypes.c_void_p(y.data_ptr()),
                                  ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return st, y


def make(kind, m, n, k, rng):
    if kind == "f32":
        w = torch.from_numpy((rng.standard_normal((n, k)) * 0.02).astype(np.float32)).cuda()
        return vs.SV_F32, w, 0, torch.from_numpy(rng.standard_normal((m, k)).astype(np.float32)).cuda()
    bits = synth.w12_window_bits(rng, (n, k))
    w, base = sd.bits_to_bf16(bits), 0
    wd = vs.SV_BF16
    if kind == "w12":
        (w, base), wd = vs.pack_w12(w), vs.SV_W12
    if kind == "w12g":   # grouped W12 of N(0, 0.02) weights with exact zeros (escapes)
        wn = (torch.randn((n, k), generator=torch.Generator().manual_seed(n + k)) * 0.02).to(torch.bfloat16)
        wn[torch.rand((n, k), generator=torch.Generator().manual_seed(k)) < 0.01] = 0
        w, wd = vs.pack_w12_grouped(wn.cuda()), vs.SV_W12
    xf = torch.from_numpy(rng.standard_normal((m, k)).astype(np.float32)).cuda()
    hi = xf.to(torch.bfloat16)
    return wd, w, base, torch.stack([hi, (xf - hi.float()).to(torch.bfloat16)])


@pytest.mark.parametrize("kind,m,n,k", [("f32", 5, 688, 256), ("bf16", 17, 6144, 4096), ("bf16", 64, 4096, 12288),
                                        ("w12", 17, 1024, 256), ("w12", 256, 688, 256), ("w12g", 17, 1024, 512)])
def test_noalloc_matches_linear_twice(kind, m, n, k):
    rng = np.random.default_rng(m * 7 + n)
    wd, w, base, x = make(kind, m, n, k, rng)
    want, _ = vs.linear(wd, w, x, n, k, base=base)
    want = want.cpu().numpy().astype(np.float64)
    scale = np.abs(want).max() + 1e-30
    for _ in range(2):
        st, y = noalloc(wd, w, base, x, n, k)
        assert st == vs.SV_OK, vs.lib.sv_last_error()
        got = y.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert np.abs(got - want).max() / scale < 1e-5


def test_noalloc_wide_shape_and_overlapping_streams():
    # 65536 x 64 weights at 32 tokens: a shape whose split-K partials (2 splits x 512
    # tiles x 16 KB) would not have fit a fixed scratch; two calls on two streams
    # at once may overlap, since the calls share no state
    m, n, k = 32, 65536, 64
    rng = np.random.default_rng(65)
    wd, w, base, x = make("bf16", m, n, k, rng)
    want, _ = vs.linear(wd, w, x, n, k, base=base)
    want = want.cpu().numpy().astype(np.float64)
    scale = np.abs(want).max() + 1e-30
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    ys = []
    for s in (s1, s2):
        with torch.cuda.stream(s):
            st, y = noalloc(wd, w, base, x, n, k)
            assert st == vs.SV_OK, vs.lib.sv_last_error()
            ys.append(y)
    torch.cuda.synchronize()
    for y in ys:
        got = y.cpu().numpy().astype(np.float64)
        assert np.isfinite(got).all()
        assert np.abs(got - want).max() / scale < 1e-5
