"""sv_linear_noalloc, the allocation-free skinny product, against sv_linear (GPU, through the C ABI).

Callers that must not allocate device memory while they run (cudaMalloc can
synchronize the device; some hosts own every allocation) use this entry
point. Its split-K scratch is a 16 MiB static device array in the library,
shared by every call, so each case below calls it twice in a row to check
that the second call is not disturbed by what the first left behind.
"""
import ctypes

import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import synth  # noqa: E402
import synth.device as sd  # noqa: E402
import verify_step_02_b300 as vs  # noqa: E402

SCRATCH = 16 << 20


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


def test_noalloc_rejects_shapes_beyond_its_scratch():
    m, k = 32, 64
    for n_tiles in range(1, 4000):
        n = n_tiles * 128
        # the allocation-free product runs the CUDA-core plan for every weight type,
        # whose scratch is what sv_linear_workspace_bytes reports for float32 weights
        if vs.lib.sv_linear_workspace_bytes(vs.SV_F32, m, n, k) > SCRATCH:
            break
    else:
        pytest.skip("no shape on this GPU needs more than the static scratch")
    w = torch.zeros((n, k), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((m, k), dtype=torch.bfloat16, device="cuda")
    st, _ = noalloc(vs.SV_BF16, w, 0, x, n, k)
    assert st == vs.SV_ERR_INVALID_ARG
    assert b"static scratch" in vs.lib.sv_last_error()
