"""The C ABI library loads and exports every function include/sv.h declares (CPU only, no compute)."""
import ctypes
import os
import re
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sv.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sv_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    import verify_step_02_b300 as vs
    names = declared_functions()
    assert len(names) >= 15
    out = subprocess.run(["nm", "-D", "--defined-only", vs.LIB_PATH], capture_output=True, text=True, check=True)
    exported = set(re.findall(r" T (sv_\w+)", out.stdout))
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    for n in names:
        assert getattr(vs.lib, n) is not None


def test_host_side_argument_errors_need_no_gpu():
    import verify_step_02_b300 as vs
    assert vs.w12_plane_bytes(1, 1) == 4096 and vs.w12_plane_bytes(65, 129) == 4 * 4096
    assert vs.w12_plane_bytes(6144, 4096) == 96 * 32 * 4096 and vs.w12_plane_bytes(0, 5) == 0
    h = ctypes.c_void_p()
    st = vs.lib.sv_model_create(None, None, None, ctypes.byref(h))
    assert st == vs.SV_ERR_INVALID_ARG and b"NULL" in vs.lib.sv_last_error()
    cfg = vs.make_config(dict(n_layers=2, d_model=256, n_heads=4, n_kv_heads=3, head_dim=64, ffn=688, vocab=1024,
                              rope_theta=1e4), vs.SV_F32, 1, 4, 128)
    st = vs.lib.sv_model_create(ctypes.byref(cfg), None, None, ctypes.byref(h))
    assert st == vs.SV_ERR_INVALID_ARG and b"multiple" in vs.lib.sv_last_error()
    cfg.n_kv_heads, cfg.head_dim = 4, 96
    assert vs.lib.sv_model_create(ctypes.byref(cfg), None, None, ctypes.byref(h)) == vs.SV_ERR_UNSUPPORTED
    st = vs.lib.sv_verify(None, 1, None, None, None, None, 0.0, 0, None, None, None, None)
    assert st == vs.SV_ERR_INVALID_ARG
    assert vs.lib.sv_unpack_w12(None, 127, 1, 1, None, None) == vs.SV_ERR_INVALID_ARG


def test_tiny_positive_temperature_is_refused_on_the_host():
    """0 < T < 1e-6 would overflow z / T in float32; the call fails before it needs a model or a GPU."""
    import verify_step_02_b300 as vs
    for t in (1e-9, 9.9e-7, -1.0, float("nan"), float("inf")):
        st = vs.lib.sv_verify(None, 1, None, None, None, None, t, 0, None, None, None, None)
        assert st == vs.SV_ERR_INVALID_ARG and b"temperature" in vs.lib.sv_last_error(), t
        st = vs.lib.sv_verify_host(None, 1, None, None, None, None, t, 0, None, None, None, None)
        assert st == vs.SV_ERR_INVALID_ARG and b"temperature" in vs.lib.sv_last_error(), t
    for t in (0.0, 1e-6, 1.0):  # accepted temperatures reach the next check (the NULL model)
        st = vs.lib.sv_verify(None, 1, None, None, None, None, t, 0, None, None, None, None)
        assert st == vs.SV_ERR_INVALID_ARG and b"model is NULL" in vs.lib.sv_last_error(), t

