"""Python binding of libsv, the B300 verify step of speculative decoding.

Argument marshalling only: every step of the verify path runs in the CUDA
kernels of libsv.so (built by verify_step_02_b300.build). PyTorch supplies
device memory and streams. Importing this package loads the library and
raises ImportError when it has not been built; there is no fallback.
"""
import ctypes
import os

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libsv.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libsv.so is not built ({LIB_PATH}); run python {os.path.join(_HERE, 'build.py')}")
lib = ctypes.CDLL(LIB_PATH)

SV_OK, SV_ERR_INVALID_ARG, SV_ERR_NOT_REPRESENTABLE, SV_ERR_KV_CAPACITY = 0, 1, 2, 3
SV_ERR_OUT_OF_MEMORY, SV_ERR_CUDA, SV_ERR_DEVICE_CHECK, SV_ERR_UNSUPPORTED = 4, 5, 6, 7
SV_F32, SV_BF16, SV_W12 = 0, 1, 2
SV_FLAG_KEEP_LOGITS, SV_FLAG_NO_PDL, SV_FLAG_CUDA_CORE_GEMM = 1, 2, 4
TRACE_KINDS = {1: "gemm", 2: "attention", 3: "attn_merge"}
KERNEL_CLASSES = ("gemm", "attention", "norm", "lm_head", "accept")


class SvError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"sv status {status}: {msg}")
        self.status = status


class Config(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in
                ("n_layers", "d_model", "n_heads", "n_kv_heads", "head_dim", "ffn", "vocab")] + \
               [("rope_theta", ctypes.c_float), ("rms_eps", ctypes.c_float)] + \
               [(n, ctypes.c_int32) for n in
                ("weight_dtype", "max_batch", "max_gamma", "page_size", "max_seq_len", "flags")]


class Matrix(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("base", ctypes.c_int32), ("row_bases", ctypes.c_void_p),
                ("esc_off", ctypes.c_void_p), ("esc", ctypes.c_void_p)]


def matrix(x):
    """sv_matrix for a dense tensor, a W12 (planes, base) pair or a grouped W12
    (planes, row_bases, esc_off, esc) tuple."""
    if isinstance(x, tuple) and len(x) == 4:
        return Matrix(x[0].data_ptr(), 0, x[1].data_ptr(), x[2].data_ptr(), x[3].data_ptr() if x[3].numel() else None)
    if isinstance(x, tuple):
        return Matrix(x[0].data_ptr(), int(x[1]), None, None, None)
    return Matrix(x.data_ptr(), 0, None, None, None)


class LayerWeights(ctypes.Structure):
    _fields_ = [("attn_norm", ctypes.c_void_p), ("wqkv", Matrix), ("wo", Matrix),
                ("mlp_norm", ctypes.c_void_p), ("wgu", Matrix), ("wd", Matrix)]


class Weights(ctypes.Structure):
    _fields_ = [("embed", ctypes.c_void_p), ("final_norm", ctypes.c_void_p), ("lm_head", Matrix),
                ("layers", ctypes.POINTER(LayerWeights))]


class KV(ctypes.Structure):
    _fields_ = [("k", ctypes.POINTER(ctypes.c_void_p)), ("v", ctypes.POINTER(ctypes.c_void_p)),
                ("n_pages", ctypes.c_int32), ("page_table", ctypes.c_void_p),
                ("max_pages_per_seq", ctypes.c_int32), ("seq_len", ctypes.c_void_p)]


_vp, _i32, _i64, _u64, _f32, _sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint64,
                                    ctypes.c_float, ctypes.c_size_t)
_SIGS = {
    "sv_model_create": (_i32, [ctypes.POINTER(Config), ctypes.POINTER(Weights), _vp, ctypes.POINTER(_vp)]),
    "sv_model_destroy": (None, [_vp]),
    "sv_verify": (_i32, [_vp, _i32, _vp, _vp, ctypes.POINTER(KV), _vp, _f32, _u64, _vp, _vp, _vp, _vp]),
    "sv_verify_host": (_i32, [_vp, _i32, _vp, _vp, ctypes.POINTER(KV), _vp, _f32, _u64, _vp, _vp, _vp, _vp]),
    "sv_model_logits": (_i32, [_vp, _vp, _i32, _vp]),
    "sv_prefill": (_i32, [_vp, _i32, _vp, _vp, ctypes.POINTER(KV), _vp, _vp]),
    "sv_verify_tree": (_i32, [_vp, _i32, _vp, _vp, _vp, ctypes.POINTER(KV), _vp, _vp, _vp, _vp]),
    "sv_model_sync_status": (_i32, [_vp, _vp]),
    "sv_model_set_timing": (_i32, [_vp, _i32]),
    "sv_model_timing": (_i32, [_vp, _vp, _vp]),
    "sv_model_set_trace": (_i32, [_vp, _vp, _i64]),
    "sv_model_trace_launches": (_i32, [_vp, _vp, _i64, ctypes.POINTER(_i64)]),
    "sv_w12_plane_bytes": (_i64, [_i64, _i64]),
    "sv_pack_w12": (_i32, [_vp, _i64, _i64, _vp, ctypes.POINTER(_i32), ctypes.POINTER(_i64), _vp]),
    "sv_unpack_w12": (_i32, [_vp, _i32, _i64, _i64, _vp, _vp]),
    "sv_w12_row_blocks": (_i64, [_i64]),
    "sv_w12_tiles": (_i64, [_i64, _i64]),
    "sv_pack_w12_grouped": (_i32, [_vp, _i64, _i64, _vp, _vp, _vp, _vp, _i64, ctypes.POINTER(_i64), _vp]),
    "sv_unpack_w12_grouped": (_i32, [_vp, _vp, _vp, _vp, _i64, _i64, _vp, _vp]),
    "sv_linear_workspace_bytes": (_sz, [_i32, _i32, _i32, _i32]),
    "sv_linear": (_i32, [_i32, ctypes.POINTER(Matrix), _i32, _i32, _vp, _i32, _i32, _vp, _vp, _sz, _vp]),
    "sv_linear_noalloc": (_i32, [_i32, ctypes.POINTER(Matrix), _i32, _i32, _vp, _i32, _i32, _vp, _vp]),
    "sv_philox_uniform": (_i32, [_u64, _i64, _i64, _i32, _i32, _vp, _vp]),
    "sv_schedule_prefix": (_i32, [_i32, _i32, _vp, _vp, _i32, _i32, _vp, ctypes.POINTER(ctypes.c_double),
                                   ctypes.POINTER(ctypes.c_double)]),
    "sv_last_error": (ctypes.c_char_p, []),
}
for _name, (_res, _args) in _SIGS.items():
    _fn = getattr(lib, _name)
    _fn.restype, _fn.argtypes = _res, _args


def _check(status):
    if status != SV_OK:
        raise SvError(status, lib.sv_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def make_config(shape, weight_dtype, max_batch, max_gamma, max_seq_len, page_size=16, rms_eps=1e-6, flags=0):
    return Config(shape["n_layers"], shape["d_model"], shape["n_heads"], shape["n_kv_heads"], shape["head_dim"],
                  shape["ffn"], shape["vocab"], float(shape["rope_theta"]), float(rms_eps), int(weight_dtype),
                  int(max_batch), int(max_gamma), int(page_size), int(max_seq_len), int(flags))


class KVCache:
    """Paged KV pools (torch tensors [n_pages, n_kv, page_size, head_dim] per layer), page table, seq_len."""

    def __init__(self, k_pools, v_pools, page_table, seq_len):
        self.k_pools, self.v_pools = list(k_pools), list(v_pools)
        self.page_table, self.seq_len = page_table, seq_len
        n = len(self.k_pools)
        self._k = (ctypes.c_void_p * n)(*[t.data_ptr() for t in self.k_pools])
        self._v = (ctypes.c_void_p * n)(*[t.data_ptr() for t in self.v_pools])
        self.struct = KV(ctypes.cast(self._k, ctypes.POINTER(ctypes.c_void_p)),
                         ctypes.cast(self._v, ctypes.POINTER(ctypes.c_void_p)),
                         int(self.k_pools[0].shape[0]), page_table.data_ptr(), int(page_table.shape[1]),
                         seq_len.data_ptr())


class Model:
    """A verify engine over caller-owned device weights (kept referenced here).

    weights: dict with "layers" (list of dicts: attn_norm, wqkv, wo, mlp_norm, wgu, wd),
    "embed", "final_norm", "lm_head"; tensors on the current CUDA device. For W12
    models each matrix entry is a (planes_tensor, base) pair (pack_w12) or a
    grouped (planes, row_bases, esc_off, esc) tuple (pack_w12_grouped).
    """

    def __init__(self, config, weights, stream=None):
        self.config = config
        self._keep = weights

        mat = matrix

        layers = weights["layers"]
        self._layers = (LayerWeights * len(layers))(*[
            LayerWeights(l["attn_norm"].data_ptr(), mat(l["wqkv"]), mat(l["wo"]), l["mlp_norm"].data_ptr(),
                         mat(l["wgu"]), mat(l["wd"])) for l in layers])
        self._w = Weights(weights["embed"].data_ptr(), weights["final_norm"].data_ptr(), mat(weights["lm_head"]),
                          ctypes.cast(self._layers, ctypes.POINTER(LayerWeights)))
        h = ctypes.c_void_p()
        _check(lib.sv_model_create(ctypes.byref(config), ctypes.byref(self._w), _stream(stream), ctypes.byref(h)))
        self.handle = h

    def close(self):
        if getattr(self, "handle", None):
            lib.sv_model_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def verify(self, tokens, verify_lens, kv, accepted_len, next_token, draft_probs=None, temperature=0.0,
               seed=0, request_ids=None, stream=None):
        """tokens, draft_probs, request_ids, accepted_len, next_token: device tensors; verify_lens: host ints."""
        lens = np.ascontiguousarray(np.asarray(verify_lens, dtype=np.int32))
        _check(lib.sv_verify(self.handle, len(lens), _ptr(tokens), lens.ctypes.data_as(ctypes.c_void_p),
                             ctypes.byref(kv.struct), _ptr(draft_probs), float(temperature), int(seed),
                             _ptr(request_ids), _ptr(accepted_len), _ptr(next_token), _stream(stream)))

    def prefill(self, tokens, block_lens, kv, next_token, stream=None):
        """Forward and commit every row of the blocks; next_token (device) = greedy token after each block."""
        lens = np.ascontiguousarray(np.asarray(block_lens, dtype=np.int32))
        _check(lib.sv_prefill(self.handle, len(lens), _ptr(tokens), lens.ctypes.data_as(ctypes.c_void_p),
                              ctypes.byref(kv.struct), _ptr(next_token), _stream(stream)))

    def verify_tree(self, tokens, parents, n_drafts, kv, accepted_len, next_token, accepted_nodes, stream=None):
        """Greedy token-tree verify: tokens, parents, outputs device tensors; n_drafts host ints."""
        n = np.ascontiguousarray(np.asarray(n_drafts, dtype=np.int32))
        _check(lib.sv_verify_tree(self.handle, len(n), _ptr(tokens), _ptr(parents), n.ctypes.data_as(ctypes.c_void_p),
                                  ctypes.byref(kv.struct), _ptr(accepted_len), _ptr(next_token),
                                  _ptr(accepted_nodes), _stream(stream)))

    def verify_host(self, tokens, verify_lens, kv, draft_probs=None, temperature=0.0, seed=0, request_ids=None,
                    stream=None, out=None):
        """Host-memory inputs and outputs (numpy or pinned torch CPU tensors); synchronizes."""
        lens = np.ascontiguousarray(np.asarray(verify_lens, dtype=np.int32))
        b = len(lens)
        if out is None:
            out = (np.zeros(b, np.int32), np.zeros(b, np.int32))

        def hp(a):
            if a is None:
                return None
            if hasattr(a, "data_ptr"):
                return ctypes.c_void_p(a.data_ptr())
            return a.ctypes.data_as(ctypes.c_void_p)

        _check(lib.sv_verify_host(self.handle, b, hp(tokens), lens.ctypes.data_as(ctypes.c_void_p),
                                  ctypes.byref(kv.struct), hp(draft_probs), float(temperature), int(seed),
                                  hp(request_ids), hp(out[0]), hp(out[1]), _stream(stream)))
        return out

    def logits(self, rows, stream=None):
        import torch
        out = torch.empty((rows, self.config.vocab), dtype=torch.float32, device="cuda")
        _check(lib.sv_model_logits(self.handle, _ptr(out), int(rows), _stream(stream)))
        return out

    def sync_status(self, stream=None):
        _check(lib.sv_model_sync_status(self.handle, _stream(stream)))

    def set_timing(self, enable):
        _check(lib.sv_model_set_timing(self.handle, int(bool(enable))))

    def timing(self):
        ms = (ctypes.c_double * 5)()
        n = (ctypes.c_int64 * 5)()
        _check(lib.sv_model_timing(self.handle, ms, n))
        return {k: (ms[i], n[i]) for i, k in enumerate(KERNEL_CLASSES)}

    def set_trace(self, records):
        """records: zero-filled device 64-bit tensor [capacity, 16], or None to stop tracing."""
        if records is None:
            _check(lib.sv_model_set_trace(self.handle, None, 0))
        else:
            _check(lib.sv_model_set_trace(self.handle, _ptr(records), int(records.shape[0])))

    def trace_launches(self):
        """[(first record, CTAs, kind name)] of the traced launches, in launch order."""
        n = ctypes.c_int64()
        _check(lib.sv_model_trace_launches(self.handle, None, 0, ctypes.byref(n)))
        buf = (ctypes.c_int64 * max(1, 3 * n.value))()
        _check(lib.sv_model_trace_launches(self.handle, buf, n.value, ctypes.byref(n)))
        return [(buf[3 * i], buf[3 * i + 1], TRACE_KINDS.get(buf[3 * i + 2], str(buf[3 * i + 2])))
                for i in range(n.value)]


def w12_plane_bytes(rows, cols):
    return int(lib.sv_w12_plane_bytes(int(rows), int(cols)))


def pack_w12(bf16, stream=None):
    """bf16 device tensor [rows, cols] -> (uint8 planes [3, plane_bytes], base). Raises SvError."""
    import torch
    rows, cols = bf16.shape
    planes = torch.empty((3, w12_plane_bytes(rows, cols)), dtype=torch.uint8, device=bf16.device)
    base, bad = ctypes.c_int32(), ctypes.c_int64()
    st = lib.sv_pack_w12(_ptr(bf16), rows, cols, _ptr(planes), ctypes.byref(base), ctypes.byref(bad),
                         _stream(stream))
    if st != SV_OK:
        err = SvError(st, lib.sv_last_error().decode())
        err.n_unrepresentable = bad.value
        raise err
    return planes, base.value


def pack_w12_grouped(bf16, stream=None):
    """bf16 device tensor [rows, cols] -> grouped W12 (planes [3, plane_bytes], row_bases, esc_off, esc)."""
    import torch
    rows, cols = bf16.shape
    dev = bf16.device
    planes = torch.empty((3, w12_plane_bytes(rows, cols)), dtype=torch.uint8, device=dev)
    bases = torch.empty(int(lib.sv_w12_row_blocks(rows)), dtype=torch.uint8, device=dev)
    off = torch.empty(int(lib.sv_w12_tiles(rows, cols)) + 1, dtype=torch.int32, device=dev)
    n = ctypes.c_int64()
    _check(lib.sv_pack_w12_grouped(_ptr(bf16), rows, cols, _ptr(planes), _ptr(bases), _ptr(off), None, 0,
                                   ctypes.byref(n), _stream(stream)))
    esc = torch.empty(max(n.value, 1), dtype=torch.int32, device=dev)
    if n.value:
        _check(lib.sv_pack_w12_grouped(_ptr(bf16), rows, cols, _ptr(planes), _ptr(bases), _ptr(off), _ptr(esc),
                                       n.value, ctypes.byref(n), _stream(stream)))
    return planes, bases, off, esc[:n.value]


def unpack_w12_grouped(planes, bases, off, esc, rows, cols, stream=None):
    import torch
    out = torch.empty((rows, cols), dtype=torch.bfloat16, device=planes.device)
    _check(lib.sv_unpack_w12_grouped(_ptr(planes), _ptr(bases), _ptr(off), _ptr(esc) if esc.numel() else None,
                                     rows, cols, _ptr(out), _stream(stream)))
    return out


def unpack_w12(planes, base, rows, cols, stream=None):
    import torch
    out = torch.empty((rows, cols), dtype=torch.bfloat16, device=planes.device)
    _check(lib.sv_unpack_w12(_ptr(planes), int(base), rows, cols, _ptr(out), _stream(stream)))
    return out


def linear(wdtype, w, x, n, k, base=0, stream=None, workspace=None):
    """y = x W^T with the verify step's GEMM kernels. Returns (y float32 [M, n], workspace).

    x: float32 [M, k] for float32 weights; bf16 [M, k], or a hi/lo pair [2, M, k], otherwise.
    """
    import torch
    planes = 2 if x.dim() == 3 else 1
    m = int(x.shape[-2])
    need = int(lib.sv_linear_workspace_bytes(int(wdtype), m, int(n), int(k)))
    if workspace is None or workspace.numel() < need:
        workspace = torch.zeros(max(need, 256), dtype=torch.uint8, device=x.device)
    y = torch.empty((m, n), dtype=torch.float32, device=x.device)
    mat = matrix(w) if isinstance(w, tuple) else Matrix(w.data_ptr(), int(base), None, None, None)
    _check(lib.sv_linear(int(wdtype), ctypes.byref(mat), int(n), int(k), _ptr(x), planes, m, _ptr(y),
                         _ptr(workspace), workspace.numel(), _stream(stream)))
    return y, workspace


def philox_uniform(seed, request_id, position0, stream_id, n, stream=None):
    import torch
    out = torch.empty(n, dtype=torch.float32, device="cuda")
    _check(lib.sv_philox_uniform(int(seed), int(request_id), int(position0), int(stream_id), int(n), _ptr(out),
                                 _stream(stream)))
    return out


def schedule_prefix(conf, step_us, early_stop=False):
    """Verify lengths maximizing expected tokens / step time (host only).

    conf: [B, gamma] draft confidences; step_us: step time for M = 1 .. len(step_us) rows.
    Returns (lens int32 [B], expected tokens, throughput in tokens/s).
    """
    c = np.ascontiguousarray(np.asarray(conf, dtype=np.float32))
    t = np.ascontiguousarray(np.asarray(step_us, dtype=np.float32))
    b, g = c.shape
    lens = np.zeros(b, np.int32)
    tau, th = ctypes.c_double(), ctypes.c_double()
    _check(lib.sv_schedule_prefix(b, g, c.ctypes.data_as(ctypes.c_void_p), t.ctypes.data_as(ctypes.c_void_p), len(t),
                                  int(bool(early_stop)), lens.ctypes.data_as(ctypes.c_void_p), ctypes.byref(tau),
                                  ctypes.byref(th)))
    return lens, tau.value, th.value

