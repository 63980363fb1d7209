"""Python binding of libtpmlp.so, the GB300 tensor-parallel MLP library.

Argument marshalling only: every function here forwards torch tensors' device pointers and
the current CUDA stream to the C entry point of the same name (see include/tp_mlp.h); every
step of the computation runs in the library's sm_103a kernels. There is no fallback: if the
shared library is missing, importing the binding raises, and the entry points refuse to run
on anything but an sm_103 device.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

__all__ = [
    "TP_F32", "TP_BF16", "TP_ACT_NONE", "TP_ACT_GELU_ERF", "TP_REDUCE_FUSED",
    "TP_REDUCE_PARTIALS", "TP_REDUCE_AUTO", "TP_REDUCE_PARTIALS_BF16", "TP_REDUCE_OVERLAP",
    "TP_COLUMN", "TP_ROW", "TpError", "MlpDesc", "LinearDesc", "lib",
    "library_path", "tp_version", "tp_last_error", "tp_mlp_workspace_size",
    "tp_linear_workspace_size", "tp_workspace_init", "tp_check_status", "tp_mlp_forward",
    "tp_mlp_backward", "tp_linear_column_forward", "tp_linear_column_backward",
    "tp_linear_row_forward", "tp_linear_row_backward", "tp_selftest_wait_timeout",
    "new_workspace", "EXPORTED_SYMBOLS", "tp_trace_start", "tp_trace_stop", "TraceRecord",
    "KERNEL_NAMES", "TAG_NAMES", "tp_linear_row_forward_noalloc", "tp_mlp_sp_workspace_size",
    "tp_mlp_forward_sp", "tp_mlp_backward_sp", "LayerNormDesc", "tp_layernorm_forward",
    "tp_layernorm_backward", "TUNE_KNOBS", "TP_TUNE_AUTO", "tp_tuning_set", "tp_tuning_get",
    "tuning",
]

TP_F32, TP_BF16 = 0, 1
TP_ACT_NONE, TP_ACT_GELU_ERF = 0, 1
TP_REDUCE_FUSED, TP_REDUCE_PARTIALS, TP_REDUCE_AUTO, TP_REDUCE_PARTIALS_BF16, TP_REDUCE_OVERLAP = 0, 1, 2, 3, 4
TP_COLUMN, TP_ROW = 0, 1
TP_BF16_TAIL_SCRATCH_BYTES = 80 * 256 * 256 * 4 + 4096

STATUS_NAMES = {
    0: "TP_OK", 1: "TP_ERR_NULL", 2: "TP_ERR_SHAPE", 3: "TP_ERR_INDIVISIBLE",
    4: "TP_ERR_ALIGN", 5: "TP_ERR_DTYPE", 6: "TP_ERR_WORKSPACE", 7: "TP_ERR_ARCH",
    8: "TP_ERR_CUDA", 9: "TP_ERR_DEVICE_TIMEOUT",
}

EXPORTED_SYMBOLS = (
    "tp_version", "tp_last_error", "tp_mlp_workspace_size", "tp_linear_workspace_size",
    "tp_workspace_init", "tp_check_status", "tp_mlp_forward", "tp_mlp_backward",
    "tp_linear_column_forward", "tp_linear_column_backward", "tp_linear_row_forward",
    "tp_linear_row_backward", "tp_selftest_wait_timeout", "tp_trace_start", "tp_trace_stop",
    "tp_linear_row_forward_noalloc", "tp_mlp_sp_workspace_size", "tp_mlp_forward_sp",
    "tp_mlp_backward_sp", "tp_layernorm_forward", "tp_layernorm_backward", "tp_tuning_set",
    "tp_tuning_get",
)

# Test and measurement hook (include/tp_mlp_tuning.h): overrides of the library's measured
# kernel choices, process-wide; TP_TUNE_AUTO gives a choice back to the library.
TP_TUNE_AUTO = -1
TUNE_KNOBS = {
    "gemm_pair": 0, "epi_warps": 1, "raster": 2, "tma_3d": 3, "split_loads": 4,
    "mma_probe": 5, "load_probe": 6, "tail_split": 7, "tail_waves": 8, "shard_split": 9,
    "simt_split": 10, "ln_reg": 11, "pdl": 12, "stage_blocks": 13, "tail_pieces": 14, "few_rows": 15,
    "dual": 16,
}

_HERE = os.path.dirname(os.path.abspath(__file__))


def library_path() -> str:
    return os.environ.get("TPMLP_LIBRARY", os.path.join(_HERE, "libtpmlp.so"))


class TpError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{self.name}: {message}")


class MlpDesc(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_int64), ("hidden", ctypes.c_int64), ("ffn", ctypes.c_int64),
                ("tp_degree", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("act", ctypes.c_int32), ("reduce", ctypes.c_int32)]


class LayerNormDesc(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_int64), ("hidden", ctypes.c_int64),
                ("tp_degree", ctypes.c_int32), ("dtype", ctypes.c_int32),
                ("eps", ctypes.c_float)]


class LinearDesc(ctypes.Structure):
    _fields_ = [("tokens", ctypes.c_int64), ("in_features", ctypes.c_int64),
                ("out_features", ctypes.c_int64), ("tp_degree", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("act", ctypes.c_int32),
                ("reduce", ctypes.c_int32), ("gather", ctypes.c_int32)]


class TraceRecord(ctypes.Structure):
    _fields_ = [("kernel", ctypes.c_int32), ("tag", ctypes.c_int32), ("flops", ctypes.c_double),
                ("bytes", ctypes.c_double), ("ms", ctypes.c_float), ("groups", ctypes.c_int32)]


KERNEL_NAMES = {1: "gemm_tc", 2: "gemm_ffma", 3: "shard_reduce", 4: "colsum", 5: "dact",
                6: "selftest", 7: "shard_copy", 8: "layernorm", 9: "ln_param_grad"}
TAG_NAMES = {1: "column_fwd", 2: "row_fwd", 3: "row_dgrad", 4: "row_wgrad", 5: "column_wgrad",
             6: "column_dgrad", 7: "reduce", 8: "bias_grad", 9: "act_grad", 10: "other",
             11: "sp_gather", 12: "sp_scatter", 13: "ln_fwd", 14: "ln_dgrad",
             15: "ln_param_grad", 16: "row_grads", 17: "column_grads"}

_P = ctypes.c_void_p
_PP = ctypes.POINTER(ctypes.c_void_p)
_SIGS = {
    "tp_version": (ctypes.c_int32, []),
    "tp_last_error": (ctypes.c_char_p, []),
    "tp_mlp_workspace_size": (ctypes.c_int, [ctypes.POINTER(MlpDesc), ctypes.POINTER(ctypes.c_size_t)]),
    "tp_linear_workspace_size": (ctypes.c_int, [ctypes.POINTER(LinearDesc), ctypes.c_int32,
                                                ctypes.POINTER(ctypes.c_size_t)]),
    "tp_workspace_init": (ctypes.c_int, [_P, ctypes.c_size_t, _P]),
    "tp_check_status": (ctypes.c_int, [_P, ctypes.c_size_t, _P]),
    "tp_mlp_forward": (ctypes.c_int, [ctypes.POINTER(MlpDesc), _P, _PP, _PP, _PP, _P, _P, _PP,
                                      _PP, _P, ctypes.c_size_t, _P]),
    "tp_mlp_backward": (ctypes.c_int, [ctypes.POINTER(MlpDesc), _P, _PP, _PP, _PP, _PP, _P, _P,
                                       _PP, _PP, _PP, _P, _P, ctypes.c_size_t, _P]),
    "tp_linear_column_forward": (ctypes.c_int, [ctypes.POINTER(LinearDesc), _P, _PP, _PP, _PP,
                                                _PP, _P, ctypes.c_size_t, _P]),
    "tp_linear_column_backward": (ctypes.c_int, [ctypes.POINTER(LinearDesc), _P, _PP, _PP, _PP,
                                                 _P, _PP, _PP, _P, ctypes.c_size_t, _P]),
    "tp_linear_row_forward": (ctypes.c_int, [ctypes.POINTER(LinearDesc), _PP, _PP, _P, _P, _P,
                                             ctypes.c_size_t, _P]),
    "tp_linear_row_backward": (ctypes.c_int, [ctypes.POINTER(LinearDesc), _PP, _PP, _P, _PP,
                                              _PP, _P, _P, ctypes.c_size_t, _P]),
    "tp_selftest_wait_timeout": (ctypes.c_int, [_P, ctypes.c_size_t, ctypes.c_uint32, _P]),
    "tp_trace_start": (ctypes.c_int, [ctypes.c_int32]),
    "tp_mlp_sp_workspace_size": (ctypes.c_int, [ctypes.POINTER(MlpDesc), ctypes.POINTER(ctypes.c_size_t)]),
    "tp_mlp_forward_sp": (ctypes.c_int, [ctypes.POINTER(MlpDesc), _PP, _PP, _PP, _PP, _P, _PP,
                                         _PP, _PP, _P, ctypes.c_size_t, _P]),
    "tp_mlp_backward_sp": (ctypes.c_int, [ctypes.POINTER(MlpDesc), _PP, _PP, _PP, _PP, _PP, _PP,
                                          _PP, _PP, _PP, _PP, _P, _P, ctypes.c_size_t, _P]),
    "tp_linear_row_forward_noalloc": (ctypes.c_int, [ctypes.POINTER(LinearDesc), _PP, _PP, _P,
                                                     _P, _P]),
    "tp_trace_stop": (ctypes.c_int, [ctypes.POINTER(TraceRecord), ctypes.c_int32,
                                     ctypes.POINTER(ctypes.c_int32)]),
    "tp_layernorm_forward": (ctypes.c_int, [ctypes.POINTER(LayerNormDesc), _PP, _PP, _PP, _PP,
                                            _P, _P, _P]),
    "tp_layernorm_backward": (ctypes.c_int, [ctypes.POINTER(LayerNormDesc), _PP, _PP, _P, _P,
                                             _PP, _PP, _PP, _PP, _P]),
    "tp_tuning_set": (ctypes.c_int, [ctypes.c_int32, ctypes.c_int32]),
    "tp_tuning_get": (ctypes.c_int32, [ctypes.c_int32]),
}


def _load():
    path = library_path()
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    so = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(so, name)
        fn.restype = res
        fn.argtypes = args
    return so


lib = _load()


def tp_version() -> int:
    return int(lib.tp_version())


def tp_last_error() -> str:
    return lib.tp_last_error().decode()


def _check(status: int):
    if status != 0:
        raise TpError(status, tp_last_error())


def tp_tuning_set(knob: str, value: int) -> None:
    """Override one measured kernel choice (tests and A/B timing only)."""
    _check(lib.tp_tuning_set(TUNE_KNOBS[knob], int(value)))


def tp_tuning_get(knob: str) -> int:
    return int(lib.tp_tuning_get(TUNE_KNOBS[knob]))


class tuning:
    """Context manager: ``with tuning(raster=1, tma_3d=0): ...`` sets the given knobs and
    restores their previous values on exit."""

    def __init__(self, **knobs):
        self.knobs = {k: int(v) for k, v in knobs.items()}
        self.saved = {}

    def __enter__(self):
        for k, v in self.knobs.items():
            self.saved[k] = tp_tuning_get(k)
            tp_tuning_set(k, v)
        return self

    def __exit__(self, *exc):
        for k, v in self.saved.items():
            tp_tuning_set(k, v)
        return False


# ------------------------------------------------------------------ marshalling helpers
def _ptr(t) -> Optional[int]:
    """Device address of a tensor (or a raw int address). The library reads every buffer as
    dense row-major device memory, so a strided view (a column slice, a transpose) or a host
    tensor is refused here instead of being read with the wrong layout or from the wrong
    memory."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_contiguous():
        raise ValueError(f"tensor of shape {tuple(t.shape)} is not contiguous (row-major); "
                         "pass .contiguous()")
    if t.device.type != "cuda":
        raise ValueError(f"tensor of shape {tuple(t.shape)} is on {t.device}; the library "
                         "reads device memory only")
    return t.data_ptr()


def _io_dtype(code):
    """torch dtype of a call's inputs, weights and saved activations for a tp_dtype code."""
    import torch

    return torch.bfloat16 if code == TP_BF16 else torch.float32


def _need(dtype, what: str, *items) -> None:
    """Every tensor among `items` (tensors, lists of tensors, None or raw int addresses) must
    have `dtype`: the library reads each buffer with the element size of its role (a bf16
    buffer read as fp32 would be read past its end)."""
    for it in items:
        for t in (it if isinstance(it, (list, tuple)) else (it,)):
            if t is None or isinstance(t, int):
                continue
            if t.dtype != dtype:
                raise ValueError(f"{what} must be {dtype}, got {t.dtype} (shape {tuple(t.shape)})")


def _f32():
    import torch

    return torch.float32


def _arr(ts: Optional[Sequence]):
    if ts is None:
        return None
    return (ctypes.c_void_p * len(ts))(*[_ptr(t) for t in ts])


def _stream(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ws(ws):
    return _ptr(ws), (ws.numel() * ws.element_size() if ws is not None else 0)


def _desc_mlp(d) -> MlpDesc:
    return d if isinstance(d, MlpDesc) else MlpDesc(**d)


def _desc_lin(d) -> LinearDesc:
    return d if isinstance(d, LinearDesc) else LinearDesc(**d)


def _desc_ln(d) -> LayerNormDesc:
    return d if isinstance(d, LayerNormDesc) else LayerNormDesc(**d)


# ------------------------------------------------------------------ entry points
def tp_mlp_workspace_size(desc) -> int:
    out = ctypes.c_size_t(0)
    _check(lib.tp_mlp_workspace_size(ctypes.byref(_desc_mlp(desc)), ctypes.byref(out)))
    return int(out.value)


def tp_linear_workspace_size(desc, kind: int) -> int:
    out = ctypes.c_size_t(0)
    _check(lib.tp_linear_workspace_size(ctypes.byref(_desc_lin(desc)), kind, ctypes.byref(out)))
    return int(out.value)


def new_workspace(nbytes: int, device="cuda", stream=None):
    """Allocate (torch) and initialise a workspace of at least nbytes."""
    import torch
    ws = torch.empty(max(int(nbytes), 256), dtype=torch.uint8, device=device)
    tp_workspace_init(ws, stream)
    return ws


def tp_workspace_init(ws, stream=None):
    p, n = _ws(ws)
    _check(lib.tp_workspace_init(p, n, _stream(stream)))


def tp_check_status(ws, stream=None):
    p, n = _ws(ws)
    _check(lib.tp_check_status(p, n, _stream(stream)))


def tp_selftest_wait_timeout(ws, limit_us: int, stream=None):
    p, n = _ws(ws)
    _check(lib.tp_selftest_wait_timeout(p, n, limit_us, _stream(stream)))


def tp_mlp_forward(desc, X, A, a, B, b, Z, Hsave, Ysave, ws, stream=None):
    io = _io_dtype(_desc_mlp(desc).dtype)
    _need(io, "X, A, a, B, b, Hsave, Ysave", X, A, a, B, b, Hsave, Ysave)
    _need(_f32(), "Z", Z)
    p, n = _ws(ws)
    _check(lib.tp_mlp_forward(ctypes.byref(_desc_mlp(desc)), _ptr(X), _arr(A), _arr(a), _arr(B),
                              _ptr(b), _ptr(Z), _arr(Hsave), _arr(Ysave), p, n, _stream(stream)))


def tp_mlp_backward(desc, X, A, B, Hsave, Ysave, dZ, dX, dA, da, dB, db, ws, stream=None):
    io = _io_dtype(_desc_mlp(desc).dtype)
    _need(io, "X, A, B, Hsave, Ysave, dZ", X, A, B, Hsave, Ysave, dZ)
    _need(_f32(), "dX, dA, da, dB, db", dX, dA, da, dB, db)
    p, n = _ws(ws)
    _check(lib.tp_mlp_backward(ctypes.byref(_desc_mlp(desc)), _ptr(X), _arr(A), _arr(B),
                               _arr(Hsave), _arr(Ysave), _ptr(dZ), _ptr(dX), _arr(dA), _arr(da),
                               _arr(dB), _ptr(db), p, n, _stream(stream)))


def tp_linear_column_forward(desc, X, W, bias, Y, Hsave, ws, stream=None):
    _need(_io_dtype(_desc_lin(desc).dtype), "X, W, bias, Y, Hsave", X, W, bias, Y, Hsave)
    p, n = _ws(ws)
    _check(lib.tp_linear_column_forward(ctypes.byref(_desc_lin(desc)), _ptr(X), _arr(W),
                                        _arr(bias), _arr(Y), _arr(Hsave), p, n, _stream(stream)))


def tp_linear_column_backward(desc, X, W, Hsave, dY, dX, dW, dbias, ws, stream=None):
    _need(_io_dtype(_desc_lin(desc).dtype), "X, W, Hsave, dY", X, W, Hsave, dY)
    _need(_f32(), "dX, dW, dbias", dX, dW, dbias)
    p, n = _ws(ws)
    _check(lib.tp_linear_column_backward(ctypes.byref(_desc_lin(desc)), _ptr(X), _arr(W),
                                         _arr(Hsave), _arr(dY), _ptr(dX), _arr(dW), _arr(dbias),
                                         p, n, _stream(stream)))


def tp_linear_row_forward(desc, X, W, bias, Z, ws, stream=None):
    _need(_io_dtype(_desc_lin(desc).dtype), "X, W, bias", X, W, bias)
    _need(_f32(), "Z", Z)
    p, n = _ws(ws)
    _check(lib.tp_linear_row_forward(ctypes.byref(_desc_lin(desc)), _arr(X), _arr(W), _ptr(bias),
                                     _ptr(Z), p, n, _stream(stream)))


def tp_linear_row_backward(desc, X, W, dZ, dX, dW, dbias, ws, stream=None):
    _need(_io_dtype(_desc_lin(desc).dtype), "X, W, dZ", X, W, dZ)
    _need(_f32(), "dX, dW, dbias", dX, dW, dbias)
    p, n = _ws(ws)
    _check(lib.tp_linear_row_backward(ctypes.byref(_desc_lin(desc)), _arr(X), _arr(W), _ptr(dZ),
                                      _arr(dX), _arr(dW), _ptr(dbias), p, n, _stream(stream)))


def tp_linear_row_forward_noalloc(desc, X, W, bias, Z, stream=None):
    _need(_io_dtype(_desc_lin(desc).dtype), "X, W, bias", X, W, bias)
    _need(_f32(), "Z", Z)
    _check(lib.tp_linear_row_forward_noalloc(ctypes.byref(_desc_lin(desc)), _arr(X), _arr(W),
                                             _ptr(bias), _ptr(Z), _stream(stream)))


def tp_mlp_sp_workspace_size(desc) -> int:
    out = ctypes.c_size_t(0)
    _check(lib.tp_mlp_sp_workspace_size(ctypes.byref(_desc_mlp(desc)), ctypes.byref(out)))
    return int(out.value)


def tp_mlp_forward_sp(desc, X_shards, A, a, B, b, Z_shards, Hsave, Ysave, ws, stream=None):
    io = _io_dtype(_desc_mlp(desc).dtype)
    _need(io, "X_shards, A, a, B, b, Hsave, Ysave", X_shards, A, a, B, b, Hsave, Ysave)
    _need(_f32(), "Z_shards", Z_shards)
    p, n = _ws(ws)
    _check(lib.tp_mlp_forward_sp(ctypes.byref(_desc_mlp(desc)), _arr(X_shards), _arr(A), _arr(a),
                                 _arr(B), _ptr(b), _arr(Z_shards), _arr(Hsave), _arr(Ysave), p,
                                 n, _stream(stream)))


def tp_mlp_backward_sp(desc, X_shards, A, B, Hsave, Ysave, dZ_shards, dX_shards, dA, da, dB, db,
                       ws, stream=None):
    io = _io_dtype(_desc_mlp(desc).dtype)
    _need(io, "X_shards, A, B, Hsave, Ysave, dZ_shards", X_shards, A, B, Hsave, Ysave, dZ_shards)
    _need(_f32(), "dX_shards, dA, da, dB, db", dX_shards, dA, da, dB, db)
    p, n = _ws(ws)
    _check(lib.tp_mlp_backward_sp(ctypes.byref(_desc_mlp(desc)), _arr(X_shards), _arr(A),
                                  _arr(B), _arr(Hsave), _arr(Ysave), _arr(dZ_shards),
                                  _arr(dX_shards), _arr(dA), _arr(da), _arr(dB), _ptr(db), p, n,
                                  _stream(stream)))


def tp_trace_start(capacity: int):
    _check(lib.tp_trace_start(capacity))


def tp_trace_stop(capacity: int = 100000):
    """Stop tracing; returns a list of dicts (kernel, tag, flops, bytes, ms, groups)."""
    buf = (TraceRecord * capacity)()
    cnt = ctypes.c_int32(0)
    _check(lib.tp_trace_stop(buf, capacity, ctypes.byref(cnt)))
    return [{"kernel": KERNEL_NAMES.get(r.kernel, str(r.kernel)),
             "tag": TAG_NAMES.get(r.tag, str(r.tag)), "flops": r.flops, "bytes": r.bytes,
             "ms": r.ms, "groups": r.groups} for r in buf[:cnt.value]]


def tp_layernorm_forward(desc, X, gamma, beta, Y, mean, rstd, stream=None):
    """LayerNorm over a hidden dimension split into desc.tp_degree column shards: lists of
    per-shard tensors X [T, H/n], gamma/beta [H/n] (or None), Y [T, H/n]; mean, rstd fp32 [T]
    (or None)."""
    _need(_io_dtype(_desc_ln(desc).dtype), "X, gamma, beta, Y", X, gamma, beta, Y)
    _need(_f32(), "mean, rstd", mean, rstd)
    _check(lib.tp_layernorm_forward(ctypes.byref(_desc_ln(desc)), _arr(X), _arr(gamma),
                                    _arr(beta), _arr(Y), _ptr(mean), _ptr(rstd),
                                    _stream(stream)))


def tp_layernorm_backward(desc, X, gamma, mean, rstd, dY, dX, dgamma, dbeta, stream=None):
    """Backward of tp_layernorm_forward: dX [T, H/n] per shard; dgamma, dbeta fp32 [H/n] per
    shard (lists, or None)."""
    _need(_io_dtype(_desc_ln(desc).dtype), "X, gamma, dY, dX", X, gamma, dY, dX)
    _need(_f32(), "mean, rstd, dgamma, dbeta", mean, rstd, dgamma, dbeta)
    _check(lib.tp_layernorm_backward(ctypes.byref(_desc_ln(desc)), _arr(X), _arr(gamma),
                                     _ptr(mean), _ptr(rstd), _arr(dY), _arr(dX), _arr(dgamma),
                                     _arr(dbeta), _stream(stream)))
