"""Weight-streaming projection kernels for GB300 (sm_103a): the Python binding.

This module only marshals arguments: it checks dtypes, shapes and devices of torch
tensors, passes their device pointers and the current CUDA stream to the C ABI of
``libpgq.so`` (declared in ``include/pgq.h``) and raises on a non-zero status.  Every
step of the computation runs in the library's CUDA kernels; there is no fallback.
If the library has not been built, every call raises ``RuntimeError``.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# PGQ_LIBRARY may name another build of the same library (e.g. an instrumented one)
LIB_PATH = os.environ.get("PGQ_LIBRARY") or os.path.join(_HERE, "libpgq.so")

# status codes and epilogues (mirrors include/pgq.h)
OK, EINVAL, EALIGN, EUNSUPPORTED, ECUDA, ETIMEOUT, ENODEV, EWORKSPACE = range(8)
EPI_NONE, EPI_RELU2, EPI_ADD = 0, 1, 2
EPILOGUES = {"none": EPI_NONE, "relu2": EPI_RELU2, "add": EPI_ADD}
QBLOCK = 32
DECODE_BMAX = 8
PASS_BMAX = 64
PASS_LMAX = 8      # layers per persistent launch of the prefill pass (PGQ_PASS_LMAX)

_vp = C.c_void_p


class Q8Job(C.Structure):
    _fields_ = [("codes", _vp), ("params", _vp), ("rows", C.c_int), ("input", C.c_int),
                ("y", _vp), ("epilogue", C.c_int), ("residual", _vp)]


class Input(C.Structure):
    _fields_ = [("x", _vp), ("gamma", _vp)]


class Q8Matrix(C.Structure):
    _fields_ = [("codes", _vp), ("params", _vp)]


class MoeLayer(C.Structure):
    _fields_ = [("router", _vp), ("up_codes", _vp), ("up_params", _vp), ("down_codes", _vp), ("down_params", _vp),
                ("E", C.c_int), ("k", C.c_int), ("hidden", C.c_int), ("inter", C.c_int), ("renorm", C.c_int)]


class MoeQ82Layer(C.Structure):
    _fields_ = [("router", _vp), ("up_codes", _vp), ("up_row_scale", _vp), ("up_col_field", _vp),
                ("down_codes", _vp), ("down_row_scale", _vp), ("down_col_field", _vp),
                ("E", C.c_int), ("k", C.c_int), ("hidden", C.c_int), ("inter", C.c_int), ("renorm", C.c_int)]


class Q82Matrix(C.Structure):
    _fields_ = [("codes", _vp), ("row_scale", _vp), ("col_field", _vp)]


class Q82Job(C.Structure):
    _fields_ = [("codes", _vp), ("row_scale", _vp), ("col_field", _vp), ("rows", C.c_int), ("y", _vp),
                ("epilogue", C.c_int), ("residual", _vp)]


class Q82Layer(C.Structure):
    _fields_ = [("q", Q82Matrix), ("k", Q82Matrix), ("v", Q82Matrix), ("o", Q82Matrix),
                ("up", Q82Matrix), ("down", Q82Matrix),
                ("hidden", C.c_int), ("kv", C.c_int), ("inter", C.c_int)]


class Q8Layer(C.Structure):
    _fields_ = [("q", Q8Matrix), ("k", Q8Matrix), ("v", Q8Matrix), ("o", Q8Matrix),
                ("up", Q8Matrix), ("down", Q8Matrix),
                ("hidden", C.c_int), ("kv", C.c_int), ("inter", C.c_int)]


_SIGS = {
    "pgq_status_string": (C.c_char_p, [C.c_int]),
    "pgq_last_error": (C.c_char_p, []),
    "pgq_abi_version": (C.c_int, []),
    "pgq_device_check": (C.c_int, []),
    "pgq_add_rmsnorm": (C.c_int, [_vp, _vp, _vp, C.c_float, C.c_int, C.c_int, _vp, _vp, _vp]),
    "pgq_add_rmsnorm_ex": (C.c_int, [_vp, _vp, _vp, C.c_float, C.c_float, C.c_int, C.c_int, C.c_int, _vp, _vp,
                                     _vp]),
    "pgq_sandwich_rmsnorm": (C.c_int, [_vp, _vp, _vp, _vp, C.c_float, C.c_float, C.c_int, C.c_int, C.c_int, _vp,
                                       _vp, _vp, _vp, _vp]),
    "pgq_relu2": (C.c_int, [_vp, C.c_size_t, _vp]),
    "pgq_gemv_f16": (C.c_int, [_vp, C.c_int, C.c_int, _vp, C.c_int, _vp, C.c_float, _vp, C.c_int, _vp, _vp]),
    "pgq_argmax_workspace_bytes": (C.c_size_t, [C.c_int]),
    "pgq_gemv_f16_argmax": (C.c_int, [_vp, C.c_int, C.c_int, _vp, C.c_int, _vp, C.c_float, _vp, _vp, _vp,
                                      C.c_size_t, _vp]),
    "pgq_argmax": (C.c_int, [_vp, C.c_int, C.c_int, _vp, _vp]),
    "pgq_gemv_f16_argmax_static": (C.c_int, [_vp, C.c_int, C.c_int, _vp, C.c_int, _vp, C.c_float, _vp, _vp, _vp]),
    "pgq_gemv_q8": (C.c_int, [_vp, _vp, C.c_int, C.c_int, _vp, C.c_int, _vp, C.c_float, _vp, C.c_int, _vp, _vp]),
    "pgq_gemv_q8_multi": (C.c_int, [C.POINTER(Q8Job), C.c_int, C.POINTER(Input), C.c_int, C.c_int, C.c_int,
                                    C.c_float, _vp]),
    "pgq_gemv_q82f": (C.c_int, [_vp, _vp, _vp, C.c_int, C.c_int, _vp, C.c_int, _vp, C.c_float, _vp, C.c_int, _vp,
                                _vp]),
    "pgq_q82f_decode_layer": (C.c_int, [C.POINTER(Q82Layer), _vp, _vp, _vp, C.c_float, _vp, _vp, _vp, _vp, _vp,
                                        _vp, C.c_int, _vp]),
    "pgq_q8_decode_layer_fused": (C.c_int, [C.POINTER(Q8Layer), _vp, _vp, _vp, C.c_float, _vp, _vp, _vp, _vp, _vp,
                                            _vp, C.c_int, _vp, _vp]),
    "pgq_mlp_f16_decode_fused": (C.c_int, [_vp, _vp, _vp, C.c_int, C.c_int, _vp, C.c_float, _vp, _vp, _vp, _vp]),
    "pgq_mlp_f16_decode": (C.c_int, [_vp, _vp, _vp, C.c_int, C.c_int, _vp, C.c_float, _vp, _vp, _vp]),
    "pgq_q8_decode_layer": (C.c_int, [C.POINTER(Q8Layer), _vp, _vp, _vp, C.c_float, _vp, _vp, _vp, _vp, _vp,
                                      _vp, _vp]),
    "pgq_q8_decode_layer_ex": (C.c_int, [C.POINTER(Q8Layer), _vp, _vp, _vp, C.c_float, _vp, _vp, _vp, _vp, _vp,
                                         _vp, C.c_int, _vp]),
    "pgq_prefill_q8_workspace_bytes": (C.c_size_t, [C.POINTER(C.c_int), C.c_int, C.c_int, C.c_int]),
    "pgq_prefill_q8": (C.c_int, [C.POINTER(Q8Job), C.c_int, _vp, C.c_int, C.c_int, _vp, C.c_size_t, _vp]),
    "pgq_prefill_q82f": (C.c_int, [C.POINTER(Q82Job), C.c_int, _vp, C.c_int, C.c_int, _vp, C.c_size_t, _vp]),
    "pgq_prefill_status": (C.c_int, [_vp, _vp]),
    "pgq_last_device_status": (C.c_int, [_vp, _vp]),
    "pgq_set_wait_limit_ns": (C.c_int, [C.c_ulonglong]),
    "pgq_wait_limit_ns": (C.c_ulonglong, []),
    "pgq_debug_stall": (C.c_int, [C.c_int]),
    "pgq_moe_router": (C.c_int, [_vp, C.c_int, C.c_int, _vp, C.c_int, _vp, _vp]),
    "pgq_moe_route_topk": (C.c_int, [_vp, C.c_int, C.c_int, C.c_int, C.c_int, _vp, _vp, _vp]),
    "pgq_moe_group_gather": (C.c_int, [_vp, C.c_int, C.c_int, C.c_int, _vp, _vp, _vp, _vp, C.c_int, C.c_int, _vp,
                                       _vp]),
    "pgq_moe_experts_q8": (C.c_int, [_vp, _vp, C.c_int, C.c_int, C.c_int, _vp, _vp, _vp, C.c_int, _vp, C.c_int, _vp,
                                     C.c_int, _vp]),
    "pgq_moe_combine_rmsnorm": (C.c_int, [_vp, _vp, _vp, _vp, C.c_int, _vp, C.c_float, C.c_int, C.c_int, _vp, _vp,
                                          _vp]),
    "pgq_moe_layer_workspace_bytes": (C.c_size_t, [C.POINTER(MoeLayer), C.c_int]),
    "pgq_moe_layer_layout": (C.c_int, [C.POINTER(MoeLayer), C.c_int, C.POINTER(C.c_size_t)]),
    "pgq_moe_prefill_layer": (C.c_int, [C.POINTER(MoeLayer), _vp, C.c_int, _vp, _vp, C.c_float, _vp, _vp,
                                        C.c_size_t, _vp]),
    "pgq_moe_q82f_layer_workspace_bytes": (C.c_size_t, [C.POINTER(MoeQ82Layer), C.c_int]),
    "pgq_moe_q82f_layer_layout": (C.c_int, [C.POINTER(MoeQ82Layer), C.c_int, C.POINTER(C.c_size_t)]),
    "pgq_moe_q82f_prefill_layer": (C.c_int, [C.POINTER(MoeQ82Layer), _vp, C.c_int, _vp, _vp, C.c_float, _vp, _vp,
                                             C.c_size_t, _vp]),
    "pgq_q8_prefill_pass_workspace_bytes": (C.c_size_t, [C.c_int, C.c_int, C.c_int, C.c_int]),
    "pgq_q8_prefill_pass_layout": (C.c_int, [C.c_int, C.c_int, C.c_int, C.c_int, C.POINTER(C.c_size_t)]),
    "pgq_q8_prefill_pass": (C.c_int, [C.POINTER(Q8Layer), C.c_int, _vp, C.c_int, _vp, _vp, C.c_float, _vp,
                                      C.c_size_t, _vp]),
    "pgq_q82f_prefill_pass": (C.c_int, [C.POINTER(Q82Layer), C.c_int, _vp, C.c_int, _vp, _vp, C.c_float, _vp,
                                        C.c_size_t, _vp]),
}

_lib = None


def lib():
    """The loaded ``libpgq.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                               "`python -m prefill_gemv_q8_gb300.build` (nvcc, sm_103a)")
        L = C.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype, fn.argtypes = res, args
        _lib = L
    return _lib


class PgqError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"pgq status {status} ({status_string(status)}): {msg}")
        self.status = status


def status_string(status: int) -> str:
    return lib().pgq_status_string(status).decode()


def _check(status: int):
    if status != OK:
        raise PgqError(status, lib().pgq_last_error().decode())


def _ptr(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _need(t, dtype, name, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    return t


def _epi(e):
    return EPILOGUES[e] if isinstance(e, str) else int(e)


# ------------------------------------------------------------------ primitives
def add_rmsnorm(h, gamma, eps, add=None, y=None, inv=None, stream=None):
    """h += add (if given); y = gamma * h / sqrt(mean(h²) + eps).  h [B][n] in place."""
    _need(h, torch.float32, "h")
    B, n = h.shape
    _need(gamma, torch.float32, "gamma", (n,))
    if add is not None:
        _need(add, torch.float32, "add", (B, n))
    y = torch.empty_like(h) if y is None else _need(y, torch.float32, "y", (B, n))
    if inv is not None:
        _need(inv, torch.float32, "inv", (B,))
    _check(lib().pgq_add_rmsnorm(_ptr(h), _ptr(add), _ptr(gamma), eps, B, n, _ptr(y), _ptr(inv), _stream(stream)))
    return y


NORM_GEMMA = 1


def add_rmsnorm_ex(h, gamma, eps, add=None, scale=0.0, gemma=False, y=None, inv=None, stream=None):
    """h <- (h + add)·scale in place (scale 0: none), y = w·(h·inv) with w = 1 + gamma
    when ``gemma``; returns y."""
    _need(h, torch.float32, "h")
    B, n = h.shape
    _need(gamma, torch.float32, "gamma", (n,))
    if add is not None:
        _need(add, torch.float32, "add", (B, n))
    if y is None:
        y = torch.empty_like(h)
    _check(lib().pgq_add_rmsnorm_ex(_ptr(h), _ptr(add), _ptr(gamma), eps, float(scale), NORM_GEMMA if gemma else 0,
                                    B, n, _ptr(y), _ptr(inv), _stream(stream)))
    return y


def sandwich_rmsnorm(x, w1, h, w2, eps, scale=0.0, gemma=False, out=None, mid=None, inv1=None, inv2=None,
                     stream=None):
    """Gemma's sandwich residual in one launch: mid = rms(x)·w1', h <- (h + mid)·scale,
    out = rms(h)·w2' (w' = 1 + w when ``gemma``); returns out."""
    _need(x, torch.float32, "x")
    B, n = x.shape
    _need(h, torch.float32, "h", (B, n))
    _need(w1, torch.float32, "w1", (n,))
    _need(w2, torch.float32, "w2", (n,))
    if out is None:
        out = torch.empty_like(h)
    _check(lib().pgq_sandwich_rmsnorm(_ptr(x), _ptr(w1), _ptr(h), _ptr(w2), eps, float(scale),
                                      NORM_GEMMA if gemma else 0, B, n, _ptr(out), _ptr(mid), _ptr(inv1), _ptr(inv2),
                                      _stream(stream)))
    return out


def relu2(v, stream=None):
    _need(v, torch.float32, "v")
    _check(lib().pgq_relu2(_ptr(v), v.numel(), _stream(stream)))
    return v


def argmax(logits, ids=None, stream=None):
    _need(logits, torch.float32, "logits")
    B, V = logits.shape
    ids = torch.empty(B, dtype=torch.int32, device=logits.device) if ids is None else ids
    _need(ids, torch.int32, "ids", (B,))
    _check(lib().pgq_argmax(_ptr(logits), B, V, _ptr(ids), _stream(stream)))
    return ids


def gemv_f16(W, x, gamma=None, eps=1e-6, epilogue="none", residual=None, y=None, stream=None):
    """y[b] = epilogue(W · xin[b]) for a binary16 W [rows][cols] and x [B][cols]."""
    _need(W, torch.float16, "W")
    rows, cols = W.shape
    _need(x, torch.float32, "x")
    B = x.shape[0]
    if gamma is not None:
        _need(gamma, torch.float32, "gamma", (cols,))
    y = torch.empty(B, rows, dtype=torch.float32, device=W.device) if y is None else y
    _need(y, torch.float32, "y", (B, rows))
    if residual is not None:
        _need(residual, torch.float32, "residual", (B, rows))
    _check(lib().pgq_gemv_f16(_ptr(W), rows, cols, _ptr(x), B, _ptr(gamma), eps, _ptr(y), _epi(epilogue),
                              _ptr(residual), _stream(stream)))
    return y


def argmax_workspace_bytes(B):
    return int(lib().pgq_argmax_workspace_bytes(B))


def gemv_f16_argmax(W, x, gamma=None, eps=1e-6, logits=True, workspace=None, ids=None, stream=None):
    """Vocab head: logits = W · xin, ids = per-position argmax.  Returns (ids, logits or None)."""
    _need(W, torch.float16, "W")
    rows, cols = W.shape
    _need(x, torch.float32, "x")
    B = x.shape[0]
    dev = W.device
    if logits is True:
        logits = torch.empty(B, rows, dtype=torch.float32, device=dev)
    elif logits is False:
        logits = None
    if logits is not None:
        _need(logits, torch.float32, "logits", (B, rows))
    ids = torch.empty(B, dtype=torch.int32, device=dev) if ids is None else ids
    _need(ids, torch.int32, "ids", (B,))
    need = argmax_workspace_bytes(B)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    _check(lib().pgq_gemv_f16_argmax(_ptr(W), rows, cols, _ptr(x), B, _ptr(gamma), eps, _ptr(logits), _ptr(ids),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream)))
    return ids, logits


def _q8_check(codes, params, name="W"):
    _need(codes, torch.int8, name + ".codes")
    rows, cols = codes.shape
    _need(params, torch.float16, name + ".params", (rows, cols // QBLOCK, 2))
    return rows, cols


def gemv_q8(codes, params, x, gamma=None, eps=1e-6, epilogue="none", residual=None, y=None, stream=None):
    """y[b] = epilogue(W · xin[b]) for a q8 block-format W (codes int8 [rows][cols],
    params binary16 [rows][cols/32][2])."""
    rows, cols = _q8_check(codes, params)
    _need(x, torch.float32, "x")
    B = x.shape[0]
    y = torch.empty(B, rows, dtype=torch.float32, device=codes.device) if y is None else y
    _need(y, torch.float32, "y", (B, rows))
    if residual is not None:
        _need(residual, torch.float32, "residual", (B, rows))
    _check(lib().pgq_gemv_q8(_ptr(codes), _ptr(params), rows, cols, _ptr(x), B, _ptr(gamma), eps, _ptr(y),
                             _epi(epilogue), _ptr(residual), _stream(stream)))
    return y


def gemv_q8_multi(jobs, inputs, eps=1e-6, stream=None):
    """jobs: list of dicts {codes, params, input, y, epilogue, residual}; inputs: list of
    (x, gamma or None).  One launch."""
    cols = jobs[0]["codes"].shape[1]
    B = inputs[0][0].shape[0]
    J = (Q8Job * len(jobs))()
    keep = []
    for i, j in enumerate(jobs):
        rows, c = _q8_check(j["codes"], j["params"])
        if c != cols:
            raise ValueError("all jobs of one launch must share cols")
        _need(j["y"], torch.float32, "y", (B, rows))
        J[i] = Q8Job(j["codes"].data_ptr(), j["params"].data_ptr(), rows, j.get("input", 0), j["y"].data_ptr(),
                     _epi(j.get("epilogue", "none")),
                     j["residual"].data_ptr() if j.get("residual") is not None else None)
    I = (Input * len(inputs))()
    for i, (x, g) in enumerate(inputs):
        _need(x, torch.float32, "x", (B, cols))
        I[i] = Input(x.data_ptr(), g.data_ptr() if g is not None else None)
    keep.append((J, I))
    _check(lib().pgq_gemv_q8_multi(J, len(jobs), I, len(inputs), cols, B, eps, _stream(stream)))


def _jobs_struct(jobs, B, cols):
    J = (Q8Job * len(jobs))()
    for i, j in enumerate(jobs):
        rows, c = _q8_check(j["codes"], j["params"])
        if c != cols:
            raise ValueError("all jobs of one launch must share cols")
        _need(j["y"], torch.float32, "y", (B, rows))
        res = j.get("residual")
        if res is not None:
            _need(res, torch.float32, "residual", (B, rows))
        J[i] = Q8Job(j["codes"].data_ptr(), j["params"].data_ptr(), rows, j.get("input", 0), j["y"].data_ptr(),
                     _epi(j.get("epilogue", "none")), res.data_ptr() if res is not None else None)
    return J


def prefill_workspace_bytes(rows, cols, B):
    rows = list(rows)
    arr = (C.c_int * len(rows))(*rows)
    return int(lib().pgq_prefill_q8_workspace_bytes(arr, len(rows), cols, B))


def prefill_workspace(rows, cols, B, device="cuda"):
    return torch.empty(prefill_workspace_bytes(rows, cols, B), dtype=torch.uint8, device=device)


def prefill_q8(jobs, X, workspace=None, stream=None):
    """Batched prefill projection: for each job {codes, params, y, epilogue, residual},
    y = epilogue(W · X[b]) for the B <= 64 positions of X [B][cols] (one launch of the
    binary16 conversion of X and one tensor-core GEMM launch)."""
    _need(X, torch.float32, "X")
    B, cols = X.shape
    J = _jobs_struct(jobs, B, cols)
    if workspace is None:
        workspace = prefill_workspace([j["codes"].shape[0] for j in jobs], cols, B, X.device)
    _check(lib().pgq_prefill_q8(J, len(jobs), _ptr(X), cols, B, _ptr(workspace), workspace.numel(),
                                _stream(stream)))
    return workspace


def prefill_q82f(jobs, X, workspace=None, stream=None):
    """prefill_q8 with q8_2f matrices: each job {codes, row_scale, col_field, y,
    epilogue, residual}."""
    _need(X, torch.float32, "X")
    B, cols = X.shape
    J = (Q82Job * len(jobs))()
    for i, j in enumerate(jobs):
        rows, c = _q82f_check(j["codes"], j["row_scale"], j["col_field"], "job")
        if c != cols:
            raise ValueError("all jobs of one launch must share cols")
        _need(j["y"], torch.float32, "y", (B, rows))
        res = j.get("residual")
        if res is not None:
            _need(res, torch.float32, "residual", (B, rows))
        J[i] = Q82Job(j["codes"].data_ptr(), j["row_scale"].data_ptr(), j["col_field"].data_ptr(), rows,
                      j["y"].data_ptr(), _epi(j.get("epilogue", "none")), res.data_ptr() if res is not None else None)
    if workspace is None:
        workspace = prefill_workspace([j["codes"].shape[0] for j in jobs], cols, B, X.device)
    _check(lib().pgq_prefill_q82f(J, len(jobs), _ptr(X), cols, B, _ptr(workspace), workspace.numel(),
                                  _stream(stream)))
    return workspace


def prefill_status(workspace, stream=None):
    return int(lib().pgq_prefill_status(_ptr(workspace), _stream(stream)))


def last_device_status(workspace=None, stream=None):
    """Status of the device-side waits since the last check (synchronises the
    stream): ``ETIMEOUT`` if a decode kernel's wait, or the last call on
    ``workspace``, ran out; ``OK`` otherwise.  Clears the decode record."""
    return int(lib().pgq_last_device_status(_ptr(workspace) if workspace is not None else None, _stream(stream)))


def set_wait_limit_ns(ns):
    """Limit of every bounded device-side wait for later launches (0: the default)."""
    _check(lib().pgq_set_wait_limit_ns(int(ns)))


def wait_limit_ns():
    return int(lib().pgq_wait_limit_ns())


def debug_stall(on):
    """Test hook: while on, decode (one position) and prefill-pass launches wait for
    an event that never comes, so their bounded waits run out."""
    _check(lib().pgq_debug_stall(1 if on else 0))


# ------------------------------------------------------------------ workloads
def mlp_f16_decode(h, W_up, W_down, gamma, eps=1e-6, u=None, y=None, stream=None):
    """y = h + W_down · relu²(W_up · rms(h)·gamma) for one position; returns (y, u)."""
    _need(h, torch.float32, "h")
    hidden = h.numel()
    inter = W_up.shape[0]
    _need(W_up, torch.float16, "W_up", (inter, hidden))
    _need(W_down, torch.float16, "W_down", (hidden, inter))
    _need(gamma, torch.float32, "gamma", (hidden,))
    u = torch.empty(inter, dtype=torch.float32, device=h.device) if u is None else u
    y = torch.empty_like(h) if y is None else y
    _check(lib().pgq_mlp_f16_decode(_ptr(h), _ptr(W_up), _ptr(W_down), hidden, inter, _ptr(gamma), eps, _ptr(u),
                                    _ptr(y), _stream(stream)))
    return y, u


def _q82f_check(codes, rs, cf, name="W"):
    _need(codes, torch.int8, name + ".codes")
    rows, cols = codes.shape
    _need(rs, torch.float16, name + ".row_scale", (rows,))
    _need(cf, torch.float16, name + ".col_field", (cols,))
    return rows, cols


def gemv_q82f(codes, row_scale, col_field, x, gamma=None, eps=1e-6, epilogue="none", residual=None, y=None,
              stream=None):
    """y[b] = epilogue(row_scale ⊙ (codes · (col_field ⊙ xin[b]))) for a q8_2f matrix."""
    _q82f_check(codes, row_scale, col_field)
    rows, cols = codes.shape
    _need(x, torch.float32, "x")
    x2 = x.view(-1, cols)
    B = x2.shape[0]
    if y is None:
        y = torch.empty(B, rows, dtype=torch.float32, device=x.device)
    _check(lib().pgq_gemv_q82f(_ptr(codes), _ptr(row_scale), _ptr(col_field), rows, cols, _ptr(x2), B, _ptr(gamma),
                               eps, _ptr(y), _epi(epilogue), _ptr(residual), _stream(stream)))
    return y


def q82f_layer_struct(mats):
    """ctypes view of a q8_2f decode layer {slot: (codes, row_scale, col_field)}."""
    L = Q82Layer()
    for s in ("q", "k", "v", "o", "up", "down"):
        c, r, f = mats[s]
        _q82f_check(c, r, f, s)
        setattr(L, s, Q82Matrix(c.data_ptr(), r.data_ptr(), f.data_ptr()))
    L.hidden, L.kv, L.inter = mats["q"][0].shape[1], mats["k"][0].shape[0], mats["up"][0].shape[0]
    return L


def q82f_decode_layer(mats, x, x_o, gamma, eps=1e-6, out=None, stream=None, weights_stable=False):
    """The decode layer with q8_2f matrices (see q8_decode_layer); ``mats`` maps slot →
    (codes, row_scale, col_field), or is a prebuilt Q82Layer."""
    L = mats if isinstance(mats, Q82Layer) else q82f_layer_struct(mats)
    if out is None:
        out = {s: torch.empty(n, dtype=torch.float32, device=x.device) for s, n in
               (("q", L.hidden), ("k", L.kv), ("v", L.kv), ("o", L.hidden), ("u", L.inter), ("down", L.hidden))}
    _check(lib().pgq_q82f_decode_layer(C.byref(L), _ptr(x), _ptr(x_o), _ptr(gamma), eps, _ptr(out["q"]),
                                       _ptr(out["k"]), _ptr(out["v"]), _ptr(out["o"]), _ptr(out["u"]),
                                       _ptr(out["down"]), WEIGHTS_STABLE if weights_stable else 0, _stream(stream)))
    return out


def q8_layer_struct(mats):
    """ctypes view of a decode layer {slot: (codes, params)}."""
    hidden = mats["q"][0].shape[1]
    L = Q8Layer()
    for s in ("q", "k", "v", "o", "up", "down"):
        c, p = mats[s]
        _q8_check(c, p, s)
        setattr(L, s, Q8Matrix(c.data_ptr(), p.data_ptr()))
    L.hidden, L.kv, L.inter = hidden, mats["k"][0].shape[0], mats["up"][0].shape[0]
    return L


WEIGHTS_STABLE = 1


def q8_decode_layer(mats, x, x_o, gamma, eps=1e-6, out=None, stream=None, weights_stable=False):
    """The q8 decode layer for one position; returns dict q, k, v, o, u, down.
    weights_stable: no work still in flight on the stream writes these weights (both
    launches may then start streaming them while the kernel before them finishes).
    ``mats`` may also be a prebuilt ``Q8Layer`` (q8_layer_struct), whose tensors the
    caller keeps alive."""
    L = mats if isinstance(mats, Q8Layer) else q8_layer_struct(mats)
    dev = x.device
    if out is None:
        out = {s: torch.empty(n, dtype=torch.float32, device=dev) for s, n in
               (("q", L.hidden), ("k", L.kv), ("v", L.kv), ("o", L.hidden), ("u", L.inter), ("down", L.hidden))}
    _check(lib().pgq_q8_decode_layer_ex(C.byref(L), _ptr(x), _ptr(x_o), _ptr(gamma), eps, _ptr(out["q"]),
                                        _ptr(out["k"]), _ptr(out["v"]), _ptr(out["o"]), _ptr(out["u"]),
                                        _ptr(out["down"]), WEIGHTS_STABLE if weights_stable else 0,
                                        _stream(stream)))
    return out


LAYER_SYNC_BYTES = 16


def layer_sync(device="cuda"):
    """A zeroed sync word for the fused (one-launch) decode layers."""
    return torch.zeros(LAYER_SYNC_BYTES // 4, dtype=torch.int32, device=device)


def q8_decode_layer_fused(mats, x, x_o, gamma, eps=1e-6, sync=None, out=None, stream=None, weights_stable=False):
    """The q8 decode layer in one launch (see q8_decode_layer); ``sync`` from
    layer_sync(), ordered on one stream between calls."""
    L = mats if isinstance(mats, Q8Layer) else q8_layer_struct(mats)
    if sync is None:
        sync = layer_sync(x.device)
    if out is None:
        out = {s: torch.empty(n, dtype=torch.float32, device=x.device) for s, n in
               (("q", L.hidden), ("k", L.kv), ("v", L.kv), ("o", L.hidden), ("u", L.inter), ("down", L.hidden))}
    _check(lib().pgq_q8_decode_layer_fused(C.byref(L), _ptr(x), _ptr(x_o), _ptr(gamma), eps, _ptr(out["q"]),
                                           _ptr(out["k"]), _ptr(out["v"]), _ptr(out["o"]), _ptr(out["u"]),
                                           _ptr(out["down"]), WEIGHTS_STABLE if weights_stable else 0, _ptr(sync),
                                           _stream(stream)))
    return out


def mlp_f16_decode_fused(h, W_up, W_down, gamma, eps=1e-6, sync=None, u=None, y=None, stream=None):
    """The tiny MLP block in one launch (see mlp_f16_decode); returns (y, u)."""
    _need(h, torch.float32, "h")
    hidden = h.numel()
    inter = W_up.shape[0]
    _need(W_up, torch.float16, "W_up", (inter, hidden))
    _need(W_down, torch.float16, "W_down", (hidden, inter))
    _need(gamma, torch.float32, "gamma", (hidden,))
    if sync is None:
        sync = layer_sync(h.device)
    if u is None:
        u = torch.empty(inter, dtype=torch.float32, device=h.device)
    if y is None:
        y = torch.empty(hidden, dtype=torch.float32, device=h.device)
    _check(lib().pgq_mlp_f16_decode_fused(_ptr(h), _ptr(W_up), _ptr(W_down), hidden, inter, _ptr(gamma), eps, _ptr(u),
                                          _ptr(y), _ptr(sync), _stream(stream)))
    return y, u


def prefill_pass_workspace(hidden, kv, inter, B, device="cuda"):
    n = int(lib().pgq_q8_prefill_pass_workspace_bytes(hidden, kv, inter, B))
    return torch.empty(n, dtype=torch.uint8, device=device)


def prefill_pass_taps(workspace, hidden, kv, inter, B):
    """Views of the last layer's n1, q, k, v, h1, n2, u inside a pass workspace."""
    off = (C.c_size_t * 7)()
    _check(lib().pgq_q8_prefill_pass_layout(hidden, kv, inter, B, off))
    sizes = (hidden, hidden, kv, kv, hidden, hidden, inter)
    names = ("n1", "q", "k", "v", "h1", "n2", "u")
    f = workspace.view(torch.uint8)
    return {nm: f[o:o + B * n * 4].view(torch.float32).view(B, n) for nm, o, n in zip(names, off, sizes)}


class PassLayers:
    """ctypes array of L layer descriptors (keeps the tensors alive)."""

    def __init__(self, layers):
        self.layers = layers
        self.arr = (Q8Layer * len(layers))(*[q8_layer_struct(m) for m in layers])
        self.hidden, self.kv, self.inter = self.arr[0].hidden, self.arr[0].kv, self.arr[0].inter


class Q82PassLayers:
    """ctypes array of L q8_2f layer descriptors (keeps the tensors alive)."""

    def __init__(self, layers):
        self.layers = layers
        self.arr = (Q82Layer * len(layers))(*[q82f_layer_struct(m) for m in layers])
        self.hidden, self.kv, self.inter = self.arr[0].hidden, self.arr[0].kv, self.arr[0].inter


def q82f_prefill_pass(layers, h, gamma1, gamma2, eps=1e-6, workspace=None, stream=None):
    """prefill_pass with q8_2f layers ({slot: (codes, row_scale, col_field)}, or a
    Q82PassLayers); the workspace is the q8 pass's."""
    if not isinstance(layers, Q82PassLayers):
        layers = Q82PassLayers(layers)
    _need(h, torch.float32, "h")
    B, H = h.shape
    L = len(layers.layers)
    _need(gamma1, torch.float32, "gamma1", (L, H))
    _need(gamma2, torch.float32, "gamma2", (L, H))
    if workspace is None:
        workspace = prefill_pass_workspace(layers.hidden, layers.kv, layers.inter, B, h.device)
    _check(lib().pgq_q82f_prefill_pass(layers.arr, L, _ptr(h), B, _ptr(gamma1), _ptr(gamma2), eps,
                                       _ptr(workspace), workspace.numel(), _stream(stream)))
    return workspace


def prefill_pass(layers, h, gamma1, gamma2, eps=1e-6, workspace=None, stream=None):
    """The batched prefill pass: h [B][hidden] updated in place through every layer.
    ``layers`` is a PassLayers (or a list of {slot: (codes, params)}); gamma1/gamma2
    [L][hidden].  Returns the workspace (it holds the last layer's intermediates)."""
    if not isinstance(layers, PassLayers):
        layers = PassLayers(layers)
    _need(h, torch.float32, "h")
    B, H = h.shape
    L = len(layers.layers)
    _need(gamma1, torch.float32, "gamma1", (L, H))
    _need(gamma2, torch.float32, "gamma2", (L, H))
    if workspace is None:
        workspace = prefill_pass_workspace(layers.hidden, layers.kv, layers.inter, B, h.device)
    _check(lib().pgq_q8_prefill_pass(layers.arr, L, _ptr(h), B, _ptr(gamma1), _ptr(gamma2), eps,
                                     _ptr(workspace), workspace.numel(), _stream(stream)))
    return workspace


# ------------------------------------------------------------------ MoE
def moe_router(R, n, logits=None, stream=None):
    _need(R, torch.float32, "R")
    E, cols = R.shape
    _need(n, torch.float32, "n")
    B = n.shape[0]
    logits = torch.empty(B, E, dtype=torch.float32, device=R.device) if logits is None else logits
    _need(logits, torch.float32, "logits", (B, E))
    _check(lib().pgq_moe_router(_ptr(R), E, cols, _ptr(n), B, _ptr(logits), _stream(stream)))
    return logits


def moe_route_topk(logits, k, renorm=False, stream=None):
    _need(logits, torch.float32, "logits")
    B, E = logits.shape
    sel = torch.empty(B, k, dtype=torch.int32, device=logits.device)
    w = torch.empty(B, k, dtype=torch.float32, device=logits.device)
    _check(lib().pgq_moe_route_topk(_ptr(logits), B, E, k, int(renorm), _ptr(sel), _ptr(w), _stream(stream)))
    return sel, w


def moe_group_gather(sel, E, x=None, xdiv=1, stream=None):
    _need(sel, torch.int32, "sel")
    B, k = sel.shape
    dev = sel.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    entries = torch.empty(B * k, dtype=torch.int32, device=dev)
    xg = None
    n = 0
    if x is not None:
        _need(x, torch.float32, "x")
        n = x.shape[1]
        xg = torch.empty(B * k, n, dtype=torch.float32, device=dev)
    _check(lib().pgq_moe_group_gather(_ptr(sel), B, k, E, _ptr(counts), _ptr(offsets), _ptr(entries), _ptr(x), n,
                                      xdiv, _ptr(xg), _stream(stream)))
    return counts, offsets, entries, xg


def moe_experts_q8(codes, params, counts, offsets, entries, x, xdiv, y, epilogue="none", stream=None):
    _need(codes, torch.int8, "codes")
    E, rows, cols = codes.shape
    _need(params, torch.float16, "params", (E, rows, cols // QBLOCK, 2))
    _need(x, torch.float32, "x")
    _need(y, torch.float32, "y")
    _check(lib().pgq_moe_experts_q8(_ptr(codes), _ptr(params), E, rows, cols, _ptr(counts), _ptr(offsets),
                                    _ptr(entries), entries.numel(), _ptr(x), xdiv, _ptr(y), _epi(epilogue),
                                    _stream(stream)))
    return y


def moe_combine_rmsnorm(h, eo, w, gamma, eps=1e-6, o=None, y=None, inv=None, stream=None):
    _need(h, torch.float32, "h")
    B, n = h.shape
    k = w.shape[1]
    y = torch.empty_like(h) if y is None else y
    _check(lib().pgq_moe_combine_rmsnorm(_ptr(h), _ptr(o), _ptr(eo), _ptr(w), k, _ptr(gamma), eps, B, n, _ptr(y),
                                         _ptr(inv), _stream(stream)))
    return y


class MoeWeights:
    """ctypes view of an MoE layer (keeps the tensors alive)."""

    def __init__(self, router, up_codes, up_params, down_codes, down_params, k, renorm=False):
        self.t = (router, up_codes, up_params, down_codes, down_params)
        E, inter, hidden = up_codes.shape
        _need(router, torch.float32, "router", (E, hidden))
        _need(down_codes, torch.int8, "down_codes", (E, hidden, inter))
        self.s = MoeLayer(router.data_ptr(), up_codes.data_ptr(), up_params.data_ptr(), down_codes.data_ptr(),
                          down_params.data_ptr(), E, k, hidden, inter, int(renorm))


class MoeQ82Weights:
    """ctypes view of an MoE layer with q8_2f experts (keeps the tensors alive)."""

    def __init__(self, router, up, down, k, renorm=False):
        (uc, urs, ucf), (dc, drs, dcf) = up, down
        self.t = (router, uc, urs, ucf, dc, drs, dcf)
        E, inter, hidden = uc.shape
        _need(router, torch.float32, "router", (E, hidden))
        _need(urs, torch.float16, "up_row_scale", (E, inter))
        _need(ucf, torch.float16, "up_col_field", (E, hidden))
        _need(dc, torch.int8, "down_codes", (E, hidden, inter))
        _need(drs, torch.float16, "down_row_scale", (E, hidden))
        _need(dcf, torch.float16, "down_col_field", (E, inter))
        self.s = MoeQ82Layer(router.data_ptr(), uc.data_ptr(), urs.data_ptr(), ucf.data_ptr(), dc.data_ptr(),
                             drs.data_ptr(), dcf.data_ptr(), E, k, hidden, inter, int(renorm))


def _moe_q82(W):
    return isinstance(W, MoeQ82Weights)


def moe_layer_workspace(W, B, device="cuda"):
    f = lib().pgq_moe_q82f_layer_workspace_bytes if _moe_q82(W) else lib().pgq_moe_layer_workspace_bytes
    n = int(f(C.byref(W.s), B))
    return torch.empty(n, dtype=torch.uint8, device=device)


def moe_layer_taps(W, workspace, B):
    off = (C.c_size_t * 9)()
    f = lib().pgq_moe_q82f_layer_layout if _moe_q82(W) else lib().pgq_moe_layer_layout
    _check(f(C.byref(W.s), B, off))
    s = W.s
    nb = B * s.k
    spec = [("n", torch.float32, (B, s.hidden)), ("logits", torch.float32, (B, s.E)), ("sel", torch.int32, (B, s.k)),
            ("w", torch.float32, (B, s.k)), ("counts", torch.int32, (s.E,)), ("offsets", torch.int32, (s.E + 1,)),
            ("entries", torch.int32, (nb,)), ("u", torch.float32, (nb, s.inter)), ("eo", torch.float32, (nb, s.hidden))]
    out = {}
    for (name, dt, shape), o in zip(spec, off):
        cnt = 1
        for d in shape:
            cnt *= d
        out[name] = workspace[o:o + cnt * 4].view(dt).view(*shape)
    return out


def moe_prefill_layer(W, h, gamma1, gamma2, eps=1e-6, y=None, workspace=None, stream=None):
    """One MoE layer over the pass h [B][hidden] (h updated in place); returns (y, workspace).
    W: MoeWeights (block-format experts) or MoeQ82Weights (q8_2f experts)."""
    _need(h, torch.float32, "h")
    B = h.shape[0]
    y = torch.empty_like(h) if y is None else y
    if workspace is None:
        workspace = moe_layer_workspace(W, B, h.device)
    f = lib().pgq_moe_q82f_prefill_layer if _moe_q82(W) else lib().pgq_moe_prefill_layer
    _check(f(C.byref(W.s), _ptr(h), B, _ptr(gamma1), _ptr(gamma2), eps, _ptr(y), _ptr(workspace), workspace.numel(),
             _stream(stream)))
    return y, workspace
