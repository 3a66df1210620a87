"""ctypes binding of libloglinear.so: argument marshalling only.

Every step of the forward and of the decode step runs in the library's CUDA kernels;
this module checks tensor placement / dtype / contiguity, allocates outputs and the
forward's workspace with PyTorch (device memory is PyTorch's job here), passes raw
pointers and sizes to the C ABI on the current CUDA stream, and turns a non-zero status
into an exception.  If the library is missing the import fails loudly: there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libloglinear.so")

LL_OK, LL_ERR_INVALID, LL_ERR_SHAPE, LL_ERR_DTYPE, LL_ERR_UNSUPPORTED, LL_ERR_CUDA, \
    LL_ERR_WORKSPACE, LL_ERR_ALIGN = range(8)
LL_F32, LL_BF16 = 0, 1
LL_PATH_AUTO, LL_PATH_SIMT, LL_PATH_TC = 0, 1, 2
PATHS = {"auto": LL_PATH_AUTO, "simt": LL_PATH_SIMT, "tc": LL_PATH_TC}

class LLStrides(ctypes.Structure):
    """ll_strides: element strides of the batch, position and head dimensions."""
    _fields_ = [("b", ctypes.c_int64), ("t", ctypes.c_int64), ("h", ctypes.c_int64)]


# Every symbol include/loglinear.h declares, with its ctypes signature.
_i64, _int, _vp, _sz = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t
_sp = ctypes.POINTER(LLStrides)
SIGNATURES = {
    "loglinear_version": (_int, []),
    "loglinear_status_string": (ctypes.c_char_p, [_int]),
    "loglinear_last_cuda_error": (ctypes.c_char_p, []),
    "loglinear_fwd_resolve_path": (_int, [_i64, _i64, _int, _int, _int]),
    "loglinear_fwd_workspace_size": (_int, [_i64, _i64, _i64, _i64, _i64, _int, _int, _int,
                                            ctypes.POINTER(_sz)]),
    "loglinear_fwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64, _i64,
                             _i64, _int, _int, _int, _int, _vp, _sz, _vp]),
    "loglinear_fwd_strided": (_int, [_vp, _sp, _vp, _sp, _vp, _sp, _vp, _vp, _vp, _sp, _i64, _i64,
                                     _i64, _i64, _i64, _i64, _i64, _int, _int, _int, _int, _vp,
                                     _sz, _vp]),
    "loglinear_prefill_with_events": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64,
                                             _i64, _i64, _i64, _i64, _int, _int, _int, _int, _vp,
                                             _sz, _vp, ctypes.POINTER(_vp), _int,
                                             ctypes.POINTER(_int)]),
    "loglinear_fwd_with_events": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                         _i64, _i64, _i64, _int, _int, _int, _int, _vp, _sz, _vp,
                                         ctypes.POINTER(_vp), _int, ctypes.POINTER(_int)]),
    "loglinear_decode_step": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _i64, _i64, _i64,
                                     _i64, _i64, _i64, _int, _int, _vp]),
    "loglinear_gdn_decode_step": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _vp, _i64, _i64,
                                         _i64, _i64, _i64, _i64, _int, _int, _vp]),
    "loglinear_gdn_fwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                 _i64, _i64, _i64, _int, _int, _vp]),
    "loglinear_gdn_fwd_chunked_workspace_size": (_int, [_i64, _i64, _i64, _i64, _i64,
                                                        ctypes.POINTER(ctypes.c_size_t)]),
    "loglinear_gdn_fwd_chunked": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64,
                                         _i64, _i64, _i64, _i64, _i64, _int, _int, _vp, _sz,
                                         _vp]),
    "loglinear_debug_level_map": (_int, [_i64, _int, _int, _vp, _vp]),
    "loglinear_device_error": (_int, [_vp, ctypes.POINTER(ctypes.c_uint)]),
    "loglinear_fwd_noalloc": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                     _i64, _i64, _int, _int, _int, _int, _vp]),
    "loglinear_prefill": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i64,
                                 _i64, _i64, _int, _int, _int, _int, _vp, _sz, _vp]),
    "loglinear_bwd_workspace_size": (_int, [_i64, _i64, _i64, _i64, _i64, _i64, _i64, _int, _int,
                                            _int, ctypes.POINTER(_sz)]),
    "loglinear_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64,
                             _i64, _i64, _i64, _i64, _i64, _int, _int, _int, _vp, _sz, _vp, _sz,
                             _vp]),
}


class LoglinearError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = f"{where}: {status_string(status)}"
        if status == LL_ERR_CUDA:
            msg += f" ({_lib.loglinear_last_cuda_error().decode()})"
        super().__init__(msg)
        self.status = status


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(
            f"{path} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


_lib = load_library()


def lib() -> ctypes.CDLL:
    return _lib


def status_string(status: int) -> str:
    return _lib.loglinear_status_string(int(status)).decode()


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.float32:
        return LL_F32
    if t.dtype == torch.bfloat16:
        return LL_BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check_dev(name, t, dtype=None, shape=None, strided=False):
    """Device, dtype and shape checks; contiguity, or with strided=True only a contiguous
    last dimension (the others are passed as strides)."""
    if t is None:
        return
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if strided:
        if t.dim() != 4 or (t.shape[-1] > 1 and t.stride(-1) != 1):
            raise ValueError(f"{name} must have a contiguous last dimension")
    elif not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def resolve_path(dk, dv, chunk, in_dtype, path="auto") -> str:
    r = _lib.loglinear_fwd_resolve_path(dk, dv, chunk, in_dtype, PATHS[path])
    if r < 0:
        raise LoglinearError(-r, "loglinear_fwd_resolve_path")
    return {LL_PATH_SIMT: "simt", LL_PATH_TC: "tc"}[r]


def fwd_workspace_size(B, T, H, dk, dv, chunk, in_dtype, path="auto") -> int:
    out = ctypes.c_size_t(0)
    st = _lib.loglinear_fwd_workspace_size(B, T, H, dk, dv, chunk, in_dtype, PATHS[path],
                                           ctypes.byref(out))
    if st != LL_OK:
        raise LoglinearError(st, "loglinear_fwd_workspace_size")
    return int(out.value)


def loglinear_fwd(q, k, v, log_a, lam, chunk, out=None, out_dtype=None, workspace=None,
                  path="auto", stream=None):
    """O = (Q K^T ⊙ M^S ⊙ M^H) V through the C ABI (q, k [B,T,Hqk,dk]; v [B,T,H,dv];
    log_a [B,T,H] fp32 or None; lam [B,T,H,L] fp32; head h reads q/k head h // (H/Hqk)).
    q, k, v and out may be strided views with a contiguous last dimension (e.g. slices of
    a fused q/k/v projection); they then go through loglinear_fwd_strided.
    Returns out [B,T,H,dv]."""
    B, T, Hqk, dk = q.shape
    H, dv, L = v.shape[2], v.shape[-1], lam.shape[-1]
    _check_dev("q", q, shape=(B, T, Hqk, dk), strided=True)
    _check_dev("k", k, q.dtype, (B, T, Hqk, dk), strided=True)
    _check_dev("v", v, q.dtype, (B, T, H, dv), strided=True)
    _check_dev("log_a", log_a, torch.float32, (B, T, H))
    _check_dev("lam", lam, torch.float32, (B, T, H, L))
    in_dt = _dtype_code(q)
    if out is None:
        out = torch.empty(B, T, H, dv, device=q.device, dtype=out_dtype or q.dtype)
    _check_dev("out", out, shape=(B, T, H, dv), strided=True)
    ws_bytes = fwd_workspace_size(B, T, H, dk, dv, chunk, in_dt, path)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), device=q.device, dtype=torch.uint8)
    _check_dev("workspace", workspace, torch.uint8)
    if all(x.is_contiguous() for x in (q, k, v, out)):
        st = _lib.loglinear_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(lam), _ptr(out),
                                B, T, H, Hqk, dk, dv, L, chunk, in_dt, _dtype_code(out),
                                PATHS[path], _ptr(workspace), workspace.numel(), _stream(stream))
    else:
        sd = [ctypes.byref(LLStrides(*x.stride()[:3])) for x in (q, k, v, out)]
        st = _lib.loglinear_fwd_strided(_ptr(q), sd[0], _ptr(k), sd[1], _ptr(v), sd[2],
                                        _ptr(log_a), _ptr(lam), _ptr(out), sd[3], B, T, H, Hqk, dk,
                                        dv, L, chunk, in_dt, _dtype_code(out), PATHS[path],
                                        _ptr(workspace), workspace.numel(), _stream(stream))
    if st != LL_OK:
        raise LoglinearError(st, "loglinear_fwd")
    return out


def loglinear_fwd_with_events(q, k, v, log_a, lam, chunk, events, out, workspace, path="auto",
                              stream=None):
    """loglinear_fwd plus torch.cuda.Event records between its kernels (events are
    created with enable_timing=True by the caller).  Returns the number of kernels."""
    B, T, Hqk, dk = q.shape
    H, dv, L = v.shape[2], v.shape[-1], lam.shape[-1]
    st_ = stream if stream is not None else torch.cuda.current_stream()
    for e in events:          # torch creates the CUDA event lazily, on its first record
        if not e.cuda_event:
            e.record(st_)
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    nk = ctypes.c_int(0)
    st = _lib.loglinear_fwd_with_events(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(lam),
                                        _ptr(out), B, T, H, Hqk, dk, dv, L, chunk, _dtype_code(q),
                                        _dtype_code(out), PATHS[path], _ptr(workspace),
                                        workspace.numel(), _stream(stream), arr, len(events),
                                        ctypes.byref(nk))
    if st != LL_OK:
        raise LoglinearError(st, "loglinear_fwd_with_events")
    return nk.value


def loglinear_decode_step(state, q, k, v, log_a, lam, t, out=None, out_dtype=None, stream=None):
    """One lssb decode step at position t; updates state [B,H,L,dk,dv] (fp32) in place
    and returns out [B,H,dv].  q, k [B,Hqk,dk] (head h reads q/k head h // (H/Hqk))."""
    B, H, L, dk, dv = state.shape
    Hqk = q.shape[1]
    _check_dev("state", state, torch.float32)
    _check_dev("q", q, shape=(B, Hqk, dk))
    _check_dev("k", k, q.dtype, (B, Hqk, dk))
    _check_dev("v", v, q.dtype, (B, H, dv))
    _check_dev("log_a", log_a, torch.float32, (B, H))
    _check_dev("lam", lam, torch.float32, (B, H, L))
    if out is None:
        out = torch.empty(B, H, dv, device=q.device, dtype=out_dtype or q.dtype)
    _check_dev("out", out, shape=(B, H, dv))
    st = _lib.loglinear_decode_step(_ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(log_a),
                                    _ptr(lam), int(t), _ptr(out), B, H, Hqk, dk, dv, L, _dtype_code(q),
                                    _dtype_code(out), _stream(stream))
    if st != LL_OK:
        raise LoglinearError(st, "loglinear_decode_step")
    return out


def loglinear_gdn_decode_step(state, q, k, v, log_a, beta, lam, t, out=None, out_dtype=None,
                              stream=None):
    """One Log-Linear Gated DeltaNet decode step at position t; updates state [B,H,L,dk,dv]
    (fp32) in place and returns out [B,H,dv].  q, k [B,Hqk,dk]; beta [B,H] fp32."""
    B, H, L, dk, dv = state.shape
    Hqk = q.shape[1]
    _check_dev("state", state, torch.float32)
    _check_dev("q", q, shape=(B, Hqk, dk))
    _check_dev("k", k, q.dtype, (B, Hqk, dk))
    _check_dev("v", v, q.dtype, (B, H, dv))
    _check_dev("log_a", log_a, torch.float32, (B, H))
    _check_dev("beta", beta, torch.float32, (B, H))
    _check_dev("lam", lam, torch.float32, (B, H, L))
    if out is None:
        out = torch.empty(B, H, dv, device=q.device, dtype=out_dtype or q.dtype)
    _check_dev("out", out, shape=(B, H, dv))
    st = _lib.loglinear_gdn_decode_step(_ptr(state), _ptr(q), _ptr(k), _ptr(v), _ptr(log_a),
                                        _ptr(beta), _ptr(lam), int(t), _ptr(out), B, H, Hqk, dk,
                                        dv, L, _dtype_code(q), _dtype_code(out), _stream(stream))
    if st != LL_OK:
        raise LoglinearError(st, "loglinear_gdn_decode_step")
    return out


def loglinear_gdn_fwd(q, k, v, log_a, beta, lam, out=None, out_dtype=None, state=None,
                      stream=None):
    """Log-Linear Gated DeltaNet over a whole sequence (recurrent form).  q, k [B,T,Hqk,dk];
    v [B,T,H,dv]; log_a [B,T,H] fp32 or None; beta [B,T,H] fp32; lam [B,T,H,L] fp32.
    Returns out [B,T,H,dv]; when `state` ([B,H,L,dk,dv] fp32) is given it receives the
    per-level state after position T-1."""
    B, T, Hqk, dk = q.shape
    H, dv, L = v.shape[2], v.shape[-1], lam.shape[-1]
    _check_dev("q", q)
    _check_dev("k", k, q.dtype, (B, T, Hqk, dk))
    _check_dev("v", v, q.dtype, (B, T, H, dv))
    _check_dev("log_a", log_a, torch.float32, (B, T, H))
    _check_dev("beta", beta, torch.float32, (B, T, H))
    _check_dev("lam", lam, torch.float32, (B, T, H, L))
    if state is not None:
        _check_dev("state", state, torch.float32, (B, H, L, dk, dv))
    if out is None:
        out = torch.empty(B, T, H, dv, device=q.device, dtype=out_dtype or q.dtype)
    _check_dev("out", out, shape=(B, T, H, dv))
    st = _lib.loglinear_gdn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(beta), _ptr(lam),
                                _ptr(out), _ptr(state), B, T, H, Hqk, dk, dv, L, _dtype_code(q),
                                _dtype_code(out), _stream(stream))
    if st != LL_OK:
        raise LoglinearError(st, "loglinear_gdn_fwd")
    return out


def gdn_fwd_chunked_workspace_size(B, T, H, dk, dv) -> int:
    out = ctypes.c_size_t(0)
    st = _lib.loglinear_gdn_fwd_chunked_workspace_size(B, T, H, dk, dv, ctypes.byref(out))
    if st != LL_OK:
        raise LoglinearError(st, "loglinear_gdn_fwd_chunked_workspace_size")
    return int(out.value)


def loglinear_gdn_fwd_chunked(q, k, v, log_a, beta, lam, out=None, out_dtype=None,
                              workspace=None, state=None, stream=None):
    """Log-Linear Gated DeltaNet over a whole sequence in chunks of 64 tokens (same inputs and
    output as loglinear_gdn_fwd; `state`, [B,H,L,dk,dv] fp32, receives the decode state after
    T-1 when given).  The workspace is allocated with torch when not given."""
    B, T, Hqk, dk = q.shape
    H, dv, L = v.shape[2], v.shape[-1], lam.shape[-1]
    _check_dev("q", q)
    _check_dev("k", k, q.dtype, (B, T, Hqk, dk))
    _check_dev("v", v, q.dtype, (B, T, H, dv))
    _check_dev("log_a", log_a, torch.float32, (B, T, H))
    _check_dev("beta", beta, torch.float32, (B, T, H))
    _check_dev("lam", lam, torch.float32, (B, T, H, L))
    if state is not None:
        _check_dev("state", state, torch.float32, (B, H, L, dk, dv))
    if out is None:
        out = torch.empty(B, T, H, dv, device=q.device, dtype=out_dtype or q.dtype)
    _check_dev("out", out, shape=(B, T, H, dv))
    sz = ctypes.c_size_t(0)
    st = _lib.loglinear_gdn_fwd_chunked_workspace_size(B, T, H, dk, dv, ctypes.byref(sz))
    if st != LL_OK:
        raise LoglinearError(st, "loglinear_gdn_fwd_chunked_workspace_size")
    if workspace is None:
        workspace = torch.empty(max(sz.value, 1), device=q.device, dtype=torch.uint8)
    st = _lib.loglinear_gdn_fwd_chunked(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(beta),
                                        _ptr(lam), _ptr(out), _ptr(state), B, T, H, Hqk, dk, dv,
                                        L,
                                        _dtype_code(q), _dtype_code(out), _ptr(workspace),
                                        workspace.numel(), _stream(stream))
    if st != LL_OK:
        raise LoglinearError(st, "loglinear_gdn_fwd_chunked")
    return out


def loglinear_prefill_with_events(q, k, v, log_a, lam, chunk, events, out, state, workspace,
                                  path="auto", stream=None):
    """loglinear_prefill plus torch.cuda.Event records between its kernels (the last
    kernel forms the decode state).  Returns the number of kernels."""
    B, T, Hqk, dk = q.shape
    H, dv, L = v.shape[2], v.shape[-1], lam.shape[-1]
    st_ = stream if stream is not None else torch.cuda.current_stream()
    for e in events:          # torch creates the CUDA event lazily, on its first record
        if not e.cuda_event:
            e.record(st_)
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    nk = ctypes.c_int(0)
    st = _lib.loglinear_prefill_with_events(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(lam),
                                            _ptr(out), _ptr(state), B, T, H, Hqk, dk, dv, L,
                                            chunk, _dtype_code(q), _dtype_code(out), PATHS[path],
                                            _ptr(workspace), workspace.numel(), _stream(stream),
                                            arr, len(events), ctypes.byref(nk))
    if st != LL_OK:
        raise LoglinearError(st, "loglinear_prefill_with_events")
    return nk.value


def loglinear_prefill(q, k, v, log_a, lam, chunk, out=None, state=None, out_dtype=None,
                      workspace=None, path="auto", stream=None):
    """loglinear_fwd over the prompt plus the per-level decode state at its last position
    (fp32 [B, H, L, dk, dv]), ready for loglinear_decode_step at t = T.
    Returns (out, state).  q/k heads as in loglinear_fwd."""
    B, T, Hqk, dk = q.shape
    H, dv, L = v.shape[2], v.shape[-1], lam.shape[-1]
    _check_dev("q", q, shape=(B, T, Hqk, dk))
    _check_dev("k", k, q.dtype, (B, T, Hqk, dk))
    _check_dev("v", v, q.dtype, (B, T, H, dv))
    _check_dev("log_a", log_a, torch.float32, (B, T, H))
    _check_dev("lam", lam, torch.float32, (B, T, H, L))
    in_dt = _dtype_code(q)
    if out is None:
        out = torch.empty(B, T, H, dv, device=q.device, dtype=out_dtype or q.dtype)
    if state is None:
        state = torch.empty(B, H, L, dk, dv, device=q.device, dtype=torch.float32)
    _check_dev("out", out, shape=(B, T, H, dv))
    _check_dev("state", state, torch.float32, (B, H, L, dk, dv))
    ws_bytes = fwd_workspace_size(B, T, H, dk, dv, chunk, in_dt, path) if T > 0 else 0
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), device=q.device, dtype=torch.uint8)
    _check_dev("workspace", workspace, torch.uint8)
    st = _lib.loglinear_prefill(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(lam), _ptr(out),
                                _ptr(state), B, T, H, Hqk, dk, dv, L, chunk, in_dt, _dtype_code(out),
                                PATHS[path], _ptr(workspace), workspace.numel(), _stream(stream))
    if st != LL_OK:
        raise LoglinearError(st, "loglinear_prefill")
    return out, state


def loglinear_fwd_noalloc(q, k, v, log_a, lam, chunk, out, path="auto", stream=None):
    """loglinear_fwd without a workspace, for callers that cannot allocate device memory:
    the scratch is the library's fixed device array (see include/loglinear.h).  `out` is
    caller-provided; nothing is allocated here either."""
    B, T, Hqk, dk = q.shape
    H, dv, L = v.shape[2], v.shape[-1], lam.shape[-1]
    for name, t in (("q", q), ("k", k), ("v", v), ("log_a", log_a), ("lam", lam), ("out", out)):
        _check_dev(name, t)
    st = _lib.loglinear_fwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(lam), _ptr(out),
                                    B, T, H, Hqk, dk, dv, L, chunk, _dtype_code(q), _dtype_code(out),
                                    PATHS[path], _stream(stream))
    if st != LL_OK:
        raise LoglinearError(st, "loglinear_fwd_noalloc")
    return out


def bwd_workspace_size(B, T, H, Hqk, dk, dv, L, in_dtype, grad_dtype, path="auto") -> int:
    out = ctypes.c_size_t(0)
    st = _lib.loglinear_bwd_workspace_size(B, T, H, Hqk, dk, dv, L, in_dtype, grad_dtype,
                                           PATHS[path], ctypes.byref(out))
    if st != LL_OK:
        raise LoglinearError(st, "loglinear_bwd_workspace_size")
    return int(out.value)


def loglinear_bwd(q, k, v, log_a, lam, dout, workspace=None, path="auto", fwd_workspace=None,
                  stream=None):
    """Gradients of sum(dout ⊙ O) for O = loglinear_fwd(q, k, v, log_a, lam): returns
    (dq, dk, dv, dlog_a, dlam); dq, dk, dv in dout's dtype, dlog_a (None without decay)
    and dlam fp32.  path: "tc" computes dq and dlam on the tensor cores (bf16, d_k = 128,
    d_v in {64, 128}), "simt" everything on CUDA cores, "auto" the tensor cores if they
    apply.  fwd_workspace: the workspace of a tensor-core loglinear_fwd over the same
    inputs, whose block states are then read instead of recomputed."""
    B, T, Hqk, dk = q.shape
    H, dv, L = v.shape[2], v.shape[-1], lam.shape[-1]
    _check_dev("q", q, shape=(B, T, Hqk, dk))
    _check_dev("k", k, q.dtype, (B, T, Hqk, dk))
    _check_dev("v", v, q.dtype, (B, T, H, dv))
    _check_dev("log_a", log_a, torch.float32, (B, T, H))
    _check_dev("lam", lam, torch.float32, (B, T, H, L))
    _check_dev("dout", dout, shape=(B, T, H, dv))
    in_dt, g_dt = _dtype_code(q), _dtype_code(dout)
    dq = torch.empty_like(q, dtype=dout.dtype)
    dk_ = torch.empty_like(k, dtype=dout.dtype)
    dv_ = torch.empty_like(v, dtype=dout.dtype)
    dla = None if log_a is None else torch.empty_like(log_a)
    dlam = torch.empty_like(lam)
    ws_bytes = bwd_workspace_size(B, T, H, Hqk, dk, dv, L, in_dt, g_dt, path)
    if workspace is None:
        workspace = torch.empty(max(ws_bytes, 1), device=q.device, dtype=torch.uint8)
    _check_dev("workspace", workspace, torch.uint8)
    if fwd_workspace is not None:
        _check_dev("fwd_workspace", fwd_workspace, torch.uint8)
    st = _lib.loglinear_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(log_a), _ptr(lam), _ptr(dout),
                            _ptr(dq), _ptr(dk_), _ptr(dv_), _ptr(dla), _ptr(dlam), B, T, H, Hqk,
                            dk, dv, L, in_dt, g_dt, PATHS[path], _ptr(fwd_workspace),
                            0 if fwd_workspace is None else fwd_workspace.numel(),
                            _ptr(workspace), workspace.numel(), _stream(stream))
    if st != LL_OK:
        raise LoglinearError(st, "loglinear_bwd")
    return dq, dk_, dv_, dla, dlam


def device_error(stream=None) -> int:
    """Reads and clears the tensor-core path's device error word (0 = no bounded wait
    ran out of time).  Synchronises the stream."""
    flags = ctypes.c_uint(0)
    st = _lib.loglinear_device_error(_stream(stream), ctypes.byref(flags))
    if st != LL_OK:
        raise LoglinearError(st, "loglinear_device_error")
    return int(flags.value)


def debug_level_map(T, chunk, path="auto", stream=None):
    """[T, T] int8 map of the level the forward's decomposition gives each (t, s)."""
    out = torch.empty(T, T, device="cuda", dtype=torch.int8)
    st = _lib.loglinear_debug_level_map(T, chunk, PATHS[path], _ptr(out), _stream(stream))
    if st != LL_OK:
        raise LoglinearError(st, "loglinear_debug_level_map")
    return out
