"""Python binding of the GB300 Sparse Delta Memory forward-step library.

Thin ctypes marshalling over ``_build/libsdm_gb300.so`` (the C ABI in
``include/sdm.h``): every function here has the name of the C entry point it
calls, checks that tensors are CUDA tensors on the current device, contiguous,
of the right dtype and at least as large as the shape implies, and passes
device pointers and the current CUDA stream.  All arithmetic runs in
the library's kernels; there is no CPU fallback.  If the library is not
built, importing works but every call raises ``SdmUnavailable``.
"""
from __future__ import annotations

import ctypes
import os

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "_build", "libsdm_gb300.so")

SDM_F32, SDM_BF16 = 0, 1
SDM_SCORE_DOT, SDM_SCORE_IDW = 0, 1
SDM_UPDATE_EQ4, SDM_UPDATE_SHARED_RESIDUAL = 0, 1

STATUS = {0: "SDM_OK", 1: "SDM_ERR_INVALID_ARG", 2: "SDM_ERR_UNSUPPORTED", 3: "SDM_ERR_CUDA",
          4: "SDM_ERR_TIMEOUT", 5: "SDM_ERR_DEVICE_BOUNDS", 6: "SDM_ERR_DUPLICATE_SLOT"}

EXPORTS = ["sdm_status_string", "sdm_subscores", "sdm_select", "sdm_address",
           "sdm_workspace_size", "sdm_scan", "sdm_scan_noalloc", "sdm_scan_logged",
           "sdm_undo_workspace_size", "sdm_scan_undo", "sdm_rmsnorm_gate", "sdm_decode",
           "sdm_forward", "sdm_forward_windows",
           "sdm_get_device_status",
           "sdm_set_scan_tuning", "sdm_selftest_wait_timeout", "sdm_measure_row_traffic"]


class SdmUnavailable(RuntimeError):
    """The CUDA library is not built or cannot be loaded."""


class SdmError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {STATUS.get(code, code)} ({status_string(code)})")


class Shape(ctypes.Structure):
    """Mirror of ``sdm_shape`` in include/sdm.h."""
    _fields_ = [("B", ctypes.c_int), ("H", ctypes.c_int), ("T", ctypes.c_int),
                ("n_sub", ctypes.c_int), ("d_h", ctypes.c_int), ("d_v", ctypes.c_int),
                ("W", ctypes.c_int), ("R", ctypes.c_int), ("k_w", ctypes.c_int),
                ("k_r", ctypes.c_int), ("in_dtype", ctypes.c_int), ("score", ctypes.c_int),
                ("idw_eps", ctypes.c_float), ("update", ctypes.c_int)]

    @property
    def N(self) -> int:
        return self.n_sub * self.n_sub

    def __repr__(self):
        return "Shape(" + ", ".join(f"{n}={getattr(self, n)}" for n, _ in self._fields_) + ")"


class Epilogue(ctypes.Structure):
    """Mirror of ``sdm_epilogue`` in include/sdm.h."""
    _fields_ = [("g", ctypes.c_void_p), ("gamma", ctypes.c_void_p), ("eps", ctypes.c_float),
                ("out", ctypes.c_void_p), ("out_dtype", ctypes.c_int)]


def make_shape(B, H, T, n_sub, d_h, d_v, W, R, k_w=0, k_r=0, in_dtype=SDM_BF16,
               score=SDM_SCORE_DOT, idw_eps=1e-3, update=SDM_UPDATE_EQ4) -> Shape:
    return Shape(B, H, T, n_sub, d_h, d_v, W, R, k_w, k_r, in_dtype, score, idw_eps, update)


_lib = None


def lib():
    """The loaded library (raises SdmUnavailable if it is missing)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise SdmUnavailable(
            f"{LIB_PATH} is not built; run `python -m sparse_state_linear_gb300.build_ext`")
    try:
        L = ctypes.CDLL(LIB_PATH)
    except OSError as e:
        raise SdmUnavailable(f"cannot load {LIB_PATH}: {e}") from e
    P, SP, I = ctypes.c_void_p, ctypes.POINTER(Shape), ctypes.c_int
    sig = {
        "sdm_status_string": ([I], ctypes.c_char_p),
        "sdm_subscores": ([SP, P, P, P, P], I),
        "sdm_select": ([SP, P, P, P, P, P, P, P], I),
        "sdm_address": ([SP, P, P, P, P, P, P, P, P], I),
        "sdm_workspace_size": ([SP], ctypes.c_size_t),
        "sdm_scan": ([SP] + [P] * 10 + [ctypes.c_size_t, P], I),
        "sdm_scan_noalloc": ([SP] + [P] * 10, I),
        "sdm_scan_logged": ([SP] + [P] * 11 + [ctypes.c_size_t, P], I),
        "sdm_undo_workspace_size": ([SP], ctypes.c_size_t),
        "sdm_scan_undo": ([SP, P, P, P, P, ctypes.c_size_t, P], I),
        "sdm_rmsnorm_gate": ([SP, P, P, P, ctypes.c_float, P, I, P], I),
        "sdm_decode": ([SP] + [P] * 12 + [ctypes.POINTER(Epilogue), P], I),
        "sdm_forward": ([SP] + [P] * 13 + [ctypes.c_size_t, P], I),
        "sdm_forward_windows": ([SP], I),
        "sdm_get_device_status": ([P], I),
        "sdm_set_scan_tuning": ([I, I], I),
        "sdm_selftest_wait_timeout": ([ctypes.c_longlong, P], I),
        "sdm_measure_row_traffic": ([P, P, ctypes.c_longlong, ctypes.c_longlong, I, I, I, I, I,
                                     ctypes.c_uint, P], I),
    }
    for name, (args, res) in sig.items():
        f = getattr(L, name)
        f.argtypes = args
        f.restype = res
    _lib = L
    return L


def status_string(code: int) -> str:
    try:
        return lib().sdm_status_string(int(code)).decode()
    except SdmUnavailable:
        return STATUS.get(code, "?")


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t: torch.Tensor | None, name: str, dtypes=None, numel: int | None = None):
    """Device pointer of `t` after checking that it is a contiguous CUDA
    tensor on the current device (the library launches there), of one of
    `dtypes`, with at least `numel` elements (the size the shape implies)."""
    if t is None:
        raise ValueError(f"{name} is required")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, but the current device is "
                         f"cuda:{torch.cuda.current_device()}; call under "
                         f"torch.cuda.device({t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtypes is not None and t.dtype not in dtypes:
        raise ValueError(f"{name} has dtype {t.dtype}, expected one of {dtypes}")
    if numel is not None and t.numel() < numel:
        raise ValueError(f"{name} has {t.numel()} elements, the shape needs {numel}")
    return ctypes.c_void_p(t.data_ptr())


def _sizes(sh: Shape):
    """Elements each argument needs for this shape."""
    bht = sh.B * sh.H * sh.T
    if bht == 0:               # no work: the library does not look at the pointers
        return dict.fromkeys(("q", "K", "S", "W", "R", "g", "v", "M", "y", "U", "gamma"), 0)
    return dict(q=bht * 2 * sh.d_h, K=sh.H * 2 * sh.n_sub * sh.d_h, S=bht * 2 * sh.n_sub,
                W=bht * sh.W, R=bht * sh.R, g=bht, v=bht * sh.d_v, M=sh.B * sh.H * sh.N * sh.d_v,
                y=bht * sh.d_v, U=bht * sh.W * sh.d_v, gamma=sh.H * sh.d_v)


def _in_dt(sh: Shape):
    return (torch.bfloat16,) if sh.in_dtype == SDM_BF16 else (torch.float32,)


def _ok(rc: int, what: str):
    if rc != 0:
        raise SdmError(rc, what)


def _empty(shape, dtype, like: torch.Tensor):
    return torch.empty(shape, dtype=dtype, device=like.device)


def sdm_subscores(sh: Shape, q, K, S=None, stream=None):
    """Sub-scores [B,H,T,2,s] float32 of one branch's half-queries q [B,H,T,2,d_h]."""
    if S is None:
        S = _empty((sh.B, sh.H, sh.T, 2, sh.n_sub), torch.float32, q)
    n = _sizes(sh)
    _ok(lib().sdm_subscores(ctypes.byref(sh), _ptr(q, "q", _in_dt(sh), n["q"]),
                            _ptr(K, "K", _in_dt(sh), n["K"]),
                            _ptr(S, "S", (torch.float32,), n["S"]), _stream(stream)),
        "sdm_subscores")
    return S


def _sel_outputs(sh: Shape, like, idx_w, wt_w, idx_r, wt_r):
    BHT = (sh.B, sh.H, sh.T)
    idx_w = _empty(BHT + (sh.W,), torch.int32, like) if idx_w is None else idx_w
    wt_w = _empty(BHT + (sh.W,), torch.float32, like) if wt_w is None else wt_w
    idx_r = _empty(BHT + (sh.R,), torch.int32, like) if idx_r is None else idx_r
    wt_r = _empty(BHT + (sh.R,), torch.float32, like) if wt_r is None else wt_r
    return idx_w, wt_w, idx_r, wt_r


def sdm_select(sh: Shape, sub_w, sub_r, idx_w=None, wt_w=None, idx_r=None, wt_r=None,
               stream=None):
    """Product-key selection from float32 sub-scores; returns (idx_w, wt_w, idx_r, wt_r)."""
    idx_w, wt_w, idx_r, wt_r = _sel_outputs(sh, sub_w, idx_w, wt_w, idx_r, wt_r)
    f32, i32, n = (torch.float32,), (torch.int32,), _sizes(sh)
    _ok(lib().sdm_select(ctypes.byref(sh), _ptr(sub_w, "sub_w", f32, n["S"]),
                         _ptr(sub_r, "sub_r", f32, n["S"]),
                         _ptr(idx_w, "idx_w", i32, n["W"]), _ptr(wt_w, "wt_w", f32, n["W"]),
                         _ptr(idx_r, "idx_r", i32, n["R"]), _ptr(wt_r, "wt_r", f32, n["R"]),
                         _stream(stream)),
        "sdm_select")
    return idx_w, wt_w, idx_r, wt_r


def sdm_address(sh: Shape, q_w, q_r, K, idx_w=None, wt_w=None, idx_r=None, wt_r=None,
                stream=None):
    """Fused sub-scores + selection; returns (idx_w, wt_w, idx_r, wt_r)."""
    idx_w, wt_w, idx_r, wt_r = _sel_outputs(sh, q_w, idx_w, wt_w, idx_r, wt_r)
    dt, f32, i32, n = _in_dt(sh), (torch.float32,), (torch.int32,), _sizes(sh)
    _ok(lib().sdm_address(ctypes.byref(sh), _ptr(q_w, "q_w", dt, n["q"]),
                          _ptr(q_r, "q_r", dt, n["q"]), _ptr(K, "K", dt, n["K"]),
                          _ptr(idx_w, "idx_w", i32, n["W"]), _ptr(wt_w, "wt_w", f32, n["W"]),
                          _ptr(idx_r, "idx_r", i32, n["R"]), _ptr(wt_r, "wt_r", f32, n["R"]),
                          _stream(stream)),
        "sdm_address")
    return idx_w, wt_w, idx_r, wt_r


def sdm_workspace_size(sh: Shape) -> int:
    """Bytes of device workspace sdm_scan / sdm_forward need for this shape."""
    return int(lib().sdm_workspace_size(ctypes.byref(sh)))


def _workspace(sh: Shape, like, workspace):
    n = sdm_workspace_size(sh)
    if workspace is None:
        workspace = torch.empty(max(n, 16), dtype=torch.uint8, device=like.device)
    return workspace, workspace.numel() * workspace.element_size()


def sdm_scan(sh: Shape, idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M, y=None, workspace=None,
             stream=None):
    """Write-then-read recurrence; M [B,H,N,d_v] float32 is updated in place; returns y."""
    if y is None:
        y = _empty((sh.B, sh.H, sh.T, sh.d_v), torch.float32, M)
    ws, nws = _workspace(sh, M, workspace)
    dt, f32, i32 = _in_dt(sh), (torch.float32,), (torch.int32,)
    n = _sizes(sh)
    _ok(lib().sdm_scan(ctypes.byref(sh), _ptr(idx_w, "idx_w", i32, n["W"]),
                       _ptr(wt_w, "wt_w", f32, n["W"]), _ptr(idx_r, "idx_r", i32, n["R"]),
                       _ptr(wt_r, "wt_r", f32, n["R"]), _ptr(alpha, "alpha", dt, n["g"]),
                       _ptr(beta, "beta", dt, n["g"]), _ptr(v, "v", dt, n["v"]),
                       _ptr(M, "M", f32, n["M"]), _ptr(y, "y", f32, n["y"]),
                       _ptr(ws, "workspace"), nws,
                       _stream(stream)), "sdm_scan")
    return y


def sdm_scan_noalloc(sh: Shape, idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M, y=None,
                     stream=None):
    """sdm_scan with the library's fixed scratch instead of a workspace (for
    callers that cannot allocate); M updated in place; returns y."""
    if y is None:
        y = _empty((sh.B, sh.H, sh.T, sh.d_v), torch.float32, M)
    dt, f32, i32 = _in_dt(sh), (torch.float32,), (torch.int32,)
    n = _sizes(sh)
    _ok(lib().sdm_scan_noalloc(ctypes.byref(sh), _ptr(idx_w, "idx_w", i32, n["W"]),
                               _ptr(wt_w, "wt_w", f32, n["W"]), _ptr(idx_r, "idx_r", i32, n["R"]),
                               _ptr(wt_r, "wt_r", f32, n["R"]),
                               _ptr(alpha, "alpha", dt, n["g"]), _ptr(beta, "beta", dt, n["g"]),
                               _ptr(v, "v", dt, n["v"]), _ptr(M, "M", f32, n["M"]),
                               _ptr(y, "y", f32, n["y"]), _stream(stream)), "sdm_scan_noalloc")
    return y


def sdm_scan_logged(sh: Shape, idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M, y=None,
                    undo=None, workspace=None, stream=None):
    """sdm_scan that also logs each step's pre-write rows; M updated in place.
    Returns (y, undo) with undo float32 [B,H,T,W,d_v]."""
    if y is None:
        y = _empty((sh.B, sh.H, sh.T, sh.d_v), torch.float32, M)
    if undo is None:
        undo = _empty((sh.B, sh.H, sh.T, sh.W, sh.d_v), torch.float32, M)
    ws, nws = _workspace(sh, M, workspace)
    dt, f32, i32 = _in_dt(sh), (torch.float32,), (torch.int32,)
    n = _sizes(sh)
    _ok(lib().sdm_scan_logged(ctypes.byref(sh), _ptr(idx_w, "idx_w", i32, n["W"]),
                              _ptr(wt_w, "wt_w", f32, n["W"]), _ptr(idx_r, "idx_r", i32, n["R"]),
                              _ptr(wt_r, "wt_r", f32, n["R"]),
                              _ptr(alpha, "alpha", dt, n["g"]), _ptr(beta, "beta", dt, n["g"]),
                              _ptr(v, "v", dt, n["v"]), _ptr(M, "M", f32, n["M"]),
                              _ptr(y, "y", f32, n["y"]), _ptr(undo, "undo", f32, n["U"]),
                              _ptr(ws, "workspace"),
                              nws, _stream(stream)), "sdm_scan_logged")
    return y, undo


def sdm_undo_workspace_size(sh: Shape) -> int:
    """Bytes of device workspace sdm_scan_undo needs for this shape."""
    return int(lib().sdm_undo_workspace_size(ctypes.byref(sh)))


def sdm_scan_undo(sh: Shape, idx_w, undo, M, workspace=None, stream=None):
    """Put M back to the table before the logged segment (in place); returns M."""
    if workspace is None:
        workspace = torch.empty(max(sdm_undo_workspace_size(sh), 16), dtype=torch.uint8,
                                device=M.device)
    nws = workspace.numel() * workspace.element_size()
    f32, i32 = (torch.float32,), (torch.int32,)
    n = _sizes(sh)
    _ok(lib().sdm_scan_undo(ctypes.byref(sh), _ptr(idx_w, "idx_w", i32, n["W"]),
                            _ptr(undo, "undo", f32, n["U"]), _ptr(M, "M", f32, n["M"]),
                            _ptr(workspace, "workspace"), nws, _stream(stream)),
        "sdm_scan_undo")
    return M


def sdm_rmsnorm_gate(sh: Shape, y, g, gamma=None, eps: float = 1e-6, out=None,
                     out_dtype=SDM_BF16, stream=None):
    """Per-head RMS-Norm and output gate on y [B,H,T,d_v] float32; g in the
    shape's input dtype; gamma [H,d_v] float32 or None.  Returns out."""
    tdt = torch.bfloat16 if out_dtype == SDM_BF16 else torch.float32
    if out is None:
        out = _empty((sh.B, sh.H, sh.T, sh.d_v), tdt, y)
    f32 = (torch.float32,)
    n = _sizes(sh)
    gp = None if gamma is None else _ptr(gamma, "gamma", f32, n["gamma"])
    _ok(lib().sdm_rmsnorm_gate(ctypes.byref(sh), _ptr(y, "y", f32, n["y"]),
                               _ptr(g, "g", _in_dt(sh), n["y"]), gp,
                               float(eps), _ptr(out, "out", (tdt,), n["y"]), int(out_dtype),
                               _stream(stream)), "sdm_rmsnorm_gate")
    return out


def sdm_decode(sh: Shape, q_w, q_r, K, alpha, beta, v, M, y=None, idx_w=None, wt_w=None,
               idx_r=None, wt_r=None, gate=None, gamma=None, eps: float = 1e-6, out=None,
               out_dtype=SDM_BF16, stream=None):
    """Fused forward for short sequences (decode); M updated in place.  With a
    gate, also the RMS-Norm + gate epilogue.  Returns dict(y, idx_w, wt_w,
    idx_r, wt_r, out)."""
    if y is None:
        y = _empty((sh.B, sh.H, sh.T, sh.d_v), torch.float32, M)
    idx_w, wt_w, idx_r, wt_r = _sel_outputs(sh, M, idx_w, wt_w, idx_r, wt_r)
    dt, f32, i32, n = _in_dt(sh), (torch.float32,), (torch.int32,), _sizes(sh)
    epi = None
    if gate is not None:
        tdt = torch.bfloat16 if out_dtype == SDM_BF16 else torch.float32
        if out is None:
            out = _empty((sh.B, sh.H, sh.T, sh.d_v), tdt, M)
        epi = Epilogue(_ptr(gate, "gate", dt, n["y"]).value,
                       None if gamma is None else _ptr(gamma, "gamma", f32, n["gamma"]).value,
                       float(eps), _ptr(out, "out", (tdt,), n["y"]).value, int(out_dtype))
    _ok(lib().sdm_decode(ctypes.byref(sh), _ptr(q_w, "q_w", dt, n["q"]),
                         _ptr(q_r, "q_r", dt, n["q"]), _ptr(K, "K", dt, n["K"]),
                         _ptr(alpha, "alpha", dt, n["g"]), _ptr(beta, "beta", dt, n["g"]),
                         _ptr(v, "v", dt, n["v"]), _ptr(M, "M", f32, n["M"]),
                         _ptr(y, "y", f32, n["y"]),
                         _ptr(idx_w, "idx_w", i32, n["W"]), _ptr(wt_w, "wt_w", f32, n["W"]),
                         _ptr(idx_r, "idx_r", i32, n["R"]), _ptr(wt_r, "wt_r", f32, n["R"]),
                         None if epi is None else ctypes.byref(epi), _stream(stream)),
        "sdm_decode")
    return dict(y=y, idx_w=idx_w, wt_w=wt_w, idx_r=idx_r, wt_r=wt_r, out=out)


def sdm_forward(sh: Shape, q_w, q_r, K, alpha, beta, v, M, y=None, idx_w=None, wt_w=None,
                idx_r=None, wt_r=None, workspace=None, stream=None):
    """Addressing then scan; M updated in place.  Returns dict(y, idx_w, wt_w, idx_r, wt_r)."""
    if y is None:
        y = _empty((sh.B, sh.H, sh.T, sh.d_v), torch.float32, M)
    idx_w, wt_w, idx_r, wt_r = _sel_outputs(sh, M, idx_w, wt_w, idx_r, wt_r)
    ws, nws = _workspace(sh, M, workspace)
    dt, f32, i32 = _in_dt(sh), (torch.float32,), (torch.int32,)
    n = _sizes(sh)
    _ok(lib().sdm_forward(ctypes.byref(sh), _ptr(q_w, "q_w", dt, n["q"]),
                          _ptr(q_r, "q_r", dt, n["q"]), _ptr(K, "K", dt, n["K"]),
                          _ptr(alpha, "alpha", dt, n["g"]), _ptr(beta, "beta", dt, n["g"]),
                          _ptr(v, "v", dt, n["v"]), _ptr(M, "M", f32, n["M"]),
                          _ptr(y, "y", f32, n["y"]),
                          _ptr(idx_w, "idx_w", i32, n["W"]), _ptr(wt_w, "wt_w", f32, n["W"]),
                          _ptr(idx_r, "idx_r", i32, n["R"]), _ptr(wt_r, "wt_r", f32, n["R"]),
                          _ptr(ws, "workspace"), nws, _stream(stream)), "sdm_forward")
    return dict(y=y, idx_w=idx_w, wt_w=wt_w, idx_r=idx_r, wt_r=wt_r)


def sdm_forward_windows(sh: Shape) -> int:
    """Step windows sdm_forward uses for this shape (1 = no overlap)."""
    return int(lib().sdm_forward_windows(ctypes.byref(sh)))


def sdm_get_device_status(stream=None) -> int:
    """Synchronize the stream, return and clear the device status code (0 = ok)."""
    return int(lib().sdm_get_device_status(_stream(stream)))


def sdm_set_scan_tuning(depth: int = 0, col_slice: int = 0):
    _ok(lib().sdm_set_scan_tuning(int(depth), int(col_slice)), "sdm_set_scan_tuning")


def sdm_selftest_wait_timeout(timeout_ns: int, stream=None):
    _ok(lib().sdm_selftest_wait_timeout(int(timeout_ns), _stream(stream)),
        "sdm_selftest_wait_timeout")


def sdm_measure_row_traffic(src, dst, col_slice: int, T: int, loads: int, stores: int,
                            seed: int = 1, stream=None) -> int:
    """Measurement reference: the scan's row traffic without its arithmetic
    on tables src, dst [chains, rows, d_v] float32; returns the bytes moved."""
    chains, rows, dv = src.shape
    if tuple(dst.shape) != (chains, rows, dv):
        raise ValueError("src and dst shapes differ")
    f32 = (torch.float32,)
    _ok(lib().sdm_measure_row_traffic(_ptr(src, "src", f32, src.numel()),
                                      _ptr(dst, "dst", f32, src.numel()), chains, rows, dv,
                                      col_slice, T, loads, stores, seed & 0xffffffff,
                                      _stream(stream)),
        "sdm_measure_row_traffic")
    return chains * dv * T * (loads + stores) * 4
