"""CPU oracle of the SDM forward step (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  It wraps ``sdm_oracle.cpp`` (plain,
single-threaded C++) with ctypes and numpy; it imports nothing from the CUDA
package, and the CUDA package imports nothing from here.

The arithmetic lives in the C++ file; this module only marshals arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sdm_oracle.cpp")
_LIB = os.path.join(_HERE, "_build", "libsdm_oracle.so")

__all__ = ["build", "Shape", "subscores", "select", "slot_weights", "scan", "forward"]


def build(force: bool = False) -> str:
    """Compile the oracle with g++ (-O2, no FMA contraction).  Returns the .so path."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "sdm_oracle.h"))
    ):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
           "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


class _CShape(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in
                ("B", "H", "T", "n_sub", "d_h", "d_v", "W", "R", "k_w", "k_r",
                 "score_kind")] + [("idw_eps", ctypes.c_double),
                                   ("update_form", ctypes.c_int)]


@dataclass
class Shape:
    B: int
    H: int
    T: int
    n_sub: int
    d_h: int
    d_v: int
    W: int
    R: int
    k_w: int = 0
    k_r: int = 0
    score_kind: int = 0      # 0 dot, 1 inverse distance
    idw_eps: float = 1e-3
    update_form: int = 0     # 0 Eq. (4) per slot, 1 Fig. 2 shared residual

    @property
    def N(self) -> int:
        return self.n_sub * self.n_sub

    def c(self) -> _CShape:
        return _CShape(self.B, self.H, self.T, self.n_sub, self.d_h, self.d_v,
                       self.W, self.R, self.k_w, self.k_r, self.score_kind,
                       float(self.idw_eps), self.update_form)


_lib = None


def _L():
    global _lib
    if _lib is None:
        _lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        sp = ctypes.POINTER(_CShape)
        _lib.sdm_ref_subscores.argtypes = [sp, P, P, P]
        _lib.sdm_ref_select.argtypes = [sp, ctypes.c_int, P, P, P, P]
        _lib.sdm_ref_slot_weights.argtypes = [sp, ctypes.c_int, P, P, P]
        _lib.sdm_ref_scan.argtypes = [sp] + [P] * 9
        _lib.sdm_ref_forward.argtypes = [sp] + [P] * 12
        _lib.sdm_ref_scan_logged.argtypes = [sp] + [P] * 10
        _lib.sdm_ref_undo.argtypes = [sp] + [P] * 3
        _lib.sdm_ref_rmsnorm_gate.argtypes = [sp, P, P, P, ctypes.c_double, P]
        for f in (_lib.sdm_ref_subscores, _lib.sdm_ref_select, _lib.sdm_ref_slot_weights,
                  _lib.sdm_ref_scan,
                  _lib.sdm_ref_forward, _lib.sdm_ref_scan_logged, _lib.sdm_ref_undo,
                  _lib.sdm_ref_rmsnorm_gate):
            f.restype = ctypes.c_int
    return _lib


def _arr(x, dtype):
    a = np.ascontiguousarray(np.asarray(x), dtype=dtype)
    return a


def _p(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _check(rc: int, what: str):
    if rc != 0:
        raise ValueError(f"oracle {what} rejected its arguments (code {rc})")


def subscores(sh: Shape, q, K) -> np.ndarray:
    """q [B,H,T,2,d_h], K [H,2,s,d_h] -> float32 S [B,H,T,2,s]."""
    q = _arr(q, np.float32)
    K = _arr(K, np.float32)
    assert q.shape == (sh.B, sh.H, sh.T, 2, sh.d_h), q.shape
    assert K.shape == (sh.H, 2, sh.n_sub, sh.d_h), K.shape
    S = np.empty((sh.B, sh.H, sh.T, 2, sh.n_sub), np.float32)
    cs = sh.c()
    _check(_L().sdm_ref_subscores(ctypes.byref(cs), _p(q), _p(K), _p(S)), "subscores")
    return S


def select(sh: Shape, which: int, S):
    """S [B,H,T,2,s] float32 -> (idx int32, score float32, wt float64) of shape [B,H,T,n]."""
    S = _arr(S, np.float32)
    assert S.shape == (sh.B, sh.H, sh.T, 2, sh.n_sub), S.shape
    n = sh.W if which == 0 else sh.R
    idx = np.empty((sh.B, sh.H, sh.T, n), np.int32)
    sc = np.empty((sh.B, sh.H, sh.T, n), np.float32)
    wt = np.empty((sh.B, sh.H, sh.T, n), np.float64)
    cs = sh.c()
    _check(_L().sdm_ref_select(ctypes.byref(cs), which, _p(S), _p(idx), _p(sc), _p(wt)),
           "select")
    return idx, sc, wt


def slot_weights(sh: Shape, which: int, S, idx) -> np.ndarray:
    """Softmax weights (float64 [B,H,T,n]) of the given slot lists idx
    [B,H,T,n] from float32 sub-scores S [B,H,T,2,s]: the oracle's weights for
    a selection made elsewhere."""
    S = _arr(S, np.float32)
    idx = _arr(idx, np.int32)
    n = sh.W if which == 0 else sh.R
    assert S.shape == (sh.B, sh.H, sh.T, 2, sh.n_sub), S.shape
    assert idx.shape == (sh.B, sh.H, sh.T, n), idx.shape
    wt = np.empty(idx.shape, np.float64)
    cs = sh.c()
    _check(_L().sdm_ref_slot_weights(ctypes.byref(cs), which, _p(S), _p(idx), _p(wt)),
           "slot_weights")
    return wt


def scan(sh: Shape, idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M0, log: bool = False):
    """Returns (M float64 [B,H,N,d_v], y float64 [B,H,T,d_v]); M0 is not modified.
    With log=True also the undo log float64 [B,H,T,W,d_v]: the value each
    written row had just before its step's write."""
    idx_w = _arr(idx_w, np.int32)
    idx_r = _arr(idx_r, np.int32)
    wt_w = _arr(wt_w, np.float64)
    wt_r = _arr(wt_r, np.float64)
    alpha = _arr(alpha, np.float32)
    beta = _arr(beta, np.float32)
    v = _arr(v, np.float32)
    M = np.array(M0, dtype=np.float64, order="C", copy=True)
    assert idx_w.shape == (sh.B, sh.H, sh.T, sh.W)
    assert idx_r.shape == (sh.B, sh.H, sh.T, sh.R)
    assert alpha.shape == (sh.B, sh.H, sh.T) and beta.shape == alpha.shape
    assert v.shape == (sh.B, sh.H, sh.T, sh.d_v)
    assert M.shape == (sh.B, sh.H, sh.N, sh.d_v)
    y = np.empty((sh.B, sh.H, sh.T, sh.d_v), np.float64)
    cs = sh.c()
    if log:
        U = np.empty((sh.B, sh.H, sh.T, sh.W, sh.d_v), np.float64)
        _check(_L().sdm_ref_scan_logged(ctypes.byref(cs), _p(idx_w), _p(wt_w), _p(idx_r),
                                        _p(wt_r), _p(alpha), _p(beta), _p(v), _p(M), _p(y),
                                        _p(U)), "scan_logged")
        return M, y, U
    _check(_L().sdm_ref_scan(ctypes.byref(cs), _p(idx_w), _p(wt_w), _p(idx_r), _p(wt_r),
                             _p(alpha), _p(beta), _p(v), _p(M), _p(y)), "scan")
    return M, y


def undo(sh: Shape, idx_w, U, M1):
    """Restore the table before a logged segment: M1 [B,H,N,d_v] after it,
    U its undo log [B,H,T,W,d_v]; returns the restored float64 table."""
    idx_w = _arr(idx_w, np.int32)
    U = _arr(U, np.float64)
    M = np.array(M1, dtype=np.float64, order="C", copy=True)
    assert idx_w.shape == (sh.B, sh.H, sh.T, sh.W)
    assert U.shape == (sh.B, sh.H, sh.T, sh.W, sh.d_v)
    assert M.shape == (sh.B, sh.H, sh.N, sh.d_v)
    cs = sh.c()
    _check(_L().sdm_ref_undo(ctypes.byref(cs), _p(idx_w), _p(U), _p(M)), "undo")
    return M


def rmsnorm_gate(sh: Shape, y, g, gamma=None, eps: float = 1e-6):
    """Per-head RMS-Norm and output gate: y [B,H,T,d_v], g [B,H,T,d_v],
    gamma [H,d_v] or None -> float64 [B,H,T,d_v]."""
    y = _arr(y, np.float64)
    g = _arr(g, np.float32)
    assert y.shape == (sh.B, sh.H, sh.T, sh.d_v) and g.shape == y.shape
    gp = None
    if gamma is not None:
        gamma = _arr(gamma, np.float32)
        assert gamma.shape == (sh.H, sh.d_v)
        gp = _p(gamma)
    out = np.empty(y.shape, np.float64)
    cs = sh.c()
    _check(_L().sdm_ref_rmsnorm_gate(ctypes.byref(cs), _p(y), _p(g), gp, float(eps), _p(out)),
           "rmsnorm_gate")
    return out


def forward(sh: Shape, q_w, q_r, K, alpha, beta, v, M0):
    """Returns dict with M, y (float64) and idx_w, wt_w, idx_r, wt_r."""
    q_w = _arr(q_w, np.float32)
    q_r = _arr(q_r, np.float32)
    K = _arr(K, np.float32)
    alpha = _arr(alpha, np.float32)
    beta = _arr(beta, np.float32)
    v = _arr(v, np.float32)
    M = np.array(M0, dtype=np.float64, order="C", copy=True)
    y = np.empty((sh.B, sh.H, sh.T, sh.d_v), np.float64)
    idx_w = np.empty((sh.B, sh.H, sh.T, sh.W), np.int32)
    idx_r = np.empty((sh.B, sh.H, sh.T, sh.R), np.int32)
    wt_w = np.empty((sh.B, sh.H, sh.T, sh.W), np.float64)
    wt_r = np.empty((sh.B, sh.H, sh.T, sh.R), np.float64)
    cs = sh.c()
    _check(_L().sdm_ref_forward(ctypes.byref(cs), _p(q_w), _p(q_r), _p(K), _p(alpha),
                                _p(beta), _p(v), _p(M), _p(y), _p(idx_w), _p(wt_w),
                                _p(idx_r), _p(wt_r)), "forward")
    return dict(M=M, y=y, idx_w=idx_w, wt_w=wt_w, idx_r=idx_r, wt_r=wt_r)
