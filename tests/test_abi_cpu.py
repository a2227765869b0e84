"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every function include/sdm.h declares, and rejects bad arguments before it
touches CUDA."""
import ctypes
import os
import re

import pytest

import sparse_state_linear_gb300 as sdm
from sparse_state_linear_gb300 import build_ext

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build_ext.build()
    return sdm.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "sdm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(sdm_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(sdm.EXPORTS)


def test_status_strings(L):
    for code in range(7):
        assert sdm.status_string(code) not in ("", "unknown status")
    assert sdm.status_string(99) == "unknown status"


def good_shape(**kw):
    base = dict(B=2, H=2, T=8, n_sub=16, d_h=16, d_v=32, W=8, R=8, in_dtype=sdm.SDM_F32)
    base.update(kw)
    return sdm.make_shape(**base)


FAKE = ctypes.c_void_p(1 << 20)        # aligned, never dereferenced
MISALIGNED = ctypes.c_void_p((1 << 20) + 4)


def scan_rc(L, sh, ptrs=None, ws_bytes=1 << 30):
    p = ptrs or [FAKE] * 9
    return L.sdm_scan(ctypes.byref(sh), *p, FAKE, ws_bytes, None)


@pytest.mark.parametrize("kw,code", [
    (dict(T=-1), 1), (dict(n_sub=0), 1), (dict(W=0), 1), (dict(d_v=0), 1),
    (dict(in_dtype=7), 1), (dict(score=3), 1), (dict(update=5), 1),
    (dict(W=300), 1),                    # W > k_w^2 with k_w = min(W, s) = 16
    (dict(k_w=17), 1),                   # k above s
    (dict(n_sub=600), 2), (dict(d_h=24), 2), (dict(d_v=40), 2), (dict(n_sub=32, W=65, R=8), 2),
    (dict(d_v=2064), 2),
])
def test_scan_rejects_bad_shapes(L, kw, code):
    assert scan_rc(L, good_shape(**kw)) == code


def test_null_and_misaligned_pointers(L):
    sh = good_shape()
    for i in range(9):
        p = [FAKE] * 9
        p[i] = None
        assert scan_rc(L, sh, p) == 1
        p[i] = MISALIGNED
        assert scan_rc(L, sh, p) == 1
    assert L.sdm_address(ctypes.byref(sh), None, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None) == 1
    assert L.sdm_select(ctypes.byref(sh), FAKE, FAKE, FAKE, FAKE, FAKE, None, None) == 1
    assert L.sdm_subscores(ctypes.byref(sh), FAKE, None, FAKE, None) == 1
    # Workspace: required, aligned and large enough.
    need = L.sdm_workspace_size(ctypes.byref(sh))
    assert need == sh.B * sh.H * sh.T * 16 * 2      # W + R = 16 codes of 2 bytes per token
    assert L.sdm_scan(ctypes.byref(sh), *([FAKE] * 9), None, need, None) == 1
    assert L.sdm_scan(ctypes.byref(sh), *([FAKE] * 9), MISALIGNED, need, None) == 1
    assert L.sdm_scan(ctypes.byref(sh), *([FAKE] * 9), FAKE, need - 1, None) == 1
    assert L.sdm_forward(ctypes.byref(sh), *([FAKE] * 12), FAKE, need - 1, None) == 1
    assert L.sdm_workspace_size(ctypes.byref(good_shape(W=0))) == 0


def test_logged_scan_and_undo_arguments(L):
    sh = good_shape()
    need = L.sdm_workspace_size(ctypes.byref(sh))
    # sdm_scan_logged: the ten tensors (undo last) must be present and aligned.
    for i in range(10):
        p = [FAKE] * 10
        p[i] = None
        assert L.sdm_scan_logged(ctypes.byref(sh), *p, FAKE, need, None) == 1
        p[i] = MISALIGNED
        assert L.sdm_scan_logged(ctypes.byref(sh), *p, FAKE, need, None) == 1
    assert L.sdm_scan_logged(ctypes.byref(sh), *([FAKE] * 10), FAKE, need - 1, None) == 1
    # sdm_scan_undo: one mark per table row of every chain.
    uneed = L.sdm_undo_workspace_size(ctypes.byref(sh))
    assert uneed == sh.B * sh.H * sh.N * 4
    assert L.sdm_undo_workspace_size(ctypes.byref(good_shape(W=0))) == 0
    for i in range(3):
        p = [FAKE] * 3
        p[i] = None
        assert L.sdm_scan_undo(ctypes.byref(sh), *p, FAKE, uneed, None) == 1
        p[i] = MISALIGNED
        assert L.sdm_scan_undo(ctypes.byref(sh), *p, FAKE, uneed, None) == 1
    assert L.sdm_scan_undo(ctypes.byref(sh), FAKE, FAKE, FAKE, None, uneed, None) == 1
    assert L.sdm_scan_undo(ctypes.byref(sh), FAKE, FAKE, FAKE, FAKE, uneed - 1, None) == 1
    assert L.sdm_scan_undo(ctypes.byref(good_shape(n_sub=600)), FAKE, FAKE, FAKE, FAKE,
                           uneed, None) == 2
    # Empty segments return before any CUDA call.
    for kw in (dict(T=0), dict(B=0)):
        e = good_shape(**kw)
        assert L.sdm_scan_undo(ctypes.byref(e), FAKE, FAKE, FAKE, None, 0, None) == 0
        assert L.sdm_scan_logged(ctypes.byref(e), *([FAKE] * 10), None, 0, None) == 0


def test_rmsnorm_gate_arguments(L):
    sh = good_shape()
    rc = lambda *a: L.sdm_rmsnorm_gate(ctypes.byref(sh), *a)
    assert rc(FAKE, FAKE, None, ctypes.c_float(0.0), FAKE, 1, None) == 1          # eps
    assert rc(FAKE, FAKE, None, ctypes.c_float(float("inf")), FAKE, 1, None) == 1
    assert rc(FAKE, FAKE, None, ctypes.c_float(1e-6), FAKE, 7, None) == 1         # out dtype
    assert rc(None, FAKE, None, ctypes.c_float(1e-6), FAKE, 1, None) == 1
    assert rc(FAKE, MISALIGNED, None, ctypes.c_float(1e-6), FAKE, 1, None) == 1
    assert rc(FAKE, FAKE, MISALIGNED, ctypes.c_float(1e-6), FAKE, 1, None) == 1
    assert rc(FAKE, FAKE, None, ctypes.c_float(1e-6), None, 0, None) == 1
    e = good_shape(T=0)
    assert L.sdm_rmsnorm_gate(ctypes.byref(e), None, None, None, ctypes.c_float(1e-6), None, 1,
                              None) == 0


def test_empty_work_is_a_no_op(L):
    # Nothing to do: returns before any CUDA call, so it works without a GPU.
    for kw in (dict(T=0), dict(B=0), dict(H=0)):
        sh = good_shape(**kw)
        assert scan_rc(L, sh) == 0
        assert L.sdm_forward(ctypes.byref(sh), *([FAKE] * 12), FAKE, 0, None) == 0
        # Empty tensors may come as NULL pointers.
        assert scan_rc(L, sh, [None] * 9) == 0
        assert L.sdm_forward(ctypes.byref(sh), *([None] * 13), 0, None) == 0
        assert L.sdm_address(ctypes.byref(sh), *([None] * 7), None) == 0
        assert L.sdm_scan_noalloc(ctypes.byref(sh), *([None] * 9), None) == 0


def test_tuning_arguments(L):
    assert L.sdm_set_scan_tuning(-1, 0) == 1
    assert L.sdm_set_scan_tuning(17, 0) == 1
    assert L.sdm_set_scan_tuning(4, 24) == 1
    assert L.sdm_set_scan_tuning(4, 32) == 0
    assert L.sdm_set_scan_tuning(0, 0) == 0
    assert L.sdm_selftest_wait_timeout(10, None) == 1


def test_python_binding_checks_tensors():
    import torch
    sh = good_shape()
    with pytest.raises(ValueError):
        sdm.sdm_scan(sh, *([torch.zeros(4)] * 8))


def test_decode_arguments(L):
    sh = good_shape(T=1)
    dec = lambda ptrs, epi=None, shape=sh: L.sdm_decode(ctypes.byref(shape), *ptrs,
                                                         ctypes.byref(epi) if epi else None,
                                                         None)
    # The twelve tensors must be present and 16-byte aligned.
    for i in range(12):
        p = [FAKE] * 12
        p[i] = None
        assert dec(p) == 1
        p[i] = MISALIGNED
        assert dec(p) == 1
    # Epilogue: eps > 0 and finite, a known output dtype, gate and output
    # present, gamma (optional) aligned.
    good = dict(g=FAKE.value, gamma=None, eps=1e-6, out=FAKE.value, out_dtype=sdm.SDM_F32)
    for bad in (dict(eps=0.0), dict(eps=float("inf")), dict(eps=float("nan")), dict(out_dtype=7),
                dict(g=None), dict(out=None), dict(gamma=MISALIGNED.value),
                dict(out=MISALIGNED.value)):
        e = sdm.Epilogue(**{**good, **bad})
        assert dec([FAKE] * 12, e) == 1, bad
    # Bad shapes are rejected before anything else.
    assert dec([FAKE] * 12, shape=good_shape(T=1, d_v=2064)) == 2
    assert dec([FAKE] * 12, shape=good_shape(T=1, W=0)) == 1
    # No work: returns before looking at the pointers (NULL is fine).
    for kw in (dict(T=0), dict(B=0), dict(H=0)):
        assert dec([None] * 12, shape=good_shape(**kw)) == 0


def test_measure_row_traffic_arguments(L):
    rc = L.sdm_measure_row_traffic
    good = (FAKE, FAKE, 4, 1024, 128, 32, 8, 128, 64, 1, None)
    # Each bad argument is refused before any CUDA call.
    bad = {2: -1, 3: 0, 4: 40, 5: 48, 6: -1, 7: 0, 8: -1}
    for i, val in bad.items():
        a = list(good)
        a[i] = val
        assert rc(*a) == 1, (i, val)
    for loads, stores in ((129, 0), (8, 9), (0, 0)):
        assert rc(FAKE, FAKE, 4, 1024, 128, 32, 8, loads, stores, 1, None) == 1
    assert rc(None, FAKE, 4, 1024, 128, 32, 8, 128, 64, 1, None) == 1
    assert rc(FAKE, MISALIGNED, 4, 1024, 128, 32, 8, 128, 64, 1, None) == 1
    assert rc(FAKE, FAKE, 4, 1 << 32, 128, 32, 8, 128, 64, 1, None) == 1     # rows >= 2^32
    # No work: nothing is launched and the pointers are not looked at.
    assert rc(None, None, 0, 1024, 128, 32, 8, 128, 64, 1, None) == 0
    assert rc(None, None, 4, 1024, 128, 32, 0, 128, 64, 1, None) == 0


def test_forward_windows(L):
    # Windows only from T = 2048 on; the FFMA addressing path (fp32, inverse
    # distance, s > 256 or d_h > 64) uses 4.  (Tensor-core shapes depend on the
    # device's shared memory and are checked in the GPU tests.)
    assert sdm.sdm_forward_windows(good_shape(T=2047)) == 1
    assert sdm.sdm_forward_windows(good_shape(T=8192, n_sub=512, d_h=256, d_v=512, W=8,
                                              R=8)) == 4
    # Window lengths are whole 64-step blocks: T = 2100 -> 525 -> 576 steps,
    # still 4 windows (the last one 372 steps); T = 2048 -> exactly 4 x 512.
    for T in (2048, 2049, 2100, 4100):
        assert sdm.sdm_forward_windows(good_shape(T=T)) == 4
    bad = good_shape()
    bad.W = 0
    assert sdm.sdm_forward_windows(bad) == 0
