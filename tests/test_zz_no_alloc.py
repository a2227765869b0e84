"""sdm_scan_noalloc (the scan for callers that cannot allocate device memory)
through the C ABI: on two calls in a row with different shapes (the second
call reuses the library's fixed scratch that the first one filled) its
results are bit-identical to sdm_scan's, which uses a caller workspace for
the same plan codes, and the first case also matches the oracle scan.
Collected last on purpose (see the file name)."""
import numpy as np
import pytest
import torch

import oracle as O
from tests._helpers import FTOL, gshape, max_rel, np32, oshape
from workloads import WORKLOADS, generate

pytestmark = pytest.mark.gpu

sdm = pytest.importorskip("sparse_state_linear_gb300")


def _inputs(w):
    x = generate(w)
    g = {k: t.to("cuda:0") for k, t in x.items()}
    sh = gshape(w, sdm)
    idx_w, wt_w, idx_r, wt_r = sdm.sdm_address(sh, g["q_w"], g["q_r"], g["K"])
    return sh, x, g, (idx_w, wt_w, idx_r, wt_r)


def test_noalloc_scan_matches_workspace_scan_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sdm.sdm_set_scan_tuning(0, 0)
    assert sdm.sdm_get_device_status() == 0
    cases = [WORKLOADS["mid"].with_(B=1, H=2, T=300),          # 600 token-heads, W=R=64
             WORKLOADS["tiny"].with_(T=200, W=4, R=6)]          # other shape, same scratch
    for i, w in enumerate(cases):
        sh, x, g, sel = _inputs(w)
        M_ref = g["M0"].clone()
        y_ref = sdm.sdm_scan(sh, *sel, g["alpha"], g["beta"], g["v"], M_ref)
        M_na = g["M0"].clone()
        y_na = sdm.sdm_scan_noalloc(sh, *sel, g["alpha"], g["beta"], g["v"], M_na)
        torch.cuda.synchronize()
        assert sdm.sdm_get_device_status() == 0
        # Same kernels, same plan codes, only the scratch differs: bit-identical.
        assert torch.equal(y_na, y_ref) and torch.equal(M_na, M_ref)
        if i == 0:
            # And against the oracle scan fed the same selections and weights.
            idx_w, wt_w, idx_r, wt_r = (t.cpu().numpy() for t in sel)
            Mo, yo = O.scan(oshape(w), idx_w, wt_w.astype(np.float64), idx_r,
                            wt_r.astype(np.float64), np32(x["alpha"]), np32(x["beta"]),
                            np32(x["v"]), x["M0"].numpy())
            assert max_rel(np32(y_na), yo) <= FTOL
            assert max_rel(np32(M_na), Mo) <= FTOL


def test_noalloc_scan_refuses_problems_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    # 40000 token-heads * 128 plan codes * 2 B > 8 MiB.  Every tensor has the
    # full size the shape implies and every slot is in range, so nothing could
    # go out of bounds even if the call were not refused before launching.
    w = WORKLOADS["mid"].with_(B=1, H=1, T=40000)
    sh = gshape(w, sdm)
    dev = "cuda:0"
    bht = (w.B, w.H, w.T)
    idx_w = torch.arange(w.W, dtype=torch.int32, device=dev).expand(*bht, w.W).contiguous()
    idx_r = torch.zeros(*bht, w.R, dtype=torch.int32, device=dev)
    wt_w = torch.zeros(*bht, w.W, device=dev)
    wt_r = torch.zeros(*bht, w.R, device=dev)
    gates = torch.zeros(*bht, dtype=torch.bfloat16, device=dev)
    v = torch.zeros(*bht, w.d_v, dtype=torch.bfloat16, device=dev)
    M = torch.zeros(w.B, w.H, w.N, w.d_v, device=dev)
    y = torch.zeros(*bht, w.d_v, device=dev)
    with pytest.raises(sdm.SdmError) as e:
        sdm.sdm_scan_noalloc(sh, idx_w, wt_w, idx_r, wt_r, gates, gates, v, M, y=y)
    assert e.value.code == 2
    torch.cuda.synchronize()
    assert sdm.sdm_get_device_status() == 0
    assert torch.count_nonzero(M) == 0 and torch.count_nonzero(y) == 0
