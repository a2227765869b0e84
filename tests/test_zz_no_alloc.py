"""sdm_scan_noalloc (the scan for callers that cannot allocate device memory)
against sdm_scan, through the C ABI, on two calls in a row with different
shapes: the second call reuses the library's fixed scratch that the first one
filled.  Collected last on purpose (see the file name)."""
import pytest
import torch

from tests._helpers import FTOL, gshape, max_rel
from workloads import WORKLOADS, generate

pytestmark = pytest.mark.gpu

sdm = pytest.importorskip("sparse_state_linear_gb300")


def _inputs(w):
    x = generate(w)
    g = {k: t.to("cuda:0") for k, t in x.items()}
    sh = gshape(w, sdm)
    idx_w, wt_w, idx_r, wt_r = sdm.sdm_address(sh, g["q_w"], g["q_r"], g["K"])
    return sh, g, (idx_w, wt_w, idx_r, wt_r)


def test_noalloc_scan_matches_workspace_scan_twice():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sdm.sdm_set_scan_tuning(0, 0)
    assert sdm.sdm_get_device_status() == 0
    cases = [WORKLOADS["mid"].with_(B=1, H=2, T=300),          # 600 token-heads, W=R=64
             WORKLOADS["tiny"].with_(T=200, W=4, R=6)]          # other shape, same scratch
    for w in cases:
        sh, g, sel = _inputs(w)
        M_ref = g["M0"].clone()
        y_ref = sdm.sdm_scan(sh, *sel, g["alpha"], g["beta"], g["v"], M_ref)
        M_na = g["M0"].clone()
        y_na = sdm.sdm_scan_noalloc(sh, *sel, g["alpha"], g["beta"], g["v"], M_na)
        torch.cuda.synchronize()
        assert sdm.sdm_get_device_status() == 0
        assert max_rel(y_na.cpu().numpy(), y_ref.cpu().double().numpy()) <= FTOL
        assert max_rel(M_na.cpu().numpy(), M_ref.cpu().double().numpy()) <= FTOL


def test_noalloc_scan_refuses_problems_beyond_its_scratch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    w = WORKLOADS["mid"].with_(B=1, H=1, T=40000)   # 40000 * 128 codes * 2 B > 8 MiB
    sh = gshape(w, sdm)
    z = torch.zeros(16, device="cuda:0")
    zi = torch.zeros(16, device="cuda:0", dtype=torch.int32)
    zb = torch.zeros(16, device="cuda:0", dtype=torch.bfloat16)
    with pytest.raises(sdm.SdmError) as e:
        sdm.sdm_scan_noalloc(sh, zi, z, zi, z, zb, zb, zb, z, y=z)
    assert e.value.code == 2
