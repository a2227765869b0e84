"""Full-size workloads through sdm_forward, in the launch configuration the
benchmark times, checked on samples the oracle computes one by one:

* addressing of a random sample of (b, h, t) tokens (the oracle's sub-scores
  and selection for just those tokens);
* the whole recurrence of sampled chains (b, h), with the oracle scan fed the
  device's selections and the oracle's own weights for them (the softmax of
  its own sums of those slots; the device's weights are checked against them
  on every token of the chain);
* rows that no step of a chain wrote are bit-identical to M_0 (all chains).
"""
import numpy as np
import pytest
import torch

import oracle as O
from tests._helpers import (FTOL, check_indices, compact_oracle_scan, gshape, max_rel, np32,
                           oracle_weights, oshape)
from workloads import ORDER, WORKLOADS, generate

pytestmark = pytest.mark.gpu

sdm = pytest.importorskip("sparse_state_linear_gb300")
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _ready():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    sdm.lib()
    sdm.sdm_set_scan_tuning(0, 0)
    assert sdm.sdm_get_device_status() == 0


@pytest.mark.parametrize("name", ORDER)
def test_fullsize_forward_sampled(name):
    w = WORKLOADS[name]
    x = generate(w)
    g = {k: t.to(DEV) for k, t in x.items() if k != "M0"}
    M = x["M0"].to(DEV)
    sh = gshape(w, sdm)
    out = sdm.sdm_forward(sh, g["q_w"], g["q_r"], g["K"], g["alpha"], g["beta"], g["v"], M)
    assert sdm.sdm_get_device_status() == 0
    iw, ir = out["idx_w"].cpu().numpy(), out["idx_r"].cpu().numpy()
    ww, wr = out["wt_w"].cpu().numpy(), out["wt_r"].cpu().numpy()
    rng = np.random.default_rng(1234)

    # Addressing on sampled tokens: a 1 x 1 x n "sequence" of the sampled rows.
    n = 512
    bs = rng.integers(0, w.B, n)
    hs = rng.integers(0, w.H, n)
    ts = rng.integers(0, w.T, n)
    ts[:4] = [0, w.T - 1, 0, w.T - 1]
    for h in np.unique(hs):
        sel = hs == h
        m = int(sel.sum())
        sub = O.Shape(B=1, H=1, T=m, n_sub=w.n_sub, d_h=w.d_h, d_v=w.d_v, W=w.W, R=w.R,
                      k_w=w.k_w, k_r=w.k_r, score_kind=w.score_kind, idw_eps=w.idw_eps)
        qw = np32(x["q_w"][bs[sel], h, ts[sel]])[None, None]
        qr = np32(x["q_r"][bs[sel], h, ts[sel]])[None, None]
        K = np32(x["K"][h:h + 1])
        S_w, S_r = O.subscores(sub, qw, K), O.subscores(sub, qr, K)
        ow, orr = O.select(sub, 0, S_w), O.select(sub, 1, S_r)
        gw = iw[bs[sel], h, ts[sel]][None, None]
        gr = ir[bs[sel], h, ts[sel]][None, None]
        # Differences are allowed only inside the 1e-5 score gap (asserted inside).
        check_indices(gw, ow[0], S_w, w.n_sub)
        check_indices(gr, orr[0], S_r, w.n_sub)
        oracle_weights(sub, S_w, S_r, gw, gr, ww[bs[sel], h, ts[sel]][None, None],
                       wr[bs[sel], h, ts[sel]][None, None])

    # Whole chains: the oracle recurrence on the device's selections.
    Mg = M  # updated in place on the device
    chains = [(0, 0), (w.B - 1, w.H - 1)] if w.B * w.H > 1 else [(0, 0)]
    for b, h in chains:
        one = O.Shape(B=1, H=1, T=w.T, n_sub=w.n_sub, d_h=w.d_h, d_v=w.d_v, W=w.W, R=w.R,
                      k_w=w.k_w, k_r=w.k_r, score_kind=w.score_kind, idw_eps=w.idw_eps)
        K = np32(x["K"][h:h + 1])
        S_w = O.subscores(one, np32(x["q_w"][b:b + 1, h:h + 1]), K)
        S_r = O.subscores(one, np32(x["q_r"][b:b + 1, h:h + 1]), K)
        cw, cr = iw[b:b + 1, h:h + 1], ir[b:b + 1, h:h + 1]
        # The chain's selections against the oracle's on every token (every
        # 16th token of the long sequence, to bound the oracle's sorting).
        st = 16 if w.T > 16384 else 1
        sub = O.Shape(B=1, H=1, T=len(range(0, w.T, st)), n_sub=w.n_sub, d_h=w.d_h,
                      d_v=w.d_v, W=w.W, R=w.R, k_w=w.k_w, k_r=w.k_r)
        check_indices(cw[:, :, ::st], O.select(sub, 0, S_w[:, :, ::st])[0], S_w[:, :, ::st],
                      w.n_sub)
        check_indices(cr[:, :, ::st], O.select(sub, 1, S_r[:, :, ::st])[0], S_r[:, :, ::st],
                      w.n_sub)
        ow_c, or_c = oracle_weights(one, S_w, S_r, cw, cr, ww[b:b + 1, h:h + 1],
                                    wr[b:b + 1, h:h + 1])
        Mo, yo = O.scan(one, cw, ow_c, cr, or_c,
                        np32(x["alpha"][b:b + 1, h:h + 1]), np32(x["beta"][b:b + 1, h:h + 1]),
                        np32(x["v"][b:b + 1, h:h + 1]), x["M0"][b:b + 1, h:h + 1].numpy())
        yg = out["y"][b, h].cpu().numpy()
        assert max_rel(yg, yo[0, 0]) <= FTOL
        assert max_rel(Mg[b, h].cpu().numpy(), Mo[0, 0]) <= FTOL

    # Untouched rows, every chain (checked on the device, bitwise).
    for b in range(w.B):
        for h in range(w.H):
            touched = torch.zeros(w.N, dtype=torch.bool, device=DEV)
            touched[out["idx_w"][b, h].reshape(-1).long()] = True
            M0bh = x["M0"][b, h].to(DEV)
            assert torch.equal(Mg[b, h][~touched], M0bh[~touched])
    del g, M, out
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,epi", [("decode_l08", False), ("decode_l13", True)])
def test_fullsize_decode_sampled(name, epi):
    """The decode workloads at full size, in the launch configuration the
    benchmark times (the 8B head shape splits each chain over column parts,
    a thread-block cluster with the epilogue): every chain's selection
    against the oracle, and the write, read and epilogue of every chain on
    the device's selections (the oracle runs on a compact table of the rows
    a chain touches, copied from M_0 before the call)."""
    w = WORKLOADS[name]
    x = generate(w, device=DEV)                 # tables of tens of GB: drawn on the device
    M = x["M0"]
    M0 = M.clone()
    sh = gshape(w, sdm)
    gate = gamma = None
    if epi:
        gen = torch.Generator(device=DEV).manual_seed(11)
        gate = torch.sigmoid(torch.randn(w.B, w.H, w.T, w.d_v, generator=gen,
                                         device=DEV)).bfloat16()
        gamma = torch.rand(w.H, w.d_v, generator=gen, device=DEV) + 0.5
    out = sdm.sdm_decode(sh, x["q_w"], x["q_r"], x["K"], x["alpha"], x["beta"], x["v"], M,
                         gate=gate, gamma=gamma, out_dtype=sdm.SDM_F32)
    assert sdm.sdm_get_device_status() == 0
    sh_o = oshape(w)
    S_w = O.subscores(sh_o, np32(x["q_w"]), np32(x["K"]))
    S_r = O.subscores(sh_o, np32(x["q_r"]), np32(x["K"]))
    ow, orr = O.select(sh_o, 0, S_w), O.select(sh_o, 1, S_r)
    iw, ir = out["idx_w"].cpu().numpy(), out["idx_r"].cpu().numpy()
    check_indices(iw, ow[0], S_w, w.n_sub)
    check_indices(ir, orr[0], S_r, w.n_sub)
    same = np.all(iw == ow[0], axis=-1) & np.all(ir == orr[0], axis=-1)
    assert same.mean() > 0.9
    ww, wr = oracle_weights(sh_o, S_w, S_r, iw, ir, np32(out["wt_w"]), np32(out["wt_r"]))
    rows, Mo, yo = compact_oracle_scan(iw, ww, ir, wr, np32(x["alpha"]), np32(x["beta"]),
                                       np32(x["v"]), M0, w.update_form)
    assert max_rel(np32(out["y"]), yo) <= FTOL
    for b in range(w.B):
        for h in range(w.H):
            r = torch.from_numpy(rows[b][h]).long().to(DEV)
            assert max_rel(M[b, h, r].cpu().numpy(), Mo[b, h, :len(r)]) <= FTOL
    if epi:
        ref = O.rmsnorm_gate(sh_o, yo, np32(gate), np32(gamma), eps=1e-6)
        assert max_rel(np32(out["out"]), ref) <= FTOL
    # Rows outside every selection are untouched: compare a random sample.
    rng = np.random.default_rng(5)
    for b, h in [(0, 0), (w.B - 1, w.H - 1)]:
        pick = rng.choice(w.N, 4096, replace=False)
        pick = np.setdiff1d(pick, iw[b, h].ravel())
        idx = torch.from_numpy(pick).long().to(DEV)
        assert torch.equal(M[b, h, idx], M0[b, h, idx])
