"""Shared parity helpers for the GPU tests (CUDA path vs the CPU oracle)."""
from __future__ import annotations

import numpy as np
import torch

import oracle as O

# Tolerances fixed by the target: slot indices exact on identical sub-scores;
# end to end, index mismatches only where oracle scores differ by < 1e-5;
# floats within max-abs 1e-4 x RMS of the oracle's output.
GAP = 1e-5
FTOL = 1e-4
# Device softmax weights (fp32, from the device's sub-scores) against the
# oracle's (double, from its own sub-scores) for the same slots.
WTOL = 1e-5


def oshape(w, T=None, B=None, H=None):
    return O.Shape(B=w.B if B is None else B, H=w.H if H is None else H,
                   T=w.T if T is None else T, n_sub=w.n_sub, d_h=w.d_h, d_v=w.d_v, W=w.W,
                   R=w.R, k_w=w.k_w, k_r=w.k_r, score_kind=w.score_kind,
                   idw_eps=w.idw_eps, update_form=w.update_form)


def gshape(w, sdm, T=None, B=None, H=None):
    return sdm.make_shape(w.B if B is None else B, w.H if H is None else H,
                          w.T if T is None else T, w.n_sub, w.d_h, w.d_v, w.W, w.R,
                          k_w=w.k_w, k_r=w.k_r,
                          in_dtype=sdm.SDM_BF16 if w.bf16 else sdm.SDM_F32,
                          score=w.score_kind, idw_eps=w.idw_eps, update=w.update_form)


def np32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def check_indices(idx_gpu, idx_ref, S_ref, n_sub, gap=GAP):
    """Compare selections row by row as sets; a slot in the symmetric
    difference must score within `gap` of the oracle's last selected score.
    Returns the number of rows that differ (as sets)."""
    idx_gpu = idx_gpu.reshape(-1, idx_gpu.shape[-1])
    idx_ref = idx_ref.reshape(-1, idx_ref.shape[-1])
    S = S_ref.reshape(-1, 2, n_sub)
    bad_rows = 0
    for r in range(idx_ref.shape[0]):
        g, o = idx_gpu[r], idx_ref[r]
        if np.array_equal(g, o):
            continue
        gs, os_ = set(g.tolist()), set(o.tolist())
        s1, s2 = S[r, 0], S[r, 1]
        score = lambda slot: np.float32(s1[slot // n_sub] + s2[slot % n_sub])
        last = score(int(o[-1]))
        assert len(gs) == len(g), f"row {r}: duplicate slots {g}"
        for slot in gs ^ os_:
            assert 0 <= slot < n_sub * n_sub
            assert abs(float(score(slot)) - float(last)) < gap, (
                f"row {r}: slot {slot} score {score(slot)} vs W-th {last}")
        if gs == os_:
            # Same set, different order: adjacent swaps only across tiny gaps.
            sg = np.array([score(int(x)) for x in g], np.float64)
            assert np.all(np.diff(sg) <= gap), f"row {r}: order {sg}"
        bad_rows += 1
    return bad_rows


def oracle_weights(sh_o, S_w, S_r, iw, ir, ww=None, wr=None):
    """The oracle's weights for the device's selections iw / ir: the softmax
    of the oracle's own float sums (from its sub-scores S_w / S_r) of exactly
    those slots, in the device's order.  With the device's weights given,
    asserts they agree within WTOL on every row.  Returns (wt_w, wt_r) float64,
    the weights a re-anchored oracle scan takes."""
    ow = O.slot_weights(sh_o, 0, S_w, iw)
    orr = O.slot_weights(sh_o, 1, S_r, ir)
    if ww is not None:
        assert np.max(np.abs(np.asarray(ww, np.float64) - ow), initial=0) < WTOL
    if wr is not None:
        assert np.max(np.abs(np.asarray(wr, np.float64) - orr), initial=0) < WTOL
    return ow, orr


def max_rel(a: np.ndarray, ref: np.ndarray) -> float:
    rms = float(np.sqrt(np.mean(np.square(ref, dtype=np.float64))))
    if rms == 0.0:
        return float(np.max(np.abs(a - ref))) if a.size else 0.0
    return float(np.max(np.abs(a.astype(np.float64) - ref))) / rms if a.size else 0.0


def compact_oracle_scan(idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M0_dev, update_form):
    """The oracle scan of a short segment on a compact table that holds only
    the rows the segment touches (exact: no other row is ever read)."""
    B, H, T, W = idx_w.shape
    R = idx_r.shape[-1]
    dv = M0_dev.shape[-1]
    rows = [[np.unique(np.concatenate([idx_w[b, h].ravel(), idx_r[b, h].ravel()]))
             for h in range(H)] for b in range(B)]
    n = max(len(r) for rr in rows for r in rr)
    s2 = int(np.ceil(np.sqrt(n)))
    Mc = np.zeros((B, H, s2 * s2, dv), np.float32)
    iw, ir = np.empty_like(idx_w), np.empty_like(idx_r)
    for b in range(B):
        for h in range(H):
            r = rows[b][h]
            Mc[b, h, :len(r)] = M0_dev[b, h, torch.from_numpy(r).long().to(M0_dev.device)].cpu().numpy()
            iw[b, h] = np.searchsorted(r, idx_w[b, h])
            ir[b, h] = np.searchsorted(r, idx_r[b, h])
    sh = O.Shape(B=B, H=H, T=T, n_sub=s2, d_h=16, d_v=dv, W=W, R=R, update_form=update_form)
    Mo, yo = O.scan(sh, iw, wt_w, ir, wt_r, alpha, beta, v, Mc)
    return rows, Mo, yo
