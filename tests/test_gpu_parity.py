"""CUDA path vs the CPU oracle, through the C ABI (needs an sm_103a GPU).

Sizes the oracle finishes in seconds, spanning several CTA tiles and a ragged
tail; full-size workloads are covered in test_gpu_sampled_fullsize.py.
"""
import numpy as np
import pytest
import torch

import oracle as O
from tests._helpers import (FTOL, check_indices, compact_oracle_scan, gshape, max_rel, np32,
                           oracle_weights, oshape)
from workloads import WORKLOADS, generate

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
    yield
    sdm.sdm_set_scan_tuning(0, 0)


def status_ok():
    assert sdm.sdm_get_device_status() == 0


# ------------------------------------------------------------------ selection

def select_both(sh_o, sh_g, S_w, S_r):
    gw = torch.from_numpy(S_w).to(DEV)
    gr = torch.from_numpy(S_r).to(DEV)
    idx_w, wt_w, idx_r, wt_r = sdm.sdm_select(sh_g, gw, gr)
    status_ok()
    ow = O.select(sh_o, 0, S_w)
    orr = O.select(sh_o, 1, S_r)
    return (idx_w.cpu().numpy(), wt_w.cpu().numpy(), idx_r.cpu().numpy(), wt_r.cpu().numpy()), ow, orr


@pytest.mark.parametrize("s,W,R,kw,kr,BT", [
    (32, 8, 8, 0, 0, (1, 37)),       # tiny shape
    (128, 64, 64, 0, 0, (2, 23)),
    (256, 64, 64, 0, 0, (3, 17)),    # GDN-matched
    (512, 8, 8, 0, 0, (1, 50)),      # FwPKM-shaped
    (256, 64, 16, 0, 0, (1, 33)),    # W != R
    (8, 64, 64, 0, 0, (1, 19)),      # every slot selected (k = s = 8)
    (64, 5, 3, 12, 2, (2, 21)),      # explicit k
    (240, 64, 64, 0, 0, (1, 20)),    # non power-of-two s
    (100, 1, 1, 0, 0, (1, 40)),      # single slot
])
def test_select_bit_exact_random(s, W, R, kw, kr, BT):
    B, T = BT
    H = 2
    rng = np.random.default_rng(s * 131 + W)
    S_w = rng.standard_normal((B, H, T, 2, s)).astype(np.float32)
    S_r = (rng.standard_normal((B, H, T, 2, s)) * 3).astype(np.float32)
    sh_o = O.Shape(B=B, H=H, T=T, n_sub=s, d_h=16, d_v=16, W=W, R=R, k_w=kw, k_r=kr)
    sh_g = sdm.make_shape(B, H, T, s, 16, 16, W, R, k_w=kw, k_r=kr, in_dtype=sdm.SDM_F32)
    (iw, ww, ir, wr), ow, orr = select_both(sh_o, sh_g, S_w, S_r)
    assert np.array_equal(iw, ow[0])
    assert np.array_equal(ir, orr[0])
    assert np.max(np.abs(ww - ow[2])) < 2e-6
    assert np.max(np.abs(wr - orr[2])) < 2e-6


@pytest.mark.parametrize("kind", ["int_ties", "constant", "signed_zeros", "dominant", "huge_range",
                                  "two_values", "neg_large"])
def test_select_bit_exact_adversarial(kind):
    rng = np.random.default_rng(7)
    B, H, T, s, W = 1, 1, 48, 64, 64
    shp = (B, H, T, 2, s)
    if kind == "int_ties":
        S = rng.integers(-3, 4, shp).astype(np.float32)
    elif kind == "constant":
        S = np.full(shp, 0.5, np.float32)
    elif kind == "signed_zeros":
        S = np.where(rng.random(shp) < 0.5, np.float32(0.0), np.float32(-0.0)).astype(np.float32)
        S[..., ::7] = 1.0
    elif kind == "dominant":
        S = rng.standard_normal(shp).astype(np.float32)
        S[..., 0, 5] = 1e6
    elif kind == "huge_range":
        S = (rng.standard_normal(shp) * 10.0 ** rng.integers(-30, 30, shp)).astype(np.float32)
    elif kind == "two_values":
        S = np.where(rng.random(shp) < 0.9, np.float32(1.0), np.float32(2.0))
    else:
        S = (-1e30 + rng.standard_normal(shp) * 1e23).astype(np.float32)
    S_r = S[..., ::-1].copy()
    sh_o = O.Shape(B=B, H=H, T=T, n_sub=s, d_h=16, d_v=16, W=W, R=16)
    sh_g = sdm.make_shape(B, H, T, s, 16, 16, W, 16, in_dtype=sdm.SDM_F32)
    (iw, ww, ir, wr), ow, orr = select_both(sh_o, sh_g, S, S_r)
    assert np.array_equal(iw, ow[0])
    assert np.array_equal(ir, orr[0])
    assert np.allclose(ww, ow[2], atol=2e-6, rtol=0)
    assert np.allclose(wr, orr[2], atol=2e-6, rtol=0)


# ------------------------------------------------------------------ sub-scores

@pytest.mark.parametrize("name", ["tiny", "mid", "gdn_matched", "fwpkm_idw"])
def test_subscores_close_to_oracle(name):
    w = WORKLOADS[name].with_(B=1, T=37, H=min(WORKLOADS[name].H, 2))
    x = generate(w)
    sh_g = gshape(w, sdm)
    S = sdm.sdm_subscores(sh_g, x["q_w"].to(DEV), x["K"].to(DEV))
    status_ok()
    ref = O.subscores(oshape(w), np32(x["q_w"]), np32(x["K"]))
    err = np.max(np.abs(np32(S) - ref))
    assert err < 1e-5 * max(1.0, float(np.max(np.abs(ref)))), err


# ------------------------------------------------------------------ addressing

REDUCED = {
    "tiny": dict(),
    "mid": dict(B=1, H=2, T=203),
    "gdn_matched": dict(B=1, H=2, T=150),
    "fwpkm_idw": dict(B=2, T=99),
    "long_seq": dict(H=2, T=301),
}


@pytest.mark.parametrize("name", list(REDUCED))
def test_address_end_to_end(name):
    w = WORKLOADS[name].with_(**REDUCED[name])
    x = generate(w)
    sh_g, sh_o = gshape(w, sdm), oshape(w)
    g = {k: t.to(DEV) for k, t in x.items()}
    iw, ww, ir, wr = sdm.sdm_address(sh_g, g["q_w"], g["q_r"], g["K"])
    status_ok()
    iw, ww, ir, wr = (t.cpu().numpy() for t in (iw, ww, ir, wr))
    # (1) Bit-exact given the device's own sub-scores.
    Sg_w = np32(sdm.sdm_subscores(sh_g, g["q_w"], g["K"]))
    Sg_r = np32(sdm.sdm_subscores(sh_g, g["q_r"], g["K"]))
    assert np.array_equal(iw, O.select(sh_o, 0, Sg_w)[0])
    assert np.array_equal(ir, O.select(sh_o, 1, Sg_r)[0])
    # (2) Against the oracle's own scores: mismatches only inside the score gap.
    S_w = O.subscores(sh_o, np32(x["q_w"]), np32(x["K"]))
    S_r = O.subscores(sh_o, np32(x["q_r"]), np32(x["K"]))
    ow, orr = O.select(sh_o, 0, S_w), O.select(sh_o, 1, S_r)
    # Differences are allowed only inside the 1e-5 score gap (asserted inside).
    check_indices(iw, ow[0], S_w, w.n_sub)
    check_indices(ir, orr[0], S_r, w.n_sub)
    # Weights on every row: the oracle's softmax of its own sums for the
    # device's slots (equal to its selection's weights where the slots agree).
    oracle_weights(sh_o, S_w, S_r, iw, ir, ww, wr)


ROW_SHAPES = [  # bf16 dot scores, s <= 256, d_h <= 64: the tensor-core kernel
    dict(n_sub=32, d_h=16, W=8, R=8, T=90),
    dict(n_sub=40, d_h=32, W=5, R=3, k_w=12, k_r=2, T=70),    # s % 16 != 0, W % 4 != 0
    dict(n_sub=200, d_h=64, W=64, R=16, T=130),
    dict(n_sub=256, d_h=64, W=1, R=64, T=66),
    dict(n_sub=16, d_h=16, W=64, R=64, T=65),                 # k = s = 16
    dict(n_sub=64, d_h=32, W=36, R=64, T=129),
]


def address_checks(w, x, sh_g, sh_o, iw, ww, ir, wr, g):
    """Bit-exact against the oracle's selection on the device's own sub-scores,
    and weights against the oracle's softmax of those selections."""
    Sg_w = np32(sdm.sdm_subscores(sh_g, g["q_w"], g["K"]))
    Sg_r = np32(sdm.sdm_subscores(sh_g, g["q_r"], g["K"]))
    ow, orr = O.select(sh_o, 0, Sg_w), O.select(sh_o, 1, Sg_r)
    assert np.array_equal(iw, ow[0])
    assert np.array_equal(ir, orr[0])
    assert np.max(np.abs(ww - ow[2])) < 1e-5
    assert np.max(np.abs(wr - orr[2])) < 1e-5


@pytest.mark.parametrize("ov", ROW_SHAPES, ids=lambda o: "s{n_sub}_W{W}_R{R}".format(**o))
def test_address_row_kernel_shapes(ov):
    w = WORKLOADS["mid"].with_(B=2, H=2, **ov)
    x = generate(w)
    sh_g, sh_o = gshape(w, sdm), oshape(w)
    g = {k: t.to(DEV) for k, t in x.items()}
    iw, ww, ir, wr = sdm.sdm_address(sh_g, g["q_w"], g["q_r"], g["K"])
    status_ok()
    address_checks(w, x, sh_g, sh_o, *(t.cpu().numpy() for t in (iw, ww, ir, wr)), g)


FFMA_SHAPES = [  # shapes the tensor-core kernel does not take: the fp32 FFMA contraction
    dict(n_sub=300, d_h=32, W=64, R=16, bf16=True),                 # s > 256: partial 2nd chunk
    dict(n_sub=128, d_h=128, W=16, R=64, bf16=True),                # d_h > 64
    dict(n_sub=64, d_h=32, W=8, R=12, bf16=True, score_kind=1),     # bf16 inverse distance
    dict(n_sub=400, d_h=16, W=8, R=8, bf16=False),                  # fp32, partial 2nd chunk
    dict(n_sub=512, d_h=256, W=64, R=8, bf16=False, score_kind=1),  # k = 64 lists at s = 512
]


@pytest.mark.parametrize("ov", FFMA_SHAPES,
                         ids=lambda o: "s{n_sub}_dh{d_h}_{}".format(
                             "idw" if o.get("score_kind") else "dot", **o))
def test_address_ffma_kernel_shapes(ov):
    ov = dict(ov)
    if ov.get("score_kind"):
        ov["qk_std"] = 1.0
    w = WORKLOADS["mid"].with_(B=1, H=2, T=45, d_v=16, **ov)
    x = generate(w)
    sh_g, sh_o = gshape(w, sdm), oshape(w)
    g = {k: t.to(DEV) for k, t in x.items()}
    # Sub-scores against the oracle's (fp32 contraction in another order).
    S = np32(sdm.sdm_subscores(sh_g, g["q_r"], g["K"]))
    ref = O.subscores(sh_o, np32(x["q_r"]), np32(x["K"]))
    assert np.max(np.abs(S - ref)) < 1e-5 * max(1.0, float(np.max(np.abs(ref))))
    iw, ww, ir, wr = sdm.sdm_address(sh_g, g["q_w"], g["q_r"], g["K"])
    status_ok()
    address_checks(w, x, sh_g, sh_o, *(t.cpu().numpy() for t in (iw, ww, ir, wr)), g)


def test_address_degenerate_rows_take_exact_path():
    """Rows the per-row kernel leaves to the exact warp kernel: all-zero
    queries (every score equal), one constant half (equal sums along a row of
    the staircase), duplicated sub-keys (equal scores inside a half)."""
    w = WORKLOADS["gdn_matched"].with_(B=1, H=2, T=200)
    x = generate(w)
    x["q_w"][0, 0, 3:40] = 0
    x["q_r"][0, 1, 10:30, 0] = 0
    x["q_w"][0, 1, 50:70, 1] = 0
    x["K"][0, 0, 100:140] = x["K"][0, 0, 20]
    x["K"][1, 1, 7:9] = x["K"][1, 1, 3]
    sh_g, sh_o = gshape(w, sdm), oshape(w)
    g = {k: t.to(DEV) for k, t in x.items()}
    iw, ww, ir, wr = sdm.sdm_address(sh_g, g["q_w"], g["q_r"], g["K"])
    status_ok()
    iw, ww, ir, wr = (t.cpu().numpy() for t in (iw, ww, ir, wr))
    assert (iw >= 0).all() and (ir >= 0).all()
    address_checks(w, x, sh_g, sh_o, iw, ww, ir, wr, g)


# ------------------------------------------------------------------ scan

def random_scan_case(rng, B, H, T, s, dv, W, R, bf16):
    N = s * s
    idx_w = np.stack([rng.choice(N, W, replace=False) for _ in range(B * H * T)])
    idx_w = idx_w.reshape(B, H, T, W).astype(np.int32)
    idx_r = rng.integers(0, N, (B, H, T, R)).astype(np.int32)
    wt_w = rng.dirichlet(np.ones(W), (B, H, T)).astype(np.float32)
    wt_r = rng.dirichlet(np.ones(R), (B, H, T)).astype(np.float32)
    dt = torch.bfloat16 if bf16 else torch.float32
    alpha = torch.from_numpy(rng.uniform(0.9, 1, (B, H, T)).astype(np.float32)).to(dt)
    beta = torch.from_numpy(rng.uniform(0, 1, (B, H, T)).astype(np.float32)).to(dt)
    v = torch.from_numpy(rng.standard_normal((B, H, T, dv)).astype(np.float32)).to(dt)
    M0 = (rng.standard_normal((B, H, N, dv)) * 0.02).astype(np.float32)
    return idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M0


def run_scan(sh_g, case, depth=0, cs=0):
    idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M0 = case
    sdm.sdm_set_scan_tuning(depth, cs)
    M = torch.from_numpy(M0).to(DEV)
    y = sdm.sdm_scan(sh_g, torch.from_numpy(idx_w).to(DEV), torch.from_numpy(wt_w).to(DEV),
                     torch.from_numpy(idx_r).to(DEV), torch.from_numpy(wt_r).to(DEV),
                     alpha.to(DEV), beta.to(DEV), v.to(DEV), M)
    status_ok()
    sdm.sdm_set_scan_tuning(0, 0)
    return M.cpu().numpy(), y.cpu().numpy()


def oracle_scan(B, H, T, s, dv, W, R, case, update_form=0):
    idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M0 = case
    sh = O.Shape(B=B, H=H, T=T, n_sub=s, d_h=16, d_v=dv, W=W, R=R, update_form=update_form)
    return O.scan(sh, idx_w, wt_w.astype(np.float64), idx_r, wt_r.astype(np.float64),
                  np32(alpha), np32(beta), np32(v), M0)


@pytest.mark.parametrize("B,H,T,s,dv,W,R,bf16", [
    (1, 1, 200, 8, 32, 16, 16, False),     # N=64: consecutive steps collide constantly
    (2, 3, 150, 16, 64, 32, 48, True),
    (1, 2, 120, 32, 128, 64, 64, True),
    (2, 1, 90, 64, 512, 8, 8, False),
    (1, 1, 64, 4, 16, 16, 16, False),      # W = N
    (1, 2, 77, 8, 48, 1, 1, False),        # d_v not a multiple of 32
])
@pytest.mark.parametrize("depth,cs", [(1, 16), (2, 32), (4, 0), (8, 16), (16, 0), (3, 64)])
def test_scan_matches_oracle(B, H, T, s, dv, W, R, bf16, depth, cs):
    if cs and dv % cs:
        cs = 16
    rng = np.random.default_rng(B * 1000 + T + W)
    case = random_scan_case(rng, B, H, T, s, dv, W, R, bf16)
    sh_g = sdm.make_shape(B, H, T, s, 16, dv, W, R,
                          in_dtype=sdm.SDM_BF16 if bf16 else sdm.SDM_F32)
    Mg, yg = run_scan(sh_g, case, depth, cs)
    Mo, yo = oracle_scan(B, H, T, s, dv, W, R, case)
    assert max_rel(yg, yo) <= FTOL
    assert max_rel(Mg, Mo) <= FTOL
    # Rows no step wrote are bit-identical to the initial table.
    idx_w, M0 = case[0], case[-1]
    for b in range(B):
        for h in range(H):
            untouched = np.ones(s * s, bool)
            untouched[idx_w[b, h].ravel()] = False
            assert np.array_equal(Mg[b, h, untouched], M0[b, h, untouched])


@pytest.mark.parametrize("B,H,dv,form", [
    (3, 17, 96, 0),     # 153 units of 32 columns: two per CTA, one idle half (152 SMs)
    (10, 8, 128, 0),    # 320 units: three per SM, one per CTA
    (5, 10, 128, 1),    # Fig. 2 form at two units per SM
])
def test_scan_many_units_matches_oracle(B, H, dv, form):
    """The launch configurations for more units than SMs, against the oracle
    (small tables and T so the oracle stays quick)."""
    T, s, W, R = 40, 16, 16, 16
    rng = np.random.default_rng(B * 100 + H + form)
    case = random_scan_case(rng, B, H, T, s, dv, W, R, True)
    sh_g = sdm.make_shape(B, H, T, s, 16, dv, W, R, in_dtype=sdm.SDM_BF16, update=form)
    Mg, yg = run_scan(sh_g, case, 0, 0)
    Mo, yo = oracle_scan(B, H, T, s, dv, W, R, case, update_form=form)
    assert max_rel(yg, yo) <= FTOL
    assert max_rel(Mg, Mo) <= FTOL


@pytest.mark.parametrize("form", [0, 1])
@pytest.mark.parametrize("depth", [2, 4, 16])
def test_scan_large_table_reused_rows(form, depth):
    """More than 65536 rows (the plan's filters then hash rows instead of
    indexing them) and every step's rows drawn from a pool of 64, so nearly
    every row is also in flight from the few steps before: the results hinge
    on the forwarded copies."""
    B, H, T, s, dv, W, R = 1, 2, 120, 300, 32, 16, 16
    rng = np.random.default_rng(90000 + depth + 7 * form)
    N = s * s
    pool = np.sort(rng.choice(N, 64, replace=False))
    assert pool.max() >= 65536
    case = list(random_scan_case(rng, B, H, T, 8, dv, W, R, False))
    case[0] = np.stack([pool[rng.choice(64, W, replace=False)] for _ in range(B * H * T)])
    case[0] = case[0].reshape(B, H, T, W).astype(np.int32)
    case[2] = pool[rng.integers(0, 64, (B, H, T, R))].astype(np.int32)
    case[-1] = (rng.standard_normal((B, H, N, dv)) * 0.02).astype(np.float32)
    sh_g = sdm.make_shape(B, H, T, s, 16, dv, W, R, in_dtype=sdm.SDM_F32, update=form)
    Mg, yg = run_scan(sh_g, case, depth, 16)
    Mo, yo = oracle_scan(B, H, T, s, dv, W, R, case, update_form=form)
    assert max_rel(yg, yo) <= FTOL
    assert max_rel(Mg[:, :, pool], Mo[:, :, pool]) <= FTOL
    untouched = np.ones(N, bool)
    untouched[pool] = False
    assert np.array_equal(Mg[:, :, untouched], case[-1][:, :, untouched])


@pytest.mark.parametrize("B,H,T,s,dv,W,R,bf16", [
    (1, 1, 200, 8, 32, 16, 16, False),     # consecutive steps collide constantly
    (2, 3, 150, 16, 64, 32, 48, True),
    (1, 2, 120, 32, 128, 64, 64, True),
    (1, 1, 64, 4, 16, 16, 16, False),      # W = N: the write set is the whole table
    (1, 2, 77, 8, 48, 1, 1, False),
    (1, 1, 40, 16, 1920, 64, 64, True),    # the 8B-scale value width
])
@pytest.mark.parametrize("depth,cs", [(1, 16), (4, 32), (8, 64), (0, 0)])
def test_scan_fig2_matches_oracle(B, H, T, s, dv, W, R, bf16, depth, cs):
    """The shared-residual write read off Fig. 2, against the oracle's form 1."""
    if cs and dv % cs:
        cs = 16
    rng = np.random.default_rng(B * 7000 + T + W)
    case = random_scan_case(rng, B, H, T, s, dv, W, R, bf16)
    sh_g = sdm.make_shape(B, H, T, s, 16, dv, W, R,
                          in_dtype=sdm.SDM_BF16 if bf16 else sdm.SDM_F32,
                          update=sdm.SDM_UPDATE_SHARED_RESIDUAL)
    Mg, yg = run_scan(sh_g, case, depth, cs)
    Mo, yo = oracle_scan(B, H, T, s, dv, W, R, case, update_form=1)
    assert max_rel(yg, yo) <= FTOL
    assert max_rel(Mg, Mo) <= FTOL
    idx_w, M0 = case[0], case[-1]
    for b in range(B):
        for h in range(H):
            untouched = np.ones(s * s, bool)
            untouched[idx_w[b, h].ravel()] = False
            assert np.array_equal(Mg[b, h, untouched], M0[b, h, untouched])


def test_scan_fig2_differs_from_eq4():
    """The two forms are different maps: the same inputs give different tables."""
    rng = np.random.default_rng(5)
    B, H, T, s, dv, W, R = 1, 1, 50, 16, 32, 8, 8
    case = random_scan_case(rng, B, H, T, s, dv, W, R, False)
    M4, _ = run_scan(sdm.make_shape(B, H, T, s, 16, dv, W, R, in_dtype=sdm.SDM_F32), case)
    M2, _ = run_scan(sdm.make_shape(B, H, T, s, 16, dv, W, R, in_dtype=sdm.SDM_F32,
                                    update=sdm.SDM_UPDATE_SHARED_RESIDUAL), case)
    assert max_rel(M4, M2) > 1e-3


def test_scan_depth_invariance_bitwise():
    rng = np.random.default_rng(99)
    B, H, T, s, dv, W, R = 1, 2, 300, 8, 64, 32, 32
    case = random_scan_case(rng, B, H, T, s, dv, W, R, True)
    sh_g = sdm.make_shape(B, H, T, s, 16, dv, W, R, in_dtype=sdm.SDM_BF16)
    M1, y1 = run_scan(sh_g, case, 1, 16)
    for depth in (2, 3, 5, 8, 13):
        M2, y2 = run_scan(sh_g, case, depth, 16)
        assert np.array_equal(M1, M2) and np.array_equal(y1, y2), depth


def test_scan_segments_equal_one_call():
    rng = np.random.default_rng(5)
    B, H, T, s, dv, W, R = 2, 2, 160, 16, 64, 16, 16
    case = random_scan_case(rng, B, H, T, s, dv, W, R, False)
    sh = sdm.make_shape(B, H, T, s, 16, dv, W, R, in_dtype=sdm.SDM_F32)
    M_one, y_one = run_scan(sh, case)
    half = sdm.make_shape(B, H, T // 2, s, 16, dv, W, R, in_dtype=sdm.SDM_F32)
    first = tuple(np.ascontiguousarray(a[:, :, :T // 2]) if isinstance(a, np.ndarray) else
                  a[:, :, :T // 2].contiguous() for a in case[:-1]) + (case[-1],)
    M_a, y_a = run_scan(half, first)
    second = tuple(np.ascontiguousarray(a[:, :, T // 2:]) if isinstance(a, np.ndarray) else
                   a[:, :, T // 2:].contiguous() for a in case[:-1]) + (M_a,)
    M_b, y_b = run_scan(half, second)
    assert np.array_equal(M_one, M_b)
    assert np.array_equal(y_one, np.concatenate([y_a, y_b], axis=2))


# ------------------------------------------------------------------ forward

@pytest.mark.parametrize("name", list(REDUCED))
def test_forward_end_to_end(name):
    forward_check(WORKLOADS[name].with_(**REDUCED[name]))


@pytest.mark.parametrize("name", ["tiny", "mid", "gdn_matched"])
def test_forward_fig2_end_to_end(name):
    forward_check(WORKLOADS[name].with_(update_form=1, **REDUCED[name]))


def forward_check(w):
    """sdm_forward against the oracle.  Selections: equal to the oracle's, or
    different only inside the score gap.  Floats: against the oracle scan
    re-anchored on the device's slots, with weights the oracle computes for
    those slots from its own sub-scores (device weights checked on every
    row); where the slots agree this is the oracle's own forward."""
    x = generate(w)
    sh_g, sh_o = gshape(w, sdm), oshape(w)
    g = {k: t.to(DEV) for k, t in x.items()}
    M = g["M0"].clone()
    out = sdm.sdm_forward(sh_g, g["q_w"], g["q_r"], g["K"], g["alpha"], g["beta"], g["v"], M)
    status_ok()
    ins = [np32(x[k]) for k in ("q_w", "q_r", "K", "alpha", "beta", "v")]
    ref = O.forward(sh_o, *ins, x["M0"].numpy())
    iw, ir = out["idx_w"].cpu().numpy(), out["idx_r"].cpu().numpy()
    S_w = O.subscores(sh_o, ins[0], ins[2])
    S_r = O.subscores(sh_o, ins[1], ins[2])
    check_indices(iw, ref["idx_w"], S_w, w.n_sub)
    check_indices(ir, ref["idx_r"], S_r, w.n_sub)
    ow, orr = oracle_weights(sh_o, S_w, S_r, iw, ir, np32(out["wt_w"]), np32(out["wt_r"]))
    Mo, yo = O.scan(sh_o, iw, ow, ir, orr, ins[3], ins[4], ins[5], x["M0"].numpy())
    assert max_rel(np32(out["y"]), yo) <= FTOL
    assert max_rel(M.cpu().numpy(), Mo) <= FTOL
    if np.array_equal(iw, ref["idx_w"]) and np.array_equal(ir, ref["idx_r"]):
        # Same selections: the re-anchored scan is the oracle's own forward.
        assert np.array_equal(yo, ref["y"]) and np.array_equal(Mo, ref["M"])
    return out, ref, yo


# ------------------------------------------------------------------ edge cases

def test_empty_inputs_are_no_ops():
    sh = sdm.make_shape(0, 2, 5, 8, 16, 32, 4, 4, in_dtype=sdm.SDM_F32)
    z = torch.zeros(16, device=DEV)
    zi = torch.zeros(16, device=DEV, dtype=torch.int32)
    sdm.sdm_scan(sh, zi, z, zi, z, z, z, z, z, y=z)
    sh = sdm.make_shape(1, 1, 0, 8, 16, 32, 4, 4, in_dtype=sdm.SDM_F32)
    sdm.sdm_forward(sh, z, z, z, z, z, z, z, y=z, idx_w=zi, wt_w=z, idx_r=zi, wt_r=z)
    status_ok()


def test_binding_checks_sizes_and_device_before_the_call():
    """The Python binding refuses a tensor smaller than the shape implies
    (before anything reaches the library) and a tensor on a device other than
    the current one."""
    w = WORKLOADS["tiny"].with_(T=10)
    x = generate(w)
    g = {k: t.to(DEV) for k, t in x.items()}
    sh = gshape(w, sdm)
    with pytest.raises(ValueError, match="elements"):
        sdm.sdm_address(sh, g["q_w"][:, :, :5].contiguous(), g["q_r"], g["K"])
    M_small = g["M0"][:, :, :16].contiguous()
    sel = sdm.sdm_address(sh, g["q_w"], g["q_r"], g["K"])
    with pytest.raises(ValueError, match="elements"):
        sdm.sdm_scan(sh, *sel, g["alpha"], g["beta"], g["v"], M_small)
    if torch.cuda.device_count() > 1:
        with pytest.raises(ValueError, match="current device"):
            sdm.sdm_address(sh, g["q_w"].to("cuda:1"), g["q_r"], g["K"])
    status_ok()


def test_single_token_and_single_slot():
    w = WORKLOADS["tiny"].with_(T=1, W=1, R=1)
    x = generate(w)
    g = {k: t.to(DEV) for k, t in x.items()}
    M = g["M0"].clone()
    out = sdm.sdm_forward(gshape(w, sdm), g["q_w"], g["q_r"], g["K"], g["alpha"], g["beta"],
                          g["v"], M)
    status_ok()
    ref = O.forward(oshape(w), *(np32(x[k]) for k in ("q_w", "q_r", "K", "alpha", "beta", "v")),
                    x["M0"].numpy())
    assert np.array_equal(out["idx_w"].cpu().numpy(), ref["idx_w"])
    assert np.all(out["wt_w"].cpu().numpy() == 1.0)
    assert max_rel(np32(out["y"]), ref["y"]) <= FTOL


def test_device_detects_bad_indices():
    B, H, T, s, dv, W, R = 1, 1, 10, 8, 32, 4, 4
    rng = np.random.default_rng(1)
    case = list(random_scan_case(rng, B, H, T, s, dv, W, R, False))
    sh = sdm.make_shape(B, H, T, s, 16, dv, W, R, in_dtype=sdm.SDM_F32)
    bad = case[0].copy()
    bad[0, 0, 3, 1] = s * s          # out of range
    case_b = [bad] + case[1:]
    M = torch.from_numpy(case[-1]).to(DEV)
    args = [torch.from_numpy(a).to(DEV) if isinstance(a, np.ndarray) else a.to(DEV)
            for a in case_b[:-1]]
    sdm.sdm_scan(sh, *args, M)
    assert sdm.sdm_get_device_status() == 5
    dup = case[0].copy()
    dup[0, 0, 4, 2] = dup[0, 0, 4, 0]
    args[0] = torch.from_numpy(dup).to(DEV)
    sdm.sdm_scan(sh, *args, M)
    assert sdm.sdm_get_device_status() == 6
    status_ok()


def test_bounded_wait_reports_timeout():
    sdm.sdm_selftest_wait_timeout(50_000_000)
    assert sdm.sdm_get_device_status() == 4
    status_ok()


# ------------------------------------------------------------------ undo log

UNDO_CASES = [  # B, H, T, s, dv, W, R, bf16
    (1, 2, 120, 4, 32, 8, 8, False),       # N = 16: rows rewritten again and again
    (2, 1, 90, 16, 64, 32, 16, True),
    (1, 1, 60, 32, 128, 64, 64, True),
]


@pytest.mark.parametrize("form", [0, 1])
@pytest.mark.parametrize("B,H,T,s,dv,W,R,bf16", UNDO_CASES)
def test_scan_logged_matches_oracle(B, H, T, s, dv, W, R, bf16, form):
    rng = np.random.default_rng(300 + T + W + form)
    case = random_scan_case(rng, B, H, T, s, dv, W, R, bf16)
    idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M0 = case
    sh_g = sdm.make_shape(B, H, T, s, 16, dv, W, R,
                          in_dtype=sdm.SDM_BF16 if bf16 else sdm.SDM_F32, update=form)
    dev = lambda a: torch.from_numpy(a).to(DEV)
    M = dev(M0)
    y, U = sdm.sdm_scan_logged(sh_g, dev(idx_w), dev(wt_w), dev(idx_r), dev(wt_r),
                               alpha.to(DEV), beta.to(DEV), v.to(DEV), M)
    status_ok()
    # Logging does not change the arithmetic.
    Mp, yp = run_scan(sh_g, case)
    assert np.array_equal(M.cpu().numpy(), Mp) and np.array_equal(y.cpu().numpy(), yp)
    sh_o = O.Shape(B=B, H=H, T=T, n_sub=s, d_h=16, d_v=dv, W=W, R=R, update_form=form)
    Mo, yo, Uo = O.scan(sh_o, idx_w, wt_w.astype(np.float64), idx_r, wt_r.astype(np.float64),
                        np32(alpha), np32(beta), np32(v), M0, log=True)
    assert max_rel(np32(U), Uo) <= FTOL
    assert max_rel(np32(y), yo) <= FTOL


@pytest.mark.parametrize("form", [0, 1])
@pytest.mark.parametrize("B,H,T,s,dv,W,R,bf16", UNDO_CASES)
def test_undo_restores_bit_exactly(B, H, T, s, dv, W, R, bf16, form):
    rng = np.random.default_rng(400 + T + W + form)
    case = random_scan_case(rng, B, H, T, s, dv, W, R, bf16)
    idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M0 = case
    dt = sdm.SDM_BF16 if bf16 else sdm.SDM_F32
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(DEV)
    gates = [alpha.to(DEV), beta.to(DEV), v.to(DEV)]
    for t0 in (0, T // 3, T - 1):
        pre = sdm.make_shape(B, H, t0, s, 16, dv, W, R, in_dtype=dt, update=form)
        tail = sdm.make_shape(B, H, T - t0, s, 16, dv, W, R, in_dtype=dt, update=form)
        M = dev(M0)
        cut = lambda a, sl: a[:, :, sl].clone() if torch.is_tensor(a) else dev(a[:, :, sl])
        P = (idx_w, wt_w, idx_r, wt_r)
        sdm.sdm_scan(pre, *(cut(a, slice(0, t0)) for a in P), *(cut(g, slice(0, t0)) for g in gates), M)
        Mp = M.clone()
        _, U = sdm.sdm_scan_logged(tail, *(cut(a, slice(t0, T)) for a in P),
                                   *(cut(g, slice(t0, T)) for g in gates), M)
        assert not torch.equal(M, Mp)
        sdm.sdm_scan_undo(tail, cut(idx_w, slice(t0, T)), U, M)
        status_ok()
        assert torch.equal(M, Mp), t0


def test_undo_reports_bad_slots():
    B, H, T, s, dv, W = 1, 1, 4, 4, 16, 2
    sh_g = sdm.make_shape(B, H, T, s, 16, dv, W, 1, in_dtype=sdm.SDM_F32)
    idx = torch.tensor([[[[0, 1], [2, 16], [3, 0], [1, 2]]]], dtype=torch.int32, device=DEV)
    U = torch.zeros(B, H, T, W, dv, device=DEV)
    M = torch.ones(B, H, s * s, dv, device=DEV)
    sdm.sdm_scan_undo(sh_g, idx, U, M)
    assert sdm.sdm_get_device_status() == 5
    # The valid rows were still restored (rows 0-3 each from their earliest write).
    assert torch.equal(M[0, 0, :4], torch.zeros(4, dv, device=DEV))
    assert torch.equal(M[0, 0, 4:], torch.ones(s * s - 4, dv, device=DEV))


# ------------------------------------------------------------------ epilogue

@pytest.mark.parametrize("B,H,T,dv,bf16", [(2, 3, 37, 128, True), (1, 2, 5, 16, False),
                                           (1, 2, 9, 1920, True), (3, 1, 64, 960, False)])
@pytest.mark.parametrize("out_dtype", [0, 1])
def test_rmsnorm_gate_matches_oracle(B, H, T, dv, bf16, out_dtype):
    rng = np.random.default_rng(B * 100 + dv + out_dtype)
    y = (rng.standard_normal((B, H, T, dv)) * rng.uniform(0.01, 3, (B, H, T, 1))).astype(np.float32)
    g32 = rng.uniform(-1.5, 1.5, (B, H, T, dv)).astype(np.float32)
    gamma = rng.uniform(0.5, 1.5, (H, dv)).astype(np.float32)
    dt = torch.bfloat16 if bf16 else torch.float32
    g = torch.from_numpy(g32).to(dt)
    sh_g = sdm.make_shape(B, H, T, 16, 16, dv, 1, 1, in_dtype=sdm.SDM_BF16 if bf16 else sdm.SDM_F32)
    out = sdm.sdm_rmsnorm_gate(sh_g, torch.from_numpy(y).to(DEV), g.to(DEV),
                               torch.from_numpy(gamma).to(DEV), eps=1e-6, out_dtype=out_dtype)
    status_ok()
    sh_o = O.Shape(B=B, H=H, T=T, n_sub=16, d_h=16, d_v=dv, W=1, R=1)
    ref = O.rmsnorm_gate(sh_o, y, np32(g), gamma, eps=1e-6)
    got = np32(out)
    scale = np.abs(ref) + 1e-30
    # fp32: a few ulps; bf16: half an ulp of the 8-bit mantissa plus the fp32 error.
    tol = 2e-6 if out_dtype == 0 else 2.0 ** -8 + 2e-6
    assert np.max(np.abs(got - ref) / np.maximum(scale, 1e-3 * np.max(np.abs(ref)))) < tol
    # gamma omitted == gamma of ones.
    ones = torch.ones(H, dv, device=DEV)
    a = sdm.sdm_rmsnorm_gate(sh_g, torch.from_numpy(y).to(DEV), g.to(DEV), None, out_dtype=out_dtype)
    b = sdm.sdm_rmsnorm_gate(sh_g, torch.from_numpy(y).to(DEV), g.to(DEV), ones, out_dtype=out_dtype)
    assert torch.equal(a, b)


def test_forward_then_epilogue_matches_oracle():
    """sdm_forward then sdm_rmsnorm_gate against the oracle epilogue of the
    re-anchored oracle read (asserts on every row, whether or not the
    device's selections equal the oracle's)."""
    w = WORKLOADS["gdn_matched"].with_(B=1, H=2, T=120)
    gate = torch.sigmoid(torch.randn(w.B, w.H, w.T, w.d_v,
                                     generator=torch.Generator().manual_seed(3))).to(torch.bfloat16)
    out, _, yo = forward_check(w)
    sh_g, sh_o = gshape(w, sdm), oshape(w)
    o = sdm.sdm_rmsnorm_gate(sh_g, out["y"], gate.to(DEV), out_dtype=sdm.SDM_F32)
    status_ok()
    ro = O.rmsnorm_gate(sh_o, yo, np32(gate), eps=1e-6)
    assert max_rel(np32(o), ro) <= FTOL


# ------------------------------------------------------------------ decode

DECODE_CASES = [  # B, H, T, s, d_h, d_v, W, R, bf16, score, form
    (3, 2, 1, 32, 16, 32, 8, 8, False, 0, 0),
    (2, 2, 1, 128, 64, 128, 64, 64, True, 0, 0),
    (2, 2, 1, 240, 64, 960, 64, 64, True, 0, 0),      # 1.4B-scale head
    (1, 2, 1, 480, 64, 1920, 64, 64, True, 0, 0),     # 8B-scale head
    (1, 1, 2, 512, 256, 512, 8, 8, False, 1, 0),      # inverse-distance scores
    (2, 1, 3, 8, 16, 64, 16, 16, False, 0, 0),        # rows reused across steps
    (2, 2, 1, 240, 64, 960, 64, 64, True, 0, 1),      # Fig. 2 form
    (2, 1, 3, 8, 16, 64, 16, 16, True, 0, 1),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=lambda c: "B{}H{}T{}s{}dv{}W{}f{}{}".format(
    c[0], c[1], c[2], c[3], c[5], c[6], c[10], "idw" if c[9] else ""))
@pytest.mark.parametrize("epi", [False, True])
def test_decode_matches_oracle(case, epi):
    B, H, T, s, dh, dv, W, R, bf16, score, form = case
    w = WORKLOADS["mid"].with_(B=B, H=H, T=T, n_sub=s, d_h=dh, d_v=16, W=W, R=R, bf16=bf16,
                               score_kind=score, update_form=form,
                               qk_std=1.0 if score else WORKLOADS["mid"].qk_std)
    x = generate(w)                                   # q, K, gates (v, M0 drawn below)
    gen = torch.Generator(device=DEV).manual_seed(s + dv)
    dt = torch.bfloat16 if bf16 else torch.float32
    v = torch.randn(B, H, T, dv, generator=gen, device=DEV).to(dt)
    M0 = torch.randn(B, H, s * s, dv, generator=gen, device=DEV) * 0.02
    sh_g = sdm.make_shape(B, H, T, s, dh, dv, W, R, in_dtype=sdm.SDM_BF16 if bf16 else sdm.SDM_F32,
                          score=score, update=form)
    g = {k: t.to(DEV) for k, t in x.items() if k in ("q_w", "q_r", "K", "alpha", "beta")}
    M = M0.clone()
    gate = gamma = None
    if epi:
        gate = torch.sigmoid(torch.randn(B, H, T, dv, generator=gen, device=DEV)).to(dt)
        gamma = torch.rand(H, dv, generator=gen, device=DEV) + 0.5
    out = sdm.sdm_decode(sh_g, g["q_w"], g["q_r"], g["K"], g["alpha"], g["beta"], v, M,
                         gate=gate, gamma=gamma, out_dtype=sdm.SDM_F32)
    status_ok()
    sh_o = O.Shape(B=B, H=H, T=T, n_sub=s, d_h=dh, d_v=dv, W=W, R=R, score_kind=score,
                   idw_eps=w.idw_eps, update_form=form)
    S_w = O.subscores(sh_o, np32(x["q_w"]), np32(x["K"]))
    S_r = O.subscores(sh_o, np32(x["q_r"]), np32(x["K"]))
    ow, orr = O.select(sh_o, 0, S_w), O.select(sh_o, 1, S_r)
    iw, ir = out["idx_w"].cpu().numpy(), out["idx_r"].cpu().numpy()
    check_indices(iw, ow[0], S_w, s)
    check_indices(ir, orr[0], S_r, s)
    # The scan part, on the device's own selections with the oracle's weights
    # for them (the device's weights checked on every row).
    ww, wr = oracle_weights(sh_o, S_w, S_r, iw, ir, np32(out["wt_w"]), np32(out["wt_r"]))
    rows, Mo, yo = compact_oracle_scan(iw, ww, ir, wr, np32(x["alpha"]), np32(x["beta"]),
                                       np32(v), M0, form)
    assert max_rel(np32(out["y"]), yo) <= FTOL
    Mg = M.cpu().numpy()
    for b in range(B):
        for h in range(H):
            r = rows[b][h]
            assert max_rel(Mg[b, h, r], Mo[b, h, :len(r)]) <= FTOL
    # Only the touched rows changed.
    changed = (M != M0).any(dim=-1).cpu().numpy()
    for b in range(B):
        for h in range(H):
            assert set(np.nonzero(changed[b, h])[0].tolist()) <= set(iw[b, h].ravel().tolist())
    if epi:
        ref = O.rmsnorm_gate(sh_o, yo, np32(gate), np32(gamma), eps=1e-6)
        assert max_rel(np32(out["out"]), ref) <= FTOL


def test_decode_agrees_with_forward():
    """Device vs device at the 1.4B-scale head: same selections wherever the
    two score paths agree, and then the same results."""
    B, H, s, dh, dv = 8, 2, 240, 64, 960
    gen = torch.Generator(device=DEV).manual_seed(7)
    q_w = (torch.randn(B, H, 1, 2, dh, generator=gen, device=DEV) / 4).bfloat16()
    q_r = (torch.randn(B, H, 1, 2, dh, generator=gen, device=DEV) / 4).bfloat16()
    K = (torch.randn(H, 2, s, dh, generator=gen, device=DEV) / 4).bfloat16()
    v = torch.randn(B, H, 1, dv, generator=gen, device=DEV).bfloat16()
    alpha = (0.9 + 0.1 * torch.rand(B, H, 1, generator=gen, device=DEV)).bfloat16()
    beta = torch.rand(B, H, 1, generator=gen, device=DEV).bfloat16()
    M0 = torch.randn(B, H, s * s, dv, generator=gen, device=DEV) * 0.02
    sh = sdm.make_shape(B, H, 1, s, dh, dv, 64, 64)
    M1, M2 = M0.clone(), M0.clone()
    a = sdm.sdm_decode(sh, q_w, q_r, K, alpha, beta, v, M1)
    b = sdm.sdm_forward(sh, q_w, q_r, K, alpha, beta, v, M2)
    status_ok()
    same = (torch.all(a["idx_w"] == b["idx_w"], -1) & torch.all(a["idx_r"] == b["idx_r"], -1))
    assert same.float().mean() > 0.9
    ya, yb = np32(a["y"]), np32(b["y"])
    sm = same.cpu().numpy()
    assert max_rel(ya[sm], yb[sm]) <= FTOL


SEGMENTED = [  # sdm_forward cuts T >= 2048 into windows and overlaps their addressing
    dict(B=3, H=17, T=2300, n_sub=64, d_h=32, d_v=96, W=16, R=16, bf16=True),    # 153 units: two per CTA, one idle half
    dict(B=1, H=2, T=4100, n_sub=64, d_h=32, d_v=64, W=32, R=32, bf16=False),    # one unit per SM, uneven last window
    dict(B=2, H=2, T=2048, n_sub=32, d_h=16, d_v=32, W=8, R=8, bf16=False, update_form=1),
]


@pytest.mark.parametrize("ov", SEGMENTED, ids=lambda o: "B{B}H{H}T{T}dv{d_v}".format(**o))
def test_forward_windows_equal_address_then_scan(ov):
    w = WORKLOADS["mid"].with_(**ov)
    x = generate(w)
    sh = gshape(w, sdm)
    g = {k: t.to(DEV) for k, t in x.items()}
    M1, M2 = g["M0"].clone(), g["M0"].clone()
    out = [torch.empty(w.B, w.H, w.T, n, dtype=dt, device=DEV)
           for n, dt in ((w.W, torch.int32), (w.W, torch.float32), (w.R, torch.int32),
                         (w.R, torch.float32))]
    y1 = sdm.sdm_forward(sh, g["q_w"], g["q_r"], g["K"], g["alpha"], g["beta"], g["v"], M1,
                         None, *out)["y"]
    sel = sdm.sdm_address(sh, g["q_w"], g["q_r"], g["K"])
    y2 = sdm.sdm_scan(sh, *sel, g["alpha"], g["beta"], g["v"], M2)
    torch.cuda.synchronize()
    status_ok()
    for a, b in zip(out, sel):
        assert torch.equal(a, b)
    assert torch.equal(y1, y2) and torch.equal(M1, M2)


def test_forward_windows_tensor_core_shapes():
    # Tensor-core addressing: 512-step windows, at most 32.
    tc = dict(n_sub=256, d_h=64, d_v=128, W=64, R=64)
    mk = lambda T: sdm.make_shape(2, 2, T, **tc)
    assert sdm.sdm_forward_windows(mk(2047)) == 1
    assert sdm.sdm_forward_windows(mk(4096)) == 8
    assert sdm.sdm_forward_windows(mk(131072)) == 32


def test_forward_windows_in_a_captured_graph():
    """The windowed forward forks onto the library's own streams and joins
    back into the caller's; captured in a CUDA graph and replayed it gives
    exactly the eager result."""
    w = WORKLOADS["mid"].with_(B=1, H=2, T=2100)            # 4 windows
    assert sdm.sdm_forward_windows(gshape(w, sdm)) > 1
    x = generate(w)
    sh = gshape(w, sdm)
    g = {k: t.to(DEV) for k, t in x.items()}
    M1 = g["M0"].clone()
    ref = sdm.sdm_forward(sh, g["q_w"], g["q_r"], g["K"], g["alpha"], g["beta"], g["v"], M1)
    M2 = g["M0"].clone()
    y2 = torch.empty_like(ref["y"])
    sel = [torch.empty_like(ref[k]) for k in ("idx_w", "wt_w", "idx_r", "wt_r")]
    ws = torch.empty(max(16, sdm.sdm_workspace_size(sh)), dtype=torch.uint8, device=DEV)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):                            # warm-up outside the capture
        sdm.sdm_forward(sh, g["q_w"], g["q_r"], g["K"], g["alpha"], g["beta"], g["v"], M2, y2,
                        *sel, workspace=ws, stream=side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=side):
        sdm.sdm_forward(sh, g["q_w"], g["q_r"], g["K"], g["alpha"], g["beta"], g["v"], M2, y2,
                        *sel, workspace=ws, stream=side)
    M2.copy_(g["M0"])
    y2.zero_()
    graph.replay()
    torch.cuda.synchronize()
    status_ok()
    assert torch.equal(y2, ref["y"]) and torch.equal(M2, M1)
    for a, k in zip(sel, ("idx_w", "wt_w", "idx_r", "wt_r")):
        assert torch.equal(a, ref[k])


@pytest.mark.parametrize("depth,cs", [(2, 16), (5, 0)])
def test_forward_windows_under_scan_tuning(depth, cs):
    w = WORKLOADS["mid"].with_(B=1, H=3, T=2200)
    x = generate(w)
    sh = gshape(w, sdm)
    g = {k: t.to(DEV) for k, t in x.items()}
    sdm.sdm_set_scan_tuning(depth, cs)
    try:
        M1, M2 = g["M0"].clone(), g["M0"].clone()
        y1 = sdm.sdm_forward(sh, g["q_w"], g["q_r"], g["K"], g["alpha"], g["beta"], g["v"],
                             M1)["y"]
        sel = sdm.sdm_address(sh, g["q_w"], g["q_r"], g["K"])
        y2 = sdm.sdm_scan(sh, *sel, g["alpha"], g["beta"], g["v"], M2)
        torch.cuda.synchronize()
        status_ok()
        assert torch.equal(y1, y2) and torch.equal(M1, M2)
    finally:
        sdm.sdm_set_scan_tuning(0, 0)
