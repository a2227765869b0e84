"""Pins of the CPU oracle against what the pages and the mathematics fix.

Every check here is independent of the oracle's own code: values printed on
the pages (tests/golden), closed forms of the recurrence, brute force over all
N slots, library routines (numpy) for the sub-scores, and the dense Gated
DeltaNet equation that the shared-residual form must reduce to.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def sh(**kw):
    base = dict(B=1, H=1, T=1, n_sub=4, d_h=4, d_v=1, W=2, R=2)
    base.update(kw)
    return O.Shape(**base)


# ----------------------------------------------------------------- addressing

def test_pkm_worked_example(oracle_mod):
    """SDM reading notes 2.3 teaching example: sums {7,6,4,3}, best two 7 and 6."""
    g = gold("pkm_addressing_example.json")
    s = g["n_sub"]
    S = np.array([g["half1"], g["half2"]], np.float32).reshape(1, 1, 1, 2, s)
    shape = sh(n_sub=s, W=g["W"], R=g["W"])
    idx, sc, wt = O.select(shape, 0, S)
    assert sc[0, 0, 0].tolist() == g["selected_sums"]
    assert idx[0, 0, 0].tolist() == g["selected_slots"]
    e = math.e
    assert wt[0, 0, 0] == pytest.approx([e / (1 + e), 1 / (1 + e)], abs=1e-15)
    # The full candidate set of the two top-2 lists: ask for all four of them.
    shape4 = sh(n_sub=s, W=4, R=4, k_w=2, k_r=2)
    idx4, sc4, _ = O.select(shape4, 0, S)
    assert sc4[0, 0, 0].tolist() == g["candidate_sums"]
    assert idx4[0, 0, 0].tolist() == [0, 1, 4, 5]


def brute_force(S, n_sel):
    """Top n_sel of all s*s float sums by (sum desc, slot asc), no pruning."""
    s = S.shape[-1]
    sums = (S[0][:, None] + S[1][None, :]).astype(np.float32).reshape(-1)
    slots = np.arange(s * s)
    order = np.lexsort((slots, -sums.astype(np.float64)))
    return slots[order[:n_sel]], sums[order[:n_sel]]


@pytest.mark.parametrize("s,W,seed", [(4, 2, 0), (8, 8, 1), (16, 16, 2), (16, 5, 3),
                                      (32, 8, 4), (8, 64, 5), (64, 64, 6)])
def test_select_matches_brute_force(oracle_mod, s, W, seed):
    rng = np.random.default_rng(seed)
    T = 40
    S = rng.standard_normal((1, 1, T, 2, s)).astype(np.float32)
    shape = sh(T=T, n_sub=s, W=W, R=W)
    idx, sc, wt = O.select(shape, 0, S)
    for t in range(T):
        bidx, bsum = brute_force(S[0, 0, t], W)
        assert np.array_equal(np.sort(sc[0, 0, t]), np.sort(bsum))
        assert idx[0, 0, t].tolist() == bidx.tolist()
        assert abs(wt[0, 0, t].sum() - 1) < 1e-12


def test_select_ties_keep_score_multiset(oracle_mod):
    """Heavily tied integer scores: the selected sums always equal brute force's;
    slots equal it except where a tie straddles the W-th position."""
    rng = np.random.default_rng(7)
    s, W, T = 8, 8, 200
    S = rng.integers(-3, 4, size=(1, 1, T, 2, s)).astype(np.float32)
    idx, sc, _ = O.select(sh(T=T, n_sub=s, W=W, R=W), 0, S)
    straddle = 0
    for t in range(T):
        bidx, bsum = brute_force(S[0, 0, t], W)
        assert sc[0, 0, t].tolist() == bsum.tolist()
        allsums = np.sort((S[0, 0, t, 0][:, None] + S[0, 0, t, 1][None, :]).ravel())[::-1]
        tie_at_edge = allsums[W - 1] == allsums[W]
        straddle += tie_at_edge
        if not tie_at_edge:
            assert idx[0, 0, t].tolist() == bidx.tolist()
        # Every selected slot really carries the reported sum.
        a, b = idx[0, 0, t] // s, idx[0, 0, t] % s
        assert np.array_equal(S[0, 0, t, 0][a] + S[0, 0, t, 1][b], sc[0, 0, t])
    assert straddle > 0


def test_select_constant_scores(oracle_mod):
    """All sums equal: the lowest slots win and each weight is exactly 1/W."""
    s, W = 16, 8
    S = np.full((1, 1, 3, 2, s), 0.37, np.float32)
    idx, sc, wt = O.select(sh(T=3, n_sub=s, W=W, R=W), 0, S)
    assert idx[0, 0, 0].tolist() == list(range(W))
    assert np.all(wt == 1.0 / W)


def test_select_single_slot_weight_one(oracle_mod):
    rng = np.random.default_rng(3)
    S = rng.standard_normal((1, 1, 5, 2, 8)).astype(np.float32)
    _, _, wt = O.select(sh(T=5, n_sub=8, W=1, R=1), 0, S)
    assert np.all(wt == 1.0)


def test_select_dominant_entry(oracle_mod):
    """One huge half-1 entry: every selected slot uses it, ordered by half 2."""
    rng = np.random.default_rng(4)
    s, W = 16, 6
    S = rng.standard_normal((1, 1, 1, 2, s)).astype(np.float32)
    S[0, 0, 0, 0, 11] = 100.0
    idx, _, _ = O.select(sh(n_sub=s, W=W, R=W), 0, S)
    a, b = idx[0, 0, 0] // s, idx[0, 0, 0] % s
    assert np.all(a == 11)
    assert b.tolist() == np.argsort(-S[0, 0, 0, 1], kind="stable")[:W].tolist()


def test_weights_entropy_range(oracle_mod):
    """u(p) = exp(H(p))/k lies in [1/k, 1] (SDM notes 4.7 / App. D.1 access metric)."""
    rng = np.random.default_rng(5)
    W = 16
    S = (rng.standard_normal((1, 1, 50, 2, 16)) * 3).astype(np.float32)
    _, _, wt = O.select(sh(T=50, n_sub=16, W=W, R=W), 0, S)
    H = -(wt * np.log(np.maximum(wt, 1e-300))).sum(-1)
    u = np.exp(H) / W
    assert np.all(u >= 1.0 / W - 1e-12) and np.all(u <= 1 + 1e-12)


def test_slot_weights_worked_example(oracle_mod):
    """SDM reading notes 2.3 example: weights of slots [0, 1] (sums 7, 6) are
    e/(1+e) and 1/(1+e), in either list order; slot 5 (sum 1 + 2 = 3)
    scores through half 1 entry 1 and half 2 entry 1."""
    g = gold("pkm_addressing_example.json")
    s = g["n_sub"]
    S = np.array([g["half1"], g["half2"]], np.float32).reshape(1, 1, 1, 2, s)
    shape = sh(n_sub=s, W=2, R=2)
    e = math.e
    wt = O.slot_weights(shape, 0, S, np.array([0, 1], np.int32).reshape(1, 1, 1, 2))
    assert wt[0, 0, 0] == pytest.approx([e / (1 + e), 1 / (1 + e)], abs=1e-15)
    wt = O.slot_weights(shape, 1, S, np.array([1, 0], np.int32).reshape(1, 1, 1, 2))
    assert wt[0, 0, 0] == pytest.approx([1 / (1 + e), e / (1 + e)], abs=1e-15)
    # Sums 7 (slot 0) and 3 (slot 5): weights 1/(1+e^-4) and e^-4/(1+e^-4).
    wt = O.slot_weights(shape, 0, S, np.array([5, 0], np.int32).reshape(1, 1, 1, 2))
    q = math.exp(-4.0)
    assert wt[0, 0, 0] == pytest.approx([q / (1 + q), 1 / (1 + q)], abs=1e-15)


def test_slot_weights_log_scores_normalise(oracle_mod):
    """Half 1 all zero and half 2 entry b = ln(b + 1): the softmax of
    ln(b + 1) over the listed slots is (b + 1) / sum(b + 1), whatever the
    half-1 index; a swapped slot map (a = slot % s) would read zeros."""
    s, n = 16, 7
    rng = np.random.default_rng(11)
    S = np.zeros((1, 1, 3, 2, s), np.float32)
    S[..., 1, :] = np.log(np.arange(1, s + 1, dtype=np.float64)).astype(np.float32)
    idx = np.stack([rng.choice(s * s, n, replace=False) for _ in range(3)]).astype(np.int32)
    idx = idx.reshape(1, 1, 3, n)
    wt = O.slot_weights(sh(T=3, n_sub=s, W=n, R=n), 0, S, idx)
    b = (idx % s).astype(np.float64)
    # Expected from the float32-rounded logs, so only the softmax is exercised.
    ev = np.exp(S[0, 0, :, 1][np.arange(3)[:, None], idx[0, 0] % s].astype(np.float64))
    assert np.allclose(wt[0, 0], ev / ev.sum(-1, keepdims=True), atol=1e-15, rtol=0)
    assert np.allclose(wt[0, 0], (b + 1) / (b + 1).sum(-1, keepdims=True), atol=1e-6)


def test_slot_weights_invariants(oracle_mod):
    """Weights sum to 1, a single slot gets exactly 1, equal sums get exactly
    1/n, and a slot outside the table is rejected."""
    rng = np.random.default_rng(12)
    s, T = 8, 20
    S = rng.standard_normal((1, 1, T, 2, s)).astype(np.float32)
    idx = np.stack([rng.choice(s * s, 8, replace=False) for _ in range(T)]).astype(np.int32)
    wt = O.slot_weights(sh(T=T, n_sub=s, W=8, R=8), 0, S, idx.reshape(1, 1, T, 8))
    assert np.all(np.abs(wt.sum(-1) - 1) < 1e-12) and np.all(wt > 0)
    one = O.slot_weights(sh(T=T, n_sub=s, W=1, R=1), 1, S, idx[:, :1].reshape(1, 1, T, 1))
    assert np.all(one == 1.0)
    flat = np.full((1, 1, 1, 2, s), 0.25, np.float32)
    eq = O.slot_weights(sh(n_sub=s, W=4, R=4), 0, flat, np.array([[[[3, 9, 60, 1]]]], np.int32))
    assert np.all(eq == 0.25)
    with pytest.raises(ValueError):
        O.slot_weights(sh(n_sub=s, W=1, R=1), 0, flat, np.array([[[[s * s]]]], np.int32))


def test_permuting_subkeys_permutes_slots(oracle_mod):
    rng = np.random.default_rng(6)
    s, dh, W = 16, 8, 8
    shape = sh(T=10, n_sub=s, d_h=dh, W=W, R=W)
    q = rng.standard_normal((1, 1, 10, 2, dh)).astype(np.float32)
    K = rng.standard_normal((1, 2, s, dh)).astype(np.float32)
    perm = rng.permutation(s)
    Kp = K.copy()
    Kp[0, 0] = K[0, 0, perm]
    idx, _, _ = O.select(shape, 0, O.subscores(shape, q, K))
    idxp, _, _ = O.select(shape, 0, O.subscores(shape, q, Kp))
    # Row j of the permuted table is row perm[j] of the original one.
    a_p, b_p = idxp // s, idxp % s
    assert np.array_equal(perm[a_p] * s + b_p, idx)


# ----------------------------------------------------------------- sub-scores

def test_dot_subscores_match_numpy(oracle_mod):
    rng = np.random.default_rng(8)
    shape = sh(B=2, H=3, T=5, n_sub=8, d_h=16)
    q = rng.standard_normal((2, 3, 5, 2, 16)).astype(np.float32)
    K = rng.standard_normal((3, 2, 8, 16)).astype(np.float32)
    S = O.subscores(shape, q, K)
    ref = np.einsum("bhtpc,hpjc->bhtpj", q.astype(np.float64), K.astype(np.float64))
    assert np.max(np.abs(S - ref.astype(np.float32))) <= 1e-6 * np.max(np.abs(ref))


def test_idw_subscores(oracle_mod):
    """FwPKM notes 2.2: s = -log(1e-3 + |q-K|^2); q equal to a key scores -ln(1e-3)."""
    rng = np.random.default_rng(9)
    shape = sh(B=1, H=1, T=4, n_sub=16, d_h=32, score_kind=1)
    K = rng.standard_normal((1, 2, 16, 32)).astype(np.float32)
    q = rng.standard_normal((1, 1, 4, 2, 32)).astype(np.float32)
    q[0, 0, 0, 0] = K[0, 0, 5]
    q[0, 0, 0, 1] = K[0, 1, 9]
    S = O.subscores(shape, q, K)
    d2 = ((q[0, 0][:, :, None, :].astype(np.float64) - K[0][None].astype(np.float64)) ** 2).sum(-1)
    ref = -np.log(1e-3 + d2)
    assert np.allclose(S[0, 0], ref, rtol=0, atol=2e-6)
    assert S[0, 0, 0, 0, 5] == np.float32(-math.log(1e-3))
    assert abs(S[0, 0, 0, 0, 5] - 6.907755) < 1e-6
    shape8 = sh(B=1, H=1, T=4, n_sub=16, d_h=32, score_kind=1, W=8, R=8)
    idx, _, _ = O.select(shape8, 0, S)
    assert idx[0, 0, 0, 0] == 5 * 16 + 9


# ----------------------------------------------------------------- recurrence

def test_eq4_and_fig2_counter_example(oracle_mod):
    """SDM reading notes 2.5: Eq. (4) gives [4, 5.5]; the Fig. 2 form [3.75, 5.75]."""
    g = gold("eq4_vs_fig2_example.json")
    for form, want in ((0, g["eq4_rows"]), (1, g["fig2_rows"])):
        shape = sh(n_sub=2, d_v=1, W=2, R=1, update_form=form)
        M0 = np.array([g["old_rows"][0], g["old_rows"][1], -7.0, 11.0]).reshape(1, 1, 4, 1)
        idx_w = np.array([0, 1], np.int32).reshape(1, 1, 1, 2)
        wt_w = np.array(g["write_weights"]).reshape(1, 1, 1, 2)
        idx_r = np.array([1], np.int32).reshape(1, 1, 1, 1)
        wt_r = np.ones((1, 1, 1, 1))
        M, y = O.scan(shape, idx_w, wt_w, idx_r, wt_r, np.full((1, 1, 1), g["alpha"]),
                      np.full((1, 1, 1), g["beta"]), np.full((1, 1, 1, 1), g["v"]), M0)
        # alpha = 0.8 enters as float32 (0.800000012); the page's arithmetic is exact.
        assert M[0, 0, :2, 0] == pytest.approx(want, rel=1e-7)
        assert M[0, 0, 2:, 0].tolist() == [-7.0, 11.0]          # untouched rows
        assert y[0, 0, 0, 0] == M[0, 0, 1, 0]                    # read sees the write


def random_scan_inputs(rng, shape, distinct=True):
    B, H, T, N = shape.B, shape.H, shape.T, shape.N
    idx_w = np.stack([rng.choice(N, shape.W, replace=False) for _ in range(B * H * T)])
    idx_w = idx_w.reshape(B, H, T, shape.W).astype(np.int32)
    idx_r = rng.integers(0, N, size=(B, H, T, shape.R)).astype(np.int32)
    wt_w = rng.dirichlet(np.ones(shape.W), size=(B, H, T))
    wt_r = rng.dirichlet(np.ones(shape.R), size=(B, H, T))
    alpha = rng.uniform(0.9, 1, (B, H, T)).astype(np.float32)
    beta = rng.uniform(0, 1, (B, H, T)).astype(np.float32)
    v = rng.standard_normal((B, H, T, shape.d_v)).astype(np.float32)
    M0 = (rng.standard_normal((B, H, N, shape.d_v)) * 0.02).astype(np.float32)
    return idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M0


def test_untouched_rows_bit_identical(oracle_mod):
    """SDM reading notes 2.4: unselected slots keep M_t[i] = M_{t-1}[i] exactly."""
    rng = np.random.default_rng(10)
    shape = sh(B=2, H=2, T=30, n_sub=16, d_v=8, W=4, R=4)
    args = random_scan_inputs(rng, shape)
    M, _ = O.scan(shape, *args)
    M0 = args[-1].astype(np.float64)
    idx_w = args[0]
    for b in range(2):
        for h in range(2):
            touched = np.zeros(shape.N, bool)
            touched[idx_w[b, h].ravel()] = True
            assert np.array_equal(M[b, h, ~touched], M0[b, h, ~touched])
            assert not np.array_equal(M[b, h, touched], M0[b, h, touched])


def test_repeated_single_slot_closed_form(oracle_mod):
    """W=1 with weight 1 on one slot and constant gates: m_t = m* + (m0-m*) r^t,
    r = alpha(1-beta), m* = beta v / (1 - r)."""
    T = 60
    shape = sh(T=T, n_sub=4, d_v=3, W=1, R=1)
    a, b = 0.93, 0.35
    v = np.array([1.5, -2.0, 0.25], np.float32)
    M0 = np.zeros((1, 1, 16, 3), np.float32)
    M0[0, 0, 6] = [0.7, 0.1, -0.4]
    idx = np.full((1, 1, T, 1), 6, np.int32)
    one = np.ones((1, 1, T, 1))
    M, y = O.scan(shape, idx, one, idx, one, np.full((1, 1, T), a, np.float32),
                  np.full((1, 1, T), b, np.float32), np.tile(v, (1, 1, T, 1)), M0)
    a64, b64 = float(np.float32(a)), float(np.float32(b))
    r = a64 * (1 - b64)
    mstar = b64 * v.astype(np.float64) / (1 - r)
    for t in range(T):
        want = mstar + (M0[0, 0, 6].astype(np.float64) - mstar) * r ** (t + 1)
        assert np.allclose(y[0, 0, t], want, rtol=1e-12, atol=1e-14)


def test_beta_one_single_slot_overwrites(oracle_mod):
    rng = np.random.default_rng(11)
    shape = sh(T=20, n_sub=8, d_v=16, W=1, R=1)
    idx_w = rng.integers(0, 64, (1, 1, 20, 1)).astype(np.int32)
    one = np.ones((1, 1, 20, 1))
    v = rng.standard_normal((1, 1, 20, 16)).astype(np.float32)
    M0 = rng.standard_normal((1, 1, 64, 16)).astype(np.float32)
    M, y = O.scan(shape, idx_w, one, idx_w, one, rng.uniform(0.5, 1, (1, 1, 20)).astype(np.float32),
                  np.ones((1, 1, 20), np.float32), v, M0)
    assert np.allclose(y[0, 0], v[0, 0].astype(np.float64), rtol=0, atol=4e-16 * 8)


def test_all_slots_selected_dense_recurrence(oracle_mod):
    """W = N: the selection covers every slot and each row follows the dense
    per-slot gated recurrence (checked in matrix form)."""
    rng = np.random.default_rng(12)
    s, T, dv, dh = 4, 12, 5, 6
    N = s * s
    shape = sh(T=T, n_sub=s, d_h=dh, d_v=dv, W=N, R=N)
    q_w = rng.standard_normal((1, 1, T, 2, dh)).astype(np.float32)
    q_r = rng.standard_normal((1, 1, T, 2, dh)).astype(np.float32)
    K = rng.standard_normal((1, 2, s, dh)).astype(np.float32)
    alpha = rng.uniform(0.9, 1, (1, 1, T)).astype(np.float32)
    beta = rng.uniform(0, 1, (1, 1, T)).astype(np.float32)
    v = rng.standard_normal((1, 1, T, dv)).astype(np.float32)
    M0 = rng.standard_normal((1, 1, N, dv)).astype(np.float32)
    out = O.forward(shape, q_w, q_r, K, alpha, beta, v, M0)
    assert all(sorted(r) == list(range(N)) for r in out["idx_w"][0, 0])
    Mref = M0[0, 0].astype(np.float64)
    for t in range(T):
        w = np.zeros(N)
        w[out["idx_w"][0, 0, t]] = out["wt_w"][0, 0, t]
        a, b = float(alpha[0, 0, t]), float(beta[0, 0, t])
        Mref = a * Mref + (b * w)[:, None] * (v[0, 0, t][None, :].astype(np.float64) - a * Mref)
    assert np.allclose(out["M"][0, 0], Mref, rtol=1e-12, atol=1e-12)


def test_fig2_form_with_all_slots_is_gated_deltanet(oracle_mod):
    """SDM reading notes 2.1 Eq. (2) / 2.5: with every slot selected and dense
    weights k, the shared-residual form is exactly Gated DeltaNet,
    M_t = a M + b k (v - a M^T k)^T."""
    rng = np.random.default_rng(13)
    s, T, dv = 4, 10, 3
    N = s * s
    shape = sh(T=T, n_sub=s, d_v=dv, W=N, R=1, update_form=1)
    idx_w = np.stack([rng.permutation(N) for _ in range(T)]).reshape(1, 1, T, N).astype(np.int32)
    wt_w = rng.dirichlet(np.ones(N), size=(1, 1, T))
    idx_r = np.zeros((1, 1, T, 1), np.int32)
    alpha = rng.uniform(0.8, 1, (1, 1, T)).astype(np.float32)
    beta = rng.uniform(0, 1, (1, 1, T)).astype(np.float32)
    v = rng.standard_normal((1, 1, T, dv)).astype(np.float32)
    M0 = rng.standard_normal((1, 1, N, dv)).astype(np.float32)
    M, _ = O.scan(shape, idx_w, wt_w, idx_r, np.ones((1, 1, T, 1)), alpha, beta, v, M0)
    Mg = M0[0, 0].astype(np.float64)
    for t in range(T):
        k = np.zeros(N)
        k[idx_w[0, 0, t]] = wt_w[0, 0, t]
        a, b = float(alpha[0, 0, t]), float(beta[0, 0, t])
        Mg = a * Mg + b * np.outer(k, v[0, 0, t].astype(np.float64) - a * Mg.T @ k)
    assert np.allclose(M[0, 0], Mg, rtol=1e-12, atol=1e-12)


def test_read_single_row(oracle_mod):
    rng = np.random.default_rng(14)
    shape = sh(B=1, H=2, T=15, n_sub=8, d_v=4, W=3, R=1)
    idx_w, wt_w, idx_r, _, alpha, beta, v, M0 = random_scan_inputs(rng, shape)
    one = np.ones((1, 2, 15, 1))
    M, y = O.scan(shape, idx_w, wt_w, idx_r, one, alpha, beta, v, M0)
    # Replaying the first t+1 steps and reading the row directly gives y_t.
    for t in (0, 7, 14):
        sub = sh(B=1, H=2, T=t + 1, n_sub=8, d_v=4, W=3, R=1)
        Mt, _ = O.scan(sub, idx_w[:, :, :t + 1], wt_w[:, :, :t + 1], idx_r[:, :, :t + 1],
                       one[:, :, :t + 1], alpha[:, :, :t + 1], beta[:, :, :t + 1],
                       v[:, :, :t + 1], M0)
        for h in range(2):
            assert np.array_equal(y[0, h, t], Mt[0, h, idx_r[0, h, t, 0]])


def test_segmented_scan_equals_single_call(oracle_mod):
    rng = np.random.default_rng(15)
    shape = sh(B=2, H=1, T=40, n_sub=8, d_v=6, W=5, R=7)
    idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M0 = random_scan_inputs(rng, shape)
    M, y = O.scan(shape, idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M0)
    half = sh(B=2, H=1, T=20, n_sub=8, d_v=6, W=5, R=7)
    sl = [slice(None), slice(None)]
    M1, y1 = O.scan(half, *(a[:, :, :20] for a in (idx_w, wt_w, idx_r, wt_r, alpha, beta, v)), M0)
    M2, y2 = O.scan(half, *(a[:, :, 20:] for a in (idx_w, wt_w, idx_r, wt_r, alpha, beta, v)), M1)
    assert np.array_equal(M, M2)
    assert np.array_equal(y, np.concatenate([y1, y2], axis=2))


def test_scan_rejects_bad_indices(oracle_mod):
    shape = sh(T=1, n_sub=2, d_v=1, W=2, R=1)
    z = np.zeros((1, 1, 1, 1))
    args = dict(wt_w=np.ones((1, 1, 1, 2)) / 2, idx_r=np.zeros((1, 1, 1, 1), np.int32),
                wt_r=np.ones((1, 1, 1, 1)), alpha=np.ones((1, 1, 1)), beta=np.ones((1, 1, 1)),
                v=z, M0=np.zeros((1, 1, 4, 1)))
    with pytest.raises(ValueError):
        O.scan(shape, np.array([0, 4], np.int32).reshape(1, 1, 1, 2), **args)
    with pytest.raises(ValueError):
        O.scan(shape, np.array([1, 1], np.int32).reshape(1, 1, 1, 2), **args)


# ------------------------------------------------------------------ undo log
# [SDM notes] 2.9 (appendix A.3, backward memory): the forward pass writes in
# place; earlier states come back by undoing the sparse writes, for O(T W d_v)
# memory -- a log of the rows each step overwrote.

def test_logged_scan_equals_plain_scan(oracle_mod):
    rng = np.random.default_rng(21)
    shape = sh(B=2, H=2, T=25, n_sub=4, d_v=5, W=6, R=3)     # N=16: heavy reuse
    args = random_scan_inputs(rng, shape)
    M, y = O.scan(shape, *args)
    M2, y2, U = O.scan(shape, *args, log=True)
    assert np.array_equal(M, M2) and np.array_equal(y, y2)
    assert U.shape == (2, 2, 25, 6, 5)


@pytest.mark.parametrize("form", [0, 1])
def test_undo_log_holds_pre_write_rows(oracle_mod, form):
    """Brute force: the log row of (t, j) is row idx_w[t, j] of the table after
    the first t steps, computed by an independent scan of those steps."""
    rng = np.random.default_rng(22 + form)
    shape = sh(B=1, H=2, T=12, n_sub=3, d_v=4, W=4, R=2, update_form=form)
    idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M0 = random_scan_inputs(rng, shape)
    _, _, U = O.scan(shape, idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M0, log=True)
    Mt = M0.astype(np.float64)
    for t in range(shape.T):
        for h in range(2):
            for j in range(shape.W):
                assert np.array_equal(U[0, h, t, j], Mt[0, h, idx_w[0, h, t, j]])
        one = sh(B=1, H=2, T=1, n_sub=3, d_v=4, W=4, R=2, update_form=form)
        st = slice(t, t + 1)
        Mt, _ = O.scan(one, idx_w[:, :, st], wt_w[:, :, st], idx_r[:, :, st], wt_r[:, :, st],
                       alpha[:, :, st], beta[:, :, st], v[:, :, st], Mt)


def test_undo_log_closed_form_single_slot(oracle_mod):
    """W=1, weight 1, constant gates: the row before step t is
    m* + (m0 - m*) r^t with r = alpha (1 - beta), m* = beta v / (1 - r)."""
    T, a, b, v0, m0 = 9, 0.9, 0.3, 2.0, 0.5
    shape = sh(T=T, n_sub=2, d_v=1, W=1, R=1)
    ones = np.ones((1, 1, T, 1))
    idx = np.full((1, 1, T, 1), 3, np.int32)
    M0 = np.zeros((1, 1, 4, 1)); M0[0, 0, 3, 0] = m0
    _, _, U = O.scan(shape, idx, ones, idx, ones, np.full((1, 1, T), a, np.float32),
                     np.full((1, 1, T), b, np.float32), np.full((1, 1, T, 1), v0, np.float32),
                     M0, log=True)
    af, bf = float(np.float32(a)), float(np.float32(b))
    r = af * (1 - bf)
    ms = bf * v0 / (1 - r)
    for t in range(T):
        assert U[0, 0, t, 0, 0] == pytest.approx(ms + (m0 - ms) * r ** t, rel=1e-12)


@pytest.mark.parametrize("form", [0, 1])
def test_undo_restores_the_segment_start(oracle_mod, form):
    """undo(tail) on the table after prefix+tail gives back exactly the table
    after the prefix (the earliest logged copy of a reused row wins)."""
    rng = np.random.default_rng(24 + form)
    full = sh(B=2, H=1, T=40, n_sub=4, d_v=3, W=5, R=2, update_form=form)
    idx_w, wt_w, idx_r, wt_r, alpha, beta, v, M0 = random_scan_inputs(rng, full)
    for t0 in (0, 1, 17, 39):
        pre = sh(B=2, H=1, T=t0, n_sub=4, d_v=3, W=5, R=2, update_form=form)
        tail = sh(B=2, H=1, T=40 - t0, n_sub=4, d_v=3, W=5, R=2, update_form=form)
        cut = lambda a, s: a[:, :, s]
        P = (idx_w, wt_w, idx_r, wt_r, alpha, beta, v)
        Mp, _ = O.scan(pre, *(cut(a, slice(0, t0)) for a in P), M0)
        Mt, _, U = O.scan(tail, *(cut(a, slice(t0, 40)) for a in P), Mp, log=True)
        Mr = O.undo(tail, idx_w[:, :, t0:], U, Mt)
        assert np.array_equal(Mr, Mp), t0


# ------------------------------------------------------------------ epilogue
# [SDM notes] 2.4, after Eq. (5): per-head RMS-Norm, then the element-wise
# output gate.

def test_rmsnorm_gate_unit_rms_and_closed_forms(oracle_mod):
    rng = np.random.default_rng(31)
    shape = sh(B=2, H=3, T=5, d_v=12)
    y = rng.standard_normal((2, 3, 5, 12))
    ones = np.ones((2, 3, 5, 12), np.float32)
    out = O.rmsnorm_gate(shape, y, ones, eps=1e-300)
    # Unit RMS per (b, h, t) row, direction kept.
    assert np.allclose(np.sqrt(np.mean(out ** 2, axis=-1)), 1.0, rtol=1e-12)
    assert np.allclose(out * np.linalg.norm(y, axis=-1, keepdims=True),
                       y * np.sqrt(12), rtol=1e-12)
    # Scale invariance of the norm and linearity in the gate and in gamma.
    assert np.allclose(O.rmsnorm_gate(shape, 7.5 * y, ones, eps=1e-300), out, rtol=1e-12)
    g = rng.uniform(-2, 2, (2, 3, 5, 12)).astype(np.float32)
    gamma = rng.uniform(0.5, 1.5, (3, 12)).astype(np.float32)
    full = O.rmsnorm_gate(shape, y, g, gamma, eps=1e-300)
    assert np.allclose(full, out * g * gamma[None, :, None, :], rtol=1e-12)
    # A constant row c gives c / sqrt(c^2 + eps) in every column.
    c = np.full((2, 3, 5, 12), 0.25)
    got = O.rmsnorm_gate(shape, c, ones, eps=0.0625)
    assert np.allclose(got, 0.25 / np.sqrt(0.0625 + 0.0625), rtol=1e-14)
    # Each head uses its own gamma row.
    gh = np.zeros((3, 12), np.float32); gh[1] = 1.0
    only1 = O.rmsnorm_gate(shape, y, ones, gh, eps=1e-300)
    assert np.all(only1[:, [0, 2]] == 0) and np.allclose(only1[:, 1], out[:, 1], rtol=1e-12)
