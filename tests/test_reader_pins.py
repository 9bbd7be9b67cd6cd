"""Pins of the channel-reader oracle (oracle/reader.py) against facts that do not come from
the oracle itself: explicit Hadamard matrices, exact ternary round trips, the exact MoE
block of the C oracle (every channel kept), full-rank recovery, brute-force selections and
a planted low-rank basis.  "Channel Selection for Mixture-of-Experts Decoding Needs No
Calibration Data", the reader's Stages 1-3."""
import numpy as np
import pytest
import scipy.linalg
import torch

import oracle
import oracle.reader as R
from routed_expert_ffn_top_gb300 import synthetic as syn


def _bf16(a):
    """Round to bf16 values (kept as float64)."""
    return torch.as_tensor(a, dtype=torch.float32).to(torch.bfloat16).to(torch.float64).numpy()


def _signs(H, seed=0):
    return syn.make_rotation_signs(H, seed=seed).numpy().astype(np.float64)


def test_hadamard_matches_the_library_matrix():
    for n in (1, 2, 8, 128):
        assert np.array_equal(R.sylvester_hadamard(n), scipy.linalg.hadamard(n))


def test_rotation_is_orthogonal_and_blockwise():
    H = 384
    s = _signs(H, 3)
    rng = np.random.default_rng(0)
    x, y = rng.standard_normal(H), rng.standard_normal(H)
    # the explicit matrix: block diagonal of H_128 / sqrt(128) times diag(signs)
    Rm = scipy.linalg.block_diag(*([scipy.linalg.hadamard(128) / np.sqrt(128)] * 3)) @ np.diag(s)
    assert np.allclose(R.rotate(x, s), Rm @ x, atol=1e-12)
    assert np.allclose(Rm @ Rm.T, np.eye(H), atol=1e-12)
    assert np.isclose(R.rotate(x, s) @ R.rotate(y, s), x @ y)
    with pytest.raises(ValueError):
        R.rotate(np.zeros(100), np.ones(100))


def test_ternary_code_round_trips_a_ternary_block():
    rng = np.random.default_rng(1)
    for frac in (0.1, 0.5, 1.0):
        c = rng.choice([-1, 0, 1], size=128, p=[frac / 2, 1 - frac, frac / 2]).astype(np.int8)
        c[0] = 1  # at least one nonzero
        alpha = 0.037
        codes, scale = R.ternary_block(alpha * c)
        assert np.array_equal(codes, c) and np.isclose(scale, alpha)
    # the threshold is 0.7 of the mean magnitude: a value just below it codes to zero
    r = np.full(128, 1.0)
    r[5] = 0.69
    r[6] = 0.71
    codes, _ = R.ternary_block(r)
    tau = 0.7 * np.mean(np.abs(r))
    assert codes[5] == (1 if 0.69 > tau else 0) and codes[6] == (1 if 0.71 > tau else 0)


def test_scan_mask_is_the_brute_force_top_set():
    rng = np.random.default_rng(2)
    xr = rng.standard_normal(256)
    xr[7] = xr[9] = 5.0  # a tie, resolved to the lower index when it matters
    for nscan in (1, 80, 128):
        m = R.scan_mask(xr, nscan)
        assert m.shape == (2, 128) and (m.sum(axis=1) == nscan).all()
        for b in range(2):
            v = np.abs(xr.reshape(2, 128)[b])
            if nscan < 128:
                assert v[m[b]].min() >= v[~m[b]].max()
    m1 = R.scan_mask(np.r_[np.full(128, 1.0), np.zeros(128)], 3)
    assert list(np.flatnonzero(m1[0])) == [0, 1, 2]  # all equal: the lowest coordinates


def test_full_scan_sketch_of_ternary_rows_is_the_exact_dot_product():
    """Rows whose rotation is exactly scale * ternary code, scanned in full, give
    ghat = g . x exactly (R is orthogonal)."""
    H = 256
    s = _signs(H, 4)
    rng = np.random.default_rng(3)
    Rm = scipy.linalg.block_diag(*([scipy.linalg.hadamard(128) / np.sqrt(128)] * 2)) @ np.diag(s)
    c = rng.choice([-1, 0, 1], size=(5, H)).astype(np.float64)
    c[:, 0] = 1
    c[:, 128] = -1
    alpha = np.repeat(rng.uniform(0.01, 0.05, (5, 2)), 128, axis=1)
    rows = (alpha * c) @ Rm  # R^T (alpha c), row by row
    codes, scales = R.ternary_sketch(rows, s)
    x = rng.standard_normal(H)
    xr = R.rotate(x, s)
    est = R.sketch_estimate(codes, scales, xr, np.ones((2, 128), bool))
    assert np.allclose(est, rows @ x, rtol=1e-10, atol=1e-12)


def _small_layer(seed=0, H=256, I=128, E=8):
    wl = syn.Workload("reader_pin", H=H, I=I, E=E, k=4, b=8, M=3)
    layer = syn.make_layer(wl, seed=seed)
    h = syn.make_hidden(wl, seed=seed)
    to64 = lambda t: t.to(torch.float64).numpy()  # noqa: E731
    return wl, layer, h, to64(layer["w_gate"]), to64(layer["w_up"]), to64(layer["w_down"])


def test_full_budget_reader_is_the_exact_block():
    """K = every candidate channel: the reader reads everything exactly and must give the
    C oracle's expert FFN + combine for the same routes."""
    wl, layer, h, wg, wu, wd = _small_layer(5)
    s = _signs(wl.H, 5)
    rd = R.build(wg, wu, wd, s, rank=16)
    ids = np.array([[0, 3, 5, 7], [1, 2, 3, 4], [6, -1, 0, 2]], np.int32)
    a = np.array([[0.4, 0.3, 0.2, 0.1], [0.25] * 4, [0.5, 0.0, 0.3, 0.2]])
    ref = oracle.expert_ffn(syn.bits(h), oracle.host_weights(layer), ids, a)
    x = h.to(torch.float64).numpy()
    for m in range(3):
        out, sel, _, _ = R.reader_token(x[m], ids[m], a[m], wg, wu, wd, rd, s,
                                        K=4 * wl.I, nscan=80)
        nvalid = int((ids[m] >= 0).sum())
        assert len(sel) == nvalid * wl.I
        assert np.allclose(out, ref[m], rtol=1e-9, atol=1e-12)


def test_zero_budget_full_rank_recovery_is_exact_on_ternary_rows():
    """K = 0 with a full-rank basis and rows whose sketches are exact: the recovered output
    equals the exact one (ahat = a, U U^T = identity)."""
    H, I, E = 256, 16, 3
    s = _signs(H, 6)
    rng = np.random.default_rng(6)
    Rm = scipy.linalg.block_diag(*([scipy.linalg.hadamard(128) / np.sqrt(128)] * 2)) @ np.diag(s)

    def ternary_rows(n):
        c = rng.choice([-1, 0, 1], size=(n, H)).astype(np.float64)
        c[:, 0] = 1
        c[:, 128] = 1
        return (0.03 * c) @ Rm

    wg = ternary_rows(E * I).reshape(E, I, H).transpose(0, 2, 1)
    wu = ternary_rows(E * I).reshape(E, I, H).transpose(0, 2, 1)
    wd = rng.standard_normal((E, I, H)) * 0.02
    rd = R.build(wg, wu, wd, s, rank=H)
    x = rng.standard_normal(H)
    experts, aff = [2, 0], [0.7, 0.3]
    exact, sel_all, _, _ = R.reader_token(x, experts, aff, wg, wu, wd, rd, s, K=2 * I, nscan=128)
    rec, sel0, scores, _ = R.reader_token(x, experts, aff, wg, wu, wd, rd, s, K=0, nscan=128)
    assert len(sel0) == 0 and len(sel_all) == 2 * I
    assert np.allclose(rec, exact, rtol=1e-9, atol=1e-12)
    # with an exact estimate, a channel's score is the length of what it adds to the output
    for j, e in enumerate(experts):
        for i in range(I):
            a = R.silu(wg[e][:, i] @ x) * (wu[e][:, i] @ x)
            assert scores[j * I + i] == pytest.approx(np.linalg.norm(aff[j] * a * wd[e][i]), rel=1e-9)


def test_selection_is_the_brute_force_top_k():
    wl, layer, h, wg, wu, wd = _small_layer(7)
    s = _signs(wl.H, 7)
    rd = R.build(wg, wu, wd, s, rank=8)
    x = h.to(torch.float64).numpy()[0]
    experts, aff = [1, 4, 6, 2], [0.4, 0.3, 0.2, 0.1]
    for K in (1, 37, 200):
        _, sel, scores, _ = R.reader_token(x, experts, aff, wg, wu, wd, rd, s, K=K)
        assert len(sel) == K
        kept = np.zeros(scores.size, bool)
        kept[sel] = True
        assert scores[kept].min() >= scores[~kept].max()


def test_down_basis_finds_a_planted_subspace():
    rng = np.random.default_rng(8)
    H, n, r = 128, 600, 32
    basis, _ = np.linalg.qr(rng.standard_normal((H, r)))
    coeff = rng.standard_normal((n, r)) * np.linspace(10, 5, r)
    D = coeff @ basis.T + 1e-3 * rng.standard_normal((n, H))
    U = R.down_basis(D.reshape(1, n, H), r)
    assert np.allclose(U.T @ U, np.eye(r), atol=1e-10)
    # principal angles between span(U) and the planted span: all cosines ~ 1
    cos = np.linalg.svd(U.T @ basis, compute_uv=False)
    assert cos.min() > 1 - 1e-6
