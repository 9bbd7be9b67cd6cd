"""fp64 oracle of the channel-sparse reader of "Channel Selection for Mixture-of-Experts
Decoding Needs No Calibration Data" (the reader's three stages).

TEST INFRASTRUCTURE ONLY.  Only the test suite and the benchmark's CPU legs may import this
module; the product never imports it and shares no code with it.

Everything is plain numpy in float64; a library matmul, sort or symmetric eigensolver
serves as a step where the definition is one.  For one token and one layer the reader:

* Stage 1 ("Screen with a Ternary Sketch"): rotates x in 128-coordinate blocks by a random
  Hadamard transform R (Sylvester Hadamard matrix / sqrt(128) times random signs, so R is
  orthogonal); every gate row g_j and up row v_j was rotated the same way and stored as a
  ternary sketch per block; from each block only the coordinates with the largest |Rx| are
  scanned (80 of 128); ghat_j, vhat_j are the sketch dot products and
  ahat_j = SiLU(ghat_j) * vhat_j.
* Stage 2 ("Compute the Top k Exactly with Output-Level Scores"): score_j =
  w_j * ||d_j|| * |ahat_j| (w_j the router weight of channel j's expert, d_j its down
  column); the K channels with the largest scores across all the token's experts are read
  exactly: a_j = SiLU(g_j . x) * (v_j . x).
* Stage 3 ("Recover Discarded Channels with a rank-32 Map"): U holds the top left singular
  vectors of all down columns of the layer, b_j = U^T d_j, and
  out = sum_{j kept} w_j a_j d_j + U sum_{j discarded} w_j ahat_j b_j.

Readings where the page is silent or garbled (its Equations 1 and 2 and the storage
format of a sketch block are missing from the text):
* the ternary code of a rotated block r is the Ternary Weight Networks rule (Li, Zhang and
  Liu, 2016): threshold 0.7 * mean|r|, code sign(r_i) where |r_i| exceeds it, else 0, and
  one scale per block, the mean |r_i| over the nonzero codes (the least-squares scale for
  those codes); 128 two-bit codes and a 4-byte scale are 36 bytes a block;
* the score is Equation 1 as the text states it: the router weight times the down-column
  norm times |ahat_j|; ties go to the lower channel index (slot, then channel);
* the partial scan keeps, per block, the nscan coordinates of largest |Rx|, ties to the
  lower coordinate;
* U is taken from the eigenvectors of D D^T for the largest eigenvalues (the left singular
  vectors of D, the H x (E I) matrix of down columns), and the output carries no residual
  (the caller adds it).
Parity status: pinned by tests/test_reader_pins.py (explicit Hadamard matrices, exact
ternary round trips, the full-budget reader against the C oracle's exact block, full-rank
recovery, brute-force selections and a planted low-rank basis).
"""
from __future__ import annotations

import numpy as np

BLOCK = 128


def sylvester_hadamard(n: int) -> np.ndarray:
    """H_1 = [1], H_2m = [[H_m, H_m], [H_m, -H_m]] (n a power of two)."""
    h = np.ones((1, 1))
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    if h.shape[0] != n:
        raise ValueError("n must be a power of two")
    return h


def rotate(x: np.ndarray, signs: np.ndarray) -> np.ndarray:
    """R x per 128-coordinate block: (H_128 / sqrt(128)) (signs * x) on every block of the
    last axis."""
    x = np.asarray(x, np.float64)
    H = x.shape[-1]
    if H % BLOCK:
        raise ValueError("H must be a multiple of 128")
    hb = sylvester_hadamard(BLOCK) / np.sqrt(BLOCK)
    y = (x * np.asarray(signs, np.float64)).reshape(x.shape[:-1] + (H // BLOCK, BLOCK))
    return np.einsum("ij,...bj->...bi", hb, y).reshape(x.shape)


def ternary_block(r: np.ndarray):
    """Ternary code and scale of one rotated block (Ternary Weight Networks threshold)."""
    r = np.asarray(r, np.float64)
    tau = 0.7 * np.mean(np.abs(r))
    codes = np.where(np.abs(r) > tau, np.sign(r), 0.0).astype(np.int8)
    nz = codes != 0
    scale = float(np.abs(r)[nz].mean()) if nz.any() else 0.0
    return codes, scale


def ternary_sketch(rows: np.ndarray, signs: np.ndarray):
    """Sketch of channel rows [n, H]: codes [n, H/128, 128] int8, scales [n, H/128]."""
    rows = np.asarray(rows, np.float64)
    n, H = rows.shape
    rot = rotate(rows, signs).reshape(n, H // BLOCK, BLOCK)
    codes = np.zeros((n, H // BLOCK, BLOCK), np.int8)
    scales = np.zeros((n, H // BLOCK))
    for j in range(n):
        for b in range(H // BLOCK):
            codes[j, b], scales[j, b] = ternary_block(rot[j, b])
    return codes, scales


def scan_mask(xr: np.ndarray, nscan: int) -> np.ndarray:
    """Per 128-block, True on the nscan coordinates of largest |xr| (ties: lower index)."""
    xr = np.asarray(xr, np.float64).reshape(-1, BLOCK)
    mask = np.zeros(xr.shape, bool)
    for b in range(xr.shape[0]):
        order = sorted(range(BLOCK), key=lambda i: (-abs(xr[b, i]), i))
        mask[b, order[:nscan]] = True
    return mask


def sketch_estimate(codes, scales, xr, mask) -> np.ndarray:
    """sum over blocks b of scale_b * sum over scanned i of code_i * xr_i, per row."""
    xr = np.asarray(xr, np.float64).reshape(-1, BLOCK)
    part = np.einsum("nbi,bi->nb", codes.astype(np.float64), xr * mask)
    return (np.asarray(scales, np.float64) * part).sum(axis=1)


def silu(z):
    z = np.asarray(z, np.float64)
    return z / (1.0 + np.exp(-z))


def down_basis(w_down: np.ndarray, rank: int) -> np.ndarray:
    """U [H, rank]: eigenvectors of D D^T for its largest eigenvalues, D = [d_{e,i}] the
    H x (E I) matrix of down columns (rows of w_down [E, I, H])."""
    D = np.asarray(w_down, np.float64).reshape(-1, w_down.shape[-1])  # [E*I, H]
    evals, evecs = np.linalg.eigh(D.T @ D)
    order = np.argsort(-evals, kind="stable")[:rank]
    return evecs[:, order]


def build(w_gate, w_up, w_down, signs, rank=32):
    """The reader's data for one layer (built once from the weights): sketches of every
    channel's gate and up row, down-column norms, U and the coefficients b = U^T d."""
    w_gate = np.asarray(w_gate, np.float64)
    w_up = np.asarray(w_up, np.float64)
    w_down = np.asarray(w_down, np.float64)
    E, H, I = w_gate.shape
    g_rows = np.transpose(w_gate, (0, 2, 1)).reshape(E * I, H)  # channel (e, i) -> row
    v_rows = np.transpose(w_up, (0, 2, 1)).reshape(E * I, H)
    gc, gs = ternary_sketch(g_rows, signs)
    vc, vs = ternary_sketch(v_rows, signs)
    U = down_basis(w_down, rank)
    return {
        "g_codes": gc.reshape(E, I, H // BLOCK, BLOCK), "g_scales": gs.reshape(E, I, H // BLOCK),
        "v_codes": vc.reshape(E, I, H // BLOCK, BLOCK), "v_scales": vs.reshape(E, I, H // BLOCK),
        "dnorm": np.linalg.norm(w_down, axis=2),  # [E, I]
        "U": U,
        "coef": w_down @ U,  # [E, I, rank]
    }


def reader_token(x, experts, affinities, w_gate, w_up, w_down, rd, signs, K, nscan=80,
                 decisions=None):
    """One token through the reader.  Returns (out [H] without residual, selected flat
    indices slot * I + i in ascending order, scores [k * I], scan mask [H/128, 128]).
    ``decisions`` may give the scan mask and the selected set to use instead of this
    function's own (for tokens whose float near-ties another precision may break
    differently)."""
    x = np.asarray(x, np.float64)
    w_gate = np.asarray(w_gate, np.float64)
    w_up = np.asarray(w_up, np.float64)
    w_down = np.asarray(w_down, np.float64)
    k = len(experts)
    E, H, I = w_gate.shape
    xr = rotate(x, signs)
    mask = scan_mask(xr, nscan) if decisions is None else decisions["mask"]
    ahat = np.zeros((k, I))
    scores = np.zeros((k, I))
    for j, e in enumerate(experts):
        if e < 0 or e >= E:
            continue
        gh = sketch_estimate(rd["g_codes"][e], rd["g_scales"][e], xr, mask)
        vh = sketch_estimate(rd["v_codes"][e], rd["v_scales"][e], xr, mask)
        ahat[j] = silu(gh) * vh
        scores[j] = affinities[j] * rd["dnorm"][e] * np.abs(ahat[j])
    valid = [j * I + i for j, e in enumerate(experts) if 0 <= e < E for i in range(I)]
    if decisions is None:
        ranked = sorted(valid, key=lambda f: (-scores.flat[f], f))
        selected = sorted(ranked[:K])
    else:
        selected = sorted(decisions["selected"])
    keep = set(selected)
    out = np.zeros(H)
    z = np.zeros(rd["U"].shape[1])
    for f in valid:
        j, i = divmod(f, I)
        e = experts[j]
        if f in keep:
            a = silu(w_gate[e][:, i] @ x) * (w_up[e][:, i] @ x)
            out += affinities[j] * a * w_down[e][i]
        else:
            z += affinities[j] * ahat[j, i] * rd["coef"][e, i]
    out += rd["U"] @ z
    return out, np.array(selected, np.int64), scores.reshape(-1), mask
