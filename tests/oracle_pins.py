"""Checks that pin the fp64 oracle to something other than itself.

Each ``pin_*`` function raises AssertionError when the oracle disagrees with an
independent fact: a brute-force enumeration on tiny inputs, a numpy/scipy library routine
applied to a special case that reduces to it, a closed form, an invariant of the
definition, or the alignment arithmetic printed on the route-block page.  The functions
take no arguments so that ``test_oracle_pins.py`` runs them against the real oracle and
``test_oracle_mutations.py`` runs them against copies of the oracle with planted mistakes.
"""
from __future__ import annotations

import itertools
import math
import os

import numpy as np
import scipy.special
import torch

import oracle
from routed_expert_ffn_top_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------------------- helpers
def f64(bits):
    """bf16 bit patterns -> exact float64 values (independent of the oracle's widening)."""
    bits = np.asarray(bits)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def bf16_bits(x):
    """Round float values to bf16 (torch's round-to-nearest-even) and return the bits."""
    return syn.bits(torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16))


def silu(x):
    return x * scipy.special.expit(x)


def small_workload(**kw):
    base = dict(name="pin", H=64, I=24, E=8, k=3, b=4, M=5)
    base.update(kw)
    return syn.Workload(**base)


def small_layer(wl, seed=0):
    layer = syn.make_layer(wl, seed=seed, device="cpu")
    h = syn.make_hidden(wl, seed=seed, device="cpu")
    return layer, h


def dense_numpy(layer):
    """Decoded float64 gate/up/down weights [E,H,I], [E,H,I], [E,I,H] from a layer dict."""
    if layer["kind"] == syn.W_DENSE:
        wg = f64(syn.bits(layer["w_gate"]))
        wu = f64(syn.bits(layer["w_up"]))
    else:
        d = layer["d"]
        cbg = f64(syn.bits(layer["cb_gate"]))
        cbu = f64(syn.bits(layer["cb_up"]))
        jg = layer["j_gate"].numpy().astype(np.int64)
        ju = layer["j_up"].numpy().astype(np.int64)
        E, Q, I = jg.shape
        # W[e, d*q + t, i] = B[J[e, q, i], t]: gather the code words, then move t next to q.
        wg = cbg[jg].transpose(0, 1, 3, 2).reshape(E, Q * d, I)
        wu = cbu[ju].transpose(0, 1, 3, 2).reshape(E, Q * d, I)
        if layer["kind"] == syn.W_VQLR:
            # the low-rank half materialised: D [H, r] times C_e [r, I], per expert
            dg, du = f64(syn.bits(layer["d_gate"])), f64(syn.bits(layer["d_up"]))
            cg, cu = f64(syn.bits(layer["c_gate"])), f64(syn.bits(layer["c_up"]))
            wg = wg + np.einsum("hr,eri->ehi", dg, cg)
            wu = wu + np.einsum("hr,eri->ehi", du, cu)
    wd = f64(syn.bits(layer["w_down"]))
    return wg, wu, wd


def brute_topk(logits_row, k):
    """Sort experts by (descending fp32 logit, ascending id) with Python's sort."""
    E = len(logits_row)
    order = sorted(range(E), key=lambda e: (-float(np.float32(logits_row[e])), e))
    return order[:k]


def brute_align(ids, E, b, cap):
    """Alignment by sorting valid (expert, route) pairs, then grouping and padding."""
    flat = [int(x) for x in np.asarray(ids).reshape(-1)]
    R = len(flat)
    pairs = sorted((e, r) for r, e in enumerate(flat) if 0 <= e < E)
    rows, blocks = [], []
    for e, grp in itertools.groupby(pairs, key=lambda t: t[0]):
        rs = [r for _, r in grp]
        nb = -(-len(rs) // b)
        rows += rs + [R] * (nb * b - len(rs))
        blocks += [e] * nb
    npad = len(rows)
    rows += [R] * (cap - npad)
    blocks += [-1] * (cap // b - len(blocks))
    return np.array(rows, dtype=np.int32), np.array(blocks, dtype=np.int32), npad


def check_alignment_invariants(ids, E, b, srt, blk, npad):
    flat = np.asarray(ids).reshape(-1)
    R = flat.size
    valid = [(r, int(e)) for r, e in enumerate(flat) if 0 <= e < E]
    counts = np.bincount([e for _, e in valid], minlength=E) if valid else np.zeros(E, int)
    assert npad == int(sum(-(-int(n) // b) * b for n in counts)), "padded rows != sum ceil(n/b)*b"
    body = srt[:npad]
    vr = body[body != R]
    assert sorted(vr.tolist()) == sorted(r for r, _ in valid), "valid routes not each once"
    assert np.all(srt[npad:] == R), "tail rows must be sentinels"
    nblk = npad // b
    assert np.all(blk[nblk:] == -1), "tail blocks must be -1"
    for q in range(nblk):
        e = blk[q]
        seg = srt[q * b:(q + 1) * b]
        rs = seg[seg != R]
        assert all(flat[r] == e for r in rs), "block holds a route of another expert"
    for e in range(E):
        pos = [i for i, r in enumerate(body) if r != R and flat[r] == e]
        rs = [int(body[i]) for i in pos]
        assert rs == sorted(rs), "routes of one expert not ascending"


# -------------------------------------------------------------------------------- router
def pin_router_hand_example():
    # h = [1, -2]; W_r = [[0.5, 1, -1], [0.25, 0, 2]] -> h W_r = [0, 1, -5]; + bias [1, 0, 0].
    h = bf16_bits([[1.0, -2.0]])
    w = bf16_bits([[0.5, 1.0, -1.0], [0.25, 0.0, 2.0]])
    got = oracle.router_logits(h, w, None, 1, 2, 3)
    assert np.array_equal(got, [[0.0, 1.0, -5.0]]), got
    got = oracle.router_logits(h, w, np.array([1.0, 0.0, 0.0], np.float32), 1, 2, 3)
    assert np.array_equal(got, [[1.0, 1.0, -5.0]]), got


def pin_router_matches_numpy_matmul():
    wl = small_workload(H=96, E=16, M=7, router_bias=True)
    layer, h = small_layer(wl, seed=3)
    hb, wb = syn.bits(h), syn.bits(layer["w_router"])
    bias = layer["bias"].numpy()
    got = oracle.router_logits(hb, wb, bias, wl.M, wl.H, wl.E)
    ref = f64(hb) @ f64(wb) + bias.astype(np.float64)[None, :]
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12), np.abs(got - ref).max()


# -------------------------------------------------------------------------------- top-k
def pin_topk_brute_force():
    rng = np.random.default_rng(11)
    for trial in range(60):
        M, E = int(rng.integers(1, 6)), int(rng.integers(1, 40))
        k = int(rng.integers(1, E + 1))
        logits = rng.standard_normal((M, E))
        if trial % 3 == 0:  # exact ties
            logits = np.round(logits * 2) / 2
        if trial % 3 == 1 and E > 1:  # pairs equal in fp32 but not in fp64
            half = E // 2
            logits[:, half:2 * half] = logits[:, :half] + 1e-12
        ids, _, _ = oracle.topk_softmax(logits, k)
        for m in range(M):
            assert ids[m].tolist() == brute_topk(logits[m], k), (trial, m)


def pin_topk_matches_numpy_stable_argsort():
    rng = np.random.default_rng(5)
    logits = np.round(rng.standard_normal((9, 32)) * 4) / 4
    ids, _, _ = oracle.topk_softmax(logits, 6)
    ref = np.argsort(-logits.astype(np.float32), axis=1, kind="stable")[:, :6]
    assert np.array_equal(ids, ref)


def pin_topk_all_ties():
    ids, wts, _ = oracle.topk_softmax(np.zeros((2, 10)), 4)
    assert ids.tolist() == [[0, 1, 2, 3]] * 2
    assert np.allclose(wts, 0.25, rtol=0, atol=1e-15)


def pin_affinities_vs_scipy_softmax():
    rng = np.random.default_rng(7)
    logits = rng.standard_normal((6, 20)) * 3
    for k in (1, 2, 5, 20):
        ids, wts, _ = oracle.topk_softmax(logits, k, renormalize=True)
        full = scipy.special.softmax(logits, axis=1)
        sel = np.take_along_axis(full, ids, axis=1)
        assert np.allclose(wts, sel / sel.sum(axis=1, keepdims=True), rtol=1e-13, atol=0)
        assert np.allclose(wts.sum(axis=1), 1.0, rtol=0, atol=1e-15)
        if k == 1:
            assert np.all(wts == 1.0)
        ids0, wts0, _ = oracle.topk_softmax(logits, k, renormalize=False)
        assert np.array_equal(ids0, ids)
        assert np.allclose(wts0, sel, rtol=1e-13, atol=0)


def pin_two_expert_logistic():
    # With k = 2 the renormalised affinity of the first expert is the logistic function of
    # the logit difference: a_0 = 1 / (1 + exp(l_1 - l_0)).
    logits = np.array([[0.3, 2.0, -1.0, 1.25]])
    ids, wts, _ = oracle.topk_softmax(logits, 2)
    assert ids.tolist() == [[1, 3]]
    assert math.isclose(wts[0, 0], 1.0 / (1.0 + math.exp(1.25 - 2.0)), rel_tol=1e-15)
    assert math.isclose(wts[0, 1], 1.0 / (1.0 + math.exp(2.0 - 1.25)), rel_tol=1e-15)


def pin_topk_gap():
    logits = np.array([[0.5, 3.0, 2.5, -1.0, 2.0]])
    _, _, gap = oracle.topk_softmax(logits, 2)
    assert gap[0] == 0.5  # selected {3.0, 2.5}; first unselected 2.0
    _, _, gap = oracle.topk_softmax(logits, 5)
    assert math.isinf(gap[0])


# ----------------------------------------------------------------------------- alignment
def pin_alignment_brute_force_random():
    rng = np.random.default_rng(2026)
    cases = 0
    for trial in range(128):
        M = int(rng.integers(0, 41))
        k = int(rng.integers(1, 9))
        E = int(rng.integers(1, 65))
        b = int(rng.choice([1, 2, 3, 4, 8, 16, 64]))
        if trial % 2 == 0 and k <= E:  # router-like: distinct experts per token
            ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]) if M else np.zeros((0, k))
        else:  # arbitrary ids, duplicates allowed
            ids = rng.integers(0, E, size=(M, k))
        ids = np.asarray(ids, dtype=np.int32).reshape(M, k)
        if trial % 4 == 1 and ids.size:  # invalid ids are excluded
            mask = rng.random(ids.shape) < 0.15
            ids[mask] = rng.choice([-1, E, E + 7, -100], size=int(mask.sum()))
        cap = oracle.align_capacity(M, k, E, b)
        srt, blk, npad = oracle.align(ids, E, b, cap)
        bs, bb, bn = brute_align(ids, E, b, cap)
        assert npad == bn and np.array_equal(srt, bs) and np.array_equal(blk, bb), trial
        check_alignment_invariants(ids, E, b, srt, blk, npad)
        cases += 1
    assert cases >= 104


def pin_alignment_adversarial():
    # every route to one expert; every expert once; E = 1; b = 1; all invalid.
    ids = np.full((5, 4), 3, np.int32)
    srt, blk, npad = oracle.align(ids, 8, 8)
    assert npad == 24 and srt[:20].tolist() == list(range(20)) and blk[:3].tolist() == [3] * 3
    ids = np.arange(16, dtype=np.int32).reshape(4, 4)[:, ::-1].copy()
    srt, blk, npad = oracle.align(ids, 16, 2)
    assert npad == 32 and blk[:16].tolist() == list(range(16))
    assert srt[0:2].tolist() == [3, 16] and srt[30:32].tolist() == [12, 16]
    ids = np.zeros((3, 1), np.int32)
    srt, blk, npad = oracle.align(ids, 1, 1)
    assert npad == 3 and srt.tolist() == [0, 1, 2] and blk.tolist() == [0, 0, 0]
    ids = np.full((2, 2), -1, np.int32)
    srt, blk, npad = oracle.align(ids, 4, 4)
    assert npad == 0 and np.all(srt == 4) and np.all(blk == -1)


def pin_alignment_capacity_error():
    ids = np.arange(8, dtype=np.int32).reshape(2, 4)
    try:
        oracle.align(ids, 8, 4, cap=31)
    except RuntimeError:
        pass
    else:
        raise AssertionError("alignment past capacity must fail")
    srt, _, npad = oracle.align(ids, 8, 4, cap=32)
    assert npad == 32


def load_fixture():
    vals = {}
    with open(os.path.join(GOLDEN, "route_block_alignment_fixture.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                key, val = line.split()
                vals[key] = int(val)
    return vals


def fixture_topk_ids(fx, seed=0):
    """A top-k id array whose histogram gives the page's 168 -> 400 rows / 50 blocks."""
    rng = np.random.default_rng(seed)
    M, k, E, b = fx["M"], fx["k"], fx["E"], fx["b"]
    n_blocks, routes = fx["active_blocks"], fx["valid_routes"]
    experts = np.sort(rng.permutation(E)[:n_blocks])
    # 168 routes over 50 experts, each holding 1..b routes (one block each).
    counts = np.full(n_blocks, routes // n_blocks)
    counts[: routes - counts.sum()] += 1
    slots = np.repeat(experts, counts)            # sorted multiset of expert ids
    ids = np.empty((M, k), np.int32)
    for s, e in enumerate(slots):                 # deal round-robin: distinct per token
        ids[s % M, s // M] = e
    for m in range(M):
        ids[m] = rng.permutation(ids[m])
    return ids


def pin_alignment_page_fixture():
    fx = load_fixture()
    ids = fixture_topk_ids(fx)
    assert all(len(set(row)) == fx["k"] for row in ids.tolist())
    srt, blk, npad = oracle.align(ids, fx["E"], fx["b"])
    R = fx["M"] * fx["k"]
    assert R == fx["valid_routes"]
    assert npad == fx["aligned_rows"], npad
    assert int((blk >= 0).sum()) == fx["active_blocks"]
    assert int((srt[:npad] != R).sum()) == fx["valid_routes"]
    check_alignment_invariants(ids, fx["E"], fx["b"], srt, blk, npad)


# ---------------------------------------------------------------------------- expert FFN
def pin_silu_hand_example():
    # H = I = E = k = 1, all weights 1: out = silu(h) * h.
    w = {"kind": syn.W_DENSE, "H": 1, "I": 1, "E": 1,
         "w_gate": bf16_bits([[[1.0]]]), "w_up": bf16_bits([[[1.0]]]),
         "w_down": bf16_bits([[[1.0]]])}
    ids = np.zeros((1, 1), np.int32)
    out = oracle.expert_ffn(bf16_bits([[1.0]]), w, ids, np.ones((1, 1)))
    assert math.isclose(out[0, 0], 0.7310585786300049, rel_tol=1e-15)   # 1 / (1 + e^-1)
    out = oracle.expert_ffn(bf16_bits([[-1.0]]), w, ids, np.ones((1, 1)))
    assert math.isclose(out[0, 0], 0.2689414213699951, rel_tol=1e-15)   # (-1/(1+e)) * (-1)
    out = oracle.expert_ffn(bf16_bits([[2.0]]), w, ids, np.full((1, 1), 0.5))
    assert math.isclose(out[0, 0], 0.5 * (2.0 / (1 + math.exp(-2.0))) * 2.0, rel_tol=1e-15)


def pin_single_expert_textbook_swiglu():
    wl = small_workload(E=1, k=1, M=4, H=48, I=40)
    layer, h = small_layer(wl, seed=1)
    wg, wu, wd = dense_numpy(layer)
    x = f64(syn.bits(h))
    res = syn.make_hidden(wl, seed=9, device="cpu", tag="res")
    ids = np.zeros((wl.M, 1), np.int32)
    out = oracle.expert_ffn(syn.bits(h), oracle.host_weights(layer), ids, np.ones((wl.M, 1)),
                            residual=syn.bits(res))
    ref = f64(syn.bits(res)) + (silu(x @ wg[0]) * (x @ wu[0])) @ wd[0]
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-13), np.abs(out - ref).max()


def _all_experts_reference(layer, h, ids, a, residual=None):
    """Dense all-experts block: every expert on every token, non-selected affinities zero."""
    wg, wu, wd = dense_numpy(layer)
    x = f64(syn.bits(h))
    M, k = ids.shape
    E = wg.shape[0]
    A = np.zeros((M, E))
    for m in range(M):
        for j in range(k):
            if 0 <= ids[m, j] < E:
                A[m, ids[m, j]] += a[m, j]
    out = np.zeros((M, wd.shape[2])) if residual is None else f64(residual).copy()
    for e in range(E):
        out += A[:, e:e + 1] * ((silu(x @ wg[e]) * (x @ wu[e])) @ wd[e])
    return out


def pin_dense_all_experts_reference():
    wl = small_workload(E=8, k=3, M=6, H=64, I=32)
    layer, h = small_layer(wl, seed=2)
    rng = np.random.default_rng(0)
    ids = np.stack([rng.permutation(wl.E)[:wl.k] for _ in range(wl.M)]).astype(np.int32)
    a = rng.random((wl.M, wl.k))
    out = oracle.expert_ffn(syn.bits(h), oracle.host_weights(layer), ids, a)
    ref = _all_experts_reference(layer, h, ids, a)
    assert np.allclose(out, ref, rtol=1e-10, atol=1e-12), np.abs(out - ref).max()


def pin_channel_view():
    # Channel j of expert e owns row j of gate/up (column j of W_gate[e] as stored [H,I])
    # and row j of W_down[e]; the output is the sum over routes and channels of
    # a * phi(g_j . x)(v_j . x) * d_j.
    wl = small_workload(E=4, k=2, M=3, H=32, I=16)
    layer, h = small_layer(wl, seed=4)
    wg, wu, wd = dense_numpy(layer)
    x = f64(syn.bits(h))
    ids = np.array([[0, 3], [2, 1], [3, 2]], np.int32)
    a = np.array([[0.7, 0.3], [0.5, 0.5], [0.9, 0.1]])
    act = np.einsum("mh,mjhc->mjc", x, wg[ids])
    act = silu(act) * np.einsum("mh,mjhc->mjc", x, wu[ids])
    ref = np.einsum("mj,mjc,mjch->mh", a, act, wd[ids])
    out = oracle.expert_ffn(syn.bits(h), oracle.host_weights(layer), ids, a)
    assert np.allclose(out, ref, rtol=1e-10, atol=1e-12)


def pin_zero_cases():
    wl = small_workload(E=4, k=2, M=3, H=32, I=16)
    layer, h = small_layer(wl, seed=6)
    res = syn.make_hidden(wl, seed=8, device="cpu", tag="res")
    ids = np.array([[0, 1], [2, 3], [1, 2]], np.int32)
    a = np.full((3, 2), 0.5)
    w = oracle.host_weights(layer)
    # h = 0  =>  out = residual
    out = oracle.expert_ffn(np.zeros_like(syn.bits(h)), w, ids, a, residual=syn.bits(res))
    assert np.array_equal(out, f64(syn.bits(res)))
    # W_gate = 0  =>  p = silu(0) * u = 0  =>  out = residual
    w0 = dict(w, w_gate=np.zeros_like(w["w_gate"]))
    out = oracle.expert_ffn(syn.bits(h), w0, ids, a, residual=syn.bits(res))
    assert np.array_equal(out, f64(syn.bits(res)))
    # zero affinities  =>  out = residual
    out = oracle.expert_ffn(syn.bits(h), w, ids, np.zeros((3, 2)), residual=syn.bits(res))
    assert np.array_equal(out, f64(syn.bits(res)))


def pin_invalid_routes_contribute_nothing():
    wl = small_workload(E=4, k=3, M=3, H=32, I=16)
    layer, h = small_layer(wl, seed=10)
    w = oracle.host_weights(layer)
    ids = np.array([[0, -1, 2], [4, 1, 3], [2, 3, 9]], np.int32)
    a = np.array([[0.2, 0.3, 0.5], [0.6, 0.3, 0.1], [0.4, 0.4, 0.2]])
    out = oracle.expert_ffn(syn.bits(h), w, ids, a)
    ref = _all_experts_reference(layer, h, ids, a)
    assert np.allclose(out, ref, rtol=1e-10, atol=1e-12)


# ------------------------------------------------------------------------------------ VQ
def vq_workload(**kw):
    base = dict(name="pin_vq", H=32, I=12, E=5, k=2, b=4, M=3, kind=syn.W_VQ, d=4, K=16)
    base.update(kw)
    return syn.Workload(**base)


def pin_vq_equals_decoded_dense():
    wl = vq_workload()
    layer, h = small_layer(wl, seed=12)
    wg, wu, wd = dense_numpy(layer)          # decoded by numpy fancy indexing
    dense = {"kind": syn.W_DENSE, "H": wl.H, "I": wl.I, "E": wl.E,
             "w_gate": bf16_bits(wg), "w_up": bf16_bits(wu), "w_down": syn.bits(layer["w_down"])}
    ids = np.array([[0, 4], [3, 1], [2, 0]], np.int32)
    a = np.array([[0.6, 0.4], [0.5, 0.5], [0.25, 0.75]])
    out_vq = oracle.expert_ffn(syn.bits(h), oracle.host_weights(layer), ids, a)
    out_dense = oracle.expert_ffn(syn.bits(h), dense, ids, a)
    assert np.array_equal(out_vq, out_dense)


def pin_vq_d8_equals_decoded_dense():
    # The same definition with 8-element code words (the pages' deployed d = 8).
    wl = vq_workload(d=8, H=64, K=16)
    layer, h = small_layer(wl, seed=16)
    wg, wu, wd = dense_numpy(layer)
    dense = {"kind": syn.W_DENSE, "H": wl.H, "I": wl.I, "E": wl.E,
             "w_gate": bf16_bits(wg), "w_up": bf16_bits(wu), "w_down": syn.bits(layer["w_down"])}
    ids = np.array([[1, 3], [4, 0], [2, 2]], np.int32)
    a = np.array([[0.7, 0.3], [0.5, 0.5], [0.4, 0.6]])
    out_vq = oracle.expert_ffn(syn.bits(h), oracle.host_weights(layer), ids, a)
    out_dense = oracle.expert_ffn(syn.bits(h), dense, ids, a)
    assert np.array_equal(out_vq, out_dense)


def pin_vq_projection_codebook():
    # "A Multi-Engine Dataflow ...", Section 4.2 (reuse of shared projections): with
    # T[q, c] = h_q . B_c for every length-d block q of h, the projection output is
    # o[i] = sum_q T[q, J[q, i]].
    wl = vq_workload(E=3, M=2, H=40, I=10, d=4, K=32)
    layer, h = small_layer(wl, seed=13)
    x = f64(syn.bits(h))
    d, Q = wl.d, wl.H // wl.d
    cbg, cbu = f64(syn.bits(layer["cb_gate"])), f64(syn.bits(layer["cb_up"]))
    jg, ju = layer["j_gate"].numpy(), layer["j_up"].numpy()
    wd = f64(syn.bits(layer["w_down"]))
    ids = np.array([[2, 0], [1, 2]], np.int32)
    a = np.array([[0.3, 0.7], [0.8, 0.2]])
    ref = np.zeros((wl.M, wl.H))
    for m in range(wl.M):
        xb = x[m].reshape(Q, d)
        Tg, Tu = xb @ cbg.T, xb @ cbu.T            # [Q, K]
        for j in range(wl.k):
            e = ids[m, j]
            g = Tg[np.arange(Q)[:, None], jg[e]].sum(axis=0)
            u = Tu[np.arange(Q)[:, None], ju[e]].sum(axis=0)
            ref[m] += a[m, j] * ((silu(g) * u) @ wd[e])
    out = oracle.expert_ffn(syn.bits(h), oracle.host_weights(layer), ids, a)
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-13)


def pin_vq_constant_index_is_dense():
    # J = const c: every d-block of a column is code word c, so W[e][h][i] = B[c][h mod d].
    wl = vq_workload(E=2, M=2, H=16, I=6, d=4, K=8)
    layer, h = small_layer(wl, seed=14)
    layer = dict(layer)
    layer["j_gate"] = torch.full_like(layer["j_gate"], 5)
    layer["j_up"] = torch.full_like(layer["j_up"], 2)
    cbg, cbu = f64(syn.bits(layer["cb_gate"])), f64(syn.bits(layer["cb_up"]))
    wg = np.broadcast_to(np.tile(cbg[5], wl.H // wl.d)[None, :, None], (wl.E, wl.H, wl.I))
    wu = np.broadcast_to(np.tile(cbu[2], wl.H // wl.d)[None, :, None], (wl.E, wl.H, wl.I))
    x = f64(syn.bits(h))
    wd = f64(syn.bits(layer["w_down"]))
    ids = np.array([[1], [0]], np.int32)
    out = oracle.expert_ffn(syn.bits(h), oracle.host_weights(layer), ids, np.ones((2, 1)))
    ref = np.stack([(silu(x[m] @ wg[ids[m, 0]]) * (x[m] @ wu[ids[m, 0]])) @ wd[ids[m, 0]]
                    for m in range(2)])
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-14)


# ------------------------------------------------------------------------------- VQ + LR
def vqlr_workload(**kw):
    base = dict(name="pin_vqlr", H=32, I=12, E=5, k=2, b=4, M=3, kind=syn.W_VQLR, d=4, K=16, r=6)
    base.update(kw)
    return syn.Workload(**base)


def pin_vqlr_equals_materialised_dense():
    # "A Multi-Engine Dataflow ...", hybrid representation (text around its Eq. (1)):
    # W_e = Q_B(J_e) + D C_e.  The oracle multiplies in the factored order (D^T h first); the
    # reference materialises W_e in numpy (einsum) and multiplies h by it directly.
    wl = vqlr_workload()
    layer, h = small_layer(wl, seed=21)
    wg, wu, wd = dense_numpy(layer)
    x = f64(syn.bits(h))
    ids = np.array([[0, 4], [3, 1], [2, 0]], np.int32)
    a = np.array([[0.6, 0.4], [0.5, 0.5], [0.25, 0.75]])
    ref = np.zeros((wl.M, wl.H))
    for m in range(wl.M):
        for j in range(wl.k):
            e = ids[m, j]
            ref[m] += a[m, j] * ((silu(x[m] @ wg[e]) * (x[m] @ wu[e])) @ wd[e])
    out = oracle.expert_ffn(syn.bits(h), oracle.host_weights(layer), ids, a)
    assert np.allclose(out, ref, rtol=1e-11, atol=1e-13)


def pin_vqlr_zero_coefficients_is_vq():
    # C_e = 0 removes the low-rank half exactly: the result is the VQ-only block, bit for bit.
    wl = vqlr_workload(E=3, M=2, r=5)
    layer, h = small_layer(wl, seed=22)
    layer = dict(layer)
    layer["c_gate"] = torch.zeros_like(layer["c_gate"])
    layer["c_up"] = torch.zeros_like(layer["c_up"])
    vq = dict(layer)
    vq["kind"] = syn.W_VQ
    ids = np.array([[2, 0], [1, 2]], np.int32)
    a = np.array([[0.3, 0.7], [0.8, 0.2]])
    out = oracle.expert_ffn(syn.bits(h), oracle.host_weights(layer), ids, a)
    out_vq = oracle.expert_ffn(syn.bits(h), oracle.host_weights(vq), ids, a)
    assert np.array_equal(out, out_vq)


def pin_vqlr_zero_codebook_is_low_rank_swiglu():
    # All code words zero: the expert is the textbook low-rank SwiGLU
    # (silu(h D_g C_g) * (h D_u C_u)) W_down, computed here with numpy matmuls.
    wl = vqlr_workload(E=2, M=2, H=24, I=10, r=4, k=1)
    layer, h = small_layer(wl, seed=23)
    layer = dict(layer)
    layer["cb_gate"] = torch.zeros_like(layer["cb_gate"])
    layer["cb_up"] = torch.zeros_like(layer["cb_up"])
    x = f64(syn.bits(h))
    dg, du = f64(syn.bits(layer["d_gate"])), f64(syn.bits(layer["d_up"]))
    cg, cu = f64(syn.bits(layer["c_gate"])), f64(syn.bits(layer["c_up"]))
    wd = f64(syn.bits(layer["w_down"]))
    ids = np.array([[1], [0]], np.int32)
    out = oracle.expert_ffn(syn.bits(h), oracle.host_weights(layer), ids, np.ones((2, 1)))
    ref = np.stack([(silu((x[m] @ dg) @ cg[ids[m, 0]]) * ((x[m] @ du) @ cu[ids[m, 0]]))
                    @ wd[ids[m, 0]] for m in range(2)])
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-14)


def pin_vqlr_projections_are_separate():
    # Gate and up keep their own basis and coefficients: swapping the up pair for the gate
    # pair makes u equal g, so p = silu(g) * g, checked against that closed form.
    wl = vqlr_workload(E=2, M=1, H=16, I=6, r=3, k=1)
    layer, h = small_layer(wl, seed=24)
    layer = dict(layer)
    layer["d_up"] = layer["d_gate"].clone()
    layer["c_up"] = layer["c_gate"].clone()
    layer["j_up"] = layer["j_gate"].clone()
    layer["cb_up"] = layer["cb_gate"].clone()
    wg, _, wd = dense_numpy(layer)
    x = f64(syn.bits(h))
    ids = np.array([[1]], np.int32)
    g = x[0] @ wg[1]
    out = oracle.expert_ffn(syn.bits(h), oracle.host_weights(layer), ids, np.ones((1, 1)))
    assert np.allclose(out[0], (silu(g) * g) @ wd[1], rtol=1e-12, atol=1e-14)


# -------------------------------------------------------------------------- whole block
def pin_decode_block_composition():
    wl = small_workload(E=8, k=3, M=4, H=64, I=16, router_bias=True)
    layer, h = small_layer(wl, seed=15)
    w = oracle.host_weights(layer)
    bias = layer["bias"].numpy()
    ids, wts, gap, out = oracle.decode_block(syn.bits(h), syn.bits(layer["w_router"]), bias,
                                             w, wl.k)
    logits = f64(syn.bits(h)) @ f64(syn.bits(layer["w_router"])) + bias.astype(np.float64)
    for m in range(wl.M):
        assert ids[m].tolist() == brute_topk(logits[m], wl.k)
    ref = _all_experts_reference(layer, h, ids, wts)
    assert np.allclose(out, ref, rtol=1e-10, atol=1e-12)
    assert np.allclose(wts.sum(axis=1), 1.0, atol=1e-15)


def pin_threads_do_not_change_results():
    """The expert loop on several threads (whole tokens each) gives the single-threaded
    results bit for bit, with the intermediates, and the all-experts reference still holds."""
    wl = small_workload(E=8, k=3, M=13, H=64, I=32)
    layer, h = small_layer(wl, seed=21)
    rng = np.random.default_rng(21)
    ids = np.stack([rng.permutation(wl.E)[:wl.k] for _ in range(wl.M)]).astype(np.int32)
    ids[3, 1] = -1  # an invalid route among them
    a = rng.random((wl.M, wl.k))
    w = oracle.host_weights(layer)
    before = oracle.set_threads(0)
    try:
        oracle.set_threads(1)
        one = oracle.expert_ffn(syn.bits(h), w, ids, a, want_intermediates=True)
        oracle.set_threads(4)
        many = oracle.expert_ffn(syn.bits(h), w, ids, a, want_intermediates=True)
    finally:
        oracle.set_threads(before)
    for x, y in zip(one, many):
        assert np.array_equal(x, y)
    ref = _all_experts_reference(layer, h, ids, a)
    assert np.allclose(many[0], ref, rtol=1e-10, atol=1e-12)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]
