"""Oracle-side helpers for the GPU parity tests: run the fp64 oracle on exactly the data the
CUDA path saw (host copies of the same seeded tensors) and compare with the stated bars.

Tolerances (the bars the parity tests enforce):
* routing ids and alignment: bit-exact;
* affinities: |gpu - oracle| <= 1e-4 * oracle + 1e-6 (fp32 softmax of fp32 logits);
* block output (bf16): relative L2 error <= 3e-3 and max-abs error <= 2e-2 * RMS(oracle).
A token whose oracle margin between the k-th and (k+1)-th logit is below NEAR_TIE may
legitimately select differently in fp32, and two selected experts whose logits lie within
NEAR_TIE may legitimately swap slots; only such tokens are excused (check_routing), at most
max(1, M // 50) of them, and their output is then checked with the GPU's ids.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from routed_expert_ffn_top_gb300 import synthetic as syn

REL_L2 = 3e-3
MAX_ABS_RMS = 2e-2
NEAR_TIE = 1e-4


def rel_l2(got, ref):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), 1e-300))


def assert_close_block(got, ref, what=""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = rel_l2(got, ref)
    rms = float(np.sqrt(np.mean(ref * ref)))
    mx = float(np.abs(got - ref).max()) if ref.size else 0.0
    assert err <= REL_L2, "%s rel L2 %.3e > %.1e" % (what, err, REL_L2)
    assert mx <= MAX_ABS_RMS * rms, "%s max-abs %.3e > %.1e * rms %.3e" % (what, mx, MAX_ABS_RMS, rms)
    return err, mx / max(rms, 1e-300)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def oracle_routing(layer, h, k, renormalize=True):
    """(ids, weights, gap, logits) from the oracle for all tokens of h."""
    bias = layer.get("bias")
    bias = None if bias is None else bias.detach().cpu().numpy()
    logits = oracle.router_logits(syn.bits(h), syn.bits(layer["w_router"]), bias,
                                  h.shape[0], layer["H"], layer["E"])
    ids, wts, gap = oracle.topk_softmax(logits, k, renormalize)
    return ids, wts, gap, logits


def check_routing(gpu_ids, gpu_wts, o_ids, o_wts, logits, k, renormalize=True, max_near=None):
    """Routing ids bit-exact against the oracle, except at documented near-ties.

    A token whose GPU ids differ from the oracle's is excused only when the difference is one
    that fp32 rounding of a near-tie can cause:
      * a different expert SET only when the oracle's own margin between its k-th and
        (k+1)-th logit (the gap it reports) is below NEAR_TIE, and every GPU expert's logit
        is at least the oracle's k-th minus NEAR_TIE;
      * a different SLOT ORDER only between experts whose logits lie within NEAR_TIE: the GPU
        slots must descend in the oracle's logits up to NEAR_TIE.
    At most `max_near` tokens (default max(1, M // 50)) may be excused.  The affinities are
    checked against the fp64 softmax of the ids actually used.  Returns (ids, weights) to
    use downstream and the number of excused tokens."""
    gpu_ids = np.asarray(gpu_ids)
    gpu_wts = np.asarray(gpu_wts, np.float64)
    M = o_ids.shape[0]
    if max_near is None:
        max_near = max(1, M // 50)
    _, _, gap = oracle.topk_softmax(logits, k, renormalize)
    ids = o_ids.copy()
    wts = o_wts.copy()
    near = 0
    for m in range(M):
        if np.array_equal(gpu_ids[m], o_ids[m]):
            continue
        l = logits[m]
        g = gpu_ids[m]
        assert len(set(g.tolist())) == k and np.all((g >= 0) & (g < l.size)), \
            "token %d: GPU ids %s are not k distinct experts" % (m, g)
        if set(g.tolist()) != set(o_ids[m].tolist()):
            assert gap[m] < NEAR_TIE, "token %d: GPU set %s, oracle %s, oracle gap %.3e" % (
                m, g, o_ids[m], gap[m])
            kth = l[o_ids[m][k - 1]]
            assert np.all(l[g] >= kth - NEAR_TIE), "token %d: GPU ids %s not a top-%d" % (m, g, k)
        for j in range(k - 1):
            assert l[g[j]] >= l[g[j + 1]] - NEAR_TIE, \
                "token %d: GPU slot %d (expert %d) below slot %d (expert %d)" % (
                    m, j, g[j], j + 1, g[j + 1])
        near += 1
        ids[m] = g
        sel = l[g]
        if renormalize:
            ex = np.exp(sel - sel.max())
            wts[m] = ex / ex.sum()
        else:
            ex = np.exp(l - l.max())
            wts[m] = np.exp(sel - l.max()) / ex.sum()
    assert near <= max_near, "%d near-tie tokens excused, at most %d allowed" % (near, max_near)
    assert np.allclose(gpu_wts, wts, rtol=1e-4, atol=1e-6), np.abs(gpu_wts - wts).max()
    return ids, wts, near


def near_tie_count(logits, k):
    """Tokens whose oracle margin between the k-th and (k+1)-th logit is below NEAR_TIE (the
    ones whose selection fp32 rounding could legitimately change)."""
    _, _, gap = oracle.topk_softmax(logits, k)
    return int((gap < NEAR_TIE).sum())


def oracle_ffn(layer, h, ids, wts, residual=None, tokens=None):
    """Oracle block output for the given tokens (default all), copying to the host only the
    experts those tokens use."""
    ids = np.asarray(ids)
    if tokens is None:
        tokens = np.arange(ids.shape[0])
    tokens = np.asarray(tokens)
    sub_ids = ids[tokens]
    E = layer["E"]
    used = sorted({int(e) for e in sub_ids.reshape(-1) if 0 <= e < E})
    remap = {e: i for i, e in enumerate(used)}
    local = np.array([[remap.get(int(e), -1) for e in row] for row in sub_ids], np.int32)
    if not used:  # no valid route at all: the block output is the residual (or zero)
        used = [0]
    w = oracle.host_weights(layer, used)
    hs = h[torch.as_tensor(tokens, device=h.device, dtype=torch.long)]
    res = None
    if residual is not None:
        res = syn.bits(residual[torch.as_tensor(tokens, device=residual.device, dtype=torch.long)])
    return oracle.expert_ffn(syn.bits(hs), w, local, np.asarray(wts, np.float64)[tokens], res)


def oracle_intermediates(layer, h, ids, wts):
    """Oracle (p [M*k, I], y [M*k, H]) per route r = m*k + j for the given routing, copying to
    the host only the experts it uses; rows of invalid routes are zero."""
    ids = np.asarray(ids)
    E = layer["E"]
    used = sorted({int(e) for e in ids.reshape(-1) if 0 <= e < E}) or [0]
    remap = {e: i for i, e in enumerate(used)}
    local = np.array([[remap.get(int(e), -1) for e in row] for row in ids], np.int32)
    w = oracle.host_weights(layer, used)
    _, p, y = oracle.expert_ffn(syn.bits(h), w, local, np.asarray(wts, np.float64),
                                want_intermediates=True)
    return p, y
