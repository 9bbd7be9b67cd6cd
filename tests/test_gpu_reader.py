"""The channel reader's CUDA path (moe_reader_build, moe_reader_ffn) against the fp64 reader
oracle ("Channel Selection for Mixture-of-Experts Decoding Needs No Calibration Data",
Stages 1-3).  Decisions taken on floats -- the scanned coordinates of each block and the
kept channels -- are checked for validity against the oracle's values, and the oracle then
evaluates the output with the GPU's decisions (the precision rule of the routing tests)."""
import numpy as np
import pytest
import torch

import gpu_ref as G
import oracle.reader as R
from routed_expert_ffn_top_gb300 import moe, synthetic as syn

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as entry
    entry.build()
    yield
    torch.cuda.synchronize()


def _f64(t):
    return t.detach().to(torch.float64).cpu().numpy()


def _pack_codes(codes):
    """int8 codes [..., nb, 128] in {-1,0,1} -> the library's words [..., nb, 8]: words 0-3
    the nonzero mask, 4-7 the negative mask, coordinate c at bit c%32 of word c/32."""
    c = np.asarray(codes, np.int64).reshape(np.shape(codes)[:-1] + (4, 32))
    bit = np.uint64(1) << np.arange(32, dtype=np.uint64)
    nz = ((c != 0).astype(np.uint64) * bit).sum(axis=-1)
    ng = ((c < 0).astype(np.uint64) * bit).sum(axis=-1)
    return np.concatenate([nz, ng], axis=-1).astype(np.uint32).view(np.int32)


def _unpack_codes(words):
    w = np.asarray(words).view(np.uint32).astype(np.uint64)
    bits = (w[..., None] >> np.arange(32, dtype=np.uint64)) & 1
    nz = bits[..., :4, :].reshape(w.shape[:-1] + (128,))
    ng = bits[..., 4:, :].reshape(w.shape[:-1] + (128,))
    return np.where(nz == 1, np.where(ng == 1, -1, 1), 0).astype(np.int8)


def _setup(H=256, I=256, E=8, k=4, M=5, rank=16, seed=0):
    wl = syn.Workload("reader_t", H=H, I=I, E=E, k=k, b=8, M=M)
    layer = syn.make_layer(wl, seed=seed, device=DEV)
    h = syn.make_hidden(wl, seed=seed, device=DEV)
    signs = syn.make_rotation_signs(H, seed=seed, device=DEV)
    wg, wu, wd = _f64(layer["w_gate"]), _f64(layer["w_up"]), _f64(layer["w_down"])
    s64 = signs.cpu().numpy().astype(np.float64)
    ref = R.build(wg, wu, wd, s64, rank=rank)
    U = torch.as_tensor(ref["U"], dtype=torch.float32, device=DEV)
    return wl, layer, h, signs, s64, (wg, wu, wd), ref, U


def _routes(M, k, E, seed):
    rng = np.random.default_rng(seed)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32)
    a = rng.uniform(0.05, 1.0, (M, k))
    a = (a / a.sum(axis=1, keepdims=True)).astype(np.float32)
    return ids, a


def test_build_matches_the_oracle():
    wl, layer, h, signs, s64, (wg, wu, wd), ref, U = _setup(seed=1)
    rd = moe.reader_build(layer, signs, U)
    torch.cuda.synchronize()
    # channel-major rows: an exact transpose
    assert torch.equal(rd["g_rows"], layer["w_gate"].transpose(1, 2).contiguous())
    assert torch.equal(rd["v_rows"], layer["w_up"].transpose(1, 2).contiguous())
    # ternary codes: equal except where the fp32 rotation lands within rounding of the
    # threshold (the decision is the kernel's, in fp32)
    for p, w in (("g", wg), ("v", wu)):
        got = _unpack_codes(rd[p + "_codes"].cpu().numpy())
        want = ref[p + "_codes"]
        rows = np.transpose(w, (0, 2, 1)).reshape(-1, wl.H)
        rot = R.rotate(rows, s64).reshape(got.shape)
        tau = 0.7 * np.abs(rot).mean(axis=-1, keepdims=True)
        diff = got != want
        assert np.all(np.abs(np.abs(rot[diff]) - np.broadcast_to(tau, rot.shape)[diff])
                      <= 1e-5 * np.broadcast_to(tau, rot.shape)[diff]), p
        assert diff.mean() < 1e-4, (p, diff.mean())
        gs = rd[p + "_scales"].cpu().numpy()
        same = ~diff.any(axis=-1)  # blocks whose codes agree: the same mean of |r|
        assert np.allclose(gs[same], ref[p + "_scales"][same], rtol=1e-5, atol=1e-9), p
        assert np.allclose(gs[~same], ref[p + "_scales"][~same], rtol=5e-2), p
    assert np.allclose(rd["dnorm"].cpu().numpy(), ref["dnorm"], rtol=1e-5)
    coef = _f64(rd["coef"])
    assert np.abs(coef - ref["coef"]).max() <= 1e-2 * np.abs(ref["coef"]).max()


def _device_reader(layer, signs, U, ref):
    """The reader's data with the oracle's sketch, norms and coefficients (the same model
    data on both sides), the rows from the library build."""
    rd = moe.reader_build(layer, signs, U)
    rd["g_codes"].copy_(torch.as_tensor(_pack_codes(ref["g_codes"]), device=DEV))
    rd["v_codes"].copy_(torch.as_tensor(_pack_codes(ref["v_codes"]), device=DEV))
    rd["g_scales"].copy_(torch.as_tensor(ref["g_scales"], dtype=torch.float32, device=DEV))
    rd["v_scales"].copy_(torch.as_tensor(ref["v_scales"], dtype=torch.float32, device=DEV))
    rd["dnorm"].copy_(torch.as_tensor(ref["dnorm"], dtype=torch.float32, device=DEV))
    rd["coef"].copy_(torch.as_tensor(ref["coef"], dtype=torch.float32, device=DEV).to(torch.bfloat16))
    return rd


def _check_decisions(x, ids, aff, wg, wu, wd, ref, s64, K, nscan, sel_gpu, xr_gpu,
                     score_tol=1e-4):
    """Validate the GPU's scan and selection against the oracle's values; return the
    decisions to evaluate the oracle with."""
    I = wg.shape[2]
    xr_o = R.rotate(x, s64).reshape(-1, 128)
    xg = xr_gpu.reshape(-1, 128)
    mask = xg != 0
    assert (mask.sum(axis=1) == nscan).all()
    assert np.allclose(xg[mask], xr_o[mask], rtol=1e-5, atol=1e-6)
    tol = 1e-5 * np.abs(xr_o).max()
    for b in range(mask.shape[0]):
        if 0 < nscan < 128:
            assert np.abs(xr_o[b][mask[b]]).min() >= np.abs(xr_o[b][~mask[b]]).max() - tol
    # the oracle's scores with the GPU's scan; the GPU's kept set must be a valid top K
    _, _, scores, _ = R.reader_token(x, ids, aff, wg, wu, wd, ref, s64, K, nscan,
                                     decisions={"mask": mask, "selected": []})
    sel = np.array(sorted(int(f) for f in sel_gpu if f >= 0), np.int64)
    nvalid = int((ids >= 0).sum()) * I
    assert len(sel) == min(K, nvalid)
    if 0 < len(sel) < nvalid:
        kept = np.zeros(scores.size, bool)
        kept[sel] = True
        valid = np.repeat(ids >= 0, I)
        stol = score_tol * scores.max()
        assert scores[kept].min() >= scores[~kept & valid].max() - stol
    return {"mask": mask, "selected": list(sel)}


@pytest.mark.parametrize("K,nscan", [(0, 80), (37, 80), (256, 128), (400, 80), (1024, 80)])
def test_decode_matches_the_oracle(K, nscan):
    wl, layer, h, signs, s64, (wg, wu, wd), ref, U = _setup(seed=2)
    rd = _device_reader(layer, signs, U, ref)
    ids, a = _routes(wl.M, wl.k, wl.E, 2)
    ids[3, 1] = -1  # an invalid route is skipped
    res = syn.make_hidden(wl, seed=9, device=DEV, tag="res")
    out, sel, xr = moe.moe_reader_ffn(h, rd, torch.as_tensor(ids, device=DEV),
                                      torch.as_tensor(a, device=DEV), K, nscan, residual=res,
                                      want_decisions=True)
    torch.cuda.synchronize()
    x = _f64(h)
    want = np.zeros((wl.M, wl.H))
    for m in range(wl.M):
        dec = _check_decisions(x[m], ids[m], a[m].astype(np.float64), wg, wu, wd, ref, s64, K,
                               nscan, sel[m].cpu().numpy(), xr[m].cpu().numpy())
        o, _, _, _ = R.reader_token(x[m], ids[m], a[m].astype(np.float64), wg, wu, wd, ref, s64,
                                    K, nscan, decisions=dec)
        want[m] = o + _f64(res[m])
    G.assert_close_block(_f64(out), want, "reader K=%d nscan=%d" % (K, nscan))


def test_decode_is_deterministic_and_batch_invariant():
    wl, layer, h, signs, s64, _, ref, U = _setup(M=7, seed=3)
    rd = _device_reader(layer, signs, U, ref)
    ids, a = _routes(wl.M, wl.k, wl.E, 3)
    t_ids, t_a = torch.as_tensor(ids, device=DEV), torch.as_tensor(a, device=DEV)
    out = moe.moe_reader_ffn(h, rd, t_ids, t_a, 100, 80)
    for _ in range(5):
        assert torch.equal(moe.moe_reader_ffn(h, rd, t_ids, t_a, 100, 80), out)
    for sub in ([0], [6, 2], list(range(1, 6))):
        sl = torch.as_tensor(sub, device=DEV)
        o = moe.moe_reader_ffn(h[sl].contiguous(), rd, t_ids[sl].contiguous(), t_a[sl].contiguous(),
                               100, 80)
        assert torch.equal(o, out[sl]), sub


def test_full_budget_reader_matches_the_exact_block():
    """Every channel read exactly: the reader's output is the block's (within the parity
    bar: the two paths add in different orders and the exact block rounds p to bf16)."""
    wl, layer, h, signs, s64, _, ref, U = _setup(M=4, seed=4)
    rd = moe.reader_build(layer, signs, U)
    ids, a = _routes(wl.M, wl.k, wl.E, 4)
    t_ids, t_a = torch.as_tensor(ids, device=DEV), torch.as_tensor(a, device=DEV)
    out = moe.moe_reader_ffn(h, rd, t_ids, t_a, wl.k * wl.I, 80)
    exact = moe.moe_expert_ffn(h, layer, t_ids, t_a, 8)
    ref_block = G.oracle_ffn(layer, h, ids, a)
    G.assert_close_block(_f64(out), ref_block, "full-budget reader")
    G.assert_close_block(_f64(exact), ref_block, "exact block")


def test_full_size_token():
    """The decode layer's shape (H=2048, I=768, E=128, k=8) for one routed token at a 12.3%
    exact-read budget: the library builds the sketch, the oracle builds its own from the
    same weights for the token's experts, both use one basis U."""
    wl = syn.workload("layer_m1")
    layer = syn.make_layer(wl, seed=5, device=DEV)
    h = syn.make_hidden(wl, seed=5, device=DEV)
    signs = syn.make_rotation_signs(wl.H, seed=5, device=DEV)
    U64 = R.down_basis(_f64(layer["w_down"]), 32)
    U = torch.as_tensor(U64, dtype=torch.float32, device=DEV)
    rd = moe.reader_build(layer, signs, U)
    ids, wts = moe.moe_route_topk(h, layer["w_router"], None, wl.k)
    K = 756
    out, sel, xr = moe.moe_reader_ffn(h, rd, ids, wts, K, 80, want_decisions=True)
    torch.cuda.synchronize()
    experts = sorted(set(int(e) for e in ids[0].tolist()))
    remap = {e: q for q, e in enumerate(experts)}
    sub = lambda t: _f64(t[torch.as_tensor(experts, device=DEV)])  # noqa: E731
    wg, wu, wd = sub(layer["w_gate"]), sub(layer["w_up"]), sub(layer["w_down"])
    s64 = signs.cpu().numpy().astype(np.float64)
    ref = R.build(wg, wu, wd, s64, rank=1)
    ref["U"] = U64
    ref["coef"] = wd @ U64
    local = np.array([remap[int(e)] for e in ids[0].tolist()], np.int32)
    aff = wts[0].cpu().numpy().astype(np.float64)
    x = _f64(h)[0]
    # each side built its own sketch (a few codes differ at the threshold), hence the looser
    # margin on the kept set
    dec = _check_decisions(x, local, aff, wg, wu, wd, ref, s64, K, 80, sel[0].cpu().numpy(),
                           xr[0].cpu().numpy(), score_tol=1e-2)
    o, _, _, _ = R.reader_token(x, local, aff, wg, wu, wd, ref, s64, K, 80, decisions=dec)
    G.assert_close_block(_f64(out)[0][None], o[None], "reader, full size")
