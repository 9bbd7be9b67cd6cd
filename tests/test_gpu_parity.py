"""CUDA path (through the C ABI) against the fp64 oracle on the same seeded inputs."""
import os

import numpy as np
import pytest
import torch

import gpu_ref as G
import oracle
import oracle_pins
from routed_expert_ffn_top_gb300 import moe, synthetic as syn

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as entry
    entry.build()
    yield
    torch.cuda.synchronize()


def _random_ids(rng, M, k, E, distinct=True):
    if distinct and k <= E:
        return np.stack([rng.permutation(E)[:k] for _ in range(M)]).astype(np.int32).reshape(M, k)
    return rng.integers(0, E, size=(M, k)).astype(np.int32)


def _random_affinities(rng, M, k):
    a = rng.random((M, k)) + 0.05
    return (a / a.sum(axis=1, keepdims=True)).astype(np.float32)


# ----------------------------------------------------------------------------- router
@pytest.mark.parametrize("E,k,H,M,bias,renorm", [
    (128, 8, 2048, 1, False, True), (128, 8, 2048, 21, False, True),
    (128, 8, 4096, 256, True, True), (8, 1, 128, 5, False, True), (64, 2, 256, 13, True, False),
    (512, 32, 1024, 3, False, True), (24, 5, 384, 9, True, True), (128, 8, 2048, 64, False, True),
])
def test_route_topk(E, k, H, M, bias, renorm):
    wl = syn.Workload("router_t", H=H, I=128, E=E, k=k, b=8, M=M, router_bias=bias)
    g = torch.Generator(device=DEV).manual_seed(E * 1000 + M)
    h = torch.randn(M, H, generator=g, device=DEV).to(torch.bfloat16)
    layer = {"H": H, "E": E,
             "w_router": (torch.randn(H, E, generator=g, device=DEV) * 0.02).to(torch.bfloat16),
             "bias": torch.randn(E, generator=g, device=DEV) if bias else None}
    ids, wts = moe.moe_route_topk(h, layer["w_router"], layer["bias"], k, renormalize=renorm)
    torch.cuda.synchronize()
    o_ids, o_wts, _, logits = G.oracle_routing(layer, h, k, renorm)
    _, _, near = G.check_routing(ids.cpu().numpy(), wts.cpu().numpy(), o_ids, o_wts, logits, k, renorm)
    assert near <= max(1, M // 50)


@pytest.mark.parametrize("pattern", ["period16", "zeros"])
@pytest.mark.parametrize("M", [1, 2, 3, 21])
def test_routing_exact_ties_go_to_the_lower_expert(pattern, M):
    """Logits that tie exactly: W_r's columns repeat with period 16 (each expert's logit is
    computed from the same column values in the same order, so experts e, e+16, e+32 ... tie
    bit for bit -- within one lane's experts and across lanes), or W_r is zero (every logit
    ties).  Ties go to the lower expert id, so the selection equals the oracle's exactly,
    through the router kernel, the one-grid block (M <= 2) and the multi-kernel block."""
    wl = syn.workload("layer_m21", M=M)
    layer = dict(_workload_layer("layer_m21"))
    g = torch.Generator(device=DEV).manual_seed(90 + M)
    if pattern == "zeros":
        wr = torch.zeros(wl.H, wl.E, dtype=torch.bfloat16, device=DEV)
    else:
        base = (torch.randn(wl.H, 16, generator=g, device=DEV) * 0.02).to(torch.bfloat16)
        wr = base.repeat(1, wl.E // 16).contiguous()
    layer["w_router"] = wr
    h = syn.make_hidden(wl, M=M, seed=90 + M, device=DEV)
    o_ids, o_wts, _, logits = G.oracle_routing(layer, h, wl.k)
    ids, wts = moe.moe_route_topk(h, wr, None, wl.k)
    assert np.array_equal(ids.cpu().numpy(), o_ids)
    assert np.allclose(wts.cpu().numpy(), o_wts, rtol=1e-4, atol=1e-6)
    ws = moe.alloc_workspace(layer, M, wl.k, 0)
    out, ids2, wts2 = moe.moe_decode_block(h, layer, wl.k, 0, workspace=ws)
    assert moe.moe_read_device_status(ws) == 0
    assert np.array_equal(ids2.cpu().numpy(), o_ids)
    assert torch.equal(wts2, wts)
    if pattern == "period16":  # the top group: one column's 8 experts, ascending
        top = int(o_ids[0, 0])
        assert o_ids[0].tolist() == [top + 16 * j for j in range(wl.k)]
    else:
        assert o_ids.tolist() == [list(range(wl.k))] * M
    G.assert_close_block(G.to_f64(out), G.oracle_ffn(layer, h, o_ids, o_wts), "ties")


# --------------------------------------------------------------------------- alignment
def _gpu_align(ids_np, E, b):
    ids = torch.as_tensor(ids_np, dtype=torch.int32, device=DEV).reshape(ids_np.shape)
    srt, blk, npad = moe.moe_align_block_size(ids, E, b)
    torch.cuda.synchronize()
    return srt.cpu().numpy(), blk.cpu().numpy(), int(npad.item())


def test_align_random_cases_bit_exact():
    rng = np.random.default_rng(104)
    n = 0
    for trial in range(128):
        M = int(rng.integers(0, 65))
        k = int(rng.integers(1, 9))
        E = int(rng.integers(1, 300))
        b = int(rng.choice([1, 2, 3, 4, 8, 16, 64]))
        ids = _random_ids(rng, M, k, E, distinct=(trial % 2 == 0)).reshape(M, k)
        if trial % 4 == 1 and ids.size:
            mask = rng.random(ids.shape) < 0.15
            ids[mask] = rng.choice([-1, E, E + 7, -100], size=int(mask.sum()))
        if M == 0:
            continue
        o_srt, o_blk, o_np = oracle.align(ids, E, b)
        g_srt, g_blk, g_np = _gpu_align(ids, E, b)
        assert g_np == o_np, trial
        assert np.array_equal(g_srt, o_srt), trial
        assert np.array_equal(g_blk[:o_blk.size], o_blk), trial
        n += 1
    assert n >= 104


def test_align_page_fixture():
    fx = oracle_pins.load_fixture()
    ids = oracle_pins.fixture_topk_ids(fx)
    g_srt, g_blk, g_np = _gpu_align(ids, fx["E"], fx["b"])
    o_srt, o_blk, o_np = oracle.align(ids, fx["E"], fx["b"])
    assert g_np == o_np == fx["aligned_rows"]
    assert int((g_blk >= 0).sum()) == fx["active_blocks"]
    assert np.array_equal(g_srt, o_srt) and np.array_equal(g_blk, o_blk)


@pytest.mark.parametrize("M,k", [(63, 8), (64, 8), (171, 3), (256, 8), (300, 6)])
def test_align_both_cta_sizes_bit_exact(M, k):
    """The stand-alone alignment runs one CTA of 256 threads below 512 routes and of 1024 from
    512 on; the positions are the same function of the ids on both sides of the switch, with
    distinct and repeated experts, invalid ids, and block sizes that do and do not divide
    the expert counts ([RBM] Section 2.1)."""
    rng = np.random.default_rng(500 + M * k)
    for E in (8, 128, 300):
        for b in (1, 3, 16, 64):
            for distinct in (True, False):
                ids = _random_ids(rng, M, k, E, distinct=distinct and k <= E).reshape(M, k)
                if not distinct:
                    mask = rng.random(ids.shape) < 0.1
                    ids[mask] = rng.choice([-1, E, E + 3], size=int(mask.sum()))
                o_srt, o_blk, o_np = oracle.align(ids, E, b)
                g_srt, g_blk, g_np = _gpu_align(ids, E, b)
                case = (M, k, E, b, distinct)
                assert g_np == o_np, case
                assert np.array_equal(g_srt, o_srt), case
                assert np.array_equal(g_blk[:o_blk.size], o_blk), case


def test_align_large_and_deterministic():
    rng = np.random.default_rng(7)
    ids = _random_ids(rng, 1024, 8, 256)
    ref = oracle.align(ids, 256, 16)
    for run in range(20):
        g = _gpu_align(ids, 256, 16)
        assert g[2] == ref[2] and np.array_equal(g[0], ref[0]) and np.array_equal(g[1], ref[1]), run


# ------------------------------------------------------------------- expert FFN, small
SMALL = [
    # M, k, E, H, I, b
    (1, 1, 8, 256, 256, 1), (5, 2, 8, 512, 256, 3), (13, 8, 16, 768, 512, 8),
    (3, 4, 32, 256, 768, 16), (37, 6, 64, 256, 256, 64), (64, 8, 128, 512, 256, 8),
    (2, 8, 8, 1024, 1280, 2), (9, 3, 40, 1280, 256, 5),
    # b = 64: 64-row tiles (several blocks per expert, ragged last blocks, single-route
    # blocks, K and channel counts over several tiles); b = 24, 128: blocks that fill part
    # of a 64-row tile, or two tiles
    (1, 1, 8, 256, 256, 64), (300, 2, 8, 512, 768, 64), (64, 8, 16, 1024, 512, 64),
    (129, 4, 8, 256, 1536, 64), (300, 8, 128, 768, 256, 64),
    (40, 4, 16, 512, 256, 24), (90, 8, 8, 256, 512, 128),
]


def _small_layer(M, k, E, H, I, b, seed=0, bias=False):
    wl = syn.Workload("small_%d_%d_%d_%d_%d_%d" % (M, k, E, H, I, b), H=H, I=I, E=E, k=k, b=b,
                      M=M, router_bias=bias)
    return wl, syn.make_layer(wl, seed=seed, device=DEV), syn.make_hidden(wl, seed=seed, device=DEV)


@pytest.mark.parametrize("M,k,E,H,I,b", SMALL)
def test_expert_ffn_small(M, k, E, H, I, b):
    wl, layer, h = _small_layer(M, k, E, H, I, b)
    rng = np.random.default_rng(M * 31 + E)
    ids = _random_ids(rng, M, k, E)
    a = _random_affinities(rng, M, k)
    res = syn.make_hidden(wl, seed=5, device=DEV, tag="res")
    t_ids = torch.as_tensor(ids, device=DEV)
    t_a = torch.as_tensor(a, device=DEV)
    ws = moe.alloc_workspace(layer, M, k, 0)
    out = moe.moe_expert_ffn(h, layer, t_ids, t_a, 0, residual=res, workspace=ws)
    assert moe.moe_read_device_status(ws) == 0
    ref = G.oracle_ffn(layer, h, ids, a, residual=res)
    G.assert_close_block(G.to_f64(out), ref, "expert_ffn %s" % (SMALL,))
    # the same routes aligned by the library in b-row blocks, and in the caller's own b-row
    # alignment (the first call aligned in 16- or 64-row blocks of the library's choice): a
    # route's bits do not depend on its block
    ws_b = moe.alloc_workspace(layer, M, k, b)
    out_b = moe.moe_expert_ffn(h, layer, t_ids, t_a, b, residual=res, workspace=ws_b)
    srt, blk, npad = moe.moe_align_block_size(t_ids, E, b)
    out2 = moe.moe_expert_ffn(h, layer, t_ids, t_a, b, alignment=(srt, blk, npad), residual=res,
                              workspace=ws_b)
    assert torch.equal(out, out_b) and torch.equal(out, out2)


def test_expert_ffn_invalid_ids_and_status():
    M, k, E, H, I, b = 6, 3, 16, 256, 256, 4
    wl, layer, h = _small_layer(M, k, E, H, I, b, seed=3)
    ids = np.array([[0, -1, 5], [16, 2, 3], [-5, -1, 99], [7, 7, 1], [15, 0, 4], [9, 10, 11]],
                   np.int32)
    a = _random_affinities(np.random.default_rng(1), M, k)
    res = syn.make_hidden(wl, seed=8, device=DEV, tag="res")
    ws = moe.alloc_workspace(layer, M, k, b)
    out = moe.moe_expert_ffn(h, layer, torch.as_tensor(ids, device=DEV),
                             torch.as_tensor(a, device=DEV), b, residual=res, workspace=ws)
    st = moe.moe_read_device_status(ws)
    assert st & moe.MOE_DEV_INVALID_EXPERT
    assert moe.moe_read_device_status(ws) == 0  # read clears
    ref = G.oracle_ffn(layer, h, ids, a, residual=res)
    G.assert_close_block(G.to_f64(out), ref, "invalid ids")
    # token 2 has no valid route: its output is exactly the residual
    assert torch.equal(out[2], res[2])


def test_vq_tensor_core_invalid_ids_and_status():
    """VQ decoded on the tensor cores with ids outside [0, E): those routes are dropped and
    flagged (the one-launch alignment raises the status bit), the rest match the oracle."""
    M, k, E, H, I, b = 6, 3, 16, 1024, 256, 4
    wl = syn.Workload("vq_tc_invalid", H=H, I=I, E=E, k=k, b=b, M=M, kind=syn.W_VQ, d=4, K=256,
                      vq_form=2)
    layer = syn.make_layer(wl, seed=17, device=DEV)
    h = syn.make_hidden(wl, seed=17, device=DEV)
    ids = np.array([[0, -1, 5], [16, 2, 3], [-5, -1, 99], [7, 7, 1], [15, 0, 4], [9, 10, 11]],
                   np.int32)
    a = _random_affinities(np.random.default_rng(2), M, k)
    res = syn.make_hidden(wl, seed=18, device=DEV, tag="res")
    ws = moe.alloc_workspace(layer, M, k, b)
    out = moe.moe_expert_ffn(h, layer, torch.as_tensor(ids, device=DEV),
                             torch.as_tensor(a, device=DEV), b, residual=res, workspace=ws)
    assert moe.moe_read_device_status(ws) & moe.MOE_DEV_INVALID_EXPERT
    G.assert_close_block(G.to_f64(out), G.oracle_ffn(layer, h, ids, a, residual=res),
                         "vq tensor cores, invalid ids")
    assert torch.equal(out[2], res[2])


@pytest.mark.parametrize("b", [2, 64])
def test_expert_ffn_bad_alignment_is_flagged(b):
    M, k, E, H, I = 4, 2, 8, 256, 256
    wl, layer, h = _small_layer(M, k, E, H, I, b, seed=4)
    ids = np.array([[0, 1], [1, 2], [2, 3], [3, 0]], np.int32)
    t_ids = torch.as_tensor(ids, device=DEV)
    a = torch.full((M, k), 0.5, device=DEV)
    srt, blk, npad = moe.moe_align_block_size(t_ids, E, b)
    srt_bad = srt.clone()
    s = srt_bad.cpu().numpy()
    s[0], s[b] = s[b], s[0]  # move a route of expert 1 into expert 0's block
    srt_bad.copy_(torch.as_tensor(s))
    ws = moe.alloc_workspace(layer, M, k, b)
    moe.moe_expert_ffn(h, layer, t_ids, a, b, alignment=(srt_bad, blk, npad), workspace=ws)
    assert moe.moe_read_device_status(ws) & moe.MOE_DEV_BAD_ALIGNMENT


def test_membership_invariance_bitwise():
    """A route's output bits do not depend on which aligned block it occupies: the
    route-block page's within-block permutation and boundary exchange both preserve them."""
    M, k, E, H, I, b = 24, 2, 8, 512, 256, 4
    wl, layer, h = _small_layer(M, k, E, H, I, b, seed=6)
    ids = np.stack([[m % 3, 3 + m % 5] for m in range(M)]).astype(np.int32)  # experts with many routes
    a = _random_affinities(np.random.default_rng(2), M, k)
    t_ids, t_a = torch.as_tensor(ids, device=DEV), torch.as_tensor(a, device=DEV)
    srt, blk, npad = moe.moe_align_block_size(t_ids, E, b)
    ws = moe.alloc_workspace(layer, M, k, b)
    base = moe.moe_expert_ffn(h, layer, t_ids, t_a, b, alignment=(srt, blk, npad), workspace=ws)
    s = srt.cpu().numpy()
    bl = blk.cpu().numpy()
    e0_rows = [i for i in range(int(npad.item())) if bl[i // b] == 0 and s[i] < M * k]
    assert len(e0_rows) >= b + 1  # spans at least two blocks
    within = s.copy()
    within[e0_rows[0]], within[e0_rows[1]] = within[e0_rows[1]], within[e0_rows[0]]
    boundary = s.copy()
    boundary[e0_rows[b - 1]], boundary[e0_rows[b]] = boundary[e0_rows[b]], boundary[e0_rows[b - 1]]
    shuffled = s.copy()
    shuffled[e0_rows] = np.random.default_rng(0).permutation(s[e0_rows])
    for variant in (within, boundary, shuffled):
        alt = torch.as_tensor(variant, device=DEV)
        out = moe.moe_expert_ffn(h, layer, t_ids, t_a, b, alignment=(alt, blk, npad), workspace=ws)
        assert torch.equal(out, base)
    assert moe.moe_read_device_status(ws) == 0


def test_expert_ffn_m0_is_noop():
    wl, layer, h = _small_layer(1, 2, 8, 256, 256, 8)
    out = torch.zeros(0, 256, dtype=torch.bfloat16, device=DEV)
    ids = torch.zeros(0, 2, dtype=torch.int32, device=DEV)
    a = torch.zeros(0, 2, dtype=torch.float32, device=DEV)
    ws = torch.zeros(1024, dtype=torch.uint8, device=DEV)
    moe.moe_expert_ffn(h[:0], layer, ids, a, 8, out=out, workspace=ws)


# ----------------------------------------------------------------- the five workloads
_cache = {}


def _workload_layer(name, layer_idx=0, seed=0):
    key = (name, layer_idx, seed)
    if key not in _cache:
        _cache.clear()
        torch.cuda.empty_cache()
        wl = syn.WORKLOADS[name]
        _cache[key] = syn.make_layer(wl, layer=layer_idx, seed=seed, device=DEV)
    return _cache[key]


def _check_block(name, M=None, tokens=None, seed=0):
    wl = syn.WORKLOADS[name]
    layer = _workload_layer(name, seed=seed)
    M = wl.M if M is None else M
    h = syn.make_hidden(wl, M=M, seed=seed, device=DEV)
    ws = moe.alloc_workspace(layer, M, wl.k, wl.b)
    out, ids, wts = moe.moe_decode_block(h, layer, wl.k, wl.b, workspace=ws)
    assert moe.moe_read_device_status(ws) == 0
    o_ids, o_wts, _, logits = G.oracle_routing(layer, h, wl.k)
    use_ids, use_wts, near = G.check_routing(ids.cpu().numpy(), wts.cpu().numpy(), o_ids, o_wts,
                                             logits, wl.k)
    ref = G.oracle_ffn(layer, h, use_ids, use_wts, tokens=tokens)
    got = G.to_f64(out) if tokens is None else G.to_f64(out)[tokens]
    G.assert_close_block(got, ref, name)
    return layer, h, ws, out, ids, wts


def test_layer_m1():
    _check_block("layer_m1")


def test_layer_m21_alignment_and_20_run_determinism():
    wl = syn.WORKLOADS["layer_m21"]
    layer, h, ws, out, ids, wts = _check_block("layer_m21")
    # alignment of the router's ids: bit-exact against the oracle
    srt, blk, npad = moe.moe_align_block_size(ids, wl.E, wl.b)
    o_srt, o_blk, o_np = oracle.align(ids.cpu().numpy(), wl.E, wl.b)
    assert int(npad.item()) == o_np
    assert np.array_equal(srt.cpu().numpy(), o_srt)
    assert np.array_equal(blk.cpu().numpy()[:o_blk.size], o_blk)
    for run in range(20):
        out2, ids2, wts2 = moe.moe_decode_block(h, layer, wl.k, wl.b, workspace=ws)
        assert torch.equal(out2, out) and torch.equal(ids2, ids) and torch.equal(wts2, wts), run


@pytest.mark.parametrize("name,M,b", [
    ("layer_m21", 1, 0), ("layer_m21", 1, 8), ("layer_m21", 2, 8), ("layer_m21", 2, 16),
    ("layer_m21", 3, 8), ("layer_m21", 8, 16), ("layer_m21", 16, 8), ("layer_m21", 16, 0),
    ("layer_m21", 21, 8), ("layer_m21", 40, 0), ("vq_d4", 1, 8), ("vq_d4", 2, 3),
    ("vq_d4", 9, 8)])
def test_decode_block_alignment_bit_exact(name, M, b):
    """The alignment the decode block itself builds -- in the router's launch for up to 2
    tokens, in one launch with the row tiles up to 128 routes, in the stand-alone kernel
    above -- equals the oracle's alignment of the call's own ids element by element: the
    sorted route ids with the sentinel tail, the block vector with its -1 tail, the row
    count.  The workspace starts dirty, so every entry must have been written."""
    wl = syn.workload(name, M=M)
    layer = _workload_layer(name)
    h = syn.make_hidden(wl, M=M, seed=40 + M, device=DEV)
    ws = moe.alloc_workspace(layer, M, wl.k, b)
    lay = moe.moe_workspace_layout(layer, M, wl.k, b)
    ws.fill_(0xFF)
    ws[:lay["zero_bytes"]] = 0  # the status word and counters start at zero, as required
    out, ids, wts = moe.moe_decode_block(h, layer, wl.k, b, workspace=ws)
    assert moe.moe_read_device_status(ws) == 0
    assert lay["b"] == (b if b else moe.moe_library_block_size(layer, M, wl.k, 0))
    srt, blk, npad = moe.workspace_alignment(ws, lay)
    o_srt, o_blk, o_np = oracle.align(ids.cpu().numpy(), wl.E, lay["b"])
    assert int(npad.item()) == o_np
    assert np.array_equal(srt.cpu().numpy(), o_srt)
    assert np.array_equal(blk.cpu().numpy(), o_blk)
    o_ids, o_wts, _, logits = G.oracle_routing(layer, h, wl.k)
    G.check_routing(ids.cpu().numpy(), wts.cpu().numpy(), o_ids, o_wts, logits, wl.k)


@pytest.mark.parametrize("M,b", [(1, 0), (2, 8), (21, 8), (40, 64)])
def test_block_surfaces_match_oracle_intermediates(M, b):
    """The intermediate surfaces one decode block leaves in its workspace -- p = SiLU(g) * u
    (bf16: the p rows of the one-grid path up to 2 tokens, else the swizzled 16- or 64-row p
    tiles) and y = p W_down (fp32) -- read back the way the bench hashes them, against the
    oracle's p and y of the same routes."""
    import bench
    wl = syn.workload("layer_m21", M=M)
    layer = _workload_layer("layer_m21")
    h = syn.make_hidden(wl, M=M, seed=70 + M, device=DEV)
    ws = moe.alloc_workspace(layer, M, wl.k, b)
    out, ids, wts = moe.moe_decode_block(h, layer, wl.k, b, workspace=ws)
    assert moe.moe_read_device_status(ws) == 0
    valid, p, y = bench.surface_tensors(moe, layer, M, wl.k, b, ws, ids)
    assert valid.numel() == M * wl.k
    o_p, o_y = G.oracle_intermediates(layer, h, ids.cpu().numpy(), wts.cpu().numpy())
    rows = valid.cpu().numpy()
    assert G.rel_l2(G.to_f64(p), o_p[rows]) <= 4e-3  # p is rounded to bf16 (2^-9 relative)
    G.assert_close_block(G.to_f64(y), o_y[rows], "y")


def test_batch_invariance_bitwise():
    wl = syn.WORKLOADS["layer_m21"]
    layer = _workload_layer("layer_m21")
    h = syn.make_hidden(wl, seed=0, device=DEV)
    out, ids, _ = moe.moe_decode_block(h, layer, wl.k, wl.b)
    for m in (0, 7, 20):
        o1, i1, _ = moe.moe_decode_block(h[m:m + 1].contiguous(), layer, wl.k, wl.b)
        assert torch.equal(i1[0], ids[m]) and torch.equal(o1[0], out[m]), m
    o5, _, _ = moe.moe_decode_block(h[3:8].contiguous(), layer, wl.k, wl.b)
    assert torch.equal(o5, out[3:8])


def test_host_entry_point_matches_device():
    wl = syn.WORKLOADS["layer_m21"]
    layer = _workload_layer("layer_m21")
    h = syn.make_hidden(wl, seed=0, device=DEV)
    ws = moe.alloc_workspace(layer, wl.M, wl.k, wl.b)
    out, ids, wts = moe.moe_decode_block(h, layer, wl.k, wl.b, workspace=ws)
    h_host = h.cpu().pin_memory()
    out_host = torch.empty_like(h_host).pin_memory()
    h_dev, out_dev = torch.empty_like(h), torch.empty_like(h)
    moe.moe_decode_block_host(h_host, layer, wl.k, wl.b, h_dev, out_dev, out_host,
                              torch.empty_like(ids), torch.empty_like(wts), ws)
    assert torch.equal(out_host, out.cpu())


VQ_SMALL = [
    # M, k, E, H, I, b, d
    (5, 2, 8, 1024, 256, 3, 4), (13, 4, 16, 2048, 512, 8, 4), (2, 8, 8, 1024, 768, 1, 4),
    (30, 3, 24, 1024, 256, 16, 4), (5, 2, 8, 1024, 256, 3, 8), (13, 4, 16, 2048, 512, 8, 8),
    (30, 3, 24, 3072, 256, 16, 8),
]


@pytest.mark.parametrize("M,k,E,H,I,b,d", VQ_SMALL)
def test_vq_expert_ffn_small(M, k, E, H, I, b, d):
    wl = syn.Workload("vq_small_%d_%d_%d_%d" % (M, k, E, d), H=H, I=I, E=E, k=k, b=b, M=M,
                      kind=syn.W_VQ, d=d, K=256)
    layer = syn.make_layer(wl, seed=2, device=DEV)
    h = syn.make_hidden(wl, seed=2, device=DEV)
    rng = np.random.default_rng(M + E)
    ids = _random_ids(rng, M, k, E)
    a = _random_affinities(rng, M, k)
    res = syn.make_hidden(wl, seed=4, device=DEV, tag="res")
    ws = moe.alloc_workspace(layer, M, k, b)
    out = moe.moe_expert_ffn(h, layer, torch.as_tensor(ids, device=DEV),
                             torch.as_tensor(a, device=DEV), b, residual=res, workspace=ws)
    assert moe.moe_read_device_status(ws) == 0
    ref = G.oracle_ffn(layer, h, ids, a, residual=res)
    G.assert_close_block(G.to_f64(out), ref, "vq expert_ffn")


VQ_TT = [
    # M, k, E, H, I, b, d: projected code books (at most 4 tokens)
    (1, 8, 16, 1024, 256, 8, 4), (3, 4, 16, 2048, 512, 1, 4), (4, 8, 8, 1024, 768, 8, 8),
    (2, 2, 8, 3072, 256, 3, 8),
]


@pytest.mark.parametrize("M,k,E,H,I,b,d", VQ_TT)
def test_vq_projected_codebooks_small(M, k, E, H, I, b, d):
    wl = syn.Workload("vq_tt_%d_%d_%d_%d" % (M, k, E, d), H=H, I=I, E=E, k=k, b=b, M=M,
                      kind=syn.W_VQ, d=d, K=256, vq_form=1)
    layer = syn.make_layer(wl, seed=12, device=DEV)
    h = syn.make_hidden(wl, seed=12, device=DEV)
    rng = np.random.default_rng(M * 7 + E)
    ids = _random_ids(rng, M, k, E)
    a = _random_affinities(rng, M, k)
    res = syn.make_hidden(wl, seed=13, device=DEV, tag="res")
    ws = moe.alloc_workspace(layer, M, k, b)
    out = moe.moe_expert_ffn(h, layer, torch.as_tensor(ids, device=DEV),
                             torch.as_tensor(a, device=DEV), b, residual=res, workspace=ws)
    assert moe.moe_read_device_status(ws) == 0
    ref = G.oracle_ffn(layer, h, ids, a, residual=res)
    G.assert_close_block(G.to_f64(out), ref, "vq projected code books")


def test_vq_projected_codebooks_block_and_invariance():
    """The VQ layer with projected code books: parity at M = 1..4, a token's bits the same
    alone and in a batch, within the bar of the shared-memory code-book form, and more
    than 4 tokens refused."""
    wl = syn.WORKLOADS["vq_d4_tt"]
    layer = _workload_layer("vq_d4_tt")
    h4 = syn.make_hidden(wl, M=4, seed=3, device=DEV)
    out4, ids4, wts4 = moe.moe_decode_block(h4, layer, wl.k, wl.b)
    o_ids, o_wts, _, logits = G.oracle_routing(layer, h4, wl.k)
    use_ids, use_wts, _ = G.check_routing(ids4.cpu().numpy(), wts4.cpu().numpy(), o_ids, o_wts,
                                          logits, wl.k)
    G.assert_close_block(G.to_f64(out4), G.oracle_ffn(layer, h4, use_ids, use_wts), "tt M=4")
    for M in (1, 2, 3):
        o, i, _ = moe.moe_decode_block(h4[:M].contiguous(), layer, wl.k, wl.b)
        assert torch.equal(i, ids4[:M]) and torch.equal(o, out4[:M]), M
    smem_form = dict(layer, vq_form=0)
    o_cb = moe.moe_expert_ffn(h4, smem_form, ids4, wts4, wl.b)
    G.assert_close_block(G.to_f64(o_cb), G.to_f64(out4).astype(np.float64), "two VQ forms")
    h5 = syn.make_hidden(wl, M=5, seed=3, device=DEV)
    with pytest.raises(moe.MoeError) as err:
        moe.moe_decode_block(h5, layer, wl.k, wl.b)
    assert err.value.status == moe.MOE_ERR_UNSUPPORTED


def test_vq_block_every_m_1_to_16():
    """The blockwise-VQ workload: parity at every M from 1 to 16 (one weight set)."""
    wl = syn.WORKLOADS["vq_d4"]
    layer = _workload_layer("vq_d4")
    for M in range(1, 17):
        h = syn.make_hidden(wl, M=M, seed=M, device=DEV)
        ws = moe.alloc_workspace(layer, M, wl.k, wl.b)
        out, ids, wts = moe.moe_decode_block(h, layer, wl.k, wl.b, workspace=ws)
        assert moe.moe_read_device_status(ws) == 0
        o_ids, o_wts, _, logits = G.oracle_routing(layer, h, wl.k)
        use_ids, use_wts, _ = G.check_routing(ids.cpu().numpy(), wts.cpu().numpy(), o_ids, o_wts,
                                              logits, wl.k)
        ref = G.oracle_ffn(layer, h, use_ids, use_wts)
        G.assert_close_block(G.to_f64(out), ref, "vq_d4 M=%d" % M)
    # bitwise determinism and batch invariance of the VQ path
    out2, _, _ = moe.moe_decode_block(h, layer, wl.k, wl.b, workspace=ws)
    assert torch.equal(out2, out)
    o1, _, _ = moe.moe_decode_block(h[3:4].contiguous(), layer, wl.k, wl.b)
    assert torch.equal(o1[0], out[3])


VQ_TC = [
    # M, k, E, H, I, b, d: index maps decoded into the tensor cores' weight operand
    (5, 2, 8, 1024, 256, 3, 4), (13, 4, 16, 2048, 512, 8, 4), (2, 8, 8, 1024, 768, 1, 4),
    (30, 3, 24, 1024, 256, 16, 4), (40, 4, 8, 1024, 256, 24, 4), (5, 2, 8, 1024, 256, 3, 8),
    (13, 4, 16, 2048, 512, 8, 8), (30, 3, 24, 3072, 256, 16, 8), (64, 8, 16, 1024, 512, 64, 8),
]


@pytest.mark.parametrize("M,k,E,H,I,b,d", VQ_TC)
def test_vq_tensor_core_small(M, k, E, H, I, b, d):
    """VQ gate/up on the tcgen05 path: parity with the oracle through the library's
    alignment and the caller's (b = 1 .. 64, so 1 to 4 sixteen-row tiles per block), the same
    bits both ways, within the bar of the shared-memory code-book form."""
    wl = syn.Workload("vq_tc_%d_%d_%d_%d" % (M, k, E, d), H=H, I=I, E=E, k=k, b=b, M=M,
                      kind=syn.W_VQ, d=d, K=256, vq_form=2)
    layer = syn.make_layer(wl, seed=14, device=DEV)
    h = syn.make_hidden(wl, seed=14, device=DEV)
    rng = np.random.default_rng(M * 3 + E + d)
    ids = _random_ids(rng, M, k, E)
    a = _random_affinities(rng, M, k)
    t_ids, t_a = torch.as_tensor(ids, device=DEV), torch.as_tensor(a, device=DEV)
    res = syn.make_hidden(wl, seed=15, device=DEV, tag="res")
    ws = moe.alloc_workspace(layer, M, k, b)
    out = moe.moe_expert_ffn(h, layer, t_ids, t_a, b, residual=res, workspace=ws)
    assert moe.moe_read_device_status(ws) == 0
    ref = G.oracle_ffn(layer, h, ids, a, residual=res)
    G.assert_close_block(G.to_f64(out), ref, "vq tensor cores")
    srt, blk, npad = moe.moe_align_block_size(t_ids, E, b)
    o = moe.moe_expert_ffn(h, layer, t_ids, t_a, b, alignment=(srt, blk, npad), residual=res)
    assert torch.equal(o, out)
    o_cb = moe.moe_expert_ffn(h, dict(layer, vq_form=0), t_ids, t_a, b, residual=res)
    G.assert_close_block(G.to_f64(o_cb), G.to_f64(out).astype(np.float64), "two VQ forms")


def test_vq_tensor_core_bits_same_in_both_tile_widths():
    """VQ on the tensor cores: 64-row tiles (the library's choice from 16 routes per expert)
    and 16-row tiles (a caller's b = 8 alignment, or a few tokens) give every route the same
    bits: one K-ordered MMA chain per element in both widths."""
    M, k, E, H, I, d = 40, 4, 8, 1024, 512, 4
    wl = syn.Workload("vq_tc_widths", H=H, I=I, E=E, k=k, b=8, M=M, kind=syn.W_VQ, d=d, K=256,
                      vq_form=2)
    layer = syn.make_layer(wl, seed=16, device=DEV)
    h = syn.make_hidden(wl, seed=16, device=DEV)
    rng = np.random.default_rng(16)
    ids = _random_ids(rng, M, k, E)
    a = _random_affinities(rng, M, k)
    t_ids, t_a = torch.as_tensor(ids, device=DEV), torch.as_tensor(a, device=DEV)
    assert moe.moe_library_block_size(layer, M, k, 0) == 64
    wide = moe.moe_expert_ffn(h, layer, t_ids, t_a, 0)  # library: 64-row blocks
    G.assert_close_block(G.to_f64(wide), G.oracle_ffn(layer, h, ids, a), "vq 64-row tiles")
    for b in (1, 8, 16, 24, 64, 128):
        srt, blk, npad = moe.moe_align_block_size(t_ids, E, b)
        o = moe.moe_expert_ffn(h, layer, t_ids, t_a, b, alignment=(srt, blk, npad))
        assert torch.equal(o, wide), b
    for sub in ([7], [0, 39], list(range(3, 9))):
        sel = torch.as_tensor(sub, device=DEV)
        o = moe.moe_expert_ffn(h[sel].contiguous(), layer, t_ids[sel].contiguous(),
                               t_a[sel].contiguous(), 0)  # library: 16-row blocks
        assert torch.equal(o, wide[sel]), sub


def test_vq_tensor_core_block_every_m_and_invariance():
    """The VQ decode layer on the tcgen05 path: parity at M = 1..16 (the router writes the
    row tiles up to 8 tokens, the row gather does above), each token's bits the same alone,
    in any batch and in a dirty workspace."""
    wl = syn.WORKLOADS["vq_d4_tc"]
    layer = _workload_layer("vq_d4_tc")
    h16 = syn.make_hidden(wl, M=16, seed=9, device=DEV)
    out16, ids16, _ = moe.moe_decode_block(h16, layer, wl.k, wl.b)
    for M in range(1, 17):
        h = h16[:M].contiguous()
        ws = moe.alloc_workspace(layer, M, wl.k, wl.b)
        if M in (1, 7, 12):
            ws.fill_(0xFF)
            ws[:moe.moe_workspace_layout(layer, M, wl.k, wl.b)["zero_bytes"]] = 0
        out, ids, wts = moe.moe_decode_block(h, layer, wl.k, wl.b, workspace=ws)
        assert moe.moe_read_device_status(ws) == 0
        assert torch.equal(ids, ids16[:M]) and torch.equal(out, out16[:M]), M
        if M in (1, 2, 5, 8, 9, 16):
            o_ids, o_wts, _, logits = G.oracle_routing(layer, h, wl.k)
            use_ids, use_wts, _ = G.check_routing(ids.cpu().numpy(), wts.cpu().numpy(), o_ids,
                                                  o_wts, logits, wl.k)
            G.assert_close_block(G.to_f64(out), G.oracle_ffn(layer, h, use_ids, use_wts),
                                 "vq_d4_tc M=%d" % M)
    for t in (0, 5, 15):
        o1, _, _ = moe.moe_decode_block(h16[t:t + 1].contiguous(), layer, wl.k, wl.b)
        assert torch.equal(o1[0], out16[t]), t
    runs = [moe.moe_decode_block(h16, layer, wl.k, wl.b)[0] for _ in range(5)]
    assert all(torch.equal(r, out16) for r in runs)
    # 256 tokens (16 routes per expert) run 64-row tiles: the 16 shared tokens keep their
    # bits; sampled parity
    assert moe.moe_library_block_size(layer, 256, wl.k, 0) == 64
    h256 = torch.cat([h16, syn.make_hidden(wl, M=240, seed=10, device=DEV)])
    out256, ids256, wts256 = moe.moe_decode_block(h256, layer, wl.k, 0)
    assert torch.equal(ids256[:16], ids16) and torch.equal(out256[:16], out16)
    o_ids, o_wts, _, logits = G.oracle_routing(layer, h256, wl.k)
    use_ids, use_wts, _ = G.check_routing(ids256.cpu().numpy(), wts256.cpu().numpy(), o_ids,
                                          o_wts, logits, wl.k)
    tokens = np.array([16, 130, 255])
    G.assert_close_block(G.to_f64(out256)[tokens],
                         G.oracle_ffn(layer, h256, use_ids, use_wts, tokens=tokens),
                         "vq_d4_tc M=256")


VQLR_SMALL = [
    # M, k, E, H, I, b, r, d
    (5, 2, 8, 1024, 256, 3, 128, 4), (13, 4, 16, 2048, 512, 8, 256, 4),
    (2, 8, 8, 1024, 768, 1, 384, 4), (30, 3, 24, 1024, 256, 16, 512, 4),
    (1, 1, 8, 1024, 256, 8, 256, 4), (13, 4, 16, 2048, 512, 8, 384, 8), (3, 2, 8, 1024, 256, 1, 128, 8),
]


@pytest.mark.parametrize("M,k,E,H,I,b,r,d", VQLR_SMALL)
def test_vqlr_expert_ffn_small(M, k, E, H, I, b, r, d):
    """VQ + low-rank gate/up through moe_expert_ffn (the projections get their own launch)."""
    wl = syn.Workload("vqlr_small_%d_%d_%d_%d_%d" % (M, k, E, r, d), H=H, I=I, E=E, k=k, b=b,
                      M=M, kind=syn.W_VQLR, d=d, K=256, r=r)
    layer = syn.make_layer(wl, seed=3, device=DEV)
    h = syn.make_hidden(wl, seed=3, device=DEV)
    rng = np.random.default_rng(M + E + r)
    ids = _random_ids(rng, M, k, E)
    a = _random_affinities(rng, M, k)
    res = syn.make_hidden(wl, seed=5, device=DEV, tag="res")
    ws = moe.alloc_workspace(layer, M, k, b)
    out = moe.moe_expert_ffn(h, layer, torch.as_tensor(ids, device=DEV),
                             torch.as_tensor(a, device=DEV), b, residual=res, workspace=ws)
    assert moe.moe_read_device_status(ws) == 0
    ref = G.oracle_ffn(layer, h, ids, a, residual=res)
    G.assert_close_block(G.to_f64(out), ref, "vqlr expert_ffn r=%d" % r)
    # the low-rank term matters: without it the output misses the bar by a wide margin
    # (the unit-scale residual dominates the relative error, hence 3x rather than more)
    vq = dict(layer)
    vq["kind"] = syn.W_VQ
    out_vq = moe.moe_expert_ffn(h, vq, torch.as_tensor(ids, device=DEV),
                                torch.as_tensor(a, device=DEV), b, residual=res)
    assert G.rel_l2(G.to_f64(out_vq), ref) > 3 * G.REL_L2


@pytest.mark.parametrize("name", ["vqlr_d4_r256", "vqlr_d8_r384"])
def test_vqlr_block_every_m_1_to_16(name):
    """The VQ + low-rank workloads ((d, r) = (4, 256) and the pages' deployed (8, 384)): the
    projections ride in the router launch; parity at every M from 1 to 16, bitwise
    determinism and batch invariance."""
    wl = syn.WORKLOADS[name]
    layer = _workload_layer(name)
    for M in range(1, 17):
        h = syn.make_hidden(wl, M=M, seed=M, device=DEV)
        ws = moe.alloc_workspace(layer, M, wl.k, wl.b)
        out, ids, wts = moe.moe_decode_block(h, layer, wl.k, wl.b, workspace=ws)
        assert moe.moe_read_device_status(ws) == 0
        o_ids, o_wts, _, logits = G.oracle_routing(layer, h, wl.k)
        use_ids, use_wts, _ = G.check_routing(ids.cpu().numpy(), wts.cpu().numpy(), o_ids, o_wts,
                                              logits, wl.k)
        ref = G.oracle_ffn(layer, h, use_ids, use_wts)
        G.assert_close_block(G.to_f64(out), ref, "%s M=%d" % (name, M))
    out2, _, _ = moe.moe_decode_block(h, layer, wl.k, wl.b, workspace=ws)
    assert torch.equal(out2, out)
    o1, _, _ = moe.moe_decode_block(h[3:4].contiguous(), layer, wl.k, wl.b)
    assert torch.equal(o1[0], out[3])
    # the decode block (projections in the router launch) and the expert entry point
    # (projections in a launch of their own) agree bit for bit
    o3 = moe.moe_expert_ffn(h, layer, ids, wts, wl.b)
    assert torch.equal(o3, out)


def test_large_m256_sampled_tokens():
    """The large-batch layer (H=4096, I=1536, b=64, biased router): 64 of its 256 tokens (every
    fourth, plus the last) against the oracle, which runs its routes on all host cores."""
    tokens = np.unique(np.concatenate([np.arange(0, 256, 4), [255]]))
    before = oracle.set_threads(0)
    oracle.set_threads(os.cpu_count() or 1)
    try:
        layer, h, ws, out, ids, wts = _check_block("large_m256", tokens=tokens)
    finally:
        oracle.set_threads(before)
    wl = syn.WORKLOADS["large_m256"]
    out2, _, _ = moe.moe_decode_block(h, layer, wl.k, wl.b, workspace=ws)
    assert torch.equal(out, out2)


def test_decode_block_picks_the_gemm_regime_for_large_batches():
    """Left to the library (b = 0), the default layer aligns in 64-row blocks (64-row tiles)
    from 24 routes per expert (one wave of 16-row units' weights fits in L2 there), below that
    in 16-row blocks; the caller's b = 8 or 64 is kept; the bits are the same every way."""
    wl = syn.workload("layer_m21", M=384)
    layer = _workload_layer("layer_m21")
    assert moe.moe_library_block_size(layer, 384, wl.k, 0) == 64
    assert moe.moe_library_block_size(layer, 64, wl.k, 0) == 16
    assert moe.moe_library_block_size(layer, 384, wl.k, 8) == 8
    h = syn.make_hidden(wl, M=384, seed=64, device=DEV)
    out8, ids, wts = moe.moe_decode_block(h, layer, wl.k, 8)
    out64, _, _ = moe.moe_decode_block(h, layer, wl.k, 64)
    out0, _, _ = moe.moe_decode_block(h, layer, wl.k, 0)
    assert torch.equal(out8, out64) and torch.equal(out8, out0)
    assert torch.equal(moe.moe_expert_ffn(h, layer, ids, wts, 8), out8)
    tokens = np.array([0, 170, 383])
    o_ids, o_wts, _, logits = G.oracle_routing(layer, h, wl.k)
    use_ids, use_wts, _ = G.check_routing(ids.cpu().numpy(), wts.cpu().numpy(), o_ids, o_wts,
                                          logits, wl.k)
    ref = G.oracle_ffn(layer, h, use_ids, use_wts, tokens=tokens)
    G.assert_close_block(G.to_f64(out8)[tokens], ref, "M=384, 64-row tiles")
    # below the threshold (M=64: 4 routes per expert) 16-row tiles run: the same tokens keep
    # their bits, and so does a caller's own 8-row alignment
    h64 = h[:64].contiguous()
    o64, ids64, wts64 = moe.moe_decode_block(h64, layer, wl.k, 8)
    assert torch.equal(ids64, ids[:64]) and torch.equal(o64, out8[:64])
    srt, blk, npad = moe.moe_align_block_size(ids64, wl.E, 8)
    assert torch.equal(moe.moe_expert_ffn(h64, layer, ids64, wts64, 8, alignment=(srt, blk, npad)),
                       o64)


def test_gemm_regime_batch_and_membership_invariance():
    """With 64-row tiles a route is one column of its tile's MMA: its bits do not
    depend on the other routes of the block, on the block's position or on M."""
    M, k, E, H, I, b = 96, 4, 8, 512, 512, 64
    wl, layer, h = _small_layer(M, k, E, H, I, b, seed=3)
    rng = np.random.default_rng(11)
    ids = _random_ids(rng, M, k, E)
    a = _random_affinities(rng, M, k)
    t_ids = torch.as_tensor(ids, device=DEV)
    t_a = torch.as_tensor(a, device=DEV)
    out = moe.moe_expert_ffn(h, layer, t_ids, t_a, b)
    for sub in ([5], [0, 95], list(range(40, 71)), list(range(95, -1, -3))):
        sel = torch.as_tensor(sub, device=DEV)
        o = moe.moe_expert_ffn(h[sel].contiguous(), layer, t_ids[sel].contiguous(),
                               t_a[sel].contiguous(), b)
        assert torch.equal(o, out[sel]), sub
    ref = G.oracle_ffn(layer, h, ids, a)
    G.assert_close_block(G.to_f64(out), ref, "gemm regime")


def test_route_bits_independent_of_batch_block_and_tile_width():
    """Every route of dense weights is one K-ordered chain of tcgen05 MMAs per projection
    (the route-block page's batch- and membership-invariance as a guarantee): a token's
    output bits are the same alone or in any batch, in blocks of 1, 8, 16, 24, 64 or 128
    rows, in 16- or 64-row tiles, through the library's own alignment or the caller's."""
    M, k, E, H, I = 72, 8, 16, 512, 768
    wl, layer, h = _small_layer(M, k, E, H, I, 8, seed=21)
    rng = np.random.default_rng(21)
    ids = _random_ids(rng, M, k, E)
    a = _random_affinities(rng, M, k)
    t_ids, t_a = torch.as_tensor(ids, device=DEV), torch.as_tensor(a, device=DEV)
    assert moe.moe_library_block_size(layer, M, k, 0) == 64
    base = moe.moe_expert_ffn(h, layer, t_ids, t_a, 0)  # library: 64-row blocks
    ref = G.oracle_ffn(layer, h, ids, a)
    G.assert_close_block(G.to_f64(base), ref, "cross-regime base")
    for b in (1, 8, 16, 24, 64, 128):
        srt, blk, npad = moe.moe_align_block_size(t_ids, E, b)
        o = moe.moe_expert_ffn(h, layer, t_ids, t_a, b, alignment=(srt, blk, npad))
        assert torch.equal(o, base), b
    for sub in ([3], [0, 71], list(range(10, 17)), list(range(71, -1, -5))):
        sel = torch.as_tensor(sub, device=DEV)
        o = moe.moe_expert_ffn(h[sel].contiguous(), layer, t_ids[sel].contiguous(),
                               t_a[sel].contiguous(), 0)  # library: 16-row blocks
        assert torch.equal(o, base[sel]), sub


@pytest.mark.parametrize("M,b", [(1, 8), (2, 8), (8, 8), (21, 8), (64, 8), (3, 64)])
def test_decode_block_on_a_dirty_workspace(M, b):
    """Every buffer of the workspace is written before it is read: a workspace whose bytes
    are all 0xFF (NaN in every float view) gives the same bits as a zeroed one, from the
    first call on.  A kernel that read a buffer before its producer finished would see NaN."""
    wl = syn.workload("layer_m21", M=M)
    layer = _workload_layer("layer_m21")
    h = syn.make_hidden(wl, M=M, seed=31, device=DEV)
    res = syn.make_hidden(wl, M=M, seed=32, device=DEV, tag="res")
    ws = moe.alloc_workspace(layer, M, wl.k, b)
    dirty = torch.full_like(ws, 0xFF)
    # the status word and the counters start clear, as the entry points require
    dirty[:moe.moe_workspace_layout(layer, M, wl.k, b)["zero_bytes"]] = 0
    out_d, ids_d, _ = moe.moe_decode_block(h, layer, wl.k, b, residual=res, workspace=dirty)
    out_z, ids_z, wts_z = moe.moe_decode_block(h, layer, wl.k, b, residual=res, workspace=ws)
    assert moe.moe_read_device_status(dirty) == 0
    assert torch.equal(ids_d, ids_z) and torch.equal(out_d, out_z)
    zb = moe.moe_workspace_layout(layer, M, wl.k, b)["zero_bytes"]
    assert int(dirty[:zb].count_nonzero().item()) == 0  # every call leaves them zero
    o_ids, o_wts, _, logits = G.oracle_routing(layer, h, wl.k)
    use_ids, use_wts, _ = G.check_routing(ids_z.cpu().numpy(), wts_z.cpu().numpy(), o_ids, o_wts,
                                          logits, wl.k)
    tokens = None if M <= 21 else np.array([0, M // 2, M - 1])
    ref = G.oracle_ffn(layer, h, use_ids, use_wts, residual=res, tokens=tokens)
    got = G.to_f64(out_z) if tokens is None else G.to_f64(out_z)[tokens]
    G.assert_close_block(got, ref, "dirty workspace M=%d" % M)


def test_decode_block_bits_same_in_both_tile_widths():
    """The default layer: M=21 runs 16-row tiles, M=384 64-row tiles; the 21 shared tokens
    keep their routing and their output bits."""
    wl = syn.WORKLOADS["layer_m21"]
    layer = _workload_layer("layer_m21")
    h384 = syn.make_hidden(wl, M=384, seed=5, device=DEV)
    o384, i384, _ = moe.moe_decode_block(h384, layer, wl.k, wl.b)
    o21, i21, _ = moe.moe_decode_block(h384[:21].contiguous(), layer, wl.k, wl.b)
    o1, i1, _ = moe.moe_decode_block(h384[40:41].contiguous(), layer, wl.k, wl.b)
    assert torch.equal(i21, i384[:21]) and torch.equal(o21, o384[:21])
    assert torch.equal(i1[0], i384[40]) and torch.equal(o1[0], o384[40])


@pytest.mark.parametrize("M", [1, 4, 16, 64])
def test_stack48_teacher_forced(M):
    """48-layer MoE-only residual stack h <- bf16(h + moe(h)); each sampled layer is checked
    against the oracle fed with that layer's GPU input (teacher forcing)."""
    wl = syn.WORKLOADS["stack48"]
    L = wl.layers
    rng = np.random.default_rng(M)
    sampled = sorted({0, 23, L - 1} | set(rng.choice(L, 3, replace=False).tolist()))
    h = syn.make_hidden(wl, M=M, seed=0, device=DEV)
    ws = None
    tokens = None if M <= 16 else np.array([0, 5, 31, 63])
    for layer_idx in range(L):
        if layer_idx not in sampled:
            # unsampled layers still run, on the same seeded weights recipe
            pass
        layer = syn.make_layer(wl, layer=layer_idx, seed=0, device=DEV)
        if ws is None:
            ws = moe.alloc_workspace(layer, M, wl.k, wl.b)
        out, ids, wts = moe.moe_decode_block(h, layer, wl.k, wl.b, residual=h, workspace=ws)
        if layer_idx in sampled:
            o_ids, o_wts, _, logits = G.oracle_routing(layer, h, wl.k)
            use_ids, use_wts, _ = G.check_routing(ids.cpu().numpy(), wts.cpu().numpy(), o_ids,
                                                  o_wts, logits, wl.k)
            ref = G.oracle_ffn(layer, h, use_ids, use_wts, residual=h, tokens=tokens)
            got = G.to_f64(out) if tokens is None else G.to_f64(out)[tokens]
            G.assert_close_block(got, ref, "stack layer %d M=%d" % (layer_idx, M))
        del layer
        h = out
    assert moe.moe_read_device_status(ws) == 0


@pytest.mark.parametrize("M", [1, 2, 3, 5, 8])
@pytest.mark.parametrize("b", [1, 8, 64])
def test_decode_block_router_fused_alignment(M, b):
    """M <= 8: the router cluster also aligns the routes; every block size and regime."""
    k, E, H, I = 4, 16, 512, 256
    wl = syn.Workload("fused_%d_%d" % (M, b), H=H, I=I, E=E, k=k, b=b, M=M, router_bias=True)
    layer = syn.make_layer(wl, seed=M + b, device=DEV)
    h = syn.make_hidden(wl, seed=M + b, device=DEV)
    res = syn.make_hidden(wl, seed=7, device=DEV, tag="res")
    ws = moe.alloc_workspace(layer, M, k, b)
    out, ids, wts = moe.moe_decode_block(h, layer, k, b, residual=res, workspace=ws)
    assert moe.moe_read_device_status(ws) == 0
    o_ids, o_wts, _, logits = G.oracle_routing(layer, h, k)
    use_ids, use_wts, _ = G.check_routing(ids.cpu().numpy(), wts.cpu().numpy(), o_ids, o_wts,
                                          logits, k)
    ref = G.oracle_ffn(layer, h, use_ids, use_wts, residual=res)
    G.assert_close_block(G.to_f64(out), ref, "fused alignment M=%d b=%d" % (M, b))
    # the same routes through the stand-alone alignment give the same bits
    out2 = moe.moe_expert_ffn(h, layer, ids, wts, b, residual=res)
    assert torch.equal(out, out2)
