"""CUDA-graph replay of the decode block: the captured launches (programmatic dependent
launches and clusters included) give the same bits as direct calls, and a replay reads the
inputs present in the captured tensors at replay time."""
import numpy as np
import pytest
import torch

import gpu_ref as G
from routed_expert_ffn_top_gb300 import moe, synthetic as syn

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as entry
    entry.build()
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("M,k,E,H,I,b", [
    (1, 8, 128, 2048, 768, 8),     # router with fused alignment and row tiles, 16-row tiles
    (21, 8, 128, 2048, 768, 8),    # separate alignment and row gather launches
    (96, 4, 16, 512, 512, 64),     # 64-row tiles
])
def test_graph_replay_bitwise(M, k, E, H, I, b):
    wl = syn.Workload("graph_%d_%d" % (M, b), H=H, I=I, E=E, k=k, b=b, M=M)
    layer = syn.make_layer(wl, seed=2, device=DEV)
    h = syn.make_hidden(wl, seed=2, device=DEV)
    res = syn.make_hidden(wl, seed=3, device=DEV, tag="res")
    ws = moe.alloc_workspace(layer, M, k, b)
    ref_out, ref_ids, ref_wts = moe.moe_decode_block(h, layer, k, b, residual=res, workspace=ws)
    torch.cuda.synchronize()

    out = torch.empty_like(ref_out)
    ids = torch.empty_like(ref_ids)
    wts = torch.empty_like(ref_wts)
    x = h.clone()
    g = moe.capture_graph(lambda s: moe.moe_decode_block(
        x, layer, k, b, residual=res, out=out, topk_ids=ids, topk_weights=wts, workspace=ws,
        stream=s))
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref_out) and torch.equal(ids, ref_ids) and torch.equal(wts, ref_wts)
    assert moe.moe_read_device_status(ws) == 0

    # new input written into the captured tensor: the replay follows it
    h2 = syn.make_hidden(wl, seed=9, device=DEV)
    x.copy_(h2)
    g.replay()
    torch.cuda.synchronize()
    ref2, ids2, wts2 = moe.moe_decode_block(h2, layer, k, b, residual=res, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(out, ref2) and torch.equal(ids, ids2) and torch.equal(wts, wts2)

    # and it is right, not just repeatable
    o_ids, o_wts, _, logits = G.oracle_routing(layer, h2, k)
    use_ids, use_wts, _ = G.check_routing(ids.cpu().numpy(), wts.cpu().numpy(), o_ids, o_wts,
                                          logits, k)
    tokens = None if M <= 32 else np.array([0, 1, M // 2, M - 1])
    ref = G.oracle_ffn(layer, h2, use_ids, use_wts, residual=res, tokens=tokens)
    got = G.to_f64(out) if tokens is None else G.to_f64(out)[tokens]
    G.assert_close_block(got, ref, "graph replay")
