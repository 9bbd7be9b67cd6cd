"""Failure detection on the GPU without a fault: a bounded device wait that nothing
completes gives up after about a second, reports MOE_DEV_WAIT_TIMEOUT through the status
word, and leaves the context usable for the next decode block."""
import time

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


def test_bounded_wait_gives_up_and_the_context_survives():
    wl = syn.Workload(name="failure_small", M=3, H=256, I=256, E=16, k=4, b=8)
    layer = syn.make_layer(wl, layer=0, seed=11, device=DEV)
    h = syn.make_hidden(wl, seed=11, device=DEV)
    ws = moe.alloc_workspace(layer, wl.M, wl.k, wl.b)
    assert moe.moe_read_device_status(ws) == 0

    torch.cuda.synchronize()
    t0 = time.perf_counter()
    moe.moe_selftest_wait_timeout(ws)
    st = moe.moe_read_device_status(ws)  # synchronises the stream
    waited = time.perf_counter() - t0
    assert st == moe.MOE_DEV_WAIT_TIMEOUT
    assert 0.9 < waited < 30.0, waited
    assert moe.moe_read_device_status(ws) == 0  # the read cleared the word

    # the same context and workspace still run a block that matches the oracle
    out, ids, wts = moe.moe_decode_block(h, layer, wl.k, wl.b, workspace=ws)
    assert moe.moe_read_device_status(ws) == 0
    o_ids, o_wts, _, logits = G.oracle_routing(layer, h, wl.k)
    use_ids, use_wts, _ = G.check_routing(ids.cpu().numpy(), wts.cpu().numpy(), o_ids, o_wts,
                                          logits, wl.k)
    ref = G.oracle_ffn(layer, h, use_ids, use_wts)
    G.assert_close_block(G.to_f64(out), ref, "after a wait timeout")
