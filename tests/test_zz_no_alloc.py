"""The allocation-free decode-block entry point (moe_decode_block_noalloc).

Callers that cannot allocate device memory -- a host program whose GPU memory belongs to
another allocator, or a deployment that allows no allocation after start-up -- call this
entry point without a workspace; the library runs the block on a fixed scratch array of
its own.  This file checks it through the C ABI against moe_decode_block with a caller
workspace, on two calls in a row, and that requests larger than the array are refused.
It is collected last so that a failure here never hides the other tests.
"""
import pytest
import torch

import gpu_ref as G
from routed_expert_ffn_top_gb300 import moe, synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__ as entry
    entry.build()


def test_noalloc_matches_workspace_entry_point_on_two_calls():
    dev = torch.device("cuda:0")
    wl = syn.WORKLOADS["layer_m21"]
    layer = syn.make_layer(wl, seed=11, device=dev)
    for call, seed in enumerate((11, 12)):  # two calls in a row, different inputs
        h = syn.make_hidden(wl, seed=seed, device=dev)
        ref, ref_ids, ref_wts = moe.moe_decode_block(h, layer, wl.k, wl.b)
        out, ids, wts = moe.moe_decode_block_noalloc(h, layer, wl.k, wl.b)
        torch.cuda.synchronize()
        assert torch.equal(ids, ref_ids), call
        assert torch.allclose(wts, ref_wts, rtol=1e-6, atol=0), call
        # the caller's 8-row blocks here, the library's 16-row blocks there: dense weights
        # give every route the same bits whatever its block
        assert torch.equal(out, ref), call


def test_noalloc_refuses_sizes_beyond_its_array():
    dev = torch.device("cuda:0")
    wl = syn.WORKLOADS["layer_m21"]
    layer = syn.make_layer(wl, seed=11, device=dev)
    h = syn.make_hidden(wl, M=256, seed=1, device=dev)
    with pytest.raises(moe.MoeError) as err:
        moe.moe_decode_block_noalloc(h, layer, wl.k, wl.b)
    assert err.value.status == moe.MOE_ERR_WORKSPACE
