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
        assert torch.equal(ids, ref_ids) and torch.equal(wts, ref_wts), call
        assert torch.equal(out, ref), call
        # the library's own block size (b = 0: 16-row blocks here) gives the same bits: dense
        # weights give every route the same bits whatever its block
        out0, _, _ = moe.moe_decode_block_noalloc(h, layer, wl.k, 0)
        assert torch.equal(out0, ref), call


def test_noalloc_refuses_sizes_beyond_its_array():
    dev = torch.device("cuda:0")
    wl = syn.WORKLOADS["layer_m21"]
    layer = syn.make_layer(wl, seed=11, device=dev)
    h = syn.make_hidden(wl, M=256, seed=1, device=dev)
    with pytest.raises(moe.MoeError) as err:
        moe.moe_decode_block_noalloc(h, layer, wl.k, wl.b)
    assert err.value.status == moe.MOE_ERR_WORKSPACE


def test_noalloc_keeps_no_state_between_calls_of_other_shapes():
    """The array keeps whatever the previous call left.  A smaller call after a larger one
    (M=21, then M=1 through the router's own alignment), and a VQ call (code books in shared
    memory, fp32 p and the sub-block table) after a dense one, each give the bits of
    moe_decode_block on a fresh zero-filled workspace with the same b."""
    dev = torch.device("cuda:0")
    wl = syn.WORKLOADS["layer_m21"]
    layer = syn.make_layer(wl, seed=13, device=dev)
    vq_wl = syn.workload("vq_d4", M=4)
    vq_layer = syn.make_layer(vq_wl, seed=13, device=dev)
    cases = [(layer, wl, 21, 31), (layer, wl, 1, 32), (vq_layer, vq_wl, 4, 33),
             (layer, wl, 2, 34)]
    for layer_i, wl_i, M, seed in cases:
        h = syn.make_hidden(wl_i, M=M, seed=seed, device=dev)
        ws = moe.alloc_workspace(layer_i, M, wl_i.k, wl_i.b)  # fresh, zero-filled
        ref, ref_ids, ref_wts = moe.moe_decode_block(h, layer_i, wl_i.k, wl_i.b, workspace=ws)
        out, ids, wts = moe.moe_decode_block_noalloc(h, layer_i, wl_i.k, wl_i.b)
        torch.cuda.synchronize()
        assert torch.equal(ids, ref_ids) and torch.equal(wts, ref_wts), (wl_i.name, M)
        assert torch.equal(out, ref), (wl_i.name, M)
