"""The C-ABI library builds, loads and exports what include/moe.h declares; host-side
validation answers without touching a GPU (no compute calls here)."""
import ctypes
import os
import re

import pytest

import __graft_entry__ as entry
from routed_expert_ffn_top_gb300 import moe, synthetic as syn

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "moe.h")


@pytest.fixture(scope="module")
def lib():
    entry.build()
    return moe.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_header_declares_binding_exports():
    assert sorted(moe.EXPORTS) == declared_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    for code in range(6):
        assert moe.moe_status_string(code)
    assert moe.moe_status_string(99) == "unknown status"


def test_align_capacity_host(lib):
    assert moe.moe_align_capacity(21, 8, 128, 8) == 168 + 128 * 7
    assert moe.moe_align_capacity(1, 8, 128, 8) == 8 + 8 * 7
    assert moe.moe_align_capacity(256, 8, 128, 64) == 2048 + 128 * 63
    assert moe.moe_align_capacity(0, 8, 128, 8) == 0
    assert moe.moe_align_capacity(-1, 8, 128, 8) == 0


def _weights(kind=0, H=2048, I=768, E=128):
    w = moe.ExpertWeights()
    w.kind, w.H, w.I, w.E, w.d, w.K = kind, H, I, E, 4, 256
    fake = 1 << 20  # a 16-byte aligned non-null address; never dereferenced by validation
    w.w_gate = w.w_up = w.w_down = fake
    w.j_gate = w.j_up = w.cb_gate = w.cb_up = fake
    return w


def test_workspace_bytes_host(lib):
    for name in ("layer_m1", "layer_m21", "large_m256"):
        wl = syn.WORKLOADS[name]
        w = _weights(H=wl.H, I=wl.I, E=wl.E)
        assert lib.moe_workspace_bytes(ctypes.byref(w), wl.M, wl.k, wl.b) > 0
    w = _weights()
    assert lib.moe_workspace_bytes(ctypes.byref(w), 4, 0, 8) == 0      # k = 0
    assert lib.moe_workspace_bytes(ctypes.byref(w), 4, 8, 12) == 0     # b > 8 not a multiple of 8
    assert lib.moe_workspace_bytes(None, 4, 8, 8) == 0


def test_validation_fails_closed_without_gpu(lib):
    vp = ctypes.c_void_p
    fake = vp(1 << 20)
    ids = vp(1 << 20)
    # unsupported E (not a multiple of 8), k > E, H not a multiple of 128
    assert lib.moe_route_topk(fake, fake, None, 1, 2048, 7, 2, 1, ids, ids, None) == moe.MOE_ERR_UNSUPPORTED
    assert lib.moe_route_topk(fake, fake, None, 1, 2048, 8, 9, 1, ids, ids, None) == moe.MOE_ERR_UNSUPPORTED
    assert lib.moe_route_topk(fake, fake, None, 1, 2000, 8, 2, 1, ids, ids, None) == moe.MOE_ERR_UNSUPPORTED
    # NULL and misaligned pointers
    assert lib.moe_route_topk(None, fake, None, 1, 2048, 128, 8, 1, ids, ids, None) == moe.MOE_ERR_INVALID_ARG
    assert lib.moe_route_topk(vp((1 << 20) + 2), fake, None, 1, 2048, 128, 8, 1, ids, ids, None) == moe.MOE_ERR_INVALID_ARG
    # M == 0 is a no-op
    assert lib.moe_route_topk(None, None, None, 0, 2048, 128, 8, 1, None, None, None) == moe.MOE_OK
    # alignment capacity too small
    assert lib.moe_align_block_size(ids, 21, 8, 128, 8, ids, ids, ids, 100, None) == moe.MOE_ERR_WORKSPACE
    # workspace too small
    w = _weights()
    assert lib.moe_expert_ffn(fake, ctypes.byref(w), 4, 8, ids, ids, None, None, None, 8, None,
                              fake, vp(1 << 20), 16, None) == moe.MOE_ERR_WORKSPACE
    # half-given alignment
    need = lib.moe_workspace_bytes(ctypes.byref(w), 4, 8, 8)
    assert lib.moe_expert_ffn(fake, ctypes.byref(w), 4, 8, ids, ids, ids, None, None, 8, None,
                              fake, vp(1 << 20), need, None) == moe.MOE_ERR_INVALID_ARG
    # VQ with unsupported d (4 and 8 are supported)
    wv = _weights(kind=1)
    wv.d = 2
    assert lib.moe_decode_block(fake, fake, None, ctypes.byref(wv), 1, 8, 8, None, fake, ids, ids,
                                vp(1 << 20), 1 << 30, None) == moe.MOE_ERR_UNSUPPORTED
    # VQ with H not a multiple of 1024 (index boxes cover 1024 rows of H)
    wv = _weights(kind=1, H=1536)
    assert lib.moe_decode_block(fake, fake, None, ctypes.byref(wv), 1, 8, 8, None, fake, ids, ids,
                                vp(1 << 20), 1 << 30, None) == moe.MOE_ERR_UNSUPPORTED
    # dense H, I not multiples of 256
    wd = _weights(H=2048 + 128)
    assert lib.moe_expert_ffn(fake, ctypes.byref(wd), 4, 8, ids, ids, None, None, None, 8, None,
                              fake, vp(1 << 20), 1 << 30, None) == moe.MOE_ERR_UNSUPPORTED
    # VQ + low rank: rank not a multiple of 128, rank too large, missing basis
    for r, expect in ((200, moe.MOE_ERR_UNSUPPORTED), (640, moe.MOE_ERR_UNSUPPORTED),
                      (0, moe.MOE_ERR_INVALID_ARG)):
        wl_ = _weights(kind=2)
        wl_.r = r
        wl_.d_gate = wl_.d_up = wl_.c_gate = wl_.c_up = 1 << 20
        assert lib.moe_decode_block(fake, fake, None, ctypes.byref(wl_), 1, 8, 8, None, fake, ids,
                                    ids, vp(1 << 20), 1 << 30, None) == expect, r
    wl_ = _weights(kind=2)
    wl_.r = 256
    wl_.d_gate = wl_.c_gate = wl_.c_up = 1 << 20  # d_up missing
    assert lib.moe_decode_block(fake, fake, None, ctypes.byref(wl_), 1, 8, 8, None, fake, ids, ids,
                                vp(1 << 20), 1 << 30, None) == moe.MOE_ERR_INVALID_ARG
    # the workspace grows by the projections z [M, 2r] fp32
    wl_.d_up = 1 << 20
    wv_ = _weights(kind=1)
    assert (lib.moe_workspace_bytes(ctypes.byref(wl_), 4, 8, 8)
            >= lib.moe_workspace_bytes(ctypes.byref(wv_), 4, 8, 8) + 4 * 2 * 256 * 4)
    # unknown weight kind
    wk = _weights(kind=7)
    assert lib.moe_decode_block(fake, fake, None, ctypes.byref(wk), 1, 8, 8, None, fake, ids, ids,
                                vp(1 << 20), 1 << 30, None) == moe.MOE_ERR_INVALID_ARG


def test_oracle_and_product_are_separate():
    """The product package never imports the oracle (and vice versa)."""
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    pkg = os.path.join(root, "routed_expert_ffn_top_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "moe_oracle" not in text, f
    for f in os.listdir(os.path.join(root, "oracle")):
        if f.endswith((".py", ".c")):
            text = open(os.path.join(root, "oracle", f)).read()
            assert not re.search(r"^\s*(import|from)\s+routed_expert_ffn_top_gb300", text, re.M), f
            assert not re.search(r'#\s*include\s*"moe', text), f


def test_selftest_wait_timeout_validates_before_launch(lib):
    L = moe.lib()
    assert L.moe_selftest_wait_timeout(None, 256, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_selftest_wait_timeout(ctypes.c_void_p((1 << 20) + 16), 256, None) == \
        moe.MOE_ERR_INVALID_ARG  # not 256-byte aligned
    assert L.moe_selftest_wait_timeout(ctypes.c_void_p(1 << 20), 0, None) == \
        moe.MOE_ERR_INVALID_ARG  # no room for the status word


def _reader(H=2048, I=768, E=128, rank=32):
    r = moe.ReaderStruct()
    r.H, r.I, r.E, r.rank = H, I, E, rank
    for name in ("signs", "g_rows", "v_rows", "w_down", "g_codes", "v_codes", "g_scales",
                 "v_scales", "dnorm", "U", "coef"):
        setattr(r, name, 1 << 20)
    return r


def test_reader_validation_without_gpu(lib):
    L = moe.lib()
    r = _reader()
    assert L.moe_reader_workspace_bytes(ctypes.byref(r), 1, 8, 756) > 0
    assert L.moe_reader_workspace_bytes(ctypes.byref(r), 1, 8, 8 * 768 + 1) == 0  # K > k*I
    assert L.moe_reader_workspace_bytes(ctypes.byref(r), 1, 32, 10) == 0  # k*I > 16384
    assert L.moe_reader_workspace_bytes(ctypes.byref(_reader(rank=33)), 1, 8, 10) == 0
    assert L.moe_reader_workspace_bytes(ctypes.byref(_reader(H=2000)), 1, 8, 10) == 0
    bad = _reader()
    bad.U = 0
    assert L.moe_reader_workspace_bytes(ctypes.byref(bad), 1, 8, 10) == 0
    vp = ctypes.c_void_p
    ws = vp(1 << 21)
    # nscan out of range and a too-small workspace fail before any launch
    assert L.moe_reader_ffn(vp(1 << 20), ctypes.byref(r), 1, 8, vp(1 << 20), vp(1 << 20), 10, 129,
                            None, vp(1 << 20), None, None, ws, 1 << 30, None) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_reader_ffn(vp(1 << 20), ctypes.byref(r), 1, 8, vp(1 << 20), vp(1 << 20), 10, 80,
                            None, vp(1 << 20), None, None, ws, 16, None) == moe.MOE_ERR_WORKSPACE
    w = _weights()
    assert L.moe_reader_build(ctypes.byref(w), ctypes.byref(_reader(I=512)), None) == moe.MOE_ERR_INVALID_ARG


def test_library_block_size_without_gpu(lib):
    """The alignment block size of the decode block: the caller's b when b > 0; for b = 0 the
    library's pick -- 8 for VQ forms 0 and 1, for dense weights and VQ form 2 a tile width
    (16 at one token; 64 for VQ form 2 from 16 routes per expert); 0 on invalid arguments."""
    L = moe.lib()
    d = _weights()
    assert L.moe_library_block_size(ctypes.byref(d), 1, 8, 8) == 8  # binding
    assert L.moe_library_block_size(ctypes.byref(d), 4096, 8, 8) == 8
    assert L.moe_library_block_size(ctypes.byref(d), 1, 8, 0) == 16  # the library's pick
    assert L.moe_library_block_size(ctypes.byref(d), 4096, 8, 0) == 64
    assert L.moe_library_block_size(ctypes.byref(d), 1, 8, 12) == 0  # invalid b
    assert L.moe_library_block_size(ctypes.byref(d), 1, 8, -8) == 0
    assert L.moe_library_block_size(None, 1, 8, 8) == 0
    v = _weights(kind=moe.MOE_W_VQ_GATEUP)
    assert L.moe_library_block_size(ctypes.byref(v), 21, 8, 3) == 3
    assert L.moe_library_block_size(ctypes.byref(v), 21, 8, 0) == 8
    v.vq_form = 2
    assert L.moe_library_block_size(ctypes.byref(v), 255, 8, 0) == 16  # 15.9 routes per expert
    assert L.moe_library_block_size(ctypes.byref(v), 256, 8, 0) == 64
    # b = 0: the workspace covers either tile width; b > 0: exactly that b's layout
    assert L.moe_workspace_bytes(ctypes.byref(d), 64, 8, 0) >= max(
        L.moe_workspace_bytes(ctypes.byref(d), 64, 8, 16),
        L.moe_workspace_bytes(ctypes.byref(d), 64, 8, 64))
    assert L.moe_workspace_bytes(ctypes.byref(d), 64, 8, -1) == 0


def test_workspace_layout_without_gpu(lib):
    """moe_workspace_layout: the alignment's place in the workspace, for the resolved b."""
    L = moe.lib()
    d = _weights()
    out = moe.WorkspaceLayout()
    for M, b, want_b in ((1, 8, 8), (21, 0, 16), (4096, 0, 64), (3, 1, 1)):
        assert L.moe_workspace_layout(ctypes.byref(d), M, 8, b, ctypes.byref(out)) == moe.MOE_OK
        assert out.b == want_b
        assert out.cap == L.moe_align_capacity(M, 8, d.E, want_b)
        # 256-byte aligned regions after the status word, each large enough, inside the size
        assert out.status == 0
        assert out.sorted_route_ids % 256 == 0 and out.sorted_route_ids >= 64
        assert out.expert_block_ids >= out.sorted_route_ids + 4 * out.cap
        assert out.num_padded >= out.expert_block_ids + 4 * (out.cap // want_b)
        assert out.num_padded + 4 <= L.moe_workspace_bytes(ctypes.byref(d), M, 8, b)
    assert L.moe_workspace_layout(ctypes.byref(d), 1, 8, 12, ctypes.byref(out)) == moe.MOE_ERR_UNSUPPORTED
    assert L.moe_workspace_layout(None, 1, 8, 8, ctypes.byref(out)) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_workspace_layout(ctypes.byref(d), 1, 8, 8, None) == moe.MOE_ERR_INVALID_ARG


def test_kernel_counts_per_path_without_gpu(lib):
    """moe_workspace_layout's `launches`: the kernels one moe_decode_block call launches, which
    the bench multiplies into its launch count.  Expected per path: dense weights at one or two
    tokens, blocks of at most 16 rows: the whole block in one grid; up to 128 routes: router,
    alignment with the row tiles, the fused expert grid, combine; above: router, alignment,
    row gather, fused grid, combine; one token with 32-row blocks: the router aligns and writes
    the rows itself.  VQ weights with code words of 4 at one or two tokens: one grid; else
    router (aligning at one or two tokens), alignment, gate/up, down, combine."""
    L = moe.lib()
    out = moe.WorkspaceLayout()
    d = _weights()
    for M, b, want in ((1, 8, 1), (2, 16, 1), (3, 16, 4), (16, 16, 4), (21, 8, 5), (256, 64, 5),
                       (1, 32, 3)):
        assert L.moe_workspace_layout(ctypes.byref(d), M, 8, b, ctypes.byref(out)) == moe.MOE_OK
        assert out.launches == want, (M, b, out.launches)
        assert (out.p_rows > 0) == (want == 1), (M, b)  # p rows: the one-grid path's only
    v = _weights(kind=moe.MOE_W_VQ_GATEUP)
    for M, want in ((1, 1), (2, 1), (4, 5), (16, 5)):
        assert L.moe_workspace_layout(ctypes.byref(v), M, 8, 8, ctypes.byref(out)) == moe.MOE_OK
        assert out.launches == want, (M, out.launches)
    v.d = 8  # no one-grid path for code words of 8
    assert L.moe_workspace_layout(ctypes.byref(v), 1, 8, 8, ctypes.byref(out)) == moe.MOE_OK
    assert out.launches == 4


def test_vq_form_validation_without_gpu(lib):
    L = moe.lib()
    w = _weights(kind=moe.MOE_W_VQ_GATEUP)
    w.vq_form = 1
    assert L.moe_workspace_bytes(ctypes.byref(w), 4, 8, 8) > 0
    w.vq_form = 3
    assert L.moe_workspace_bytes(ctypes.byref(w), 4, 8, 8) == 0
    w.vq_form = -1
    assert L.moe_workspace_bytes(ctypes.byref(w), 4, 8, 8) == 0
    # the tensor-core form holds 16-row tiles: x and p tiles but no fp32 p or sub-blocks
    w.vq_form = 0
    smem_form = L.moe_workspace_bytes(ctypes.byref(w), 4, 8, 8)
    w.vq_form = 2
    tc_form = L.moe_workspace_bytes(ctypes.byref(w), 4, 8, 8)
    assert tc_form > 0 and tc_form != smem_form
    assert L.moe_workspace_bytes(ctypes.byref(w), 300, 8, 64) > 0  # any M
    d = _weights()
    for form in (1, 2):  # projected code books and tensor-core decoding are VQ forms only
        d.vq_form = form
        assert L.moe_workspace_bytes(ctypes.byref(d), 4, 8, 8) == 0
    lr = _weights(kind=moe.MOE_W_VQLR_GATEUP)
    lr.vq_form = 2
    assert L.moe_workspace_bytes(ctypes.byref(lr), 4, 8, 8) == 0
