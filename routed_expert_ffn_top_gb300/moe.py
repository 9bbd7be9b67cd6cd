"""Thin ctypes binding of the C ABI in ``include/moe.h`` (argument marshalling only).

Every function here has the name of the C entry point it calls and does no arithmetic of
its own: it checks dtypes/devices/contiguity of torch tensors, allocates outputs the
caller did not pass, hands raw device pointers and the current CUDA stream to the library,
and raises :class:`MoeError` on a non-zero status.  The library must have been built
(``python -m routed_expert_ffn_top_gb300.build`` or ``__graft_entry__.build()``); there is
no fallback of any kind when it is missing.
"""
from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional

import torch

from . import build as _build

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED = 2
MOE_ERR_WORKSPACE = 3
MOE_ERR_CUDA = 4
MOE_ERR_DEVICE = 5

MOE_DEV_INVALID_EXPERT = 0x1
MOE_DEV_WAIT_TIMEOUT = 0x2
MOE_DEV_BAD_ALIGNMENT = 0x4

MOE_W_DENSE_BF16 = 0
MOE_W_VQ_GATEUP = 1
MOE_W_VQLR_GATEUP = 2

# Every symbol include/moe.h declares (checked against the header by the tests).
EXPORTS = (
    "moe_status_string", "moe_route_topk", "moe_align_capacity", "moe_align_block_size",
    "moe_workspace_bytes", "moe_expert_ffn", "moe_decode_block", "moe_decode_block_host",
    "moe_read_device_status", "moe_set_trace_events", "moe_decode_block_noalloc",
    "moe_selftest_wait_timeout", "moe_reader_build", "moe_reader_workspace_bytes",
    "moe_reader_ffn", "moe_library_block_size", "moe_workspace_layout",
)


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, moe_status_string(status), status))


class ExpertWeights(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int32), ("H", ctypes.c_int32), ("I", ctypes.c_int32),
        ("E", ctypes.c_int32),
        ("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p),
        ("j_gate", ctypes.c_void_p), ("j_up", ctypes.c_void_p),
        ("cb_gate", ctypes.c_void_p), ("cb_up", ctypes.c_void_p),
        ("d", ctypes.c_int32), ("K", ctypes.c_int32),
        ("w_down", ctypes.c_void_p),
        ("d_gate", ctypes.c_void_p), ("d_up", ctypes.c_void_p),
        ("c_gate", ctypes.c_void_p), ("c_up", ctypes.c_void_p),
        ("r", ctypes.c_int32),
        ("vq_form", ctypes.c_int32),
    ]


class WorkspaceLayout(ctypes.Structure):
    _fields_ = [
        ("b", ctypes.c_int32), ("kn", ctypes.c_int32), ("cap", ctypes.c_int64),
        ("status", ctypes.c_size_t), ("sorted_route_ids", ctypes.c_size_t),
        ("expert_block_ids", ctypes.c_size_t), ("num_padded", ctypes.c_size_t),
        ("y", ctypes.c_size_t), ("p_tiles", ctypes.c_size_t),
        ("tpb", ctypes.c_int32), ("zero_bytes", ctypes.c_int32),
        ("launches", ctypes.c_int32), ("reserved", ctypes.c_int32),
        ("p_rows", ctypes.c_size_t),
    ]


class ReaderStruct(ctypes.Structure):
    _fields_ = [
        ("H", ctypes.c_int32), ("I", ctypes.c_int32), ("E", ctypes.c_int32),
        ("rank", ctypes.c_int32),
        ("signs", ctypes.c_void_p), ("g_rows", ctypes.c_void_p), ("v_rows", ctypes.c_void_p),
        ("w_down", ctypes.c_void_p), ("g_codes", ctypes.c_void_p), ("v_codes", ctypes.c_void_p),
        ("g_scales", ctypes.c_void_p), ("v_scales", ctypes.c_void_p), ("dnorm", ctypes.c_void_p),
        ("U", ctypes.c_void_p), ("coef", ctypes.c_void_p),
    ]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def lib():
    """The loaded CDLL (raises if the library has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    "CUDA library %s is missing: build it with "
                    "`python -m routed_expert_ffn_top_gb300.build`" % path)
            L = ctypes.CDLL(path)
            vp, ci, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            wp = ctypes.POINTER(ExpertWeights)
            L.moe_status_string.argtypes = [ci]
            L.moe_status_string.restype = ctypes.c_char_p
            L.moe_route_topk.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, vp, vp, vp]
            L.moe_align_capacity.argtypes = [ci, ci, ci, ci]
            L.moe_align_capacity.restype = sz
            L.moe_align_block_size.argtypes = [vp, ci, ci, ci, ci, vp, vp, vp, sz, vp]
            L.moe_workspace_bytes.argtypes = [wp, ci, ci, ci]
            L.moe_workspace_bytes.restype = sz
            L.moe_library_block_size.argtypes = [wp, ci, ci, ci]
            L.moe_library_block_size.restype = ci
            L.moe_workspace_layout.argtypes = [wp, ci, ci, ci, ctypes.POINTER(WorkspaceLayout)]
            L.moe_expert_ffn.argtypes = [vp, wp, ci, ci, vp, vp, vp, vp, vp, ci, vp, vp, vp, sz, vp]
            L.moe_decode_block.argtypes = [vp, vp, vp, wp, ci, ci, ci, vp, vp, vp, vp, vp, sz, vp]
            L.moe_decode_block_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, wp, ci, ci, ci,
                                                vp, vp, vp, sz, vp]
            L.moe_read_device_status.argtypes = [vp, vp, vp]
            L.moe_set_trace_events.argtypes = [vp, ci]
            L.moe_decode_block_noalloc.argtypes = [vp, vp, vp, wp, ci, ci, ci, vp, vp, vp, vp, vp]
            L.moe_selftest_wait_timeout.argtypes = [vp, sz, vp]
            rp = ctypes.POINTER(ReaderStruct)
            L.moe_reader_build.argtypes = [wp, rp, vp]
            L.moe_reader_workspace_bytes.argtypes = [rp, ci, ci, ci]
            L.moe_reader_workspace_bytes.restype = sz
            L.moe_reader_ffn.argtypes = [vp, rp, ci, ci, vp, vp, ci, ci, vp, vp, vp, vp, vp, sz, vp]
            for f in ("moe_route_topk", "moe_align_block_size", "moe_expert_ffn",
                      "moe_decode_block", "moe_decode_block_host", "moe_read_device_status",
                      "moe_set_trace_events", "moe_decode_block_noalloc",
                      "moe_selftest_wait_timeout", "moe_reader_build", "moe_reader_ffn"):
                getattr(L, f).restype = ci
            _lib = L
    return _lib


# ----------------------------------------------------------------------------- marshalling
def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        stream = stream.cuda_stream
    return ctypes.c_void_p(int(stream))


def _need(t, dtype, name, device=None):
    if t is None:
        raise ValueError("%s is required" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if device is not None and t.device != device:
        raise ValueError("%s must be on %s, got %s" % (name, device, t.device))
    return t


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def moe_status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def expert_weights(layer: dict) -> ExpertWeights:
    """C weight descriptor for a layer dict (as made by :mod:`.synthetic`).

    The descriptor holds raw pointers; the caller keeps ``layer``'s tensors alive.
    """
    w = ExpertWeights()
    w.kind = int(layer.get("kind", MOE_W_DENSE_BF16))
    w.H, w.I, w.E = int(layer["H"]), int(layer["I"]), int(layer["E"])
    w.d, w.K = int(layer.get("d", 0) or 0), int(layer.get("K", 0) or 0)
    w.vq_form = int(layer.get("vq_form", 0) or 0)
    dev = layer["w_down"].device
    _need(layer["w_down"], torch.bfloat16, "w_down", dev)
    w.w_down = layer["w_down"].data_ptr()
    if w.kind == MOE_W_DENSE_BF16:
        w.w_gate = _need(layer["w_gate"], torch.bfloat16, "w_gate", dev).data_ptr()
        w.w_up = _need(layer["w_up"], torch.bfloat16, "w_up", dev).data_ptr()
    else:
        w.j_gate = _need(layer["j_gate"], torch.uint8, "j_gate", dev).data_ptr()
        w.j_up = _need(layer["j_up"], torch.uint8, "j_up", dev).data_ptr()
        w.cb_gate = _need(layer["cb_gate"], torch.bfloat16, "cb_gate", dev).data_ptr()
        w.cb_up = _need(layer["cb_up"], torch.bfloat16, "cb_up", dev).data_ptr()
    if w.kind == MOE_W_VQLR_GATEUP:
        w.r = int(layer["r"])
        w.d_gate = _need(layer["d_gate"], torch.bfloat16, "d_gate", dev).data_ptr()
        w.d_up = _need(layer["d_up"], torch.bfloat16, "d_up", dev).data_ptr()
        w.c_gate = _need(layer["c_gate"], torch.bfloat16, "c_gate", dev).data_ptr()
        w.c_up = _need(layer["c_up"], torch.bfloat16, "c_up", dev).data_ptr()
    return w


# ------------------------------------------------------------------------------ entry points
def moe_route_topk(h, w_router, bias, k, renormalize=True, topk_ids=None, topk_weights=None,
                   stream=None):
    dev = h.device
    _need(h, torch.bfloat16, "h", dev)
    _need(w_router, torch.bfloat16, "w_router", dev)
    if bias is not None:
        _need(bias, torch.float32, "bias", dev)
    M, H = h.shape
    E = w_router.shape[1]
    if topk_ids is None:
        topk_ids = torch.empty((M, k), dtype=torch.int32, device=dev)
    if topk_weights is None:
        topk_weights = torch.empty((M, k), dtype=torch.float32, device=dev)
    _need(topk_ids, torch.int32, "topk_ids", dev)
    _need(topk_weights, torch.float32, "topk_weights", dev)
    _check(lib().moe_route_topk(_ptr(h), _ptr(w_router), _ptr(bias), M, H, E, k,
                                int(bool(renormalize)), _ptr(topk_ids), _ptr(topk_weights),
                                _stream(stream)), "moe_route_topk")
    return topk_ids, topk_weights


def moe_align_capacity(M, k, E, b) -> int:
    return int(lib().moe_align_capacity(M, k, E, b))


def moe_align_block_size(topk_ids, E, b, sorted_route_ids=None, expert_block_ids=None,
                         num_padded=None, stream=None):
    dev = topk_ids.device
    _need(topk_ids, torch.int32, "topk_ids", dev)
    M, k = topk_ids.shape
    cap = moe_align_capacity(M, k, E, b)
    if sorted_route_ids is None:
        sorted_route_ids = torch.empty((cap,), dtype=torch.int32, device=dev)
    if expert_block_ids is None:
        expert_block_ids = torch.empty((max(cap // b, 1),), dtype=torch.int32, device=dev)
    if num_padded is None:
        num_padded = torch.empty((1,), dtype=torch.int32, device=dev)
    _need(sorted_route_ids, torch.int32, "sorted_route_ids", dev)
    _need(expert_block_ids, torch.int32, "expert_block_ids", dev)
    _need(num_padded, torch.int32, "num_padded", dev)
    if expert_block_ids.numel() < sorted_route_ids.numel() // b:
        raise ValueError("expert_block_ids must hold cap // b entries")
    _check(lib().moe_align_block_size(_ptr(topk_ids), M, k, E, b, _ptr(sorted_route_ids),
                                      _ptr(expert_block_ids), _ptr(num_padded),
                                      sorted_route_ids.numel(), _stream(stream)),
           "moe_align_block_size")
    return sorted_route_ids, expert_block_ids, num_padded


def moe_workspace_bytes(layer: dict, M, k, b) -> int:
    w = expert_weights(layer)
    return int(lib().moe_workspace_bytes(ctypes.byref(w), M, k, b))


def moe_library_block_size(layer: dict, M, k, b) -> int:
    """The block size moe_decode_block aligns with for these weights and sizes."""
    w = expert_weights(layer)
    return int(lib().moe_library_block_size(ctypes.byref(w), M, k, b))


def moe_workspace_layout(layer: dict, M, k, b) -> dict:
    """Block size, capacity and byte offsets of the alignment inside the workspace of
    moe_decode_block / moe_expert_ffn (library alignment) for these sizes."""
    w = expert_weights(layer)
    out = WorkspaceLayout()
    _check(lib().moe_workspace_layout(ctypes.byref(w), M, k, b, ctypes.byref(out)),
           "moe_workspace_layout")
    return {f: int(getattr(out, f)) for f, _ in WorkspaceLayout._fields_ if f != "reserved"}


def workspace_alignment(workspace: torch.Tensor, layout: dict):
    """Views (sorted_route_ids, expert_block_ids, num_padded) of the alignment a call left in
    `workspace`, at the offsets of `layout` (moe_workspace_layout)."""
    cap, b = layout["cap"], layout["b"]

    def view(off, n):
        return workspace[off:off + 4 * n].view(torch.int32)

    return (view(layout["sorted_route_ids"], cap), view(layout["expert_block_ids"], cap // b),
            view(layout["num_padded"], 1))


def alloc_workspace(layer: dict, M, k, b, device=None) -> torch.Tensor:
    """A zero-filled workspace of the size the library asks for (256-byte aligned)."""
    n = moe_workspace_bytes(layer, M, k, b)
    if n == 0:
        raise MoeError(MOE_ERR_UNSUPPORTED, "moe_workspace_bytes")
    device = layer["w_down"].device if device is None else device
    return torch.zeros((n,), dtype=torch.uint8, device=device)


def moe_expert_ffn(h, layer, topk_ids, topk_weights, b, alignment=None, residual=None,
                   out=None, workspace=None, stream=None):
    dev = h.device
    _need(h, torch.bfloat16, "h", dev)
    _need(topk_ids, torch.int32, "topk_ids", dev)
    _need(topk_weights, torch.float32, "topk_weights", dev)
    M, k = topk_ids.shape
    w = expert_weights(layer)
    if residual is not None:
        _need(residual, torch.bfloat16, "residual", dev)
    if out is None:
        out = torch.empty((M, w.H), dtype=torch.bfloat16, device=dev)
    _need(out, torch.bfloat16, "out", dev)
    if workspace is None:
        workspace = alloc_workspace(layer, M, k, b, dev)
    srt = blk = npad = None
    if alignment is not None:
        srt, blk, npad = alignment
    _check(lib().moe_expert_ffn(_ptr(h), ctypes.byref(w), M, k, _ptr(topk_ids),
                                _ptr(topk_weights), _ptr(srt), _ptr(blk), _ptr(npad), b,
                                _ptr(residual), _ptr(out), _ptr(workspace), workspace.numel(),
                                _stream(stream)), "moe_expert_ffn")
    return out


def moe_decode_block(h, layer, k, b, residual=None, out=None, topk_ids=None, topk_weights=None,
                     workspace=None, stream=None):
    dev = h.device
    _need(h, torch.bfloat16, "h", dev)
    M = h.shape[0]
    w = expert_weights(layer)
    w_router = _need(layer["w_router"], torch.bfloat16, "w_router", dev)
    bias = layer.get("bias")
    if bias is not None:
        _need(bias, torch.float32, "bias", dev)
    if residual is not None:
        _need(residual, torch.bfloat16, "residual", dev)
    if out is None:
        out = torch.empty((M, w.H), dtype=torch.bfloat16, device=dev)
    if topk_ids is None:
        topk_ids = torch.empty((M, k), dtype=torch.int32, device=dev)
    if topk_weights is None:
        topk_weights = torch.empty((M, k), dtype=torch.float32, device=dev)
    if workspace is None:
        workspace = alloc_workspace(layer, M, k, b, dev)
    _need(out, torch.bfloat16, "out", dev)
    _need(topk_ids, torch.int32, "topk_ids", dev)
    _need(topk_weights, torch.float32, "topk_weights", dev)
    _check(lib().moe_decode_block(_ptr(h), _ptr(w_router), _ptr(bias), ctypes.byref(w), M, k, b,
                                  _ptr(residual), _ptr(out), _ptr(topk_ids), _ptr(topk_weights),
                                  _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_decode_block")
    return out, topk_ids, topk_weights


def moe_decode_block_noalloc(h, layer, k, b, residual=None, out=None, topk_ids=None,
                             topk_weights=None, stream=None):
    """moe_decode_block without a workspace: for callers that cannot allocate device memory,
    the library runs the block on its own fixed scratch array (see include/moe.h).  Outputs
    the caller does not pass are allocated here by torch, as for the other wrappers."""
    dev = h.device
    _need(h, torch.bfloat16, "h", dev)
    M = h.shape[0]
    w = expert_weights(layer)
    w_router = _need(layer["w_router"], torch.bfloat16, "w_router", dev)
    bias = layer.get("bias")
    if bias is not None:
        _need(bias, torch.float32, "bias", dev)
    if residual is not None:
        _need(residual, torch.bfloat16, "residual", dev)
    if out is None:
        out = torch.empty((M, w.H), dtype=torch.bfloat16, device=dev)
    if topk_ids is None:
        topk_ids = torch.empty((M, k), dtype=torch.int32, device=dev)
    if topk_weights is None:
        topk_weights = torch.empty((M, k), dtype=torch.float32, device=dev)
    _need(out, torch.bfloat16, "out", dev)
    _need(topk_ids, torch.int32, "topk_ids", dev)
    _need(topk_weights, torch.float32, "topk_weights", dev)
    _check(lib().moe_decode_block_noalloc(_ptr(h), _ptr(w_router), _ptr(bias), ctypes.byref(w),
                                          M, k, b, _ptr(residual), _ptr(out), _ptr(topk_ids),
                                          _ptr(topk_weights), _stream(stream)),
           "moe_decode_block_noalloc")
    return out, topk_ids, topk_weights


def moe_decode_block_host(h_host, layer, k, b, h_dev, out_dev, out_host, topk_ids, topk_weights,
                          workspace, residual_host=None, residual_dev=None, stream=None):
    """Host in, host out: the library copies h to the device and the result back, and
    synchronises the stream before returning."""
    w = expert_weights(layer)
    bias = layer.get("bias")
    M = h_host.shape[0]
    _check(lib().moe_decode_block_host(_ptr(h_host), _ptr(residual_host), _ptr(out_host),
                                       _ptr(h_dev), _ptr(residual_dev), _ptr(out_dev),
                                       _ptr(layer["w_router"]), _ptr(bias), ctypes.byref(w), M, k,
                                       b, _ptr(topk_ids), _ptr(topk_weights), _ptr(workspace),
                                       workspace.numel(), _stream(stream)),
           "moe_decode_block_host")
    return out_host


def moe_read_device_status(workspace, stream=None) -> int:
    """Synchronises the stream, returns the device status bits and clears them."""
    out = ctypes.c_int32(0)
    rc = lib().moe_read_device_status(_ptr(workspace), _stream(stream), ctypes.byref(out))
    if rc not in (MOE_OK, MOE_ERR_DEVICE):
        raise MoeError(rc, "moe_read_device_status")
    return int(out.value)


def moe_selftest_wait_timeout(workspace, stream=None):
    """Enqueue the failure-detection self-test (include/moe.h): one CTA whose bounded wait
    runs out after about a second and sets MOE_DEV_WAIT_TIMEOUT in the workspace's status."""
    _check(lib().moe_selftest_wait_timeout(_ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_selftest_wait_timeout")


def moe_set_trace_events(events=None):
    """Record the given six torch.cuda.Event objects around the block's kernels on every
    later call from this thread (see include/moe.h); ``None`` stops tracing."""
    if events is None:
        _check(lib().moe_set_trace_events(None, 0), "moe_set_trace_events")
        return
    events = list(events)
    for e in events:  # torch creates the CUDA event lazily, on first record
        if e.cuda_event == 0:
            e.record()
    arr = (ctypes.c_void_p * len(events))(*[e.cuda_event for e in events])
    _check(lib().moe_set_trace_events(arr, len(events)), "moe_set_trace_events")


# ------------------------------------------------------------------------------ CUDA graphs
def capture_graph(fn, stream: Optional[torch.cuda.Stream] = None) -> torch.cuda.CUDAGraph:
    """Capture ``fn(stream)`` -- one or more calls of the entry points above on ``stream`` --
    into a CUDA graph, after one eager run of it on the same stream.

    Decoding repeats the same block shapes step after step.  Replaying the captured
    launches (programmatic dependent launches included) skips the per-call host work:
    argument checks, marshalling, tensor-map encoding and one launch per kernel.  At small
    M that host work takes longer than the block's GPU time.  The graph keeps the raw
    pointers of the tensors ``fn`` used: a replay reads the inputs that are in those same
    tensors at that time and writes the same outputs.  Its workspace must not be shared
    with calls that run at the same time.
    """
    if stream is None:
        stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):
        fn(stream)  # eager run: one-time kernel attributes are set outside the capture
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        fn(stream)
    torch.cuda.current_stream().wait_stream(stream)
    return graph


# ------------------------------------------------------------------------ channel reader
def _reader_struct(rd: dict) -> ReaderStruct:
    s = ReaderStruct()
    s.H, s.I, s.E, s.rank = rd["H"], rd["I"], rd["E"], rd["rank"]
    for name in ("signs", "g_rows", "v_rows", "w_down", "g_codes", "v_codes", "g_scales",
                 "v_scales", "dnorm", "U", "coef"):
        setattr(s, name, rd[name].data_ptr())
    return s


def reader_build(layer: dict, signs: torch.Tensor, U: torch.Tensor, stream=None) -> dict:
    """Allocate and build the reader's data for a dense layer (see include/moe.h)."""
    E, H, I = layer["E"], layer["H"], layer["I"]
    rank = U.shape[1]
    dev = layer["w_down"].device
    nb = H // 128
    rd = {"H": H, "I": I, "E": E, "rank": rank, "signs": signs.contiguous(),
          "U": U.to(torch.float32).contiguous(), "w_down": layer["w_down"],
          "g_rows": torch.empty((E, I, H), dtype=torch.bfloat16, device=dev),
          "v_rows": torch.empty((E, I, H), dtype=torch.bfloat16, device=dev),
          "g_codes": torch.empty((E, I, nb, 8), dtype=torch.int32, device=dev),
          "v_codes": torch.empty((E, I, nb, 8), dtype=torch.int32, device=dev),
          "g_scales": torch.empty((E, I, nb), dtype=torch.float32, device=dev),
          "v_scales": torch.empty((E, I, nb), dtype=torch.float32, device=dev),
          "dnorm": torch.empty((E, I), dtype=torch.float32, device=dev),
          "coef": torch.empty((E, I, rank), dtype=torch.bfloat16, device=dev)}
    w = expert_weights(layer)
    s = _reader_struct(rd)
    _check(lib().moe_reader_build(ctypes.byref(w), ctypes.byref(s), _stream(stream)),
           "moe_reader_build")
    return rd


def reader_workspace(rd: dict, M: int, k: int, K: int, device=None) -> torch.Tensor:
    s = _reader_struct(rd)
    n = lib().moe_reader_workspace_bytes(ctypes.byref(s), M, k, K)
    if n == 0:
        raise MoeError(MOE_ERR_UNSUPPORTED, "moe_reader_workspace_bytes")
    return torch.zeros((n,), dtype=torch.uint8, device=rd["w_down"].device if device is None else device)


def moe_reader_ffn(h, rd: dict, topk_ids, topk_weights, K: int, nscan: int = 80, residual=None,
                   out=None, workspace=None, want_decisions=False, stream=None):
    """The reader's decode (include/moe.h).  Returns out, or (out, selected [M,K] int32,
    xr [M,H] fp32) with ``want_decisions``."""
    M, k = topk_ids.shape
    if out is None:
        out = torch.empty_like(h)
    if workspace is None:
        workspace = reader_workspace(rd, M, k, K)
    sel = xr = None
    if want_decisions:
        sel = torch.empty((M, max(K, 1)), dtype=torch.int32, device=h.device)
        xr = torch.empty((M, rd["H"]), dtype=torch.float32, device=h.device)
    s = _reader_struct(rd)
    _check(lib().moe_reader_ffn(_ptr(h), ctypes.byref(s), M, k, _ptr(topk_ids), _ptr(topk_weights),
                                K, nscan, _ptr(residual), _ptr(out), _ptr(sel), _ptr(xr),
                                _ptr(workspace), workspace.numel(), _stream(stream)),
           "moe_reader_ffn")
    if want_decisions:
        return out, sel[:, :K], xr
    return out
