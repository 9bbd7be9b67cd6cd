"""fp64 CPU oracle for the small-batch MoE decode block.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()`` and the
benchmark's ``cpu_baseline`` / ``--impl reference`` legs may import this package.  The
product (``routed_expert_ffn_top_gb300``) never imports it and shares no code with it.

The arithmetic lives in ``moe_oracle.c`` (plain loops, double precision); this module only
compiles it with gcc and marshals numpy arrays into it.  bf16 tensors travel as their
``uint16`` bit patterns.  See ``moe_oracle.c`` for the passages each function follows:

* "A Multi-Engine Dataflow for MoE Decoding on Scratchpad-Based Tensor Accelerators" --
  the MoE block (router, gate/up, activation, down, accumulated summation) and blockwise
  VQ (Section 2.3);
* "Channel Selection for Mixture-of-Experts Decoding Needs No Calibration Data" -- the
  channel view of one expert (Background: Channels and Retention Rules);
* "Route-Block Membership Selects Packed-AWQ Arithmetic" -- route flattening and padded
  expert blocks (Section 2.1), stable (expert, route) construction (Section 5.3).

Parity status: every function is pinned by ``tests/test_oracle_pins.py`` (brute force,
closed forms, textbook reductions, invariants and the alignment arithmetic printed in
Section 2.1 of the route-block page).
"""
from __future__ import annotations

import contextlib
import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libmoe_oracle.so")

W_DENSE = 0
W_VQ = 1
W_VQLR = 2

_lock = threading.RLock()
_lib = None


def build(force: bool = False) -> str:
    """Compile ``moe_oracle.c`` into ``oracle/_build/libmoe_oracle.so`` with gcc."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    # -ffp-contract=off: no fused multiply-add contraction, so the rounding of every
    # product and sum is the one written in the source on every host architecture.
    # -fopenmp: the expert loop may take routes on several threads (each route's arithmetic
    # unchanged; the combine runs afterwards in slot order), so the results do not depend on
    # the thread count; without an OpenMP runtime the same source builds serial.
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", _SRC, "-o", tmp]
    if subprocess.run(base + ["-fopenmp", "-lm"], capture_output=True).returncode != 0:
        subprocess.run(base + ["-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Weights(ctypes.Structure):
    _fields_ = [
        ("kind", ctypes.c_int), ("H", ctypes.c_int), ("I", ctypes.c_int), ("E", ctypes.c_int),
        ("w_gate", ctypes.c_void_p), ("w_up", ctypes.c_void_p),
        ("j_gate", ctypes.c_void_p), ("j_up", ctypes.c_void_p),
        ("cb_gate", ctypes.c_void_p), ("cb_up", ctypes.c_void_p),
        ("d", ctypes.c_int), ("K", ctypes.c_int),
        ("w_down", ctypes.c_void_p),
        ("d_gate", ctypes.c_void_p), ("d_up", ctypes.c_void_p),
        ("c_gate", ctypes.c_void_p), ("c_up", ctypes.c_void_p),
        ("r", ctypes.c_int),
    ]


def load_library(path):
    """Open a compiled oracle library and declare its signatures."""
    lib = ctypes.CDLL(path)
    vp, ci, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    lib.oracle_router_logits.argtypes = [vp, vp, vp, ci, ci, ci, vp]
    lib.oracle_topk_softmax.argtypes = [vp, ci, ci, ci, ci, vp, vp, vp]
    lib.oracle_align.argtypes = [vp, ci, ci, ci, ci, vp, vp, vp, i64]
    lib.oracle_expert_ffn.argtypes = [vp, ctypes.POINTER(_Weights), ci, ci, vp, vp,
                                      vp, vp, vp, vp]
    lib.oracle_decode_block.argtypes = [vp, vp, vp, ctypes.POINTER(_Weights), ci, ci,
                                        ci, vp, vp, vp, vp, vp]
    lib.oracle_set_threads.argtypes = [ci]
    for f in ("oracle_router_logits", "oracle_topk_softmax", "oracle_align",
              "oracle_expert_ffn", "oracle_decode_block", "oracle_set_threads"):
        getattr(lib, f).restype = ctypes.c_int
    return lib


@contextlib.contextmanager
def using_library(path):
    """Route every call in this module through another build of ``moe_oracle.c``.

    The pin tests use it to run the same checks against deliberately broken copies of the
    oracle source and confirm that each planted mistake is caught.
    """
    global _lib
    with _lock:
        saved = _load()
        _lib = load_library(path)
    try:
        yield
    finally:
        with _lock:
            _lib = saved


def _load():
    global _lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            lib = load_library(build())
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _bits(a):
    """bf16 payload as a C-contiguous uint16 array (accepts uint16/int16 numpy arrays)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.int16:
        a = a.view(np.uint16)
    if a.dtype != np.uint16:
        raise TypeError("bf16 arrays are passed as uint16 bit patterns, got %s" % a.dtype)
    return a


def _check(rc, what):
    if rc != 0:
        raise RuntimeError("%s failed with oracle status %d" % (what, rc))


def set_threads(n: int) -> int:
    """Threads the expert loop uses (whole tokens per thread; results do not depend on it).
    n <= 0 only reports the count.  Returns the count in effect (1 without OpenMP)."""
    return int(_load().oracle_set_threads(int(n)))


def router_logits(h, w_router, bias, M, H, E):
    """logits [M,E] float64 = h W_r (+ bias)."""
    h, w_router = _bits(h), _bits(w_router)
    bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    out = np.zeros((M, E), dtype=np.float64)
    _check(_load().oracle_router_logits(_ptr(h), _ptr(w_router), _ptr(bias), M, H, E,
                                        _ptr(out)), "oracle_router_logits")
    return out


def topk_softmax(logits, k, renormalize=True):
    """(topk_ids int32 [M,k], topk_weights float64 [M,k], gap float64 [M])."""
    logits = np.ascontiguousarray(logits, dtype=np.float64)
    M, E = logits.shape
    ids = np.zeros((M, k), dtype=np.int32)
    wts = np.zeros((M, k), dtype=np.float64)
    gap = np.zeros((M,), dtype=np.float64)
    _check(_load().oracle_topk_softmax(_ptr(logits), M, E, k, int(bool(renormalize)),
                                       _ptr(ids), _ptr(wts), _ptr(gap)), "oracle_topk_softmax")
    return ids, wts, gap


def align_capacity(M, k, E, b):
    """Rows needed in the worst case: every valid route plus b-1 padding rows per expert."""
    R = M * k
    return R + min(E, R) * (b - 1)


def align(topk_ids, E, b, cap=None):
    """(sorted_route_ids [cap], expert_block_ids [cap//b], num_padded)."""
    topk_ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    M, k = topk_ids.shape
    if cap is None:
        cap = align_capacity(M, k, E, b)
    srt = np.zeros((cap,), dtype=np.int32)
    blk = np.zeros((max(cap // b, 0),), dtype=np.int32)
    npad = np.zeros((1,), dtype=np.int32)
    _check(_load().oracle_align(_ptr(topk_ids), M, k, E, b, _ptr(srt),
                                _ptr(blk) if blk.size else None, _ptr(npad), cap),
           "oracle_align")
    return srt, blk, int(npad[0])


def _weights_struct(w, keep):
    """Build the C weights struct from a dict of numpy arrays; ``keep`` pins buffers."""
    kind = w.get("kind", W_DENSE)
    s = _Weights()
    s.kind, s.H, s.I, s.E = kind, w["H"], w["I"], w["E"]
    s.d, s.K = w.get("d", 0), w.get("K", 0)

    def put(name, arr, conv):
        if arr is None:
            return None
        arr = conv(arr)
        keep.append(arr)
        return arr.ctypes.data

    s.w_gate = put("w_gate", w.get("w_gate"), _bits)
    s.w_up = put("w_up", w.get("w_up"), _bits)
    s.j_gate = put("j_gate", w.get("j_gate"), lambda a: np.ascontiguousarray(a, dtype=np.uint8))
    s.j_up = put("j_up", w.get("j_up"), lambda a: np.ascontiguousarray(a, dtype=np.uint8))
    s.cb_gate = put("cb_gate", w.get("cb_gate"), _bits)
    s.cb_up = put("cb_up", w.get("cb_up"), _bits)
    s.w_down = put("w_down", w.get("w_down"), _bits)
    s.d_gate = put("d_gate", w.get("d_gate"), _bits)
    s.d_up = put("d_up", w.get("d_up"), _bits)
    s.c_gate = put("c_gate", w.get("c_gate"), _bits)
    s.c_up = put("c_up", w.get("c_up"), _bits)
    s.r = w.get("r", 0) or 0
    return s


def expert_ffn(h, weights, topk_ids, topk_weights, residual=None, want_intermediates=False):
    """out [M,H] float64 (and p [M*k,I], y [M*k,H] when ``want_intermediates``)."""
    keep = []
    s = _weights_struct(weights, keep)
    h = _bits(h)
    topk_ids = np.ascontiguousarray(topk_ids, dtype=np.int32)
    M, k = topk_ids.shape
    a = np.ascontiguousarray(topk_weights, dtype=np.float64)
    res = None if residual is None else _bits(residual)
    out = np.zeros((M, s.H), dtype=np.float64)
    p = y = None
    if want_intermediates:
        p = np.zeros((M * k, s.I), dtype=np.float64)
        y = np.zeros((M * k, s.H), dtype=np.float64)
    _check(_load().oracle_expert_ffn(_ptr(h), ctypes.byref(s), M, k, _ptr(topk_ids), _ptr(a),
                                     _ptr(res), _ptr(out), _ptr(p), _ptr(y)),
           "oracle_expert_ffn")
    if want_intermediates:
        return out, p, y
    return out


def decode_block(h, w_router, bias, weights, k, renormalize=True, residual=None):
    """(topk_ids [M,k], topk_weights [M,k] float64, gap [M], out [M,H] float64)."""
    keep = []
    s = _weights_struct(weights, keep)
    h = _bits(h)
    M = h.shape[0]
    w_router = _bits(w_router)
    bias = None if bias is None else np.ascontiguousarray(bias, dtype=np.float32)
    res = None if residual is None else _bits(residual)
    ids = np.zeros((M, k), dtype=np.int32)
    wts = np.zeros((M, k), dtype=np.float64)
    gap = np.zeros((M,), dtype=np.float64)
    out = np.zeros((M, s.H), dtype=np.float64)
    _check(_load().oracle_decode_block(_ptr(h), _ptr(w_router), _ptr(bias), ctypes.byref(s), M,
                                       k, int(bool(renormalize)), _ptr(res), _ptr(ids),
                                       _ptr(wts), _ptr(gap), _ptr(out)), "oracle_decode_block")
    return ids, wts, gap, out


def host_weights(layer: dict, experts=None) -> dict:
    """Host copies of a layer's expert weights (a dict of torch tensors as the seeded input
    generator makes them) in the dict form the functions above take.  Marshalling only:
    bf16 tensors become their uint16 bit patterns, index maps uint8 arrays.

    ``experts`` (optional, sorted list of expert ids) restricts the copy to those experts
    and renumbers them 0..len-1; the caller must renumber routes the same way.
    """
    import torch

    def sel(t):
        if t is None:
            return None
        if experts is not None:
            t = t[torch.as_tensor(experts, device=t.device, dtype=torch.long)]
        return t

    def bits(t):
        if t.dtype != torch.bfloat16:
            raise TypeError("expected a bf16 tensor")
        return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)

    kind = layer["kind"]
    w = {"kind": kind, "H": layer["H"], "I": layer["I"],
         "E": layer["E"] if experts is None else len(experts),
         "d": layer.get("d", 0), "K": layer.get("K", 0)}
    if kind == W_DENSE:
        w["w_gate"] = bits(sel(layer["w_gate"]))
        w["w_up"] = bits(sel(layer["w_up"]))
    else:
        w["j_gate"] = sel(layer["j_gate"]).cpu().numpy()
        w["j_up"] = sel(layer["j_up"]).cpu().numpy()
        w["cb_gate"] = bits(layer["cb_gate"])
        w["cb_up"] = bits(layer["cb_up"])
    if kind == W_VQLR:
        w["r"] = layer["r"]
        w["d_gate"] = bits(layer["d_gate"])
        w["d_up"] = bits(layer["d_up"])
        w["c_gate"] = bits(sel(layer["c_gate"]))
        w["c_up"] = bits(sel(layer["c_up"]))
    w["w_down"] = bits(sel(layer["w_down"]))
    return w
