"""Seeded synthetic inputs for the MoE decode block.

This module holds no arithmetic of the method: it only draws random tensors with the
shapes and distributions of the pages' workload (a Qwen3-30B-A3B-shaped MoE layer:
H=2048, I=768, E=128 experts, top-8) and of the large-batch case (H=4096, I=1536), and
converts them to the bit patterns the CPU oracle takes.  Both the CUDA path and the oracle
receive the very same tensors from here.

Recipe (every tensor has its own sub-seed, a CRC32 of "<workload>/<layer>/<tensor>" mixed
with the run seed, so any tensor can be regenerated alone):

* h ~ N(0, 1) rounded to bf16, shape [M, H];
* router W_r ~ N(0, 0.02) bf16 [H, E]; optional per-expert router bias ~ N(0, 1) fp32 [E];
* dense W_gate, W_up ~ N(0, 0.02) bf16 [E, H, I]; W_down ~ N(0, 0.02) bf16 [E, I, H];
* blockwise VQ gate/up: index maps J uniform in [0, K) uint8 [E, H/d, I]; layer-shared code
  books ~ N(0, 0.02) bf16 [K, d] (one for gate, one for up); down stays dense bf16;
* VQ + low-rank gate/up: the VQ tensors above plus, per projection, a layer-shared basis
  D ~ N(0, 0.02) bf16 [H, r] and per-expert coefficients C ~ N(0, 0.02) bf16 [E, r, I].
"""
from __future__ import annotations

import dataclasses
import zlib
from typing import Optional

import numpy as np
import torch

W_DENSE = 0
W_VQ = 1
W_VQLR = 2


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    H: int
    I: int
    E: int
    k: int
    b: int
    M: int
    kind: int = W_DENSE
    d: int = 4
    K: int = 256
    r: int = 0
    router_bias: bool = False
    layers: int = 1
    residual: bool = False
    w_std: float = 0.02
    h_std: float = 1.0
    # channel reader (dense weights): channels read exactly per token (0: not a reader
    # workload), coordinates scanned per 128-block, rank of the recovery map
    reader_K: int = 0
    reader_nscan: int = 80
    reader_rank: int = 32
    # VQ gate/up form: 0 code books in shared memory, 1 projected code books (<= 4 tokens),
    # 2 decoded into the tensor cores' weight operand (16-row tcgen05 tiles)
    vq_form: int = 0


# The five workloads: a single decode layer at one token, the same layer at 21 tokens (the
# route-block page's fixture size), a 48-layer MoE-only residual stack, a VQ gate/up layer,
# and a large-batch layer with a biased router.
WORKLOADS = {
    "layer_m1": Workload("layer_m1", H=2048, I=768, E=128, k=8, b=8, M=1),
    "layer_m21": Workload("layer_m21", H=2048, I=768, E=128, k=8, b=8, M=21),
    "stack48": Workload("stack48", H=2048, I=768, E=128, k=8, b=8, M=1, layers=48,
                        residual=True),
    "vq_d4": Workload("vq_d4", H=2048, I=768, E=128, k=8, b=8, M=1, kind=W_VQ, d=4, K=256),
    "vqlr_d4_r256": Workload("vqlr_d4_r256", H=2048, I=768, E=128, k=8, b=8, M=1,
                             kind=W_VQLR, d=4, K=256, r=256),
    "vq_d8": Workload("vq_d8", H=2048, I=768, E=128, k=8, b=8, M=1, kind=W_VQ, d=8, K=256),
    "vq_d4_tt": Workload("vq_d4_tt", H=2048, I=768, E=128, k=8, b=8, M=1, kind=W_VQ, d=4,
                         K=256, vq_form=1),
    "vq_d4_tc": Workload("vq_d4_tc", H=2048, I=768, E=128, k=8, b=8, M=1, kind=W_VQ, d=4,
                         K=256, vq_form=2),
    "vqlr_d8_r384": Workload("vqlr_d8_r384", H=2048, I=768, E=128, k=8, b=8, M=1,
                             kind=W_VQLR, d=8, K=256, r=384),
    "large_m256": Workload("large_m256", H=4096, I=1536, E=128, k=8, b=64, M=256,
                           router_bias=True),
    # the decode layer at one token through the channel reader: 756 of the 8 x 768 candidate
    # channels (12.3%) read exactly, 80 of 128 coordinates scanned, a rank-32 map
    "reader_m1": Workload("reader_m1", H=2048, I=768, E=128, k=8, b=8, M=1, reader_K=756),
}


def workload(name: str, **overrides) -> Workload:
    return dataclasses.replace(WORKLOADS[name], **overrides)


def sub_seed(seed: int, wl_name: str, layer: int, tensor: str) -> int:
    tag = ("%s/%d/%s" % (wl_name, layer, tensor)).encode()
    return (zlib.crc32(tag) ^ (seed * 0x9E3779B1)) & 0x7FFFFFFFFFFF


def _gen(device, s):
    g = torch.Generator(device=device)
    g.manual_seed(s)
    return g


def _normal_bf16(shape, std, device, s):
    t = torch.randn(*shape, generator=_gen(device, s), device=device, dtype=torch.float32)
    if std != 1.0:
        t.mul_(std)
    return t.to(torch.bfloat16)


def make_hidden(wl: Workload, M: Optional[int] = None, seed: int = 0, device="cpu",
                tag: str = "h") -> torch.Tensor:
    M = wl.M if M is None else M
    return _normal_bf16((M, wl.H), wl.h_std, device, sub_seed(seed, wl.name, 0, tag))


def make_layer(wl: Workload, layer: int = 0, seed: int = 0, device="cpu") -> dict:
    """All parameters of one MoE layer as torch tensors on ``device``."""
    H, I, E = wl.H, wl.I, wl.E
    s = lambda t: sub_seed(seed, wl.name, layer, t)  # noqa: E731
    p = {"kind": wl.kind, "H": H, "I": I, "E": E, "d": wl.d, "K": wl.K, "r": wl.r,
         "vq_form": wl.vq_form}
    p["w_router"] = _normal_bf16((H, E), wl.w_std, device, s("w_router"))
    if wl.router_bias:
        p["bias"] = torch.randn(E, generator=_gen(device, s("bias")), device=device,
                                dtype=torch.float32)
    else:
        p["bias"] = None
    if wl.kind == W_DENSE:
        p["w_gate"] = _normal_bf16((E, H, I), wl.w_std, device, s("w_gate"))
        p["w_up"] = _normal_bf16((E, H, I), wl.w_std, device, s("w_up"))
    else:
        if H % wl.d:
            raise ValueError("H must be a multiple of d")
        p["j_gate"] = torch.randint(0, wl.K, (E, H // wl.d, I), generator=_gen(device, s("j_gate")),
                                    device=device, dtype=torch.int32).to(torch.uint8)
        p["j_up"] = torch.randint(0, wl.K, (E, H // wl.d, I), generator=_gen(device, s("j_up")),
                                  device=device, dtype=torch.int32).to(torch.uint8)
        p["cb_gate"] = _normal_bf16((wl.K, wl.d), wl.w_std, device, s("cb_gate"))
        p["cb_up"] = _normal_bf16((wl.K, wl.d), wl.w_std, device, s("cb_up"))
    if wl.kind == W_VQLR:
        p["d_gate"] = _normal_bf16((H, wl.r), wl.w_std, device, s("d_gate"))
        p["d_up"] = _normal_bf16((H, wl.r), wl.w_std, device, s("d_up"))
        p["c_gate"] = _normal_bf16((E, wl.r, I), wl.w_std, device, s("c_gate"))
        p["c_up"] = _normal_bf16((E, wl.r, I), wl.w_std, device, s("c_up"))
    p["w_down"] = _normal_bf16((E, I, H), wl.w_std, device, s("w_down"))
    return p


def make_rotation_signs(H: int, seed: int = 0, device="cpu", tag: str = "reader/signs") -> torch.Tensor:
    """The random signs of a block-Hadamard rotation (one +1/-1 per coordinate of H) as int8:
    the random numbers the channel reader draws once, passed to both of its implementations."""
    g = _gen(device, sub_seed(seed, tag, 0, "signs"))
    return (torch.randint(0, 2, (H,), generator=g, device=device, dtype=torch.int32) * 2 - 1).to(torch.int8)


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> C-contiguous numpy uint16 bit patterns (on the host)."""
    if t.dtype != torch.bfloat16:
        raise TypeError("expected a bf16 tensor")
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
