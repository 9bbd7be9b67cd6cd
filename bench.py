#!/usr/bin/env python3
"""Benchmark of the MoE decode block (one JSON line on stdout, rank 0).

A step is one pass of the whole block -- router GEMV + softmax top-k, alignment, gate/up +
SiLU, down + weighted combine -- over one batch of seeded synthetic input, through the C ABI
(moe_decode_block).  Default workload: one Qwen3-30B-A3B-shaped MoE layer (H=2048, I=768,
E=128, k=8, b=8) at M=21 decode tokens.  Successive steps cycle through several
independently drawn weight sets, so every step reads its experts from HBM, not from L2.

value   = decode tokens/s over all ranks (M * steps * ranks / max-over-ranks time);
e2e     = the same metric through moe_decode_block_host (host h in, host out back, the
          copies inside the timed region);
roofline= the gate/up kernel (the dominant one): algorithmic bytes per launch / its mean
          duration from CUDA events recorded around it on its stream, over a traced pass of
          the same steps right after the timed region;
cpu_baseline = the fp64 CPU oracle on a bounded sample of the same workload.

`--impl reference` times the oracle alone (the reference arm: there is no other
implementation of this block to run) and prints the same line with "impl": "reference".
Under torchrun every rank runs its own replica of the workload on its own GPU.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from routed_expert_ffn_top_gb300 import synthetic as syn  # noqa: E402

METRIC = "MoE-block decode µs/layer, tokens/s & HBM GB/s vs ~8 TB/s peak, M=1..256"
UNIT = "tokens/s"
FALLBACK_HBM_GBS = 6800.0
PROFILES = os.path.join(ROOT, "profiles")


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="layer_m21", choices=sorted(syn.WORKLOADS))
    p.add_argument("--M", type=int, default=None, help="override the token count")
    p.add_argument("--graph", action="store_true",
                   help="time CUDA-graph replays of the block instead of direct calls")
    p.add_argument("--b", type=int, default=None,
                   help="override the alignment block size (64 selects the tcgen05 regime)")
    p.add_argument("--E", type=int, default=None,
                   help="override the expert count (smaller captures of the same kernels)")
    p.add_argument("--vq-form", type=int, default=None, choices=[0, 1, 2],
                   help="override the VQ gate/up form (VQ workloads): 0 code books in shared "
                        "memory, 1 projected code books, 2 decoded on the tensor cores")
    p.add_argument("--weight-sets", type=int, default=8,
                   help="independent weight sets cycled by single-layer workloads")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--no-per-config", action="store_true",
                   help="skip the per-configuration entries (the other configurations' timings)")
    p.add_argument("--no-extras", action="store_true",
                   help="time the block only (no trace, e2e, CPU baseline): for profilers")
    return p.parse_args()


# ------------------------------------------------------------------------------ ranks
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int) -> float:
    if world == 1:
        return value
    import torch.distributed as dist
    dev = torch.device("cuda", torch.cuda.current_device()) if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ----------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle-reason samples every 200 ms while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            with open(self.path) as f:
                for line in f:
                    parts = [x.strip() for x in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
        finally:
            if self.path and os.path.exists(self.path):
                os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------- helpers
NOMINAL_HBM_GBS = 8000.0  # the headline metric's "~8 TB/s"


def bootstrap_median_ci(values, resamples=10000, seed=0):
    """95% bootstrap interval of the median of `values` (resampled with replacement)."""
    rng = np.random.default_rng(seed)
    v = np.asarray(values, dtype=np.float64)
    meds = np.median(rng.choice(v, size=(resamples, v.size), replace=True), axis=1)
    lo, hi = np.percentile(meds, [2.5, 97.5])
    return [round(float(lo), 3), round(float(hi), 3)]


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def overrides(args) -> dict:
    out = {}
    if args.M:
        out["M"] = args.M
    if args.E:
        out["E"] = args.E
    if args.b:
        out["b"] = args.b
    if args.vq_form is not None:
        out["vq_form"] = args.vq_form
    return out


def gemm_regime(wl) -> bool:
    """Dense weights (and VQ gate/up decoded on the tensor cores) run as tcgen05 grouped
    GEMMs over tiles of the aligned blocks."""
    return wl.kind == syn.W_DENSE or (wl.kind == syn.W_VQ and wl.vq_form == 2)


def gateup_kernel_name(wl) -> str:
    if gemm_regime(wl):
        return "gemm_gateup_vq_kernel" if wl.kind == syn.W_VQ else "gemm_gateup_kernel"
    return "vq_ttable_partial_kernel" if wl.vq_form == 1 else "gateup_vq_kernel"


KERNEL_SOURCES = {
    "decode_small_kernel": ("decode_small.cu", "gemm_core.cuh", "route_core.cuh", "align_core.cuh",
                            "small_route.cuh"),
    "gemm_fused_kernel": ("gemm_tc05.cu", "gemm_core.cuh"),
    "gemm_gateup_vq_kernel": ("gemm_tc05.cu", "gemm_core.cuh"),
}


def kernel_source_hash(kernel: str = "gemm_fused_kernel"):
    """Hash of the sources a kernel is built from (its traffic record is void once they change)."""
    h = hashlib.sha256()
    srcs = KERNEL_SOURCES.get(kernel, ("gemv.cu",))
    for name in srcs + ("ptx.cuh", "moe_internal.cuh"):
        with open(os.path.join(ROOT, "routed_expert_ffn_top_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel: str, workload: str, unique_experts: float):
    """DRAM bytes per launch of `kernel`, from the committed ncu record
    (profiles/dram_traffic.txt: kernel, workload, kernel-source hash, unique experts of the
    captured launch, dram read+write bytes of that launch), scaled to `unique_experts`
    routed experts.  None when there is no record taken on the current kernel source."""
    path = os.path.join(PROFILES, "dram_traffic.txt")
    try:
        with open(path) as f:
            for line in f:
                parts = line.split()
                if len(parts) != 5 or line.startswith("#"):
                    continue
                k, wl, src, u, b = parts
                if k == kernel and wl == workload and src == kernel_source_hash(kernel):
                    return float(b) / float(u) * unique_experts
    except (OSError, ValueError):
        return None
    return None


def expert_bytes(wl):
    """Bytes of one expert's weights that the block streams (gate/up representation + down)."""
    if wl.kind == syn.W_DENSE:
        gu = 2 * wl.H * wl.I * 2
    else:
        gu = 2 * (wl.H // wl.d) * wl.I          # uint8 index maps of gate and up
        if wl.kind == syn.W_VQLR:
            gu += 2 * wl.r * wl.I * 2          # bf16 low-rank coefficients C_gate, C_up
    return gu, wl.I * wl.H * 2


def shared_bytes(wl):
    """Layer-shared weights read once per block: the router (and the low-rank bases)."""
    b = wl.H * wl.E * 2
    if wl.kind == syn.W_VQLR:
        b += 2 * wl.H * wl.r * 2
    return b


def surface_tensors(moe, layer, M, k, b, ws, ids):
    """The block's intermediate surfaces as one call left them in its workspace (dense
    weights): (valid route ids ascending, p = SiLU(g) * u [bf16, one row per valid route],
    y = p W_down [fp32, one row per valid route]).  p is read from the one-grid path's
    p rows, or de-swizzled from the p tiles the down GEMM reads."""
    lay = moe.moe_workspace_layout(layer, M, k, b)
    I, H = layer["I"], layer["H"]
    R = M * k
    idl = ids.flatten().long()
    valid = torch.nonzero((idl >= 0) & (idl < layer["E"])).flatten()
    y = ws[lay["y"]:lay["y"] + R * H * 4].view(torch.float32).view(R, H)[valid]
    if lay["p_rows"]:
        p = ws[lay["p_rows"]:lay["p_rows"] + R * I * 2].view(torch.bfloat16).view(R, I)[valid]
    else:  # the swizzled p tiles: row n of tile t, 64-wide chunk c, 16-byte piece j
        srt, _, _ = moe.workspace_alignment(ws, lay)
        b, kn, tpb = lay["b"], lay["kn"], lay["tpb"]
        pos = torch.full((R,), -1, dtype=torch.long, device=ws.device)
        srt_l = srt.long()
        rows = torch.nonzero((srt_l >= 0) & (srt_l < R)).flatten()
        pos[srt_l[rows]] = rows
        pv = pos[valid]
        t = (pv // b) * tpb + (pv % b) // kn
        n = (pv % b) % kn
        c = torch.arange(I // 64, device=ws.device)
        j = torch.arange(8, device=ws.device)
        off = (t[:, None, None] * (I // 64) * kn * 128 + c[None, :, None] * kn * 128
               + n[:, None, None] * 128 + ((j[None, None, :] ^ (n[:, None, None] & 7)) << 4))
        pieces = ws[lay["p_tiles"]:].view(-1)
        byte_idx = (off[..., None] + torch.arange(16, device=ws.device)).reshape(len(pv), -1)
        p = pieces[byte_idx].contiguous().view(torch.bfloat16).view(len(pv), I)
    return valid, p, y


def surface_hashes(moe, layer, wl, M, h, ws, ids, out):
    """SHA-256 of the block's surfaces after one call (the route-block page's exact-trajectory
    record): the activation p = SiLU(g) * u (bf16) and the routed down outputs y (fp32) of the
    valid routes in ascending route order, and the final output (bf16), each hashed as its
    raw bytes.  The gate/up GEMM's own output (g, u) is never stored on this path: SiLU and
    the product are applied to the accumulators."""
    _, p, y = surface_tensors(moe, layer, M, wl.k, wl.b, ws, ids)

    def digest(t):
        raw = t.contiguous().view(-1).view(torch.uint8)
        return hashlib.sha256(raw.cpu().numpy().tobytes()).hexdigest()
    return {"w13": "not stored (SiLU(g) * u formed in the gate/up epilogue)",
            "activation": digest(p), "routed_w2": digest(y), "final": digest(out)}


def block_launches(layer, wl, M):
    """Kernels one moe_decode_block call launches (the library's own count)."""
    from routed_expert_ffn_top_gb300 import moe
    return moe.moe_workspace_layout(layer, M, wl.k, wl.b)["launches"]


# The configurations of the headline metric, each measured in its own timed region: the
# decode layer at 1 and 21 tokens, the 48-layer stack at 1, 4, 16 and 64 tokens, the VQ layer
# at 1 to 16 tokens, and the large-batch layer.
PER_CONFIG = [("layer_m1", 1), ("layer_m21", 21), ("stack48", 1), ("stack48", 4),
              ("stack48", 16), ("stack48", 64), ("vq_d4", 1), ("vq_d4", 2), ("vq_d4", 4),
              ("vq_d4", 8), ("vq_d4", 16), ("large_m256", 256)]


def measured_bf16_tflops():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["bf16_tflops"]), "measured"
    except (OSError, KeyError, ValueError):
        return 1900.0, "fallback"


def near_tie_counts(inputs):
    """Tokens of each configuration whose routing is a near tie: the oracle's fp64 margin
    between the k-th and (k+1)-th logit below 1e-4 (where fp32 rounding may legitimately pick
    differently).  inputs: key -> (h, [layers]) as the configurations ran; the count is over
    the tokens of h against each layer's router."""
    import oracle
    out = {}
    for key, (h, layers) in inputs.items():
        n = 0
        for layer in layers:
            bias = layer.get("bias")
            bias = None if bias is None else bias.detach().cpu().numpy()
            logits = oracle.router_logits(syn.bits(h), syn.bits(layer["w_router"]), bias,
                                          h.shape[0], layer["H"], layer["E"])
            k = layer.get("k", 8)
            _, _, gap = oracle.topk_softmax(logits, k)
            n += int((gap < 1e-4).sum())
        out[key] = n
    return out


def per_config_entries(dev, local, min_seconds=0.4, near_inputs=None):
    """µs per layer, tokens/s and HBM fractions of every configuration, each timed with CUDA
    events over whole steps (a step = one layer, or the 48 layers of the stack) after
    warm-up, with its own clock samples.  Single layers cycle 8 independently drawn weight
    sets (9.7 GB, or 38.6 GB at H=4096), the stack reads 48 distinct layers (58 GB): every
    step's expert weights come from HBM.  Blocks align with the configuration's own b."""
    from routed_expert_ffn_top_gb300 import moe

    peak, _ = measured_peaks()
    tpeak, _ = measured_bf16_tflops()
    stream = torch.cuda.current_stream()
    entries = {}
    cache = {}
    for name, M in PER_CONFIG:
        wl = syn.workload(name, M=M)
        if cache.get("name") != name:
            cache.clear()
            torch.cuda.empty_cache()
            n_sets = wl.layers if wl.layers > 1 else 8
            cache["name"] = name
            cache["layers"] = [syn.make_layer(wl, layer=i, seed=1, device=dev) for i in range(n_sets)]
        layers = cache["layers"]
        stack = wl.layers > 1
        h0 = syn.make_hidden(wl, M=M, seed=1, device=dev)
        ws = moe.alloc_workspace(layers[0], M, wl.k, wl.b, dev)
        out = [torch.empty_like(h0) for _ in range(2)]
        ids = torch.empty((M, wl.k), dtype=torch.int32, device=dev)
        wts = torch.empty((M, wl.k), dtype=torch.float32, device=dev)

        def step(i):
            if stack:
                h = h0
                for li, layer in enumerate(layers):
                    moe.moe_decode_block(h, layer, wl.k, wl.b, residual=h, out=out[li % 2],
                                         topk_ids=ids, topk_weights=wts, workspace=ws)
                    h = out[li % 2]
            else:
                moe.moe_decode_block(h0, layers[i % len(layers)], wl.k, wl.b, out=out[0],
                                     topk_ids=ids, topk_weights=wts, workspace=ws)

        # routing of every weight set, or of every layer of the stack (the bytes a step streams)
        uniq, npad_rows = [], []
        b_used = moe.moe_library_block_size(layers[0], M, wl.k, wl.b)
        h = h0
        for li, layer in enumerate(layers):
            moe.moe_decode_block(h, layer, wl.k, wl.b, residual=h if stack else None,
                                 out=out[li % 2], topk_ids=ids, topk_weights=wts, workspace=ws)
            if stack:
                h = out[li % 2]
            uniq.append(int(torch.unique(ids).numel()))
            n_e = torch.bincount(ids.flatten().long(), minlength=wl.E)
            npad_rows.append(int(((n_e + b_used - 1) // b_used * b_used).sum().item()))
        for i in range(5):
            step(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step(0)
        torch.cuda.synchronize()
        per_step = max(time.perf_counter() - t0, 1e-6)
        steps = int(max(10, min(20000, min_seconds / per_step)))
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as clk:
            torch.cuda.synchronize()
            ev0.record(stream)
            for i in range(steps):
                step(i)
            ev1.record(stream)
            torch.cuda.synchronize()
        t_ms = ev0.elapsed_time(ev1)
        if moe.moe_read_device_status(ws) != 0:
            raise RuntimeError("device status set in the %s M=%d entry" % (name, M))
        layers_per_step = len(layers) if stack else 1
        us_layer = t_ms * 1e3 / (steps * layers_per_step)
        gu_b, dn_b = expert_bytes(wl)
        u_mean = statistics.mean(uniq)
        gbs = (u_mean * (gu_b + dn_b) + shared_bytes(wl)) / (us_layer * 1e-6) / 1e9
        e = {"workload": name, "M": M, "b": wl.b, "b_effective": b_used, "steps": steps,
             "us_per_layer": round(us_layer, 3),
             "tokens_per_s": round(M / (us_layer * 1e-6 * layers_per_step), 2),
             "unique_experts_per_layer": round(u_mean, 2),
             "hbm_gbs_unique_expert_bytes": round(gbs, 1),
             "hbm_frac": {"measured": round(gbs / peak, 4),
                          "nominal_8tbs": round(gbs / NOMINAL_HBM_GBS, 4)},
             "gpu_launches": block_launches(layers[0], wl, M) * layers_per_step * steps,
             "clocks": clk.summary()}
        if gemm_regime(wl):
            # the MMAs' N side: every block of b rows is tpb tiles of kn columns
            lay = moe.moe_workspace_layout(layers[0], M, wl.k, wl.b)
            cols = statistics.mean(npad_rows) / b_used * lay["tpb"] * lay["kn"]
            gu_flop = 2.0 * cols * (2 * wl.H * wl.I if wl.kind == syn.W_DENSE else 0)
            flops = gu_flop + 2.0 * cols * wl.I * wl.H
            e["tensor_tflops_issued"] = round(flops / (us_layer * 1e-6) / 1e12, 2)
            e["tensor_frac_measured"] = round(flops / (us_layer * 1e-6) / 1e12 / tpeak, 4)
        entries["%s_M%d" % (name, M)] = e
        if near_inputs is not None:
            router = {"H": wl.H, "E": wl.E, "k": wl.k, "w_router": layers[0]["w_router"].cpu(),
                      "bias": None if layers[0].get("bias") is None else layers[0]["bias"].cpu()}
            near_inputs["%s_M%d" % (name, M)] = (h0.cpu(), [router])
        del ws, out, h0
    cache.clear()
    torch.cuda.empty_cache()
    entries["reader_m1_M1"] = reader_config_entry(dev, local, min_seconds)
    torch.cuda.empty_cache()
    return entries


def reader_config_entry(dev, local, min_seconds=0.4):
    """The channel reader at one token (router + reader per layer, 8 rotating weight sets), in
    its own timed region with clock samples, beside the exact block on the same weights."""
    from routed_expert_ffn_top_gb300 import moe

    wl = syn.WORKLOADS["reader_m1"]
    M, K, nscan = wl.M, wl.reader_K, wl.reader_nscan
    layers, readers = [], []
    for li in range(8):
        layer = syn.make_layer(wl, layer=li, seed=1, device=dev)
        signs = syn.make_rotation_signs(wl.H, seed=li, device=dev)
        readers.append(moe.reader_build(layer, signs, reader_basis(layer["w_down"], wl.reader_rank)))
        layers.append(layer)
    h0 = syn.make_hidden(wl, seed=1, device=dev)
    out = torch.empty_like(h0)
    ids = torch.empty((M, wl.k), dtype=torch.int32, device=dev)
    wts = torch.empty((M, wl.k), dtype=torch.float32, device=dev)
    ws = moe.reader_workspace(readers[0], M, wl.k, K)
    ws_exact = moe.alloc_workspace(layers[0], M, wl.k, wl.b, dev)

    def reader_step(i):
        li = i % len(layers)
        moe.moe_route_topk(h0, layers[li]["w_router"], layers[li]["bias"], wl.k, topk_ids=ids,
                           topk_weights=wts)
        moe.moe_reader_ffn(h0, readers[li], ids, wts, K, nscan, out=out, workspace=ws)

    def exact_step(i):
        moe.moe_decode_block(h0, layers[i % len(layers)], wl.k, wl.b, out=out, topk_ids=ids,
                             topk_weights=wts, workspace=ws_exact)

    def timed(step, clocks=False):
        for i in range(5):
            step(i)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        step(0)
        torch.cuda.synchronize()
        steps = int(max(10, min(20000, min_seconds / max(time.perf_counter() - t0, 1e-6))))
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with ClockSampler(local) as clk:
            torch.cuda.synchronize()
            ev0.record()
            for i in range(steps):
                step(i)
            ev1.record()
            torch.cuda.synchronize()
        return ev0.elapsed_time(ev1) * 1e3 / steps, steps, clk.summary()

    us, steps, clocks = timed(reader_step)
    exact_us, _, _ = timed(exact_step)
    nvalid = M * wl.k * wl.I
    kept = M * min(K, wl.k * wl.I)
    sk_b, ex_b, rc_b = reader_bytes(wl, nvalid, kept)
    full = M * wl.k * (2 * wl.H * wl.I * 2 + wl.I * wl.H * 2)
    return {"workload": "reader_m1", "M": M, "reader_K": K, "reader_nscan": nscan,
            "steps": steps, "us_per_layer": round(us, 3), "tokens_per_s": round(M / (us * 1e-6), 2),
            "exact_block_us_per_layer": round(exact_us, 3),
            "bytes_read_fraction_of_routed": round((sk_b + ex_b + rc_b) / full, 4),
            "gpu_launches": 2 * steps, "clocks": clocks}


# ------------------------------------------------------------------------------ ours
def run_ours(args, world, rank, local):
    from routed_expert_ffn_top_gb300 import build as lib_build
    from routed_expert_ffn_top_gb300 import moe

    lib_build.build()
    dev = torch.device("cuda", local)
    wl = syn.workload(args.workload, **overrides(args))
    if wl.reader_K > 0:
        return run_reader(args, world, rank, local, wl)
    M = wl.M
    stack = wl.layers > 1
    n_sets = wl.layers if stack else max(1, args.weight_sets)
    layers = [syn.make_layer(wl, layer=i, seed=1 + rank, device=dev) for i in range(n_sets)]
    h0 = syn.make_hidden(wl, seed=1 + rank, device=dev)
    ws = moe.alloc_workspace(layers[0], M, wl.k, wl.b, dev)
    out = [torch.empty_like(h0) for _ in range(2)]
    ids = torch.empty((M, wl.k), dtype=torch.int32, device=dev)
    wts = torch.empty((M, wl.k), dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    # router (+ alignment, and the row tiles of the grouped GEMMs, when one router cluster
    # holds every token), else alignment [+ row gather for dense weights]; gate/up, down,
    # combine
    gemm = gemm_regime(wl)
    launches_per_block = block_launches(layers[0], wl, M)
    one_kernel = launches_per_block == 1

    def eager_step(i, s):
        """One step: a single layer, or all L layers of the residual stack."""
        if stack:
            h = h0
            for li in range(n_sets):
                o = out[li % 2]
                moe.moe_decode_block(h, layers[li], wl.k, wl.b, residual=h, out=o, topk_ids=ids,
                                     topk_weights=wts, workspace=ws, stream=s)
                h = o
        else:
            moe.moe_decode_block(h0, layers[i % n_sets], wl.k, wl.b, out=out[0], topk_ids=ids,
                                 topk_weights=wts, workspace=ws, stream=s)

    # The timed steps call moe_decode_block directly.  With --graph they replay CUDA graphs
    # of the same calls (one per weight set, or one of the whole stack) instead; the other
    # form is timed after the main region for comparison.
    graphs = []
    if args.graph:
        if stack:
            graphs.append(moe.capture_graph(lambda s: eager_step(0, s)))
        else:
            for li in range(n_sets):
                graphs.append(moe.capture_graph(lambda s, li=li: eager_step(li, s)))
        torch.cuda.synchronize()

    def step(i):
        if graphs:
            graphs[i % len(graphs)].replay()
        else:
            eager_step(i, stream)

    blocks_per_step = n_sets if stack else 1

    # unique experts each weight set routes to (bytes actually streamed per block)
    gu_b, dn_b = expert_bytes(wl)
    per_set_unique = []
    padded_rows = []  # aligned rows sum_e ceil(n_e / b) * b of each probe
    b_lib = moe.moe_library_block_size(layers[0], M, wl.k, wl.b)

    def note_routing():
        per_set_unique.append(int(torch.unique(ids).numel()))
        n_e = torch.bincount(ids.flatten().long(), minlength=wl.E)
        padded_rows.append(int(((n_e + b_lib - 1) // b_lib * b_lib).sum().item()))

    if stack:
        h = h0
        for li in range(n_sets):
            o = out[li % 2]
            moe.moe_decode_block(h, layers[li], wl.k, wl.b, residual=h, out=o, topk_ids=ids,
                                 topk_weights=wts, workspace=ws)
            note_routing()
            h = o
    else:
        for li in range(n_sets):
            moe.moe_decode_block(h0, layers[li], wl.k, wl.b, out=out[0], topk_ids=ids,
                                 topk_weights=wts, workspace=ws)
            note_routing()
    torch.cuda.synchronize()

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    if moe.moe_read_device_status(ws) != 0:
        raise RuntimeError("device status set during warm-up")

    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
        barrier(world)
    t_ms = ev0.elapsed_time(ev1)
    t_ms = max_over_ranks(t_ms, world)
    clocks = clk.summary()
    status = moe.moe_read_device_status(ws)
    if status != 0:
        raise RuntimeError("device status %#x after the timed region" % status)

    # the other launch form over the same steps, for comparison
    other_ms = None
    if not args.no_extras:
        other = graphs
        if not graphs:
            if stack:
                other = [moe.capture_graph(lambda s: eager_step(0, s))]
            else:
                other = [moe.capture_graph(lambda s, li=li: eager_step(li, s))
                         for li in range(n_sets)]
        torch.cuda.synchronize()
        ev0.record(stream)
        for i in range(args.steps):
            if graphs:
                eager_step(i, stream)
            else:
                other[i % len(other)].replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        other_ms = max_over_ranks(ev0.elapsed_time(ev1), world) / args.steps
        del other

    # the route-block page's protocol: 20 warm-up calls, then 7 blocks of 50 calls, each timed
    # with CUDA events; the median block and a 10,000-resample bootstrap interval of it
    protocol = None
    if not args.no_extras:
        for i in range(20):
            step(i)
        block_us = []
        for blk in range(7):
            torch.cuda.synchronize()
            ev0.record(stream)
            for i in range(50):
                step(blk * 50 + i)
            ev1.record(stream)
            torch.cuda.synchronize()
            block_us.append(ev0.elapsed_time(ev1) * 1e3 / (50 * blocks_per_step))
        protocol = {"calls_per_block": 50, "blocks": 7, "warmup_calls": 20,
                    "median_us_per_layer": round(statistics.median(block_us), 3),
                    "bootstrap95_us_per_layer": bootstrap_median_ci(block_us),
                    "block_us_per_layer": [round(v, 3) for v in block_us]}

    ms_per_step = t_ms / args.steps
    tokens = M * args.steps * world
    value = tokens / (t_ms / 1e3)
    # unique routed-expert bytes of the steps that ran
    if stack:
        step_bytes = sum(per_set_unique) * (gu_b + dn_b)
    else:
        step_bytes = statistics.mean(per_set_unique[i % n_sets] for i in range(args.steps)) * (gu_b + dn_b)
    router_bytes = shared_bytes(wl) * blocks_per_step
    hbm_gbs = (step_bytes + router_bytes) / (ms_per_step * 1e-3) / 1e9
    us_per_layer = ms_per_step * 1e3 / blocks_per_step

    result = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) hidden states, N(0,0.02) bf16 weights)",
        "config": {"workload": wl.name, "M": M, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
                   "b": wl.b, "layers_per_step": blocks_per_step,
                   "weight_kind": "dense_bf16" if wl.kind == syn.W_DENSE else "vq_d%d" % wl.d,
                   "vq_form": None if wl.kind == syn.W_DENSE else wl.vq_form,
                   "l2": ("inputs larger than L2: %d independent weight sets of %.2f GB cycled"
                          % (n_sets, wl.E * (gu_b + dn_b) / 1e9)),
                   "parallelism": "replicas" if world > 1 else "single"},
        "us_per_layer": round(us_per_layer, 3),
        "launch": "cuda_graph_replay" if graphs else "direct_calls",
        ("direct_call_us_per_layer" if graphs else "graph_replay_us_per_layer"):
            None if other_ms is None else round(other_ms * 1e3 / blocks_per_step, 3),
        "hbm_gbs_unique_expert_bytes": round(hbm_gbs, 1),
        "hbm_frac": {"measured": round(hbm_gbs / measured_peaks()[0], 4),
                     "nominal_8tbs": round(hbm_gbs / NOMINAL_HBM_GBS, 4)},
        "unique_experts_per_layer": round(statistics.mean(per_set_unique), 2),
        "unique_experts_per_set": per_set_unique,
        "gpu_launches": launches_per_block * blocks_per_step * args.steps,
        "clocks": clocks,
    }
    if protocol is not None:
        result["protocol"] = protocol
    if args.no_extras:
        if rank == 0:
            print(json.dumps(result), flush=True)
        return

    # --- traced pass: per-kernel durations from events recorded around the kernels
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    dur = {"router": [], "align": [], "gateup": [], "down": [], "combine": []}

    def traced_block(h, li, res, o):
        moe.moe_set_trace_events(evs)
        try:
            moe.moe_decode_block(h, layers[li], wl.k, wl.b, residual=res, out=o, topk_ids=ids,
                                 topk_weights=wts, workspace=ws, stream=stream)
        finally:
            moe.moe_set_trace_events(None)
        evs[5].synchronize()
        dur["router"].append(evs[0].elapsed_time(evs[1]))
        dur["align"].append(evs[1].elapsed_time(evs[2]))
        dur["gateup"].append(evs[2].elapsed_time(evs[3]))
        dur["down"].append(evs[3].elapsed_time(evs[4]))
        dur["combine"].append(evs[4].elapsed_time(evs[5]))

    for i in range(args.steps):
        if stack:
            h = h0
            for li in range(n_sets):
                traced_block(h, li, h, out[li % 2])
                h = out[li % 2]
        else:
            traced_block(h0, i % n_sets, None, out[0])
    mean_ms = {k: statistics.mean(v) for k, v in dur.items()}
    peak, peak_kind = measured_peaks()
    u_mean = statistics.mean(per_set_unique)
    p_bytes = 2 if gemm else 4
    if one_kernel:
        # the whole block in one grid: the routed experts' weights and W_r in, h in, out back
        kernel = "decode_small_kernel"
        alg = u_mean * (gu_b + dn_b) + shared_bytes(wl) + 2 * M * wl.H * 2
        k_ms = sum(mean_ms.values())
    elif wl.kind == syn.W_DENSE:
        # gate/up and down in one grid (its trace interval is the gate/up one): the routed
        # experts' weights, h rows in, p out and back, y out
        kernel = "gemm_fused_kernel"
        alg = (u_mean * (gu_b + dn_b) + M * wl.H * 2 + 2 * M * wl.k * wl.I * p_bytes
               + M * wl.k * wl.H * 4)
        k_ms = mean_ms["gateup"] + mean_ms["down"]
    else:
        # weights of the routed experts + h read once + p written (fp32 per route from the VQ
        # kernels on the CUDA cores, bf16 per route from the tensor-core one)
        kernel = gateup_kernel_name(wl)
        alg = u_mean * gu_b + M * wl.H * 2 + M * wl.k * wl.I * p_bytes
        k_ms = mean_ms["gateup"]
    achieved = alg / (k_ms * 1e-3) / 1e9
    traffic = recorded_traffic(kernel, wl.name, u_mean)
    if one_kernel:  # every trace point follows the one grid
        traced = {kernel: k_ms}
    elif wl.kind == syn.W_DENSE:  # the row gather counts with the alignment interval
        traced = {"router": mean_ms["router"], "align": mean_ms["align"], kernel: k_ms,
                  "combine": mean_ms["combine"]}
    else:
        traced = mean_ms
    result["roofline"] = {
        "kernel": kernel, "bound": "hbm", "achieved": round(achieved, 1),
        "peak": peak, "peak_source": peak_kind, "unit": "GB/s", "frac": round(achieved / peak, 4),
        "frac_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
        "traffic": None if traffic is None else int(traffic),
        "algorithmic_bytes_per_launch": int(alg),
        "kernel_ms": round(k_ms, 5),
        "kernel_ms_traced": {k: round(v, 5) for k, v in traced.items()},
    }
    if not one_kernel and wl.kind != syn.W_DENSE:
        dn_alg = u_mean * dn_b + M * wl.k * (wl.I * p_bytes + wl.H * 4)
        result["down_kernel_gbs"] = round(dn_alg / (mean_ms["down"] * 1e-3) / 1e9, 1)
    if gemm:
        # tensor work actually issued: every MMA column (tpb tiles of kn per block of b rows,
        # valid or padding) x 2 flops per MAC
        lay = moe.moe_workspace_layout(layers[0], M, wl.k, wl.b)
        cols = float(sum(padded_rows) / len(padded_rows)) / lay["b"] * lay["tpb"] * lay["kn"]
        flops = 2 * cols * (2 * wl.H * wl.I if wl.kind == syn.W_DENSE else 0)
        if wl.kind == syn.W_DENSE:
            flops += 2 * cols * wl.I * wl.H
        result["roofline"]["tensor_tflops_issued"] = round(flops / (k_ms * 1e-3) / 1e12, 1)

    # --- e2e: host h in, host out back, copies inside the timed region
    h_host = h0.cpu().pin_memory()
    out_host = torch.empty_like(h_host).pin_memory()
    h_dev = torch.empty_like(h0)

    def e2e_step(i):
        if stack:  # one host round trip around the whole L-layer stack
            h_dev.copy_(h_host, non_blocking=True)
            h = h_dev
            for li in range(n_sets):
                moe.moe_decode_block(h, layers[li], wl.k, wl.b, residual=h, out=out[li % 2],
                                     topk_ids=ids, topk_weights=wts, workspace=ws, stream=stream)
                h = out[li % 2]
            out_host.copy_(h, non_blocking=True)
            stream.synchronize()
        else:  # the C ABI's host entry point: copy in, block, copy out, synchronise
            moe.moe_decode_block_host(h_host, layers[i % n_sets], wl.k, wl.b, h_dev, out[0],
                                      out_host, ids, wts, ws, stream=stream)

    for i in range(max(1, args.warmup)):
        e2e_step(i)
    barrier(world)
    t0 = time.perf_counter()
    for i in range(args.steps):
        e2e_step(i)
    t_e2e = max_over_ranks(time.perf_counter() - t0, world)
    result["e2e"] = {"value": round(M * args.steps * world / t_e2e, 3), "unit": UNIT,
                     "h2d_bytes_per_step": M * wl.H * 2, "d2h_bytes_per_step": M * wl.H * 2}

    # --- the exact-trajectory record: surface hashes of two calls on the same inputs (dense
    # weights: their p is in the tiles or rows the workspace layout names)
    if wl.kind == syn.W_DENSE:
        hashes = []
        for _ in range(2):
            ws.zero_()
            o = torch.empty_like(h0)
            moe.moe_decode_block(h0, layers[0], wl.k, wl.b, out=o, topk_ids=ids,
                                 topk_weights=wts, workspace=ws)
            torch.cuda.synchronize()
            hashes.append(surface_hashes(moe, layers[0], wl, M, h0, ws, ids, o))
        result["surface_hashes"] = dict(hashes[0], repeat_identical=hashes[0] == hashes[1])
    else:
        result["surface_hashes"] = "recorded for dense weights only"
    result["config"]["b_effective"] = moe.moe_library_block_size(layers[0], M, wl.k, wl.b)
    result["config"]["launches_per_layer"] = launches_per_block

    # --- every configuration of the metric, each in its own timed region (N = 1 only)
    near_inputs = {wl.name + "_M%d" % M: (h0, [dict(layers[0], k=wl.k)])}
    if world == 1 and not args.no_per_config:
        result["per_config"] = per_config_entries(dev, local, near_inputs=near_inputs)

    # --- CPU baseline: the oracle on a bounded sample (rank 0 only, N = 1 only), and the
    # oracle's count of near-tie tokens of each configuration's routing
    if rank == 0 and world == 1:
        result["cpu_baseline"] = cpu_baseline(wl, layers[0], h0, args.cpu_seconds)
        nt = near_tie_counts(near_inputs)
        result["near_tie_tokens"] = nt.get(wl.name + "_M%d" % M)
        for key, entry in result.get("per_config", {}).items():
            entry["near_tie_tokens"] = nt.get(key)
    if rank == 0:
        print(json.dumps(result), flush=True)


# ---------------------------------------------------------------------- channel reader
def reader_bytes(wl, nvalid_channels, kept):
    """Algorithmic bytes of one reader decode for one token: the sketch (two-bit codes and
    fp32 scales of gate and up, the down norm) of every candidate channel, the exact rows
    (gate, up, down) of the kept ones, the recovery coefficients of the discarded ones, U."""
    nb = wl.H // 128
    sketch = nvalid_channels * (2 * nb * (32 + 4) + 4)
    exact = kept * 3 * wl.H * 2
    recover = (nvalid_channels - kept) * wl.reader_rank * 2 + wl.H * wl.reader_rank * 4
    return sketch, exact, recover


def reader_basis(w_down: torch.Tensor, rank: int = 32) -> torch.Tensor:
    """The reader's recovery basis U [H, rank] fp32 -- model data the caller supplies, built
    once per layer offline, not part of the decode path: the top left singular vectors of the
    H x (E I) matrix of down columns, from the eigenvectors of D^T D (torch's symmetric
    eigensolver on the host)."""
    D = w_down.reshape(-1, w_down.shape[-1]).to(torch.float64)
    evals, evecs = torch.linalg.eigh((D.T @ D).cpu())  # H x H
    order = torch.argsort(evals, descending=True, stable=True)[:rank]
    return evecs[:, order].to(device=w_down.device, dtype=torch.float32).contiguous()


def run_reader(args, world, rank, local, wl):
    from routed_expert_ffn_top_gb300 import moe

    dev = torch.device("cuda", local)
    M, K, nscan = wl.M, wl.reader_K, wl.reader_nscan
    n_sets = max(1, args.weight_sets)
    layers, readers = [], []
    for li in range(n_sets):
        layer = syn.make_layer(wl, layer=li, seed=1 + rank, device=dev)
        signs = syn.make_rotation_signs(wl.H, seed=li, device=dev)
        U = reader_basis(layer["w_down"], wl.reader_rank)  # offline, once per layer
        readers.append(moe.reader_build(layer, signs, U))
        layers.append(layer)
    torch.cuda.synchronize()
    h0 = syn.make_hidden(wl, seed=1 + rank, device=dev)
    out = torch.empty_like(h0)
    ids = torch.empty((M, wl.k), dtype=torch.int32, device=dev)
    wts = torch.empty((M, wl.k), dtype=torch.float32, device=dev)
    ws = moe.reader_workspace(readers[0], M, wl.k, K)
    stream = torch.cuda.current_stream()

    def step(i, s=None):
        li = i % n_sets
        moe.moe_route_topk(h0, layers[li]["w_router"], layers[li]["bias"], wl.k, topk_ids=ids,
                           topk_weights=wts, stream=s)
        moe.moe_reader_ffn(h0, readers[li], ids, wts, K, nscan, out=out, workspace=ws, stream=s)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        ev0.record()
        for i in range(args.steps):
            step(i)
        ev1.record()
        torch.cuda.synchronize()
        barrier(world)
    ms_per_step = max_over_ranks(ev0.elapsed_time(ev1) / args.steps, world)
    clocks = clk.summary()
    value = M * world / (ms_per_step * 1e-3)

    # the exact block on the same weights and tokens, for comparison
    ws_exact = moe.alloc_workspace(layers[0], M, wl.k, wl.b, dev)
    for i in range(args.warmup):
        moe.moe_decode_block(h0, layers[i % n_sets], wl.k, wl.b, out=out, topk_ids=ids,
                             topk_weights=wts, workspace=ws_exact)
    torch.cuda.synchronize()
    ev0.record()
    for i in range(args.steps):
        moe.moe_decode_block(h0, layers[i % n_sets], wl.k, wl.b, out=out, topk_ids=ids,
                             topk_weights=wts, workspace=ws_exact)
    ev1.record()
    torch.cuda.synchronize()
    exact_us = ev0.elapsed_time(ev1) * 1e3 / args.steps

    # traced pass: the reader's stages
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(6)]
    names = ("scan_sketch", "select", "exact", "recover", "final")
    dur = {n: [] for n in names}
    for i in range(args.steps):
        li = i % n_sets
        moe.moe_route_topk(h0, layers[li]["w_router"], layers[li]["bias"], wl.k, topk_ids=ids,
                           topk_weights=wts)
        moe.moe_set_trace_events(evs)
        try:
            moe.moe_reader_ffn(h0, readers[li], ids, wts, K, nscan, out=out, workspace=ws)
        finally:
            moe.moe_set_trace_events(None)
        evs[5].synchronize()
        for q, n in enumerate(names):
            dur[n].append(evs[q].elapsed_time(evs[q + 1]))
    mean_ms = {n: statistics.mean(v) for n, v in dur.items()}
    nvalid = M * wl.k * wl.I
    kept = M * min(K, wl.k * wl.I)
    sk_b, ex_b, rc_b = reader_bytes(wl, nvalid, kept)
    peak, peak_kind = measured_peaks()
    one_grid = M == 1  # one token: the five stages run as one kernel (every trace point after it)
    if one_grid:
        kernel = "reader_one_kernel"
        alg = sk_b + ex_b + rc_b
        k_ms = sum(mean_ms.values())
        traced = {kernel: k_ms}
    else:
        dominant = "sketch" if mean_ms["scan_sketch"] >= mean_ms["exact"] else "exact"
        kernel = "reader_%s_kernel" % dominant
        alg = sk_b if dominant == "sketch" else ex_b
        k_ms = mean_ms["scan_sketch" if dominant == "sketch" else "exact"]
        traced = mean_ms
    achieved = alg / (k_ms * 1e-3) / 1e9
    full = M * wl.k * (2 * wl.H * wl.I * 2 + wl.I * wl.H * 2)  # the routed experts' full bytes
    result = {
        "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) hidden states, N(0,0.02) bf16 weights)",
        "config": {"workload": wl.name, "M": M, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
                   "reader_K": K, "reader_nscan": nscan, "reader_rank": wl.reader_rank,
                   "l2": "inputs larger than L2: %d independent weight sets and readers cycled"
                         % n_sets,
                   "parallelism": "replicas" if world > 1 else "single"},
        "us_per_layer": round(ms_per_step * 1e3, 3),
        "exact_block_us_per_layer": round(exact_us, 3),
        "read_fraction_of_routed_bytes": round((sk_b + ex_b + rc_b) / full, 4),
        "reader_bytes": {"sketch": sk_b, "exact": ex_b, "recover": rc_b},
        "roofline": {"kernel": kernel, "bound": "hbm",
                     "achieved": round(achieved, 1), "peak": peak, "peak_source": peak_kind,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "frac_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4), "traffic": None,
                     "algorithmic_bytes_per_launch": int(alg), "kernel_ms": round(k_ms, 5),
                     "kernel_ms_traced": {n: round(v, 5) for n, v in traced.items()}},
        # the router, then the reader's one grid (one token) or five kernels
        "gpu_launches": (2 if one_grid else 6) * args.steps,
        "clocks": clocks,
    }
    if not args.no_extras:
        h_host = h0.cpu().pin_memory()
        out_host = torch.empty_like(h_host).pin_memory()
        h_dev = torch.empty_like(h0)

        def e2e_step(i):
            li = i % n_sets
            h_dev.copy_(h_host, non_blocking=True)
            moe.moe_route_topk(h_dev, layers[li]["w_router"], layers[li]["bias"], wl.k,
                               topk_ids=ids, topk_weights=wts)
            moe.moe_reader_ffn(h_dev, readers[li], ids, wts, K, nscan, out=out, workspace=ws)
            out_host.copy_(out, non_blocking=True)
            stream.synchronize()

        for i in range(max(1, args.warmup)):
            e2e_step(i)
        barrier(world)
        t0 = time.perf_counter()
        for i in range(args.steps):
            e2e_step(i)
        t_e2e = max_over_ranks(time.perf_counter() - t0, world)
        result["e2e"] = {"value": round(M * args.steps * world / t_e2e, 3), "unit": UNIT,
                         "h2d_bytes_per_step": M * wl.H * 2, "d2h_bytes_per_step": M * wl.H * 2}
        if rank == 0 and world == 1:
            result["cpu_baseline"] = reader_cpu_baseline(wl, layers[0], readers[0], h0,
                                                         args.cpu_seconds)
    if rank == 0:
        print(json.dumps(result), flush=True)


def _reader_oracle_sample(wl, layer, signs, U, h):
    """Host data for the reader oracle: the token's routing and its experts' sketches (the
    sketch is built once per layer, outside the timed decode)."""
    import oracle
    import oracle.reader as R
    hb = syn.bits(h[:1])
    logits = oracle.router_logits(hb, syn.bits(layer["w_router"]), None, 1, wl.H, wl.E)
    ids, wts, _ = oracle.topk_softmax(logits, wl.k)
    experts = sorted(set(ids.reshape(-1).tolist()))
    sel = torch.as_tensor(experts, device=layer["w_down"].device)
    f64 = lambda t: t[sel].to(torch.float64).cpu().numpy()  # noqa: E731
    wg, wu, wd = f64(layer["w_gate"]), f64(layer["w_up"]), f64(layer["w_down"])
    s64 = signs.cpu().numpy().astype(np.float64)
    rd = R.build(wg, wu, wd, s64, rank=1)
    rd["U"] = U.to(torch.float64).cpu().numpy()
    rd["coef"] = wd @ rd["U"]
    local = np.array([experts.index(e) for e in ids[0]], np.int32)
    x = h[0].to(torch.float64).cpu().numpy()
    return x, local, wts[0], wg, wu, wd, rd, s64


def reader_cpu_baseline(wl, layer, reader, h, seconds):
    import oracle.reader as R
    x, local, a, wg, wu, wd, rd, s64 = _reader_oracle_sample(wl, layer, reader["signs"],
                                                             reader["U"], h)
    total, n = 0.0, 0
    while total < seconds or n == 0:
        t0 = time.perf_counter()
        R.reader_token(x, local, a, wg, wu, wd, rd, s64, wl.reader_K, wl.reader_nscan)
        total += time.perf_counter() - t0
        n += 1
    return {"value": round(n / total, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "%d decodes of one token through the fp64 numpy reader oracle (its "
                      "experts' sketches prebuilt), %.1f s" % (n, total)}


def _oracle_block_sample(wl, layer, h, tokens):
    """Host copies for the oracle: full router, and only the experts the sample uses."""
    import oracle
    bias = layer.get("bias")
    bias = None if bias is None else bias.detach().cpu().numpy()
    hb = syn.bits(h[:tokens])
    wr = syn.bits(layer["w_router"])
    logits = oracle.router_logits(hb, wr, bias, tokens, wl.H, wl.E)
    ids, _, _ = oracle.topk_softmax(logits, wl.k)
    used = sorted(set(ids.reshape(-1).tolist()))
    w = oracle.host_weights(layer, used)
    remap = {e: i for i, e in enumerate(used)}
    return hb, wr, bias, w, remap


def _time_oracle_block(wl, hb, wr, bias, w, remap, tokens):
    """One timed oracle pass over the sample: routing + expert FFN + combine."""
    import oracle
    t0 = time.perf_counter()
    logits = oracle.router_logits(hb, wr, bias, tokens, wl.H, wl.E)
    ids, wts, _ = oracle.topk_softmax(logits, wl.k)
    local = np.vectorize(remap.get)(ids).astype(np.int32)
    oracle.expert_ffn(hb, w, local, wts)
    return time.perf_counter() - t0


def cpu_baseline(wl, layer, h, seconds):
    """The fp64 oracle on a bounded sample of the batch, timed single-threaded and on all the
    host's cores (OpenMP over routes; the results do not depend on the thread count)."""
    import oracle
    oracle.build()
    # a bounded sample: whole passes over at most 32 tokens of the batch
    tokens = min(h.shape[0], 32)
    hb, wr, bias, w, remap = _oracle_block_sample(wl, layer, h, tokens)
    ncpu = os.cpu_count() or 1
    before = oracle.set_threads(0)
    legs = {}
    try:
        for name, threads in (("single_thread", 1), ("all_cores", ncpu)):
            used = oracle.set_threads(threads)
            total, n = 0.0, 0
            while total < seconds / 2 or n == 0:
                total += _time_oracle_block(wl, hb, wr, bias, w, remap, tokens)
                n += 1
            legs[name] = {"value": round(tokens * n / total, 4), "threads": used, "passes": n,
                          "seconds": round(total, 2)}
    finally:
        oracle.set_threads(before)
    best = legs["all_cores"]
    return {"value": best["value"], "unit": UNIT, "cores": best["threads"], "kind": "oracle",
            "host_cpu_count": ncpu, "single_thread": legs["single_thread"],
            "sample": "passes of the %s block over %d of its %d tokens (router, all their routed "
                      "experts, combine) through the fp64 C oracle: %.1f s on %d threads (OpenMP "
                      "over routes), %.1f s on one" % (wl.name, tokens, h.shape[0],
                                                       best["seconds"], best["threads"],
                                                       legs["single_thread"]["seconds"])}


# ------------------------------------------------------------------------- reference
def run_reference(args, world, rank):
    if rank != 0:
        return
    import oracle
    oracle.build()
    wl = syn.workload(args.workload, **overrides(args))
    layer = syn.make_layer(wl, layer=0, seed=1, device="cpu")
    h = syn.make_hidden(wl, seed=1, device="cpu")
    if wl.reader_K > 0:
        return run_reader_reference(args, world, wl, layer, h)
    # each step: the oracle's full block on a sample of at most 8 tokens of the batch
    tokens = min(wl.M, 8)
    hb, wr, bias, w, remap = _oracle_block_sample(wl, layer, h, tokens)
    for _ in range(args.warmup):
        _time_oracle_block(wl, hb, wr, bias, w, remap, tokens)
    times = [_time_oracle_block(wl, hb, wr, bias, w, remap, tokens) for _ in range(args.steps)]
    total = sum(times)
    value = tokens * args.steps / total
    blocks = wl.layers if wl.layers > 1 else 1
    sample = ("%d of the %d tokens of the %s batch per step (one layer), single-threaded fp64 "
              "C oracle" % (tokens, wl.M, wl.name))
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "M": wl.M, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
                   "b": wl.b, "layers_per_step": blocks},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def run_reader_reference(args, world, wl, layer, h):
    """The reader oracle as the reference arm: one token's decode per step."""
    import oracle.reader as R
    signs = syn.make_rotation_signs(wl.H, seed=0)
    U = torch.as_tensor(R.down_basis(layer["w_down"].to(torch.float64).numpy(), wl.reader_rank))
    x, local, a, wg, wu, wd, rd, s64 = _reader_oracle_sample(wl, layer, signs, U, h)
    for _ in range(args.warmup):
        R.reader_token(x, local, a, wg, wu, wd, rd, s64, wl.reader_K, wl.reader_nscan)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        R.reader_token(x, local, a, wg, wu, wd, rd, s64, wl.reader_K, wl.reader_nscan)
        times.append(time.perf_counter() - t0)
    total = sum(times)
    value = args.steps / total
    sample = "one token of the %s layer per step through the fp64 numpy reader oracle" % wl.name
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(total / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": wl.name, "M": wl.M, "H": wl.H, "I": wl.I, "E": wl.E, "k": wl.k,
                   "reader_K": wl.reader_K, "reader_nscan": wl.reader_nscan},
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    args = parse_args()
    world, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
