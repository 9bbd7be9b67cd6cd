"""The bench's host-side bookkeeping on CPU: the committed DRAM traffic records are used only
while their kernel's sources are unchanged, and are scaled by the routed experts of the
measured launch; the per-expert byte counts the roofline divides by follow the weight
representation."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from routed_expert_ffn_top_gb300 import synthetic as syn  # noqa: E402


def _records():
    out = []
    with open(os.path.join(ROOT, "profiles", "dram_traffic.txt")) as f:
        for line in f:
            parts = line.split()
            if line.startswith("#") or len(parts) != 5:
                continue
            k, wl, src, u, b = parts
            out.append((k, wl, src, float(u), float(b)))
    return out


def test_traffic_records_scale_by_routed_experts_and_expire_with_the_sources(monkeypatch):
    recs = _records()
    assert recs, "no traffic record committed"
    for k, wl, src, u, b in recs:
        # pretend the sources are the ones the record was taken on
        monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel, src=src: src)
        assert bench.recorded_traffic(k, wl, u) == b
        assert bench.recorded_traffic(k, wl, 2 * u) == 2 * b
        assert bench.recorded_traffic(k, "no_such_workload", u) is None
        # any change of the kernel's sources voids the record
        monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel: "0" * 16)
        assert bench.recorded_traffic(k, wl, u) is None


def test_source_hash_covers_each_kernels_files(tmp_path, monkeypatch):
    """The hash of a kernel changes when a file of its list (or a shared header) changes, and
    not when another kernel's file does."""
    csrc = os.path.join(ROOT, "routed_expert_ffn_top_gb300", "csrc")
    copy = tmp_path / "routed_expert_ffn_top_gb300" / "csrc"
    copy.mkdir(parents=True)
    for name in os.listdir(csrc):
        p = os.path.join(csrc, name)
        if os.path.isfile(p):
            (copy / name).write_bytes(open(p, "rb").read())
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    for kernel, files in bench.KERNEL_SOURCES.items():
        base = bench.kernel_source_hash(kernel)
        for name in files + ("ptx.cuh", "moe_internal.cuh"):
            f = copy / name
            old = f.read_bytes()
            f.write_bytes(old + b"\n")
            assert bench.kernel_source_hash(kernel) != base, (kernel, name)
            f.write_bytes(old)
        assert bench.kernel_source_hash(kernel) == base
    # the VQ GEMV file is not a source of the fused dense grid
    base = bench.kernel_source_hash("gemm_fused_kernel")
    f = copy / "gemv.cu"
    f.write_bytes(f.read_bytes() + b"\n")
    assert bench.kernel_source_hash("gemm_fused_kernel") == base


def test_expert_bytes_follow_the_weight_representation():
    dense = syn.workload("layer_m21")
    gu, dn = bench.expert_bytes(dense)
    assert gu == 2 * 2048 * 768 * 2 and dn == 768 * 2048 * 2  # bf16 gate + up, bf16 down
    vq = syn.workload("vq_d4")
    gu, dn = bench.expert_bytes(vq)
    assert gu == 2 * (2048 // 4) * 768 and dn == 768 * 2048 * 2  # uint8 index maps, bf16 down
