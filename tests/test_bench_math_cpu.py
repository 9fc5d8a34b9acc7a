"""The bench's measurement arithmetic on the host: algorithmic bytes and
operations per call, the clock-sample summary that decides whether a run is
kept, the lookup of the committed DRAM traffic record, and the roofline
denominators."""

from __future__ import annotations

import json
import os
import sys
from types import SimpleNamespace

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def proj(m, k, n, x_dtype="bf16"):
    return SimpleNamespace(m=m, k=k, n=n, x_dtype=x_dtype)


def test_decode_bytes_of_the_2b_projection():
    """M=1, K=2560 -> N=6912, bf16 x: packed W 4,423,680 B, x 5,120 B, y
    27,648 B, gamma 4 B and one scale 4 B: 4,456,456 B."""
    b = bench.row_bytes(proj(1, 2560, 6912))
    assert b["forward"] == 4_423_680 + 5_120 + 27_648 + 4 + 4 == 4_456_456
    # packing: the compulsory traffic, the fp32 weight read once, packed bytes and gamma written
    assert b["pack_weights"] == 4 * 6912 * 2560 + 6912 * 2560 // 4 + 4


def test_fp32_activations_count_four_bytes():
    assert bench.row_bytes(proj(4, 256, 256, "f32"))["forward"] - bench.row_bytes(proj(4, 256, 256))["forward"] \
        == 2 * 4 * 256


def test_prefill_operations():
    # 72.48 G operations per 2B-class projection at M = 2048
    assert bench.row_ops(proj(2048, 2560, 6912))["forward"] == 2 * 2048 * 6912 * 2560 == 72_477_573_120
    projs = [proj(2048, 2560, 6912), proj(2048, 6912, 2560)]
    assert bench.workload_units(projs, "TOPS") == 2 * 72_477_573_120


def test_workload_units_sums_the_forward_bytes():
    projs = [proj(1, 2560, 6912), proj(1, 6912, 2560)]
    assert bench.workload_units(projs, "GB/s") == sum(bench.row_bytes(p)["forward"] for p in projs)
    assert bench.workload_units(projs, "GB/s", rows=("forward", "pack_weights")) == \
        sum(bench.row_bytes(p)["forward"] + bench.row_bytes(p)["pack_weights"] for p in projs)
    # the table-lookup alternative moves the same algorithmic bytes as the dp4a forward
    assert all(bench.row_bytes(p)["forward_lut"] == bench.row_bytes(p)["forward"] for p in projs)
    assert bench.lut_applies(bench.WORKLOADS["decode_2b"]) and bench.lut_applies(bench.WORKLOADS["stack_7b_decode"])
    assert not bench.lut_applies(bench.WORKLOADS["prefill_2b"])


def test_rotation_covers_twice_the_l2(monkeypatch):
    """The decode pool of packed weights is at least twice the L2 size."""
    monkeypatch.setattr(bench, "l2_bytes", lambda device: 126 * 2 ** 20)
    wl = bench.WORKLOADS["decode_2b"]
    slots = bench.decode_slots(wl, None)
    per_slot = sum(p.n * p.k // 4 for p in wl.projections)
    assert slots * per_slot >= 2 * 126 * 2 ** 20 and (slots - 1) * per_slot < 2 * 126 * 2 ** 20
    assert bench.decode_slots(bench.WORKLOADS["stack_7b_decode"], None) == 1     # 1.26 GB of weights
    assert bench.prefill_slots(bench.WORKLOADS["prefill_2b"], None) >= 2


def test_oracle_work_split_covers_the_sample_once():
    """The all-cores oracle's work items cover every sampled row and token of
    every projection exactly once."""
    projs = [proj(1, 2560, 6912), proj(2048, 6912, 2560)]
    for p, nm in zip(projs, ("a", "b")):
        p.name = nm
    items = bench._split(projs, 1000, 7)
    for j, p in enumerate(projs):
        cover = np.zeros((p.m, min(1000, p.n)), dtype=int)
        for jj, r0, r1, t0, t1 in items:
            if jj == j:
                cover[t0:t1, r0:r1] += 1
        assert (cover == 1).all()


@pytest.mark.parametrize("m,k,want", [
    (1, 2560, ["bl_gemv_dp4a"]), (4, 2560, ["bl_gemv_dp4a"]), (4, 32768, ["bl_act_tq", "bl_gemv_w"]),
    (8, 2560, ["bl_decode_mma"]), (16, 2560, ["bl_act_quant", "bl_decode_mma"]),
    (17, 2560, ["bl_act_perm", "bl_gemm_tc"]), (2048, 6912, ["bl_act_perm", "bl_gemm_tc"]),
])
def test_row_kernels_follow_the_library_dispatch(m, k, want):
    assert bench.row_kernels(proj(m, k, 6912))["forward"] == want


@pytest.mark.parametrize("m,want", [(1, ["bl_gemv_grouped"]), (2, ["bl_act_quant_grouped", "bl_gemm_grouped"]),
                                    (2048, ["bl_act_quant_grouped", "bl_gemm_grouped"])])
def test_grouped_row_kernels_follow_the_library_dispatch(m, want):
    # one token: the fused per-group kernel; more: the activation pass, then the contraction
    assert bench.row_kernels(proj(m, 2560, 6912))["forward_grouped"] == want


class _Done:
    def terminate(self):
        pass

    def wait(self, timeout=None):
        return 0


def _sampler(rows, t0=10.0, t1=20.0):
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc, s.thread, s.t0, s.t1 = _Done(), None, t0, t1
    s.samples = [(t, [c.strip() for c in r.split(",")]) for t, r in rows]
    return s


def test_clock_summary_uses_samples_inside_the_timed_region(monkeypatch):
    monkeypatch.setattr(bench.time, "sleep", lambda _s: None)
    rows = [
        (9.0, "1200, 2032, 200.0, 0x0, Not Active, Not Active, Not Active, Not Active"),      # before
        (11.0, "2032, 2032, 900.5, 0x0, Not Active, Not Active, Not Active, Not Active"),
        (12.0, "1965, 2032, 1090.0, 0x4, Not Active, Not Active, Not Active, Active"),
        (13.0, "1957, 2032, 1088.0, 0x4, Not Active, Not Active, Not Active, Active"),
        (25.0, "2032, 2032, 150.0, 0x0, Active, Not Active, Not Active, Not Active"),          # after
    ]
    c = _sampler(rows).stop()
    assert c["samples"] == 3 and c["sm_mhz"] == 1965.0 and c["sm_max_mhz"] == 2032.0
    assert c["power_w_max"] == 1090.0
    assert c["reasons"] == ["sw_power_cap"]          # the hw_slowdown sample lies outside


def test_clock_summary_reports_every_throttle_reason(monkeypatch):
    monkeypatch.setattr(bench.time, "sleep", lambda _s: None)
    rows = [(15.0, "1500, 2032, 700.0, 0x68, Active, Active, Active, Not Active")]
    c = _sampler(rows).stop()
    assert c["reasons"] == ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"]


def test_clock_summary_without_nvidia_smi():
    s = bench.ClockSampler.__new__(bench.ClockSampler)
    s.proc = None
    assert s.stop()["reasons"] == ["nvidia-smi unavailable"]


def test_traffic_record_is_keyed_to_the_kernel_source(monkeypatch, tmp_path):
    rec = tmp_path / "dram_traffic.txt"
    h = bench.source_hash("pack.cu")
    rec.write_text(f"# header\ntraffic pack_weights {h} decode_2b 141814400 note\n"
                   f"traffic pack_weights 0123456789abcdef decode_2b 1 stale\n")
    monkeypatch.setattr(bench, "TRAFFIC_PATH", str(rec))
    assert bench.traffic_record("pack_weights", "decode_2b") == 141814400
    assert bench.traffic_record("pack_weights", "no_such_workload") is None
    assert bench.traffic_record("prefill", "decode_2b") is None
    monkeypatch.setattr(bench, "source_hash", lambda src: "0000000000000000")
    assert bench.traffic_record("pack_weights", "decode_2b") is None   # a changed kernel has no record


def test_peaks_come_from_the_measured_file():
    hbm, bf16, sustained, source = bench.peaks()
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if not os.path.exists(path):
        assert source == "fallback" and (hbm, bf16) == (bench.FALLBACK_HBM_GBS, bench.FALLBACK_BF16_TFLOPS)
        return
    d = json.load(open(path))
    assert source == "measured" and hbm == float(d["hbm_gbs"]) and bf16 == float(d["bf16_tflops"])
    assert sustained <= bf16


def test_step_sets_build_every_call_kind_on_cpu(monkeypatch):
    """ForwardSet and PackSet with a stand-in library on CPU tensors: every
    call kind (dp4a forward, table lookup, per-group) is built and callable."""
    import torch
    calls = []

    class FakeLib:
        def __getattr__(self, name):
            def f(*a):
                calls.append(name)
                return 1024 if name.endswith("_workspace_bytes") else 0
            return f

    class Grouped:
        def __init__(self, n, k):
            self.wp = torch.zeros(n, k // 4, dtype=torch.uint8)
            self.gammas = torch.zeros(n, k // 64)

    class FakeBlt:
        lib = FakeLib()
        BL_BF16, BL_F32 = 1, 0
        forward_workspace_bytes = staticmethod(lambda m, n, k: 1024)
        pack_workspace_bytes = staticmethod(lambda n, k: 1024)
        PackedWeight = staticmethod(lambda *a: a)
        pack_weights = staticmethod(lambda w, out=None: out)
        pack_weights_grouped = staticmethod(lambda w: Grouped(*w.shape))

    monkeypatch.setattr(torch.cuda, "synchronize", lambda *a, **k: None)
    wl = bench.WORKLOADS["cpu_small"]
    fs = bench.ForwardSet(FakeBlt, wl.projections, torch.device("cpu"), 2)
    for _, c in fs.calls(0):
        c(0)
    fs.lut = True
    for _, c in fs.calls(1):
        c(0)
    fs.lut = False
    fs.add_grouped()
    fs.grouped = True
    for _, c in fs.calls(1):
        c(0)
    assert [n for n in calls if n in ("bitlinear_forward", "bitlinear_forward_lut", "bitlinear_forward_grouped")] == \
        ["bitlinear_forward", "bitlinear_forward_lut", "bitlinear_forward_grouped"]
    assert len(bench.PackSet(FakeBlt, wl.projections, torch.device("cpu"), 2).calls(0)) == len(wl.projections)


def test_traffic_records_match_the_kernel_sources():
    # every DRAM-traffic record the bench reports is keyed to the current
    # source of its kernel: an edit of the source (or of the shared headers)
    # must come with a new capture, or a re-keyed record after an edit that
    # changes no code, else the bench line reports the traffic as null
    seen = set()
    with open(bench.TRAFFIC_PATH) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 5 and parts[0] == "traffic":
                seen.add((parts[1], parts[3]))
    assert {k for k, _ in seen} == set(bench.KERNEL_SOURCE)
    for kind, workload in sorted(seen):
        assert bench.traffic_record(kind, workload) is not None, (kind, workload)
