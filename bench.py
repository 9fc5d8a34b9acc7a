#!/usr/bin/env python
"""Benchmark of the BitLinear W1.58A8 hot path on one B300 (or N replicas).

One step runs every step of the path, through the C ABI, on every projection
of the workload, with inputs resident in HBM:

    a1-a3   bitlinear_pack_weights   gamma = mean|W| (exact), ternary codes,
                                     four per byte (W is read twice: gamma
                                     must be complete before any code is)
    a4-a6   bitlinear_forward        per-token absmax int8 activations, ternary x
                                     int8 contraction, fp32 rescale (x_q and s
                                     are written out too)

The default workload is the 2B-class decode GEMV (M=1, K=2560->N=6912 and
K=6912->N=2560, fp32 weights packed to 2 bits, bf16 activations). The step
is captured once in a CUDA graph (external event nodes between the calls give
each call's device time) and the timed region replays it.

Prints one JSON line. `--impl reference` times the CPU oracle instead (on the
host cores, on a bounded sample of the same workload).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from workloads import WORKLOADS, make_projection_inputs  # noqa: E402

FALLBACK_HBM_GBS = 6400.0
FALLBACK_BF16_TFLOPS = 1800.0
METRIC = "BitLinear W1.58A8 GB/s (decode) & int8 TOPS (prefill), % of roofline, 1xB300"


# --------------------------------------------------------------------------- algorithmic work
def row_bytes(p):
    """Compulsory bytes of each call on one projection (inputs read once, outputs written once)."""
    nk, mk, mn = p.n * p.k, p.m * p.k, p.m * p.n
    xb = 2 if p.x_dtype == "bf16" else 4
    return {
        "pack_weights": 8 * nk + nk // 4 + 4,                     # read W twice, write Wp and gamma
        # read x, Wp, gamma; write y and the quantised activations (x_q, s)
        "forward": xb * mk + nk // 4 + 4 + 4 * mn + mk + 4 * p.m,
    }


def row_ops(p):
    return {"forward": 2 * p.m * p.n * p.k}


ROWS = ["pack_weights", "forward"]
FUSED_MAX_M = 8     # the forward quantises activations inside the contraction up to this M


def row_kernels(p):
    if p.k % 64 == 0 and p.m >= 17:
        fwd = ["bl_act_perm", "bl_gemm_tc"]
    elif p.k % 64 == 0 and p.m <= 4:
        fwd = ["bl_act_tq", "bl_gemv_w"]
    elif p.k % 64 == 0 and p.m <= FUSED_MAX_M:
        fwd = ["bl_decode_mma"]
    else:
        fwd = ["bl_act_quant", "bl_decode_mma"]
    return {"pack_weights": ["bl_absum_partials", "bl_quant_pack"],
            "forward": fwd}


def workload_units(projs, unit, rows=None):
    rows = rows or ROWS
    if unit == "GB/s":
        return sum(sum(v for r, v in row_bytes(p).items() if r in rows) for p in projs)
    return sum(row_ops(p)["forward"] for p in projs)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1400.0, "fallback"


# --------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi samples (200 ms) of SM clock and throttle reasons during the timed region."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        try:
            self.index = "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            self.index = str(device.index or 0)
        self.samples = []
        self.proc = None
        self.thread = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.index, f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.5)

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.time(), [c.strip() for c in line.split(",")]))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        inside = [s for t, s in self.samples if self.t0 is not None and self.t0 <= t <= self.t1 + 0.2]
        if not inside and self.samples:
            inside = [self.samples[-1][1]]
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = set()
        mhz, mx, pw = [], [], []
        for s in inside:
            try:
                mhz.append(float(s[0]))
                mx.append(float(s[1]))
                pw.append(float(s[2]))
            except ValueError:
                continue
            for nm, v in zip(names[1:], s[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None, "samples": len(mhz), "reasons": sorted(reasons)}


# --------------------------------------------------------------------------- ncu traffic record
def source_hash(src):
    """sha256 (16 hex digits) of a kernel source and the headers every kernel includes."""
    h = hashlib.sha256()
    for name in (src, "kernels.cuh", "common.cuh", "async.cuh"):
        with open(os.path.join(ROOT, "bit_ternary_forward_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_record(kernel_row, workload, prefill=False):
    """DRAM bytes per launch from the committed ncu summary of this workload, if the kernel source is unchanged."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    src = {"pack_weights": "pack.cu", "forward": "gemv_fused.cu"}[kernel_row]
    if kernel_row == "forward" and prefill:
        src = "prefill.cu"
    h = source_hash(src)
    best = None
    for line in open(path):
        parts = line.split()
        if len(parts) >= 5 and parts[0] == "traffic" and parts[1] == kernel_row and parts[2] == h and parts[3] == workload:
            best = float(parts[4])
    return best


# --------------------------------------------------------------------------- oracle (CPU) timing
def oracle_step(inputs, rows_per_proj, pack=True):
    """One oracle step on the first rows_per_proj weight rows of each projection.
    With pack=False the codes come from the set-up (packed once, reused)."""
    import oracle
    done = 0
    for (w, x, p, pre) in inputs:
        n = min(rows_per_proj, p.n)
        if pack:
            wn = w[:n]
            g = oracle.absmean_gamma(wn)
            c = oracle.ternary_codes(wn, g)
            oracle.pack_codes(c)
        else:
            g, c = pre[0], pre[1][:n]
        xq, s = oracle.quant_act(x)
        acc = oracle.ternary_int8_matmul(xq, c)
        oracle.rescale(acc, g, s)
        done += n
    return done


def oracle_inputs(projs, pack=True):
    import oracle
    out = []
    for p in projs:
        w, x = make_projection_inputs(p)
        if x.dtype == torch.bfloat16:
            xf = oracle.bf16_bits_to_f32(x.view(torch.int16).numpy().view(np.uint16))
        else:
            xf = x.numpy()
        wn = w.numpy()
        pre = None
        if not pack:
            g = oracle.absmean_gamma(wn)
            pre = (g, oracle.ternary_codes(wn, g))
        out.append((wn, xf, p, pre))
    return out


def sampled_units(projs, n_rows, unit, rows=None):
    tot = 0
    for p in projs:
        n = min(n_rows, p.n)
        q = type(p)(p.name, p.m, p.k, n, p.w_seed, p.x_seed, p.w_dist, p.x_dist, p.x_dtype)
        tot += workload_units([q], unit, rows)
    return tot


def time_oracle(projs, unit, budget_s, steps=None, warmup=0, rows=None):
    """Oracle throughput on a row sample sized so that `steps` steps take about budget_s.
    rows: the bench rows the step covers (without the packing rows the codes
    are made once before timing, as the packed-once workloads do)."""
    pack = rows is None or "pack_weights" in rows
    inputs = oracle_inputs(projs, pack)
    t = time.perf_counter()
    oracle_step(inputs, 64, pack)
    t64 = max(time.perf_counter() - t, 1e-3)
    n_steps = steps if steps else 1
    n_rows = int(64 * (budget_s / n_steps) / t64)
    n_rows = max(1, min(n_rows, max(p.n for p in projs)))
    for _ in range(warmup):
        oracle_step(inputs, n_rows, pack)
    t = time.perf_counter()
    for _ in range(n_steps):
        oracle_step(inputs, n_rows, pack)
    el = time.perf_counter() - t
    units = sampled_units(projs, n_rows, unit, rows) * n_steps
    scale = 1e9 if unit == "GB/s" else 1e12
    return {"value": units / el / scale, "unit": unit, "cores": 1, "kind": "oracle", "seconds": el,
            "steps": n_steps,
            "sample": f"first {n_rows} weight rows of each of {len(projs)} projection(s) (all tokens), "
                      f"{n_steps} step(s); numpy oracle, single thread"}


# --------------------------------------------------------------------------- the GPU step
class Step:
    """The timed step. Single-projection workloads pack weights inside the step
    (pack_weights, forward); the 7B-class stacks pack every layer
    once at set-up and reuse it, so their step is the forward of every
    projection."""

    def __init__(self, projs, device, rotate, pack_in_step=True):
        import bit_ternary_forward_b300 as blt
        from workloads.synth import gaussian_activations_on, student_t_weights_on
        self.blt = blt
        self.lib = blt.lib
        self.projs = projs
        self.device = device
        self.pack_in_step = pack_in_step
        self.rows = ROWS if pack_in_step else ["forward"]
        self.slots = []
        for r in range(rotate):
            slot = []
            for p in projs:
                nws = max(blt.pack_workspace_bytes(p.n, p.k), blt.forward_workspace_bytes(p.m, p.n, p.k))
                d = {
                    "p": p,
                    "gamma": torch.empty(1, dtype=torch.float32, device=device),
                    "wp": torch.empty((p.n, p.k // 4), dtype=torch.uint8, device=device),
                    "xq": torch.empty((p.m, p.k), dtype=torch.int8, device=device),
                    "s": torch.empty(p.m, dtype=torch.float32, device=device),
                    "y": torch.empty((p.m, p.n), dtype=torch.float32, device=device),
                    "ws_t": torch.empty(nws + 256, dtype=torch.uint8, device=device),
                    "nws": nws,
                }
                d["ws"] = (d["ws_t"].data_ptr() + 255) // 256 * 256
                if pack_in_step:
                    w, x = make_projection_inputs(p)
                    d["w"] = (w.clone() if r else w).to(device)
                    d["x"] = x.to(device)
                else:
                    w = student_t_weights_on(device, p.n, p.k, p.w_seed) if p.w_dist == "t4" else \
                        make_projection_inputs(p)[0].to(device)
                    blt.pack_weights(w, out=blt.PackedWeight(d["wp"], d["gamma"], p.n, p.k))
                    torch.cuda.synchronize(device)
                    del w
                    d["x"] = gaussian_activations_on(device, p.m, p.k, p.x_seed + 7919 * r)
                d["xdt"] = blt.BL_BF16 if d["x"].dtype == torch.bfloat16 else blt.BL_F32
                slot.append(d)
            self.slots.append(slot)
        self.rotate = rotate

    def run(self, i, stream, events=None):
        """One step on rotation slot i; events receives external event records between calls."""
        lib = self.lib
        st = stream.cuda_stream
        for d in self.slots[i % self.rotate]:
            p = d["p"]
            if self.pack_in_step:
                if events is not None:
                    events.mark(stream)
                self._ok(lib.bitlinear_pack_weights(d["w"].data_ptr(), p.n, p.k, d["wp"].data_ptr(),
                                                    d["gamma"].data_ptr(), d["ws"], d["nws"], st))
            if events is not None:
                events.mark(stream)
            self._ok(lib.bitlinear_forward(d["x"].data_ptr(), d["xdt"], p.m, d["wp"].data_ptr(), d["gamma"].data_ptr(),
                                           p.n, p.k, d["y"].data_ptr(), d["xq"].data_ptr(), d["s"].data_ptr(),
                                           d["ws"], d["nws"], st))
        if events is not None:
            events.mark(stream)

    def _ok(self, st):
        if st != 0:
            raise RuntimeError(self.lib.bitlinear_last_error().decode())

    def launches_per_step(self):
        return sum(len(k) for p in self.projs for r, k in row_kernels(p).items() if r in self.rows)


class GraphEvents:
    def __init__(self, pre_created):
        from cuda.bindings import runtime as rt
        self.rt = rt
        self.pool = pre_created
        self.used = 0

    def mark(self, stream):
        ev = self.pool[self.used]
        self.used += 1
        err, = self.rt.cudaEventRecordWithFlags(ev.cuda_event, stream.cuda_stream, self.rt.cudaEventRecordExternal)
        if int(err) != 0:
            raise RuntimeError(f"cudaEventRecordWithFlags failed: {err}")


# --------------------------------------------------------------------------- main
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, device):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


STEP_DESC = ("pack_weights (absmean, codes, packing) + forward (act quant, contraction, rescale) per projection")


def base_config(wl, world):
    """The config fields both arms report for a workload."""
    return {"workload": wl.name, "description": wl.description,
            "projections": [f"{p.name}: M={p.m} K={p.k} N={p.n}"
                            for p in wl.projections[:len(wl.projections) // max(wl.layers, 1)]],
            "layers": wl.layers,
            "step": STEP_DESC if wl.layers == 1 else "forward (act quant, contraction, rescale) of every projection; "
                                                      "weights packed once at set-up",
            "parallelism": f"replicas x{world}"}


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    wl = WORKLOADS[args.workload]
    projs = wl.projections if wl.layers == 1 else wl.projections[:4]
    unit = "GB/s" if args.unit == "GB/s" else "TOPS"
    rows = ROWS if wl.layers == 1 else ["forward"]
    r = time_oracle(projs, unit, budget_s=args.reference_budget, steps=args.steps, warmup=min(args.warmup, 3),
                    rows=rows)
    line = {"metric": METRIC, "impl": "reference", "value": r["value"], "unit": unit, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * r["seconds"] / r["steps"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int64/f32",
            "data": "synthetic (seeded generators)",
            "config": base_config(wl, world),
            "cpu_baseline": {"value": r["value"], "unit": unit, "cores": r["cores"], "kind": "oracle",
                             "sample": r["sample"]},
            "e2e": {"value": r["value"], "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default="decode_2b", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--graph-steps", type=int, default=250, help="steps per captured graph")
    ap.add_argument("--rotate", type=int, default=2, help="input copies cycled between steps")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=15.0)
    ap.add_argument("--reference-budget", type=float, default=90.0)
    args = ap.parse_args(argv)
    wl = WORKLOADS[args.workload]
    args.unit = "GB/s" if all(p.m <= 64 for p in wl.projections) else "TOPS"

    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        return run_reference(args, world, rank)

    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    projs = wl.projections
    pack_in_step = wl.layers == 1
    step = Step(projs, device, args.rotate if pack_in_step else 1, pack_in_step)
    rows_used = step.rows
    stream = torch.cuda.Stream(device)
    hbm, bf16, bf16_sus, peak_src = peaks()

    # warm-up (eager), also the first use of every kernel
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            step.run(i, stream)
    stream.synchronize()

    # Two graphs of G steps: the timed one holds the calls alone, so each
    # kernel may start (programmatic dependent launch) while the one before
    # it drains; the second has external event nodes between the calls, which
    # end that overlap, and gives each call's own device time.
    G = max(1, min(args.graph_steps, args.steps))
    while args.steps % G:
        G -= 1
    replays = args.steps // G
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        for i in range(G):
            step.run(i, stream)
    graph.replay()
    n_marks = G * (len(projs) * len(rows_used) + 1)
    pool = [torch.cuda.Event(enable_timing=True) for _ in range(n_marks)]
    for ev in pool:
        ev.record(stream)
    stream.synchronize()
    gev = GraphEvents(pool)
    marked = torch.cuda.CUDAGraph()
    with torch.cuda.graph(marked, stream=stream):
        for i in range(G):
            step.run(i, stream, events=gev)
    marked.replay()
    stream.synchronize()

    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(device)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize(device)
    clocks.mark("t0")
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for _ in range(replays):
            graph.replay()
        t_end.record(stream)
    torch.cuda.synchronize(device)
    clocks.mark("t1")
    barrier(world)
    clk = clocks.stop()
    ms = t_start.elapsed_time(t_end)
    ms = max_over_ranks(ms, world, device)

    # per-call device times: a second timed pass over the marked graph
    with torch.cuda.stream(stream):
        for _ in range(min(replays, 3)):
            marked.replay()
    torch.cuda.synchronize(device)
    # per-call device times from the last replay's external events
    per_row = {r: [] for r in rows_used}
    marks_per_step = len(projs) * len(rows_used) + 1
    for i in range(G):
        k = i * marks_per_step
        for p in projs:
            for r in rows_used:
                per_row[r].append((p, pool[k].elapsed_time(pool[k + 1])))
                k += 1
    unit = args.unit
    scale = 1e9 if unit == "GB/s" else 1e12
    units_step = workload_units(projs, unit, rows_used)
    value = world * units_step * args.steps / (ms * 1e-3) / scale

    rows = []
    for r in rows_used:
        tot_ms = sum(t for _, t in per_row[r])
        launches = len(per_row[r])
        avg_ms = tot_ms / launches
        byts = sum(row_bytes(p)[r] for p, _ in per_row[r]) / launches
        gbs = byts / (avg_ms * 1e-3) / 1e9
        kern = sorted({k for p, _ in per_row[r] for k in row_kernels(p)[r]})
        entry = {"row": r, "kernels": kern, "avg_us": 1e3 * avg_ms, "share": None,
                 "bytes_per_launch": byts, "gbs": gbs, "hbm_frac": gbs / hbm}
        if r == "forward":
            ops = sum(row_ops(p)["forward"] for p, _ in per_row[r]) / launches
            entry["tops"] = ops / (avg_ms * 1e-3) / 1e12
        entry["_tot"] = tot_ms
        rows.append(entry)
    tot_all = sum(e["_tot"] for e in rows)
    for e in rows:
        e["share"] = e.pop("_tot") / tot_all
    dom = max(rows, key=lambda e: e["share"])
    if unit == "GB/s" or dom["row"] != "forward":
        roof = {"bound": "hbm", "achieved": dom["gbs"], "peak": hbm, "unit": "GB/s", "frac": dom["gbs"] / hbm,
                "traffic": traffic_record(dom["row"], wl.name, unit != "GB/s"),
                "kernel": dom["row"] + " (" + "+".join(dom["kernels"]) + ")",
                "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_src})"}
    else:
        roof = {"bound": "tensor", "achieved": dom["tops"], "peak": bf16, "unit": "TFLOP/s",
                "frac": dom["tops"] / bf16, "traffic": traffic_record(dom["row"], wl.name, True),
                "kernel": dom["row"] + " (" + "+".join(dom["kernels"]) + "; fp16 tcgen05.mma, exact)",
                "peak_source": f"MEASURED_PEAKS.json bf16_tflops burst ({peak_src}); fp16 runs at the bf16 rate",
                "frac_of_sustained": dom["tops"] / bf16_sus}

    # end to end through the public API with host buffers
    e2e = run_e2e(step, projs, device, stream, args.e2e_steps, unit, scale)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = time_oracle(projs if pack_in_step else projs[:4], unit, budget_s=args.cpu_budget,
                          rows=rows_used)
        cpu = {k: cpu[k] for k in ("value", "unit", "cores", "kind", "sample")}

    n_launch = step.launches_per_step() * args.steps
    line = {
        "metric": METRIC, "value": value, "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms / args.steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "u8/i8/i32 (f32 scales)", "data": "synthetic (seeded generators)",
        "config": {**base_config(wl, world),
                   "units_per_step": units_step,
                   "l2": f"inputs larger than L2: {args.rotate} rotating input sets of "
                         f"{sum(4 * p.n * p.k + 2 * p.m * p.k for p in projs) / 1e6:.1f} MB",
                   "graph_steps": G,
                   "rows_timing": "rows and roofline from a second timed pass whose graph has event nodes "
                                  "between the calls (each call alone, no overlap with its neighbours)"},
        "roofline": roof,
        "rows": rows,
        "clocks": clk,
        "e2e": e2e,
        "gpu_launches": n_launch,
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_e2e(step, projs, device, stream, steps, unit, scale):
    """Host-resident inputs: H2D copies, the public API calls and a D2H of y, every step.

    With packing in the step the fp32 weights are inputs too (copied and packed
    every step); for the packed-once stacks the packed weights stay resident
    as model state and only the activations travel."""
    import bit_ternary_forward_b300 as blt
    host = []
    for p, d in zip(projs, step.slots[0]):
        hx = d["x"].cpu().pin_memory()
        hw = d["w"].cpu().pin_memory() if step.pack_in_step else None
        host.append((p, d, hw, hx, torch.empty((p.m, p.n), dtype=torch.float32).pin_memory()))
    dev = [(torch.empty((p.n, p.k), dtype=torch.float32, device=device) if hw is not None else None,
            torch.empty((p.m, p.k), dtype=hx.dtype, device=device)) for p, _, hw, hx, _ in host]
    h2d = sum((hw.numel() * 4 if hw is not None else 0) + hx.numel() * hx.element_size() for _, _, hw, hx, _ in host)
    d2h = sum(hy.numel() * 4 for _, _, _, _, hy in host)

    def one():
        for (p, d, hw, hx, hy), (dw, dx) in zip(host, dev):
            dx.copy_(hx, non_blocking=True)
            if hw is not None:
                dw.copy_(hw, non_blocking=True)
                packed = blt.pack_weights(dw)
            else:
                packed = blt.PackedWeight(d["wp"], d["gamma"], p.n, p.k)
            y = blt.forward(dx, packed)
            hy.copy_(y, non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(3):
            one()
        stream.synchronize()
        t0 = torch.cuda.Event(enable_timing=True)
        t1 = torch.cuda.Event(enable_timing=True)
        t0.record(stream)
        for _ in range(steps):
            one()
        t1.record(stream)
    stream.synchronize()
    ms = t0.elapsed_time(t1)
    rows = step.rows
    return {"value": workload_units(projs, unit, rows) * steps / (ms * 1e-3) / scale, "unit": unit,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "api": "bit_ternary_forward_b300." + ("pack_weights + forward" if step.pack_in_step else "forward") +
                   ", pinned host buffers"}


if __name__ == "__main__":
    sys.exit(main())
