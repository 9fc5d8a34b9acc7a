#!/usr/bin/env python
"""Benchmark of the BitLinear W1.58A8 forward on one B300 (or N replicas).

The metric has two halves, GB/s for decode and int8-equivalent TOPS for
prefill, each against its roofline. One default run measures both:

decode (the line's `value`)
    One step is bitlinear_forward on every projection of the workload
    (default decode_2b: M=1, K=2560->N=6912 and K=6912->N=2560, bf16
    activations) over weights packed once at set-up, as a deployed model's
    are. Distinct packed-weight buffers totalling at least twice the L2 size
    are rotated between steps, so every forward streams its packed weights
    from HBM. Bytes per projection (the algorithmic traffic):
        N*K/4 (packed W) + xb*M*K (x) + 4*M*N (y) + 4 (gamma) + 4*M (scales).
prefill (`prefill` object and rows)
    The same step at M=2048 on the prefill_2b projections; operations
    2*M*N*K per projection.
pack_weights (a row)
    bitlinear_pack_weights (gamma = exact mean|W|, codes, four per byte) is
    one-time work per layer and sits outside the timed step; its compulsory
    bytes are 4*N*K + N*K/4 + 4 (W read once), and the measured DRAM traffic
    (W read twice: gamma must be complete before any code) is reported beside.

Each step is captured in a CUDA graph and replayed in the timed region
(events on the launching stream, barrier and synchronize on both sides). A
second graph of the same calls with event nodes between them gives each
call's own device time (the rows). `e2e` repeats the decode step through the
public Python API with host buffers: every step copies x in from pinned
memory and y out. `cpu_baseline` times the CPU oracle on a row sample, on one
core and on every host core.

--workload selects another workload (skinny_2b, prefill_2b, stack_7b_decode,
stack_7b_prefill, cpu_small) as the line's own step; --impl reference times
the oracle on the host cores instead (the reference arm).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
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
FALLBACK_L2_BYTES = 126 * 2 ** 20
METRIC = "BitLinear W1.58A8 GB/s (decode) & int8 TOPS (prefill), % of roofline, 1xB300"
PREFILL_COMPANION = "prefill_2b"     # the prefill half measured beside the default decode line


# --------------------------------------------------------------------------- algorithmic work
def x_bytes(p):
    return 2 if p.x_dtype == "bf16" else 4


def row_bytes(p):
    """Algorithmic bytes of each call on one projection.

    forward: packed W, x and y once, gamma and the per-token scales.
    pack_weights: the compulsory traffic, W read once, Wp and gamma written."""
    nk, mk, mn = p.n * p.k, p.m * p.k, p.m * p.n
    fwd = nk // 4 + x_bytes(p) * mk + 4 * mn + 4 + 4 * p.m
    return {
        "forward": fwd,
        "forward_lut": fwd,
        "forward_grouped": fwd + nk // 16 - 4,             # per-group scales in place of one gamma
        "pack_weights": 4 * nk + nk // 4 + 4,
        "pack_grouped": 4 * nk + nk // 4 + nk // 16,
    }


def row_ops(p):
    return {"forward": 2 * p.m * p.n * p.k, "forward_lut": 2 * p.m * p.n * p.k, "forward_grouped": 2 * p.m * p.n * p.k}


def row_kernels(p):
    """The kernels one call launches, following the library's dispatch."""
    mt = 1 if p.m <= 1 else (2 if p.m <= 2 else 4)
    if p.k % 64 == 0 and p.m >= 17:
        fwd = ["bl_act_perm", "bl_gemm_tc"]
    elif p.k % 64 == 0 and p.m <= 4 and mt * p.k <= 65536:
        fwd = ["bl_gemv_dp4a"]
    elif p.k % 64 == 0 and p.m <= 4:
        fwd = ["bl_act_tq", "bl_gemv_w"]
    elif p.k % 64 == 0 and p.m <= 8:
        fwd = ["bl_decode_mma"]
    elif p.k % 64 == 0:
        fwd = ["bl_act_quant", "bl_decode_mma"]
    else:
        fwd = ["bl_act_quant", "bl_gemv_w2a8"]
    return {"pack_weights": ["bl_absum_partials", "bl_quant_pack"], "forward": fwd, "forward_lut": ["bl_gemv_lut"],
            "forward_grouped": ["bl_gemv_grouped"] if p.m == 1 else ["bl_act_quant_grouped", "bl_gemm_grouped"],
            "pack_grouped": ["bl_pack_grouped"]}


def workload_units(projs, unit, rows=("forward",)):
    if unit == "GB/s":
        return sum(row_bytes(p)[r] for p in projs for r in rows)
    return sum(row_ops(p)["forward"] for p in projs)


def is_decode(wl):
    return all(p.m <= 64 for p in wl.projections)


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1400.0, "fallback"


MAX_ORACLE_PROCESSES = 32   # each process holds its own copy of the sampled inputs


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


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
            # the timed region was shorter than the sampling period: the sample nearest to it
            mid = 0.5 * (self.t0 + self.t1) if self.t0 is not None else self.samples[-1][0]
            inside = [min(self.samples, key=lambda ts: abs(ts[0] - mid))[1]]
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
KERNEL_SOURCE = {"pack_weights": "pack.cu", "decode": "gemv_dp4a.cu", "prefill": "prefill.cu"}
TRAFFIC_PATH = os.path.join(ROOT, "profiles", "dram_traffic.txt")


def source_hash(src):
    """sha256 (16 hex digits) of a kernel source and the headers every kernel includes."""
    h = hashlib.sha256()
    for name in (src, "kernels.cuh", "common.cuh", "async.cuh"):
        with open(os.path.join(ROOT, "bit_ternary_forward_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def traffic_record(kind, workload):
    """DRAM bytes per launch from the committed ncu summary of this workload,
    if the kernel source is unchanged since the capture (else None)."""
    path = TRAFFIC_PATH
    if not os.path.exists(path) or kind not in KERNEL_SOURCE:
        return None
    h = source_hash(KERNEL_SOURCE[kind])
    best = None
    for line in open(path):
        parts = line.split()
        if len(parts) >= 5 and parts[0] == "traffic" and parts[1] == kind and parts[2] == h and parts[3] == workload:
            best = float(parts[4])
    return best


# --------------------------------------------------------------------------- oracle (CPU) timing
def _oracle_prepare(projs, pack):
    """Per projection: (W fp32, x fp32, projection, (gamma, codes) or None)."""
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
            wn = None                      # only the codes are needed from here on
        out.append((wn, xf, p, pre))
    return out


def _oracle_part(inputs, j, r0, r1, t0, t1, pack):
    """The oracle on weight rows [r0, r1) and tokens [t0, t1) of projection j."""
    import oracle
    wn, xf, p, pre = inputs[j]
    if pack:
        wr = wn[r0:r1]
        g = oracle.absmean_gamma(wr)
        c = oracle.ternary_codes(wr, g)
        oracle.pack_codes(c)
    else:
        g, c = pre[0], pre[1][r0:r1]
    xq, s = oracle.quant_act(xf[t0:t1])
    acc = oracle.ternary_int8_matmul(xq, c)
    oracle.rescale(acc, g, s)


def _split(projs, n_rows, parts):
    """Work items (projection, row range, token range) covering the first n_rows
    rows of every projection in about `parts` pieces: by tokens when a
    projection has many, else by rows."""
    items = []
    for j, p in enumerate(projs):
        n = min(n_rows, p.n)
        if p.m >= 64:
            cuts = np.linspace(0, p.m, min(parts, p.m) + 1).astype(int)
            items += [(j, 0, n, int(a), int(b)) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
        else:
            cuts = np.linspace(0, n, min(parts, n) + 1).astype(int)
            items += [(j, int(a), int(b), 0, p.m) for a, b in zip(cuts[:-1], cuts[1:]) if b > a]
    return items


_POOL_INPUTS = None


def _pool_init(names, pack):
    global _POOL_INPUTS
    import torch as _t
    _t.set_num_threads(1)
    projs = [p for name, idx in names for p in [WORKLOADS[name].projections[idx]]]
    _POOL_INPUTS = (_oracle_prepare(projs, pack), pack)


def _pool_task(item):
    inputs, pack = _POOL_INPUTS
    _oracle_part(inputs, *item, pack)
    return 0


def sampled_units(projs, n_rows, unit, rows):
    tot = 0
    for p in projs:
        n = min(n_rows, p.n)
        q = type(p)(p.name, p.m, p.k, n, p.w_seed, p.x_seed, p.w_dist, p.x_dist, p.x_dtype)
        tot += workload_units([q], unit, rows)
    return tot


class OracleTimer:
    """The CPU oracle, as it stands, on a row sample of a workload: on one core
    and on every host core (a spawned process pool over row or token ranges,
    started before the first CUDA call)."""

    def __init__(self, wl_name, projs_idx, unit, rows, cores=None):
        self.wl = WORKLOADS[wl_name]
        self.names = [(wl_name, i) for i in projs_idx]
        self.projs = [self.wl.projections[i] for i in projs_idx]
        self.unit, self.rows = unit, rows
        self.pack = "pack_weights" in rows
        self.host = host_cores()
        self.cores = cores or min(self.host, MAX_ORACLE_PROCESSES)
        self.pool = None
        if self.cores > 1:
            ctx = mp.get_context("spawn")
            self.pool = ctx.Pool(self.cores, initializer=_pool_init, initargs=(self.names, self.pack))

    def close(self):
        if self.pool is not None:
            self.pool.terminate()
            self.pool.join()

    def _scale(self):
        return 1e9 if self.unit == "GB/s" else 1e12

    def single(self, budget_s, steps=1, warmup=0):
        inputs = _oracle_prepare(self.projs, self.pack)
        t = time.perf_counter()
        for j, p in enumerate(self.projs):
            _oracle_part(inputs, j, 0, min(64, p.n), 0, p.m, self.pack)
        t64 = max(time.perf_counter() - t, 1e-3)
        n_rows = max(1, min(int(64 * (budget_s / steps) / t64), max(p.n for p in self.projs)))
        for _ in range(warmup):
            self._run_single(inputs, n_rows)
        t = time.perf_counter()
        for _ in range(steps):
            self._run_single(inputs, n_rows)
        el = time.perf_counter() - t
        units = sampled_units(self.projs, n_rows, self.unit, self.rows) * steps
        return {"value": units / el / self._scale(), "unit": self.unit, "cores": 1, "kind": "oracle",
                "seconds": el, "steps": steps,
                "sample": f"first {n_rows} weight rows of each of {len(self.projs)} projection(s) (all tokens), "
                          f"{steps} step(s); numpy oracle, one process"}

    def _run_single(self, inputs, n_rows):
        for j, p in enumerate(self.projs):
            _oracle_part(inputs, j, 0, min(n_rows, p.n), 0, p.m, self.pack)

    def parallel(self, budget_s, steps=1, warmup=0):
        if self.pool is None:
            r = self.single(budget_s, steps, warmup)
            return r
        # a short calibration run across the pool, then a sample sized to the budget
        n_rows = 64 * self.cores
        t = time.perf_counter()
        self.pool.map(_pool_task, _split(self.projs, n_rows, self.cores), chunksize=1)
        tc = max(time.perf_counter() - t, 1e-3)
        n_rows = max(1, min(int(n_rows * (budget_s / steps) / tc), max(p.n for p in self.projs)))
        items = _split(self.projs, n_rows, self.cores)
        for _ in range(max(1, warmup)):
            self.pool.map(_pool_task, items, chunksize=1)
        t = time.perf_counter()
        for _ in range(steps):
            self.pool.map(_pool_task, items, chunksize=1)
        el = time.perf_counter() - t
        units = sampled_units(self.projs, n_rows, self.unit, self.rows) * steps
        return {"value": units / el / self._scale(), "unit": self.unit, "cores": self.cores, "kind": "oracle",
                "seconds": el, "steps": steps,
                "sample": f"first {n_rows} weight rows of each of {len(self.projs)} projection(s) (all tokens), "
                          f"{steps} step(s); numpy oracle, {self.cores} processes over row or token ranges "
                          f"({self.host} host cores)"}


def oracle_projection_indices(wl):
    """The projections the oracle samples: all of a one-layer workload, one layer of a stack."""
    return list(range(len(wl.projections) if wl.layers == 1 else len(wl.projections) // wl.layers))


# --------------------------------------------------------------------------- the GPU sets
def l2_bytes(device):
    try:
        return int(torch.cuda.get_device_properties(device).L2_cache_size) or FALLBACK_L2_BYTES
    except Exception:
        return FALLBACK_L2_BYTES


def _check(lib, st):
    if st != 0:
        raise RuntimeError(lib.bitlinear_last_error().decode())


class ForwardSet:
    """Packed-once weights, activations and outputs of a list of projections in
    `slots` distinct copies. Slot 0 holds the seeded workload (weights packed
    by the library at set-up); further slots hold copies of its packed bytes
    and fresh activations in their own buffers, so that rotating the slots
    makes every forward read its packed weights from HBM."""

    def __init__(self, blt, projs, device, slots):
        from workloads.synth import gaussian_activations_on, student_t_weights_on
        self.blt, self.lib, self.projs, self.device = blt, blt.lib, projs, device
        self.lut = False          # calls go to bitlinear_forward_lut (the table-lookup GEMV) when set
        self.grouped = False      # calls go to bitlinear_forward_grouped (per-group scales) when set
        self.slots = []
        for r in range(slots):
            slot = []
            for j, p in enumerate(projs):
                nws = blt.forward_workspace_bytes(p.m, p.n, p.k)
                d = {"p": p, "y": torch.empty((p.m, p.n), dtype=torch.float32, device=device),
                     "ws_t": torch.empty(nws + 256, dtype=torch.uint8, device=device), "nws": nws}
                d["ws"] = (d["ws_t"].data_ptr() + 255) // 256 * 256
                if r == 0:
                    d["wp"] = torch.empty((p.n, p.k // 4), dtype=torch.uint8, device=device)
                    d["gamma"] = torch.empty(1, dtype=torch.float32, device=device)
                    if p.w_dist == "t4" and p.n * p.k > 8_000_000:
                        w = student_t_weights_on(device, p.n, p.k, p.w_seed)
                        x = gaussian_activations_on(device, p.m, p.k, p.x_seed)
                    else:
                        w, x = make_projection_inputs(p)
                        w, x = w.to(device), x.to(device)
                    blt.pack_weights(w, out=blt.PackedWeight(d["wp"], d["gamma"], p.n, p.k))
                    torch.cuda.synchronize(device)
                    del w
                    d["x"] = x
                else:
                    src = self.slots[0][j]
                    d["wp"] = src["wp"].clone()
                    d["gamma"] = src["gamma"].clone()
                    d["x"] = gaussian_activations_on(device, p.m, p.k, p.x_seed + 7919 * r,
                                                     dtype=src["x"].dtype)
                d["xdt"] = blt.BL_BF16 if d["x"].dtype == torch.bfloat16 else blt.BL_F32
                slot.append(d)
            self.slots.append(slot)

    def calls(self, i):
        """The forward calls of step i (slot i mod slots), as closures on a stream."""
        lib = self.lib
        out = []
        for d in self.slots[i % len(self.slots)]:
            p = d["p"]

            def call(st, d=d, p=p):
                _check(lib, lib.bitlinear_forward(d["x"].data_ptr(), d["xdt"], p.m, d["wp"].data_ptr(),
                                                  d["gamma"].data_ptr(), p.n, p.k, d["y"].data_ptr(), None, None,
                                                  d["ws"], d["nws"], st))

            def call_lut(st, d=d, p=p):
                _check(lib, lib.bitlinear_forward_lut(d["x"].data_ptr(), d["xdt"], p.m, d["wp"].data_ptr(),
                                                      d["gamma"].data_ptr(), p.n, p.k, d["y"].data_ptr(), st))

            def call_grouped(st, d=d, p=p):
                _check(lib, lib.bitlinear_forward_grouped(d["x"].data_ptr(), d["xdt"], p.m, d["wpg"].data_ptr(),
                                                          d["gammas"].data_ptr(), p.n, p.k, d["y"].data_ptr(), None,
                                                          None, d["gws"], d["ngws"], st))
            out.append((p, call_grouped if self.grouped else (call_lut if self.lut else call)))
        return out

    def add_grouped(self):
        """Per-group packed weights of every projection (slot 0 packed from the
        seeded W, the other slots copies) and the grouped forward's workspaces."""
        blt = self.blt
        for j, p in enumerate(self.projs):
            w, _ = make_projection_inputs(p)
            g = blt.pack_weights_grouped(w.to(self.device))
            torch.cuda.synchronize(self.device)
            del w
            for r, slot in enumerate(self.slots):
                d = slot[j]
                d["wpg"] = g.wp if r == 0 else g.wp.clone()
                d["gammas"] = g.gammas if r == 0 else g.gammas.clone()
                n = int(blt.lib.bitlinear_forward_grouped_workspace_bytes(p.m, p.n, p.k))
                d["gws_t"] = torch.empty(n + 256, dtype=torch.uint8, device=self.device)
                d["gws"] = (d["gws_t"].data_ptr() + 255) // 256 * 256
                d["ngws"] = n

    def weight_bytes_per_slot(self):
        return sum(p.n * p.k // 4 for p in self.projs)


class PackSet:
    """fp32 weights of a list of projections in `slots` copies (each larger
    than L2 in total) and their packed outputs, for timing bitlinear_pack_weights."""

    def __init__(self, blt, projs, device, slots):
        self.blt, self.lib, self.projs = blt, blt.lib, projs
        self.slots = []
        for r in range(slots):
            slot = []
            for p in projs:
                w, _ = make_projection_inputs(p)
                nws = blt.pack_workspace_bytes(p.n, p.k)
                d = {"p": p, "w": w.to(device),
                     "wp": torch.empty((p.n, p.k // 4), dtype=torch.uint8, device=device),
                     "gamma": torch.empty(1, dtype=torch.float32, device=device),
                     "ws_t": torch.empty(nws + 256, dtype=torch.uint8, device=device), "nws": nws}
                d["ws"] = (d["ws_t"].data_ptr() + 255) // 256 * 256
                slot.append(d)
            self.slots.append(slot)

    def calls(self, i):
        lib = self.lib
        out = []
        for d in self.slots[i % len(self.slots)]:
            p = d["p"]

            def call(st, d=d, p=p):
                _check(lib, lib.bitlinear_pack_weights(d["w"].data_ptr(), p.n, p.k, d["wp"].data_ptr(),
                                                       d["gamma"].data_ptr(), d["ws"], d["nws"], st))
            out.append((p, call))
        return out


# --------------------------------------------------------------------------- graphs and timing
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


def capture(step_set, G, stream, marked=False):
    """A CUDA graph of steps 0..G-1 of `step_set`; with marked=True an external
    event node sits before every call and after the last (returns the events)."""
    pool = None
    gev = None
    if marked:
        n = G * len(step_set.projs) + 1
        pool = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        for ev in pool:
            ev.record(stream)
        stream.synchronize()
        gev = GraphEvents(pool)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(G):
            for _, call in step_set.calls(i):
                if gev is not None:
                    gev.mark(stream)
                call(stream.cuda_stream)
        if gev is not None:
            gev.mark(stream)
    g.replay()
    stream.synchronize()
    return g, pool


def time_graph(graph, replays, stream, world, device, clocks=None):
    """ms of `replays` back-to-back replays, max over ranks. A short GPU sleep
    ahead of the start event keeps the GPU busy while the host enqueues the
    graph, so the timed region holds the graph's own work."""
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(device)
    if clocks is not None:
        clocks.mark("t0")
    with torch.cuda.stream(stream):
        torch.cuda._sleep(200_000)
        t_start.record(stream)
        for _ in range(replays):
            graph.replay()
        t_end.record(stream)
    torch.cuda.synchronize(device)
    if clocks is not None:
        clocks.mark("t1")
    barrier(world)
    return max_over_ranks(t_start.elapsed_time(t_end), world, device)


def per_call_ms(step_set, marked_graph, pool, G, stream):
    """[(projection, ms)] of every call of one replay of the marked graph."""
    with torch.cuda.stream(stream):
        marked_graph.replay()
    stream.synchronize()
    out = []
    k = 0
    for i in range(G):
        for p, _ in step_set.calls(i):
            out.append((p, pool[k].elapsed_time(pool[k + 1])))
            k += 1
    return out


def graph_steps_for(steps, cap):
    G = max(1, min(cap, steps))
    while steps % G:
        G -= 1
    return G


def row_entry(name, timings, kind, hbm):
    """Per-call statistics of one row from [(projection, ms)]."""
    launches = len(timings)
    avg_ms = sum(t for _, t in timings) / launches
    byts = sum(row_bytes(p)[kind] for p, _ in timings) / launches
    e = {"row": name, "kernels": sorted({k for p, _ in timings for k in row_kernels(p)[kind]}),
         "calls": launches, "avg_us": 1e3 * avg_ms, "bytes_per_call": byts,
         "gbs": byts / (avg_ms * 1e-3) / 1e9}
    e["hbm_frac"] = e["gbs"] / hbm
    if kind == "forward":
        ops = sum(row_ops(p)["forward"] for p, _ in timings) / launches
        e["tops"] = ops / (avg_ms * 1e-3) / 1e12
    return e


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


def base_config(wl, world):
    """The config fields both arms report for a workload."""
    return {"workload": wl.name, "description": wl.description,
            "projections": [f"{p.name}: M={p.m} K={p.k} N={p.n}"
                            for p in wl.projections[:len(wl.projections) // max(wl.layers, 1)]],
            "layers": wl.layers,
            "step": "bitlinear_forward (activation quantisation, ternary x int8 contraction, rescale) of every "
                    "projection over weights packed once at set-up",
            "parallelism": f"replicas x{world}"}


def unit_of(wl):
    return "GB/s" if is_decode(wl) else "TOPS"


def run_reference(args, world, rank):
    if rank != 0:
        return 0
    wl = WORKLOADS[args.workload]
    unit = unit_of(wl)
    t = OracleTimer(wl.name, oracle_projection_indices(wl), unit, ("forward",), cores=args.cpu_cores)
    try:
        r = t.parallel(args.reference_budget, steps=args.steps, warmup=min(args.warmup, 1))
    finally:
        t.close()
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


def measure_forward(blt, wl, device, stream, args, world, hbm, bf16, bf16_sus, peak_src, slots, clocks=None):
    """Whole-step throughput of the forward step of `wl` and its per-call rows."""
    fs = ForwardSet(blt, wl.projections, device, slots)
    unit = unit_of(wl)
    # eager warm-up: the first use of every kernel
    with torch.cuda.stream(stream):
        for i in range(max(args.warmup, 3)):
            for _, call in fs.calls(i):
                call(stream.cuda_stream)
    stream.synchronize()
    G = graph_steps_for(args.steps, args.graph_steps)
    graph, _ = capture(fs, G, stream)
    marked, pool = capture(fs, G, stream, marked=True)
    if clocks is not None:
        clocks.start()
    ms = time_graph(graph, args.steps // G, stream, world, device, clocks)
    clk = clocks.stop() if clocks is not None else None
    per_call = per_call_ms(fs, marked, pool, G, stream)
    scale = 1e9 if unit == "GB/s" else 1e12
    units_step = workload_units(wl.projections, unit)
    value = world * units_step * args.steps / (ms * 1e-3) / scale
    row = row_entry("forward", per_call, "forward", hbm)
    launches_per_step = sum(len(row_kernels(p)["forward"]) for p in wl.projections)
    if unit == "GB/s":
        # the timed step holds only forward calls: their throughput in the timed region
        achieved = units_step * args.steps / (ms * 1e-3) / 1e9
        roof = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                "traffic": traffic_record("decode", wl.name),
                "kernel": "forward (" + "+".join(row["kernels"]) + ")",
                "achieved_timing": "algorithmic bytes of the timed forwards / the timed region (the step is "
                                   "forward calls only, consecutive calls overlapping as in a decode loop)",
                "alone": {"gbs": row["gbs"], "frac": row["gbs"] / hbm, "avg_us": row["avg_us"]},
                "peak_source": f"MEASURED_PEAKS.json hbm_gbs ({peak_src})"}
    else:
        achieved = units_step * args.steps / (ms * 1e-3) / 1e12
        roof = {"bound": "tensor", "achieved": achieved, "peak": bf16, "unit": "TFLOP/s", "frac": achieved / bf16,
                "frac_of_sustained": achieved / bf16_sus, "traffic": traffic_record("prefill", wl.name),
                "kernel": "forward (" + "+".join(row["kernels"]) + "; fp16 tcgen05.mma made exact)",
                "achieved_timing": "2*M*N*K of the timed forwards / the timed region",
                "alone": {"tflops": row["tops"], "frac": row["tops"] / bf16, "avg_us": row["avg_us"]},
                "peak_source": f"MEASURED_PEAKS.json bf16_tflops burst ({peak_src}); fp16 runs at the bf16 rate"}
    by_proj = []
    for p in wl.projections[:len(wl.projections) // max(wl.layers, 1)]:
        ts = [(q, t) for q, t in per_call if q.name == p.name or q.name.split(".")[-1] == p.name.split(".")[-1]]
        e = row_entry("forward " + p.name.split(".")[-1], ts, "forward", hbm)
        e["frac_of_bf16_burst"] = e["tops"] / bf16 if unit == "TOPS" else None
        by_proj.append(e)
    return {"fs": fs, "ms": ms, "value": value, "unit": unit, "units_step": units_step, "roofline": roof,
            "row": row, "rows_by_projection": by_proj, "clocks": clk, "G": G,
            "launches": launches_per_step * args.steps,
            "slot_bytes": sum(4 * p.m * p.n + x_bytes(p) * p.m * p.k + p.n * p.k // 4 for p in wl.projections)}


LUT_MAX_K = 16384


def lut_applies(wl):
    return all(p.m == 1 and p.k % 64 == 0 and p.k <= LUT_MAX_K for p in wl.projections)


def measure_lut(fs, wl, device, stream, args, world, hbm, dp4a_value):
    """The same decode step through the table-lookup GEMV (bitlinear_forward_lut),
    timed the same way on the same rotating slots, for the comparison with the
    dp4a GEMV of the main line."""
    fs.lut = True
    try:
        with torch.cuda.stream(stream):
            for i in range(3):
                for _, call in fs.calls(i):
                    call(stream.cuda_stream)
        stream.synchronize()
        G = graph_steps_for(args.steps, args.graph_steps)
        graph, _ = capture(fs, G, stream)
        marked, pool = capture(fs, G, stream, marked=True)
        ms = time_graph(graph, args.steps // G, stream, world, device)
        per_call = per_call_ms(fs, marked, pool, G, stream)
    finally:
        fs.lut = False
    units_step = workload_units(wl.projections, "GB/s", rows=("forward_lut",))
    value = world * units_step * args.steps / (ms * 1e-3) / 1e9
    row = row_entry("forward by table lookup (alternative kernel, each call alone)", per_call, "forward_lut", hbm)
    return {"kernel": "bl_gemv_lut", "value": value, "unit": "GB/s", "frac": value / hbm,
            "ms_per_step": ms / args.steps, "alone_us": row["avg_us"], "vs_dp4a": value / dp4a_value,
            "timing": "the main line's method on the same slots: graph of the step's calls, no event nodes"}, row


def grouped_applies(wl):
    return all(p.k % 64 == 0 for p in wl.projections)


def measure_grouped(fs, wl, device, stream, args, world, hbm, dp4a_value):
    """The same step through the per-group forward (bitlinear_forward_grouped)
    on per-group packed copies of the workload's weights, timed the same way."""
    fs.add_grouped()
    fs.grouped = True
    try:
        with torch.cuda.stream(stream):
            for i in range(3):
                for _, call in fs.calls(i):
                    call(stream.cuda_stream)
        stream.synchronize()
        G = graph_steps_for(args.steps, args.graph_steps)
        graph, _ = capture(fs, G, stream)
        marked, pool = capture(fs, G, stream, marked=True)
        ms = time_graph(graph, args.steps // G, stream, world, device)
        per_call = per_call_ms(fs, marked, pool, G, stream)
    finally:
        fs.grouped = False
    unit = unit_of(wl)
    rows = ("forward_grouped",)
    units_step = (workload_units(wl.projections, "GB/s", rows=rows) if unit == "GB/s"
                  else sum(row_ops(p)["forward_grouped"] for p in wl.projections))
    value = world * units_step * args.steps / (ms * 1e-3) / (1e9 if unit == "GB/s" else 1e12)
    row = row_entry("forward with per-group (64) scales (each call alone)", per_call, "forward_grouped", hbm)
    return {"kernels": sorted({k for p in wl.projections for k in row_kernels(p)["forward_grouped"]}), "value": value,
            "unit": unit,
            "frac": value / hbm if unit == "GB/s" else None, "ms_per_step": ms / args.steps,
            "alone_us": row["avg_us"], "vs_per_tensor": value / dp4a_value,
            "timing": "the main line's method on the same slots: graph of the step's calls, no event nodes"}, row


def measure_pack_grouped(blt, wl, device, stream, hbm):
    """Per-call time of bitlinear_pack_weights_grouped on the workload's fp32
    weights (two rotating copies)."""
    ps = PackSet(blt, wl.projections, device, 2)
    for slot in ps.slots:
        for d in slot:
            d["gam_g"] = torch.empty((d["p"].n, d["p"].k // 64), dtype=torch.float32, device=device)
    lib = blt.lib

    class _Grouped:
        projs = ps.projs

        @staticmethod
        def calls(i):
            out = []
            for d in ps.slots[i % len(ps.slots)]:
                p = d["p"]

                def call(st, d=d, p=p):
                    _check(lib, lib.bitlinear_pack_weights_grouped(d["w"].data_ptr(), p.n, p.k, d["wp"].data_ptr(),
                                                                   d["gam_g"].data_ptr(), st))
                out.append((p, call))
            return out
    gs = _Grouped()
    with torch.cuda.stream(stream):
        for i in range(3):
            for _, call in gs.calls(i):
                call(stream.cuda_stream)
    stream.synchronize()
    G = 8
    marked, pool = capture(gs, G, stream, marked=True)
    per_call = per_call_ms(gs, marked, pool, G, stream)
    e = row_entry("pack_weights_grouped (one-time, outside the step)", per_call, "pack_grouped", hbm)
    e["bytes_note"] = "compulsory 4*N*K + N*K/4 + N*K/16 (W read once, Wp and the scales written)"
    del ps
    torch.cuda.empty_cache()
    return e


def measure_pack(blt, wl, device, stream, args, world, hbm):
    """Per-call time of bitlinear_pack_weights on the workload's weights (two
    rotating fp32 copies, each larger than L2 for the 2B shapes)."""
    ps = PackSet(blt, wl.projections, device, 2)
    with torch.cuda.stream(stream):
        for i in range(3):
            for _, call in ps.calls(i):
                call(stream.cuda_stream)
    stream.synchronize()
    G = 8
    marked, pool = capture(ps, G, stream, marked=True)
    per_call = per_call_ms(ps, marked, pool, G, stream)
    e = row_entry("pack_weights (one-time, outside the step)", per_call, "pack_weights", hbm)
    e["bytes_note"] = "compulsory 4*N*K + N*K/4 + 4 (W read once); traffic = measured DRAM bytes per call"
    e["traffic"] = traffic_record("pack_weights", wl.name)
    del ps
    torch.cuda.empty_cache()
    return e


MAX_SLOTS = 256


def decode_slots(wl, device):
    """Rotation slots so that the packed weights of all slots total at least 2x
    L2 (at most MAX_SLOTS: the CPU-scale case stays in L2 and is a parity case)."""
    wbytes = sum(p.n * p.k // 4 for p in wl.projections)
    return max(1, min(MAX_SLOTS, math.ceil(2 * l2_bytes(device) / wbytes)))


def prefill_slots(wl, device):
    """Rotation slots so that each slot's activations, packed weights and outputs
    total at least 2x L2 over all slots."""
    b = sum(4 * p.m * p.n + x_bytes(p) * p.m * p.k + p.n * p.k // 4 for p in wl.projections)
    return max(1, min(MAX_SLOTS, math.ceil(2 * l2_bytes(device) / b)))


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", default="decode_2b", choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--graph-steps", type=int, default=200, help="steps per captured graph")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-companions", action="store_true", help="skip the pack and prefill rows")
    ap.add_argument("--cpu-budget", type=float, default=8.0)
    ap.add_argument("--cpu-cores", type=int, default=0, help="processes of the all-cores oracle (0: all)")
    ap.add_argument("--reference-budget", type=float, default=60.0)
    args = ap.parse_args(argv)
    wl = WORKLOADS[args.workload]

    world, rank, local = dist_setup(args)
    if args.impl == "reference":
        return run_reference(args, world, rank)

    # the all-cores oracle pool is spawned before the first CUDA call
    timer = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        timer = OracleTimer(wl.name, oracle_projection_indices(wl), unit_of(wl), ("forward",),
                            cores=args.cpu_cores or None)

    import bit_ternary_forward_b300 as blt
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.Stream(device)
    hbm, bf16, bf16_sus, peak_src = peaks()

    decode = is_decode(wl)
    slots = decode_slots(wl, device) if decode else prefill_slots(wl, device)
    main_res = measure_forward(blt, wl, device, stream, args, world, hbm, bf16, bf16_sus, peak_src, slots,
                               clocks=ClockSampler(device))
    rows = [dict(main_res["row"], row="forward (all calls of the step, each alone)")] + main_res["rows_by_projection"]

    e2e = run_e2e(blt, main_res["fs"], wl.projections, device, stream, args.e2e_steps, main_res["unit"])
    companions = {}
    if decode and not args.no_companions and lut_applies(wl):
        companions["lut_gemv"], lut_row = measure_lut(main_res["fs"], wl, device, stream, args, world, hbm,
                                                      main_res["value"])
        rows.append(lut_row)
    if not args.no_companions and wl.layers == 1 and wl.name != "cpu_small" and grouped_applies(wl):
        companions["per_group"], g_row = measure_grouped(main_res["fs"], wl, device, stream, args, world, hbm,
                                                         main_res["value"])
        rows.append(g_row)
    del main_res["fs"]
    torch.cuda.empty_cache()

    if not args.no_companions and wl.layers == 1 and wl.name != "cpu_small":
        rows.append(measure_pack(blt, wl, device, stream, args, world, hbm))
        if grouped_applies(wl):
            rows.append(measure_pack_grouped(blt, wl, device, stream, hbm))
        if decode and wl.name == "decode_2b":
            pwl = WORKLOADS[PREFILL_COMPANION]
            pslots = prefill_slots(pwl, device)
            pargs = argparse.Namespace(**vars(args))
            pargs.steps = max(10, min(args.steps, 50))
            pre = measure_forward(blt, pwl, device, stream, pargs, world, hbm, bf16, bf16_sus, peak_src, pslots,
                                  clocks=ClockSampler(device))
            del pre["fs"]
            torch.cuda.empty_cache()
            companions["prefill"] = {
                "workload": pwl.name, "description": pwl.description, "value": pre["value"], "unit": "TOPS",
                "steps": pargs.steps, "ms_per_step": pre["ms"] / pargs.steps, "roofline": pre["roofline"],
                "clocks": pre["clocks"], "slots": pslots, "gpu_launches": pre["launches"]}
            rows += pre["rows_by_projection"]

    cpu = None
    if timer is not None:
        try:
            one = timer.single(args.cpu_budget)
            allc = timer.parallel(args.cpu_budget)
        finally:
            timer.close()
        cpu = {k: allc[k] for k in ("value", "unit", "cores", "kind", "sample")}
        cpu["single_core"] = {k: one[k] for k in ("value", "unit", "cores", "sample")}

    unit = main_res["unit"]
    slot_mb = main_res["slot_bytes"] / 1e6
    line = {
        "metric": METRIC, "value": main_res["value"], "unit": unit, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": main_res["ms"] / args.steps, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8/i8/i32 (f32 scales)",
        "data": "synthetic (seeded generators)",
        "config": {**base_config(wl, world),
                   "units_per_step": main_res["units_step"],
                   "l2": f"inputs larger than L2: {slots} rotating slot(s) of packed weights, activations and "
                         f"outputs ({slot_mb:.1f} MB each; {slots * slot_mb:.0f} MB in all against "
                         f"{l2_bytes(device) / 2 ** 20:.0f} MiB of L2)",
                   "graph_steps": main_res["G"],
                   "rows_timing": "rows from a second graph of the same calls with event nodes between them "
                                  "(each call alone, no overlap with its neighbours)"},
        "roofline": main_res["roofline"],
        "rows": rows,
        **companions,
        "clocks": main_res["clocks"],
        "e2e": e2e,
        "gpu_launches": main_res["launches"],
        "cpu_baseline": cpu,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def run_e2e(blt, fs, projs, device, stream, steps, unit):
    """The step through the public Python API with host buffers: every step
    copies each projection's activations from pinned host memory, runs
    bit_ternary_forward_b300.forward on the resident packed weights (into a
    preallocated output, as a serving loop would) and reads y back into pinned
    host memory. Timed eagerly (one API call per projection per step), and
    again with the same calls captured once in a CUDA graph and replayed per
    step (the copies from and to the pinned buffers run on every replay)."""
    slot = fs.slots[0]
    host = []
    for d in slot:
        p = d["p"]
        host.append((d, d["x"].cpu().pin_memory(), torch.empty((p.m, p.n), dtype=torch.float32).pin_memory(),
                     torch.empty_like(d["x"]), torch.empty((p.m, p.n), dtype=torch.float32, device=device),
                     blt.PackedWeight(d["wp"], d["gamma"], p.n, p.k)))
    h2d = sum(hx.numel() * hx.element_size() for _, hx, _, _, _, _ in host)
    d2h = sum(hy.numel() * 4 for _, _, hy, _, _, _ in host)

    def one():
        for d, hx, hy, dx, dy, packed in host:
            dx.copy_(hx, non_blocking=True)
            blt.forward(dx, packed, y=dy)
            hy.copy_(dy, non_blocking=True)

    scale = 1e9 if unit == "GB/s" else 1e12
    units = workload_units(projs, unit)
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
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        one()
    with torch.cuda.stream(stream):
        g.replay()
        stream.synchronize()
        t0.record(stream)
        for _ in range(steps):
            g.replay()
        t1.record(stream)
    stream.synchronize()
    ms_g = t0.elapsed_time(t1)
    return {"value": units * steps / (ms * 1e-3) / scale, "unit": unit,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": steps,
            "api": "bit_ternary_forward_b300.forward on packed-once weights into preallocated outputs, x and y "
                   "through pinned host buffers, one eager call per projection per step",
            "graph": {"value": units * steps / (ms_g * 1e-3) / scale, "unit": unit,
                      "api": "the same copies and forward calls captured once in a CUDA graph and replayed every "
                             "step (host-to-device and device-to-host copies included in every replay)"}}


if __name__ == "__main__":
    sys.exit(main())
