"""Benchmark of the packed low-bit GEMV / GEMM path on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-rows]

Headline workload (one JSON line on stdout, rank 0): the ternary decode layer set of a 27B-class
block (hidden 5120, FFN 17408: q, o 5120x5120; gate, up 17408x5120; down 5120x17408; codes iid
{-1,0,+1} with p = (0.3, 0.4, 0.3); scales |N(0, 0.02)| in fp16; x bf16 N(0, 1); batch 1), the
largest decode configuration of the workload list.  One step decodes one token through LAYERS
distinct copies of that layer set, each issued the way a decoder layer issues it: [q] (lb_gemv),
[o] (lb_gemv), [gate, up] on one activation vector (one lb_gemv_batched launch), [down]
(lb_gemv), i.e. 4 launches per copy.  The weights a step streams (~680 MB) exceed 4x the 126 MB
L2, so every step reads them from HBM.  The K timed steps are one CUDA-graph replay, timed with
CUDA events on the launching stream.

``value`` is the algorithmic packed-weight bandwidth (packed codes + scales + x + y bytes per step
divided by the step time), in GB/s.  ``rows`` adds the other steps of the path measured the same
way: both packers, the GEMVs of every decode configuration (1-bit 2048x2048 fp16; the 1.7B-class
ternary layer set; the 151936x2048 LM head at batch 1 and 4; the 27B-class layer sets at batch 1
and 5, both formats), the prefill GEMM (512 x 5120 -> 17408, TFLOP/s), the embedding gather, the
SiLU-gated pair, and the read-only reference launches of the same byte counts (lb_read_probe).
``e2e`` is the headline metric measured through the public API with host buffers: every step
copies x from pinned host memory, runs the layer-set GEMVs and copies y back.

``--impl reference`` times the CPU oracle (FP64 numpy) on a bounded sample of the same workload.
With torchrun (N > 1) every rank runs an independent replica (the products shard by rows without
any exchange); value is the sum over ranks divided by the slowest rank's time.
"""

from __future__ import annotations

import argparse
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from gemm_lb_gemv_02_b300 import synth  # noqa: E402

HEADLINE = "c4t"                 # the 27B-class ternary decode layer set
LAYERS = 8                       # distinct layer-set copies per step (8 x 85 MB >> L2)
L2_BYTES = 126 * 2 ** 20
# ncu DRAM bytes of the headline layer set, tied to the GEMV source they were measured on
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "gemv_traffic.json")
GEMV_SOURCE = os.path.join(ROOT, "gemm_lb_gemv_02_b300", "csrc", "lb_gemv.cu")
METRIC = "packed-weight GEMV HBM GB/s (% of peak) at batch 1; prefill GEMM TFLOP/s"


def _peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": d["hbm_gbs"], "bf16_tflops": d["bf16_tflops"],
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained"), "source": "measured"}
    return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ------------------------------------------------------------------------------------ dist
def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def _barrier(ws):
    if ws > 1:
        torch.distributed.barrier()


def _max_over_ranks(v: float, ws: int) -> float:
    if ws == 1:
        return v
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while active."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, busy_mhz_floor: float = 0.0):
        if not self.path or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((float(parts[1]), float(parts[2]), parts[3], parts[5:9]))
            except ValueError:
                continue
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i, v in enumerate(r[3]) if v.lower().startswith("active")})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------------------------------ helpers
def _copies_for(bytes_per_copy: int, minimum: int = 2) -> int:
    return max(minimum, -(-4 * L2_BYTES // max(1, bytes_per_copy)))


def _pack_workload(wl, lbt, storage=None):
    """Pack every matrix of a workload on the device (via the library's packers); storage
    "ternary5" stores a ternary workload's codes five per byte."""
    packed = []
    for i in range(len(wl.matrices)):
        inp = synth.matrix_inputs(wl, i)
        if wl.fmt == "1bit":
            packed.append(lbt.pack_1bit(inp["w"].cuda()))
        elif storage == "ternary5":
            packed.append(lbt.pack_ternary5(inp["t"].cuda(), inp["s"].cuda()))
        else:
            packed.append(lbt.pack_ternary(inp["t"].cuda(), inp["s"].cuda()))
    torch.cuda.synchronize()
    return packed


def _clone(pw):
    from gemm_lb_gemv_02_b300.tensors import PackedWeight
    return PackedWeight(pw.fmt, pw.n, pw.k, pw.codes.clone(), pw.scales.clone())


def _gemv_bytes(pw, batch):
    return pw.codes.numel() + pw.scales.numel() * 2 + 2 * batch * (pw.k + pw.n)


def _graph(fn):
    """Capture fn() (a sequence of library calls on the current stream) into a CUDA graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()                                    # eager run: loads modules, sets attributes
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _busy(g, seconds: float) -> None:
    """Replay graph g back to back for about `seconds` (one replay in flight at a time)."""
    t_end = time.perf_counter() + seconds
    while time.perf_counter() < t_end:
        g.replay()
        torch.cuda.synchronize()


def _time_graph(g, reps: int = 1) -> float:
    """Milliseconds per replay, CUDA events on the replay stream, synchronised on both sides."""
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for _ in range(reps):
        g.replay()
    e1.record()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / reps


# How a decoder layer issues its matrices: each inner list is one launch (lb_gemv for one matrix,
# lb_gemv_batched for several); the matrices of a launch read the same activations.
LAYER_GROUPING = {
    "c2": [["q", "k", "v"], ["o"], ["gate", "up"], ["down"]],
    "c4t": [["q"], ["o"], ["gate", "up"], ["down"]],
    "c4b": [["q"], ["o"], ["gate", "up"], ["down"]],
}


def grouping_of(wl, mode):
    """mode: 'separate' (one launch per matrix), 'layer' (LAYER_GROUPING), 'one' (a single launch)."""
    names = [m.name for m in wl.matrices]
    if mode == "separate" or wl.key not in LAYER_GROUPING:
        return [[i] for i in range(len(names))]
    if mode == "one":
        return [list(range(len(names)))]
    return [[names.index(n) for n in grp] for grp in LAYER_GROUPING[wl.key]]


class GemvSet:
    """Rotating copies of a workload's matrices; one 'step' runs every matrix of one copy, issued as
    the grouping says (matrices of one launch share the first one's activations)."""

    def __init__(self, wl, batch, lbt, copies=None, layers_per_step=None, grouping="separate", storage=None):
        self.wl, self.batch, self.lbt = wl, batch, lbt
        base = _pack_workload(wl, lbt, storage)
        per_copy = sum(_gemv_bytes(pw, batch) for pw in base)
        self.copies = copies or _copies_for(per_copy)
        self.sets = [base] + [[_clone(pw) for pw in base] for _ in range(self.copies - 1)]
        self.layers = layers_per_step or 1
        self.groups = grouping_of(wl, grouping)
        self.grouping = grouping
        own = [synth.workload_activations(wl, i, batch).cuda() for i in range(len(wl.matrices))]
        self.x = list(own)
        for grp in self.groups:                  # same-K members of a launch share one vector
            for i in grp:
                if wl.matrices[i].k == wl.matrices[grp[0]].k:
                    self.x[i] = own[grp[0]]
        self.y = [torch.empty(batch, m.n, dtype=self.x[i].dtype, device="cuda") for i, m in enumerate(wl.matrices)]
        self.bytes_per_layer = sum(_gemv_bytes(pw, batch) for pw in base) - sum(
            2 * batch * base[i].k for grp in self.groups for i in grp[1:]
            if self.x[i] is self.x[grp[0]])           # a shared x is read once
        self.launches_per_layer = len(self.groups)
        self.cursor = 0

    def run_layer(self, mats):
        for grp in self.groups:
            if len(grp) == 1:
                i = grp[0]
                self.lbt.gemv(mats[i], self.x[i], self.y[i])
            else:
                self.lbt.gemv_batched([(mats[i], self.x[i]) for i in grp], [self.y[i] for i in grp])

    def step(self):
        for _ in range(self.layers):
            self.run_layer(self.sets[self.cursor % self.copies])
            self.cursor += 1

    @property
    def bytes_per_step(self):
        return self.bytes_per_layer * self.layers


# ------------------------------------------------------------------------------------ measurements
def _want(name, sel):
    return sel is None or any(name.startswith(p) for p in sel)


GEMV_ROWS = (  # row name, workload, batch, grouping[, storage]
    ("gemv_c1_b1", "c1", 1, "separate"),
    ("gemv_c2_b1", "c2", 1, "layer"),
    ("gemv_c2_b1_7launches", "c2", 1, "separate"),
    ("gemv_c2_b1_1launch", "c2", 1, "one"),
    ("gemv_c3_b1", "c3", 1, "separate"),
    ("gemv_c3_b4", "c3", 4, "separate"),
    ("gemv_c4t_b1", "c4t", 1, "layer"),
    ("gemv_c4t_b5", "c4t", 5, "layer"),
    ("gemv_c4b_b1", "c4b", 1, "layer"),
    ("gemv_c4b_b5", "c4b", 5, "layer"),
    ("gemv_c4t_b1_5launches", "c4t", 1, "separate"),
    ("gemv_c2_b1_ternary5", "c2", 1, "layer", "ternary5"),
    ("gemv_c2_b1_ternary5_7launches", "c2", 1, "separate", "ternary5"),
    ("gemv_c4t_b1_ternary5", "c4t", 1, "layer", "ternary5"),
    ("gemv_c4t_b1_ternary5_5launches", "c4t", 1, "separate", "ternary5"),
    ("gemv_c4t_b5_ternary5_5launches", "c4t", 5, "separate", "ternary5"),
)


def measure_gemv_rows(lbt, peaks, sel=None):
    rows = {}
    for name, key, b, grouping, *storage in GEMV_ROWS:
        wl = synth.WORKLOADS[key]
        if not _want(name, sel):
            continue
        st = storage[0] if storage else None
        gs = GemvSet(wl, b, lbt, grouping=grouping, storage=st)
        steps = gs.copies * 2
        g = _graph(lambda: [gs.step() for _ in range(steps)])
        _time_graph(g)
        ms = _time_graph(g, reps=3) / steps
        gbs = gs.bytes_per_step / (ms * 1e-3) / 1e9
        rows[name] = {
            "shape": [[m.n, m.k] for m in wl.matrices], "fmt": st or wl.fmt, "x": wl.xdtype, "batch": b,
            "launches": [[wl.matrices[i].name for i in grp] for grp in gs.groups],
            "us_per_layer_set": round(ms * 1e3, 3), "GB_s": round(gbs, 1),
            "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 3),
            "frac_of_8TBs_nominal": round(gbs / 8000.0, 3), "copies_rotated": gs.copies}
        del gs, g
        torch.cuda.empty_cache()
    return rows


def measure_pack_rows(lbt, peaks, sel=None):
    rows = {}
    if not _want("pack", sel):
        return rows
    wl = synth.WORKLOADS["c1"]
    w = synth.matrix_inputs(wl, 0)["w"]
    reps = 48                                            # 48 distinct 16 MB inputs > 4x L2
    ws = [w.cuda().clone() for _ in range(reps)]
    outs = [lbt.PackedWeight.empty(1, 2048, 2048) for _ in range(reps)]
    torch.cuda.synchronize()
    from gemm_lb_gemv_02_b300 import lb as lbl
    for i in range(reps):                                # warm
        lbl.lb_pack_1bit(ws[i], 2048, 2048, outs[i].codes, outs[i].scales)
    t0 = time.perf_counter()
    for i in range(reps):
        lbl.lb_pack_1bit(ws[i], 2048, 2048, outs[i].codes, outs[i].scales)
    dt = (time.perf_counter() - t0) / reps
    by = 2048 * 2048 * 4 + 2048 * 2048 // 8 + 2048 * 16 * 2
    rows["pack_1bit_c1"] = {"shape": [2048, 2048], "us_per_call_incl_sync": round(dt * 1e6, 1),
                            "GB_s_incl_sync": round(by / dt / 1e9, 1),
                            "note": "synchronous call (reads the validation word back); host wall time"}
    del ws, outs
    wl = synth.WORKLOADS["c5"]
    inp = synth.matrix_inputs(wl, 0)
    t, s = inp["t"].cuda(), inp["s"].cuda()
    n, k = t.shape
    out = lbt.PackedWeight.empty(2, n, k)
    for _ in range(2):
        lbl.lb_pack_ternary(t, s, n, k, out.codes, out.scales)
    reps = 10
    t0 = time.perf_counter()
    for _ in range(reps):
        lbl.lb_pack_ternary(t, s, n, k, out.codes, out.scales)
    dt = (time.perf_counter() - t0) / reps
    by = n * k + n * k // 4 + 2 * n * (k // 128) * 2
    rows["pack_ternary_c5"] = {"shape": [n, k], "us_per_call_incl_sync": round(dt * 1e6, 1),
                               "GB_s_incl_sync": round(by / dt / 1e9, 1),
                               "note": "synchronous call (reads the validation word back); host wall time"}
    return rows


GEMM_ROWS = (
    # name, workload, matrix index, tokens
    ("gemm_c5", "c5", 0, 512),
    ("gemm_c4b_1bit_gate", "c4b", 2, 512),
    ("gemm_c5_m8", "c5", 0, 8),
    ("gemm_c5_m16", "c5", 0, 16),
    ("gemm_c5_m32", "c5", 0, 32),
    ("gemm_c5_m64", "c5", 0, 64),
    ("gemm_c5_m128", "c5", 0, 128),
)


def _gemm_one(lbt, peaks, wl_key, index, m):
    wl = synth.WORKLOADS[wl_key]
    base = _pack_workload(wl, lbt)[index]
    x = synth.workload_activations(wl, index, m).cuda()
    wbytes = _gemv_bytes(base, 0)
    per_copy = wbytes + x.numel() * 2 + m * base.n * 2
    copies = _copies_for(per_copy)
    ws = [base] + [_clone(base) for _ in range(copies - 1)]
    xs = [x.clone() for _ in range(copies)]
    y = torch.empty(m, base.n, dtype=torch.bfloat16, device="cuda")
    wsp = torch.empty(lbt.lb.lb_gemm_workspace_bytes(m, base.n, base.k, lbt.lb.LB_BF16), dtype=torch.uint8,
                      device="cuda")
    steps = copies * 2
    g = _graph(lambda: [lbt.gemm(ws[i % copies], xs[i % copies], torch.bfloat16, y, wsp) for i in range(steps)])
    _time_graph(g)
    ms = _time_graph(g, reps=3) / steps
    flops = 2.0 * m * base.n * base.k
    tf = flops / (ms * 1e-3) / 1e12
    return {"format": wl.fmt, "shape": [m, base.k, base.n], "us_per_gemm": round(ms * 1e3, 2),
            "TFLOP_s": round(tf, 1), "frac_of_measured_bf16_burst": round(tf / peaks["bf16_tflops"], 3),
            "frac_of_measured_bf16_sustained": round(tf / peaks["bf16_tflops_sustained"], 3)
            if peaks.get("bf16_tflops_sustained") else None,
            "weight_GB_s": round(wbytes / (ms * 1e-3) / 1e9, 1),
            "includes": "activation conversion prologue + GEMM kernel", "copies_rotated": copies}


def measure_gemm_row(lbt, peaks, sel=None):
    rows = {}
    for name, wl_key, index, m in GEMM_ROWS:
        if _want(name, sel):
            rows[name] = _gemm_one(lbt, peaks, wl_key, index, m)
    return rows


def measure_copy_reference(peaks, sel=None):
    """Context for the GEMV rows: a plain device-to-device copy (cudaMemcpyAsync through torch) of
    44 MB, the LM-head GEMV's byte count, rotated over buffers larger than L2.  The measured peak
    comes from a 4 GB copy; one launch of this size pays its ramp-up and tail."""
    name = "ref_copy_44MB"
    if not _want(name, sel):
        return {}
    nb = 44 * 1000 * 1000
    copies = _copies_for(2 * nb)
    src = [torch.empty(nb, dtype=torch.uint8, device="cuda") for _ in range(copies)]
    dst = [torch.empty(nb, dtype=torch.uint8, device="cuda") for _ in range(copies)]
    steps = copies * 2
    g = _graph(lambda: [dst[i % copies].copy_(src[i % copies]) for i in range(steps)])
    _time_graph(g)
    ms = _time_graph(g, reps=3) / steps
    gbs = 2 * nb / (ms * 1e-3) / 1e9
    del src, dst, g
    torch.cuda.empty_cache()
    return {name: {"bytes_read_plus_written": 2 * nb, "us_per_copy": round(ms * 1e3, 2), "GB_s": round(gbs, 1),
                   "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 3),
                   "note": "library copy, not this library's kernel: the bandwidth one launch of this size reaches"}}


def measure_read_probe_rows(lbt, peaks, sel=None):
    """The practical read ceiling of one launch: lb_read_probe (plain 16-byte loads, the GEMV's
    launch behaviour) over the byte counts of the headline's launches and of the LM-head GEMV,
    rotated over > 4x L2 and graph-timed exactly like the GEMV rows.  The layer-set row issues the
    headline's four byte counts in sequence, as the headline issues its four launches."""
    from gemm_lb_gemv_02_b300 import lb as lbl
    rows = {}
    wl = synth.WORKLOADS[HEADLINE]
    mats = {m.name: m for m in wl.matrices}

    def gemv_bytes(names, batch=1):
        by = 0
        for nm in names:
            m = mats[nm]
            cb, sb = lbl.lb_packed_bytes(lbl.FORMATS[wl.fmt], m.n, m.k)
            by += cb + sb + 2 * batch * m.n
        return by + 2 * batch * mats[names[0]].k
    c3 = synth.WORKLOADS["c3"].matrices[0]
    cb3, sb3 = lbl.lb_packed_bytes(lbl.LB_FMT_1BIT_G128, c3.n, c3.k)
    launches = [gemv_bytes(grp) for grp in LAYER_GROUPING[HEADLINE]]
    cases = [("read_probe_c3_44MB", [cb3 + sb3 + 2 * (c3.n + c3.k)])]
    cases += [(f"read_probe_{HEADLINE}_{'_'.join(grp)}", [b]) for grp, b in zip(LAYER_GROUPING[HEADLINE], launches)]
    cases.append((f"read_probe_{HEADLINE}_layer_set", launches))
    sink = torch.zeros(4, dtype=torch.int32, device="cuda")
    for name, sizes in cases:
        if not _want(name, sel):
            continue
        sizes = [(b + 15) // 16 * 16 for b in sizes]
        copies = _copies_for(sum(sizes))
        bufs = [[torch.empty(b, dtype=torch.uint8, device="cuda") for b in sizes] for _ in range(copies)]
        steps = copies * 2
        g = _graph(lambda: [lbl.lb_read_probe(buf, buf.numel(), sink) for i in range(steps) for buf in bufs[i % copies]])
        _time_graph(g)
        ms = _time_graph(g, reps=3) / steps
        gbs = sum(sizes) / (ms * 1e-3) / 1e9
        rows[name] = {"bytes_per_launch": sizes, "us_per_step": round(ms * 1e3, 3), "GB_s": round(gbs, 1),
                      "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 3), "copies_rotated": copies,
                      "note": "read-only reference launch (no compute), not the method's work"}
        del bufs, g
        torch.cuda.empty_cache()
    return rows


SWIGLU_ROWS = (  # row name, workload, batch[, storage]
    ("swiglu_c2_b1", "c2", 1),
    ("swiglu_c4t_b1", "c4t", 1),
    ("swiglu_c4t_b5", "c4t", 5),
    ("swiglu_c4t_b1_ternary5", "c4t", 1, "ternary5"),
)


def measure_swiglu_rows(lbt, peaks, sel=None):
    """The feed-forward gate / up pair: h = silu(W_gate x) * (W_up x) in one fused launch, against
    the same pair issued as one grouped launch of two GEMVs (g and u written out)."""
    rows = {}
    for name, key, b, *storage in SWIGLU_ROWS:
        if not _want(name, sel):
            continue
        wl = synth.WORKLOADS[key]
        idx = [next(i for i, m in enumerate(wl.matrices) if m.name == nm) for nm in ("gate", "up")]
        base = []
        for i in idx:
            inp = synth.matrix_inputs(wl, i)
            if wl.fmt == "1bit":
                base.append(lbt.pack_1bit(inp["w"].cuda()))
            elif storage and storage[0] == "ternary5":
                base.append(lbt.pack_ternary5(inp["t"].cuda(), inp["s"].cuda()))
            else:
                base.append(lbt.pack_ternary(inp["t"].cuda(), inp["s"].cuda()))
        per_copy = _gemv_bytes(base[0], b) + _gemv_bytes(base[1], b)
        copies = _copies_for(per_copy)
        pairs = [base] + [[_clone(pw) for pw in base] for _ in range(copies - 1)]
        x = synth.workload_activations(wl, idx[0], b).cuda()
        n = base[0].n
        h = torch.empty(b, n, dtype=x.dtype, device="cuda")
        yg, yu = torch.empty_like(h), torch.empty_like(h)
        steps = copies * 2
        g_f = _graph(lambda: [lbt.gemv_swiglu(pairs[i % copies][0], pairs[i % copies][1], x, h) for i in range(steps)])
        _time_graph(g_f)
        ms_f = _time_graph(g_f, reps=3) / steps
        g_u = _graph(lambda: [lbt.gemv_batched([(pairs[i % copies][0], x), (pairs[i % copies][1], x)], [yg, yu])
                              for i in range(steps)])
        _time_graph(g_u)
        ms_u = _time_graph(g_u, reps=3) / steps
        hc = torch.empty_like(h)

        def unfused_combined(i):                    # grouped launch + the silu(g) * u combine kernel
            lbt.gemv_batched([(pairs[i % copies][0], x), (pairs[i % copies][1], x)], [yg, yu])
            torch.mul(torch.nn.functional.silu(yg), yu, out=hc)

        g_c = _graph(lambda: [unfused_combined(i) for i in range(steps)])
        _time_graph(g_c)
        ms_c = _time_graph(g_c, reps=3) / steps
        by = per_copy - 2 * b * base[0].k - 2 * b * n     # x read once, one output vector
        gbs = by / (ms_f * 1e-3) / 1e9
        rows[name] = {"shape": [n, base[0].k], "fmt": storage[0] if storage else wl.fmt, "batch": b,
                      "us_per_pair": round(ms_f * 1e3, 2),
                      "GB_s": round(gbs, 1), "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 3),
                      "unfused_grouped_us": round(ms_u * 1e3, 2),
                      "unfused_grouped_plus_combine_us": round(ms_c * 1e3, 2),
                      "note": "unfused: one grouped launch writing g and u; plus_combine adds the "
                              "elementwise silu(g) * u (torch) the unfused path needs to produce h",
                      "copies_rotated": copies}
        del pairs, g_f, g_u, g_c
        torch.cuda.empty_cache()
    return rows


def measure_embed_rows(lbt, peaks, sel=None):
    """Embedding-row gather from the 1-bit 151936 x 2048 table: 32768 token ids (a long prefill),
    bfloat16 rows out (134 MB, larger than L2)."""
    name = "embed_c3_1bit_bf16_32k"
    if not _want(name, sel):
        return {}
    wl = synth.WORKLOADS["c3"]
    pw = _pack_workload(wl, lbt)[0]
    count = 32768
    g = torch.Generator().manual_seed(2024)
    ids = torch.randint(0, pw.n, (count,), generator=g, dtype=torch.int32).cuda()
    out = torch.empty(count, pw.k, dtype=torch.bfloat16, device="cuda")
    reps = 8
    gr = _graph(lambda: [lbt.embed(pw, ids, torch.bfloat16, out) for _ in range(reps)])
    _time_graph(gr)
    ms = _time_graph(gr, reps=3) / reps
    row_in = pw.k // 8 + 2 * (pw.k // 128)
    by = count * (row_in + 4 + 2 * pw.k)
    gbs = by / (ms * 1e-3) / 1e9
    return {name: {"table": [pw.n, pw.k], "fmt": "1bit", "tokens": count, "out": "bf16",
                   "us_per_call": round(ms * 1e3, 2), "GB_s": round(gbs, 1),
                   "frac_of_measured_hbm": round(gbs / peaks["hbm_gbs"], 3),
                   "bytes_basis": "codes + scales of each gathered row + ids + rows written"}}


# ------------------------------------------------------------------------------------ CPU oracle
# The oracle is timed on a bounded sample of the headline workload: the first 1/ORACLE_ROW_FRACTION of
# the rows of every matrix of one layer set (the same K, codes, scales and x as the GPU's), so that
# one pass is a fraction of a second.  The same sample serves the CPU-baseline leg and the
# reference arm.
ORACLE_ROW_FRACTION = 16


def _oracle_sample():
    from oracle import lb_oracle as orc
    wl = synth.WORKLOADS[HEADLINE]
    mats = []
    for i, m in enumerate(wl.matrices):
        inp = synth.matrix_inputs(wl, i)
        rows = m.n // ORACLE_ROW_FRACTION
        c, s = orc.pack_ternary(inp["t"][:rows].numpy(), inp["s"][:rows].numpy().view(np.uint16))
        x = orc.decode_activation_bits(synth.workload_activations(wl, i, 1).view(torch.int16).numpy().view(np.uint16),
                                       wl.xdtype)
        mats.append((c, s, m.k, x, c.nbytes + s.nbytes + 2 * (m.k + rows)))
    return mats


def _oracle_pass(mats) -> int:
    from oracle import lb_oracle as orc
    for c, s, k, x, _ in mats:
        orc.matvec(orc.FMT_TERNARY, c, s, k, x)
    return sum(m[4] for m in mats)


_ORACLE_MATS = None


def _oracle_init():
    """Per process: one BLAS thread, and the sample built once."""
    global _ORACLE_MATS
    try:
        from threadpoolctl import threadpool_limits
        threadpool_limits(1)
    except Exception:
        pass
    _ORACLE_MATS = _oracle_sample()
    _oracle_pass(_ORACLE_MATS)                               # warm (first allocations)


def _oracle_step(_=None) -> int:
    return _oracle_pass(_ORACLE_MATS)


def _oracle_timed(seconds: float):
    """Oracle passes over this process's sample for about `seconds`."""
    done, nbytes = 0, 0
    t0 = time.perf_counter()
    while time.perf_counter() - t0 < seconds or done == 0:
        nbytes += _oracle_pass(_ORACLE_MATS)
        done += 1
    return nbytes, time.perf_counter() - t0, done


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def cpu_model() -> str:
    try:
        for line in open("/proc/cpuinfo"):
            if line.startswith("model name"):
                return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


def cpu_baseline(seconds: float = 10.0):
    """The oracle as it stands, timed on the host cores: in one spawned process with one thread, then
    in one spawned process per core (so no process forks after the GPU was touched), each over the
    whole sample; GB/s of algorithmic bytes."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    with ctx.Pool(1, initializer=_oracle_init) as pool:
        nb1, dt1, _ = pool.apply(_oracle_timed, (seconds / 2,))
    cores = host_cores()
    with ctx.Pool(cores, initializer=_oracle_init) as pool:
        res = pool.map(_oracle_timed, [seconds / 2] * cores)
    wall = max(r[1] for r in res)
    return {"single_thread_GB_s": nb1 / dt1 / 1e9, "all_cores_GB_s": sum(r[0] for r in res) / wall / 1e9,
            "cores": cores, "passes_all_cores": sum(r[2] for r in res), "seconds": seconds}


# ------------------------------------------------------------------------------------ arms
def run_reference(args, ws, rank):
    if rank != 0:
        return
    import multiprocessing as mp
    cores = host_cores()
    # each step: one pass over the sample in every one of `cores` spawned processes
    with mp.get_context("spawn").Pool(cores, initializer=_oracle_init) as pool:
        for _ in range(args.warmup):
            pool.map(_oracle_step, range(cores), chunksize=1)
        t0 = time.perf_counter()
        nbytes = 0
        for _ in range(args.steps):
            nbytes += sum(pool.map(_oracle_step, range(cores), chunksize=1))
        dt = time.perf_counter() - t0
    v = nbytes / dt / 1e9
    sample = (f"1/{ORACLE_ROW_FRACTION} of the rows of each of the 5 matrices of the {HEADLINE} layer set per "
              f"process, {cores} spawned processes (one BLAS thread each), FP64 numpy oracle")
    line = {"impl": "reference", "metric": METRIC, "value": round(v, 3), "unit": "GB/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": _config(),
            "cpu_baseline": {"value": round(v, 3), "unit": "GB/s", "cores": cores, "kind": "oracle",
                             "sample": sample, "cpu": cpu_model()},
            "e2e": {"value": round(v, 3), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _config():
    return {"workload": f"{HEADLINE}: ternary g128 decode layer set of a 27B-class block (hidden 5120, FFN "
                        "17408: q, o 5120x5120; gate, up 17408x5120; down 5120x17408), batch 1, x bf16, FP32 "
                        f"accumulate; one step = one token through {LAYERS} distinct copies of the set, each "
                        "issued as a decoder layer issues it: [q], [o], [gate, up] on one x (one grouped "
                        "launch), [down]",
            "global_batch": 1, "layers_per_step": LAYERS, "parallelism": "replicas",
            "l2": f"inputs larger than L2: {LAYERS} rotated copies (> 4x 126 MB) per step",
            "seeds": f"synth.WORKLOADS['{HEADLINE}'].seed = {synth.WORKLOADS[HEADLINE].seed}"}


def _traffic_per_launch():
    """ncu DRAM bytes per headline launch, if they were measured on the current GEMV source."""
    import hashlib
    try:
        rec = json.load(open(TRAFFIC_FILE))
        sha = hashlib.sha256(open(GEMV_SOURCE, "rb").read()).hexdigest()
    except (OSError, ValueError):
        return None, "no capture on record"
    if rec.get("gemv_source_sha256") != sha:
        return None, "the GEMV source changed since the last capture"
    return rec.get("dram_bytes_per_launch"), rec.get("basis", "")


def run_ours(args, ws, rank, local):
    from gemm_lb_gemv_02_b300 import lb as lbl
    from gemm_lb_gemv_02_b300 import tensors as lbt
    torch.cuda.set_device(local)
    peaks = _peaks()
    wl = synth.WORKLOADS[HEADLINE]
    gs = GemvSet(wl, 1, lbt, copies=LAYERS, layers_per_step=LAYERS, grouping="layer")
    warm = _graph(lambda: [gs.step() for _ in range(max(1, args.warmup))])
    timed = _graph(lambda: [gs.step() for _ in range(args.steps)])
    timed.replay()                    # a graph's first launch uploads it: keep that out of the timing
    torch.cuda.synchronize()
    launches_per_layer = gs.launches_per_layer
    launches = args.steps * LAYERS * launches_per_layer

    with ClockSampler(local) as clocks:
        # soak: keep the same load running for ~1.5 s so that the sampler sees it (one replay in
        # flight at a time, so the soak ends when its time is up)
        _busy(warm, args.soak)
        torch.cuda.synchronize()
        _barrier(ws)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        timed.replay()
        e1.record()
        torch.cuda.synchronize()
        _barrier(ws)
        ms = e0.elapsed_time(e1)
        for _ in range(3):                       # keep loading while the sampler finishes its interval
            warm.replay()
        torch.cuda.synchronize()
    clk = clocks.summary()
    ms_max = _max_over_ranks(ms, ws)
    by_step = gs.bytes_per_step
    value = by_step * args.steps * ws / (ms_max * 1e-3) / 1e9
    per_rank_gbs = by_step * args.steps / (ms * 1e-3) / 1e9

    # end to end through the public API with host buffers: per step the token's activation
    # vectors (one per launch group) come from pinned host memory, all layers run eagerly through
    # lb_gemv / lb_gemv_batched, and the outputs of the last layer are read back
    heads = sorted({id(gs.x[i]): i for grp in gs.groups for i in grp}.values())   # distinct vectors
    xs_h = {i: gs.x[i].cpu().pin_memory() for i in heads}
    ys_h = [torch.empty(y.shape, dtype=y.dtype).pin_memory() for y in gs.y]
    h2d = sum(x.numel() * x.element_size() for x in xs_h.values())
    d2h = sum(y.numel() * y.element_size() for y in ys_h)
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        for i in heads:
            gs.x[i].copy_(xs_h[i], non_blocking=True)
        for layer in range(LAYERS):
            gs.run_layer(gs.sets[layer % gs.copies])
        for i in range(len(gs.y)):
            ys_h[i].copy_(gs.y[i], non_blocking=True)
        torch.cuda.current_stream().synchronize()

    # an idle GPU lowers its clocks, and the host-paced eager loop does not raise them again: bring
    # the GPU back to the working state of a serving loop with the same load first, then warm up
    _busy(warm, 0.3)
    for _ in range(max(3, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    e2e_dt = (time.perf_counter() - t0) / e2e_steps
    e2e_value = by_step / e2e_dt / 1e9

    # the same step as a serving loop issues it: the copies and all launches captured once into a
    # CUDA graph (through the same public calls), replayed per step; host wall clock, synchronised
    def e2e_body():
        for i in heads:
            gs.x[i].copy_(xs_h[i], non_blocking=True)
        for layer in range(LAYERS):
            gs.run_layer(gs.sets[layer % gs.copies])
        for i in range(len(gs.y)):
            ys_h[i].copy_(gs.y[i], non_blocking=True)

    e2e_graph = _graph(e2e_body)
    _busy(warm, 0.1)
    for _ in range(3):
        e2e_graph.replay()
        torch.cuda.current_stream().synchronize()
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_graph.replay()
        torch.cuda.current_stream().synchronize()
    e2e_graph_value = by_step / ((time.perf_counter() - t0) / e2e_steps) / 1e9
    del e2e_graph
    e2e_c = run_e2e_c(LAYERS, e2e_steps, max(3, args.warmup))

    del gs, warm, timed
    torch.cuda.empty_cache()
    rows = {}
    sel = None if args.rows == "all" else [r for r in args.rows.split(",") if r]
    if rank == 0 and not args.no_rows and args.rows != "none":
        rows.update(measure_pack_rows(lbt, peaks, sel))
        rows.update(measure_gemv_rows(lbt, peaks, sel))
        rows.update(measure_gemm_row(lbt, peaks, sel))
        rows.update(measure_embed_rows(lbt, peaks, sel))
        rows.update(measure_swiglu_rows(lbt, peaks, sel))
        rows.update(measure_read_probe_rows(lbt, peaks, sel))
        rows.update(measure_copy_reference(peaks, sel))
    assert lbl.lb_device_error(clear=True) == 0, "device error word set"

    if rank != 0:
        return
    cpu = cpu_baseline(args.cpu_seconds)
    traffic, traffic_basis = _traffic_per_launch()
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic", "config": _config(),
        "roofline": {"bound": "hbm", "achieved": round(per_rank_gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                     "frac": round(per_rank_gbs / peaks["hbm_gbs"], 4), "traffic": traffic,
                     "traffic_basis": traffic_basis,
                     "kernel": "gemv_kernel<ternary, bf16 x, batch 1> (4 launches per layer set: q, o, "
                               "gate/up grouped, down)",
                     "achieved_basis": "algorithmic bytes (packed codes + scales + x + y) per launch / "
                                       "(timed region / launches), CUDA events, so launch gaps count against it",
                     "algorithmic_bytes_per_launch": round(by_step / (LAYERS * launches_per_layer)),
                     "peak_basis": f"{peaks['source']} STREAM-style copy bandwidth"},
        "cpu_baseline": {"value": round(cpu["all_cores_GB_s"], 4), "unit": "GB/s", "cores": cpu["cores"],
                         "kind": "oracle", "cpu": cpu_model(),
                         "single_thread_value": round(cpu["single_thread_GB_s"], 4),
                         "sample": f"1/{ORACLE_ROW_FRACTION} of the rows of each matrix of the {HEADLINE} layer set, "
                                   f"FP64 numpy oracle; one spawned process per core with one BLAS thread each, "
                                   f"{cpu['passes_all_cores']} passes in {cpu['seconds'] / 2:.1f} s (value), and "
                                   "one process with one thread (single_thread_value)"},
        "e2e": {"value": round(e2e_value, 1), "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "per step: the activation vectors (one per launch group) copied from pinned host "
                       "memory, LAYERS x 4 eager lb_gemv / lb_gemv_batched calls through the Python binding, "
                       "the outputs copied back, one stream synchronize; host wall clock, after 0.3 s of "
                       "the same load and W warm-up steps (an idle GPU's lowered clocks are not raised "
                       "again by this host-paced loop)",
                "graph_value": round(e2e_graph_value, 1),
                "graph_how": "the same copies and calls captured once into a CUDA graph, one replay + "
                             "synchronize per step; host wall clock",
                "c_abi": e2e_c},
        "gpu_launches": launches,
        "clocks": clk,
        "peaks": peaks,
        "rows": rows,
    }
    print(json.dumps(line), flush=True)


def run_e2e_c(layers: int, steps: int, warmup: int):
    """The same end-to-end step from a plain C++ caller of the C ABI (gemm_lb_gemv_02_b300/e2e_c.cpp,
    compiled here against liblb.so): its GB/s and the host microseconds spent inside each lb_* call."""
    import subprocess
    pkg = os.path.join(ROOT, "gemm_lb_gemv_02_b300")
    src, exe = os.path.join(pkg, "e2e_c.cpp"), os.path.join(pkg, "_build", "e2e_c")
    lib = os.path.join(pkg, "liblb.so")
    try:
        if not os.path.exists(exe) or os.path.getmtime(exe) < max(os.path.getmtime(src), os.path.getmtime(lib)):
            os.makedirs(os.path.dirname(exe), exist_ok=True)
            subprocess.run(["nvcc", "-O2", "-std=c++17", "-I", os.path.join(ROOT, "include"), "-o", exe, src,
                            "-L" + pkg, "-llb", "-Xlinker", "-rpath=" + pkg], check=True, capture_output=True)
        r = subprocess.run([exe, str(layers), str(steps), str(warmup)], capture_output=True, text=True, timeout=300)
        if r.returncode != 0:
            return {"unavailable": (r.stderr or r.stdout).strip()[-300:]}
        out = json.loads(r.stdout.strip().splitlines()[-1])
        out["how"] = ("e2e_c.cpp: the same step (pinned host x in, 4 calls per layer, outputs back, one "
                      "stream synchronize) made by a C++ caller of include/lb.h; host wall clock; "
                      "host_us_per_call = time inside the lb_* calls / calls")
        return out
    except Exception as e:                                    # the line still prints without it
        return {"unavailable": f"{type(e).__name__}: {e}"[:300]}


def run_rows_only(args, local):
    from gemm_lb_gemv_02_b300 import tensors as lbt
    torch.cuda.set_device(local)
    peaks = _peaks()
    sel = [r for r in args.rows.split(",") if r] if args.rows not in ("all", "none") else None
    rows = {}
    rows.update(measure_gemv_rows(lbt, peaks, sel))
    rows.update(measure_gemm_row(lbt, peaks, sel))
    rows.update(measure_swiglu_rows(lbt, peaks, sel))
    rows.update(measure_read_probe_rows(lbt, peaks, sel))
    print(json.dumps({"rows_only": True, "rows": rows}), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-rows", action="store_true", help="skip the per-row measurements")
    ap.add_argument("--rows", default="all",
                    help="comma-separated prefixes of the rows to measure (pack, gemv_c3, gemm_c5, ...), "
                         "'all' or 'none'")
    ap.add_argument("--soak", type=float, default=1.5,
                    help="seconds of untimed load before the timed region (clock sampling)")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="oracle CPU-baseline duration")
    ap.add_argument("--rows-only", action="store_true",
                    help="measure only the rows selected by --rows and print them (no headline, e2e or CPU "
                         "leg); for profiling one kernel under ncu")
    args = ap.parse_args()
    ws, rank, local = _dist()
    if ws > 1:
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        torch.distributed.init_process_group(backend)
    try:
        if args.impl == "reference":
            run_reference(args, ws, rank)
        elif args.rows_only:
            run_rows_only(args, local)
        else:
            run_ours(args, ws, rank, local)
    finally:
        if ws > 1:
            torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
