"""Per-CTA phase trace of one GEMV launch inside a decoder layer's launch chain.

    python -m gemm_lb_gemv_02_b300.trace_gemv [--workload c4t] [--launch 2] [--batch 1]

Builds the phase-trace variant of the library (liblb_trace.so, compiled with -DLB_GEMV_TRACE; the
product library is not touched), packs the workload's matrices, runs the layer's launches (each
inner list of LAYERS is one launch) a few times to warm up, then clears the trace, runs the
launches 0 .. --launch once more on one stream (programmatic dependent launch between them, as in
the layer) and reads the trace, which then holds the last launch's events.  Prints a Markdown
summary: when the CTAs start, how long each phase takes (median and 10th / 90th percentile over
the CTAs), the steady-state stage period and the launch's span.

Durations inside a CTA come from clock64 (SM cycles); positions on the launch's time line come
from %globaltimer (ns), which all SMs share.
"""

from __future__ import annotations

import argparse
import ctypes
import os
import sys

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

LAYERS = {
    "c2": [["q", "k", "v"], ["o"], ["gate", "up"], ["down"]],
    "c4t": [["q"], ["o"], ["gate", "up"], ["down"]],
    "c4b": [["q"], ["o"], ["gate", "up"], ["down"]],
}
CTAS, EVENTS = 2048, 40
EV_START, EV_COPY0, EV_COPYN, EV_GRIDDEP, EV_PROLOGUE, EV_STAGE0, EV_UNIT0, EV_DONE, EV_END = 0, 1, 2, 3, 4, 5, 21, 29, 30
EV_P_INIT, EV_P_ARRIVED, EV_P_LOOP, EV_P_SLOT0 = 31, 32, 33, 34


def _pct(v, q):
    return float(np.percentile(v, q)) if len(v) else float("nan")


def summarize(tr: np.ndarray, clock_ghz: float) -> str:
    """tr: [CTAS][EVENTS][2] uint64 (globaltimer ns, clock64).  Markdown summary of the CTAs that
    recorded a start and an end."""
    ns, cyc = tr[:, :, 0].astype(np.int64), tr[:, :, 1].astype(np.int64)
    # CTA 0 always belongs to the traced (last) launch; CTAs whose events an earlier launch of
    # another grid shape wrote are left out
    grid = tr[:, EVENTS - 1, :]
    same = (grid[:, 0] == grid[0, 0]) & (grid[:, 1] == grid[0, 1])
    ncta = int(grid[0, 0] * grid[0, 1])
    live = np.flatnonzero(same & (np.arange(len(tr)) < ncta) & (ns[:, EV_START] > 0) & (ns[:, EV_END] > 0))
    if len(live) == 0:
        return "no CTA recorded a start and an end\n"
    ns, cyc = ns[live], cyc[live]
    # events an earlier launch of the chain left in slots this launch does not reach (fewer stages
    # or units) predate the CTA's start: drop them
    stale = ns < ns[:, EV_START:EV_START + 1]
    ns, cyc = np.where(stale, 0, ns), np.where(stale, 0, cyc)
    t0 = ns[:, EV_START].min()
    span = (ns[:, EV_END].max() - t0) / 1e3
    lines = [f"grid {int(grid[0, 0])} x {int(grid[0, 1])}; CTAs traced: {len(live)}; "
             f"launch span (first start .. last end): {span:.2f} us", "",
             "| phase | median | p10 | p90 |", "|---|---:|---:|---:|"]

    def row(name, v, unit):
        v = v[np.isfinite(v)]
        if len(v):
            lines.append(f"| {name} | {np.median(v):.2f} {unit} | {_pct(v, 10):.2f} | {_pct(v, 90):.2f} |")

    us = lambda a, b: np.where((ns[:, a] > 0) & (ns[:, b] > 0), (ns[:, b] - ns[:, a]) / 1e3, np.nan)
    kc = lambda a, b: np.where((cyc[:, a] > 0) & (cyc[:, b] > 0), (cyc[:, b] - cyc[:, a]) / 1e3, np.nan)
    row("CTA start after the first CTA's start", (ns[:, EV_START] - t0) / 1e3, "us")
    row("start -> producer's first copy issued", kc(EV_START, EV_COPY0), "kcyc")
    row("  producer: start -> barriers initialised and fenced", kc(EV_START, EV_P_INIT), "kcyc")
    row("  producer: -> past its start-up arrivals", kc(EV_P_INIT, EV_P_ARRIVED), "kcyc")
    row("  producer: -> at the start of its copy loop", kc(EV_P_ARRIVED, EV_P_LOOP), "kcyc")
    row("  producer: -> first slot granted", kc(EV_P_LOOP, EV_P_SLOT0), "kcyc")
    row("  producer: -> first copy issued", kc(EV_P_SLOT0, EV_COPY0), "kcyc")
    row("start -> consumers past griddepcontrol.wait", us(EV_START, EV_GRIDDEP), "us")
    row("griddepcontrol.wait -> x prologue done", kc(EV_GRIDDEP, EV_PROLOGUE), "kcyc")
    row("x prologue done -> first stage's data ready", kc(EV_PROLOGUE, EV_STAGE0), "kcyc")
    st = cyc[:, EV_STAGE0:EV_STAGE0 + 16].astype(np.float64)
    st[st == 0] = np.nan
    d = np.diff(st, axis=1)
    has = np.isfinite(d).any(axis=1)
    row("stage period (warp 0, stage i -> i+1)", np.nanmedian(d[has], axis=1) / 1e3, "kcyc")
    u = cyc[:, EV_UNIT0:EV_UNIT0 + 8].astype(np.float64)
    u[u == 0] = np.nan
    row("first stage ready -> first unit done", (u[:, 0] - cyc[:, EV_STAGE0]) / 1e3, "kcyc")
    two = np.isfinite(u[:, 1])
    row("first unit done -> second unit done", (u[two, 1] - u[two, 0]) / 1e3, "kcyc")
    row("consumers done -> CTA end", kc(EV_DONE, EV_END), "kcyc")
    row("producer: first -> last copy issued", kc(EV_COPY0, EV_COPYN), "kcyc")
    row("CTA start -> CTA end", kc(EV_START, EV_END), "kcyc")
    row("CTA end after the first CTA's start", (ns[:, EV_END] - t0) / 1e3, "us")
    lines.append("")
    lines.append(f"(kcyc = 1000 SM cycles, {1 / clock_ghz:.3f} us at the {clock_ghz:.2f} GHz maximum SM clock the device reports)")
    return "\n".join(lines) + "\n"


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="c4t", help="a layer workload (c2, c4t, c4b) or a single-matrix one (c1, c3)")
    ap.add_argument("--launch", type=int, default=2, help="index of the traced launch in the layer")
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--xdtype", choices=["bf16", "f16"], default=None,
                    help="activation type (default: the workload's own)")
    ap.add_argument("--ternary5", action="store_true",
                    help="store a ternary workload's codes five per byte")
    a = ap.parse_args()

    from gemm_lb_gemv_02_b300 import build
    lib_path = build.build(trace=True)
    os.environ["LB_LIBRARY"] = lib_path
    import torch

    from gemm_lb_gemv_02_b300 import lb, synth, tensors
    assert lb.LIB_PATH == lib_path, "the product library was loaded before the trace build"
    reader = ctypes.CDLL(lib_path).lb_gemv_trace_read
    reader.argtypes, reader.restype = [ctypes.c_void_p, ctypes.c_longlong], ctypes.c_longlong

    wl = synth.WORKLOADS[a.workload]
    names = [m.name for m in wl.matrices]
    packed = []
    for i in range(len(wl.matrices)):
        inp = synth.matrix_inputs(wl, i)
        if wl.fmt == "1bit":
            packed.append(tensors.pack_1bit(inp["w"].cuda()))
        else:
            pack = tensors.pack_ternary5 if a.ternary5 else tensors.pack_ternary
            packed.append(pack(inp["t"].cuda(), inp["s"].cuda()))
    layers = LAYERS.get(a.workload, [[n] for n in names])
    groups = [[names.index(n) for n in g] for g in layers]
    xs = {g[0]: synth.workload_activations(wl, g[0], a.batch).cuda() for g in groups}
    if a.xdtype:
        xs = {i: x.to(torch.bfloat16 if a.xdtype == "bf16" else torch.float16) for i, x in xs.items()}

    def launch(g):
        if len(g) == 1:
            tensors.gemv(packed[g[0]], xs[g[0]])
        else:
            tensors.gemv_batched([(packed[i], xs[g[0]]) for i in g])

    for _ in range(a.warmup):
        for g in groups:
            launch(g)
    torch.cuda.synchronize()
    buf = np.zeros((CTAS, EVENTS, 2), dtype=np.uint64)
    assert reader(buf.ctypes.data, buf.nbytes) == buf.nbytes            # clears the trace
    for g in groups[:a.launch + 1]:
        launch(g)
    torch.cuda.synchronize()
    assert reader(buf.ctypes.data, buf.nbytes) == buf.nbytes
    assert lb.lb_device_error(clear=True) == 0
    clock_ghz = torch.cuda.get_device_properties(0).clock_rate / 1e6 if hasattr(
        torch.cuda.get_device_properties(0), "clock_rate") else 1.92
    print(f"## GEMV phase trace: {a.workload}, launch {a.launch} "
          f"({'+'.join(layers[a.launch])}), batch {a.batch}, x {next(iter(xs.values())).dtype}"
          f"{', five per byte' if a.ternary5 else ''}\n")
    print(summarize(buf, clock_ghz))


if __name__ == "__main__":
    main()
