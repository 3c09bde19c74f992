"""CPU checks of the GEMV phase-trace summary (gemm_lb_gemv_02_b300/trace_gemv.py): phase lengths
from a synthetic trace, and events that an earlier launch of the chain left behind are ignored."""

import numpy as np

from gemm_lb_gemv_02_b300 import trace_gemv as T


def _trace(ncta=4, stale=False):
    tr = np.zeros((T.CTAS, T.EVENTS, 2), dtype=np.uint64)
    tr[:ncta, T.EVENTS - 1, 0] = 1            # grid 1 x ncta
    tr[:ncta, T.EVENTS - 1, 1] = ncta
    for c in range(ncta):
        t_ns, t_cyc = 10_000_000 + 40 * c, 500_000 + 1000 * c
        stamps = {T.EV_START: 0, T.EV_P_INIT: 400, T.EV_P_ARRIVED: 550, T.EV_P_LOOP: 600,
                  T.EV_P_SLOT0: 700, T.EV_COPY0: 1100, T.EV_GRIDDEP: 900, T.EV_PROLOGUE: 2600,
                  T.EV_STAGE0: 3100, T.EV_STAGE0 + 1: 5900, T.EV_STAGE0 + 2: 8700,
                  T.EV_UNIT0: 9000, T.EV_DONE: 9100, T.EV_END: 10800, T.EV_COPYN: 2000}
        for ev, dc in stamps.items():          # cycles at 2 GHz: ns = cycles / 2
            tr[c, ev, 0] = t_ns + dc // 2
            tr[c, ev, 1] = t_cyc + dc
        if stale:                               # a later stage and a second unit of an earlier launch
            for ev in (T.EV_STAGE0 + 6, T.EV_UNIT0 + 1):
                tr[c, ev, 0] = 4_000_000
                tr[c, ev, 1] = 3
    return tr


def _rows(text):
    out = {}
    for line in text.splitlines():
        if line.startswith("| ") and not line.startswith("| phase") and not line.startswith("|---"):
            cells = [x.strip() for x in line.strip("|").split("|")]
            out[cells[0]] = float(cells[1].split()[0])
    return out


def test_phase_lengths():
    r = _rows(T.summarize(_trace(), 2.0))
    assert r["start -> producer's first copy issued"] == 1.1
    assert r["producer: start -> barriers initialised and fenced"] == 0.4
    assert r["producer: -> past its start-up arrivals"] == 0.15
    assert r["producer: -> first copy issued"] == 0.4
    assert r["griddepcontrol.wait -> x prologue done"] == 1.7
    assert r["stage period (warp 0, stage i -> i+1)"] == 2.8
    assert r["first stage ready -> first unit done"] == 5.9
    assert r["CTA start -> CTA end"] == 10.8


def test_stale_events_are_ignored():
    clean = T.summarize(_trace(), 2.0)
    dirty = T.summarize(_trace(stale=True), 2.0)
    assert dirty == clean
    assert "second unit done" not in dirty


def test_other_grid_is_left_out():
    tr = _trace(ncta=4)
    tr[2, T.EVENTS - 1, 1] = 99                 # CTA 2 last written by a launch of another grid
    assert "CTAs traced: 3" in T.summarize(tr, 2.0)
