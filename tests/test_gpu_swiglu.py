"""SiLU-gated feed-forward pair (lb_gemv_swiglu) on the GPU against the FP64 oracle."""

import numpy as np
import pytest
import torch

from gemm_lb_gemv_02_b300 import synth
from oracle import lb_oracle as orc
from tests.helpers import oracle_pack, u16

pytestmark = pytest.mark.gpu

lb = pytest.importorskip("gemm_lb_gemv_02_b300.lb")
from gemm_lb_gemv_02_b300 import tensors  # noqa: E402


def _inputs(fmt, n, k, seed):
    if fmt == "1bit":
        return {"w": synth.weights_fp32(n, k, 0.05, seed)}
    return {"t": synth.ternary_codes(n, k, seed), "s": synth.ternary_scales_bits(n, k, 0.02, seed + 1)}


def _device(fmt, inp):
    if fmt == "1bit":
        return tensors.pack_1bit(inp["w"].cuda())
    if fmt == "ternary5":
        return tensors.pack_ternary5(inp["t"].cuda(), inp["s"].cuda())
    return tensors.pack_ternary(inp["t"].cuda(), inp["s"].cuda())


def _oracle(fmt, inp, rows=None):
    sel = slice(None) if rows is None else rows
    if fmt == "1bit":
        return orc.pack_1bit(inp["w"].numpy()[sel])
    if fmt == "ternary5":
        return orc.pack_ternary5(inp["t"].numpy()[sel], inp["s"].numpy().view(np.uint16)[sel])
    return orc.pack_ternary(inp["t"].numpy()[sel], inp["s"].numpy().view(np.uint16)[sel])


def _check(fmt, ig, iu, h, x, rows=None):
    xdt = "bf16" if x.dtype == torch.bfloat16 else "f16"
    cg, sg = _oracle(fmt, ig, rows)
    cu, su = _oracle(fmt, iu, rows)
    xv = orc.decode_activation_bits(u16(x), xdt)
    f = {"1bit": orc.FMT_1BIT, "ternary": orc.FMT_TERNARY, "ternary5": orc.FMT_TERNARY5}[fmt]
    h_ref, g, a_g, u, a_u = orc.swiglu(f, cg, sg, cu, su, ig["w"].shape[1] if fmt == "1bit" else ig["t"].shape[1], xv)
    hv = orc.decode_activation_bits(u16(h), xdt)
    if rows is not None:
        hv = hv[:, rows]
    tol = orc.swiglu_tolerance(h_ref, g, a_g, u, a_u, hv, xdt)
    err = np.abs(hv - h_ref)
    worst = np.unravel_index(np.argmax(err / tol), err.shape)
    assert (err <= tol).all(), f"h {hv[worst]} vs {h_ref[worst]} (tol {tol[worst]}) at {worst}"


def _run_guarded(pg, pu, x):
    b, n = x.shape[0], pg.n
    pad = 64
    buf = torch.full((b * n + 2 * pad,), 12345, dtype=torch.int16, device="cuda")
    h = buf[pad:pad + b * n].view(x.dtype).view(b, n)
    tensors.gemv_swiglu(pg, pu, x, h)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 12345) and torch.all(buf[pad + b * n:] == 12345), "write outside h"
    assert lb.lb_device_error(clear=True) == 0
    return h


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
@pytest.mark.parametrize("xdt", ["f16", "bf16"])
@pytest.mark.parametrize("n,k", [(16, 128), (100, 384), (333, 1024), (64, 8192), (6144, 2048), (20, 49152)])
def test_swiglu_shapes(fmt, xdt, n, k):
    """Ragged row counts, one and many groups, a long K with few rows (split across a cluster),
    and the 1.7B-class gate/up shape."""
    ig, iu = _inputs(fmt, n, k, seed=n + k), _inputs(fmt, n, k, seed=n + k + 7)
    pg, pu = _device(fmt, ig), _device(fmt, iu)
    for batch in (1, 2, 5, 8):
        x = synth.activations(batch, k, xdt, seed=n + batch).cuda()
        h = _run_guarded(pg, pu, x)
        _check(fmt, ig, iu, h, x)


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
def test_swiglu_matches_two_gemvs(fmt):
    """The fused pair computes exactly what silu(lb_gemv(gate)) * lb_gemv(up) would, up to the
    rounding of the two intermediate vectors, which the fused path never stores."""
    n, k = 512, 2048
    ig, iu = _inputs(fmt, n, k, seed=3), _inputs(fmt, n, k, seed=4)
    pg, pu = _device(fmt, ig), _device(fmt, iu)
    x = synth.activations(1, k, "bf16", seed=5).cuda()
    h = _run_guarded(pg, pu, x)
    g = tensors.gemv(pg, x).float()
    u = tensors.gemv(pu, x).float()
    h2 = (g / (1 + torch.exp(-g)) * u).to(torch.bfloat16)
    _check(fmt, ig, iu, h, x)
    # both are close to each other within the bfloat16 rounding of g and u
    assert torch.allclose(h.float(), h2.float(), rtol=3e-2, atol=1e-3)


def test_swiglu_c4t_block_sampled():
    """The 27B-class ternary gate / up pair (17408 x 5120) at batch 1 and 5, outputs checked on
    sampled rows (the oracle packs only those rows)."""
    wl = synth.WORKLOADS["c4t"]
    gi = next(i for i, m in enumerate(wl.matrices) if m.name == "gate")
    ui = next(i for i, m in enumerate(wl.matrices) if m.name == "up")
    ig, iu = synth.matrix_inputs(wl, gi), synth.matrix_inputs(wl, ui)
    pg, pu = _device("ternary", ig), _device("ternary", iu)
    n = wl.matrices[gi].n
    rng = np.random.default_rng(8)
    rows = np.unique(np.concatenate([np.arange(8), np.arange(n - 8, n), rng.integers(0, n, 1200)]))
    for batch in (1, 5):
        x = synth.workload_activations(wl, gi, batch).cuda()
        h = tensors.gemv_swiglu(pg, pu, x)
        torch.cuda.synchronize()
        assert lb.lb_device_error(clear=True) == 0
        _check("ternary", ig, iu, h, x, rows=rows)


@pytest.mark.parametrize("xdt", ["f16", "bf16"])
@pytest.mark.parametrize("n,k", [(100, 1024), (333, 4096), (64, 16384), (6144, 2048)])
def test_swiglu_ternary5(xdt, n, k):
    """Five-per-byte gate / up at batch 1 (the lookup-table form with one table build for both
    units; 16384-wide K splits over a cluster).  Other batches and K not a multiple of 1024 are
    refused."""
    ig, iu = _inputs("ternary5", n, k, seed=n + k), _inputs("ternary5", n, k, seed=n + k + 7)
    pg, pu = _device("ternary5", ig), _device("ternary5", iu)
    x = synth.activations(1, k, xdt, seed=n + 1).cuda()
    h = _run_guarded(pg, pu, x)
    _check("ternary5", ig, iu, h, x)
    with pytest.raises(lb.LBError) as e:
        tensors.gemv_swiglu(pg, pu, synth.activations(2, k, xdt, seed=1).cuda())
    assert e.value.name == "LB_ERR_UNSUPPORTED"


def test_swiglu_ternary5_c4t_sampled():
    """The 27B-class gate / up pair stored five per byte at batch 1, sampled rows."""
    wl = synth.WORKLOADS["c4t"]
    gi = next(i for i, m in enumerate(wl.matrices) if m.name == "gate")
    ui = next(i for i, m in enumerate(wl.matrices) if m.name == "up")
    ig, iu = synth.matrix_inputs(wl, gi), synth.matrix_inputs(wl, ui)
    pg, pu = _device("ternary5", ig), _device("ternary5", iu)
    n = wl.matrices[gi].n
    rb = np.arange(0, n, 128)
    rng = np.random.default_rng(9)
    rows = np.unique(np.concatenate([rb, rb + 127, rng.integers(0, n, 600)]))
    x = synth.workload_activations(wl, gi, 1).cuda()
    h = tensors.gemv_swiglu(pg, pu, x)
    torch.cuda.synchronize()
    assert lb.lb_device_error(clear=True) == 0
    _check("ternary5", ig, iu, h, x, rows=rows)

