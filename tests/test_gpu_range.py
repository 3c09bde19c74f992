"""Activation range: every product against the FP64 oracle on inputs that span the numeric range of
binary16 and bfloat16 (largest finite values, 1e30, 1e5, groups that mix ~1e4 with ~1e-4, all-zero
rows, signed zeros, subnormal and tiny normal values).  The bound is the same as everywhere else,
|y - y_ref| <= 2e-3 * sum|s t x| + 1e-5 (+ half an ulp of the stored output)."""

import numpy as np
import pytest
import torch

from gemm_lb_gemv_02_b300 import synth
from oracle import lb_oracle as orc
from tests.helpers import check_products, u16

pytestmark = pytest.mark.gpu

lb = pytest.importorskip("gemm_lb_gemv_02_b300.lb")
from gemm_lb_gemv_02_b300 import tensors  # noqa: E402

FMAX = {"f16": 65504.0, "bf16": 3.3895313892515355e38}


def _packed(fmt, n, k, seed):
    """Weights whose products stay finite for the largest activations: 1-bit from N(0, 0.002^2),
    ternary scales |N(0, 0.02^2)|."""
    if fmt == "1bit":
        w = synth.weights_fp32(n, k, 0.002, seed)
        return tensors.pack_1bit(w.cuda()), orc.pack_1bit(w.numpy())
    t, s = synth.ternary_codes(n, k, seed), synth.ternary_scales_bits(n, k, 0.02, seed + 1)
    if fmt == "ternary5":
        return tensors.pack_ternary5(t.cuda(), s.cuda()), orc.pack_ternary5(t.numpy(), s.numpy().view(np.uint16))
    return tensors.pack_ternary(t.cuda(), s.cuda()), orc.pack_ternary(t.numpy(), s.numpy().view(np.uint16))


def _oracle(fmt, codes, scales, k, x):
    xdt = "bf16" if x.dtype == torch.bfloat16 else "f16"
    f = {"1bit": orc.FMT_1BIT, "ternary": orc.FMT_TERNARY, "ternary5": orc.FMT_TERNARY5}[fmt]
    y_ref, a = orc.matvec(f, codes, scales, k, orc.decode_activation_bits(u16(x.cpu()), xdt))
    assert np.all(np.abs(y_ref) + orc.tolerance(y_ref, a) < FMAX[xdt]), "test input overflows the output format"
    return y_ref, a


@pytest.mark.parametrize("fmt", ["1bit", "ternary", "ternary5"])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
@pytest.mark.parametrize("n,k", [(300, 2176), (1100, 5120)])
def test_gemv_wide_range(fmt, xdt, n, k):
    pw, (codes, scales) = _packed(fmt, n, k, seed=n + k)
    x8 = synth.activations_wide_range(8, k, xdt, seed=k + 3).cuda()
    for j in range(8):                                               # every row kind alone at batch 1
        x = x8[j:j + 1].contiguous()
        y = tensors.gemv(pw, x)
        torch.cuda.synchronize()
        y_ref, a = _oracle(fmt, codes, scales, k, x)
        check_products(y, y_ref, a, f"{fmt} {xdt} n={n} k={k} row kind {j}")
    for batch in (5, 8):                                             # mixed kinds in one launch
        x = x8[8 - batch:].contiguous() if batch == 5 else x8
        y = tensors.gemv(pw, x)
        torch.cuda.synchronize()
        y_ref, a = _oracle(fmt, codes, scales, k, x)
        check_products(y, y_ref, a, f"{fmt} {xdt} n={n} k={k} batch {batch}")
    assert lb.lb_device_error(clear=True) == 0


@pytest.mark.parametrize("fmt", ["1bit", "ternary", "ternary5"])
@pytest.mark.parametrize("batch", [1, 5])
def test_gemv_batched_wide_range(fmt, batch):
    shapes = [(300, 2176), (17, 640), (1100, 512)]
    packed = [_packed(fmt, n, k, seed=3 * n + k) for n, k in shapes]
    xs = [synth.activations_wide_range(8, k, "bf16", seed=n)[8 - batch:].contiguous().cuda() for n, k in shapes]
    ys = tensors.gemv_batched([(pw, x) for (pw, _), x in zip(packed, xs)])
    torch.cuda.synchronize()
    for (pw, (codes, scales)), (n, k), x, y in zip(packed, shapes, xs, ys):
        y_ref, a = _oracle(fmt, codes, scales, k, x)
        check_products(y, y_ref, a, f"batched {fmt} n={n} k={k} batch={batch}")
    assert lb.lb_device_error(clear=True) == 0


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
def test_swiglu_wide_range(fmt, xdt):
    """The row kinds whose h = silu(g) u stays finite in the output format: bfloat16 kinds 2..7 and
    binary16 kinds 1, 3..7 (the others hold elements large enough that g u overflows)."""
    n, k = 300, 2176
    pg, (cg, sg) = _packed(fmt, n, k, seed=5)
    pu, (cu, su) = _packed(fmt, n, k, seed=6)
    kinds = [2, 3, 4, 5, 6, 7] if xdt == "bf16" else [1, 3, 4, 5, 6, 7]
    x = synth.activations_wide_range(8, k, xdt, seed=9)[kinds].contiguous().cuda()
    h = tensors.gemv_swiglu(pg, pu, x)
    torch.cuda.synchronize()
    f = orc.FMT_1BIT if fmt == "1bit" else orc.FMT_TERNARY
    xv = orc.decode_activation_bits(u16(x.cpu()), xdt)
    h_ref, g, a_g, u, a_u = orc.swiglu(f, cg, sg, cu, su, k, xv)
    assert np.all(np.isfinite(h_ref)) and np.all(np.abs(h_ref) < FMAX[xdt] / 2)
    hv = orc.decode_activation_bits(u16(h), xdt)
    tol = orc.swiglu_tolerance(h_ref, g, a_g, u, a_u, hv, xdt)
    err = np.abs(hv - h_ref)
    worst = np.unravel_index(np.argmax(err / tol), err.shape)
    assert (err <= tol).all(), f"h {hv[worst]} vs {h_ref[worst]} (tol {tol[worst]}) at {worst}"
    assert lb.lb_device_error(clear=True) == 0


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
@pytest.mark.parametrize("m,n,k", [(40, 272, 640), (24, 1104, 5120)])
def test_gemm_wide_range(fmt, xdt, m, n, k):
    """Token rows cycle through the eight row kinds; the GEMM accepts every finite input."""
    pw, (codes, scales) = _packed(fmt, n, k, seed=m + n)
    x = synth.activations_wide_range(m, k, xdt, seed=k + 11)
    for out in (torch.bfloat16,) if xdt == "bf16" else (torch.float16, torch.bfloat16):
        y = tensors.gemm(pw, x.cuda(), out_dtype=out)
        torch.cuda.synchronize()
        assert lb.lb_device_error(clear=True) == 0
        y_ref, a = _oracle(fmt, codes, scales, k, x)
        if out == torch.float16:
            keep = np.all(np.abs(y_ref) + orc.tolerance(y_ref, a) < FMAX["f16"], axis=1)
            check_products(y[torch.as_tensor(np.flatnonzero(keep), device=y.device)], y_ref[keep], a[keep],
                           f"gemm {fmt} x={xdt} y=f16 m={m} n={n} k={k}")
        else:
            check_products(y, y_ref, a, f"gemm {fmt} x={xdt} y=bf16 m={m} n={n} k={k}")
