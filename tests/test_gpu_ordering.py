"""Launch order on one stream.  The GEMV family is launched with programmatic dependent launch: it
may start while the preceding kernel runs, reads x and writes y only after that kernel completed,
and streams the packed weights before (so the weights must not come from the immediately
preceding kernel; the synchronous packers satisfy that).  These tests issue the producers and
consumers of x, W and y back to back on one stream, with no copy or synchronisation in between,
and compare with the FP64 oracle."""

import numpy as np
import pytest
import torch

from gemm_lb_gemv_02_b300 import synth
from oracle import lb_oracle as orc
from tests.helpers import check_products, oracle_pack, oracle_products

pytestmark = pytest.mark.gpu

lb = pytest.importorskip("gemm_lb_gemv_02_b300.lb")
from gemm_lb_gemv_02_b300 import tensors  # noqa: E402


def _inputs(fmt, n, k, seed):
    if fmt == "1bit":
        return {"w": synth.weights_fp32(n, k, 0.05, seed)}
    return {"t": synth.ternary_codes(n, k, seed), "s": synth.ternary_scales_bits(n, k, 0.02, seed + 1)}


def _pack_on_device(fmt, inp):
    if fmt == "1bit":
        return tensors.pack_1bit(inp["w"].cuda())
    return tensors.pack_ternary(inp["t"].cuda(), inp["s"].cuda())


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
def test_pack_then_gemv_back_to_back(fmt):
    """x already on the device before packing; the GEMV follows the packer with nothing between."""
    n, k = 1100, 5120
    inp = _inputs(fmt, n, k, seed=21)
    x = synth.activations(1, k, "bf16", seed=22).cuda()
    y = torch.empty(1, n, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    pw = _pack_on_device(fmt, inp)
    tensors.gemv(pw, x, y)
    torch.cuda.synchronize()
    codes, scales = oracle_pack(fmt, inp)
    y_ref, a = oracle_products(fmt, codes, scales, k, x.cpu())
    check_products(y, y_ref, a, f"{fmt} pack then gemv")


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
def test_x_from_the_preceding_kernel(fmt):
    """x is written by a torch kernel immediately before the GEMV on the same stream."""
    n, k = 700, 2048
    inp = _inputs(fmt, n, k, seed=31)
    pw = _pack_on_device(fmt, inp)
    codes, scales = oracle_pack(fmt, inp)
    src = synth.activations(4, k, "f16", seed=32).cuda()
    x = torch.zeros(4, k, dtype=torch.float16, device="cuda")
    torch.cuda.synchronize()
    for rep in range(3):                                 # x changes every time, right before the GEMV
        torch.mul(src, float(rep + 1), out=x)
        y = tensors.gemv(pw, x)
        torch.cuda.synchronize()
        y_ref, a = oracle_products(fmt, codes, scales, k, x.cpu())
        check_products(y, y_ref, a, f"{fmt} x from the preceding kernel, rep {rep}")


def test_gemv_chain_through_y():
    """The second GEMV's x is the first GEMV's y: o(q(x)) on one stream, as a layer chains them."""
    n, k = 2048, 2048
    inp1, inp2 = _inputs("ternary", n, k, seed=41), _inputs("ternary", n, k, seed=43)
    pw1, pw2 = _pack_on_device("ternary", inp1), _pack_on_device("ternary", inp2)
    c1, s1 = oracle_pack("ternary", inp1)
    c2, s2 = oracle_pack("ternary", inp2)
    x = synth.activations(1, k, "bf16", seed=44).cuda()
    y1 = torch.empty(1, n, dtype=torch.bfloat16, device="cuda")
    y2 = torch.empty(1, n, dtype=torch.bfloat16, device="cuda")
    torch.cuda.synchronize()
    for _ in range(3):
        tensors.gemv(pw1, x, y1)
        tensors.gemv(pw2, y1, y2)
    total = y2.float().sum()                             # a consumer right after the second GEMV
    torch.cuda.synchronize()
    y_ref1, a1 = oracle_products("ternary", c1, s1, k, x.cpu())
    check_products(y1, y_ref1, a1, "first GEMV")
    y_ref2, a2 = oracle_products("ternary", c2, s2, k, y1.cpu())   # against the y1 the GPU produced
    check_products(y2, y_ref2, a2, "second GEMV (x = first y)")
    assert np.isclose(float(total), float(y2.float().cpu().double().sum()), rtol=1e-4, atol=1e-3)
