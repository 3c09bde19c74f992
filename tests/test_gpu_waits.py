"""The give-up path of the kernels' bounded pipeline waits, exercised without any GPU fault.

A test-only switch of the library (lb_testing_fault_next_launch, exported for this suite and not
declared in lb.h) makes the next GEMV or GEMM launch issue none of its asynchronous copies and bound
every mbarrier wait by 1 ms instead of 2 s.  Every wait then runs out: the kernel must set bit 0 of
the device error word, skip its compute, still join every barrier (cluster barriers included) and
release its tensor memory, and return.  The next normal launch must then give oracle-exact
results, which shows that nothing was left behind (no held TMEM, no stale barrier state)."""

import ctypes

import numpy as np
import pytest
import torch

from gemm_lb_gemv_02_b300 import synth
from oracle import lb_oracle as orc
from tests.helpers import check_products, oracle_pack, oracle_products, u16

pytestmark = pytest.mark.gpu

lb = pytest.importorskip("gemm_lb_gemv_02_b300.lb")
from gemm_lb_gemv_02_b300 import tensors  # noqa: E402

GEMV, GEMM = 1, 2


def _fault_next(kernel: int) -> None:
    fn = ctypes.CDLL(lb.LIB_PATH).lb_testing_fault_next_launch
    fn.argtypes, fn.restype = [ctypes.c_int], ctypes.c_int
    assert fn(kernel) == lb.LB_OK


def _packed(fmt, n, k, seed):
    if fmt == "1bit":
        inp = {"w": synth.weights_fp32(n, k, 0.05, seed)}
        pw = tensors.pack_1bit(inp["w"].cuda())
    else:
        inp = {"t": synth.ternary_codes(n, k, seed), "s": synth.ternary_scales_bits(n, k, 0.02, seed + 1)}
        pw = tensors.pack_ternary(inp["t"].cuda(), inp["s"].cuda())
    return pw, *oracle_pack(fmt, inp)


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
@pytest.mark.parametrize("n,k", [(300, 2176), (64, 8192)])     # persistent CTAs; K split across a cluster
def test_gemv_wait_gives_up_then_recovers(fmt, n, k):
    pw, codes, scales = _packed(fmt, n, k, seed=n + k)
    x = synth.activations(2, k, "bf16", seed=5).cuda()
    assert lb.lb_device_error(clear=True) == 0
    _fault_next(GEMV)
    tensors.gemv(pw, x)
    torch.cuda.synchronize()
    assert lb.lb_device_error(clear=True) & 1, "the waits did not give up"
    y = tensors.gemv(pw, x)
    torch.cuda.synchronize()
    assert lb.lb_device_error(clear=True) == 0
    y_ref, a = oracle_products(fmt, codes, scales, k, x.cpu())
    check_products(y, y_ref, a, f"{fmt} after a given-up launch")


def test_gemv_batched_wait_gives_up_then_recovers():
    shapes = [(300, 2176), (17, 640)]
    packed = [_packed("ternary", n, k, seed=n) for n, k in shapes]
    xs = [synth.activations(1, k, "f16", seed=k).cuda() for _, k in shapes]
    _fault_next(GEMV)
    tensors.gemv_batched([(pw, x) for (pw, _, _), x in zip(packed, xs)])
    torch.cuda.synchronize()
    assert lb.lb_device_error(clear=True) & 1
    ys = tensors.gemv_batched([(pw, x) for (pw, _, _), x in zip(packed, xs)])
    torch.cuda.synchronize()
    assert lb.lb_device_error(clear=True) == 0
    for (pw, codes, scales), (n, k), x, y in zip(packed, shapes, xs, ys):
        y_ref, a = oracle_products("ternary", codes, scales, k, x.cpu())
        check_products(y, y_ref, a, f"batched n={n} after a given-up launch")


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
@pytest.mark.parametrize("m", [40, 16])                       # the tensor-memory path; the few-token path
def test_gemm_wait_gives_up_then_recovers(fmt, m):
    n, k = 256, 1024
    pw, codes, scales = _packed(fmt, n, k, seed=3)
    x = synth.activations(m, k, "bf16", seed=4)
    assert lb.lb_device_error(clear=True) == 0
    _fault_next(GEMM)
    tensors.gemm(pw, x.cuda(), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert lb.lb_device_error(clear=True) & 1, "the waits did not give up"
    for _ in range(2):                        # TMEM was released: later launches allocate it again
        y = tensors.gemm(pw, x.cuda(), out_dtype=torch.bfloat16)
        torch.cuda.synchronize()
        assert lb.lb_device_error(clear=True) == 0
        f = orc.FMT_1BIT if fmt == "1bit" else orc.FMT_TERNARY
        y_ref, a = orc.gemm(f, codes, scales, k, orc.bf16_bits_to_f64(u16(x)))
        check_products(y, y_ref, a, f"gemm {fmt} after a given-up launch")
