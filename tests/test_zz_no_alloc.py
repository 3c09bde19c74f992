"""lb_gemm_noalloc: the GEMM entry point for callers that cannot allocate device memory.

Plug-in style hosts that hand a kernel only its input and output buffers, and serving loops that
must not call cudaMalloc (it can synchronise the device), cannot give lb_gemm a workspace; this
entry point stages activations in a scratch array owned by the library instead.  The test calls it
through the C ABI twice in a row, on different inputs and for both formats, and checks each
result bit for bit against lb_gemm's on the same inputs and against the oracle's bound.  It is collected last so that a run
stopping at the first failure has already run everything else.
"""

import ctypes

import numpy as np
import pytest
import torch

from gemm_lb_gemv_02_b300 import synth
from oracle import lb_oracle as orc
from tests.helpers import u16

pytestmark = pytest.mark.gpu

lb = pytest.importorskip("gemm_lb_gemv_02_b300.lb")
from gemm_lb_gemv_02_b300 import tensors  # noqa: E402


def _noalloc(pw, x, out_dtype):
    y = torch.empty(x.shape[0], pw.n, dtype=out_dtype, device="cuda")
    W = pw.struct()
    st = lb.library().lb_gemm_noalloc(ctypes.byref(W), ctypes.c_void_p(x.data_ptr()),
                                      tensors.dtype_code(x.dtype), x.shape[0], ctypes.c_void_p(y.data_ptr()),
                                      tensors.dtype_code(out_dtype),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == lb.LB_OK, lb.lb_last_error()
    return y


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
def test_noalloc_matches_gemm_on_two_calls(fmt):
    """Same kernels, same staging layout: the result equals lb_gemm's bit for bit, and both are
    within the product bound of the oracle."""
    n, k = 512, 1280
    if fmt == "1bit":
        w = synth.weights_fp32(n, k, 0.05, seed=70)
        pw = tensors.pack_1bit(w.cuda())
        codes, scales = orc.pack_1bit(w.numpy())
        f = orc.FMT_1BIT
    else:
        t = synth.ternary_codes(n, k, seed=71)
        s = synth.ternary_scales_bits(n, k, 0.02, seed=72)
        pw = tensors.pack_ternary(t.cuda(), s.cuda())
        codes, scales = orc.pack_ternary(t.numpy(), s.numpy().view(np.uint16))
        f = orc.FMT_TERNARY
    for call, (m, xdt, out) in enumerate(((300, "bf16", torch.bfloat16), (130, "f16", torch.float16))):
        x = synth.activations(m, k, xdt, seed=73 + call).cuda()
        y_gemm = tensors.gemm(pw, x, out_dtype=out)          # the existing entry point
        y = _noalloc(pw, x, out)
        torch.cuda.synchronize()
        assert lb.lb_device_error(clear=True) == 0
        assert np.array_equal(u16(y), u16(y_gemm)), f"call {call}: noalloc differs from lb_gemm"
        dt = "bf16" if out == torch.bfloat16 else "f16"
        xv = orc.decode_activation_bits(u16(x), xdt)
        y_ref, a = orc.gemm(f, codes, scales, k, xv)
        yv = orc.decode_activation_bits(u16(y), dt)
        assert orc.within_tolerance(yv, y_ref, a, dt).all(), f"call {call}: outside the product bound"


def test_noalloc_rejects_oversized_request():
    n, k = 256, 16384
    pw = tensors.PackedWeight.empty(lb.LB_FMT_TERNARY_G128, n, k)
    m = lb.LB_GEMM_NOALLOC_SCRATCH_BYTES // (2 * k) + 129          # staging larger than the scratch
    assert lb.lb_gemm_workspace_bytes(m, n, k, lb.LB_BF16) > lb.LB_GEMM_NOALLOC_SCRATCH_BYTES
    x = torch.empty(m, k, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(m, n, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(lb.LBError) as e:
        lb.lb_gemm_noalloc(pw.struct(), x, lb.LB_BF16, m, y, lb.LB_BF16)
    assert e.value.name == "LB_ERR_WORKSPACE"
