"""Streams and host threads: every entry point honours the stream it is given, and concurrent
calls from several host threads (each on its own stream) give the same bits as serial calls.
Every product here has a fixed reduction order, so repeated results are bit-identical."""

import threading

import numpy as np
import pytest
import torch

from gemm_lb_gemv_02_b300 import synth

pytestmark = pytest.mark.gpu

lb = pytest.importorskip("gemm_lb_gemv_02_b300.lb")
from gemm_lb_gemv_02_b300 import tensors  # noqa: E402


def _ternary(n, k, seed):
    return tensors.pack_ternary(synth.ternary_codes(n, k, seed).cuda(), synth.ternary_scales_bits(n, k, 0.02, seed + 1).cuda())


def _bits(t):
    return t.view(torch.int16).cpu().numpy()


def _all_products(pw, pu, x1, x5, xm, ids, stream=None):
    """Every product entry point once, on `stream` (None: torch's current stream)."""
    return [
        tensors.gemv(pw, x1, stream=stream),
        tensors.gemv(pw, x5, stream=stream),
        *tensors.gemv_batched([(pw, x1), (pu, x1)], stream=stream),
        tensors.gemv_swiglu(pw, pu, x1, stream=stream),
        tensors.gemm(pw, xm, stream=stream),
        tensors.embed(pw, ids, stream=stream),
    ]


def test_explicit_streams_match_default_stream():
    n, k = 512, 1024
    pw, pu = _ternary(n, k, 1), _ternary(n, k, 3)
    x1 = synth.activations(1, k, "bf16", seed=5).cuda()
    x5 = synth.activations(5, k, "bf16", seed=6).cuda()
    xm = synth.activations(70, k, "bf16", seed=7).cuda()
    ids = torch.tensor([0, 511, 7], dtype=torch.int32, device="cuda")
    ref = _all_products(pw, pu, x1, x5, xm, ids)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    out = _all_products(pw, pu, x1, x5, xm, ids, stream=s)        # passed explicitly
    s.synchronize()
    for a, b in zip(ref, out):
        assert np.array_equal(_bits(a), _bits(b))
    s2 = torch.cuda.Stream()
    s2.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s2):                                    # torch's current stream
        out2 = _all_products(pw, pu, x1, x5, xm, ids)
    s2.synchronize()
    for a, b in zip(ref, out2):
        assert np.array_equal(_bits(a), _bits(b))
    assert lb.lb_device_error(clear=True) == 0


def test_concurrent_host_threads():
    """Four host threads, each with its own weights and stream, 25 rounds of GEMV / grouped GEMV /
    GEMM each: the library's host caches (tensor maps, kernel attributes) are shared."""
    k = 2048
    work = []
    for t in range(4):
        pw, pu = _ternary(256 + 64 * t, k, 10 + 2 * t), _ternary(256 + 64 * t, k, 11 + 2 * t)
        x1 = synth.activations(1, k, "f16", seed=20 + t).cuda()
        xm = synth.activations(40 + t, k, "bf16", seed=30 + t).cuda()
        ref = [tensors.gemv(pw, x1), *tensors.gemv_batched([(pw, x1), (pu, x1)]), tensors.gemm(pw, xm)]
        work.append((pw, pu, x1, xm, ref))
    torch.cuda.synchronize()
    refs = [[_bits(r) for r in w[4]] for w in work]
    errors = []

    def run(t):
        try:
            pw, pu, x1, xm, _ = work[t]
            s = torch.cuda.Stream()
            for _ in range(25):
                outs = [tensors.gemv(pw, x1, stream=s), *tensors.gemv_batched([(pw, x1), (pu, x1)], stream=s),
                        tensors.gemm(pw, xm, stream=s)]
            s.synchronize()
            for a, b in zip(outs, refs[t]):
                if not np.array_equal(_bits(a), b):
                    errors.append(f"thread {t}: result differs")
        except Exception as e:                                     # reported below
            errors.append(f"thread {t}: {e!r}")

    threads = [threading.Thread(target=run, args=(t,)) for t in range(4)]
    for th in threads:
        th.start()
    for th in threads:
        th.join()
    assert not errors, errors
    assert lb.lb_device_error(clear=True) == 0
