"""Packers at every workload's own size: every matrix of every configuration is packed on the GPU
with the library's packers and compared byte for byte with the oracle's packing of the same raw
inputs (all rows for the 2048-wide workloads, the first, last and 1500 random rows of the 27B-class
matrices and of the prefill matrix)."""

import numpy as np
import pytest
import torch

from gemm_lb_gemv_02_b300 import synth
from oracle import lb_oracle as orc
from tests.helpers import u16, u8

pytestmark = pytest.mark.gpu

lb = pytest.importorskip("gemm_lb_gemv_02_b300.lb")
from gemm_lb_gemv_02_b300 import tensors  # noqa: E402


def _rows(n, sample):
    if sample is None or n <= sample:
        return np.arange(n)
    rng = np.random.default_rng(n)
    return np.unique(np.concatenate([[0, 1, n - 2, n - 1], rng.integers(0, n, sample)]))


@pytest.mark.parametrize("key,sample", [("c1", None), ("c2", None), ("c4t", 1500), ("c4b", 1500), ("c5", 1500)])
def test_pack_workload_bit_exact(key, sample):
    wl = synth.WORKLOADS[key]
    for i, mat in enumerate(wl.matrices):
        inp = synth.matrix_inputs(wl, i)
        if wl.fmt == "1bit":
            pw = tensors.pack_1bit(inp["w"].cuda())
            bytes_per_row = mat.k // 8
        else:
            pw = tensors.pack_ternary(inp["t"].cuda(), inp["s"].cuda())
            bytes_per_row = mat.k // 4
        torch.cuda.synchronize()
        codes = u8(pw.codes).reshape(mat.n, bytes_per_row)
        scales = u16(pw.scales).reshape(mat.n, mat.k // 128)
        rows = _rows(mat.n, sample)
        if wl.fmt == "1bit":
            rc, rs = orc.pack_1bit(inp["w"].numpy()[rows])
        else:
            rc, rs = orc.pack_ternary(inp["t"].numpy()[rows], inp["s"].numpy().view(np.uint16)[rows])
        assert np.array_equal(codes[rows], rc), f"{key}/{mat.name}: codes differ"
        assert np.array_equal(scales[rows], rs), f"{key}/{mat.name}: scales differ"
        del pw
