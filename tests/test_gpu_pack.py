"""Packers on the GPU against the oracle: bit-exact codes and scales, and the error statuses."""

import numpy as np
import pytest
import torch

from gemm_lb_gemv_02_b300 import synth
from oracle import lb_oracle as orc
from tests.helpers import u16, u8

pytestmark = pytest.mark.gpu

lb = pytest.importorskip("gemm_lb_gemv_02_b300.lb")
from gemm_lb_gemv_02_b300 import tensors  # noqa: E402


def _pack1(w_cpu: torch.Tensor):
    pw = tensors.pack_1bit(w_cpu.cuda())
    torch.cuda.synchronize()
    n, k = w_cpu.shape
    return u8(pw.codes).reshape(n, k // 8), u16(pw.scales).reshape(n, k // 128)


@pytest.mark.parametrize("n,k", [(1, 128), (7, 384), (129, 256), (16, 2048), (33, 640)])
def test_pack_1bit_shapes(n, k):
    w = synth.weights_fp32(n, k, 0.1, seed=n * 1000 + k)
    codes, scales = _pack1(w)
    rc, rs = orc.pack_1bit(w.numpy())
    assert np.array_equal(codes, rc)
    assert np.array_equal(scales, rs)


def test_pack_1bit_edge_values():
    w = synth.weights_fp32(6, 256, 1.0, seed=5)
    w[0, :128] = 0.0                                  # all-zero group -> scale 0, all bits 1
    w[1, 3] = -0.0
    w[1, 4] = 0.0
    w[2, :128] = torch.tensor(np.float32(2.0 ** -130)) * torch.sign(w[2, :128])   # subnormal fp32
    w[3, 7] = 65519.0                                  # rounds down to 65504
    w[4, 9] = -6.0e-8                                  # binary16 subnormal scale region
    w[4, :128] *= 1e-7
    w[5, 200] = 1e-30
    codes, scales = _pack1(w)
    rc, rs = orc.pack_1bit(w.numpy())
    assert np.array_equal(codes, rc) and np.array_equal(scales, rs)
    assert scales[0, 0] == 0 and np.all(codes[0, :16] == 0xFF)
    assert scales[3, 0] == 0x7BFF


@pytest.mark.parametrize("bad,status", [(float("nan"), "LB_ERR_NONFINITE"), (float("inf"), "LB_ERR_NONFINITE"),
                                        (-float("inf"), "LB_ERR_NONFINITE"), (65520.0, "LB_ERR_RANGE"),
                                        (-1e6, "LB_ERR_RANGE")])
def test_pack_1bit_errors(bad, status):
    w = synth.weights_fp32(3, 256, 0.1, seed=9)
    w[2, 131] = bad
    with pytest.raises(lb.LBError) as e:
        tensors.pack_1bit(w.cuda())
    assert e.value.name == status
    # the library stays usable after an error
    codes, scales = _pack1(synth.weights_fp32(2, 128, 0.1, seed=10))
    rc, rs = orc.pack_1bit(synth.weights_fp32(2, 128, 0.1, seed=10).numpy())
    assert np.array_equal(codes, rc) and np.array_equal(scales, rs)


@pytest.mark.parametrize("n,k", [(1, 128), (7, 384), (129, 256), (64, 5120)])
def test_pack_ternary_shapes(n, k):
    t = synth.ternary_codes(n, k, seed=n + k)
    s = synth.ternary_scales_bits(n, k, 0.02, seed=n + k + 1)
    pw = tensors.pack_ternary(t.cuda(), s.cuda())
    torch.cuda.synchronize()
    rc, rs = orc.pack_ternary(t.numpy(), s.numpy().view(np.uint16))
    assert np.array_equal(u8(pw.codes).reshape(n, k // 4), rc)
    assert np.array_equal(u16(pw.scales).reshape(n, k // 128), rs)


@pytest.mark.parametrize("bad", [2, -2, 3, 127, -128])
def test_pack_ternary_bad_code(bad):
    t = synth.ternary_codes(4, 256, seed=3)
    t[3, 255] = bad
    s = synth.ternary_scales_bits(4, 256, 0.02, seed=4)
    with pytest.raises(lb.LBError) as e:
        tensors.pack_ternary(t.cuda(), s.cuda())
    assert e.value.name == "LB_ERR_CODE"


def test_pack_full_size_lm_head_sampled():
    """151936 x 2048 1-bit (the LM-head workload): all rows packed on the GPU, sampled rows
    (first, last and 2000 random) compared bit-exactly with the oracle."""
    wl = synth.WORKLOADS["c3"]
    w = synth.matrix_inputs(wl, 0)["w"]
    n, k = w.shape
    pw = tensors.pack_1bit(w.cuda())
    torch.cuda.synchronize()
    codes = u8(pw.codes).reshape(n, k // 8)
    scales = u16(pw.scales).reshape(n, k // 128)
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 1, n - 2, n - 1], rng.integers(0, n, 2000)]))
    rc, rs = orc.pack_1bit(w.numpy()[rows])
    assert np.array_equal(codes[rows], rc) and np.array_equal(scales[rows], rs)


def _config_matrices():
    out = []
    for key in ("c1", "c2", "c4t", "c4b", "c5"):
        wl = synth.WORKLOADS[key]
        for i, m in enumerate(wl.matrices):
            out.append((key, i, m.name))
    return out


@pytest.mark.parametrize("key,index,name", _config_matrices())
def test_pack_every_config_matrix(key, index, name):
    """Every matrix of every configuration at its own size, packed on the GPU with the library's
    packers and compared bit-exactly with the oracle's packing: whole matrices up to 4096 rows,
    otherwise the first, last and 1500 random rows.  Ternary matrices are also checked five per
    byte."""
    wl = synth.WORKLOADS[key]
    inp = synth.matrix_inputs(wl, index)
    n, k = wl.matrices[index].n, wl.matrices[index].k
    rng = np.random.default_rng(index + 7)
    rows = np.arange(n) if n <= 4096 else np.unique(np.concatenate([[0, 1, n - 2, n - 1], rng.integers(0, n, 1500)]))
    if wl.fmt == "1bit":
        codes, scales = _pack1(inp["w"])
        rc, rs = orc.pack_1bit(inp["w"].numpy()[rows])
        assert np.array_equal(codes[rows], rc) and np.array_equal(scales[rows], rs), f"{key}/{name} 1-bit"
        return
    t, s = inp["t"], inp["s"]
    packers = [(tensors.pack_ternary, orc.pack_ternary, 32), (tensors.pack_ternary5, orc.pack_ternary5, 26)]
    for dev_pack, ora_pack, gbytes in packers:
        pw = dev_pack(t.cuda(), s.cuda())
        torch.cuda.synchronize()
        codes = u8(pw.codes).reshape(n, (k // 128) * gbytes)
        scales = u16(pw.scales).reshape(n, k // 128)
        rc, rs = ora_pack(t.numpy()[rows], s.numpy().view(np.uint16)[rows])
        assert np.array_equal(codes[rows], rc) and np.array_equal(scales[rows], rs), f"{key}/{name} {gbytes} B/group"
        del pw
