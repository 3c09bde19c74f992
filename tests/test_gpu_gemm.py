"""Prefill GEMM (tcgen05) on the GPU against the FP64 oracle."""

import numpy as np
import pytest
import torch

from gemm_lb_gemv_02_b300 import synth
from oracle import lb_oracle as orc
from tests.helpers import check_products, oracle_pack, u16

pytestmark = pytest.mark.gpu

lb = pytest.importorskip("gemm_lb_gemv_02_b300.lb")
from gemm_lb_gemv_02_b300 import tensors  # noqa: E402


def _packed(fmt, n, k, seed):
    if fmt == "1bit":
        inp = {"w": synth.weights_fp32(n, k, 0.05, seed)}
        pw = tensors.pack_1bit(inp["w"].cuda())
    else:
        inp = {"t": synth.ternary_codes(n, k, seed), "s": synth.ternary_scales_bits(n, k, 0.02, seed + 1)}
        pw = tensors.pack_ternary(inp["t"].cuda(), inp["s"].cuda())
    codes, scales = oracle_pack(fmt, inp)
    return pw, codes, scales


def _check(pw, codes, scales, x, out_dtype, what, rows=None, cols=None):
    y = tensors.gemm(pw, x.cuda(), out_dtype=out_dtype)
    torch.cuda.synchronize()
    assert lb.lb_device_error(clear=True) == 0
    xs = x if rows is None else x[rows]
    c, s = (codes, scales) if cols is None else (codes[cols], scales[cols])
    xv = orc.decode_activation_bits(u16(xs), "bf16" if x.dtype == torch.bfloat16 else "f16")
    fmt = orc.FMT_1BIT if pw.fmt == lb.LB_FMT_1BIT_G128 else orc.FMT_TERNARY
    y_ref, a = orc.gemm(fmt, c, s, pw.k, xv)
    yd = y if rows is None else y[torch.as_tensor(rows, device=y.device)]
    return check_products(yd, y_ref, a, what, cols=cols)


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
@pytest.mark.parametrize("m,n,k", [(1, 256, 128), (5, 16, 256), (128, 256, 384), (130, 272, 256),
                                   (300, 512, 640), (64, 48, 1024)])
@pytest.mark.parametrize("xdt", ["bf16", "f16"])
def test_gemm_small_shapes(fmt, m, n, k, xdt):
    pw, codes, scales = _packed(fmt, n, k, seed=m + n + k)
    x = synth.activations(m, k, xdt, seed=m * 3 + k)
    for out in (torch.bfloat16, torch.float16):
        _check(pw, codes, scales, x, out, f"gemm {fmt} m={m} n={n} k={k} x={xdt} y={out}")


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
@pytest.mark.parametrize("m", [2, 9, 16, 17, 33, 100, 127, 129, 255, 256, 257, 383])
def test_gemm_token_counts(fmt, m):
    """Token counts around every width the tensor-core product takes (multiples of 16 up to 256,
    one or two 128-token tiles, a trailing tile of 1 token)."""
    n, k = 384, 768
    pw, codes, scales = _packed(fmt, n, k, seed=40 + m)
    x = synth.activations(m, k, "bf16", seed=41 + m)
    _check(pw, codes, scales, x, torch.bfloat16, f"gemm {fmt} m={m}")


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
def test_gemm_integer_exact(fmt):
    m, n, k = 200, 256, 512
    if fmt == "1bit":
        w = synth.weights_fp32(n, k, 1.0, seed=20)
        w[:, ::128] = 1.0                                          # group max |w| == 1 -> scale 1.0
        w = w.clamp(-1.0, 1.0)
        pw = tensors.pack_1bit(w.cuda())
        codes, scales = orc.pack_1bit(w.numpy())
        f = orc.FMT_1BIT
    else:
        t = synth.ternary_codes(n, k, seed=21)
        s = torch.full((n, k // 128), 0x3C00, dtype=torch.int16)
        pw = tensors.pack_ternary(t.cuda(), s.cuda())
        codes, scales = orc.pack_ternary(t.numpy(), s.numpy().view(np.uint16))
        f = orc.FMT_TERNARY
    assert np.all(scales == 0x3C00)
    g = torch.Generator().manual_seed(22)
    x = torch.randint(-3, 4, (m, k), generator=g).to(torch.bfloat16)
    y = tensors.gemm(pw, x.cuda(), out_dtype=torch.float16)
    torch.cuda.synchronize()
    y_ref, _ = orc.gemm(f, codes, scales, k, orc.bf16_bits_to_f64(u16(x)))
    assert np.array_equal(orc.f16_bits_to_f64(u16(y)), y_ref)


def test_gemm_c5_prefill_sampled():
    """The 512 x 5120 -> 17408 prefill workload at full size, outputs checked on sampled rows and
    columns (the whole GEMM runs; the oracle recomputes 96 token rows x 1200 weight rows)."""
    wl = synth.WORKLOADS["c5"]
    mat = wl.matrices[0]
    inp = synth.matrix_inputs(wl, 0)
    pw = tensors.pack_ternary(inp["t"].cuda(), inp["s"].cuda())
    x = synth.workload_activations(wl, 0, 512)
    codes, scales = oracle_pack("ternary", inp)
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 127, 128, 511], rng.integers(0, 512, 92)]))
    cols = np.unique(np.concatenate([np.arange(8), np.arange(mat.n - 8, mat.n), rng.integers(0, mat.n, 1184)]))
    _check(pw, codes, scales, x, torch.bfloat16, "c5 prefill", rows=rows, cols=cols)


def test_gemm_1bit_block_prefill_sampled():
    """A 1-bit 17408 x 5120 block matrix (the 5120 -> 17408 projection of the 1-bit block workload)
    as a 512-token prefill, outputs checked on sampled token rows and weight rows."""
    wl = synth.WORKLOADS["c4b"]
    idx = next(i for i, mt in enumerate(wl.matrices) if mt.n == 17408)
    mat = wl.matrices[idx]
    inp = synth.matrix_inputs(wl, idx)
    pw = tensors.pack_1bit(inp["w"].cuda())
    x = synth.workload_activations(wl, idx, 512)
    codes, scales = oracle_pack("1bit", inp)
    rng = np.random.default_rng(6)
    rows = np.unique(np.concatenate([[0, 255, 256, 511], rng.integers(0, 512, 60)]))
    cols = np.unique(np.concatenate([np.arange(8), np.arange(mat.n - 8, mat.n), rng.integers(0, mat.n, 600)]))
    _check(pw, codes, scales, x, torch.bfloat16, "1-bit block prefill", rows=rows, cols=cols)


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
def test_gemm_many_token_tiles(fmt):
    """4096 tokens (16 token tiles of 256) with a ragged row count; every output checked."""
    m, n, k = 4096, 400, 1024
    pw, codes, scales = _packed(fmt, n, k, seed=90)
    x = synth.activations(m, k, "bf16", seed=91)
    _check(pw, codes, scales, x, torch.bfloat16, f"gemm {fmt} m={m}")


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
def test_gemm_long_k(fmt):
    """K = 17536 (137 groups: the scale rows are not a multiple of 16 bytes, so the scales take
    the non-TMA path, and 274 pipeline stages), 300 tokens."""
    m, n, k = 300, 256, 17536
    pw, codes, scales = _packed(fmt, n, k, seed=92)
    x = synth.activations(m, k, "bf16", seed=93)
    _check(pw, codes, scales, x, torch.bfloat16, f"gemm {fmt} k={k}")


@pytest.mark.parametrize("fmt,m", [("ternary", 8), ("ternary", 16), ("ternary", 32), ("1bit", 12), ("1bit", 32)])
def test_gemm_small_m_block_matrix(fmt, m):
    """The few-token path (verification width, short prefill chunks) on a 17408 x 5120 block
    matrix: every token row, first / last and 1500 sampled weight rows."""
    key = "c5" if fmt == "ternary" else "c4b"
    wl = synth.WORKLOADS[key]
    idx = next(i for i, mt in enumerate(wl.matrices) if mt.n == 17408)
    mat = wl.matrices[idx]
    inp = synth.matrix_inputs(wl, idx)
    pw = tensors.pack_1bit(inp["w"].cuda()) if fmt == "1bit" else tensors.pack_ternary(inp["t"].cuda(), inp["s"].cuda())
    x = synth.workload_activations(wl, idx, m)
    codes, scales = oracle_pack(fmt, inp)
    rng = np.random.default_rng(7 + m)
    cols = np.unique(np.concatenate([np.arange(8), np.arange(mat.n - 8, mat.n), rng.integers(0, mat.n, 1500)]))
    _check(pw, codes, scales, x, torch.bfloat16, f"{key} m={m}", cols=cols)
