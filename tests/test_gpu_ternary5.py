"""Ternary codes stored five per byte: packer (bit-exact) and GEMV on the GPU against the oracle."""

import numpy as np
import pytest
import torch

from gemm_lb_gemv_02_b300 import synth
from oracle import lb_oracle as orc
from tests.helpers import check_products, u8, u16

pytestmark = pytest.mark.gpu

lb = pytest.importorskip("gemm_lb_gemv_02_b300.lb")
from gemm_lb_gemv_02_b300 import tensors  # noqa: E402


def _inputs(n, k, seed):
    return synth.ternary_codes(n, k, seed), synth.ternary_scales_bits(n, k, 0.02, seed + 1)


@pytest.mark.parametrize("n,k", [(1, 128), (7, 256), (33, 640), (300, 2048), (1000, 5120)])
def test_pack_ternary5_bit_exact(n, k):
    t, s = _inputs(n, k, seed=n + k)
    pw = tensors.pack_ternary5(t.cuda(), s.cuda())
    codes, scales = orc.pack_ternary5(t.numpy(), s.numpy().view(np.uint16))
    assert np.array_equal(u8(pw.codes).reshape(codes.shape), codes)
    assert np.array_equal(u16(pw.scales).reshape(scales.shape), scales)


def test_pack_ternary5_rejects_bad_code():
    t, s = _inputs(16, 256, seed=3)
    t[5, 200] = 2
    with pytest.raises(lb.LBError) as e:
        tensors.pack_ternary5(t.cuda(), s.cuda())
    assert e.value.name == "LB_ERR_CODE"


def _run_guarded(pw, x):
    b, n = x.shape[0], pw.n
    pad = 64
    buf = torch.full((b * n + 2 * pad,), 12345, dtype=torch.int16, device="cuda")
    y = buf[pad:pad + b * n].view(x.dtype).view(b, n)
    tensors.gemv(pw, x, y)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 12345) and torch.all(buf[pad + b * n:] == 12345), "write outside y"
    return y


@pytest.mark.parametrize("xdt", ["f16", "bf16"])
@pytest.mark.parametrize("n,k", [(1, 128), (7, 256), (65, 640), (300, 2176), (1000, 4096), (100, 17408)])
def test_gemv_ternary5_shapes(xdt, n, k):
    """Ragged row counts (CTAs of 64 rows), one group, a K that is not a multiple of the 2048-wide
    activation chunk, and long K; batch 1..8."""
    t, s = _inputs(n, k, seed=2 * n + k)
    pw = tensors.pack_ternary5(t.cuda(), s.cuda())
    codes, scales = orc.pack_ternary5(t.numpy(), s.numpy().view(np.uint16))
    for batch in (1, 2, 3, 4, 5, 6, 7, 8):
        x = synth.activations(batch, k, xdt, seed=n + batch).cuda()
        y = _run_guarded(pw, x)
        xv = orc.decode_activation_bits(u16(x), xdt)
        y_ref, a = orc.matvec(orc.FMT_TERNARY5, codes, scales, k, xv)
        check_products(y, y_ref, a, f"ternary5 {xdt} n={n} k={k} batch={batch}")


def test_gemv_ternary5_c4t_gate_sampled():
    """The 27B-class ternary gate matrix (17408 x 5120) in five-per-byte storage, batch 1 and 5,
    sampled rows (the oracle packs only those rows)."""
    wl = synth.WORKLOADS["c4t"]
    gi = next(i for i, m in enumerate(wl.matrices) if m.name == "gate")
    inp = synth.matrix_inputs(wl, gi)
    pw = tensors.pack_ternary5(inp["t"].cuda(), inp["s"].cuda())
    n, k = wl.matrices[gi].n, wl.matrices[gi].k
    rng = np.random.default_rng(12)
    rows = np.unique(np.concatenate([np.arange(8), np.arange(n - 8, n), rng.integers(0, n, 1500)]))
    codes, scales = orc.pack_ternary5(inp["t"].numpy()[rows], inp["s"].numpy().view(np.uint16)[rows])
    for batch in (1, 5):
        x = synth.workload_activations(wl, gi, batch).cuda()
        y = tensors.gemv(pw, x)
        torch.cuda.synchronize()
        y_ref, a = orc.matvec(orc.FMT_TERNARY5, codes, scales, k, orc.decode_activation_bits(u16(x), "bf16"))
        check_products(y, y_ref, a, f"c4t gate ternary5 batch={batch}", cols=rows)


def test_gemv_ternary5_integer_exact():
    """Scales 1 and small-integer x: every partial sum is an exactly representable integer."""
    n, k = 64, 1024
    t = synth.ternary_codes(n, k, seed=14)
    s = torch.full((n, k // 128), 0x3C00, dtype=torch.int16)
    pw = tensors.pack_ternary5(t.cuda(), s.cuda())
    codes, scales = orc.pack_ternary5(t.numpy(), s.numpy().view(np.uint16))
    g = torch.Generator().manual_seed(15)
    x = torch.randint(-4, 5, (3, k), generator=g).to(torch.float16)
    y = tensors.gemv(pw, x.cuda())
    torch.cuda.synchronize()
    y_ref, _ = orc.matvec(orc.FMT_TERNARY5, codes, scales, k, orc.f16_bits_to_f64(u16(x)))
    assert np.array_equal(orc.f16_bits_to_f64(u16(y)), y_ref)


@pytest.mark.parametrize("name", ["gate", "down"])
def test_gemv_ternary5_c4t_sampled_rows(name):
    """The 27B-class gate (17408 x 5120) and down (5120 x 17408) matrices in five-per-byte storage
    at batch 1 (lookup-table path; down splits K over 6-CTA clusters that take two row blocks
    each), sampled rows including the first and last of every row block."""
    wl = synth.WORKLOADS["c4t"]
    gi = next(i for i, m in enumerate(wl.matrices) if m.name == name)
    inp = synth.matrix_inputs(wl, gi)
    pw = tensors.pack_ternary5(inp["t"].cuda(), inp["s"].cuda())
    n, k = wl.matrices[gi].n, wl.matrices[gi].k
    x = synth.workload_activations(wl, gi, 1).cuda()
    y = tensors.gemv(pw, x)
    torch.cuda.synchronize()
    rb = np.arange(0, n, 128)
    rng = np.random.default_rng(16)
    rows = np.unique(np.concatenate([rb, rb + 127, rng.integers(0, n, 1000)]))
    codes, scales = orc.pack_ternary5(inp["t"].numpy()[rows], inp["s"].numpy().view(np.uint16)[rows])
    y_ref, a = orc.matvec(orc.FMT_TERNARY5, codes, scales, k, orc.decode_activation_bits(u16(x), "bf16"))
    check_products(y, y_ref, a, f"c4t {name} ternary5", cols=rows)


@pytest.mark.parametrize("batch", [1, 3])
def test_gemv_ternary5_batched(batch):
    """Grouped five-per-byte GEMVs: at batch 1 one lookup-table launch (problems sharing x and K run
    on persistent CTAs with one table build; the others one CTA per row block), at batch 3 one
    CUDA-core launch per problem.  Mixed n and k, a shared x."""
    specs = [(1000, 4096, 0), (700, 4096, 0), (300, 2048, 1)]
    xs = [synth.activations(batch, 4096, "bf16", seed=60).cuda(), synth.activations(batch, 2048, "bf16", seed=61).cuda()]
    pws, refs = [], []
    for i, (n, k, xi) in enumerate(specs):
        t, s = _inputs(n, k, seed=62 + i)
        pws.append(tensors.pack_ternary5(t.cuda(), s.cuda()))
        refs.append(orc.pack_ternary5(t.numpy(), s.numpy().view(np.uint16)))
    for group in ([0, 1], [0, 1, 2]):
        ys = tensors.gemv_batched([(pws[i], xs[specs[i][2]]) for i in group])
        torch.cuda.synchronize()
        for i, y in zip(group, ys):
            n, k, xi = specs[i]
            xv = orc.decode_activation_bits(u16(xs[xi]), "bf16")
            y_ref, a = orc.matvec(orc.FMT_TERNARY5, refs[i][0], refs[i][1], k, xv)
            check_products(y, y_ref, a, f"ternary5 batched {group} problem {i} batch={batch}")



def test_gemv_ternary5_many_row_blocks():
    """Five per byte at batch 1 with 299 row blocks on persistent CTAs, the last one ragged."""
    n, k = 299 * 128 - 77, 1024
    t, s = _inputs(n, k, seed=80)
    pw = tensors.pack_ternary5(t.cuda(), s.cuda())
    codes, scales = orc.pack_ternary5(t.numpy(), s.numpy().view(np.uint16))
    x = synth.activations(1, k, "bf16", seed=81).cuda()
    y = _run_guarded(pw, x)
    y_ref, a = orc.matvec(orc.FMT_TERNARY5, codes, scales, k, orc.decode_activation_bits(u16(x), "bf16"))
    check_products(y, y_ref, a, f"ternary5 {n}x{k} persistent")


def test_gemv_ternary5_c4t_gate_up_grouped():
    """The 27B-class gate and up matrices (17408 x 5120 each) stored five per byte in one grouped
    launch on one x at batch 1: persistent CTAs over both matrices' row blocks with one table
    build per CTA.  Sampled rows of both outputs, including every row block's first and last."""
    wl = synth.WORKLOADS["c4t"]
    idx = [next(i for i, m in enumerate(wl.matrices) if m.name == nm) for nm in ("gate", "up")]
    inps = [synth.matrix_inputs(wl, i) for i in idx]
    pws = [tensors.pack_ternary5(inp["t"].cuda(), inp["s"].cuda()) for inp in inps]
    x = synth.workload_activations(wl, idx[0], 1).cuda()
    ys = tensors.gemv_batched([(pw, x) for pw in pws])
    torch.cuda.synchronize()
    n, k = wl.matrices[idx[0]].n, wl.matrices[idx[0]].k
    rb = np.arange(0, n, 128)
    rng = np.random.default_rng(17)
    rows = np.unique(np.concatenate([rb, rb + 127, rng.integers(0, n, 600)]))
    xv = orc.decode_activation_bits(u16(x), "bf16")
    for name, inp, y in zip(("gate", "up"), inps, ys):
        codes, scales = orc.pack_ternary5(inp["t"].numpy()[rows], inp["s"].numpy().view(np.uint16)[rows])
        y_ref, a = orc.matvec(orc.FMT_TERNARY5, codes, scales, k, xv)
        check_products(y, y_ref, a, f"c4t {name} ternary5 grouped", cols=rows)
