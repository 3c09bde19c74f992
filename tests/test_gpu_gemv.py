"""Decode / small-batch GEMV on the GPU against the FP64 oracle (|y - y_ref| <= 2e-3 a + 1e-5)."""

import numpy as np
import pytest
import torch

from gemm_lb_gemv_02_b300 import synth
from oracle import lb_oracle as orc
from tests.helpers import check_products, oracle_pack, oracle_products, u16

pytestmark = pytest.mark.gpu

lb = pytest.importorskip("gemm_lb_gemv_02_b300.lb")
from gemm_lb_gemv_02_b300 import tensors  # noqa: E402

TDT = {"f16": torch.float16, "bf16": torch.bfloat16}


def _packed(fmt, n, k, seed):
    if fmt == "1bit":
        inp = {"w": synth.weights_fp32(n, k, 0.05, seed)}
        pw = tensors.pack_1bit(inp["w"].cuda())
    else:
        inp = {"t": synth.ternary_codes(n, k, seed), "s": synth.ternary_scales_bits(n, k, 0.02, seed + 1)}
        pw = tensors.pack_ternary(inp["t"].cuda(), inp["s"].cuda())
    codes, scales = oracle_pack(fmt, inp)
    return pw, codes, scales


def _run_guarded(pw, x):
    """gemv into the middle of a canary-filled buffer; checks the canaries afterwards."""
    b, n = x.shape[0], pw.n
    pad = 64
    buf = torch.full((b * n + 2 * pad,), 12345, dtype=torch.int16, device="cuda")
    y = buf[pad:pad + b * n].view(x.dtype).view(b, n)
    tensors.gemv(pw, x, y)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 12345) and torch.all(buf[pad + b * n:] == 12345), "write outside y"
    return y


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
@pytest.mark.parametrize("xdt", ["f16", "bf16"])
@pytest.mark.parametrize("n,k", [(1, 128), (7, 256), (16, 128), (17, 640), (100, 384), (333, 1024), (1100, 512),
                                 (300, 2176), (37893, 384)])
def test_gemv_small_shapes(fmt, xdt, n, k):
    pw, codes, scales = _packed(fmt, n, k, seed=n * 7 + k)
    for batch in (1, 2, 3, 5, 8):
        x = synth.activations(batch, k, xdt, seed=n + k + batch).cuda()
        y = _run_guarded(pw, x)
        y_ref, a = oracle_products(fmt, codes, scales, k, x.cpu())
        check_products(y, y_ref, a, f"{fmt} {xdt} n={n} k={k} batch={batch}")


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
@pytest.mark.parametrize("xdt", ["f16", "bf16"])
def test_gemv_integer_exact(fmt, xdt):
    """Scales 1 and small-integer x: every partial sum is an exactly representable integer, so the
    result must be exact (checks the decode offsets cancel exactly)."""
    n, k = 64, 512
    if fmt == "1bit":
        w = synth.weights_fp32(n, k, 1.0, seed=11)
        w[:, ::128] = 1.0                                          # group max |w| == 1 -> scale 1.0
        w = w.clamp(-1.0, 1.0)
        pw = tensors.pack_1bit(w.cuda())
        codes, scales = orc.pack_1bit(w.numpy())
    else:
        t = synth.ternary_codes(n, k, seed=12)
        s = torch.full((n, k // 128), 0x3C00, dtype=torch.int16)  # 1.0
        pw = tensors.pack_ternary(t.cuda(), s.cuda())
        codes, scales = orc.pack_ternary(t.numpy(), s.numpy().view(np.uint16))
    assert np.all(scales == 0x3C00)
    g = torch.Generator().manual_seed(13)
    x = torch.randint(-4, 5, (4, k), generator=g).to(TDT[xdt])
    y = tensors.gemv(pw, x.cuda())
    torch.cuda.synchronize()
    y_ref, _ = oracle_products(fmt, codes, scales, k, x)
    yv = orc.decode_activation_bits(u16(y), xdt)
    assert np.array_equal(yv, y_ref)


def _workload_check(key, batch, sample_rows=None):
    wl = synth.WORKLOADS[key]
    worst = 0.0
    for i, mat in enumerate(wl.matrices):
        inp = synth.matrix_inputs(wl, i)
        if wl.fmt == "1bit":
            pw = tensors.pack_1bit(inp["w"].cuda())
        else:
            pw = tensors.pack_ternary(inp["t"].cuda(), inp["s"].cuda())
        x = synth.workload_activations(wl, i, batch).cuda()
        y = tensors.gemv(pw, x)
        torch.cuda.synchronize()
        rows = None
        if sample_rows and mat.n > sample_rows:
            rng = np.random.default_rng(i)
            rows = np.unique(np.concatenate([np.arange(16), np.arange(mat.n - 16, mat.n),
                                             rng.integers(0, mat.n, sample_rows)]))
        # the oracle packs the checked rows itself from the raw inputs (packing is row by row)
        sel = slice(None) if rows is None else rows
        if wl.fmt == "1bit":
            codes, scales = orc.pack_1bit(inp["w"].numpy()[sel])
        else:
            codes, scales = orc.pack_ternary(inp["t"].numpy()[sel], inp["s"].numpy().view(np.uint16)[sel])
        y_ref, a = oracle_products(wl.fmt, codes, scales, mat.k, x.cpu())
        worst = max(worst, check_products(y, y_ref, a, f"{key}/{mat.name} batch={batch}", cols=rows))
        del pw, x, y
    return worst


def test_gemv_c1_full():
    _workload_check("c1", 1)


def test_gemv_c2_layer_set_full():
    _workload_check("c2", 1)


@pytest.mark.parametrize("batch", [1, 4])
def test_gemv_c3_lm_head(batch):
    _workload_check("c3", batch, sample_rows=3000)


@pytest.mark.parametrize("key", ["c4t", "c4b"])
@pytest.mark.parametrize("batch", [1, 5])
def test_gemv_c4_layer_set(key, batch):
    _workload_check(key, batch, sample_rows=1500)


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
@pytest.mark.parametrize("xdt", ["f16", "bf16"])
@pytest.mark.parametrize("batch", [1, 3, 8])
def test_gemv_batched_mixed_shapes(fmt, xdt, batch):
    """One grouped launch over problems of different n and k (ragged row blocks, partial stages,
    group counts that are not multiples of 8), some sharing one x: each y matches the oracle and
    nothing is written outside any y."""
    shapes = [(300, 2176), (17, 640), (1100, 512), (129, 128), (2048, 1024)]
    packed = [_packed(fmt, n, k, seed=n + 3 * k) for n, k in shapes]
    xs = {k: synth.activations(batch, k, xdt, seed=k + batch).cuda() for _, k in shapes}
    pad = 64
    bufs, ys = [], []
    for n, k in shapes:
        buf = torch.full((batch * n + 2 * pad,), 12345, dtype=torch.int16, device="cuda")
        bufs.append(buf)
        ys.append(buf[pad:pad + batch * n].view(TDT[xdt]).view(batch, n))
    tensors.gemv_batched([(pw, xs[k]) for (pw, _, _), (n, k) in zip(packed, shapes)], ys)
    torch.cuda.synchronize()
    for (pw, codes, scales), (n, k), y, buf in zip(packed, shapes, ys, bufs):
        assert torch.all(buf[:pad] == 12345) and torch.all(buf[pad + batch * n:] == 12345), "write outside y"
        y_ref, a = oracle_products(fmt, codes, scales, k, xs[k].cpu())
        check_products(y, y_ref, a, f"batched {fmt} {xdt} n={n} k={k} batch={batch}")


def test_gemv_batched_c2_layer_set_grouping():
    """The 1.7B-class ternary layer set as a decoder layer issues it: [q, k, v] on one x, [o],
    [gate, up] on one x, [down]; every output matches the oracle."""
    wl = synth.WORKLOADS["c2"]
    mats = {}
    for i, mat in enumerate(wl.matrices):
        inp = synth.matrix_inputs(wl, i)
        mats[mat.name] = (tensors.pack_ternary(inp["t"].cuda(), inp["s"].cuda()), mat, oracle_pack("ternary", inp))
    x_attn = synth.activations(1, 2048, "f16", seed=71).cuda()
    x_o = synth.activations(1, 2048, "f16", seed=72).cuda()
    x_ffn = synth.activations(1, 2048, "f16", seed=73).cuda()
    x_down = synth.activations(1, 6144, "f16", seed=74).cuda()
    groups = [[("q", x_attn), ("k", x_attn), ("v", x_attn)], [("o", x_o)], [("gate", x_ffn), ("up", x_ffn)],
              [("down", x_down)]]
    for grp in groups:
        ys = tensors.gemv_batched([(mats[name][0], x) for name, x in grp])
        torch.cuda.synchronize()
        for (name, x), y in zip(grp, ys):
            pw, mat, (codes, scales) = mats[name]
            y_ref, a = oracle_products("ternary", codes, scales, mat.k, x.cpu())
            check_products(y, y_ref, a, f"c2/{name} grouped")


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
@pytest.mark.parametrize("batch", [1, 5])
def test_gemv_batched_k_split_with_empty_chunks(fmt, batch):
    """A long-K problem with few rows makes the grouped launch split K over a cluster; the short
    problems of the same launch then have K chunks with no groups, which must add nothing."""
    shapes = [(64, 8192), (16, 256), (200, 1024), (130, 128)]
    packed = [_packed(fmt, n, k, seed=2 * n + k) for n, k in shapes]
    xs = [synth.activations(batch, k, "bf16", seed=n + k).cuda() for n, k in shapes]
    ys = tensors.gemv_batched([(pw, x) for (pw, _, _), x in zip(packed, xs)])
    torch.cuda.synchronize()
    for (pw, codes, scales), (n, k), x, y in zip(packed, shapes, xs, ys):
        y_ref, a = oracle_products(fmt, codes, scales, k, x.cpu())
        check_products(y, y_ref, a, f"batched split {fmt} n={n} k={k} batch={batch}")


@pytest.mark.parametrize("fmt,batch,k", [("1bit", 1, 327680), ("1bit", 2, 180224), ("1bit", 4, 90112),
                                         ("1bit", 8, 49152), ("ternary", 1, 344064), ("ternary", 2, 188416),
                                         ("ternary", 4, 98304), ("ternary", 8, 49152)])
def test_gemv_at_k_limit(fmt, batch, k):
    """Each batch class at the largest K lb_gemv accepts (the K split then uses the widest
    cluster), with a ragged row count."""
    n = 20
    pw, codes, scales = _packed(fmt, n, k, seed=k + batch)
    x = synth.activations(batch, k, "bf16", seed=batch).cuda()
    y = _run_guarded(pw, x)
    y_ref, a = oracle_products(fmt, codes, scales, k, x.cpu())
    check_products(y, y_ref, a, f"{fmt} k-limit batch={batch} k={k}")


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
@pytest.mark.parametrize("batch", [1, 8])
def test_gemv_two_row_blocks_per_cluster(fmt, batch):
    """9600 x 8192 splits K over 3-CTA clusters, and 75 row blocks x 3 CTAs do not fit the SMs in
    one wave, so each cluster takes two row blocks (the second one grid-height row blocks after the
    first) and reduces both through one exchange.  Sampled rows cover the first and last rows of
    every row block."""
    n, k = 9600, 8192
    if fmt == "1bit":
        inp = {"w": synth.weights_fp32(n, k, 0.05, seed=51)}
        pw = tensors.pack_1bit(inp["w"].cuda())
    else:
        inp = {"t": synth.ternary_codes(n, k, seed=51), "s": synth.ternary_scales_bits(n, k, 0.02, seed=52)}
        pw = tensors.pack_ternary(inp["t"].cuda(), inp["s"].cuda())
    x = synth.activations(batch, k, "bf16", seed=53).cuda()
    y = _run_guarded(pw, x)
    rb = np.arange(0, n, 128)
    rng = np.random.default_rng(54)
    rows = np.unique(np.concatenate([rb, rb + 127, rng.integers(0, n, 1500)]))
    sub = {key: v.numpy()[rows] for key, v in inp.items()}
    if fmt == "1bit":
        codes, scales = orc.pack_1bit(sub["w"])
    else:
        codes, scales = orc.pack_ternary(sub["t"], sub["s"].view(np.uint16))
    y_ref, a = oracle_products(fmt, codes, scales, k, x.cpu())
    check_products(y, y_ref, a, f"{fmt} {n}x{k} batch={batch}", cols=rows)



@pytest.mark.parametrize("xdt", ["f16", "bf16"])
def test_gemv_1bit_table_many_row_blocks(xdt):
    """1-bit at batch 1 (table form) with 299 row blocks on persistent CTAs, the last one ragged:
    every row is checked."""
    n, k = 299 * 128 - 50, 1024
    pw, codes, scales = _packed("1bit", n, k, seed=71)
    x = synth.activations(1, k, xdt, seed=72).cuda()
    y = _run_guarded(pw, x)
    y_ref, a = oracle_products("1bit", codes, scales, k, x.cpu())
    check_products(y, y_ref, a, f"1-bit {n}x{k} persistent")
