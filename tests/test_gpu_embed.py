"""Embedding-row gather on the GPU against the FP64 oracle: bit-exact output patterns."""

import numpy as np
import pytest
import torch

from gemm_lb_gemv_02_b300 import synth
from oracle import lb_oracle as orc
from tests.helpers import oracle_pack, u16

pytestmark = pytest.mark.gpu

lb = pytest.importorskip("gemm_lb_gemv_02_b300.lb")
from gemm_lb_gemv_02_b300 import tensors  # noqa: E402

ODT = {"f16": torch.float16, "bf16": torch.bfloat16}


def _packed(fmt, n, k, seed):
    if fmt == "1bit":
        inp = {"w": synth.weights_fp32(n, k, 0.05, seed)}
        pw = tensors.pack_1bit(inp["w"].cuda())
    else:
        inp = {"t": synth.ternary_codes(n, k, seed), "s": synth.ternary_scales_bits(n, k, 0.02, seed + 1)}
        pw = tensors.pack_ternary(inp["t"].cuda(), inp["s"].cuda())
    codes, scales = oracle_pack(fmt, inp)
    return pw, codes, scales


def _run_guarded(pw, ids, odt):
    """lb_embed into the middle of a canary-filled buffer; checks the canaries afterwards."""
    count, k = ids.shape[0], pw.k
    pad = 64
    buf = torch.full((count * k + 2 * pad,), 12345, dtype=torch.int16, device="cuda")
    out = buf[pad:pad + count * k].view(ODT[odt]).view(count, k)
    tensors.embed(pw, ids.cuda(), out_dtype=ODT[odt], out=out)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == 12345) and torch.all(buf[pad + count * k:] == 12345), "write outside out"
    return out


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
@pytest.mark.parametrize("odt", ["f16", "bf16"])
@pytest.mark.parametrize("n,k,count", [(1, 128, 1), (37, 384, 5), (300, 2048, 333), (1000, 640, 64), (9, 17536, 40)])
def test_embed_shapes(fmt, odt, n, k, count):
    pw, codes, scales = _packed(fmt, n, k, seed=n + k)
    g = torch.Generator().manual_seed(count + n)
    ids = torch.randint(0, n, (count,), generator=g, dtype=torch.int32)
    ids[0] = n - 1                                                 # last row, and a repeat below
    if count > 2:
        ids[2] = ids[0]
    out = _run_guarded(pw, ids, odt)
    assert lb.lb_device_error(clear=True) == 0
    ref, bad = orc.embed_rows(orc.FMT_1BIT if fmt == "1bit" else orc.FMT_TERNARY, codes, scales, k,
                              ids.numpy(), odt)
    assert not bad.any()
    assert np.array_equal(u16(out), ref)


@pytest.mark.parametrize("fmt", ["1bit", "ternary"])
def test_embed_out_of_range_ids(fmt):
    """Ids outside [0, n) give +0 rows and set bit 2 of the device error word; the other rows are
    unaffected."""
    n, k = 50, 256
    pw, codes, scales = _packed(fmt, n, k, seed=3)
    ids = torch.tensor([4, -1, 49, 50, 2 ** 31 - 1, 0], dtype=torch.int32)
    lb.lb_device_error(clear=True)
    out = _run_guarded(pw, ids, "bf16")
    assert lb.lb_device_error(clear=True) == 4
    ref, bad = orc.embed_rows(orc.FMT_1BIT if fmt == "1bit" else orc.FMT_TERNARY, codes, scales, k,
                              ids.numpy(), "bf16")
    assert bad.tolist() == [False, True, False, True, True, False]
    assert np.array_equal(u16(out), ref)
    assert lb.lb_device_error() == 0


def test_embed_negative_scale_signed_zero():
    """t = 0 under a negative scale is -0 (IEEE s * 0), t = -1 under +0 is -0."""
    n, k = 4, 256
    t = synth.ternary_codes(n, k, seed=5)
    s = synth.ternary_scales_bits(n, k, 0.02, seed=6)
    s[1, 0] = s[1, 0] | -32768                                     # negative scale
    s[2, 1] = 0                                                    # +0 scale
    pw = tensors.pack_ternary(t.cuda(), s.cuda())
    codes, scales = orc.pack_ternary(t.numpy(), s.numpy().view(np.uint16))
    ids = torch.tensor([1, 2, 3, 0], dtype=torch.int32)
    out = _run_guarded(pw, ids, "f16")
    ref, _ = orc.embed_rows(orc.FMT_TERNARY, codes, scales, k, ids.numpy(), "f16")
    assert np.array_equal(u16(out), ref)
    assert (u16(out)[0, :128][t[1, :128].numpy() == 0] == 0x8000).all()


def test_embed_c3_table_sampled():
    """The 151936 x 2048 1-bit table (the LM-head matrix of the 1-bit workload, used as a tied
    embedding), 4096 token ids with the first and last rows; every gathered row is checked. The
    oracle packs only the sampled rows (packing is row by row)."""
    wl = synth.WORKLOADS["c3"]
    mat = wl.matrices[0]
    inp = synth.matrix_inputs(wl, 0)
    pw = tensors.pack_1bit(inp["w"].cuda())
    g = torch.Generator().manual_seed(77)
    ids = torch.randint(0, mat.n, (4096,), generator=g, dtype=torch.int32)
    ids[:2] = torch.tensor([0, mat.n - 1], dtype=torch.int32)
    out = tensors.embed(pw, ids.cuda(), out_dtype=torch.bfloat16)
    torch.cuda.synchronize()
    assert lb.lb_device_error(clear=True) == 0
    uniq, inv = np.unique(ids.numpy(), return_inverse=True)
    codes, scales = orc.pack_1bit(inp["w"].numpy()[uniq])
    ref, bad = orc.embed_rows(orc.FMT_1BIT, codes, scales, mat.k, inv, "bf16")
    assert not bad.any()
    assert np.array_equal(u16(out), ref)
