"""Pins of the CPU oracle against what the pages and the mathematics fix (no GPU needed).

Each ``pin_*`` function raises AssertionError when the oracle disagrees with an
independent fact: a number printed on a page, the page's own demo statements re-run in
CPython, a library routine for a special case, a closed form, an invariant, or exact
rational arithmetic on tiny inputs.  ``test_mutations_are_caught`` plants plausible
mistakes in the oracle (on the CPU) and checks that some pin fails for each of them.
"""

import json
import math
import os
import random
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import lb_oracle as orc

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------- codecs

def pin_f16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.f16_bits_to_f64(bits)
    lib = bits.view(np.float16).astype(np.float64)
    same = (ours == lib) | (np.isnan(ours) & np.isnan(lib))
    assert same.all(), f"binary16 decode differs at {np.flatnonzero(~same)[:5]}"
    assert np.array_equal(np.signbit(ours[~np.isnan(ours)]), np.signbit(lib[~np.isnan(lib)]))


def pin_bf16_decode_exhaustive():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = orc.bf16_bits_to_f64(bits)
    lib = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    same = (ours == lib) | (np.isnan(ours) & np.isnan(lib))
    assert same.all(), f"bfloat16 decode differs at {np.flatnonzero(~same)[:5]}"


def pin_f16_encode():
    # every finite binary16 value maps back to its own pattern
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = bits.view(np.float16).astype(np.float64)
    fin = np.isfinite(vals)
    assert np.array_equal(orc.f64_to_f16_bits_rne(vals[fin]), bits[fin])
    # midpoints between neighbours (ties) and quarter points, against numpy's conversion
    pos = np.sort(np.unique(np.abs(vals[fin])))
    mids = np.concatenate([(pos[:-1] + pos[1:]) / 2, pos[:-1] * 0.75 + pos[1:] * 0.25])
    mids = np.concatenate([mids, -mids, [65519.0, 65520.0, 65535.0, 1e9, 2.0 ** -25, 3 * 2.0 ** -26]])
    with np.errstate(over="ignore"):
        lib = mids.astype(np.float16).view(np.uint16)
    ours = orc.f64_to_f16_bits_rne(mids)
    assert np.array_equal(ours, lib), f"RNE differs at {mids[ours != lib][:5]}"
    # a dense random sweep of float32 inputs across the exponent range
    rng = np.random.default_rng(7)
    f32 = (rng.standard_normal(200000) * np.exp2(rng.integers(-30, 20, 200000))).astype(np.float32)
    with np.errstate(over="ignore"):
        lib = f32.astype(np.float16).view(np.uint16)
    assert np.array_equal(orc.f64_to_f16_bits_rne(f32.astype(np.float64)), lib)


def pin_bf16_encode():
    # every finite bfloat16 value maps back to its own pattern
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = orc.bf16_bits_to_f64(bits)
    fin = np.isfinite(vals)
    assert np.array_equal(orc.f64_to_bf16_bits_rne(vals[fin]), bits[fin])
    # ties, quarter points and the overflow edge, against torch's float32 -> bfloat16 conversion
    pos = np.sort(np.unique(np.abs(vals[fin])))
    mids = np.concatenate([(pos[:-1] + pos[1:]) / 2, pos[:-1] * 0.75 + pos[1:] * 0.25])
    top = float(pos[-1])
    mids = np.concatenate([mids, -mids, [top * (1 + 2.0 ** -9), top * (1 + 2.0 ** -8) * 0.999999]])
    mids = mids[np.abs(mids) < 3.4e38]                     # float32-representable inputs
    lib = torch.from_numpy(mids.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ours = orc.f64_to_bf16_bits_rne(mids.astype(np.float32).astype(np.float64))
    assert np.array_equal(ours, lib), f"RNE differs at {mids[ours != lib][:5]}"
    # a dense random sweep of float32 inputs across the exponent range (subnormals included)
    rng = np.random.default_rng(8)
    f32 = (rng.standard_normal(200000) * np.exp2(rng.integers(-140, 120, 200000))).astype(np.float32)
    lib = torch.from_numpy(f32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.f64_to_bf16_bits_rne(f32.astype(np.float64)), lib)


def pin_embed():
    """Embedding rows against the raw inputs, with numpy's binary16 and torch's bfloat16
    arithmetic: a 1-bit row is sign(w) * fp16(max |w| of the group); a ternary row is t * s."""
    rng = np.random.default_rng(9)
    n, k = 37, 384
    w = (rng.standard_normal((n, k)) * 0.1).astype(np.float32)
    w[3, :128] = 0.0                                       # an all-zero group: s = 0, bits 1 -> +0
    codes, scales = orc.pack_1bit(w)
    ids = np.array([5, 0, 36, 3, 5, -1, 37, 12])
    s_ref = np.abs(w).reshape(n, k // 128, 128).max(axis=2).astype(np.float16)       # numpy RNE
    for dt in ("f16", "bf16"):
        out, bad = orc.embed_rows(orc.FMT_1BIT, codes, scales, k, ids, dt)
        assert bad.tolist() == [False] * 5 + [True, True, False]
        assert not out[bad].any()
        for r, i in enumerate(ids):
            if bad[r]:
                continue
            v = np.where(w[i] >= 0, 1.0, -1.0).astype(np.float16) * np.repeat(s_ref[i], 128)
            if dt == "f16":
                exp = v.view(np.uint16)
            else:
                exp = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            assert np.array_equal(out[r], exp), (dt, r)
    t = rng.integers(-1, 2, (n, k)).astype(np.int8)
    sb = (np.abs(rng.standard_normal((n, k // 128))) * 0.02).astype(np.float16)
    sb[7, 1] = -sb[7, 1]                                   # a negative scale: t = 0 gives -0
    codes, scales = orc.pack_ternary(t, sb.view(np.uint16))
    ids = np.array([7, 7, 0, 36])
    out, bad = orc.embed_rows(orc.FMT_TERNARY, codes, scales, k, ids, "f16")
    assert not bad.any()
    for r, i in enumerate(ids):
        exp = (t[i].astype(np.float16) * np.repeat(sb[i], 128)).view(np.uint16)
        assert np.array_equal(out[r], exp), r
    assert (out[0, 128:256][t[7, 128:256] == 0] == 0x8000).all()


def pin_ternary5():
    """Five-digit base-3 storage: hand-computed bytes, exact round trip, the printed sizes, and
    the same products as the 2-bit storage of the same codes."""
    g = _load("sizes.json")
    # sizes: 26 bytes of codes + 2 of scale per 128 weights = 1.75 bpw; the page's "five
    # three-state values in a byte" is 8 / 5 bits, and 1.75 lies between the printed 1.71 and 1.76
    c, sc = orc.packed_bytes(orc.FMT_TERNARY5, 1, orc.GROUP)
    assert (c, sc) == (26, 2) and orc.bits_per_weight(orc.FMT_TERNARY5) == 1.75
    assert 8 / 5 == g["p4_five_trits_per_byte_bits"]["value"]
    assert g["p2_ternary_info_bpw"]["value"] <= 1.75 <= g["p3_ternary_effective_bpw"]["value"]
    # hand-computed bytes (digit f = t + 1, first weight of a byte in the lowest digit)
    one = np.ones((1, 128), dtype=np.int8)
    s1 = np.full((1, 1), 0x3C00, dtype=np.uint16)
    c, _ = orc.pack_ternary5(one, s1)                              # f = 2 everywhere
    assert c[0, :25].tolist() == [242] * 25 and c[0, 25] == 2 + 6 + 18
    c, _ = orc.pack_ternary5(-one, s1)                             # f = 0
    assert not c.any()
    t = np.zeros((1, 128), dtype=np.int8)
    c, _ = orc.pack_ternary5(t, s1)                                # f = 1: 1 + 3 + 9 + 27 + 81
    assert c[0, :25].tolist() == [121] * 25 and c[0, 25] == 13
    t[0, 7] = 1                                                    # byte 1, digit 2: + 3^2
    t[0, 126] = -1                                                 # byte 25, digit 1: - 3
    c, _ = orc.pack_ternary5(t, s1)
    assert c[0, 1] == 130 and c[0, 25] == 10 and c[0, 0] == 121
    # round trip and equal products with the 2-bit storage
    rng = np.random.default_rng(11)
    n, k = 13, 640
    t = rng.integers(-1, 2, (n, k)).astype(np.int8)
    sb = (np.abs(rng.standard_normal((n, k // 128))) * 0.03).astype(np.float16).view(np.uint16)
    c5, s5 = orc.pack_ternary5(t, sb)
    assert c5.shape == (n, 26 * (k // 128)) and np.array_equal(orc.unpack_ternary5(c5, k), t)
    c2, s2 = orc.pack_ternary(t, sb)
    x = rng.standard_normal((3, k))
    y5, a5 = orc.matvec(orc.FMT_TERNARY5, c5, s5, k, x)
    y2, a2 = orc.matvec(orc.FMT_TERNARY, c2, s2, k, x)
    assert np.array_equal(y5, y2) and np.array_equal(a5, a2)
    bad = c5.copy()
    bad[0, 25] = 27                                                # a digit past weight 127
    with pytest.raises(orc.OracleError):
        orc.unpack_ternary5(bad, k)


def pin_silu():
    """silu against 50-digit mpmath, its limits, and the slope constant of the SwiGLU bound."""
    import mpmath
    mpmath.mp.dps = 50
    z = np.concatenate([np.linspace(-60, 60, 2401), [0.0, -0.0, 1e-300, -1e-300, 700.0, -700.0, 800.0, -800.0]])
    ours = orc.silu(z)
    ref = np.array([float(mpmath.mpf(float(v)) / (1 + mpmath.exp(-mpmath.mpf(float(v))))) for v in z])
    assert np.allclose(ours, ref, rtol=1e-14, atol=0.0), np.max(np.abs(ours - ref) / np.maximum(np.abs(ref), 1e-300))
    # the limits, reached at finite arguments (a product of finite binary16 inputs stays finite)
    assert orc.silu(np.array([800.0]))[0] == 800.0 and orc.silu(np.array([-800.0]))[0] == 0.0
    assert orc.silu(np.array([np.log(3.0)]))[0] == pytest.approx(0.75 * np.log(3.0), rel=1e-15)
    # the slope of silu: sigma(z) (1 + z (1 - sigma(z))); its maximum is the constant of the bound
    zz = np.linspace(-20, 20, 400001)
    sg = 1.0 / (1.0 + np.exp(-zz))
    slope = np.abs(sg * (1.0 + zz * (1.0 - sg)))
    assert slope.max() <= orc.SILU_SLOPE_MAX and slope.max() > orc.SILU_SLOPE_MAX - 1e-4


def pin_swiglu():
    """A tiny pair by brute force from the raw inputs in 50-digit arithmetic, and the tolerance
    bound checked at the corners of the allowed product errors."""
    import mpmath
    mpmath.mp.dps = 50
    rng = np.random.default_rng(10)
    n, k, b = 3, 256, 2
    tg = rng.integers(-1, 2, (n, k)).astype(np.int8)
    tu = rng.integers(-1, 2, (n, k)).astype(np.int8)
    sg = (np.abs(rng.standard_normal((n, k // 128))) * 0.05).astype(np.float16)
    su = (np.abs(rng.standard_normal((n, k // 128))) * 0.05).astype(np.float16)
    x = rng.standard_normal((b, k)).astype(np.float16).astype(np.float64)
    cg, scg = orc.pack_ternary(tg, sg.view(np.uint16))
    cu, scu = orc.pack_ternary(tu, su.view(np.uint16))
    h, g, a_g, u, a_u = orc.swiglu(orc.FMT_TERNARY, cg, scg, cu, scu, k, x)
    for bi in range(b):
        for r in range(n):
            gm = sum(mpmath.mpf(float(sg[r, i // 128])) * int(tg[r, i]) * mpmath.mpf(x[bi, i]) for i in range(k))
            um = sum(mpmath.mpf(float(su[r, i // 128])) * int(tu[r, i]) * mpmath.mpf(x[bi, i]) for i in range(k))
            hm = gm / (1 + mpmath.exp(-gm)) * um
            assert abs(h[bi, r] - float(hm)) <= 1e-12 * max(1.0, abs(float(hm))), (bi, r)
    # perturb g and u to the corners of their product bounds: the bound still holds
    dg = orc.TOL_REL * a_g + orc.TOL_ABS
    du = orc.TOL_REL * a_u + orc.TOL_ABS
    tol = orc.swiglu_tolerance(h, g, a_g, u, a_u)
    for sgn_g in (-1, 1):
        for sgn_u in (-1, 1):
            hp = orc.silu(g + sgn_g * dg) * (u + sgn_u * du)
            assert (np.abs(hp - h) <= tol).all()


# --------------------------------------------------------------------------- sizes

def pin_sizes():
    g = _load("sizes.json")
    c, s = orc.packed_bytes(orc.FMT_1BIT, 1, orc.GROUP)
    assert c + s == g["p1_demo_group_bytes_1bit"]["value"]
    assert orc.bits_per_weight(orc.FMT_1BIT) == g["p1_box_bpw_1bit"]["value"]
    ratio = g["p1_demo_group_bytes_fp16"]["value"] / (c + s)
    assert f"{ratio:.1f}" == g["p1_ratio_printed"]["value"]
    assert round(16 / orc.bits_per_weight(orc.FMT_1BIT), 1) == g["p2_binary_reduction"]["value"]
    # 3.44 GB of FP16 weights at 1.125 bpw
    assert round(g["p1_model_gb_fp16"]["value"] * orc.bits_per_weight(orc.FMT_1BIT) / 16, 2) == \
        g["p1_model_gb_1bit"]["value"]
    # the pages' ternary figure is an information rate, log2(3) + 16/128
    info = math.log2(3) + 16 / orc.GROUP
    assert round(info, 2) == g["p2_ternary_info_bpw"]["value"]
    assert round(16 / info, 1) == g["p2_ternary_reduction"]["value"]
    # stored ternary: 2-bit fields + one fp16 scale per 128 -> 34 bytes per group
    c, s = orc.packed_bytes(orc.FMT_TERNARY, 1, orc.GROUP)
    assert (c, s) == (32, 2) and orc.bits_per_weight(orc.FMT_TERNARY) == 2.125
    assert orc.packed_bytes(orc.FMT_1BIT, 2048, 2048) == (2048 * 256, 2048 * 16 * 2)
    assert orc.packed_bytes(orc.FMT_TERNARY, 17408, 5120) == (17408 * 1280, 17408 * 40 * 2)


# --------------------------------------------------------------------------- the page's demo

def _page_demo_group():
    """The statements of the demo in [P1] section 7, run in CPython."""
    random.seed(42)
    weights = [random.gauss(0, 0.1) for _ in range(128)]
    scale = max(abs(w) for w in weights)
    quantized = [1 if w >= 0 else 0 for w in weights]
    dequantized = [scale if b == 1 else -scale for b in quantized]
    mse = sum((a - b) ** 2 for a, b in zip(weights, dequantized)) / 128
    return weights, scale, quantized, mse


def pin_demo_group():
    weights, scale, quantized, mse = _page_demo_group()
    w32 = np.array(weights, dtype=np.float32)[None, :]
    assert np.array_equal(np.sign(w32[0]) >= 0, np.array(quantized) == 1)   # no fp32 sign flips
    codes, scales = orc.pack_1bit(w32)
    t = orc.unpack_1bit(codes, 128)[0]
    assert list((t > 0).astype(int)) == quantized
    assert int(scales[0, 0]) == int(np.float16(scale).view(np.uint16))
    w_hat = orc.dequantize(orc.FMT_1BIT, codes, scales, 128)[0]
    # the page's dequantised values, with its float scale replaced by the stored fp16 scale
    s16 = float(np.float16(scale))
    assert np.array_equal(w_hat, np.array([s16 if b else -s16 for b in quantized]))
    mse16 = float(np.mean((np.array(weights) - w_hat) ** 2))
    # |s16 - scale| <= 2^-11 scale changes the MSE by at most about 2 |ds| mean|w - w_hat|
    assert abs(mse16 - mse) <= 2 * abs(s16 - scale) * 2 * scale + 1e-12


# --------------------------------------------------------------------------- layout fixtures

def pin_layout_fixtures():
    g = _load("layout.json")
    for case in g["onebit"]:
        w = np.full((1, 128), case["background"], dtype=np.float32)
        for i, v in case["set"].items():
            w[0, int(i)] = v
        codes, _ = orc.pack_1bit(w)
        expect = np.full(16, int(case.get("bytes_all", "0x00"), 16), dtype=np.uint8)
        for i, b in case["bytes"].items():
            expect[int(i)] = int(b, 16)
        assert np.array_equal(codes[0], expect), case["why"]
    for case in g["ternary"]:
        t = np.zeros((1, 128), dtype=np.int8)
        t[0, :4] = case["t_prefix"]
        codes, _ = orc.pack_ternary(t, np.zeros((1, 1), dtype=np.uint16))
        assert int(codes[0, 0]) == int(case["byte0"], 16), case["why"]
        assert np.all(codes[0, 1:] == 0x55)


# --------------------------------------------------------------------------- round trips

def pin_roundtrip_1bit():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((5, 384)) * 0.1).astype(np.float32)
    w[1, 128:256] = 0.0                                         # all-zero group
    w[2, 5] = -0.0
    codes, scales = orc.pack_1bit(w)
    gmax = np.abs(w).reshape(5, 3, 128).max(axis=2).astype(np.float16).astype(np.float64)
    expect = np.where(w >= 0, 1.0, -1.0) * np.repeat(gmax, 128, axis=1)
    assert np.array_equal(orc.dequantize(orc.FMT_1BIT, codes, scales, 384), expect)


def pin_roundtrip_ternary():
    rng = np.random.default_rng(4)
    t = rng.integers(-1, 2, size=(6, 256)).astype(np.int8)
    s = np.abs(rng.standard_normal((6, 2)) * 0.02).astype(np.float16).view(np.uint16)
    codes, s2 = orc.pack_ternary(t, s)
    assert np.array_equal(orc.unpack_ternary(codes, 256), t)
    assert np.array_equal(s2, s)


# --------------------------------------------------------------------------- invariants

def _popcount_group_bytes(row_bytes):
    return int.from_bytes(bytes(row_bytes), "little").bit_count()


def pin_rowsum_invariant():
    rng = np.random.default_rng(5)
    n, k = 7, 512
    w = (rng.standard_normal((n, k)) * 0.05).astype(np.float32)
    codes, scales = orc.pack_1bit(w)
    y, _ = orc.matvec(orc.FMT_1BIT, codes, scales, k, np.ones((1, k)))
    s = scales.view(np.float16).astype(np.float64)
    for r in range(n):
        expect = 0.0
        for g in range(k // 128):
            pos = _popcount_group_bytes(codes[r, 16 * g:16 * g + 16])
            expect += s[r, g] * (pos - (128 - pos))
        assert y[0, r] == expect, (r, y[0, r], expect)
    # ternary: s * (#(+1) - #(-1)) counted from the raw fields
    t = rng.integers(-1, 2, size=(n, k)).astype(np.int8)
    sb = np.abs(rng.standard_normal((n, k // 128)) * 0.02).astype(np.float16).view(np.uint16)
    codes, scales = orc.pack_ternary(t, sb)
    y, _ = orc.matvec(orc.FMT_TERNARY, codes, scales, k, np.ones((1, k)))
    s = sb.view(np.float16).astype(np.float64)
    for r in range(n):
        expect = 0.0
        for g in range(k // 128):
            fields = [(int(b) >> (2 * j)) & 3 for b in codes[r, 32 * g:32 * g + 32] for j in range(4)]
            expect += s[r, g] * (fields.count(2) - fields.count(0))
        assert y[0, r] == expect


def pin_unit_vectors():
    rng = np.random.default_rng(6)
    n, k = 5, 256
    w = (rng.standard_normal((n, k))).astype(np.float32)
    codes, scales = orc.pack_1bit(w)
    s = scales.view(np.float16).astype(np.float64)
    for col in (0, 1, 7, 8, 127, 128, 200, 255):
        x = np.zeros((1, k))
        x[0, col] = 1.0
        y, _ = orc.matvec(orc.FMT_1BIT, codes, scales, k, x)
        for r in range(n):
            bit = (int(codes[r, col // 8]) >> (col % 8)) & 1
            assert y[0, r] == (s[r, col // 128] if bit else -s[r, col // 128])
    t = rng.integers(-1, 2, size=(n, k)).astype(np.int8)
    codes, scales = orc.pack_ternary(t, scales)
    for col in (0, 3, 4, 129, 255):
        x = np.zeros((1, k))
        x[0, col] = 1.0
        y, _ = orc.matvec(orc.FMT_TERNARY, codes, scales, k, x)
        for r in range(n):
            f = (int(codes[r, col // 4]) >> (2 * (col % 4))) & 3
            assert y[0, r] == (f - 1) * s[r, col // 128]


def _exact_products(codes, scales_bits, k, x_bits, fmt, xdt):
    """Pure-Python exact rational y and a, decoding every field by hand."""
    n = codes.shape[0]
    dec = orc.f16_bits_to_f64 if xdt == "f16" else orc.bf16_bits_to_f64
    xs = [[Fraction(float(v)) for v in dec(row)] for row in x_bits]
    ss = [[Fraction(float(v)) for v in orc.f16_bits_to_f64(row)] for row in scales_bits]
    y = [[Fraction(0)] * n for _ in xs]
    a = [[Fraction(0)] * n for _ in xs]
    for r in range(n):
        for kk in range(k):
            if fmt == orc.FMT_1BIT:
                t = 1 if (int(codes[r, kk // 8]) >> (kk % 8)) & 1 else -1
            else:
                t = ((int(codes[r, kk // 4]) >> (2 * (kk % 4))) & 3) - 1
            wv = ss[r][kk // 128] * t
            for b, xb in enumerate(xs):
                y[b][r] += wv * xb[kk]
                a[b][r] += abs(wv * xb[kk])
    return y, a


def pin_bruteforce_exact():
    rng = np.random.default_rng(8)
    for fmt in (orc.FMT_1BIT, orc.FMT_TERNARY):
        for (n, k, b, xdt) in ((1, 128, 1, "f16"), (3, 256, 2, "bf16"), (4, 128, 3, "f16")):
            if fmt == orc.FMT_1BIT:
                codes, scales = orc.pack_1bit((rng.standard_normal((n, k)) * 0.1).astype(np.float32))
            else:
                t = rng.integers(-1, 2, size=(n, k)).astype(np.int8)
                sb = np.abs(rng.standard_normal((n, k // 128)) * 0.02).astype(np.float16).view(np.uint16)
                codes, scales = orc.pack_ternary(t, sb)
            xf = rng.standard_normal((b, k))
            if xdt == "f16":
                x_bits = xf.astype(np.float16).view(np.uint16)
            else:
                x_bits = torch.from_numpy(xf).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
            x = orc.decode_activation_bits(x_bits, xdt)
            y, a = orc.matvec(fmt, codes, scales, k, x)
            ye, ae = _exact_products(codes, scales, k, x_bits, fmt, xdt)
            for bb in range(b):
                for r in range(n):
                    bound = 1e-13 * float(ae[bb][r]) + 1e-300
                    assert abs(Fraction(y[bb, r]) - ye[bb][r]) <= Fraction(bound), (fmt, n, k, bb, r)
                    assert abs(Fraction(a[bb, r]) - ae[bb][r]) <= Fraction(bound)


def pin_linearity_and_scaling():
    rng = np.random.default_rng(9)
    n, k = 9, 384
    t = rng.integers(-1, 2, size=(n, k)).astype(np.int8)
    sb = np.abs(rng.standard_normal((n, k // 128)) * 0.02 + 0.01).astype(np.float16).view(np.uint16)
    codes, scales = orc.pack_ternary(t, sb)
    x1, x2 = rng.standard_normal((2, 1, k))
    y1, a1 = orc.matvec(orc.FMT_TERNARY, codes, scales, k, x1)
    y2, _ = orc.matvec(orc.FMT_TERNARY, codes, scales, k, x2)
    y12, _ = orc.matvec(orc.FMT_TERNARY, codes, scales, k, x1 + x2)
    assert np.allclose(y12, y1 + y2, rtol=0, atol=1e-12 * (a1.max() + 1))
    doubled = (scales.astype(np.int64) + 0x400).astype(np.uint16)      # exponent + 1 (normal values)
    assert np.all(((scales >> 10) & 0x1F) > 0) and np.all(((scales >> 10) & 0x1F) < 30)
    yd, ad = orc.matvec(orc.FMT_TERNARY, codes, doubled, k, x1)
    assert np.array_equal(yd, 2 * y1) and np.array_equal(ad, 2 * a1)


def pin_errors():
    def raises(kind, fn, *args):
        with pytest.raises(orc.OracleError) as e:
            fn(*args)
        assert e.value.kind == kind, e.value

    w = np.zeros((2, 128), dtype=np.float32)
    raises("shape", orc.pack_1bit, np.zeros((2, 100), dtype=np.float32))
    raises("shape", orc.pack_1bit, np.zeros((0, 128), dtype=np.float32))
    for bad in (np.nan, np.inf, -np.inf):
        w2 = w.copy()
        w2[1, 5] = bad
        raises("nonfinite", orc.pack_1bit, w2)
    w3 = w.copy()
    w3[0, 0] = 65520.0                                                   # rounds to binary16 inf
    raises("range", orc.pack_1bit, w3)
    w3[0, 0] = 65519.0                                                   # rounds to 65504
    c, s = orc.pack_1bit(w3)
    assert int(s[0, 0]) == 0x7BFF
    t = np.zeros((1, 128), dtype=np.int8)
    t[0, 7] = 2
    raises("code", orc.pack_ternary, t, np.zeros((1, 1), dtype=np.uint16))
    raises("code", orc.unpack_ternary, np.full((1, 32), 0xFF, dtype=np.uint8), 128)


def pin_tolerance_rule():
    y_ref = np.array([1.0, -2.0, 0.0])
    a = np.array([10.0, 4.0, 0.0])
    slack = 2e-3 * a + 1e-5
    assert orc.within_tolerance(y_ref + 0.99 * slack, y_ref, a).all()
    assert not orc.within_tolerance(y_ref + 1.01 * slack, y_ref, a).any()
    # stored outputs: the nearest bfloat16 / binary16 of the exact value always passes, even with
    # a == |y| where 2e-3 * a is below the format's own rounding error
    rng = np.random.default_rng(11)
    y = rng.standard_normal(20000) * np.exp2(rng.integers(-20, 20, 20000))
    bf = torch.from_numpy(y).to(torch.bfloat16).to(torch.float64).numpy()
    f16 = y.astype(np.float16).astype(np.float64)
    zero = np.zeros_like(y)
    assert orc.within_tolerance(bf, y, zero, "bf16").all()
    assert orc.within_tolerance(f16[np.abs(y) < 6e4], y[np.abs(y) < 6e4], zero[np.abs(y) < 6e4], "f16").all()
    # half an ulp exactly: 4.39 sits in the bfloat16 binade [4, 8) with ulp 2^-5
    assert np.isclose(orc.output_half_ulp(4.39, "bf16"), 2.0 ** -6)
    assert np.isclose(orc.output_half_ulp(4.39, "f16"), 2.0 ** -9)
    assert np.isclose(orc.output_half_ulp(1e-9, "f16"), 2.0 ** -25)
    # one full ulp off is rejected when a == 0
    assert not orc.within_tolerance(np.array([4.0 + 2.0 ** -5 + 2.0 ** -9]), np.array([4.0]), np.array([0.0]),
                                    "bf16").any()


ALL_PINS = [pin_f16_decode_exhaustive, pin_bf16_decode_exhaustive, pin_f16_encode, pin_bf16_encode, pin_embed,
            pin_silu, pin_swiglu, pin_ternary5,
            pin_sizes,
            pin_demo_group, pin_layout_fixtures, pin_roundtrip_1bit, pin_roundtrip_ternary,
            pin_rowsum_invariant, pin_unit_vectors, pin_bruteforce_exact,
            pin_linearity_and_scaling, pin_errors, pin_tolerance_rule]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin()


# --------------------------------------------------------------------------- planted mistakes

def _mut_bitorder_big(monkeypatch):
    real = np.packbits
    monkeypatch.setattr(orc.np, "packbits", lambda a, axis=None, bitorder="big": real(a, axis=axis, bitorder="big"))


def _mut_sign_strict(monkeypatch):
    real = orc.pack_1bit

    def bad(w):
        codes, scales = real(w)
        w = np.asarray(w, dtype=np.float32)
        return np.packbits((w > 0).astype(np.uint8), axis=1, bitorder="little"), scales
    monkeypatch.setattr(orc, "pack_1bit", bad)


def _mut_scale_mean(monkeypatch):
    real = orc.pack_1bit

    def bad(w):
        codes, _ = real(w)
        w = np.asarray(w, dtype=np.float32)
        n, k = w.shape
        m = np.abs(w).reshape(n, k // 128, 128).mean(axis=2)
        return codes, orc.f64_to_f16_bits_rne(m)
    monkeypatch.setattr(orc, "pack_1bit", bad)


def _mut_ternary_field(monkeypatch):
    real = orc.pack_ternary

    def bad(t, s):
        t = np.asarray(t)
        f = (t.astype(np.int64) & 3).reshape(t.shape[0], -1, 4)           # t instead of t + 1
        codes = (f[:, :, 0] | (f[:, :, 1] << 2) | (f[:, :, 2] << 4) | (f[:, :, 3] << 6)).astype(np.uint8)
        return codes, np.asarray(s, dtype=np.uint16).copy()
    monkeypatch.setattr(orc, "pack_ternary", bad)


def _mut_drop_scale(monkeypatch):
    real = orc.dequantize
    monkeypatch.setattr(orc, "dequantize",
                        lambda fmt, c, s, k: real(fmt, c, np.full_like(np.asarray(s), 0x3C00), k))


def _mut_scale_axis(monkeypatch):
    def bad(fmt, codes, scales, k):
        t = orc.unpack_1bit(codes, k) if fmt == orc.FMT_1BIT else orc.unpack_ternary(codes, k)
        s = orc.f16_bits_to_f64(np.asarray(scales, dtype=np.uint16))
        return t * np.tile(s, (1, 128))                                   # wrong group indexing
    monkeypatch.setattr(orc, "dequantize", bad)


def _mut_f16_bias(monkeypatch):
    real = orc.f16_bits_to_f64
    monkeypatch.setattr(orc, "f16_bits_to_f64", lambda b: real(b) * 2.0)


def _mut_abs_sum(monkeypatch):
    real = orc.matvec

    def bad(fmt, codes, scales, k, x):
        y, a = real(fmt, codes, scales, k, x)
        return y, np.abs(y)                                              # |sum| instead of sum |.|
    monkeypatch.setattr(orc, "matvec", bad)


def _mut_rne_truncate(monkeypatch):
    real = orc.f64_to_f16_bits_rne

    def bad(v):
        v = np.asarray(v, dtype=np.float64)
        return real(np.where(np.abs(v) > 0, v * (1 - 2.0 ** -12), v))     # biased toward zero
    monkeypatch.setattr(orc, "f64_to_f16_bits_rne", bad)


def _mut_bf16_truncate(monkeypatch):
    real = orc.f64_to_bf16_bits_rne

    def bad(v):
        v = np.asarray(v, dtype=np.float64)
        return real(np.where(np.abs(v) > 0, v * (1 - 2.0 ** -9), v))      # biased toward zero
    monkeypatch.setattr(orc, "f64_to_bf16_bits_rne", bad)


def _mut_embed_row_offset(monkeypatch):
    real = orc.embed_rows

    def bad(fmt, codes, scales, k, ids, out_dtype):
        return real(fmt, codes, scales, k, np.asarray(ids) + 1, out_dtype)   # off-by-one row
    monkeypatch.setattr(orc, "embed_rows", bad)


def _mut_silu_sign(monkeypatch):
    monkeypatch.setattr(orc, "silu", lambda z: np.asarray(z, dtype=np.float64) / (1.0 + np.exp(np.asarray(z, dtype=np.float64))))


def _mut_swiglu_swap(monkeypatch):
    real = orc.swiglu

    def bad(fmt, cg, sg, cu, su, k, x):
        return real(fmt, cu, su, cg, sg, k, x)                            # gate and up exchanged
    monkeypatch.setattr(orc, "swiglu", bad)


def _mut_t5_digit_order(monkeypatch):
    real = orc.pack_ternary5

    def bad(t, s):
        t = np.asarray(t)
        n, k = t.shape
        g = k // 128
        f = np.zeros((n, g, 130), dtype=np.int64)
        f[:, :, :128] = t.astype(np.int64).reshape(n, g, 128) + 1
        f = f.reshape(n, g, 26, 5)
        codes = sum(f[..., i] * 3 ** (4 - i) for i in range(5)).astype(np.uint8)   # first weight highest
        return codes.reshape(n, g * 26), np.asarray(s, dtype=np.uint16).copy()
    monkeypatch.setattr(orc, "pack_ternary5", bad)


MUTATIONS = [_mut_t5_digit_order, _mut_silu_sign, _mut_swiglu_swap, _mut_bitorder_big, _mut_sign_strict, _mut_scale_mean, _mut_ternary_field,
             _mut_drop_scale, _mut_scale_axis, _mut_f16_bias, _mut_abs_sum, _mut_rne_truncate,
             _mut_bf16_truncate, _mut_embed_row_offset]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=lambda m: m.__name__)
def test_mutations_are_caught(mutation, monkeypatch):
    mutation(monkeypatch)
    failed = []
    for pin in ALL_PINS:
        try:
            pin()
        except (Exception, pytest.fail.Exception):
            failed.append(pin.__name__)
    assert failed, f"no pin caught {mutation.__name__}"
