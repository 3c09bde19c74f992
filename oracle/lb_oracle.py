"""FP64 CPU oracle for the packed low-bit (1-bit and ternary, group 128) weight path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import or call this module:
only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline / reference
legs use it.  It shares no code, table or helper with the CUDA library; it is a plain,
slow, obviously-checkable restatement of what the pages define, written with numpy.

Sources (web pages, cited by title and section):

* [P1] 7minutos.es, "Un tutorial de codificación para ejecutar PrismML Bonsai 1-bit LLM en
  CUDA con GGUF …", section "7 · Q1_0_g128 Cuantización: qué está pasando bajo el capó":
  the weight-representation box (1 bit per weight, 0 -> -scale, 1 -> +scale, 128 weights
  share one FP16 scale, 1 + 16/128 = 1.125 bpw, 3.44 GB -> 0.24 GB, 14.2x) and the Python
  demo that quantises one group (scale = max |w|, bit = 1 if w >= 0 else 0, dequantised
  value = +scale if bit else -scale, 18 bytes vs 256 bytes per group).
* [P2] 7minutos.es, "PrismML lanza Bonsai 27B: compilaciones ternarias y de 1 bit …",
  section "Cómo funciona la compresión": every weight is a code with one FP16 scale per
  group of 128, effective weight w_i = s_g · t_i; ternary alphabet {-1, 0, +1}.
* [P3] kerneldigest.dev, "Compresión ternaria de modelos LLM: Bonsai 2 27B …", section
  "Arquitectura del Sistema": ternary {-1, 0, +1} weights with group-wise FP16 scaling.

Readings of points the pages leave open (each is also listed in the design notes):

* groups run along K (the reduction axis), contiguous inside a row; K % 128 == 0;
* 1-bit codes: weight k of a row is bit (k mod 8) of byte k // 8 (LSB first), so a row of
  K weights is K/8 bytes and group g of that row is bytes 16g .. 16g+15;
* ternary codes: 2-bit field f = t + 1 (0 -> -1, 1 -> 0, 2 -> +1; 3 is invalid); weight k
  is field (k mod 4) of byte k // 4, LSB first (bits 2(k mod 4), 2(k mod 4)+1);
* scales: one IEEE binary16 per (row, group), stored as its 16-bit pattern, [N][K/128];
* the 1-bit scale is the fp32 maximum of |w| over the group rounded to binary16 with
  round-to-nearest-even; a maximum that rounds to infinity, or any NaN/Inf weight, is an
  error (the page's Python demo does not meet either case);
* products: y[b][n] = sum_k w_hat[n][k] * x[b][k] computed in FP64 from the decoded
  binary16/bfloat16 inputs; a[b][n] = sum_k |w_hat[n][k] * x[b][k]| sizes the tolerance
  |y - y_ref| <= 2e-3 * a + 1e-5 for the FP32-accumulated value; a result stored as
  binary16 / bfloat16 is additionally allowed half an ulp of that format (bfloat16's unit
  roundoff 2^-8 is larger than 2e-3, so the bound cannot apply to the stored value alone).
"""

from __future__ import annotations

import numpy as np

GROUP = 128          # [P1] box: "cada 128 pesos comparten un factor de escala FP16"
FMT_1BIT = 1
FMT_TERNARY = 2
FMT_TERNARY5 = 3     # ternary codes stored 5 per byte (base 3), 26 bytes per 128-weight group
T5_GROUP_BYTES = 26  # 25 bytes of 5 digits + 1 byte of 3 digits
TOL_REL = 2e-3
TOL_ABS = 1e-5


class OracleError(ValueError):
    """Raised for inputs the method rejects; ``kind`` names the reason."""

    def __init__(self, kind: str, msg: str):
        super().__init__(f"{kind}: {msg}")
        self.kind = kind


# ---------------------------------------------------------------------------------------
# IEEE-754 codecs written from the format definitions (binary16: 1 sign, 5 exponent with
# bias 15, 10 fraction bits; bfloat16: 1 sign, 8 exponent with bias 127, 7 fraction bits).
# ---------------------------------------------------------------------------------------

def f16_bits_to_f64(bits) -> np.ndarray:
    """Decode binary16 bit patterns to float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where(b >> 15, -1.0, 1.0)
    exp = (b >> 10) & 0x1F
    frac = (b & 0x3FF).astype(np.float64)
    sub = frac * 2.0 ** -24                                    # exponent field 0
    nrm = (1024.0 + frac) * np.exp2((exp - 25).astype(np.float64))
    out = np.where(exp == 0, sub, nrm)
    out = np.where(exp == 31, np.where(frac == 0, np.inf, np.nan), out)
    return sign * out


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Decode bfloat16 bit patterns to float64 (exact)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.int64)
    sign = np.where(b >> 15, -1.0, 1.0)
    exp = (b >> 7) & 0xFF
    frac = (b & 0x7F).astype(np.float64)
    sub = frac * 2.0 ** -133
    nrm = (128.0 + frac) * np.exp2((exp - 134).astype(np.float64))
    out = np.where(exp == 0, sub, nrm)
    out = np.where(exp == 255, np.where(frac == 0, np.inf, np.nan), out)
    return sign * out


def f64_to_f16_bits_rne(values) -> np.ndarray:
    """Round float64 values to binary16 with round-to-nearest, ties to even.

    Intended for values that are exactly representable in float64 (float32 inputs are).
    NaN maps to 0x7E00; overflow maps to +/-infinity (0x7C00 / 0xFC00).
    """
    v = np.asarray(values, dtype=np.float64)
    neg = np.signbit(v)
    a = np.abs(v)
    out = np.zeros(a.shape, dtype=np.int64)
    finite = np.isfinite(a)
    # exponent of the leading bit: a = m * 2**e2 with m in [0.5, 1)
    _, e2 = np.frexp(np.where(finite & (a > 0), a, 1.0))
    e = e2.astype(np.int64) - 1                                # a in [2**e, 2**(e+1))
    subn = a < 2.0 ** -14
    # subnormal grid: multiples of 2**-24
    q_sub = np.rint(np.where(finite, a, 0.0) * 2.0 ** 24)      # rint = ties to even
    # normal grid: 11 significant bits
    q_nrm = np.rint(np.where(finite, a, 0.0) * np.exp2((10 - e).astype(np.float64)))
    carry = q_nrm >= 2048.0
    e_n = np.where(carry, e + 1, e)
    q_n = np.where(carry, 1024.0, q_nrm)
    nrm_bits = ((e_n + 15) << 10) | (q_n.astype(np.int64) - 1024)
    nrm_bits = np.where(e_n + 15 >= 31, 0x7C00, nrm_bits)
    out = np.where(subn, q_sub.astype(np.int64), nrm_bits)    # q_sub == 1024 is 2**-14
    out = np.where(np.isinf(a), 0x7C00, out)
    out = np.where(np.isnan(a), 0x7E00, out)
    out = np.where(neg & ~np.isnan(a), out | 0x8000, out)
    return out.astype(np.uint16)


def f64_to_bf16_bits_rne(values) -> np.ndarray:
    """Round float64 values to bfloat16 with round-to-nearest, ties to even.

    bfloat16: 8 significant bits, exponent bias 127, normal minimum 2^-126, subnormal spacing
    2^-133, largest finite (2 - 2^-7) * 2^127.  Intended for values exactly representable in
    float64 (binary16 and float32 values are).  NaN maps to 0x7FC0; overflow to +/-infinity.
    """
    v = np.asarray(values, dtype=np.float64)
    neg = np.signbit(v)
    a = np.abs(v)
    finite = np.isfinite(a)
    _, e2 = np.frexp(np.where(finite & (a > 0), a, 1.0))
    e = e2.astype(np.int64) - 1                                # a in [2**e, 2**(e+1))
    subn = a < 2.0 ** -126
    q_sub = np.rint(np.where(finite & subn, a, 0.0) * 2.0 ** 133)   # multiples of 2**-133
    q_nrm = np.rint(np.where(finite, a, 0.0) * np.exp2((7 - e).astype(np.float64)))
    carry = q_nrm >= 256.0
    e_n = np.where(carry, e + 1, e)
    q_n = np.where(carry, 128.0, q_nrm)
    nrm_bits = ((e_n + 127) << 7) | (q_n.astype(np.int64) - 128)
    nrm_bits = np.where(e_n + 127 >= 255, 0x7F80, nrm_bits)
    out = np.where(subn, q_sub.astype(np.int64), nrm_bits)    # q_sub == 128 is 2**-126
    out = np.where(np.isinf(a), 0x7F80, out)
    out = np.where(np.isnan(a), 0x7FC0, out)
    out = np.where(neg & ~np.isnan(a), out | 0x8000, out)
    return out.astype(np.uint16)


def encode_output_bits(values, dtype: str) -> np.ndarray:
    """float64 -> 16-bit patterns of 'f16' or 'bf16', round-to-nearest-even."""
    if dtype == "f16":
        return f64_to_f16_bits_rne(values)
    if dtype == "bf16":
        return f64_to_bf16_bits_rne(values)
    raise OracleError("dtype", f"unknown output dtype {dtype!r}")


def decode_activation_bits(bits, dtype: str) -> np.ndarray:
    """x or y stored as 16-bit patterns -> float64.  dtype is 'f16' or 'bf16'."""
    if dtype == "f16":
        return f16_bits_to_f64(bits)
    if dtype == "bf16":
        return bf16_bits_to_f64(bits)
    raise OracleError("dtype", f"unknown activation dtype {dtype!r}")


# ---------------------------------------------------------------------------------------
# Sizes.  [P1] box: 1 bit + 16/128 bit = 1.125 bpw; demo: 128/8 + 2 = 18 bytes per group.
# Ternary storage is 2-bit fields: 128*2/8 + 2 = 34 bytes per group (2.125 bpw).
# ---------------------------------------------------------------------------------------

def packed_bytes(fmt: int, n: int, k: int) -> tuple[int, int]:
    """(code bytes, scale bytes) of an n x k matrix in the packed format."""
    _check_shape(n, k)
    groups = n * (k // GROUP)
    if fmt == FMT_1BIT:
        return n * k // 8, groups * 2
    if fmt == FMT_TERNARY:
        return n * k // 4, groups * 2
    if fmt == FMT_TERNARY5:
        return groups * T5_GROUP_BYTES, groups * 2
    raise OracleError("format", f"unknown format {fmt}")


def bits_per_weight(fmt: int) -> float:
    c, s = packed_bytes(fmt, 1, GROUP)
    return 8.0 * (c + s) / GROUP


def _check_shape(n: int, k: int) -> None:
    if n < 1 or k < GROUP or k % GROUP:
        raise OracleError("shape", f"need n >= 1 and k a positive multiple of {GROUP}, got n={n} k={k}")


# ---------------------------------------------------------------------------------------
# Packing.
# ---------------------------------------------------------------------------------------

def pack_1bit(w) -> tuple[np.ndarray, np.ndarray]:
    """Sign / max-abs quantiser of [P1] section 7 applied to every (row, group).

    w: float32 [N][K].  For each group: scale = max |w| (exact in fp32), stored as binary16
    (round to nearest even); bit = 1 if w >= 0 else 0 (so +0.0 and -0.0 give 1).
    Returns codes uint8 [N][K/8] (LSB-first) and scales uint16 [N][K/128].
    """
    w = np.asarray(w, dtype=np.float32)
    if w.ndim != 2:
        raise OracleError("shape", "w must be 2-D")
    n, k = w.shape
    _check_shape(n, k)
    if not np.all(np.isfinite(w)):
        raise OracleError("nonfinite", "weights contain NaN or Inf")
    groups = w.reshape(n, k // GROUP, GROUP)
    smax = np.max(np.abs(groups), axis=2)                      # fp32, exact
    scales = f64_to_f16_bits_rne(smax.astype(np.float64))
    if np.any((scales & 0x7FFF) == 0x7C00):
        raise OracleError("range", "a group maximum rounds to binary16 infinity")
    bits = (w >= 0).astype(np.uint8)                           # 1 -> +scale, 0 -> -scale
    codes = np.packbits(bits, axis=1, bitorder="little")
    return codes, scales


def pack_ternary(t, s) -> tuple[np.ndarray, np.ndarray]:
    """Ternary codes t in {-1, 0, +1} ([P2] "Cómo funciona la compresión") and given
    binary16 scales -> packed 2-bit fields (f = t + 1) and the scales unchanged.

    t: int8 [N][K]; s: uint16 [N][K/128].
    """
    t = np.asarray(t)
    s = np.asarray(s, dtype=np.uint16)
    if t.ndim != 2:
        raise OracleError("shape", "t must be 2-D")
    n, k = t.shape
    _check_shape(n, k)
    if s.shape != (n, k // GROUP):
        raise OracleError("shape", f"scales must be {(n, k // GROUP)}, got {s.shape}")
    if not np.all((t == -1) | (t == 0) | (t == 1)):
        raise OracleError("code", "ternary codes must be -1, 0 or +1")
    f = (t.astype(np.int64) + 1).reshape(n, k // 4, 4)
    codes = (f[:, :, 0] | (f[:, :, 1] << 2) | (f[:, :, 2] << 4) | (f[:, :, 3] << 6)).astype(np.uint8)
    return codes, s.copy()


def pack_ternary5(t, s) -> tuple[np.ndarray, np.ndarray]:
    """Ternary codes stored five to a byte ([P4] es.news.hada.io topic 31450, comments: five
    three-state values fit one byte, 1.6 bits each; [P3] "Arquitectura del Sistema": 1.76
    effective bits per weight).  Reading used here: digit f = t + 1 in {0, 1, 2}; within each
    128-weight group, byte j holds weights 5j .. 5j+4 as sum_i f_(5j+i) 3^i (first weight in the
    lowest digit); byte 25 holds weights 125..127 (its two upper digits are 0).  26 bytes per
    group, row-major [N][26 K/128]; scales unchanged.
    """
    t = np.asarray(t)
    s = np.asarray(s, dtype=np.uint16)
    if t.ndim != 2:
        raise OracleError("shape", "t must be 2-D")
    n, k = t.shape
    _check_shape(n, k)
    if s.shape != (n, k // GROUP):
        raise OracleError("shape", f"scales must be {(n, k // GROUP)}, got {s.shape}")
    if not np.all((t == -1) | (t == 0) | (t == 1)):
        raise OracleError("code", "ternary codes must be -1, 0 or +1")
    g = k // GROUP
    f = np.zeros((n, g, 5 * T5_GROUP_BYTES), dtype=np.int64)
    f[:, :, :GROUP] = t.astype(np.int64).reshape(n, g, GROUP) + 1
    f = f.reshape(n, g, T5_GROUP_BYTES, 5)
    codes = sum(f[..., i] * 3 ** i for i in range(5)).astype(np.uint8)
    return codes.reshape(n, g * T5_GROUP_BYTES), s.copy()


# ---------------------------------------------------------------------------------------
# Unpacking and dequantisation: w_hat = s_g * t_i ([P2] "Cómo funciona la compresión").
# ---------------------------------------------------------------------------------------

def unpack_1bit(codes, k: int) -> np.ndarray:
    """codes uint8 [N][K/8] -> t int8 [N][K] in {-1, +1} ([P1]: 0 -> -1, 1 -> +1)."""
    codes = np.asarray(codes, dtype=np.uint8)
    b = np.unpackbits(codes, axis=1, bitorder="little")[:, :k].astype(np.int8)
    return (2 * b - 1).astype(np.int8)


def unpack_ternary(codes, k: int) -> np.ndarray:
    """codes uint8 [N][K/4] -> t int8 [N][K] in {-1, 0, +1}; field 3 is rejected."""
    codes = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    n = codes.shape[0]
    f = np.stack([(codes >> (2 * j)) & 3 for j in range(4)], axis=2).reshape(n, -1)[:, :k]
    if np.any(f == 3):
        raise OracleError("code", "field value 3 is not a ternary code")
    return (f - 1).astype(np.int8)


def unpack_ternary5(codes, k: int) -> np.ndarray:
    """codes uint8 [N][26 K/128] (five base-3 digits per byte) -> t int8 [N][K]; a byte above
    242, or a last byte of a group with a non-zero upper digit, is rejected."""
    codes = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    n, g = codes.shape[0], k // GROUP
    b = codes.reshape(n, g, T5_GROUP_BYTES)
    if np.any(b > 242) or np.any(b[:, :, -1] >= 27):
        raise OracleError("code", "not a base-3 code byte of this layout")
    digits = np.stack([(b // 3 ** i) % 3 for i in range(5)], axis=3).reshape(n, g, 5 * T5_GROUP_BYTES)
    return (digits[:, :, :GROUP] - 1).reshape(n, k).astype(np.int8)


def dequantize(fmt: int, codes, scales, k: int) -> np.ndarray:
    """Packed weights -> dense float64 [N][K] with w_hat[n][k] = s[n][k // 128] * t[n][k]."""
    if fmt == FMT_1BIT:
        t = unpack_1bit(codes, k)
    elif fmt == FMT_TERNARY:
        t = unpack_ternary(codes, k)
    elif fmt == FMT_TERNARY5:
        t = unpack_ternary5(codes, k)
    else:
        raise OracleError("format", f"unknown format {fmt}")
    s = f16_bits_to_f64(np.asarray(scales, dtype=np.uint16))
    return t.astype(np.float64) * np.repeat(s, GROUP, axis=1)


# ---------------------------------------------------------------------------------------
# Embedding rows.  The low-bit representation also covers the embedding table ([P2] "Cómo
# funciona la compresión"; [P4] es.news.hada.io topic 31450, "Configuración multimodal y de bajo
# bit de extremo a extremo"), so the step before the first GEMV dequantises one table row per
# token: out[i][k] = s[id_i][k // 128] * t[id_i][k], rounded to the output format.
# ---------------------------------------------------------------------------------------

def embed_rows(fmt: int, codes, scales, k: int, ids, out_dtype: str) -> tuple[np.ndarray, np.ndarray]:
    """ids int [count] -> (out 16-bit patterns [count][K], bad bool [count]).

    A row id outside [0, N) is not a table row: its output row is all +0 and it is flagged.
    """
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.uint16)
    n = codes.shape[0]
    ids = np.asarray(ids, dtype=np.int64).reshape(-1)
    bad = (ids < 0) | (ids >= n)
    rows = np.where(bad, 0, ids)
    w = dequantize(fmt, codes[rows], scales[rows], k) if len(ids) else np.zeros((0, k))
    out = encode_output_bits(w, out_dtype)
    out[bad] = 0
    return out, bad


# ---------------------------------------------------------------------------------------
# Products.  y = W x for a batch of activation rows (decode GEMV, small-batch verify GEMV)
# and for M token rows (prefill GEMM); they are the same definition.
# ---------------------------------------------------------------------------------------

def matvec(fmt: int, codes, scales, k: int, x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """x float64 [B][K] -> (y [B][N], a [B][N]) with y = x W_hat^T and a = |x| |W_hat|^T."""
    w = dequantize(fmt, codes, scales, k)
    x = np.asarray(x, dtype=np.float64)
    if x.ndim != 2 or x.shape[1] != k:
        raise OracleError("shape", f"x must be [B][{k}]")
    y = x @ w.T
    a = np.abs(x) @ np.abs(w).T
    return y, a


def gemm(fmt: int, codes, scales, k: int, x: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """Prefill product Y[m][n] = sum_k X[m][k] w_hat[n][k] (same definition, M rows)."""
    return matvec(fmt, codes, scales, k, x)


# ---------------------------------------------------------------------------------------
# SiLU-gated feed-forward pair: h = silu(W_gate x) * (W_up x).  The pages name the fastest decode
# kernels as specialised at the matvec / FFN level ([P5] "Detalles técnicos") and the models as
# builds of a Qwen3-family base ([P2]), whose feed-forward block gates the up projection with
# silu(z) = z * sigmoid(z) = z / (1 + e^-z) of the gate projection.
# ---------------------------------------------------------------------------------------

SILU_SLOPE_MAX = 1.0999     # bounds max over z of |d/dz silu(z)| = 1.09984 (near z = 2.40)


def silu(z) -> np.ndarray:
    """z / (1 + e^-z) in float64; e^-z overflowing to infinity gives the limit, a signed zero."""
    z = np.asarray(z, dtype=np.float64)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu(fmt: int, codes_g, scales_g, codes_u, scales_u, k: int, x: np.ndarray):
    """x float64 [B][K] -> (h [B][N], g, a_g, u, a_u): h = silu(g) * u with g, u the two products
    and a_g, a_u their sums of absolute terms (for the tolerance)."""
    g, a_g = matvec(fmt, codes_g, scales_g, k, x)
    u, a_u = matvec(fmt, codes_u, scales_u, k, x)
    return silu(g) * u, g, a_g, u, a_u


def swiglu_tolerance(h_ref, g, a_g, u, a_u, h_test=None, out_dtype: str | None = None) -> np.ndarray:
    """Allowed |h_test - h_ref| when g and u are each FP32-accumulated within the product bound
    dg = 2e-3 * a_g + 1e-5, du = 2e-3 * a_u + 1e-5 and h is formed from them in FP32:
    |silu(g') u' - silu(g) u| <= SILU_SLOPE_MAX * dg * (|u| + du) + |silu(g)| * du, plus 1e-6 |h|
    for the FP32 evaluation of silu and the product, plus half an ulp of the output format."""
    dg = TOL_REL * np.asarray(a_g) + TOL_ABS
    du = TOL_REL * np.asarray(a_u) + TOL_ABS
    h_ref = np.asarray(h_ref, dtype=np.float64)
    mag = np.abs(h_ref)
    if h_test is not None:
        mag = np.maximum(mag, np.abs(np.asarray(h_test, dtype=np.float64)))
    return (SILU_SLOPE_MAX * dg * (np.abs(u) + du) + np.abs(silu(g)) * du + 1e-6 * mag
            + output_half_ulp(mag, out_dtype))


def output_half_ulp(v, dtype: str | None) -> np.ndarray:
    """Half a unit in the last place of the output format at magnitude |v| (0 if dtype is None).

    binary16: 11 significant bits, subnormal spacing 2^-24; bfloat16: 8 significant bits,
    subnormal spacing 2^-133.
    """
    v = np.abs(np.asarray(v, dtype=np.float64))
    if dtype is None:
        return np.zeros_like(v)
    if dtype == "f16":
        bits, emin, tiny = 11, -14, 2.0 ** -24
    elif dtype == "bf16":
        bits, emin, tiny = 8, -126, 2.0 ** -133
    else:
        raise OracleError("dtype", f"unknown output dtype {dtype!r}")
    _, e2 = np.frexp(np.where(v > 0, v, 1.0))
    e = np.maximum(e2.astype(np.int64) - 1, emin)          # binade of v (at least the normal minimum)
    ulp = np.where(v > 0, np.exp2((e - (bits - 1)).astype(np.float64)), tiny)
    return 0.5 * np.maximum(ulp, tiny)


def tolerance(y_ref, a, y_test=None, out_dtype: str | None = None) -> np.ndarray:
    """Allowed |y_test - y_ref|: 2e-3 * a + 1e-5 for the FP32-accumulated value, plus half an ulp
    of the output format when the result is stored as binary16 / bfloat16 (a stored bfloat16 has
    unit roundoff 2^-8 > 2e-3, so the final rounding is granted on top of the accumulation bound;
    the binade is taken from the larger of |y_ref| and |y_test|)."""
    mag = np.abs(np.asarray(y_ref, dtype=np.float64))
    if y_test is not None:
        mag = np.maximum(mag, np.abs(np.asarray(y_test, dtype=np.float64)))
    return TOL_REL * np.asarray(a) + TOL_ABS + output_half_ulp(mag, out_dtype)


def within_tolerance(y_test, y_ref, a, out_dtype: str | None = None) -> np.ndarray:
    """Element-wise |y_test - y_ref| <= tolerance(y_ref, a, y_test, out_dtype)."""
    y_test = np.asarray(y_test, dtype=np.float64)
    return np.abs(y_test - y_ref) <= tolerance(y_ref, a, y_test, out_dtype)


def tolerance_ratio(y_test, y_ref, a, out_dtype: str | None = None) -> float:
    """max over elements of |y_test - y_ref| / tolerance; <= 1 means pass."""
    y_test = np.asarray(y_test, dtype=np.float64)
    r = np.abs(y_test - y_ref) / tolerance(y_ref, a, y_test, out_dtype)
    return float(np.max(r)) if r.size else 0.0
