"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle legs.

This module only draws random numbers with the shapes and distributions of the benchmark
workloads.  It holds none of the method's arithmetic (no quantisation, packing, decoding
or products), so both the CUDA path and the CPU oracle can take their inputs from here.
Everything is generated on the CPU with ``torch.Generator`` and returned as CPU tensors;
callers copy to the device themselves.

Workloads (group size 128 along K, batch = number of activation rows):

* ``c1``  1-bit GEMV 2048 x 2048; W ~ N(0, 0.1) fp32, packed by sign / max-abs; x fp16
  N(0, 1); batch 1.
* ``c2``  ternary decode layer set of a 1.7B-class block (hidden 2048, FFN 6144): q, k, v, o
  2048 x 2048, gate, up 6144 x 2048, down 2048 x 6144; codes iid {-1, 0, +1} with
  probabilities (0.3, 0.4, 0.3); scales |N(0, 0.02)| rounded to fp16; x fp16 N(0, 1); batch 1.
* ``c3``  1-bit LM head 151936 x 2048; W ~ N(0, 0.05) fp32; x bf16 N(0, 1); batch 1 and 4.
* ``c4``  27B-class decode layer set (hidden 5120, FFN 17408), ternary and 1-bit: q, o
  5120 x 5120, gate, up 17408 x 5120, down 5120 x 17408; x bf16 N(0, 1); batch 1 and 5.
  The 1-bit weights are drawn from N(0, 0.02) (the workload does not fix sigma).
* ``c5``  ternary prefill GEMM: 512 tokens x K 5120 -> N 17408; X bf16 N(0, 1).
"""

from __future__ import annotations

from dataclasses import dataclass, field

import torch

GROUP = 128


@dataclass(frozen=True)
class Matrix:
    name: str
    n: int          # output rows
    k: int          # reduction length


@dataclass(frozen=True)
class Workload:
    key: str
    fmt: str                    # "1bit" or "ternary"
    matrices: tuple             # tuple[Matrix, ...]
    xdtype: str                 # "f16" or "bf16"
    batches: tuple              # activation rows per product (GEMV batch or GEMM M)
    seed: int
    w_sigma: float = 0.0        # 1-bit: std of the fp32 weights before packing
    s_sigma: float = 0.02       # ternary: std of the normal whose |.| gives the scales
    p_ternary: tuple = (0.3, 0.4, 0.3)
    gemm: bool = False
    note: str = field(default="", compare=False)

    @property
    def weights(self) -> int:
        return sum(m.n * m.k for m in self.matrices)


def _block(h: int, f: int, full_qkv: bool) -> tuple:
    if full_qkv:
        mats = [Matrix("q", h, h), Matrix("k", h, h), Matrix("v", h, h), Matrix("o", h, h)]
    else:
        mats = [Matrix("q", h, h), Matrix("o", h, h)]
    mats += [Matrix("gate", f, h), Matrix("up", f, h), Matrix("down", h, f)]
    return tuple(mats)


WORKLOADS = {
    "c1": Workload("c1", "1bit", (Matrix("w", 2048, 2048),), "f16", (1,), seed=1001, w_sigma=0.1),
    "c2": Workload("c2", "ternary", _block(2048, 6144, True), "f16", (1,), seed=1002),
    "c3": Workload("c3", "1bit", (Matrix("lm_head", 151936, 2048),), "bf16", (1, 4), seed=1003,
                   w_sigma=0.05),
    "c4t": Workload("c4t", "ternary", _block(5120, 17408, False), "bf16", (1, 5), seed=1004),
    "c4b": Workload("c4b", "1bit", _block(5120, 17408, False), "bf16", (1, 5), seed=1014,
                    w_sigma=0.02),
    "c5": Workload("c5", "ternary", (Matrix("up", 17408, 5120),), "bf16", (512,), seed=1005,
                   gemm=True),
}


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def weights_fp32(n: int, k: int, sigma: float, seed: int) -> torch.Tensor:
    """Dense fp32 weights N(0, sigma^2), shape [n][k] (input of the 1-bit packer)."""
    return torch.randn(n, k, generator=_gen(seed), dtype=torch.float32) * sigma


def ternary_codes(n: int, k: int, seed: int, p=(0.3, 0.4, 0.3)) -> torch.Tensor:
    """iid codes in {-1, 0, +1} with probabilities p, int8 [n][k]."""
    u = torch.rand(n, k, generator=_gen(seed), dtype=torch.float32)
    t = torch.zeros(n, k, dtype=torch.int8)
    t[u < p[0]] = -1
    t[u >= p[0] + p[1]] = 1
    return t


def ternary_scales_bits(n: int, k: int, sigma: float, seed: int) -> torch.Tensor:
    """|N(0, sigma^2)| drawn in fp32, stored as fp16; returned as int16 bit patterns [n][k/128]."""
    s = torch.randn(n, k // GROUP, generator=_gen(seed), dtype=torch.float32).abs() * sigma
    return s.to(torch.float16).view(torch.int16)


def activations(b: int, k: int, dtype: str, seed: int) -> torch.Tensor:
    """x ~ N(0, 1) in fp16 or bf16, shape [b][k]."""
    tdt = {"f16": torch.float16, "bf16": torch.bfloat16}[dtype]
    return torch.randn(b, k, generator=_gen(seed), dtype=torch.float32).to(tdt)


def matrix_seed(w: Workload, index: int, salt: int = 0) -> int:
    return w.seed * 1000 + index * 10 + salt


def matrix_inputs(w: Workload, index: int):
    """Raw inputs of matrix ``index`` of workload ``w``.

    1-bit: ``{"w": fp32 [n][k]}``.  Ternary: ``{"t": int8 [n][k], "s": int16 bits [n][k/128]}``.
    """
    m = w.matrices[index]
    if w.fmt == "1bit":
        return {"w": weights_fp32(m.n, m.k, w.w_sigma, matrix_seed(w, index))}
    return {"t": ternary_codes(m.n, m.k, matrix_seed(w, index), w.p_ternary),
            "s": ternary_scales_bits(m.n, m.k, w.s_sigma, matrix_seed(w, index, 1))}


def workload_activations(w: Workload, index: int, batch: int) -> torch.Tensor:
    m = w.matrices[index]
    return activations(batch, m.k, w.xdtype, matrix_seed(w, index, 2 + batch))


def activations_wide_range(b: int, k: int, dtype: str, seed: int) -> torch.Tensor:
    """Activation rows that stress the numeric range of the 16-bit inputs, shape [b][k] (b >= 5).

    bfloat16 rows: 0 N(0,1) scaled so that max |x| = 3e38 (near the largest finite bfloat16);
    1 N(0,1) * 1e30; 2 N(0,1) * 1e5; 3 N(0,1) * 1e-4 with one element of magnitude ~1e4 per 128
    (ratio 1e8 inside a group); 4 all zeros (+0), 5 N(0,1) * 1e-4 with one ~1e4 element in the
    whole row, 6 N(0,1) with +-0 in every fourth position, 7 N(0,1) * 2^-120 (tiny normals).
    binary16 rows: 0 N(0,1) with one element of magnitude ~6e4 per 128; 1 subnormals
    (N(0,1) * 2^-20); 2 N(0,1) * 1e-3 with a few elements ~3e4; 3 N(0,1); 4 all zeros (+0);
    5 N(0,1) with +-0 in every fourth position; 6 N(0,1) * 100; 7 N(0,1) * 2^-14.
    Rows beyond b are dropped; rows are chosen by index modulo 8.
    """
    g = _gen(seed)
    z = torch.randn(8, k, generator=g, dtype=torch.float64)
    u = torch.rand(8, k, generator=g, dtype=torch.float64)
    pos_group = (torch.arange(k) % GROUP) == (seed % GROUP)
    one_pos = torch.arange(k) == ((seed * 7919) % k)
    rows = torch.zeros(8, k, dtype=torch.float64)
    if dtype == "bf16":
        rows[0] = z[0] / z[0].abs().max() * 3e38
        rows[1] = z[1] * 1e30
        rows[2] = z[2] * 1e5
        rows[3] = torch.where(pos_group, torch.sign(z[3]) * (1e4 + 1e3 * u[3]), z[3] * 1e-4)
        rows[4] = 0.0
        rows[5] = torch.where(one_pos, torch.sign(z[5]) * (1e4 + 1e3 * u[5]), z[5] * 1e-4)
        rows[6] = torch.where(torch.arange(k) % 4 == 0, torch.where(u[6] < 0.5, 0.0, -0.0), z[6])
        rows[7] = z[7] * 2.0 ** -120
        tdt = torch.bfloat16
    else:
        rows[0] = torch.where(pos_group, torch.sign(z[0]) * (5e4 + 1e4 * u[0]), z[0])
        rows[1] = z[1] * 2.0 ** -20
        rows[2] = torch.where(torch.arange(k) % 509 == 3, torch.sign(z[2]) * 3e4, z[2] * 1e-3)
        rows[3] = z[3]
        rows[4] = 0.0
        rows[5] = torch.where(torch.arange(k) % 4 == 0, torch.where(u[5] < 0.5, 0.0, -0.0), z[5])
        rows[6] = z[6] * 100.0
        rows[7] = z[7] * 2.0 ** -14
        tdt = torch.float16
    idx = torch.arange(b) % 8
    return rows[idx].to(torch.float32).to(tdt)
