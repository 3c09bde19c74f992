"""Shared helpers for the GPU parity tests: move synthetic inputs to the device, call the library,
and compare with the CPU oracle element by element."""

import numpy as np
import torch

from oracle import lb_oracle as orc


def u16(t: torch.Tensor) -> np.ndarray:
    """Any 16-bit tensor (fp16 / bf16 / int16) -> numpy uint16 bit patterns."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.detach().contiguous().cpu().numpy().view(np.uint8)


def xdt_name(dtype: torch.dtype) -> str:
    return {torch.float16: "f16", torch.bfloat16: "bf16"}[dtype]


def oracle_pack(fmt: str, inputs: dict):
    if fmt == "1bit":
        return orc.pack_1bit(inputs["w"].numpy())
    return orc.pack_ternary(inputs["t"].numpy(), inputs["s"].numpy().view(np.uint16))


def oracle_products(fmt: str, codes, scales, k: int, x: torch.Tensor, rows=None):
    """y_ref, a (float64 [B][rows]) for the selected weight rows (all if rows is None)."""
    f = orc.FMT_1BIT if fmt == "1bit" else orc.FMT_TERNARY
    if rows is not None:
        codes, scales = codes[rows], scales[rows]
    xv = orc.decode_activation_bits(u16(x), xdt_name(x.dtype))
    return orc.matvec(f, codes, scales, k, xv)


def check_products(y_dev: torch.Tensor, y_ref, a, what: str, cols=None):
    """Compare device output (16-bit, [B][N]) against oracle values; raises with the worst element."""
    yb = u16(y_dev)
    if cols is not None:
        yb = yb[:, cols]
    dt = xdt_name(y_dev.dtype)
    yv = orc.decode_activation_bits(yb, dt)
    ok = orc.within_tolerance(yv, y_ref, a, dt)
    if not ok.all():
        bad = np.argwhere(~ok)
        b, n = bad[0]
        raise AssertionError(f"{what}: {len(bad)} of {ok.size} outside tolerance; first at {tuple(bad[0])}: "
                             f"got {yv[b, n]!r} want {y_ref[b, n]!r} (a={a[b, n]!r}); "
                             f"worst ratio {orc.tolerance_ratio(yv, y_ref, a, dt):.3f}")
    return orc.tolerance_ratio(yv, y_ref, a, dt)
