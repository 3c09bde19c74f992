"""Convenience wrappers over the C ABI that allocate outputs as torch CUDA tensors.

Every function calls exactly one liblb entry point (plus torch allocations); no arithmetic of the
method happens here.
"""

from __future__ import annotations

import contextlib
from dataclasses import dataclass, field

import torch

from . import lb

_TORCH = {lb.LB_F16: torch.float16, lb.LB_BF16: torch.bfloat16}


def _alloc_on(stream):
    """Context for allocating a call's outputs and workspace: a torch stream owns what is allocated
    under it, so torch's caching allocator does not hand the memory to another stream while the
    call's kernels may still use it.  A raw stream handle (or None) allocates on the current
    stream, and keeping those buffers alive is then the caller's job."""
    return torch.cuda.stream(stream) if isinstance(stream, torch.cuda.Stream) else contextlib.nullcontext()


def dtype_code(t: torch.dtype) -> int:
    if t == torch.float16:
        return lb.LB_F16
    if t == torch.bfloat16:
        return lb.LB_BF16
    raise TypeError(f"activations must be float16 or bfloat16, got {t}")


@dataclass
class PackedWeight:
    """A packed matrix on the device: codes uint8 plane + scales (binary16 bits, int16 storage)."""
    fmt: int
    n: int
    k: int
    codes: torch.Tensor
    scales: torch.Tensor
    _struct: object = field(default=None, repr=False, compare=False)

    def struct(self) -> lb.lb_weight:
        """The C lb_weight of this matrix (rebuilt only when a plane was replaced)."""
        key = (self.fmt, self.n, self.k, self.codes.data_ptr(), self.scales.data_ptr())
        if self._struct is None or self._struct[0] != key:
            self._struct = (key, lb.make_weight(self.fmt, self.n, self.k, self.codes, self.scales))
        return self._struct[1]

    @classmethod
    def empty(cls, fmt: int, n: int, k: int, device="cuda") -> "PackedWeight":
        cb, sb = lb.lb_packed_bytes(fmt, n, k)
        return cls(fmt, n, k, torch.empty(cb, dtype=torch.uint8, device=device),
                   torch.empty(sb // 2, dtype=torch.int16, device=device))


def pack_1bit(w: torch.Tensor, stream=None) -> PackedWeight:
    """fp32 [n][k] CUDA tensor -> PackedWeight via lb_pack_1bit."""
    assert w.is_cuda and w.dtype == torch.float32 and w.is_contiguous() and w.dim() == 2
    n, k = w.shape
    pw = PackedWeight.empty(lb.LB_FMT_1BIT_G128, n, k, device=w.device)
    lb.lb_pack_1bit(w, n, k, pw.codes, pw.scales, stream)
    return pw


def pack_ternary(t: torch.Tensor, s: torch.Tensor, stream=None) -> PackedWeight:
    """int8 codes [n][k] + binary16 scales [n][k/128] (int16 or float16 storage) -> PackedWeight."""
    assert t.is_cuda and t.dtype == torch.int8 and t.is_contiguous() and t.dim() == 2
    n, k = t.shape
    pw = PackedWeight.empty(lb.LB_FMT_TERNARY_G128, n, k, device=t.device)
    lb.lb_pack_ternary(t, s.contiguous(), n, k, pw.codes, pw.scales, stream)
    return pw


def pack_ternary5(t: torch.Tensor, s: torch.Tensor, stream=None) -> PackedWeight:
    """int8 codes [n][k] + binary16 scales [n][k/128] -> PackedWeight, five codes per byte."""
    assert t.is_cuda and t.dtype == torch.int8 and t.is_contiguous() and t.dim() == 2
    n, k = t.shape
    pw = PackedWeight.empty(lb.LB_FMT_TERNARY5_G128, n, k, device=t.device)
    lb.lb_pack_ternary5(t, s.contiguous(), n, k, pw.codes, pw.scales, stream)
    return pw


def gemv(W: PackedWeight, x: torch.Tensor, y: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """y[b][n] = W x[b] for x [batch][k] (batch 1..8), output in the dtype of x."""
    assert x.is_cuda and x.is_contiguous() and x.dim() == 2 and x.shape[1] == W.k
    if y is None:
        with _alloc_on(stream):
            y = torch.empty(x.shape[0], W.n, dtype=x.dtype, device=x.device)
    lb.lb_gemv(W.struct(), x, dtype_code(x.dtype), x.shape[0], y, stream)
    return y


def gemv_batched(problems, ys=None, stream=None) -> list:
    """Several GEMVs in one launch: problems = [(PackedWeight, x)], every x [batch][k] of one dtype
    and batch (x tensors may be shared).  Returns the outputs y [batch][n] (or fills `ys`)."""
    assert problems
    x0 = problems[0][1]
    batch, dt = x0.shape[0], x0.dtype
    if ys is None:
        with _alloc_on(stream):
            ys = [torch.empty(batch, W.n, dtype=dt, device=x.device) for W, x in problems]
    for W, x in problems:
        assert x.is_cuda and x.is_contiguous() and x.dim() == 2 and x.shape == (batch, W.k) and x.dtype == dt
    lb.lb_gemv_batched([(W.struct(), x, y) for (W, x), y in zip(problems, ys)], dtype_code(dt), batch, stream)
    return ys


def gemv_swiglu(Wg: PackedWeight, Wu: PackedWeight, x: torch.Tensor, h: torch.Tensor | None = None,
                stream=None) -> torch.Tensor:
    """h[b] = silu(Wg x[b]) * (Wu x[b]) for x [batch][k] (batch 1..8), output in the dtype of x."""
    assert x.is_cuda and x.is_contiguous() and x.dim() == 2 and x.shape[1] == Wg.k
    if h is None:
        with _alloc_on(stream):
            h = torch.empty(x.shape[0], Wg.n, dtype=x.dtype, device=x.device)
    lb.lb_gemv_swiglu(Wg.struct(), Wu.struct(), x, dtype_code(x.dtype), x.shape[0], h, stream)
    return h


def gemm(W: PackedWeight, x: torch.Tensor, out_dtype: torch.dtype = torch.bfloat16,
         y: torch.Tensor | None = None, workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Y[m][n] = X W^T for X [m][k]; output dtype out_dtype."""
    assert x.is_cuda and x.is_contiguous() and x.dim() == 2 and x.shape[1] == W.k
    m = x.shape[0]
    xdt = dtype_code(x.dtype)
    need = lb.lb_gemm_workspace_bytes(m, W.n, W.k, xdt)
    with _alloc_on(stream):
        if y is None:
            y = torch.empty(m, W.n, dtype=out_dtype, device=x.device)
        if workspace is None or workspace.numel() < need:
            workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    lb.lb_gemm(W.struct(), x, xdt, m, y, dtype_code(y.dtype), workspace, workspace.numel(), stream)
    return y


def embed(W: PackedWeight, ids: torch.Tensor, out_dtype: torch.dtype = torch.bfloat16,
          out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Embedding rows out[i] = dequantised row ids[i] of the packed table W (ids: int32 CUDA tensor)."""
    assert ids.is_cuda and ids.dtype == torch.int32 and ids.is_contiguous() and ids.dim() == 1
    count = ids.shape[0]
    if out is None:
        with _alloc_on(stream):
            out = torch.empty(count, W.k, dtype=out_dtype, device=ids.device)
    assert out.is_cuda and out.is_contiguous() and out.shape == (count, W.k)
    lb.lb_embed(W.struct(), ids, count, out, dtype_code(out.dtype), stream)
    return out
