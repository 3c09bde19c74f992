"""Thin ctypes binding of liblb (see include/lb.h).  Argument marshalling only.

Each ``lb_*`` function here has the name, arguments and meaning of the C entry point: device
buffers are passed as torch CUDA tensors (or raw integer device addresses), ``stream`` is a
``torch.cuda.Stream``, a raw ``cudaStream_t`` integer or ``None`` for torch's current stream.
A non-OK status raises :class:`LBError`.  Every computation runs in liblb's CUDA kernels; there is
no Python or CPU fallback, and importing this module fails loudly if liblb.so has not been built.
"""

from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
# LB_LIBRARY selects another build of the same library (the phase-trace build, see trace_gemv.py)
LIB_PATH = os.environ.get("LB_LIBRARY") or os.path.join(HERE, "liblb.so")

LB_OK = 0
LB_FMT_1BIT_G128 = 1
LB_FMT_TERNARY_G128 = 2
LB_FMT_TERNARY5_G128 = 3
LB_F16 = 1
LB_BF16 = 2
FORMATS = {"1bit": LB_FMT_1BIT_G128, "ternary": LB_FMT_TERNARY_G128, "ternary5": LB_FMT_TERNARY5_G128}
DTYPES = {"f16": LB_F16, "bf16": LB_BF16}

STATUS_NAMES = {0: "LB_OK", 1: "LB_ERR_NULL", 2: "LB_ERR_SHAPE", 3: "LB_ERR_ALIGN", 4: "LB_ERR_DTYPE",
                5: "LB_ERR_CODE", 6: "LB_ERR_NONFINITE", 7: "LB_ERR_RANGE", 8: "LB_ERR_CUDA",
                9: "LB_ERR_UNSUPPORTED", 10: "LB_ERR_WORKSPACE"}

# Symbols declared in include/lb.h (checked by the tests against the header and the library).
EXPORTED = ("lb_status_string", "lb_last_error", "lb_version", "lb_packed_bytes", "lb_pack_1bit",
            "lb_pack_ternary", "lb_gemv", "lb_gemm_workspace_bytes", "lb_gemm", "lb_device_error",
            "lb_gemm_noalloc", "lb_gemv_batched", "lb_embed", "lb_gemv_swiglu", "lb_pack_ternary5",
            "lb_read_probe")
LB_GEMM_NOALLOC_SCRATCH_BYTES = (8 << 20) + (64 << 10)
LB_GEMV_BATCH_MAX = 8


class LBError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        self.name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{where}: {self.name}: {detail}")


class lb_weight(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("reserved", ctypes.c_int32), ("n", ctypes.c_int64),
                ("k", ctypes.c_int64), ("codes", ctypes.c_void_p), ("scales", ctypes.c_void_p)]


class lb_gemv_problem(ctypes.Structure):
    _fields_ = [("W", lb_weight), ("x", ctypes.c_void_p), ("y", ctypes.c_void_p)]


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"liblb.so not found at {LIB_PATH}; build it with "
                          "`python -m gemm_lb_gemv_02_b300.build` (the CUDA library is required)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    sz_p = ctypes.POINTER(ctypes.c_size_t)
    sig = {
        "lb_status_string": ([i32], ctypes.c_char_p),
        "lb_last_error": ([], ctypes.c_char_p),
        "lb_version": ([], i32),
        "lb_packed_bytes": ([i32, i64, i64, sz_p, sz_p], i32),
        "lb_pack_1bit": ([vp, i64, i64, vp, vp, vp], i32),
        "lb_pack_ternary": ([vp, vp, i64, i64, vp, vp, vp], i32),
        "lb_pack_ternary5": ([vp, vp, i64, i64, vp, vp, vp], i32),
        "lb_gemv": ([ctypes.POINTER(lb_weight), vp, i32, i32, vp, vp], i32),
        "lb_gemm_workspace_bytes": ([i64, i64, i64, i32, sz_p], i32),
        "lb_gemm": ([ctypes.POINTER(lb_weight), vp, i32, i64, vp, i32, vp, ctypes.c_size_t, vp], i32),
        "lb_device_error": ([ctypes.POINTER(ctypes.c_uint32), i32], i32),
        "lb_gemm_noalloc": ([ctypes.POINTER(lb_weight), vp, i32, i64, vp, i32, vp], i32),
        "lb_gemv_batched": ([ctypes.POINTER(lb_gemv_problem), i32, i32, i32, vp], i32),
        "lb_embed": ([ctypes.POINTER(lb_weight), vp, i64, vp, i32, vp], i32),
        "lb_gemv_swiglu": ([ctypes.POINTER(lb_weight), ctypes.POINTER(lb_weight), vp, i32, i32, vp, vp], i32),
        "lb_read_probe": ([vp, ctypes.c_size_t, vp, vp], i32),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


_lib = _load()


def library():
    """The loaded ctypes.CDLL of liblb.so."""
    return _lib


def _ptr(obj) -> int | None:
    if obj is None:
        return None
    if hasattr(obj, "data_ptr"):
        return obj.data_ptr()
    return int(obj)


_torch = None
_have_cuda = None


def _stream(stream) -> int | None:
    global _torch, _have_cuda
    if stream is None:
        if _have_cuda is None:
            import torch
            _torch = torch
            _have_cuda = torch.cuda.is_available()
            if _have_cuda:
                torch.cuda.init()
        if not _have_cuda:
            return None
        # torch's current stream on the current device, as a raw cudaStream_t
        return _torch._C._cuda_getCurrentRawStream(_torch._C._cuda_getDevice())
    if hasattr(stream, "cuda_stream"):
        return stream.cuda_stream
    return int(stream)


def _check(status: int, where: str) -> None:
    if status != LB_OK:
        raise LBError(status, where, _lib.lb_last_error().decode(errors="replace"))


def lb_status_string(status: int) -> str:
    return _lib.lb_status_string(status).decode()


def lb_last_error() -> str:
    return _lib.lb_last_error().decode(errors="replace")


def lb_version() -> int:
    return _lib.lb_version()


def lb_packed_bytes(fmt: int, n: int, k: int) -> tuple[int, int]:
    c, s = ctypes.c_size_t(), ctypes.c_size_t()
    _check(_lib.lb_packed_bytes(fmt, n, k, ctypes.byref(c), ctypes.byref(s)), "lb_packed_bytes")
    return c.value, s.value


def lb_pack_1bit(w, n: int, k: int, codes, scales, stream=None) -> None:
    _check(_lib.lb_pack_1bit(_ptr(w), n, k, _ptr(codes), _ptr(scales), _stream(stream)), "lb_pack_1bit")


def lb_pack_ternary(t, s_in, n: int, k: int, codes, scales, stream=None) -> None:
    _check(_lib.lb_pack_ternary(_ptr(t), _ptr(s_in), n, k, _ptr(codes), _ptr(scales), _stream(stream)),
           "lb_pack_ternary")


def lb_pack_ternary5(t, s_in, n: int, k: int, codes, scales, stream=None) -> None:
    _check(_lib.lb_pack_ternary5(_ptr(t), _ptr(s_in), n, k, _ptr(codes), _ptr(scales), _stream(stream)),
           "lb_pack_ternary5")


def make_weight(fmt: int, n: int, k: int, codes, scales) -> lb_weight:
    return lb_weight(fmt, 0, n, k, _ptr(codes), _ptr(scales))


def lb_gemv(W: lb_weight, x, xdt: int, batch: int, y, stream=None) -> None:
    _check(_lib.lb_gemv(ctypes.byref(W), _ptr(x), xdt, batch, _ptr(y), _stream(stream)), "lb_gemv")


def lb_gemv_batched(problems, xdt: int, batch: int, stream=None) -> None:
    """problems: sequence of (lb_weight, x, y) triples (device tensors or addresses)."""
    arr = (lb_gemv_problem * max(1, len(problems)))()
    for i, (W, x, y) in enumerate(problems):
        arr[i] = lb_gemv_problem(W, _ptr(x), _ptr(y))
    _check(_lib.lb_gemv_batched(arr, len(problems), xdt, batch, _stream(stream)), "lb_gemv_batched")


def lb_gemm_workspace_bytes(m: int, n: int, k: int, xdt: int) -> int:
    b = ctypes.c_size_t()
    _check(_lib.lb_gemm_workspace_bytes(m, n, k, xdt, ctypes.byref(b)), "lb_gemm_workspace_bytes")
    return b.value


def lb_gemm(W: lb_weight, x, xdt: int, m: int, y, ydt: int, workspace, workspace_bytes: int,
            stream=None) -> None:
    _check(_lib.lb_gemm(ctypes.byref(W), _ptr(x), xdt, m, _ptr(y), ydt, _ptr(workspace), workspace_bytes,
                        _stream(stream)), "lb_gemm")


def lb_gemm_noalloc(W: lb_weight, x, xdt: int, m: int, y, ydt: int, stream=None) -> None:
    """lb_gemm without a workspace: the library stages activations in its own static scratch."""
    _check(_lib.lb_gemm_noalloc(ctypes.byref(W), _ptr(x), xdt, m, _ptr(y), ydt, _stream(stream)), "lb_gemm_noalloc")


def lb_gemv_swiglu(Wg: lb_weight, Wu: lb_weight, x, xdt: int, batch: int, h, stream=None) -> None:
    """h = silu(Wg x) * (Wu x) in one launch."""
    _check(_lib.lb_gemv_swiglu(ctypes.byref(Wg), ctypes.byref(Wu), _ptr(x), xdt, batch, _ptr(h), _stream(stream)),
           "lb_gemv_swiglu")


def lb_embed(W: lb_weight, ids, count: int, out, out_dtype: int, stream=None) -> None:
    """Embedding rows out[i] = dequantised row ids[i] of W (ids: int32 device tensor)."""
    _check(_lib.lb_embed(ctypes.byref(W), _ptr(ids), count, _ptr(out), out_dtype, _stream(stream)), "lb_embed")


def lb_read_probe(data, nbytes: int, sink, stream=None) -> None:
    """Read nbytes of device memory (the read-bandwidth reference of one launch); sink: uint32."""
    _check(_lib.lb_read_probe(_ptr(data), nbytes, _ptr(sink), _stream(stream)), "lb_read_probe")


def lb_device_error(clear: bool = False) -> int:
    w = ctypes.c_uint32()
    _check(_lib.lb_device_error(ctypes.byref(w), 1 if clear else 0), "lb_device_error")
    return w.value
