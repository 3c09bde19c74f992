"""The C ABI library loads and exports every symbol include/lb.h declares; host-side argument
validation returns the documented status before touching the GPU (runs without a GPU)."""

import ctypes
import os
import re

import pytest

from gemm_lb_gemv_02_b300 import lb

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "lb.h")


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(lb_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_expected_entry_points():
    names = declared_functions()
    assert set(names) == set(lb.EXPORTED), names


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(lb.LIB_PATH)
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings():
    for code, name in lb.STATUS_NAMES.items():
        assert lb.lb_status_string(code).startswith(name)


def test_packed_bytes():
    assert lb.lb_packed_bytes(lb.LB_FMT_1BIT_G128, 2048, 2048) == (2048 * 2048 // 8, 2048 * 16 * 2)
    assert lb.lb_packed_bytes(lb.LB_FMT_TERNARY_G128, 17408, 5120) == (17408 * 5120 // 4, 17408 * 40 * 2)
    for bad in ((lb.LB_FMT_1BIT_G128, 0, 128), (lb.LB_FMT_1BIT_G128, 4, 100), (lb.LB_FMT_1BIT_G128, 4, 0)):
        with pytest.raises(lb.LBError) as e:
            lb.lb_packed_bytes(*bad)
        assert e.value.name == "LB_ERR_SHAPE"
    with pytest.raises(lb.LBError) as e:
        lb.lb_packed_bytes(7, 4, 128)
    assert e.value.name == "LB_ERR_DTYPE"


def _status(fn, *args):
    try:
        fn(*args)
    except lb.LBError as e:
        return e.name
    return "LB_OK"


# The largest k lb_gemv takes per batch class (batch 1, 2, 3-4, 5-8), as include/lb.h states them.
GEMV_K_LIMITS = {lb.LB_FMT_1BIT_G128: ((1, 327680), (2, 180224), (4, 90112), (8, 49152)),
                 lb.LB_FMT_TERNARY_G128: ((1, 344064), (2, 188416), (4, 98304), (8, 49152))}

# Fake, never-dereferenced device addresses: validation must reject before any CUDA call.
A16 = 0x10000
MIS = 0x10001


def test_pack_validation():
    assert _status(lb.lb_pack_1bit, None, 4, 128, A16, A16, 0) == "LB_ERR_NULL"
    assert _status(lb.lb_pack_1bit, A16, 4, 100, A16, A16, 0) == "LB_ERR_SHAPE"
    assert _status(lb.lb_pack_1bit, A16, 0, 128, A16, A16, 0) == "LB_ERR_SHAPE"
    assert _status(lb.lb_pack_1bit, MIS, 4, 128, A16, A16, 0) == "LB_ERR_ALIGN"
    assert _status(lb.lb_pack_ternary, A16, None, 4, 128, A16, A16, 0) == "LB_ERR_NULL"
    assert _status(lb.lb_pack_ternary, A16, A16, 4, 129, A16, A16, 0) == "LB_ERR_SHAPE"
    assert _status(lb.lb_pack_ternary, A16, A16, 4, 128, MIS, A16, 0) == "LB_ERR_ALIGN"


def test_gemv_validation():
    W = lb.make_weight(lb.LB_FMT_1BIT_G128, 16, 128, A16, A16)
    assert _status(lb.lb_gemv, W, None, lb.LB_F16, 1, A16, 0) == "LB_ERR_NULL"
    assert _status(lb.lb_gemv, W, A16, 9, 1, A16, 0) == "LB_ERR_DTYPE"
    assert _status(lb.lb_gemv, W, A16, lb.LB_F16, 0, A16, 0) == "LB_ERR_SHAPE"
    assert _status(lb.lb_gemv, W, A16, lb.LB_F16, 9, A16, 0) == "LB_ERR_SHAPE"
    assert _status(lb.lb_gemv, W, MIS, lb.LB_F16, 1, A16, 0) == "LB_ERR_ALIGN"
    assert _status(lb.lb_gemv, lb.make_weight(4, 16, 128, A16, A16), A16, lb.LB_F16, 1, A16, 0) == "LB_ERR_DTYPE"
    assert _status(lb.lb_gemv, lb.make_weight(1, 16, 130, A16, A16), A16, lb.LB_F16, 1, A16, 0) == "LB_ERR_SHAPE"
    assert _status(lb.lb_gemv, lb.make_weight(1, 16, 128, MIS, A16), A16, lb.LB_F16, 1, A16, 0) == "LB_ERR_ALIGN"
    assert _status(lb.lb_gemv, lb.make_weight(1, 16, 128, None, A16), A16, lb.LB_F16, 1, A16, 0) == "LB_ERR_NULL"


def test_gemm_validation():
    W = lb.make_weight(lb.LB_FMT_TERNARY_G128, 256, 256, A16, A16)
    need = lb.lb_gemm_workspace_bytes(5, 256, 256, lb.LB_BF16)
    assert need == 128 * (256 * 2 + 4)                   # binary16 tiles + one FP32 factor per padded row
    assert _status(lb.lb_gemm, W, A16, lb.LB_BF16, 5, A16, lb.LB_BF16, None, 0, 0) == "LB_ERR_WORKSPACE"
    assert _status(lb.lb_gemm, W, A16, lb.LB_BF16, 5, A16, lb.LB_BF16, A16, need - 1, 0) == "LB_ERR_WORKSPACE"
    assert _status(lb.lb_gemm, W, A16, lb.LB_BF16, 5, A16, lb.LB_BF16, A16 + 16, need, 0) == "LB_ERR_ALIGN"
    assert _status(lb.lb_gemm, W, A16, lb.LB_BF16, 0, A16, lb.LB_BF16, A16, need, 0) == "LB_ERR_SHAPE"
    assert _status(lb.lb_gemm, lb.make_weight(2, 250, 256, A16, A16), A16, lb.LB_BF16, 5, A16, lb.LB_BF16,
                   A16, need, 0) == "LB_ERR_SHAPE"
    assert _status(lb.lb_gemm, lb.make_weight(1, 250, 256, A16, A16), A16, lb.LB_BF16, 5, A16, lb.LB_BF16,
                   A16, need, 0) == "LB_ERR_SHAPE"
    assert _status(lb.lb_gemm, W, A16, 5, 5, A16, lb.LB_BF16, A16, need, 0) == "LB_ERR_DTYPE"
    # launch-shape limit: 65535 token tiles of 256; beyond it only the workspace bounds a call
    W128 = lb.make_weight(lb.LB_FMT_TERNARY_G128, 256, 128, A16, A16)
    assert _status(lb.lb_gemm, W128, A16, lb.LB_BF16, 65535 * 256 + 1, A16, lb.LB_BF16, A16, need, 0) == "LB_ERR_SHAPE"
    assert _status(lb.lb_gemm, W128, A16, lb.LB_BF16, 65535 * 256, A16, lb.LB_BF16, A16, need, 0) == "LB_ERR_WORKSPACE"
    Wk = lb.make_weight(lb.LB_FMT_TERNARY_G128, 256, 1 << 24, A16, A16)
    assert _status(lb.lb_gemm, Wk, A16, lb.LB_BF16, 1 << 20, A16, lb.LB_BF16, A16, need, 0) == "LB_ERR_WORKSPACE"


def test_ternary5_entry_points():
    """The five-per-byte format: sizes, packer validation, and the calls that do not take it."""
    assert lb.lb_packed_bytes(lb.LB_FMT_TERNARY5_G128, 3, 1024) == (3 * 8 * 26, 3 * 8 * 2)
    assert _status(lb.lb_pack_ternary5, A16, A16, 4, 100, A16, A16) == "LB_ERR_SHAPE"
    assert _status(lb.lb_pack_ternary5, None, A16, 4, 128, A16, A16) == "LB_ERR_NULL"
    assert _status(lb.lb_pack_ternary5, A16, A16, 4, 128, MIS, A16) == "LB_ERR_ALIGN"
    W5 = lb.make_weight(lb.LB_FMT_TERNARY5_G128, 256, 256, A16, A16)
    need = lb.lb_gemm_workspace_bytes(5, 256, 256, lb.LB_BF16)
    assert _status(lb.lb_gemm, W5, A16, lb.LB_BF16, 5, A16, lb.LB_BF16, A16, need, 0) == "LB_ERR_UNSUPPORTED"
    assert _status(lb.lb_gemm_noalloc, W5, A16, lb.LB_BF16, 5, A16, lb.LB_BF16) == "LB_ERR_UNSUPPORTED"
    assert _status(lb.lb_embed, W5, A16, 3, A16, lb.LB_BF16, 0) == "LB_ERR_UNSUPPORTED"
    # the grouped GEMV takes the format, but not mixed with another one in one call
    W2 = lb.make_weight(lb.LB_FMT_TERNARY_G128, 256, 256, A16, A16)
    assert _status(lb.lb_gemv_batched, [(W5, A16, A16), (W2, A16, A16)], lb.LB_F16, 1) == "LB_ERR_UNSUPPORTED"
    assert _status(lb.lb_gemv_swiglu, W5, W5, A16, lb.LB_F16, 1, A16, 0) == "LB_ERR_UNSUPPORTED"
    assert _status(lb.lb_gemv, W5, A16, lb.LB_F16, 9, A16, 0) == "LB_ERR_SHAPE"


def test_embed_validation():
    W = lb.make_weight(lb.LB_FMT_1BIT_G128, 64, 256, A16, A16)
    assert _status(lb.lb_embed, W, A16, 0, None, lb.LB_BF16, 0) == "LB_OK"            # nothing to do
    assert _status(lb.lb_embed, W, A16, -1, A16, lb.LB_BF16, 0) == "LB_ERR_SHAPE"
    assert _status(lb.lb_embed, W, A16, 2 ** 31, A16, lb.LB_BF16, 0) == "LB_ERR_SHAPE"
    wide = lb.make_weight(lb.LB_FMT_1BIT_G128, 64, 1 << 24, A16, A16)                # 16384 pieces per row
    assert _status(lb.lb_embed, wide, A16, 2 ** 20 + 1, A16, lb.LB_BF16, 0) == "LB_ERR_SHAPE"
    assert _status(lb.lb_embed, W, None, 3, A16, lb.LB_BF16, 0) == "LB_ERR_NULL"
    assert _status(lb.lb_embed, W, A16, 3, None, lb.LB_BF16, 0) == "LB_ERR_NULL"
    assert _status(lb.lb_embed, W, A16, 3, A16, 7, 0) == "LB_ERR_DTYPE"
    assert _status(lb.lb_embed, W, A16 + 2, 3, A16, lb.LB_F16, 0) == "LB_ERR_ALIGN"     # ids: 4-byte
    assert _status(lb.lb_embed, W, A16, 3, A16 + 8, lb.LB_F16, 0) == "LB_ERR_ALIGN"     # out: 16-byte
    assert _status(lb.lb_embed, lb.make_weight(4, 64, 256, A16, A16), A16, 3, A16, lb.LB_F16, 0) == "LB_ERR_DTYPE"
    assert _status(lb.lb_embed, lb.make_weight(2, 64, 200, A16, A16), A16, 3, A16, lb.LB_F16, 0) == "LB_ERR_SHAPE"


def test_gemv_swiglu_validation():
    Wg = lb.make_weight(lb.LB_FMT_TERNARY_G128, 64, 256, A16, A16)
    Wu = lb.make_weight(lb.LB_FMT_TERNARY_G128, 64, 256, A16, A16)
    assert _status(lb.lb_gemv_swiglu, Wg, Wu, None, lb.LB_F16, 1, A16, 0) == "LB_ERR_NULL"
    assert _status(lb.lb_gemv_swiglu, Wg, Wu, A16, lb.LB_F16, 1, None, 0) == "LB_ERR_NULL"
    assert _status(lb.lb_gemv_swiglu, Wg, Wu, A16, 9, 1, A16, 0) == "LB_ERR_DTYPE"
    assert _status(lb.lb_gemv_swiglu, Wg, Wu, A16, lb.LB_F16, 0, A16, 0) == "LB_ERR_SHAPE"
    assert _status(lb.lb_gemv_swiglu, Wg, Wu, A16, lb.LB_F16, 9, A16, 0) == "LB_ERR_SHAPE"
    assert _status(lb.lb_gemv_swiglu, Wg, Wu, MIS, lb.LB_F16, 1, A16, 0) == "LB_ERR_ALIGN"
    assert _status(lb.lb_gemv_swiglu, Wg, Wu, A16, lb.LB_F16, 1, MIS, 0) == "LB_ERR_ALIGN"
    assert _status(lb.lb_gemv_swiglu, Wg, lb.make_weight(2, 48, 256, A16, A16), A16, lb.LB_F16, 1, A16, 0) == "LB_ERR_SHAPE"
    assert _status(lb.lb_gemv_swiglu, Wg, lb.make_weight(2, 64, 384, A16, A16), A16, lb.LB_F16, 1, A16, 0) == "LB_ERR_SHAPE"
    assert _status(lb.lb_gemv_swiglu, Wg, lb.make_weight(1, 64, 256, A16, A16), A16, lb.LB_F16, 1, A16, 0) == "LB_ERR_UNSUPPORTED"
    assert _status(lb.lb_gemv_swiglu, Wg, lb.make_weight(2, 64, 256, None, A16), A16, lb.LB_F16, 1, A16, 0) == "LB_ERR_NULL"


def test_grouped_launch_row_block_limit():
    """More than 65535 blocks of 128 rows cannot be one grouped launch: a clean error, no launch."""
    big = lb.make_weight(lb.LB_FMT_1BIT_G128, 65536 * 128, 128, A16, A16)
    assert _status(lb.lb_gemv_batched, [(big, A16, A16)], lb.LB_F16, 1) == "LB_ERR_SHAPE"
    assert _status(lb.lb_gemv_swiglu, big, big, A16, lb.LB_F16, 1, A16, 0) == "LB_ERR_SHAPE"


def test_gemv_batched_validation():
    W1 = lb.make_weight(lb.LB_FMT_1BIT_G128, 16, 128, A16, A16)
    Wt = lb.make_weight(lb.LB_FMT_TERNARY_G128, 16, 128, A16, A16)
    ok = (W1, A16, A16)
    raw = lb.library().lb_gemv_batched
    assert lb.lb_status_string(raw(None, 1, lb.LB_F16, 1, None)).startswith("LB_ERR_NULL")
    assert _status(lb.lb_gemv_batched, [], lb.LB_F16, 1) == "LB_ERR_SHAPE"
    assert _status(lb.lb_gemv_batched, [ok] * (lb.LB_GEMV_BATCH_MAX + 1), lb.LB_F16, 1) == "LB_ERR_SHAPE"
    assert _status(lb.lb_gemv_batched, [ok], 9, 1) == "LB_ERR_DTYPE"
    assert _status(lb.lb_gemv_batched, [ok], lb.LB_F16, 9) == "LB_ERR_SHAPE"
    assert _status(lb.lb_gemv_batched, [ok, (Wt, A16, A16)], lb.LB_F16, 1) == "LB_ERR_UNSUPPORTED"
    assert _status(lb.lb_gemv_batched, [ok, (W1, None, A16)], lb.LB_F16, 1) == "LB_ERR_NULL"
    assert _status(lb.lb_gemv_batched, [ok, (W1, A16, MIS)], lb.LB_F16, 1) == "LB_ERR_ALIGN"
    assert _status(lb.lb_gemv_batched, [ok, (lb.make_weight(1, 16, 130, A16, A16), A16, A16)], lb.LB_F16, 1) == "LB_ERR_SHAPE"
    # the documented k limits (an 8-CTA split), for the grouped and the single call
    for fmt, limits in GEMV_K_LIMITS.items():
        for batch, kmax in limits:
            long_w = lb.make_weight(fmt, 16, kmax + 128, A16, A16)
            assert _status(lb.lb_gemv_batched, [(long_w, A16, A16)], lb.LB_F16, batch) == "LB_ERR_UNSUPPORTED"
            assert _status(lb.lb_gemv, long_w, A16, lb.LB_F16, batch, A16, 0) == "LB_ERR_UNSUPPORTED"
