"""The C-ABI library loads without a GPU, exports every entry point that
include/qmv.h declares, and rejects bad arguments before touching CUDA."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qmv.h")


@pytest.fixture(scope="module")
def lib():
    from gemm_decode_prefill_gb300 import build
    build.build()
    from gemm_decode_prefill_gb300 import qmv
    return qmv


def _declared():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^QMV_API\s+[^;(]*?\b(\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_hot_path():
    names = _declared()
    for n in ["qmv_q8row", "qmv_q2g64", "qmv_q2g128", "qmm_q8row", "moe_select_topk",
              "moe_ffn_q8row", "qmv_pack_q8row", "qmv_pack_q2"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    raw = ctypes.CDLL(lib.LIB_PATH)
    for name in _declared():
        assert hasattr(raw, name), name
    assert set(_declared()) == set(lib.EXPORTS)


def test_status_strings(lib):
    assert lib.status_string(0) == "QMV_OK"
    assert lib.status_string(1) == "QMV_ERR_INVALID_ARG"
    assert lib.status_string(5) == "QMV_ERR_DEVICE_STATUS"
    assert lib.status_string(99) == "QMV_ERR_UNKNOWN"
    assert lib.version() >= 100


def test_null_arguments_are_rejected_without_cuda(lib):
    L = lib._lib
    h = ctypes.c_void_p()
    assert L.qmv_q8row(None, None, None, None) == 1
    assert L.qmv_q2g64(None, None, None, None) == 1
    assert L.qmv_q2g128(None, None, None, None) == 1
    assert L.qmm_q8row(None, None, 4, None, None) == 1
    assert L.qmv_pack_q8row(None, None, 1, 4, 16, None, ctypes.byref(h)) == 1
    assert L.qmv_pack_q2(None, None, 64, 4, 64, None, ctypes.byref(h)) == 1
    assert L.moe_select_topk(None, 8, 2, 1, None, None, 0, None, None, None, None) == 1
    assert L.moe_ffn_q8row(None, None, None, None, None, 9, None, None, None) == 1
    buf = ctypes.create_string_buffer(256)
    assert L.qmv_last_error(buf, 256) == 1
    assert b"null" in buf.value


def test_shape_rules_are_checked_before_cuda(lib):
    L = lib._lib
    h = ctypes.c_void_p()
    fake = ctypes.c_void_p(4096)  # never dereferenced: validation fails first
    assert L.qmv_pack_q8row(fake, fake, 1, 4, 24, None, ctypes.byref(h)) == 1   # cols % 16
    assert L.qmv_pack_q8row(fake, fake, 0, 4, 32, None, ctypes.byref(h)) == 1   # experts
    assert L.qmv_pack_q2(fake, fake, 32, 4, 64, None, ctypes.byref(h)) == 1     # group
    assert L.qmv_pack_q2(fake, fake, 64, 4, 96, None, ctypes.byref(h)) == 1     # cols % group
    assert L.qmv_pack_q2(fake, fake, 128, 4, 65536, None, ctypes.byref(h)) == 2  # too wide
    assert L.moe_select_topk(fake, 2000, 2, 1, None, None, 0, None, fake, fake, None) == 1
    assert L.moe_select_topk(fake, 8, 9, 1, None, None, 0, None, fake, fake, None) == 1
    assert L.moe_select_topk(fake, 8, 0, 1, None, None, 0, None, fake, fake, None) == 1
    assert h.value is None
