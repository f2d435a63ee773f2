"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/uq.h declares, sizes the cache as the pages state,
and rejects bad arguments before touching the device."""
import ctypes as C
import os
import re

import numpy as np
import pytest

import oracle
import ue8m0_kv_cache_gb300 as uq

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "uq.h")


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(uq_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ["uq_quantize_append", "uq_decode_attention", "uq_decode_attention_fp8",
              "uq_decode_attention_bf16", "uq_decode_workspace_bytes", "uq_check_device_status"]:
        assert n in names


def test_library_exports_every_declared_symbol():
    lib = C.CDLL(uq.LIB_PATH)
    missing = [n for n in _declared() if not hasattr(lib, n)]
    assert not missing, missing
    assert sorted(uq.EXPORTED) == _declared()


def test_status_strings():
    for code, name in uq.STATUS_NAMES.items():
        assert uq.uq_status_string(code) == name


def _struct(dtype=uq.FP4_UE8M0, pages=10, hkv=8, ps=16, d=128, ptr=0x100000):
    return uq.UqCacheStruct(dtype, pages, hkv, ps, d, ptr, ptr, ptr, ptr, 1.0, 1.0, 42)


class _FakeCache:
    def __init__(self, s):
        self.struct = s


def test_cache_bytes_follow_the_17_bytes_per_32_layout():
    c = _FakeCache(_struct())
    rows = 10 * 8 * 16
    codes, scales = uq.uq_cache_bytes(c, 0), uq.uq_cache_bytes(c, 1)
    assert codes == rows * 64 and scales == rows * 4
    assert (codes + scales) * 8 / (rows * 128) == 4.25
    assert uq.uq_cache_bytes(_FakeCache(_struct(uq.FP8_E4M3)), 0) == rows * 128
    assert uq.uq_cache_bytes(_FakeCache(_struct(uq.FP8_E4M3)), 1) == 0
    assert uq.uq_cache_bytes(_FakeCache(_struct(uq.BF16)), 2) == rows * 256


def test_rotation_signs_match_oracle():
    for seed in (0, 42, 2 ** 63 + 5):
        assert uq.uq_rotation_signs(seed, 128) == oracle.signs(seed, 128).tolist()


def _append(struct, k=0x200000, v=0x200000, in_dtype=0, T=4, slots=0x300000):
    return uq._lib.uq_quantize_append(k, v, in_dtype, T, None, 0, slots, C.byref(struct), None)


def _decode(struct, q=0x200000, bt=0x300000, sl=0x300000, B=2, hq=8, out=0x400000, ws=0x500000, wsb=1 << 20,
            fn=None):
    fn = fn or uq._lib.uq_decode_attention
    return fn(q, C.byref(struct), bt, 4, sl, B, hq, 0.0, out, ws, wsb, None)


def test_argument_validation_without_a_device():
    E = {v: k for k, v in uq.STATUS_NAMES.items()}
    assert _append(_struct(), T=0) == 0  # no-op
    assert _append(_struct(), k=None) == E["UQ_ERR_INVALID_ARG"]
    assert _append(_struct(), T=-1) == E["UQ_ERR_INVALID_ARG"]
    assert _append(_struct(), in_dtype=7) == E["UQ_ERR_INVALID_ARG"]
    assert _append(_struct(), k=0x200004) == E["UQ_ERR_ALIGNMENT"]
    assert _append(_struct(d=96)) == E["UQ_ERR_UNSUPPORTED"]
    assert _append(_struct(ps=8)) == E["UQ_ERR_UNSUPPORTED"]
    assert _append(_struct(ps=48)) == E["UQ_ERR_UNSUPPORTED"]
    assert _append(_struct(dtype=9)) == E["UQ_ERR_INVALID_ARG"]
    assert _append(_struct(ptr=0)) == E["UQ_ERR_INVALID_ARG"]
    assert _decode(_struct(), B=0) == 0
    assert _decode(_struct(), q=None) == E["UQ_ERR_INVALID_ARG"]
    assert _decode(_struct(), hq=12) == E["UQ_ERR_INVALID_ARG"]  # not a multiple of Hkv
    assert _decode(_struct(), out=0x400008) == E["UQ_ERR_ALIGNMENT"]
    assert _decode(_struct(), B=5000) == E["UQ_ERR_UNSUPPORTED"]
    assert _decode(_struct(), fn=uq._lib.uq_decode_attention_fp8) == E["UQ_ERR_INVALID_ARG"]
    assert _decode(_struct(uq.BF16), fn=uq._lib.uq_decode_attention_fp8) == E["UQ_ERR_INVALID_ARG"]
    s = _struct(uq.FP8_E4M3)
    s.k_scale = 0.0
    assert _decode(s, fn=uq._lib.uq_decode_attention_fp8) == E["UQ_ERR_INVALID_ARG"]
    assert uq._lib.uq_test_cvt_e4m3(0x200000, 3, 0x300000, None) == E["UQ_ERR_INVALID_ARG"]
    assert uq._lib.uq_test_cvt_e2m1(0x200000, 3, 0x300000, None) == E["UQ_ERR_INVALID_ARG"]
    assert uq._lib.uq_test_cvt_e2m1(0, 2, 0x300000, None) == E["UQ_ERR_INVALID_ARG"]
    assert uq._lib.uq_test_scale_byte(0x200000, -1, 0x300000, None) == E["UQ_ERR_INVALID_ARG"]
    assert uq._lib.uq_test_scale_byte(0x200000, 0, 0x300000, None) == E["UQ_OK"]
    assert uq._lib.uq_test_rotate(0x200000, 4, 96, 0, 0, 0x300000, None) == E["UQ_ERR_UNSUPPORTED"]
    assert uq._lib.uq_test_rotate(0x200000, 4, 128, 0, 2, 0x300000, None) == E["UQ_ERR_INVALID_ARG"]
    assert uq._lib.uq_test_rotate(0x200000, 4, 128, 0, -1, 0x300000, None) == E["UQ_ERR_INVALID_ARG"]
    assert uq._lib.uq_test_rotate(0x200000, 0, 128, 0, 1, 0x300000, None) == E["UQ_OK"]


def test_workspace_size_is_positive_and_monotone():
    a = uq.uq_decode_workspace_bytes(8, 64, 8, 128)
    b = uq.uq_decode_workspace_bytes(64, 64, 8, 128)
    assert 0 < a < b
    assert uq.uq_decode_workspace_bytes(8, 12, 8, 128) == 0


def _cascade(struct, q=0x200000, bt=0x300000, sl=0x300000, B=2, hq=8, cu=0x600000, pre=0x600100, ng=1,
             max_prefix=4096, min_rows=0, out=0x400000, ws=0x500000, wsb=1 << 30):
    return uq._lib.uq_cascade_decode_attention(q, C.byref(struct), bt, 4, sl, B, hq, cu, pre, ng, max_prefix,
                                               min_rows, 0.0, out, ws, wsb, None)


def test_cascade_argument_validation_without_a_device():
    E = {v: k for k, v in uq.STATUS_NAMES.items()}
    assert _cascade(_struct(uq.FP8_E4M3)) == E["UQ_ERR_UNSUPPORTED"]
    assert _cascade(_struct(d=256)) == E["UQ_ERR_UNSUPPORTED"]
    assert _cascade(_struct(), ng=-1) == E["UQ_ERR_INVALID_ARG"]
    assert _cascade(_struct(), min_rows=-3) == E["UQ_ERR_INVALID_ARG"]
    assert _cascade(_struct(), max_prefix=-1) == E["UQ_ERR_INVALID_ARG"]
    assert _cascade(_struct(), cu=None) == E["UQ_ERR_INVALID_ARG"]
    assert _cascade(_struct(), pre=None) == E["UQ_ERR_INVALID_ARG"]
    assert _cascade(_struct(), B=0) == 0  # no-op
    assert _cascade(_struct(), q=None) == E["UQ_ERR_INVALID_ARG"]
    assert _cascade(_struct(), out=0x400008) == E["UQ_ERR_ALIGNMENT"]
    assert _cascade(_struct(), wsb=64) == E["UQ_ERR_WORKSPACE"]


def test_cascade_workspace_covers_the_decode_workspace():
    dec = uq.uq_decode_workspace_bytes(4, 64, 8, 128)
    a = uq.uq_cascade_workspace_bytes(4, 1, 64, 8, 128, 98304)
    b = uq.uq_cascade_workspace_bytes(4, 0, 64, 8, 128, 98304)
    assert a > dec and b >= dec
    assert uq.uq_cascade_workspace_bytes(4, 1, 64, 8, 256, 98304) == 0
    assert uq.uq_cascade_workspace_bytes(4, -1, 64, 8, 128, 98304) == 0


def test_calibration_and_constant_argument_validation_without_a_device():
    E = {v: k for k, v in uq.STATUS_NAMES.items()}
    cs = (C.c_float * 2)(0.156, 0.2)
    bad = (C.c_float * 2)(0.156, -1.0)
    f = uq._lib.uq_calibrate_c
    assert f(0x200000, 0, 16, 96, 42, C.cast(cs, C.c_void_p), 2, 0, 0x300000, None) == E["UQ_ERR_UNSUPPORTED"]
    assert f(0x200000, 5, 16, 128, 42, C.cast(cs, C.c_void_p), 2, 0, 0x300000, None) == E["UQ_ERR_INVALID_ARG"]
    assert f(0x200000, 0, 16, 128, 42, C.cast(cs, C.c_void_p), 0, 0, 0x300000, None) == E["UQ_ERR_INVALID_ARG"]
    assert f(0x200000, 0, 16, 128, 42, C.cast(cs, C.c_void_p), 65, 0, 0x300000, None) == E["UQ_ERR_INVALID_ARG"]
    assert f(0x200000, 0, 16, 128, 42, C.cast(cs, C.c_void_p), 2, 1, 0x300000, None) == E["UQ_ERR_INVALID_ARG"]
    assert f(0x200000, 0, 16, 128, 42, C.cast(bad, C.c_void_p), 2, 0, 0x300000, None) == E["UQ_ERR_INVALID_ARG"]
    assert f(0x200004, 0, 16, 128, 42, C.cast(cs, C.c_void_p), 2, 0, 0x300000, None) == E["UQ_ERR_ALIGNMENT"]
    assert f(0x200000, 0, 16, 128, 42, C.cast(cs, C.c_void_p), 2, 0, 0x300004, None) == E["UQ_ERR_ALIGNMENT"]
    s = _struct()
    s.fp4_c = -0.5
    assert _append(s) == E["UQ_ERR_INVALID_ARG"]
    s.fp4_c = float("nan")
    assert _decode(s) == E["UQ_ERR_INVALID_ARG"]


def test_timeout_hook_rejects_negative_arguments_on_the_host():
    # only invalid arguments here: a valid call would arm the next decode launch of this process
    for cta, budget in ((-1, 1000), (0, -1)):
        with pytest.raises(uq.UqError):
            uq.uq_test_arm_decode_timeout(cta, budget)
