"""Host-side checks of the C ABI: the library loads, exports what include/mxq.h declares, and
rejects bad arguments before any launch. No call here reaches a kernel: every call either fails
validation or is an empty call (M == 0 or K == 0), so fake pointers are never dereferenced."""

import ctypes
import os
import re
import subprocess

import pytest

import mx_microscaling_quantize_gb300 as mxq
from mx_microscaling_quantize_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mxq.h")

OK, NULL, SHAPE, ALIGN, UNSUP = 0, 1, 2, 3, 4
P = 1 << 20  # a 16-byte aligned fake device address, never dereferenced


@pytest.fixture(scope="module")
def L():
    _build.build()
    return mxq.lib()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^(?:mx_status|const char\*)\s+(mx_\w+)\(", text, re.M)))


def test_header_declares_the_binding_exports():
    assert declared_functions() == sorted(mxq.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    out = subprocess.run(["nm", "-D", "--defined-only", mxq.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in declared_functions():
        assert name in exported, name
        assert getattr(L, name) is not None


def test_macros_match_binding():
    text = open(HEADER).read()
    macros = dict(re.findall(r"#define (MX_\w+) (\d+)", text))
    assert int(macros["MX_FMT_E2M1"]) == mxq.E2M1 and int(macros["MX_FMT_E4M3"]) == mxq.E4M3
    assert int(macros["MX_SCALES_LINEAR"]) == mxq.LINEAR
    assert int(macros["MX_SCALES_SWIZZLED"]) == mxq.SWIZZLED
    assert int(macros["MX_ROUND_RNE"]) == mxq.RNE
    assert int(macros["MX_ROUND_QUEST"]) == mxq.QUEST
    assert int(macros["MX_ROT_DENSE"]) == mxq.ROT_DENSE
    assert int(macros["MX_ROT_HADAMARD"]) == mxq.ROT_HADAMARD
    assert int(macros["MX_ROT_AUTO"]) == mxq.ROT_AUTO


def test_status_strings(L):
    for s in range(6):
        assert mxq.mx_status_string(s).startswith("MX_")
    assert "unknown" in mxq.mx_status_string(99)


@pytest.mark.parametrize("M,K,layout,want", [
    (1, 32, 0, (1, 1)), (1, 32, 1, (128, 4)), (128, 4096, 0, (128, 128)),
    (129, 96, 1, (256, 4)), (300, 416, 1, (384, 16)), (0, 64, 1, (0, 4)),
    (8192, 28672, 1, (8192, 896)),
])
def test_scales_shape(L, M, K, layout, want):
    assert mxq.mx_scales_shape(M, K, layout) == want


def test_grouped_scales_shape(L):
    assert mxq.mx_grouped_scales_shape(16384, 128, 2048, mxq.SWIZZLED) == (32640, 64)
    assert mxq.mx_grouped_scales_shape(16384, 128, 2048, mxq.LINEAR) == (16384, 64)
    # the bound holds for every split of the rows: n_e = 1 for 127 experts, rest in one
    counts = [1] * 127 + [16384 - 127]
    need = sum(-(-c // 128) * 128 for c in counts)
    assert need <= mxq.mx_grouped_scales_shape(16384, 128, 2048, mxq.SWIZZLED)[0]


def shape_status(L, M, K, group=32, layout=0):
    r, c = ctypes.c_int64(), ctypes.c_int64()
    return L.mx_scales_shape(M, K, group, layout, ctypes.byref(r), ctypes.byref(c))


def test_scales_shape_errors(L):
    assert shape_status(L, -1, 32) == SHAPE
    assert shape_status(L, 4, 48) == SHAPE
    assert shape_status(L, 4, 64, group=16) == UNSUP
    assert shape_status(L, 4, 64, layout=7) == UNSUP
    assert L.mx_scales_shape(4, 64, 32, 0, None, None) == NULL


def test_quantize_validation(L):
    q = L.mx_quantize
    assert q(P, -1, 64, 1, 32, 0, 0, P, P, None) == SHAPE
    assert q(P, 4, 48, 1, 32, 0, 0, P, P, None) == SHAPE
    assert q(P, 4, 64, 3, 32, 0, 0, P, P, None) == UNSUP
    assert q(P, 4, 64, 1, 16, 0, 0, P, P, None) == UNSUP
    assert q(P, 4, 64, 1, 32, 2, 0, P, P, None) == UNSUP
    assert q(P, 4, 64, 1, 32, 0, 2, P, P, None) == UNSUP  # unknown rounding
    assert q(P, 4, 64, 2, 32, 0, 1, P, P, None) == UNSUP  # Quest-like scale: MXFP4 only
    assert q(P, 4, 48, 1, 32, 0, 1, P, P, None) == SHAPE  # the other checks still apply
    assert q(None, 4, 64, 1, 32, 0, 1, P, P, None) == NULL
    assert q(None, 4, 64, 1, 32, 0, 0, P, P, None) == NULL
    assert q(P, 4, 64, 1, 32, 0, 0, None, P, None) == NULL
    assert q(P, 4, 64, 1, 32, 0, 0, P, None, None) == NULL
    assert q(P + 8, 4, 64, 1, 32, 0, 0, P, P, None) == ALIGN
    assert q(P + 16, 4, 64, 1, 32, 0, 0, P, P, None) == ALIGN
    assert q(P, 4, 64, 2, 32, 0, 0, P + 16, P, None) == ALIGN
    assert q(P, 4, 64, 1, 32, 0, 0, P + 4, P, None) == ALIGN
    assert q(P, 4, 64, 1, 32, 1, 0, P, P + 1, None) == ALIGN
    # empty calls launch nothing and succeed, even with NULL buffers
    assert q(None, 0, 64, 1, 32, 0, 0, None, None, None) == OK
    assert q(None, 5, 0, 2, 32, 1, 0, None, None, None) == OK
    # absurd sizes are rejected, not overflowed
    assert q(P, 1 << 40, 1 << 20, 1, 32, 0, 0, P, P, None) == SHAPE


def test_qdq_and_rotation_validation(L):
    q = L.mx_qdq  # (x, M, K, fmt, group, rounding, H, g, rot_kind, y, stream)
    for rk in (0, 1, 2):  # MX_ROT_DENSE, MX_ROT_HADAMARD, MX_ROT_AUTO
        assert q(P, 4, 64, 1, 32, 0, P, 8, rk, P, None) == UNSUP     # g = 8
        assert q(P, 4, 96, 1, 32, 0, P, 64, rk, P, None) == SHAPE    # K % g
        assert q(P, 4, 64, 1, 32, 0, P + 1, 32, rk, P, None) == ALIGN
        assert q(P, 4, 64, 1, 32, 0, P + 8, 32, rk, P, None) == ALIGN
    assert q(P, 4, 64, 1, 32, 0, P, 32, 3, P, None) == UNSUP         # unknown rot_kind
    assert q(P, 4, 64, 2, 32, 1, P, 32, 0, P, None) == UNSUP         # Quest-like: MXFP4 only
    assert q(P, 4, 64, 2, 32, 1, None, 0, 0, P, None) == UNSUP
    assert q(P, 4, 64, 1, 32, 3, None, 0, 0, P, None) == UNSUP       # unknown rounding
    assert q(P, 4, 64, 1, 32, 0, None, 0, 7, None, None) == NULL     # no H: rot_kind ignored
    assert q(P, 4, 64, 1, 32, 0, None, 0, 0, P + 2, None) == ALIGN
    assert q(P, 4, 64, 1, 32, 0, None, 0, 0, P + 16, None) == ALIGN
    r = L.mx_rotate_quantize  # (x, M, K, H, g, rot_kind, fmt, group, layout, rnd, codes, scales, s)
    for rk in (0, 1, 2):
        assert r(P, 4, 64, P, 48, rk, 1, 32, 1, 0, P, P, None) == UNSUP
        assert r(P, 4, 192, P, 128, rk, 1, 32, 1, 0, P, P, None) == SHAPE
        assert r(P, 4, 64, None, 32, rk, 1, 32, 1, 0, P, P, None) == NULL
        assert r(P, 4, 64, P, 32, rk, 1, 32, 1, 0, P, P + 8, None) == ALIGN
        assert r(None, 0, 64, None, 32, rk, 1, 32, 1, 0, None, None, None) == OK
    assert r(P, 4, 64, P, 32, -1, 1, 32, 1, 0, P, P, None) == UNSUP
    assert r(P, 4, 64, P, 32, 3, 1, 32, 1, 0, P, P, None) == UNSUP
    assert r(P, 4, 64, P, 32, 0, 2, 32, 1, 1, P, P, None) == UNSUP  # Quest-like: MXFP4 only
    assert r(P, 4, 64, P, 32, 0, 1, 32, 1, 1, P, P + 8, None) == ALIGN
    d = L.mx_rotate_debug  # (x, M, K, H, g, rot_kind, y, stream)
    assert d(P, 4, 64, P, 24, 0, P, None) == UNSUP
    assert d(P, 4, 64, P, 32, 3, P, None) == UNSUP
    assert d(P, 4, 64, None, 32, 1, P, None) == NULL
    assert d(P, 4, 64, P, 32, 1, P + 16, None) == ALIGN


def test_grouped_validation(L):
    g = L.mx_quantize_grouped
    assert g(P, P, 0, 16, 64, 1, 32, 1, 0, P, P, None) == SHAPE       # E = 0
    assert g(P, P, 1025, 16, 64, 1, 32, 1, 0, P, P, None) == SHAPE    # E > 1024
    assert g(P, None, 4, 16, 64, 1, 32, 1, 0, P, P, None) == NULL
    assert g(P, P + 4, 4, 16, 64, 1, 32, 1, 0, P, P, None) == ALIGN
    assert g(P, P, 4, 16, 64, 1, 32, 1, 0, P, P + 8, None) == ALIGN
    assert g(P, P, 4, 16, 48, 1, 32, 1, 0, P, P, None) == SHAPE
    assert g(None, None, 4, 0, 64, 1, 32, 1, 0, None, None, None) == OK
    assert g(P, P, 4, 16, 64, 1, 32, 1, 1, P, P, None) == UNSUP  # no grouped Quest-like scale


def test_dequantize_validation(L):
    d = L.mx_dequantize  # (codes, scales, M, K, fmt, group, layout, y, stream)
    assert d(P, P, -1, 64, 1, 32, 0, P, None) == SHAPE
    assert d(P, P, 4, 48, 1, 32, 0, P, None) == SHAPE
    assert d(P, P, 4, 64, 3, 32, 0, P, None) == UNSUP
    assert d(P, P, 4, 64, 1, 16, 0, P, None) == UNSUP
    assert d(P, P, 4, 64, 1, 32, 2, P, None) == UNSUP
    assert d(None, P, 4, 64, 1, 32, 0, P, None) == NULL
    assert d(P, None, 4, 64, 1, 32, 0, P, None) == NULL
    assert d(P, P, 4, 64, 1, 32, 0, None, None) == NULL
    assert d(P + 16, P, 4, 64, 2, 32, 0, P, None) == ALIGN
    assert d(P, P, 4, 64, 2, 32, 0, P + 16, None) == ALIGN
    assert d(P, P + 8, 4, 64, 2, 32, 1, P, None) == ALIGN
    assert d(None, None, 0, 64, 1, 32, 1, None, None) == OK
    assert d(P, P, 1 << 40, 1 << 20, 1, 32, 0, P, None) == SHAPE


def test_nvfp4_shapes_and_validation(L):
    assert mxq.mx_nvfp4_scales_shape(1, 32, mxq.SWIZZLED) == (128, 4)
    assert mxq.mx_nvfp4_scales_shape(300, 416, mxq.SWIZZLED) == (384, 28)
    assert mxq.mx_nvfp4_scales_shape(300, 416, mxq.LINEAR) == (300, 26)
    q = L.mx_quantize_nvfp4  # (x, M, K, H, g, rot_kind, gs, layout, codes, scales, stream)
    assert q(P, 4, 48, None, 0, 0, P, 0, P, P, None) == SHAPE
    assert q(P, 4, 64, None, 0, 0, P, 2, P, P, None) == UNSUP
    assert q(P, 4, 64, P, 8, 0, P, 0, P, P, None) == UNSUP
    assert q(P, 4, 64, P, 32, 3, P, 0, P, P, None) == UNSUP          # unknown rot_kind
    assert q(P, 4, 96, P, 64, 1, P, 0, P, P, None) == SHAPE
    assert q(P, 4, 64, None, 0, 0, None, 0, P, P, None) == NULL
    assert q(None, 4, 64, None, 0, 0, P, 0, P, P, None) == NULL
    assert q(P, 4, 64, None, 0, 0, P, 0, None, P, None) == NULL
    assert q(P, 4, 64, None, 0, 0, P + 2, 0, P, P, None) == ALIGN
    assert q(P, 4, 64, None, 0, 0, P, 0, P + 16, P, None) == ALIGN
    assert q(P, 4, 64, None, 0, 0, P, 0, P, P + 1, None) == ALIGN
    assert q(P, 4, 64, None, 0, 0, P, 1, P, P + 2, None) == ALIGN
    for rk in (0, 1, 2):
        assert q(P, 4, 64, P + 8, 32, rk, P, 1, P, P, None) == ALIGN
    assert q(None, 0, 64, None, 0, 0, None, 1, None, None, None) == OK
    d = L.mx_qdq_nvfp4  # (x, M, K, H, g, rot_kind, gs, y, stream)
    assert d(P, 4, 64, None, 0, 0, P, None, None) == NULL
    assert d(P, 4, 64, None, 0, 0, P, P + 16, None) == ALIGN
    assert d(P, -1, 64, None, 0, 0, P, P, None) == SHAPE
    assert d(P, 4, 64, P, 32, 5, P, P, None) == UNSUP
    assert mxq.mx_nvfp4_grouped_scales_shape(300, 4, 416, mxq.SWIZZLED) == (768, 28)
    assert mxq.mx_nvfp4_grouped_scales_shape(300, 4, 416, mxq.LINEAR) == (300, 26)
    gq = L.mx_quantize_nvfp4_grouped  # (x, off, E, M, K, gs, layout, codes, scales, stream)
    assert gq(P, P, 0, 4, 64, P, 0, P, P, None) == SHAPE
    assert gq(P, P, 1025, 4, 64, P, 0, P, P, None) == SHAPE
    assert gq(P, P, 2, 4, 48, P, 0, P, P, None) == SHAPE
    assert gq(P, P, 2, 4, 64, P, 2, P, P, None) == UNSUP
    assert gq(P, P, 2, 4, 64, None, 0, P, P, None) == NULL
    assert gq(P, None, 2, 4, 64, P, 0, P, P, None) == NULL
    assert gq(P, P + 4, 2, 4, 64, P, 0, P, P, None) == ALIGN
    assert gq(P, P, 2, 4, 64, P + 2, 0, P, P, None) == ALIGN
    assert gq(P, P, 2, 4, 64, P, 0, P, P + 1, None) == ALIGN
    assert gq(P, P, 2, 4, 64, P, 1, P, P + 2, None) == ALIGN
    assert gq(None, None, 2, 0, 64, None, 1, None, None, None) == OK
    u = L.mx_dequantize_nvfp4  # (codes, scales, M, K, gs, layout, y, stream)
    assert u(P, P, 4, 48, P, 0, P, None) == SHAPE
    assert u(P, P, -1, 64, P, 0, P, None) == SHAPE
    assert u(P, P, 4, 64, P, 2, P, None) == UNSUP
    assert u(None, P, 4, 64, P, 0, P, None) == NULL
    assert u(P, None, 4, 64, P, 0, P, None) == NULL
    assert u(P, P, 4, 64, None, 0, P, None) == NULL
    assert u(P, P, 4, 64, P, 0, None, None) == NULL
    assert u(P + 16, P, 4, 64, P, 0, P, None) == ALIGN
    assert u(P, P, 4, 64, P, 0, P + 16, None) == ALIGN
    assert u(P, P + 1, 4, 64, P, 0, P, None) == ALIGN
    assert u(P, P + 2, 4, 64, P, 1, P, None) == ALIGN
    assert u(P, P, 4, 64, P + 2, 0, P, None) == ALIGN
    assert u(None, None, 0, 64, None, 1, None, None) == OK
    assert u(P, P, 1 << 40, 1 << 20, P, 0, P, None) == SHAPE


def test_device_errors_null(L):
    assert L.mx_device_errors(None) == NULL


def test_selftest_bounded_wait_validation(L):
    assert L.mx_selftest_bounded_wait(0, None) == SHAPE
    assert L.mx_selftest_bounded_wait(-5, None) == SHAPE
    assert L.mx_selftest_bounded_wait(100_000_001, None) == SHAPE


def test_selftest_rotate_give_up_validation(L):
    f = L.mx_selftest_rotate_give_up
    assert f(P, 128, 256, P, 32, P, P, 0, None) == SHAPE            # limit out of range
    assert f(P, 128, 256, P, 32, P, P, 100_000_001, None) == SHAPE
    assert f(P, 16, 256, P, 32, P, P, 1000, None) == SHAPE          # the few-row kernel's call
    assert f(P, 0, 256, P, 32, P, P, 1000, None) == SHAPE           # empty
    assert f(P, 128, 96, P, 64, P, P, 1000, None) == SHAPE          # K % g
    assert f(P, 128, 256, P, 48, P, P, 1000, None) == UNSUP         # g
    assert f(None, 128, 256, P, 32, P, P, 1000, None) == NULL
    assert f(P + 16, 128, 256, P, 32, P, P, 1000, None) == ALIGN    # x 32-byte aligned


def test_gemm_validation(L):
    f = L.mx_gemm  # (a_codes, a_scales, b_codes, b_scales, M, N, K, fmt, group, layout, alpha, c, stream)
    assert f(P, P, P, P, 128, 128, 96, 1, 32, 1, 1.0, P, None) == SHAPE     # K % 64
    assert f(P, P, P, P, 128, 128, 0, 1, 32, 1, 1.0, P, None) == SHAPE      # K == 0
    assert f(P, P, P, P, 128, 100, 64, 1, 32, 1, 1.0, P, None) == SHAPE     # N % 8
    assert f(P, P, P, P, -1, 128, 64, 1, 32, 1, 1.0, P, None) == SHAPE
    assert f(P, P, P, P, 65535 * 128 + 1, 8, 64, 1, 32, 1, 1.0, P, None) == SHAPE
    assert f(P, P, P, P, 1 << 34, 8, 64, 1, 32, 1, 1.0, P, None) == SHAPE
    assert f(P, P, P, P, 128, 128, 64, 3, 32, 1, 1.0, P, None) == UNSUP     # fmt (NVFP4 is 3)
    assert f(P, P, P, P, 128, 128, 64, 1, 16, 1, 1.0, P, None) == UNSUP     # group
    assert f(P, P, P, P, 128, 128, 64, 1, 32, 2, 1.0, P, None) == UNSUP     # layout
    for i in range(5):
        args = [P, P, P, P]
        if i < 4:
            args[i] = None
        assert f(*args, 128, 128, 64, 1, 32, 1, 1.0, None if i == 4 else P, None) == NULL
    assert f(P + 8, P, P, P, 128, 128, 64, 1, 32, 1, 1.0, P, None) == ALIGN
    assert f(P, P, P + 8, P, 128, 128, 64, 2, 32, 1, 1.0, P, None) == ALIGN
    assert f(P, P, P, P, 128, 128, 64, 1, 32, 1, 1.0, P + 2, None) == ALIGN
    assert f(P, P + 1, P, P, 128, 128, 64, 1, 32, 1, 1.0, P, None) == ALIGN  # swizzled scales
    assert f(P, P, P, P + 4, 128, 128, 64, 1, 32, 1, 1.0, P, None) == ALIGN
    assert f(P, P + 1, P, P, 128, 128, 64, 1, 32, 0, 1.0, P, None) == ALIGN   # linear: 2 bytes
    assert f(P, P, P, P + 3, 128, 128, 64, 2, 32, 0, 1.0, P, None) == ALIGN
    assert f(None, None, None, None, 0, 128, 64, 1, 32, 1, 1.0, None, None) == OK
    assert f(None, None, None, None, 128, 0, 64, 2, 32, 0, 1.0, None, None) == OK


def test_selftest_gemm_give_up_validation(L):
    f = L.mx_selftest_gemm_give_up  # (a, sa, b, sb, M, N, K, fmt, layout, c, limit_ns, stream)
    assert f(P, P, P, P, 128, 128, 64, 1, 1, P, 0, None) == SHAPE             # limit out of range
    assert f(P, P, P, P, 128, 128, 64, 1, 1, P, 100_000_001, None) == SHAPE
    assert f(P, P, P, P, 0, 128, 64, 1, 1, P, 1000, None) == SHAPE            # empty
    assert f(P, P, P, P, 128, 0, 64, 1, 1, P, 1000, None) == SHAPE
    assert f(P, P, P, P, 128, 128, 96, 1, 1, P, 1000, None) == SHAPE          # K % 64
    assert f(P, P, P, P, 128, 128, 64, 3, 1, P, 1000, None) == UNSUP
    assert f(None, P, P, P, 128, 128, 64, 1, 1, P, 1000, None) == NULL
    assert f(P, P, P, P, 128, 128, 64, 1, 1, P + 8, 1000, None) == ALIGN


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(mxq, "_lib", None)
    monkeypatch.setattr(mxq, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        mxq.lib()
