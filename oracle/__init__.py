"""CPU oracle for OCP-MX block quantization -- TEST INFRASTRUCTURE ONLY.

A plain, slow, double-precision C++ definition of what the GPU path computes (mx_oracle.cpp),
loaded through ctypes. Only tests/, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of bench.py may import this package. The product library never
imports, links or calls it, and the two share no code.

Every function takes and returns numpy arrays in host memory. bf16 tensors travel as their raw
uint16 bit patterns. Format ids: ``E2M1`` (MXFP4) and ``E4M3`` (MXFP8); scale layouts:
``LINEAR`` ([M, K/32] row-major) and ``SWIZZLED`` (128x4 blocked, padded).
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

E2M1 = 1
E4M3 = 2
LINEAR = 0
SWIZZLED = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mx_oracle.cpp")
_LIB = os.path.join(_HERE, "libmx_oracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile mx_oracle.cpp into libmx_oracle.so beside it (plain g++, no fast-math)."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["g++", "-std=c++17", "-O2", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
             _SRC, "-o", tmp])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
    p = ctypes.c_void_p
    sig = {
        "mxo_emax": (i32, [i32]),
        "mxo_decode": (dbl, [i32, i32]),
        "mxo_bf16_to_double": (dbl, [ctypes.c_uint16]),
        "mxo_double_to_bf16": (ctypes.c_uint16, [dbl]),
        "mxo_scale_byte": (i32, [i32, dbl]),
        "mxo_quantize_block": (i32, [i32, p, i32, i32, p]),
        "mxo_dequant_bf16": (ctypes.c_uint16, [i32, i32, i32]),
        "mxo_swizzled_offset": (i64, [i64, i64, i64]),
        "mxo_scales_shape": (None, [i64, i64, i32, p, p]),
        "mxo_quantize": (None, [p, i64, i64, i32, i32, p, p]),
        "mxo_qdq": (None, [p, i64, i64, i32, p]),
        "mxo_dequantize": (None, [p, p, i64, i64, i32, i32, p]),
        "mxo_rotate": (None, [p, i64, i64, p, i32, p]),
        "mxo_rotate_quantize": (None, [p, i64, i64, p, i32, i32, i32, p, p]),
        "mxo_rotate_qdq": (None, [p, i64, i64, p, i32, i32, p]),
        "mxo_quantize_values": (None, [p, i64, i64, i32, i32, p, p]),
        "mxo_qdq_values": (None, [p, i64, i64, i32, p]),
        "mxo_nvfp4_values": (None, [p, i64, i64, ctypes.c_float, i32, p, p, p]),
        "mxo_quest_alpha": (dbl, []),
        "mxo_quest_scale_byte": (i32, [p, i32]),
        "mxo_quest_quantize_block": (i32, [p, i32, p]),
        "mxo_quest_quantize_values": (None, [p, i64, i64, i32, p, p]),
        "mxo_quest_qdq_values": (None, [p, i64, i64, p]),
        "mxo_quantize_grouped": (None, [p, p, i32, i64, i32, i32, i64, p, p]),
        "mxo_nvfp4_scales_shape": (None, [i64, i64, i32, p, p]),
        "mxo_nvfp4_block": (i32, [p, i32, ctypes.c_float, p]),
        "mxo_nvfp4_dequant_bf16": (ctypes.c_uint16, [i32, i32, ctypes.c_float]),
        "mxo_nvfp4_quantize": (None, [p, i64, i64, p, i32, ctypes.c_float, i32, p, p]),
        "mxo_nvfp4_qdq": (None, [p, i64, i64, p, i32, ctypes.c_float, p]),
        "mxo_nvfp4_dequantize": (None, [p, p, i64, i64, ctypes.c_float, i32, p]),
        "mxo_nvfp4_quantize_grouped": (None, [p, p, i32, i64, p, i32, i64, p, p]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def _bits(x) -> np.ndarray:
    x = np.ascontiguousarray(x)
    assert x.dtype == np.uint16, "bf16 tensors are passed as uint16 bit patterns"
    return x


# ----------------------------------------------------------------------------------------------
# scalar helpers
# ----------------------------------------------------------------------------------------------
def emax(fmt: int) -> int:
    return _load().mxo_emax(fmt)


def decode(fmt: int, code: int) -> float:
    """Value of one element code (sign included), scale 2^0."""
    return _load().mxo_decode(fmt, code)


def bf16_to_double(bits: int) -> float:
    return _load().mxo_bf16_to_double(bits)


def double_to_bf16(v: float) -> int:
    """Round a double to bf16 once (nearest, ties to even); returns the bit pattern."""
    return _load().mxo_double_to_bf16(v)


def scale_byte(fmt: int, amax: float) -> int:
    """E8M0 byte of a block with the given (finite, non-negative) abs-max."""
    return _load().mxo_scale_byte(fmt, amax)


def quantize_block(fmt: int, values, forced_byte: int = -1):
    """Quantize one block of float64 values; returns (scale byte, unpacked codes uint8)."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    codes = np.zeros(v.size, dtype=np.uint8)
    b = _load().mxo_quantize_block(fmt, _ptr(v), v.size, forced_byte, _ptr(codes))
    return b, codes


def dequant_bf16(fmt: int, code: int, scale: int) -> int:
    return _load().mxo_dequant_bf16(fmt, code, scale)


def swizzled_offset(r: int, c: int, padded_cols: int) -> int:
    return _load().mxo_swizzled_offset(r, c, padded_cols)


def scales_shape(M: int, K: int, layout: int):
    rows = ctypes.c_int64()
    cols = ctypes.c_int64()
    _load().mxo_scales_shape(M, K, layout, ctypes.byref(rows), ctypes.byref(cols))
    return rows.value, cols.value


def grouped_scales_rows(counts, layout: int) -> int:
    counts = [int(c) for c in counts]
    if layout == LINEAR:
        return sum(counts)
    return sum(-(-c // 128) * 128 for c in counts)


def code_bytes_per_row(fmt: int, K: int) -> int:
    return K if fmt == E4M3 else K // 2


# ----------------------------------------------------------------------------------------------
# tensor operations
# ----------------------------------------------------------------------------------------------
def quantize(x_bits, fmt: int, layout: int):
    """-> (codes uint8 [M, K or K/2], scales uint8 [rows, cols])."""
    x = _bits(x_bits)
    M, K = x.shape
    codes = np.zeros((M, code_bytes_per_row(fmt, K)), dtype=np.uint8)
    scales = np.zeros(scales_shape(M, K, layout), dtype=np.uint8)
    _load().mxo_quantize(_ptr(x), M, K, fmt, layout, _ptr(codes), _ptr(scales))
    return codes, scales


def qdq(x_bits, fmt: int) -> np.ndarray:
    """-> bf16 bits [M, K]."""
    x = _bits(x_bits)
    M, K = x.shape
    out = np.zeros((M, K), dtype=np.uint16)
    _load().mxo_qdq(_ptr(x), M, K, fmt, _ptr(out))
    return out


def dequantize(codes, scales, K: int, fmt: int, layout: int) -> np.ndarray:
    """codes [M, K or K/2] uint8 and scales (linear [M, K/32] or swizzled) -> bf16 bits [M, K].
    Scale byte 0xFF and E4M3 NaN codes give the bf16 NaN 0x7FC0."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    M = c.shape[0]
    assert c.shape[1] == code_bytes_per_row(fmt, K)
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    assert s.shape == scales_shape(M, K, layout)
    out = np.zeros((M, K), dtype=np.uint16)
    _load().mxo_dequantize(_ptr(c), _ptr(s), M, K, fmt, layout, _ptr(out))
    return out


def rotate(x_bits, H_bits) -> np.ndarray:
    """Pre-quantization rotated values y (float64 [M, K]), y_chunk = x_chunk @ H."""
    x = _bits(x_bits)
    H = _bits(H_bits)
    M, K = x.shape
    g = H.shape[0]
    y = np.zeros((M, K), dtype=np.float64)
    _load().mxo_rotate(_ptr(x), M, K, _ptr(H), g, _ptr(y))
    return y


def rotate_quantize(x_bits, H_bits, fmt: int, layout: int):
    x = _bits(x_bits)
    H = _bits(H_bits)
    M, K = x.shape
    codes = np.zeros((M, code_bytes_per_row(fmt, K)), dtype=np.uint8)
    scales = np.zeros(scales_shape(M, K, layout), dtype=np.uint8)
    _load().mxo_rotate_quantize(_ptr(x), M, K, _ptr(H), H.shape[0], fmt, layout, _ptr(codes),
                                _ptr(scales))
    return codes, scales


def rotate_qdq(x_bits, H_bits, fmt: int) -> np.ndarray:
    x = _bits(x_bits)
    H = _bits(H_bits)
    M, K = x.shape
    out = np.zeros((M, K), dtype=np.uint16)
    _load().mxo_rotate_qdq(_ptr(x), M, K, _ptr(H), H.shape[0], fmt, _ptr(out))
    return out


def _values(v) -> np.ndarray:
    v = np.ascontiguousarray(v, dtype=np.float64)
    assert v.ndim == 2
    return v


def quantize_values(v, fmt: int, layout: int):
    """Quantize float64 values [M, K] (rotated values from ``rotate``, for instance): the same
    steps as ``quantize`` after its bf16 decode. -> (codes, scales)."""
    v = _values(v)
    M, K = v.shape
    codes = np.zeros((M, code_bytes_per_row(fmt, K)), dtype=np.uint8)
    scales = np.zeros(scales_shape(M, K, layout), dtype=np.uint8)
    _load().mxo_quantize_values(_ptr(v), M, K, fmt, layout, _ptr(codes), _ptr(scales))
    return codes, scales


def qdq_values(v, fmt: int) -> np.ndarray:
    """QDQ of float64 values [M, K] -> bf16 bits [M, K] (``qdq`` after its bf16 decode)."""
    v = _values(v)
    M, K = v.shape
    out = np.zeros((M, K), dtype=np.uint16)
    _load().mxo_qdq_values(_ptr(v), M, K, fmt, _ptr(out))
    return out


# ----------------------------------------------------------------------------------------------
# Quest-like scale (MXFP4): E8M0 scale from the clip point alpha * RMS of the block instead of its
# abs-max (mx_oracle.cpp, quest_scale_byte, states the reading); E2M1 elements.
# ----------------------------------------------------------------------------------------------
def quest_alpha() -> float:
    """The clip ratio alpha the oracle uses (clip point over the block's RMS)."""
    return _load().mxo_quest_alpha()


def quest_scale_byte(values) -> int:
    """E8M0 byte of one block of finite values under the Quest-like rule."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    return _load().mxo_quest_scale_byte(_ptr(v), v.size)


def quest_quantize_block(values):
    """-> (scale byte, unpacked E2M1 codes uint8 [n]) of one block under the Quest-like rule."""
    v = np.ascontiguousarray(values, dtype=np.float64)
    codes = np.zeros(v.size, dtype=np.uint8)
    byte = _load().mxo_quest_quantize_block(_ptr(v), v.size, _ptr(codes))
    return byte, codes


def quest_quantize_values(v, layout: int):
    """Quest-like MXFP4 quantize of float64 values [M, K] -> (codes [M, K/2], scales)."""
    v = _values(v)
    M, K = v.shape
    codes = np.zeros((M, K // 2), dtype=np.uint8)
    scales = np.zeros(scales_shape(M, K, layout), dtype=np.uint8)
    _load().mxo_quest_quantize_values(_ptr(v), M, K, layout, _ptr(codes), _ptr(scales))
    return codes, scales


def quest_qdq_values(v) -> np.ndarray:
    """Quest-like MXFP4 QDQ of float64 values [M, K] -> bf16 bits [M, K]."""
    v = _values(v)
    M, K = v.shape
    out = np.zeros((M, K), dtype=np.uint16)
    _load().mxo_quest_qdq_values(_ptr(v), M, K, _ptr(out))
    return out


def _quest_inputs(x_bits, H_bits):
    return bf16_bits_to_double(_bits(x_bits)) if H_bits is None else rotate(x_bits, H_bits)


def quest_quantize(x_bits, layout: int, H_bits=None):
    """Quest-like MXFP4 quantize of bf16 x [M, K], rotated first by H when given."""
    return quest_quantize_values(_quest_inputs(x_bits, H_bits), layout)


def quest_qdq(x_bits, H_bits=None) -> np.ndarray:
    """Quest-like MXFP4 QDQ of bf16 x [M, K] (in the rotated basis when H is given)."""
    return quest_qdq_values(_quest_inputs(x_bits, H_bits))


def quantize_grouped(x_bits, offsets, fmt: int, layout: int, scale_rows: int | None = None):
    """Per-expert quantize. offsets: int64 [E+1] row offsets (host)."""
    x = _bits(x_bits)
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    E = off.size - 1
    M, K = x.shape
    assert off[E] == M
    counts = np.diff(off)
    if scale_rows is None:
        scale_rows = grouped_scales_rows(counts, layout)
    cols = K // 32 if layout == LINEAR else -(-(K // 32) // 4) * 4
    codes = np.zeros((M, code_bytes_per_row(fmt, K)), dtype=np.uint8)
    scales = np.zeros((scale_rows, cols), dtype=np.uint8)
    _load().mxo_quantize_grouped(_ptr(x), _ptr(off), E, K, fmt, layout, scale_rows, _ptr(codes),
                                 _ptr(scales))
    return codes, scales


def bf16_bits_to_double(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 values (exact: a bf16 is the upper half of an fp32)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def gemm(a_codes, a_scales, b_codes, b_scales, K: int, fmt: int, layout: int,
         alpha: float = 1.0) -> np.ndarray:
    """Block-scaled GEMM of stored MX data, float64 [M, N]:
    alpha * dequantize(A) @ dequantize(B)^T, A and B dequantized by ``dequantize`` (each value
    decode(code) * 2^(scale byte - 127) rounded to bf16 once) and multiplied in float64 (the
    QuTLASS MXFP4 test's reference: the matmul of the dequantized operands)."""
    da = bf16_bits_to_double(dequantize(a_codes, a_scales, K, fmt, layout))
    db = bf16_bits_to_double(dequantize(b_codes, b_scales, K, fmt, layout))
    return alpha * (da @ db.T)


# ----------------------------------------------------------------------------------------------
# NVFP4: E2M1 codes in blocks of 16, E4M3 block scales under an fp32 global scale gs
# ----------------------------------------------------------------------------------------------
def nvfp4_scales_shape(M: int, K: int, layout: int):
    rows = ctypes.c_int64()
    cols = ctypes.c_int64()
    _load().mxo_nvfp4_scales_shape(M, K, layout, ctypes.byref(rows), ctypes.byref(cols))
    return rows.value, cols.value


def nvfp4_block(values, gs: float):
    """One block of fp32 values -> (E4M3 scale byte, unpacked E2M1 codes)."""
    v = np.ascontiguousarray(values, dtype=np.float32)
    codes = np.zeros(v.size, dtype=np.uint8)
    b = _load().mxo_nvfp4_block(_ptr(v), v.size, float(np.float32(gs)), _ptr(codes))
    return b, codes


def nvfp4_dequant_bf16(code: int, scale: int, gs: float) -> int:
    return _load().mxo_nvfp4_dequant_bf16(code, scale, float(np.float32(gs)))


def nvfp4_quantize(x_bits, gs: float, layout: int, H_bits=None):
    """-> (codes uint8 [M, K/2], E4M3 scales uint8 [rows, cols]); H_bits rotates each g-chunk."""
    x = _bits(x_bits)
    M, K = x.shape
    H = None if H_bits is None else _bits(H_bits)
    codes = np.zeros((M, K // 2), dtype=np.uint8)
    scales = np.zeros(nvfp4_scales_shape(M, K, layout), dtype=np.uint8)
    _load().mxo_nvfp4_quantize(_ptr(x), M, K, None if H is None else _ptr(H),
                               0 if H is None else H.shape[0], float(np.float32(gs)), layout,
                               _ptr(codes), _ptr(scales))
    return codes, scales


def nvfp4_qdq(x_bits, gs: float, H_bits=None) -> np.ndarray:
    x = _bits(x_bits)
    M, K = x.shape
    H = None if H_bits is None else _bits(H_bits)
    out = np.zeros((M, K), dtype=np.uint16)
    _load().mxo_nvfp4_qdq(_ptr(x), M, K, None if H is None else _ptr(H),
                          0 if H is None else H.shape[0], float(np.float32(gs)), _ptr(out))
    return out


def nvfp4_values(v, gs: float, layout: int, codes=True, scales=True, qdq=True):
    """NVFP4 of float64 values [M, K] (rotated values from ``rotate``, for instance), each
    rounded to fp32 once first: -> (codes [M, K/2], scales, QDQ bf16 bits [M, K]), None for an
    output not asked for."""
    v = _values(v)
    M, K = v.shape
    c = np.zeros((M, K // 2), dtype=np.uint8) if codes else None
    s = np.zeros(nvfp4_scales_shape(M, K, layout), dtype=np.uint8) if scales else None
    q = np.zeros((M, K), dtype=np.uint16) if qdq else None
    _load().mxo_nvfp4_values(_ptr(v), M, K, float(np.float32(gs)), layout,
                             None if c is None else _ptr(c), None if s is None else _ptr(s),
                             None if q is None else _ptr(q))
    return c, s, q


def nvfp4_dequantize(codes, scales, K: int, gs: float, layout: int) -> np.ndarray:
    """Stored NVFP4 codes [M, K/2] + E4M3 scales (linear or swizzled) -> bf16 bits [M, K]."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    s = np.ascontiguousarray(scales, dtype=np.uint8)
    M = c.shape[0]
    y = np.zeros((M, K), dtype=np.uint16)
    _load().mxo_nvfp4_dequantize(_ptr(c), _ptr(s), M, K, float(np.float32(gs)), layout, _ptr(y))
    return y


def nvfp4_quantize_grouped(x_bits, offsets, gs, layout: int, scale_rows: int | None = None):
    """Per-expert NVFP4 quantize. offsets: int64 [E+1] row offsets; gs: fp32 [E] global scales
    (one per expert). -> (codes [M, K/2], scales: linear [M, K/16] or per-expert padded
    swizzled [scale_rows, ceil(K/64)*4])."""
    x = _bits(x_bits)
    off = np.ascontiguousarray(offsets, dtype=np.int64)
    g = np.ascontiguousarray(gs, dtype=np.float32)
    E = off.size - 1
    M, K = x.shape
    assert off[E] == M and g.size == E
    if scale_rows is None:
        scale_rows = grouped_scales_rows(np.diff(off), layout)
    cols = nvfp4_scales_shape(0, K, layout)[1]
    codes = np.zeros((M, K // 2), dtype=np.uint8)
    scales = np.zeros((scale_rows, cols), dtype=np.uint8)
    _load().mxo_nvfp4_quantize_grouped(_ptr(x), _ptr(off), E, K, _ptr(g), layout, scale_rows,
                                       _ptr(codes), _ptr(scales))
    return codes, scales
