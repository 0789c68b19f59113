"""Pins for the CPU oracle: each test checks it against something other than itself.

Sources of truth used here: the format definitions (spec constants and structure), closed forms
worked by hand (tests/golden/), torch's CPU float8_e4m3fn / float8_e8m0fnu / bfloat16 casts
(library routines), numpy/scipy routines, brute force and invariants.
"""

import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from mx_microscaling_quantize_gb300 import workloads as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16(values) -> np.ndarray:
    return W.to_bf16_bits(np.asarray(values, dtype=np.float32))


def all_finite_bf16() -> np.ndarray:
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return b[((b >> 7) & 0xFF) != 0xFF]


# ---------------------------------------------------------------------------------------------
# element grids
# ---------------------------------------------------------------------------------------------
def test_e2m1_grid_from_spec_properties():
    """E2M1: 8 magnitudes, strictly increasing; 0; min subnormal 0.5; min normal 1.0;
    max normal 6.0; two values per binade (one mantissa bit); sign-magnitude codes."""
    mags = [O.decode(O.E2M1, c) for c in range(8)]
    assert mags[0] == 0.0
    assert all(a < b for a, b in zip(mags, mags[1:]))
    assert mags[1] == 0.5 and mags[2] == 1.0 and mags[7] == 6.0
    for e in range(0, 3):  # binades [1,2), [2,4), [4,8)
        inside = [m for m in mags if 2.0 ** e <= m < 2.0 ** (e + 1)]
        assert len(inside) == 2 and inside[0] == 2.0 ** e
        assert inside[1] - inside[0] == 2.0 ** (e - 1)
    for c in range(8):
        assert O.decode(O.E2M1, c | 8) == -mags[c]
        assert math.copysign(1.0, O.decode(O.E2M1, c | 8)) == -1.0


def test_e4m3_decode_matches_torch_all_bytes():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    for c in range(256):
        if c & 0x7F == 0x7F:
            assert np.isnan(ref[c])  # the format's only NaN; quantization never emits it
            assert np.isnan(O.decode(O.E4M3, c))
            continue
        assert O.decode(O.E4M3, c) == ref[c], hex(c)
        assert math.copysign(1.0, O.decode(O.E4M3, c)) == math.copysign(1.0, ref[c])


def test_e4m3_encode_matches_torch_cast_in_range():
    """At scale byte 127 (s = 0) the element code is torch's RNE float8_e4m3fn cast, for every
    finite bf16 value whose magnitude is below 464 (beyond, torch returns NaN, no saturation)."""
    bits = all_finite_bf16()
    vals = W.bf16_bits_to_float(bits).astype(np.float64)
    keep = np.abs(vals) < 464
    bits, vals = bits[keep], vals[keep]
    _, codes = O.quantize_block(O.E4M3, vals, forced_byte=127)
    ref = torch.from_numpy(vals.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8)
    np.testing.assert_array_equal(codes, ref.numpy())


def test_e4m3_saturates():
    vals = np.array([464.0, 465.0, 480.0, 1e6, 3.0e38, -464.0, -1e30])
    _, codes = O.quantize_block(O.E4M3, vals, forced_byte=127)
    np.testing.assert_array_equal(codes, [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE])


def test_e2m1_nearest_and_ties_brute_force():
    """For t on a fine grid, the E2M1 code is a nearest grid point and, on ties, the even code."""
    mags = np.array([O.decode(O.E2M1, c) for c in range(8)])
    t = np.arange(-8 * 64, 8 * 64 + 1) / 64.0
    _, codes = O.quantize_block(O.E2M1, t, forced_byte=127)
    for ti, c in zip(t, codes):
        m = mags[c & 7]
        a = min(abs(ti), 6.0)
        d = np.abs(mags - a)
        assert abs(m - a) == d.min(), (ti, c)
        if np.sum(d == d.min()) == 2:
            assert (c & 1) == 0, (ti, c)
        assert bool(c & 8) == (ti < 0 or (ti == 0 and math.copysign(1, ti) < 0)), (ti, c)


def _read_worked_blocks(name):
    blocks = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split()
        if parts[0] == "block":
            blocks.append((parts[1], int(parts[2]), []))
        else:
            blocks[-1][2].append((float(parts[0]), int(parts[1], 16)))
    return blocks


@pytest.mark.parametrize("fmt,name", [(O.E2M1, "e2m1_worked_blocks.txt"),
                                      (O.E4M3, "e4m3_worked_blocks.txt")])
def test_worked_blocks(fmt, name):
    for bname, byte, entries in _read_worked_blocks(name):
        v = np.zeros(32)
        want = np.zeros(32, dtype=np.uint8)
        for i, (val, code) in enumerate(entries):
            v[i] = val
            want[i] = code
        assert bf16(v).astype(np.uint32).tolist() == bf16(v).tolist()
        assert (W.bf16_bits_to_float(bf16(v)) == v.astype(np.float32)).all(), bname
        got_byte, got = O.quantize_block(fmt, v)
        assert got_byte == byte, bname
        np.testing.assert_array_equal(got, want, err_msg=bname)
        # the same block through the tensor entry point (packing / linear scale layout)
        codes, scales = O.quantize(bf16(v).reshape(1, 32), fmt, O.LINEAR)
        assert scales[0, 0] == byte
        if fmt == O.E4M3:
            np.testing.assert_array_equal(codes[0], want)
        else:
            np.testing.assert_array_equal(codes[0] & 0xF, want[0::2])
            np.testing.assert_array_equal(codes[0] >> 4, want[1::2])


# ---------------------------------------------------------------------------------------------
# scales
# ---------------------------------------------------------------------------------------------
def test_scale_bytes_closed_form_table():
    for line in open(os.path.join(GOLDEN, "scale_bytes.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        a, b2, b8 = line.split()
        amax = 2.0 ** int(a[2:]) if a.startswith("2^") else float(a)
        assert O.scale_byte(O.E2M1, amax) == int(b2), a
        assert O.scale_byte(O.E4M3, amax) == int(b8), a
        # through a whole block (amax placed at a varying position)
        v = np.zeros(32)
        v[int(b2) % 32] = -amax
        assert O.quantize_block(O.E2M1, v)[0] == int(b2)
        assert O.quantize_block(O.E4M3, v)[0] == int(b8)


@pytest.mark.parametrize("fmt", [O.E2M1, O.E4M3])
def test_scale_bracket_invariant_every_bf16_amax(fmt):
    """For every non-negative finite bf16 amax: 2^(s+emax) <= amax < 2^(s+emax+1) unless the
    scale is clamped at s = -127 (then amax < 2^(-127+emax+1)); decode via torch's e8m0."""
    emax = 2 if fmt == O.E2M1 else 8
    bits = all_finite_bf16()
    bits = bits[bits < 0x8000]
    vals = W.bf16_bits_to_float(bits).astype(np.float64)
    e8 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).double().numpy()
    for amax in vals:
        byte = O.scale_byte(fmt, float(amax))
        assert 0 <= byte <= 254
        scale = e8[byte]
        if amax == 0:
            assert byte == 0
            continue
        lo = scale * 2.0 ** emax
        if byte > 0:
            assert lo <= amax < 2 * lo, (amax, byte)
        else:
            assert amax < 2 * lo, (amax, byte)
            assert amax < 2.0 ** (-126 + emax) or lo <= amax


def test_zero_block():
    for fmt in (O.E2M1, O.E4M3):
        b, codes = O.quantize_block(fmt, np.zeros(32))
        assert b == 0 and not codes.any()
        v = np.zeros(32)
        v[3] = -0.0
        b, codes = O.quantize_block(fmt, v)
        sign = 0x8 if fmt == O.E2M1 else 0x80
        assert b == 0 and codes[3] == sign and codes.sum() == sign


def test_nan_and_inf_blocks():
    for fmt, fill in ((O.E2M1, 0), (O.E4M3, 0x7F)):
        for bad in (float("nan"), float("inf"), -float("inf")):
            v = np.linspace(-1, 1, 32)
            v[7] = bad
            b, codes = O.quantize_block(fmt, v)
            assert b == 0xFF and (codes == fill).all()
            x = bf16(v).reshape(1, 32)
            assert (O.qdq(x, fmt) == 0x7FC0).all()


# ---------------------------------------------------------------------------------------------
# round trip, dequantization, idempotence
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", [O.E2M1, O.E4M3])
def test_every_representable_value_round_trips_at_scale_one(fmt):
    n = 16 if fmt == O.E2M1 else 256
    sign = 0x8 if fmt == O.E2M1 else 0x80
    anchor = 6.0 if fmt == O.E2M1 else 448.0  # amax in [2^emax, 2^(emax+1)) forces s = 0
    for c in range(n):
        if fmt == O.E4M3 and (c & 0x7F) == 0x7F:
            continue
        v = np.zeros(32)
        v[0] = anchor
        v[1] = O.decode(fmt, c)
        b, codes = O.quantize_block(fmt, v)
        assert b == 127
        assert codes[1] == c or (v[1] == 0 and (codes[1] & ~sign) == 0 and codes[1] == c)
        x = bf16(v).reshape(1, 32)
        out = O.qdq(x, fmt)
        np.testing.assert_array_equal(out, x)


def test_dequant_matches_torch_bf16_rounding():
    """decode(code) * 2^s rounded once to bf16 == torch's float64 -> bfloat16 cast of the same
    exact product (exact in float32, so torch's float path rounds it once)."""
    for fmt, codes in ((O.E2M1, range(16)), (O.E4M3, [c for c in range(256) if c & 0x7F != 0x7F])):
        for byte in list(range(0, 12)) + list(range(120, 135)) + list(range(240, 255)):
            for c in codes:
                exact = O.decode(fmt, c) * 2.0 ** (byte - 127)
                want = torch.tensor([exact], dtype=torch.float64).to(torch.bfloat16)
                want = int(want.view(torch.int16).item()) & 0xFFFF
                assert O.dequant_bf16(fmt, c, byte) == want, (fmt, c, byte)


def test_bf16_conversions_against_torch():
    bits = all_finite_bf16()
    for b in bits[::97]:
        v = O.bf16_to_double(int(b))
        t = torch.tensor([int(b)], dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
        assert v == t.double().item() and math.copysign(1, v) == math.copysign(1, t.item())
        assert O.double_to_bf16(v) == b
    rng = np.random.default_rng(5)
    vals = rng.standard_normal(2000).astype(np.float32) * np.float32(2.0) ** rng.integers(
        -140, 120, 2000).astype(np.float32)
    want = W.to_bf16_bits(vals)
    got = np.array([O.double_to_bf16(float(v)) for v in vals], dtype=np.uint16)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("fmt", [O.E2M1, O.E4M3])
def test_qdq_idempotent(fmt):
    x = W.mxfp4_qdq_activation(64, 256)
    y = O.qdq(x, fmt)
    z = O.qdq(y, fmt)
    np.testing.assert_array_equal(z, y)
    x = W.mxfp4_qdq_weight(64, 256)
    y = O.qdq(x, fmt)
    np.testing.assert_array_equal(O.qdq(y, fmt), y)


def test_qdq_equals_dequantized_codes():
    x = W.mxfp8_linear_quant(8, 256)
    for fmt in (O.E2M1, O.E4M3):
        codes, scales = O.quantize(x, fmt, O.LINEAR)
        out = O.qdq(x, fmt)
        for r in range(8):
            for k in range(0, 256, 7):
                if fmt == O.E4M3:
                    c = codes[r, k]
                else:
                    c = (codes[r, k // 2] >> (4 * (k % 2))) & 0xF
                assert out[r, k] == O.dequant_bf16(fmt, int(c), int(scales[r, k // 32]))


# ---------------------------------------------------------------------------------------------
# dequantization of stored codes and scales
# ---------------------------------------------------------------------------------------------
E2M1_SPEC_VALUES = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]  # OCP MX E2M1 magnitudes, codes 0..7


def torch_bf16_bits(values: torch.Tensor) -> np.ndarray:
    return values.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("layout", [O.LINEAR, O.SWIZZLED])
@pytest.mark.parametrize("M,K", [(1, 32), (130, 416), (64, 4096)])
def test_dequantize_of_quantize_is_qdq(M, K, layout):
    x = W.mxfp4_qdq_activation(M, K) if K % 1024 == 0 else W.mxfp8_linear_quant(M, K, stream=K)
    for fmt in (O.E2M1, O.E4M3):
        codes, scales = O.quantize(x, fmt, layout)
        np.testing.assert_array_equal(O.dequantize(codes, scales, K, fmt, layout), O.qdq(x, fmt))


def test_dequantize_e4m3_every_code_and_scale_against_torch():
    """Random E4M3 bytes (NaN codes included) under every E8M0 byte: torch's float8_e4m3fn and
    float8_e8m0fnu decodes, multiplied in float64 (exact) and cast once to bfloat16."""
    rng = np.random.default_rng(21)
    M, K = 256, 1024
    codes = rng.integers(0, 256, (M, K), dtype=np.uint8)
    codes[0, :256] = np.arange(256, dtype=np.uint8)
    scales = rng.integers(0, 256, (M, K // 32), dtype=np.uint8)
    scales[1:, 0] = np.arange(255, dtype=np.uint8)
    v = torch.from_numpy(codes).view(torch.float8_e4m3fn).double()
    s = torch.from_numpy(scales).view(torch.float8_e8m0fnu).double().repeat_interleave(32, dim=1)
    want = torch_bf16_bits(v * s)
    got = O.dequantize(codes, scales, K, O.E4M3, O.LINEAR)
    nan = np.isnan((v * s).numpy())
    assert nan.any() and (got[nan] == 0x7FC0).all()
    np.testing.assert_array_equal(got[~nan], want[~nan])
    assert (got == 0x7F80).any() and (got == 0x0000).any()  # overflow to Inf and underflow hit


def test_dequantize_e2m1_nibbles_against_spec_table():
    """Packed E2M1 bytes: the even K index in the low nibble, magnitudes from the OCP table,
    sign bit 0x8; scales read through the 128x4 blocked layout give the same values."""
    rng = np.random.default_rng(22)
    M, K = 200, 640
    packed = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    scales = rng.integers(0, 256, (M, K // 32), dtype=np.uint8)
    nib = np.empty((M, K), dtype=np.int64)
    nib[:, 0::2] = packed & 0xF
    nib[:, 1::2] = packed >> 4
    table = np.array(E2M1_SPEC_VALUES + [-v for v in E2M1_SPEC_VALUES])
    v = torch.from_numpy(table[nib])
    s = torch.from_numpy(scales).view(torch.float8_e8m0fnu).double().repeat_interleave(32, dim=1)
    want = torch_bf16_bits(v * s)
    want[np.isnan((v * s).numpy())] = 0x7FC0
    np.testing.assert_array_equal(O.dequantize(packed, scales, K, O.E2M1, O.LINEAR), want)
    swz = to_blocked_reference(torch.from_numpy(scales)).numpy()
    swz = swz.reshape(O.scales_shape(M, K, O.SWIZZLED))
    np.testing.assert_array_equal(O.dequantize(packed, swz, K, O.E2M1, O.SWIZZLED), want)


def test_dequantize_subnormal_and_overflow_closed_forms():
    """Worked by hand: bf16 subnormals are m * 2^-133. E4M3 0x0F = 1.875 * 2^-6 under 2^-127 is
    1.875 * 2^-133 -> 2 * 2^-133 (0x0002); 0x0C = 1.5 * 2^-133 ties to even -> 0x0002; 0x09 ->
    0x0001; 0x01 = 2^-136 -> +0; 0x8F -> 0x8002. E2M1 6 * 2^127 overflows to Inf (0x7F80,
    0xFF80 for code 0xF); E4M3 448 * 2^119 = 1.75 * 2^127 is exact: 0x7F60."""
    cases = [(O.E4M3, 0x0F, 0, 0x0002), (O.E4M3, 0x0C, 0, 0x0002), (O.E4M3, 0x09, 0, 0x0001),
             (O.E4M3, 0x01, 0, 0x0000), (O.E4M3, 0x8F, 0, 0x8002), (O.E2M1, 0x7, 254, 0x7F80),
             (O.E2M1, 0xF, 254, 0xFF80), (O.E4M3, 0x7E, 246, 0x7F60), (O.E2M1, 0x1, 0, 0x0020),
             (O.E4M3, 0x7F, 127, 0x7FC0), (O.E2M1, 0x2, 255, 0x7FC0)]
    for fmt, code, byte, want in cases:
        K = 32
        if fmt == O.E4M3:
            codes = np.full((1, K), code, dtype=np.uint8)
        else:
            codes = np.full((1, K // 2), code | (code << 4), dtype=np.uint8)
        out = O.dequantize(codes, np.full((1, 1), byte, dtype=np.uint8), K, fmt, O.LINEAR)
        assert (out == want).all(), (fmt, hex(code), byte, hex(int(out[0, 0])))


# ---------------------------------------------------------------------------------------------
# NVFP4 (two-level reading: E4M3 block scale of 16 under an fp32 global scale)
# ---------------------------------------------------------------------------------------------
def read_nvfp4_golden():
    out = []
    for line in open(os.path.join(GOLDEN, "nvfp4_worked_blocks.txt")):
        if not line.strip() or line.startswith("#"):
            continue
        name, gs, vals, sc, codes, qdq = [f.strip() for f in line.split("|")]
        out.append((name, float(gs), [float(v) for v in vals.split()], int(sc, 16),
                    [int(c, 16) for c in codes.split()], [int(q, 16) for q in qdq.split()]))
    return out


@pytest.mark.parametrize("case", read_nvfp4_golden(), ids=lambda c: c[0])
def test_nvfp4_worked_blocks(case):
    name, gs, vals, sc, codes, qdq = case
    b, c = O.nvfp4_block(vals, gs)
    assert b == sc and list(c) == codes
    x = bf16(vals).reshape(1, 16)
    x = np.concatenate([x, x], axis=1)  # K = 32: two identical blocks
    np.testing.assert_array_equal(O.nvfp4_qdq(x, gs)[0, :16], np.array(qdq, dtype=np.uint16))
    cq, sq = O.nvfp4_quantize(x, gs, O.LINEAR)
    assert list(sq[0]) == [sc, sc]
    assert [(cq[0, k // 2] >> (4 * (k % 2))) & 0xF for k in range(16)] == codes


def test_nvfp4_special_block():
    v = [1.0] * 16
    v[3] = float("nan")
    b, c = O.nvfp4_block(v, 1.0)
    assert b == 0x7F and not c.any()
    assert O.nvfp4_dequant_bf16(2, 0x7F, 1.0) == 0x7FC0


def test_nvfp4_scale_is_torch_e4m3_cast_of_the_fp32_scale():
    """The scale byte is torch's RNE float8_e4m3fn cast of s_f = amax * (gs / 6) (fp32 ops in
    numpy), for scales inside the E4M3 range."""
    rng = np.random.default_rng(31)
    for _ in range(400):
        v = (rng.standard_normal(16) * 2.0 ** rng.integers(-20, 20)).astype(np.float32)
        gs = np.float32(2.0 ** rng.uniform(-8, 12))
        s_f = np.abs(v).max() * (gs / np.float32(6.0))
        if s_f >= 448:
            continue
        want = torch.tensor([float(s_f)], dtype=torch.float32).to(torch.float8_e4m3fn)
        b, _ = O.nvfp4_block(v, gs)
        assert b == int(want.view(torch.uint8).item()), (s_f, b)


def test_nvfp4_codes_are_mx_e2m1_rounding_of_the_scaled_values():
    """Codes = the (pinned) MX E2M1 rounding at scale 2^0 of t = v * (gs / decode(sc))."""
    rng = np.random.default_rng(32)
    e4m3 = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
    for _ in range(300):
        v = (rng.standard_normal(16) * 2.0 ** rng.integers(-10, 10)).astype(np.float32)
        gs = np.float32(2.0 ** rng.uniform(-6, 10))
        b, codes = O.nvfp4_block(v, gs)
        s_dec = np.float32(e4m3[b])
        enc = gs / s_dec if s_dec != 0 else np.float32(0)
        t = (v * enc).astype(np.float64)
        byte, want = O.quantize_block(O.E2M1, t, forced_byte=127)
        assert byte == 127
        np.testing.assert_array_equal(codes, want)


def test_nvfp4_identity_rotation_and_layouts():
    x = W.mxfp4_qdq_activation(130, 256)
    gs = np.float32(448 * 6) / np.float32(W.bf16_bits_to_float(x).__abs__().max())
    eye = W.to_bf16_bits(np.eye(32))
    c0, s0 = O.nvfp4_quantize(x, gs, O.LINEAR)
    c1, s1 = O.nvfp4_quantize(x, gs, O.LINEAR, H_bits=eye)
    np.testing.assert_array_equal(c0, c1)
    np.testing.assert_array_equal(s0, s1)
    np.testing.assert_array_equal(O.nvfp4_qdq(x, gs), O.nvfp4_qdq(x, gs, H_bits=eye))
    _, sw = O.nvfp4_quantize(x, gs, O.SWIZZLED)
    want = to_blocked_reference(torch.from_numpy(s0)).numpy()
    np.testing.assert_array_equal(sw.reshape(-1), want)
    # QDQ output is the dequantization of the stored codes and scales
    q = O.nvfp4_qdq(x, gs)
    for r in range(0, 130, 13):
        for k in range(0, 256, 11):
            code = (c0[r, k // 2] >> (4 * (k % 2))) & 0xF
            assert q[r, k] == O.nvfp4_dequant_bf16(int(code), int(s0[r, k // 16]), float(gs))


def test_nvfp4_dequantize_every_code_and_scale_in_fp32_steps():
    """All 16 E2M1 codes under all 256 E4M3 scale bytes and three global scales: decode(code)
    from the OCP value table, decode(scale) by torch's float8_e4m3fn (sign included), then the
    two fp32 operations of the reading, dq = decode(scale) / gs and decode(code) * dq, in
    numpy float32 (correctly rounded), and torch's float32 -> bfloat16 cast; NaN scale bytes
    (0x7F, 0xFF) give 0x7FC0."""
    K = 32
    codes = np.tile(np.array([(2 * i) | ((2 * i + 1) << 4) for i in range(8)], np.uint8), (256, 2))
    scales = np.repeat(np.arange(256, dtype=np.uint8)[:, None], 2, axis=1)
    table = np.array(E2M1_SPEC_VALUES + [-v for v in E2M1_SPEC_VALUES], dtype=np.float32)
    code_val = np.tile(table, (256, 2))
    s_dec = torch.from_numpy(scales).view(torch.float8_e4m3fn).float().numpy()
    for gs in (1.0, 0.3712, 2.0 ** -10 * 3.0):
        g32 = np.float32(gs)
        dq = np.where(s_dec == 0, np.float32(0), s_dec / g32).astype(np.float32)
        y = (code_val * np.repeat(dq, 16, axis=1)).astype(np.float32)
        want = torch_bf16_bits(torch.from_numpy(y))
        nan = np.isnan(y)
        want[nan] = 0x7FC0
        got = O.nvfp4_dequantize(codes, scales, K, gs, O.LINEAR)
        assert nan[0x7F].all() and nan[0xFF].all() and nan.sum() == 2 * K
        np.testing.assert_array_equal(got, want)
        assert (got[0x85] != got[0x05]).any()  # the scale's sign bit is honoured


@pytest.mark.parametrize("rotated", [False, True])
def test_nvfp4_dequantize_of_quantize_is_qdq(rotated):
    x = W.mxfp4_qdq_activation(130, 512)
    H = W.normalized_hadamard_bf16(32) if rotated else None
    gs = np.float32(448 * 6) / np.float32(np.abs(W.bf16_bits_to_float(x)).max())
    q = O.nvfp4_qdq(x, gs, H_bits=H)
    for layout in (O.LINEAR, O.SWIZZLED):
        c, s = O.nvfp4_quantize(x, gs, layout, H_bits=H)
        np.testing.assert_array_equal(O.nvfp4_dequantize(c, s, 512, gs, layout), q)


# ---------------------------------------------------------------------------------------------
# layouts
# ---------------------------------------------------------------------------------------------
def to_blocked_reference(scales: torch.Tensor) -> torch.Tensor:
    """The 128x4 blocked rearrangement written with tensor reshapes (pad, cut into 128x4 tiles,
    row-block-major; inside a tile the 4 row-quarters of 32 rows are interleaved per row)."""
    rows, cols = scales.shape
    R = -(-rows // 128) * 128
    C = -(-cols // 4) * 4
    p = torch.zeros((R, C), dtype=scales.dtype)
    p[:rows, :cols] = scales
    t = p.view(R // 128, 128, C // 4, 4).permute(0, 2, 1, 3)   # [rb, cb, 128, 4]
    t = t.reshape(-1, 4, 32, 4).transpose(1, 2)                # [tile, 32, 4 quarters, 4]
    return t.reshape(-1)


@pytest.mark.parametrize("M,K", [(1, 32), (5, 96), (128, 128), (130, 416), (300, 4096)])
def test_swizzled_layout_matches_reshape_formulation_and_is_bijective(M, K):
    x = W.mxfp8_linear_quant(M, K, stream=M)
    for fmt in (O.E2M1, O.E4M3):
        codes_l, lin = O.quantize(x, fmt, O.LINEAR)
        codes_s, swz = O.quantize(x, fmt, O.SWIZZLED)
        np.testing.assert_array_equal(codes_l, codes_s)
        want = to_blocked_reference(torch.from_numpy(lin)).numpy()
        np.testing.assert_array_equal(swz.reshape(-1), want)
        R, C = swz.shape
        assert R == -(-M // 128) * 128 and C == -(-(K // 32) // 4) * 4
        offs = {O.swizzled_offset(r, c, C) for r in range(R) for c in range(C)}
        assert offs == set(range(R * C))


def test_e2m1_nibble_order():
    v = np.zeros(32)
    v[0], v[1] = 1.0, -6.0  # codes 0x2 and 0xF
    codes, _ = O.quantize(bf16(v).reshape(1, 32), O.E2M1, O.LINEAR)
    assert codes[0, 0] == 0xF2


# ---------------------------------------------------------------------------------------------
# rotation
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("g", [16, 32, 64, 128])
def test_hadamard_input_generator(g):
    import scipy.linalg
    h = W.sylvester_hadamard(g)
    np.testing.assert_array_equal(h, scipy.linalg.hadamard(g))
    hn = h * g ** -0.5
    np.testing.assert_allclose(hn @ hn.T, np.eye(g), atol=1e-15)
    hb = W.bf16_bits_to_float(W.normalized_hadamard_bf16(g)).astype(np.float64)
    assert np.all(np.abs(hb - hn) <= 2.0 ** -9 * np.abs(hn))
    if g in (16, 64):
        np.testing.assert_array_equal(hb, hn)


@pytest.mark.parametrize("g", [16, 32, 64, 128])
def test_rotation_against_numpy_matmul(g):
    K = 256
    x = W.rotation_sweep_input("attn_in", 6, K)
    H = W.normalized_hadamard_bf16(g)
    y = O.rotate(x, H)
    xd = W.bf16_bits_to_float(x).astype(np.float64)
    hd = W.bf16_bits_to_float(H).astype(np.float64)
    want = (xd.reshape(6, K // g, g) @ hd).reshape(6, K)
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-12 * np.abs(xd).max())


def test_rotation_identity_reduces_to_plain_path():
    x = W.mxfp4_qdq_activation(8, 512)
    for g in (16, 32, 64, 128):
        eye = W.to_bf16_bits(np.eye(g))
        np.testing.assert_array_equal(O.rotate(x, eye), W.bf16_bits_to_float(x))
        for fmt in (O.E2M1, O.E4M3):
            for layout in (O.LINEAR, O.SWIZZLED):
                a = O.rotate_quantize(x, eye, fmt, layout)
                b = O.quantize(x, fmt, layout)
                np.testing.assert_array_equal(a[0], b[0])
                np.testing.assert_array_equal(a[1], b[1])
            np.testing.assert_array_equal(O.rotate_qdq(x, eye, fmt), O.qdq(x, fmt))


def test_rotation_spike_gives_hadamard_row_and_norm_is_kept():
    g = 64
    H = W.normalized_hadamard_bf16(g)
    hd = W.bf16_bits_to_float(H).astype(np.float64)
    x = np.zeros((1, 128), dtype=np.float32)
    x[0, 64 + 5] = 2.0
    y = O.rotate(W.to_bf16_bits(x), H)
    assert (y[0, :64] == 0).all()
    np.testing.assert_array_equal(y[0, 64:], 2.0 * hd[5])
    xr = W.rotation_sweep_input("o_proj_in", 4, 512)
    y = O.rotate(xr, H)  # g = 64: bf16(64^-0.5) = 1/8 exactly, H orthonormal
    xd = W.bf16_bits_to_float(xr).astype(np.float64)
    for c in range(0, 512, 64):
        np.testing.assert_allclose(np.linalg.norm(y[:, c:c + 64], axis=1),
                                   np.linalg.norm(xd[:, c:c + 64], axis=1), rtol=1e-14)


def test_rotate_quantize_is_quantize_of_rotated_values():
    x = W.rotate_quant_activation(3, 256)
    H = W.normalized_hadamard_bf16(32)
    y = O.rotate(x, H)
    codes, scales = O.rotate_quantize(x, H, O.E2M1, O.LINEAR)
    for r in range(3):
        for j in range(8):
            b, c = O.quantize_block(O.E2M1, y[r, 32 * j:32 * j + 32])
            assert scales[r, j] == b
            packed = c[0::2] | (c[1::2] << 4)
            np.testing.assert_array_equal(codes[r, 16 * j:16 * j + 16], packed)


# ---------------------------------------------------------------------------------------------
# grouped (MoE)
# ---------------------------------------------------------------------------------------------
def test_grouped_single_expert_equals_plain():
    x = W.mxfp8_linear_quant(200, 256)
    off = np.array([0, 200])
    for fmt in (O.E2M1, O.E4M3):
        for layout in (O.LINEAR, O.SWIZZLED):
            a = O.quantize_grouped(x, off, fmt, layout)
            b = O.quantize(x, fmt, layout)
            np.testing.assert_array_equal(a[0], b[0])
            np.testing.assert_array_equal(a[1], b[1])


def test_grouped_experts_are_independent_blocks():
    counts = [0, 5, 128, 0, 130, 1]
    off = np.concatenate([[0], np.cumsum(counts)])
    x = W.mxfp8_linear_quant(int(off[-1]), 160)
    codes, swz = O.quantize_grouped(x, off, O.E4M3, O.SWIZZLED)
    assert swz.shape == (128 + 128 + 256 + 128, 8)
    prow = 0
    for e, n in enumerate(counts):
        if n == 0:
            continue
        c, s = O.quantize(x[off[e]:off[e + 1]], O.E4M3, O.SWIZZLED)
        np.testing.assert_array_equal(codes[off[e]:off[e + 1]], c)
        flat = swz.reshape(-1)[prow * 8:(prow + s.shape[0]) * 8]
        np.testing.assert_array_equal(flat, s.reshape(-1))
        prow += s.shape[0]


def test_nvfp4_grouped_experts_are_independent_blocks():
    """Each expert's codes and scales are the plain NVFP4 quantization of its own rows under its
    own global scale; swizzled scales sit in the expert's own run of 128-row tiles, pads zero;
    one expert covering every row is the plain call."""
    counts = [0, 5, 128, 0, 130, 1]
    off = np.concatenate([[0], np.cumsum(counts)])
    x = W.mxfp8_linear_quant(int(off[-1]), 192)
    gs = np.array([1.0, 3.0, 0.25, 7.0, 448 * 6 / 40.0, 0.5], dtype=np.float32)
    codes, swz = O.nvfp4_quantize_grouped(x, off, gs, O.SWIZZLED)
    cl, lin = O.nvfp4_quantize_grouped(x, off, gs, O.LINEAR)
    np.testing.assert_array_equal(codes, cl)
    assert swz.shape == (128 + 128 + 256 + 128, 12) and lin.shape == (264, 12)
    prow = 0
    for e, n in enumerate(counts):
        if n == 0:
            continue
        c, s = O.nvfp4_quantize(x[off[e]:off[e + 1]], gs[e], O.SWIZZLED)
        _, sl = O.nvfp4_quantize(x[off[e]:off[e + 1]], gs[e], O.LINEAR)
        np.testing.assert_array_equal(codes[off[e]:off[e + 1]], c)
        np.testing.assert_array_equal(lin[off[e]:off[e + 1]], sl)
        flat = swz.reshape(-1)[prow * 12:(prow + s.shape[0]) * 12]
        np.testing.assert_array_equal(flat, s.reshape(-1))
        prow += s.shape[0]
    one = O.nvfp4_quantize_grouped(x, np.array([0, off[-1]]), gs[4:5], O.SWIZZLED)
    plain = O.nvfp4_quantize(x, gs[4], O.SWIZZLED)
    np.testing.assert_array_equal(one[0], plain[0])
    np.testing.assert_array_equal(one[1], plain[1])


def test_weight_generator_row_ranges_match_the_whole():
    full = W.weight_rotate_quant(5000, 64)
    for r0, r1 in ((0, 1), (2047, 2049), (4095, 5000), (100, 4200)):
        np.testing.assert_array_equal(W.weight_rotate_quant(5000, 64, r0, r1), full[r0:r1])
    v = W.bf16_bits_to_float(full)
    assert abs(v.std() - 0.02) < 0.001 and abs(v.mean()) < 0.001


def test_workload_recipes():
    x = W.mxfp8_linear_quant(128, 4096)
    assert x.shape == (128, 4096) and x.dtype == np.uint16
    f = W.bf16_bits_to_float(x)
    for r in range(128):
        j = (37 * r) % 128
        assert (f[r, 32 * j:32 * j + 32] == 0).all()
    assert 0.005 < (np.abs(f) > 6).mean() < 0.02
    counts = W.moe_counts()
    assert counts.sum() == 16384 and counts.size == 128 and counts.max() > 1000
    np.testing.assert_array_equal(W.mxfp8_linear_quant(4, 64), W.mxfp8_linear_quant(4, 64))


@pytest.mark.parametrize("g", [16, 32, 128])
def test_rotation_orientation_with_non_symmetric_matrix(g):
    """y_chunk = x_chunk @ H (row vector times matrix), checked with a random, non-symmetric H
    against numpy's matmul; the transposed product must differ."""
    rng = np.random.default_rng(g)
    H = W.to_bf16_bits(rng.standard_normal((g, g)) / np.sqrt(g))
    x = W.rotate_quant_activation(5, 2 * g)
    y = O.rotate(x, H)
    xd = W.bf16_bits_to_float(x).astype(np.float64).reshape(5, 2, g)
    hd = W.bf16_bits_to_float(H).astype(np.float64)
    np.testing.assert_allclose(y, (xd @ hd).reshape(5, 2 * g), rtol=0, atol=1e-12)
    assert np.abs(y - (xd @ hd.T).reshape(5, 2 * g)).max() > 1e-3



# ---------------------------------------------------------------------------------------------
# block-scaled GEMM of stored MX data: dequantize, then matmul
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", [O.E2M1, O.E4M3])
def test_gemm_of_unit_codes_is_k_times_alpha(fmt):
    """Every code 1.0 (E2M1 nibble 0x2, E4M3 byte 0x38) under scale byte 127 (2^0): each
    entry of C is alpha * K; under scale bytes 129 (A) and 126 (B) it is alpha * K * 2."""
    M, N, K = 3, 5, 128
    byte = 0x22 if fmt == O.E2M1 else 0x38
    cols = O.code_bytes_per_row(fmt, K)
    a = np.full((M, cols), byte, dtype=np.uint8)
    b = np.full((N, cols), byte, dtype=np.uint8)
    sa = np.full((M, K // 32), 127, dtype=np.uint8)
    sb = np.full((N, K // 32), 127, dtype=np.uint8)
    np.testing.assert_array_equal(O.gemm(a, sa, b, sb, K, fmt, O.LINEAR, alpha=0.5),
                                  np.full((M, N), 0.5 * K))
    sa[:] = 129
    sb[:] = 126
    np.testing.assert_array_equal(O.gemm(a, sa, b, sb, K, fmt, O.LINEAR), np.full((M, N), 2.0 * K))


@pytest.mark.parametrize("layout", [O.LINEAR, O.SWIZZLED])
@pytest.mark.parametrize("fmt", [O.E2M1, O.E4M3])
def test_gemm_matches_a_brute_force_sum(fmt, layout):
    """Random codes and scale bytes: each entry equals alpha * sum_k of the products of the
    element-by-element dequantized values (oracle scalar dequant), summed in Python."""
    rng = np.random.default_rng(fmt * 10 + layout)
    M, N, K = 3, 4, 64
    cols = O.code_bytes_per_row(fmt, K)
    a = rng.integers(0, 256, (M, cols), dtype=np.uint8)
    b = rng.integers(0, 256, (N, cols), dtype=np.uint8)
    if fmt == O.E4M3:  # no NaN codes
        a[(a & 0x7F) == 0x7F] ^= 0x01
        b[(b & 0x7F) == 0x7F] ^= 0x01
    la = rng.integers(120, 135, (M, K // 32), dtype=np.uint8)
    lb = rng.integers(120, 135, (N, K // 32), dtype=np.uint8)

    def stored(lin, rows):
        if layout == O.LINEAR:
            return lin
        sw = np.zeros(O.scales_shape(rows, K, O.SWIZZLED), dtype=np.uint8).reshape(-1)
        cp = O.scales_shape(rows, K, O.SWIZZLED)[1]
        for r in range(rows):
            for j in range(K // 32):
                sw[O.swizzled_offset(r, j, cp)] = lin[r, j]
        return sw.reshape(O.scales_shape(rows, K, O.SWIZZLED))

    def value(codes, lin, r, k):
        if fmt == O.E4M3:
            code = int(codes[r, k])
        else:
            byte = int(codes[r, k // 2])
            code = byte & 0xF if k % 2 == 0 else byte >> 4
        return O.bf16_to_double(O.dequant_bf16(fmt, code, int(lin[r, k // 32])))

    C = O.gemm(a, stored(la, M), b, stored(lb, N), K, fmt, layout, alpha=1.5)
    for i in range(M):
        for j in range(N):
            want = 1.5 * sum(value(a, la, i, k) * value(b, lb, j, k) for k in range(K))
            assert C[i, j] == pytest.approx(want, rel=1e-15, abs=1e-300)


# ---------------------------------------------------------------------------------------------
# Quest-like MXFP4 scale (clip point alpha * RMS in place of the abs-max)
# ---------------------------------------------------------------------------------------------
E2M1_GRID = (0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0)  # the format's magnitudes (1 sign, E2M1)


def gaussian_grid_mse(alpha: float) -> float:
    """E[(Z - q(Z))^2] for Z ~ N(0, 1) and q the E2M1 grid stretched so that 6 sits at alpha
    (nearest grid point, saturating), integrated piecewise between the decision points."""
    from scipy import integrate, stats
    t = alpha / 6.0
    mids = [(a + b) / 2 for a, b in zip(E2M1_GRID, E2M1_GRID[1:])]
    edges = [0.0] + [t * m for m in mids] + [math.inf]
    total = 0.0
    for k, level in enumerate(E2M1_GRID):
        f = lambda z, q=level * t: (z - q) ** 2 * stats.norm.pdf(z)
        total += integrate.quad(f, edges[k], edges[k + 1], epsabs=1e-14, epsrel=1e-13)[0]
    return 2.0 * total


def test_quest_alpha_minimises_gaussian_mse_of_e2m1_grid():
    """The oracle's clip ratio is the minimiser of the grid's mean squared error on a standard
    normal variable (the Gaussian clipping of the QuEST method), found here by quadrature."""
    from scipy import optimize
    res = optimize.minimize_scalar(gaussian_grid_mse, bounds=(1.0, 6.0), method="bounded",
                                   options={"xatol": 1e-10})
    alpha = O.quest_alpha()
    assert abs(alpha - res.x) < 2e-6
    best = gaussian_grid_mse(alpha)
    assert best <= res.fun * (1 + 1e-9)
    for d in (-0.05, -0.01, 0.01, 0.05):  # a minimum, not a flat stretch
        assert gaussian_grid_mse(alpha + d) > best


def _read_quest_blocks():
    blocks = []
    for line in open(os.path.join(GOLDEN, "quest_worked_blocks.txt")):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split()
        if parts[0] == "block":
            blocks.append((parts[1], int(parts[2]), []))
        else:
            blocks[-1][2].append((int(parts[0]), float(parts[1]), int(parts[2], 16)))
    return blocks


@pytest.mark.parametrize("case", _read_quest_blocks(), ids=lambda c: c[0])
def test_quest_worked_blocks(case):
    name, byte, entries = case
    v = np.zeros(32)
    want = np.zeros(32, dtype=np.uint8)
    i = 0
    for count, val, code in entries:
        v[i:i + count] = val
        want[i:i + count] = code
        i += count
    assert (W.bf16_bits_to_float(bf16(v)) == v.astype(np.float32)).all(), name
    got_byte, got = O.quest_quantize_block(v)
    assert got_byte == byte, name
    np.testing.assert_array_equal(got, want, err_msg=name)
    assert O.quest_scale_byte(v) == byte
    codes, scales = O.quest_quantize(bf16(v).reshape(1, 32), O.LINEAR)
    assert scales[0, 0] == byte
    np.testing.assert_array_equal(codes[0] & 0xF, want[0::2])
    np.testing.assert_array_equal(codes[0] >> 4, want[1::2])


def _quest_byte_exact(v) -> int:
    """Scale byte by exact rational arithmetic: k = floor(log2 c) is the k with
    4^k <= c^2 < 4^(k+1), c^2 = alpha^2 * sum(v^2) / 32, alpha taken as the decimal 2.922475."""
    from fractions import Fraction
    alpha = Fraction(2922475, 10 ** 6)
    c2 = alpha * alpha * sum(Fraction(float(x)) ** 2 for x in v) / 32
    if c2 == 0:
        return 0
    k = (c2.numerator.bit_length() - c2.denominator.bit_length()) // 2 - 2
    while Fraction(4) ** (k + 1) <= c2:
        k += 1
    while Fraction(4) ** k > c2:
        k -= 1
    return min(max(k - 2, -127), 127) + 127


def test_quest_scale_byte_matches_exact_arithmetic():
    rng = np.random.default_rng(11)
    blocks = []
    for e in (-140, -126, -60, -3, 0, 5, 60, 120, 126):  # spread over the whole exponent range
        blocks.append(rng.standard_normal(32) * 2.0 ** e)
        blocks.append(rng.uniform(-1, 1, 32) * 2.0 ** e)
    for e in range(-130, 128, 7):  # blocks whose c sits next to a power of two, every binade
        blocks.append(np.full(32, 1.375 * 2.0 ** e))
        blocks.append(np.full(32, 1.3671875 * 2.0 ** e))
    for _ in range(300):
        blocks.append(rng.standard_normal(32) * 2.0 ** rng.integers(-20, 20))
    for v in blocks:
        v = W.bf16_bits_to_float(bf16(v)).astype(np.float64)  # bf16 inputs, as on the path
        assert O.quest_scale_byte(v) == _quest_byte_exact(v), v


def test_quest_scale_invariants():
    """Power-of-two equivariance, sign symmetry, and the bounds RMS in [amax/sqrt(32), amax]
    give against the abs-max byte: floor(log2 c) - floor(log2 amax) in [-1, 2]."""
    rng = np.random.default_rng(12)
    cases = [rng.standard_normal(32) for _ in range(200)]
    cases += [np.eye(32)[i] * rng.uniform(1, 2) for i in range(32)]       # one-hot (RMS low)
    cases += [np.full(32, rng.uniform(1, 2)) * rng.choice([-1, 1], 32) for _ in range(32)]
    for v in cases:
        v = W.bf16_bits_to_float(bf16(v)).astype(np.float64)
        b, codes = O.quest_quantize_block(v)
        b_abs = O.scale_byte(O.E2M1, float(np.abs(v).max()))
        assert -1 <= b - b_abs <= 2
        for k in (-40, -1, 3, 50):
            b2, codes2 = O.quest_quantize_block(v * 2.0 ** k)
            assert b2 == b + k
            np.testing.assert_array_equal(codes2, codes)
        bn, codesn = O.quest_quantize_block(-v)
        assert bn == b
        np.testing.assert_array_equal(codesn ^ 8, codes)
    nan_block = np.ones(32)
    nan_block[5] = np.nan
    assert O.quest_quantize_block(nan_block)[0] == 0xFF
    inf_block = np.ones(32)
    inf_block[7] = -np.inf
    b, codes = O.quest_quantize_block(inf_block)
    assert b == 0xFF and not codes.any()


def test_quest_gaussian_qdq_error_reaches_the_optimum():
    """On normal data the Quest-like scale's QDQ error is within 1.5% of the continuous
    optimum (the grid's Gaussian MSE at alpha) and below the abs-max scale's."""
    rng = np.random.default_rng(13)
    v = rng.standard_normal((2000, 320))
    qd = W.bf16_bits_to_float(O.quest_qdq_values(v)).astype(np.float64)
    qa = W.bf16_bits_to_float(O.qdq_values(v, O.E2M1)).astype(np.float64)
    mse_q = float(((qd - v) ** 2).mean())
    mse_a = float(((qa - v) ** 2).mean())
    optimum = gaussian_grid_mse(O.quest_alpha())
    assert abs(mse_q / optimum - 1) < 0.015
    assert mse_q < 0.98 * mse_a


def test_quest_tensor_entry_points_assemble_the_blocks():
    """Tensor calls (linear / swizzled scales, QDQ, rotated input) against block-by-block calls
    and the dequantize definition."""
    rng = np.random.default_rng(14)
    M, K = 130, 192
    x = bf16(rng.standard_normal((M, K)) * np.exp(rng.uniform(-3, 3, (M, 1))))
    v = W.bf16_bits_to_float(x).astype(np.float64)
    codes_l, scales_l = O.quest_quantize(x, O.LINEAR)
    codes_s, scales_s = O.quest_quantize(x, O.SWIZZLED)
    np.testing.assert_array_equal(codes_l, codes_s)
    rows, cols = O.scales_shape(M, K, O.SWIZZLED)
    for r in range(M):
        for j in range(K // 32):
            b, c = O.quest_quantize_block(v[r, 32 * j:32 * j + 32])
            assert scales_l[r, j] == b
            assert scales_s.reshape(-1)[O.swizzled_offset(r, j, cols)] == b
            packed = codes_l[r, 16 * j:16 * j + 16]
            np.testing.assert_array_equal(packed & 0xF, c[0::2])
            np.testing.assert_array_equal(packed >> 4, c[1::2])
    np.testing.assert_array_equal(O.quest_qdq(x), O.dequantize(codes_l, scales_l, K, O.E2M1,
                                                                O.LINEAR))
    g = 32
    h = np.array([[1.0]])
    while h.shape[0] < g:
        h = np.block([[h, h], [h, -h]])
    H = bf16(h / math.sqrt(g))
    y = O.rotate(x, H)
    np.testing.assert_array_equal(O.quest_quantize(x, O.SWIZZLED, H)[1],
                                  O.quest_quantize_values(y, O.SWIZZLED)[1])
    np.testing.assert_array_equal(O.quest_qdq(x, H), O.quest_qdq_values(y))
