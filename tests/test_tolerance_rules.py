"""CPU checks of the rotated-path tolerance rules in mx_testlib: they accept the oracle's own
results and the exemptions the rules allow, and reject codes or scales that are wrong."""

import numpy as np
import pytest

import oracle as O
from mx_microscaling_quantize_gb300 import workloads as W
import mx_testlib as T


def identity(g):
    return W.to_bf16_bits(np.eye(g))


@pytest.mark.parametrize("fmt", [O.E2M1, O.E4M3])
def test_rules_accept_oracle_results(fmt):
    x = W.rotate_quant_activation(4, 256)
    H = W.normalized_hadamard_bf16(32)
    c, s = O.rotate_quantize(x, H, fmt, O.LINEAR)
    stats = T.check_rotated_codes(x, H, fmt, c, s)
    assert stats["exempt_blocks"] == 0
    assert T.check_rotated_qdq(x, H, fmt, O.rotate_qdq(x, H, fmt))["exempt_blocks"] == 0


def test_rules_reject_a_wrong_code_away_from_midpoints():
    x = W.rotate_quant_activation(4, 256)
    H = W.normalized_hadamard_bf16(32)
    c, s = O.rotate_quantize(x, H, O.E2M1, O.LINEAR)
    y = O.rotate(x, H)
    # pick an element whose scaled value is far from every midpoint and bump its code
    t = y[0, :32] / 2.0 ** (int(s[0, 0]) - 127)
    i = int(np.argmin(np.abs(np.abs(t) - 1.0)))  # |t| close to a grid point (1.0)
    bad = c.copy()
    nib = (bad[0, i // 2] >> (4 * (i % 2))) & 0xF
    new = (nib & 0x8) | min((nib & 7) + 1, 7)
    bad[0, i // 2] = (bad[0, i // 2] & (0xF0 if i % 2 == 0 else 0x0F)) | (new << (4 * (i % 2)))
    with pytest.raises(AssertionError):
        T.check_rotated_codes(x, H, O.E2M1, bad, s)
    bad_s = s.copy()
    bad_s[1, 3] += 1
    with pytest.raises(AssertionError):
        T.check_rotated_codes(x, H, O.E2M1, c, bad_s)
    out = O.rotate_qdq(x, H, O.E2M1)
    out[2, 40] ^= 0x0040
    with pytest.raises(AssertionError):
        T.check_rotated_qdq(x, H, O.E2M1, out)


def test_rules_allow_midpoint_and_power_of_two_exemptions():
    g = 32
    v = np.zeros((1, 32))
    v[0, 0] = 4.0     # amax exactly 2^2: E2M1 byte 127, a flip to 126 is allowed
    v[0, 1] = 0.75    # exact midpoint of 0.5 and 1.0 at scale 1
    x = W.to_bf16_bits(v)
    H = identity(g)
    c, s = O.rotate_quantize(x, H, O.E2M1, O.LINEAR)
    alt = c.copy()
    alt[0, 0] = (alt[0, 0] & 0x0F) | (0x1 << 4)  # element 1 -> 0.5 instead of 1.0
    stats = T.check_rotated_codes(x, H, O.E2M1, alt, s)
    assert stats["exempt_codes"] == 1
    b, codes = O.quantize_block(O.E2M1, v[0], forced_byte=126)
    packed = (codes[0::2] | (codes[1::2] << 4)).reshape(1, 16)
    stats = T.check_rotated_codes(x, H, O.E2M1, packed, np.array([[126]], dtype=np.uint8))
    assert stats["scale_flips"] == 1


def test_unswizzle_inverts_oracle_layout():
    x = W.mxfp8_linear_quant(200, 416)
    _, lin = O.quantize(x, O.E4M3, O.LINEAR)
    _, swz = O.quantize(x, O.E4M3, O.SWIZZLED)
    np.testing.assert_array_equal(T.unswizzle(swz, 200, 416), lin)
    assert not T.swizzle_pads(swz, 200, 416).any()


def test_converter_sweep_covers_every_scale():
    xs = T.converter_sweep()
    _, s2 = O.quantize(xs[:400], O.E2M1, O.LINEAR)
    assert xs.shape[1] == 2048 and xs.shape[0] > 4000
    fin = T.finite_bf16()
    assert np.isin(fin, xs).all()


def nvfp4_gs(x_bits) -> np.float32:
    return np.float32(448 * 6) / np.float32(np.abs(W.bf16_bits_to_float(x_bits)).max())


def test_nvfp4_rules_accept_oracle_and_reject_planted_errors():
    x = W.rotate_quant_activation(4, 256)
    H = W.normalized_hadamard_bf16(32)
    gs = nvfp4_gs(x)
    c, s = O.nvfp4_quantize(x, gs, O.LINEAR, H_bits=H)
    assert T.check_rotated_nvfp4(x, H, gs, c, s)["exempt_blocks"] == 0
    assert T.check_rotated_nvfp4_qdq(x, H, gs, O.nvfp4_qdq(x, gs, H_bits=H))["exempt_blocks"] == 0
    # a code two grid steps away
    bad = c.copy()
    nib = bad[1, 3] & 0xF
    bad[1, 3] = (bad[1, 3] & 0xF0) | ((nib & 0x8) | ((nib & 7) + 2 if (nib & 7) < 6 else 0))
    with pytest.raises(AssertionError):
        T.check_rotated_nvfp4(x, H, gs, bad, s)
    # a scale byte far from the rounding of s_f
    bad_s = s.copy()
    bad_s[2, 5] = min(int(bad_s[2, 5]) + 3, 0x7E)
    with pytest.raises(AssertionError):
        T.check_rotated_nvfp4(x, H, gs, c, bad_s)
    # a QDQ output that no allowed code gives
    q = O.nvfp4_qdq(x, gs, H_bits=H)
    q[3, 17] ^= 0x0040
    with pytest.raises(AssertionError):
        T.check_rotated_nvfp4_qdq(x, H, gs, q)


def test_nvfp4_scale_candidates_bracket_the_rounding():
    gs = np.float32(6.0)  # r6 = 1: s_f = amax
    assert T.nvfp4_scale_candidates(1.0, 0.0, gs) == {0x38}          # 1.0 exactly
    # 1.0625 is the midpoint of 1.0 (0x38) and 1.125 (0x39): a tolerance around it allows both
    assert T.nvfp4_scale_candidates(1.0625, 1e-6, gs) == {0x38, 0x39}
    assert T.nvfp4_scale_candidates(1.03, 1e-6, gs) == {0x38}


def _packed_e2m1(codes):
    return (codes[0::2] | (codes[1::2] << 4)).reshape(1, -1).astype(np.uint8)


def test_scale_flip_only_toward_the_nearby_power_of_two():
    """A block's abs-max within tolerance of 2^k (the bottom of its binade) lets the GPU's
    scale byte be one lower, never one higher; within tolerance of 2^(k+1) (the top), one
    higher, never one lower. Planted flips in the wrong direction are rejected even though the
    codes are exactly what the oracle gives under the planted byte."""
    g = 32
    # bottom of the binade: amax = 4.0 exactly (E2M1 byte 127)
    v = np.zeros((1, 32))
    v[0, 0], v[0, 1] = 4.0, 0.75
    x = W.to_bf16_bits(v)
    H = identity(g)
    _, s = O.rotate_quantize(x, H, O.E2M1, O.LINEAR)
    assert int(s[0, 0]) == 127
    for byte, ok in ((126, True), (128, False)):
        _, codes = O.quantize_block(O.E2M1, v[0], forced_byte=byte)
        sb = np.array([[byte]], dtype=np.uint8)
        if ok:
            assert T.check_rotated_codes(x, H, O.E2M1, _packed_e2m1(codes), sb)["scale_flips"] == 1
        else:
            with pytest.raises(AssertionError):
                T.check_rotated_codes(x, H, O.E2M1, _packed_e2m1(codes), sb)
    # top of the binade: every element 7.9375 * (1 + 2^-7) = 7.99951..., 4.9e-4 below 8; with
    # g = 128 the chunk norm is about 90.5 (tolerance 9.05e-4); H = (1 + 2^-7) I is exact in
    # bf16. The flip is planted in the first of the row's four blocks.
    g = 128
    v = np.full((1, 128), 7.9375)
    x = W.to_bf16_bits(v)
    H = W.to_bf16_bits(np.eye(g) * (1.0 + 2.0 ** -7))
    y = O.rotate(x, H)
    assert 0 < 8.0 - y.max() < 1e-5 * np.linalg.norm(y)
    c, s = O.rotate_quantize(x, H, O.E2M1, O.LINEAR)
    assert (s == 127).all()
    for byte, ok in ((128, True), (126, False)):
        _, codes = O.quantize_block(O.E2M1, y[0, :32], forced_byte=byte)
        cb, sb = c.copy(), s.copy()
        cb[0, :16] = _packed_e2m1(codes)[0]
        sb[0, 0] = byte
        if ok:
            assert T.check_rotated_codes(x, H, O.E2M1, cb, sb)["scale_flips"] == 1
        else:
            with pytest.raises(AssertionError):
                T.check_rotated_codes(x, H, O.E2M1, cb, sb)
    # QDQ outputs follow the same rule: that block dequantized under byte 126 is rejected,
    # under 128 accepted
    for byte, ok in ((128, True), (126, False)):
        _, codes = O.quantize_block(O.E2M1, y[0, :32], forced_byte=byte)
        out = O.rotate_qdq(x, H, O.E2M1)
        out[0, :32] = [O.dequant_bf16(O.E2M1, int(cd), byte) for cd in codes]
        if ok:
            assert T.check_rotated_qdq(x, H, O.E2M1, out)["exempt_blocks"] == 1
        else:
            with pytest.raises(AssertionError):
                T.check_rotated_qdq(x, H, O.E2M1, out)


def test_chunked_checks_cover_every_row():
    """The whole-output checks split rows over a thread pool: a planted error in the last row
    of a many-row input is still found, and per-chunk counts add up to the whole."""
    x = W.rotate_quant_activation(97, 256, stream=5)
    H = W.normalized_hadamard_bf16(32)
    c, s = O.rotate_quantize(x, H, O.E4M3, O.LINEAR)
    stats = T.check_rotated_codes(x, H, O.E4M3, c, s)
    assert stats["blocks"] == 97 * 256 // 32 and stats["exempt_blocks"] == 0
    bad = c.copy()
    bad[96, 200] ^= 0x03
    with pytest.raises(AssertionError, match="row 96"):
        T.check_rotated_codes(x, H, O.E4M3, bad, s)
    q = O.qdq(x, O.E2M1)
    T.assert_rows_equal(q, T.oracle_qdq_rows(x, O.E2M1))
    q[96, 255] ^= 1
    with pytest.raises(AssertionError, match="rows"):
        T.assert_rows_equal(q, T.oracle_qdq_rows(x, O.E2M1))


# ---------------------------------------------------------------------------------------------
# Quest-like scale checker
# ---------------------------------------------------------------------------------------------
def _packed(codes):
    return (codes[0::2] | (codes[1::2] << 4)).astype(np.uint8)


@pytest.mark.parametrize("rotated", [False, True])
def test_quest_rules_accept_oracle_and_reject_planted_errors(rotated):
    x = W.rotate_quant_activation(6, 256)
    H = W.normalized_hadamard_bf16(32) if rotated else None
    c, s = O.quest_quantize(x, O.LINEAR, H)
    q = O.quest_qdq(x, H)
    stats = T.check_quest(x, H, codes=(c, s), qdq=q)
    assert stats["codes"]["exempt_blocks"] == 0 and stats["qdq"]["exempt_blocks"] == 0
    assert stats["codes"]["blocks"] == 6 * 8
    bad_s = s.copy()
    bad_s[2, 5] += 1
    with pytest.raises(AssertionError):
        T.check_quest(x, H, codes=(c, bad_s))
    bad_c = c.copy()
    bad_c[4, 9] ^= 0x22  # two codes two grid steps off: never a midpoint exemption
    with pytest.raises(AssertionError):
        T.check_quest(x, H, codes=(bad_c, s))
    bad_q = q.copy()
    bad_q[1, 77] ^= 0x0080
    with pytest.raises(AssertionError):
        T.check_quest(x, H, qdq=bad_q)


def test_quest_scale_flip_only_toward_the_nearby_power_of_two():
    """A block with c = 3.99995 (1.2e-5 below 4): under a rotation (tolerance about 6e-5 of c
    here) the byte may step up to 127 but never down to 125; without a rotation (exact inputs,
    only the kernel's fp32 sum can move it) it must stay 126."""
    v = np.full(32, 1.375)
    v[0] = 1.15625
    x = W.to_bf16_bits(v.reshape(1, 32))
    assert abs(T.quest_clip(v) / 4 - 1) < 2e-5 and T.quest_clip(v) < 4
    ref_byte, _ = O.quest_quantize_block(v)
    assert ref_byte == 126
    H = identity(32)
    for b, ok_rot in ((127, True), (125, False)):
        _, codes = O.quantize_block(O.E2M1, v, forced_byte=b)
        got = (_packed(codes).reshape(1, 16), np.array([[b]], dtype=np.uint8))
        if ok_rot:
            assert T.check_quest(x, H, codes=got)["codes"]["scale_flips"] == 1
        else:
            with pytest.raises(AssertionError):
                T.check_quest(x, H, codes=got)
        with pytest.raises(AssertionError):
            T.check_quest(x, None, codes=got)
