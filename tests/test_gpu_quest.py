"""GPU parity of the Quest-like MXFP4 scale (rounding = QUEST: the E8M0 scale from the clip point
alpha * RMS of the block instead of its abs-max) against the CPU oracle, through the C ABI.

Plain calls (no rotation) quantize exact bf16 inputs: codes, scale bytes and QDQ outputs equal
the oracle's bit for bit except where the oracle's clip point lies within 2^-20 of a power of two
(the kernel sums the squares in fp32), where the byte may step toward that power and the codes
follow it. Rotated calls (tensor-core, FMA and Walsh-Hadamard kernels) follow the rotated-path
rules of mx_testlib with the Quest-like threshold (mx_testlib.check_quest).
"""

import numpy as np
import pytest
import torch

import __graft_entry__
import mx_microscaling_quantize_gb300 as mxq
import oracle as O
from mx_microscaling_quantize_gb300 import workloads as W
import mx_testlib as T

pytestmark = pytest.mark.gpu
LAYOUTS = [O.LINEAR, O.SWIZZLED]
Q = mxq.QUEST


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()
    yield
    assert mxq.mx_device_errors() == 0


def quest_outputs(xb, H=None, rot_kind=mxq.ROT_DENSE):
    """GPU codes (linear and swizzled scales; the codes of both calls must agree) and QDQ."""
    x = T.to_gpu(xb)
    Hd = None if H is None else T.to_gpu(H)
    M, K = xb.shape
    out = {}
    for layout in LAYOUTS:
        if Hd is None:
            c, s = mxq.mx_quantize(x, mxq.E2M1, layout, rounding=Q)
        else:
            c, s = mxq.mx_rotate_quantize(x, Hd, mxq.E2M1, layout, rounding=Q, rot_kind=rot_kind)
        out[layout] = (T.u8(c), T.u8(s))
    c_lin, s_lin = out[O.LINEAR]
    c_swz, s_swz = out[O.SWIZZLED]
    np.testing.assert_array_equal(c_swz, c_lin)
    assert not T.swizzle_pads(s_swz, M, K).any()
    np.testing.assert_array_equal(T.unswizzle(s_swz, M, K), s_lin)
    q = T.bf16_bits(mxq.mx_qdq(x, mxq.E2M1, Hd, rounding=Q, rot_kind=rot_kind))
    return c_lin, s_lin, q


def range_rows(K):
    """Constant blocks on both sides of the kernels' plain-sum range [2^-80, 2^100] (outside it
    the squares are summed again after a power-of-two scaling), tiny and huge random rows (the
    scaled sum throughout)."""
    rng = np.random.default_rng(K)
    rows = np.zeros((6, K))
    for i, e in enumerate((-42, -44, 46, 48)):  # sums 2^-78.1, 2^-82.1, 2^97.9, 2^101.9
        rows[i] = 1.375 * 2.0 ** e
    rows[4] = rng.standard_normal(K) * 2.0 ** -60
    rows[5] = rng.standard_normal(K) * 2.0 ** 100
    return W.to_bf16_bits(rows)


def special_rows(K):
    """Rows that reach the edges of the rule: all zero, subnormal-only (scale clamped at byte
    0), near the bf16 maximum (byte 254 and its subnormal inverse scale), a NaN and an infinity
    in one block each, one-hot blocks (c below the abs-max) and constant blocks (c above it),
    and range_rows."""
    return np.concatenate([_special_rows(K), range_rows(K)])


def _special_rows(K):
    rows = np.zeros((8, K))
    rows[1] = 2.0 ** -131 * (np.arange(K) % 7)
    rows[2] = 1.5 * 2.0 ** 127 * np.where(np.arange(K) % 3 == 0, -1.0, 1.0)
    rows[3] = np.linspace(-3, 3, K)
    rows[3, 5] = np.nan
    rows[4] = np.linspace(-1, 1, K)
    rows[4, K - 3] = np.inf
    rows[5, ::32] = 1.75
    rows[6] = 1.375
    rows[7, ::2] = -1.3671875
    return W.to_bf16_bits(rows)


@pytest.mark.parametrize("M,K", [(1, 32), (7, 96), (129, 416), (300, 1024), (1000, 8192)])
def test_quest_plain_matches_oracle(M, K):
    xb = np.concatenate([W.mxfp4_qdq_activation(M, K, stream=M + K), special_rows(K)])
    c, s, q = quest_outputs(xb)
    stats = T.check_quest(xb, None, codes=(c, s), qdq=q)
    assert stats["codes"]["exempt_blocks"] <= stats["codes"]["scale_flips"], stats
    assert stats["codes"]["scale_flips"] <= 2, stats
    # the special rows exactly
    r0 = M
    rc, rs = O.quest_quantize(xb[r0:], O.LINEAR)
    np.testing.assert_array_equal(s[r0:], rs)
    np.testing.assert_array_equal(c[r0:], rc)
    np.testing.assert_array_equal(q[r0:], O.quest_qdq(xb[r0:]))
    assert (rs[2] == 254).all() and (rs[1] == 0).all()
    assert rs[3, 0] == 255 and rs[4, (K - 3) // 32] == 255


def test_quest_dequantize_equals_qdq():
    """dequantize(quantize(x)) == QDQ(x) under the Quest-like scale, plain and rotated."""
    xb = W.rotate_quant_activation(300, 2048)
    H = T.to_gpu(W.normalized_hadamard_bf16(32))
    x = T.to_gpu(xb)
    for Hd in (None, H):
        for layout in LAYOUTS:
            if Hd is None:
                c, s = mxq.mx_quantize(x, mxq.E2M1, layout, rounding=Q)
            else:
                c, s = mxq.mx_rotate_quantize(x, Hd, mxq.E2M1, layout, rounding=Q)
            y = mxq.mx_dequantize(c, s, 2048, mxq.E2M1, layout)
            torch.testing.assert_close(y.view(torch.int16),
                                       mxq.mx_qdq(x, mxq.E2M1, Hd, rounding=Q).view(torch.int16),
                                       rtol=0, atol=0)


@pytest.mark.parametrize("kind", ["dense", "hadamard"])
@pytest.mark.parametrize("g", [16, 32, 64, 128])
@pytest.mark.parametrize("M,K", [(1, 384), (16, 1024), (129, 640), (300, 2048)])
def test_quest_rotated_rules(M, K, g, kind):
    """Tensor-core (M > 16) and FMA (M <= 16, M * g <= 512) kernels under ROT_DENSE; the
    Walsh-Hadamard kernel under ROT_HADAMARD for g <= 64 (g = 128 runs on the tensor cores)."""
    xb = np.concatenate([W.rotate_quant_activation(M, K, stream=7 * M + g), range_rows(K)[4:]])
    H = W.normalized_hadamard_bf16(g)
    rk = mxq.ROT_HADAMARD if kind == "hadamard" else mxq.ROT_DENSE
    c, s, q = quest_outputs(xb, H, rk)
    stats = T.check_quest(xb, H, codes=(c, s), qdq=q)
    assert stats["codes"]["exempt_blocks"] <= 0.01 * stats["codes"]["blocks"] + 2, stats
    assert stats["qdq"]["exempt_blocks"] <= 0.01 * stats["qdq"]["blocks"] + 2, stats


@pytest.mark.parametrize("g", [16, 32, 64, 128])
def test_quest_identity_rotation(g):
    """x * I is exact in fp32. The tensor-core kernel (M > 16) and the Walsh-Hadamard kernel's
    dense fallback add a block's squares in the plain kernel's order, so they equal the plain
    Quest-like path bit for bit; the FMA kernel (M <= 16) adds them in another order, so it
    meets the plain-path rule (scale steps only where c is within 2^-20 of a power of two)."""
    I = W.to_bf16_bits(np.eye(g))
    for M in (3, 200):
        xb = np.concatenate([W.mxfp4_qdq_activation(M, 512, stream=g + M), range_rows(512)])
        M = xb.shape[0]
        plain = quest_outputs(xb)
        for rk in (mxq.ROT_DENSE, mxq.ROT_HADAMARD):
            c, s, q = quest_outputs(xb, I, rk)
            fma_kernel = M <= 16 and M * g <= 512 and not (rk == mxq.ROT_HADAMARD and g <= 64)
            if not fma_kernel:
                for a, b in zip(plain, (c, s, q)):
                    np.testing.assert_array_equal(a, b)
            else:
                stats = T.check_quest(xb, None, codes=(c, s), qdq=q)
                assert stats["codes"]["exempt_blocks"] <= stats["codes"]["scale_flips"] <= 1


def test_quest_full_size_rotate_quantize_and_qdq():
    """The rotate + quantize workload at its full size, x[8192, 8192] with g = 32, whole
    outputs; and the plain Quest-like QDQ of the MXFP4 weight x[8192, 8192]."""
    xb = W.rotate_quant_activation(8192, 8192)
    H = W.normalized_hadamard_bf16(32)
    c, s, q = quest_outputs(xb, H)
    stats = T.check_quest(xb, H, codes=(c, s), qdq=q)
    assert stats["codes"]["exempt_blocks"] <= 0.01 * stats["codes"]["blocks"], stats
    wb = W.mxfp4_qdq_weight()
    q = T.bf16_bits(mxq.mx_qdq(T.to_gpu(wb), mxq.E2M1, rounding=Q))
    stats = T.check_quest(wb, None, qdq=q)
    assert stats["qdq"]["exempt_blocks"] <= 4, stats


@pytest.mark.parametrize("rot_kind", [mxq.ROT_DENSE, mxq.ROT_HADAMARD])
def test_quest_full_size_wide_rows(rot_kind):
    """Quest-like rotate + quantize of x[8192, 28672] (g = 32), the size the benchmark times,
    whole outputs, on the tensor-core and the Walsh-Hadamard kernels."""
    xb = W.rotate_quant_activation(8192, 28672)
    H = W.normalized_hadamard_bf16(32)
    x, Hd = T.to_gpu(xb), T.to_gpu(H)
    c, s = mxq.mx_rotate_quantize(x, Hd, mxq.E2M1, mxq.LINEAR, rounding=Q, rot_kind=rot_kind)
    stats = T.check_quest(xb, H, codes=(T.u8(c), T.u8(s)))
    assert stats["codes"]["exempt_blocks"] <= 0.01 * stats["codes"]["blocks"], stats


def test_quest_rejected_where_unsupported():
    x = torch.zeros(128, 256, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(mxq.MXError):
        mxq.mx_quantize(x, mxq.E4M3, rounding=Q)
    off = torch.tensor([0, 64, 128], dtype=torch.int64, device="cuda")
    with pytest.raises(mxq.MXError):
        mxq.mx_quantize_grouped(x, off, mxq.E2M1, rounding=Q)
