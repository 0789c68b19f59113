"""Past 2^31 elements: x[65600, 32768] (2,149,580,800 bf16, 4.3 GB) built on the device by
repeating a seeded 64-row block, so that the expected result of row r is the oracle's result for
row r % 64 of the block. Rows on both sides of the 2^31-element boundary (row 65536) are checked:
every index the kernels form past it must be 64-bit."""

import numpy as np
import pytest
import torch

import __graft_entry__
import mx_microscaling_quantize_gb300 as mxq
import oracle as O
from mx_microscaling_quantize_gb300 import workloads as W
import mx_testlib as T

pytestmark = pytest.mark.gpu
M, K, B = 65600, 32768, 64
ROWS = np.array([0, 1, 63, 4097, 65535, 65536, 65537, 65599])


@pytest.fixture(scope="module")
def big():
    __graft_entry__.build()
    assert M * K > 2 ** 31
    base = W.mxfp4_qdq_activation(B, K)
    x = T.to_gpu(base).repeat(M // B + 1, 1)[:M].contiguous()
    yield base, x
    del x
    torch.cuda.empty_cache()
    assert mxq.mx_device_errors() == 0


def rows_of(t):
    return t[torch.from_numpy(ROWS).cuda()]


def test_qdq_and_dequantize_past_2pow31(big):
    base, x = big
    y = mxq.mx_qdq(x, mxq.E2M1)
    want = O.qdq(base[ROWS % B], O.E2M1)
    np.testing.assert_array_equal(T.bf16_bits(rows_of(y)), want)
    del y
    c, s = mxq.mx_quantize(x, mxq.E2M1, mxq.SWIZZLED)
    rc, rs = O.quantize(base, O.E2M1, O.LINEAR)
    np.testing.assert_array_equal(T.u8(rows_of(c)), rc[ROWS % B])
    lin = T.unswizzle(T.u8(s), M, K)
    np.testing.assert_array_equal(lin[ROWS], rs[ROWS % B])
    assert not T.swizzle_pads(T.u8(s), M, K).any()
    y = mxq.mx_dequantize(c, s, K, mxq.E2M1, mxq.SWIZZLED)
    np.testing.assert_array_equal(T.bf16_bits(rows_of(y)), want)


def test_mxfp8_quantize_linear_past_2pow31(big):
    base, x = big
    c, s = mxq.mx_quantize(x, mxq.E4M3, mxq.LINEAR)
    rc, rs = O.quantize(base[ROWS % B], O.E4M3, O.LINEAR)
    np.testing.assert_array_equal(T.u8(rows_of(c)), rc)
    np.testing.assert_array_equal(T.u8(rows_of(s)), rs)


def test_rotate_quantize_past_2pow31(big):
    base, x = big
    H = W.normalized_hadamard_bf16(32)
    c, s = mxq.mx_rotate_quantize(x, T.to_gpu(H), mxq.E2M1, mxq.SWIZZLED)
    lin = T.unswizzle(T.u8(s), M, K)
    stats = T.check_rotated_codes(base[ROWS % B], H, O.E2M1, T.u8(rows_of(c)), lin[ROWS])
    assert stats["exempt_blocks"] <= 0.01 * stats["blocks"] + 2, stats
