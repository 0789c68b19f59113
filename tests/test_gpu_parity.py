"""GPU parity: the CUDA path (called through the C ABI) against the CPU oracle.

Bar: bit-exact codes, E8M0 bytes and bf16 QDQ outputs on the non-rotated paths; the rotated
paths follow the tolerance rules of mx_testlib (pre-quantization values within 1e-5 of the
chunk norm, code differences only next to rounding midpoints, scale flips only next to powers
of two). Inputs are the seeded synthetic workloads at sizes the oracle finishes in seconds
(several tiles plus ragged tails), and every workload at its full size, whole outputs: the
oracle runs over row chunks on all host cores (mx_testlib.map_row_chunks).
"""

import functools

import numpy as np
import pytest
import torch

import __graft_entry__
import mx_microscaling_quantize_gb300 as mxq
import oracle as O
from mx_microscaling_quantize_gb300 import workloads as W
import mx_testlib as T

pytestmark = pytest.mark.gpu
FMTS = [O.E2M1, O.E4M3]
LAYOUTS = [O.LINEAR, O.SWIZZLED]
GUARD = 4096
CANARY = 0xA5


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()
    yield
    assert mxq.mx_device_errors() == 0


@functools.lru_cache(maxsize=2)
def full_input(name, *args):
    """A full-size workload input, drawn once for the tests that share it (bf16 bits, read
    only)."""
    x = getattr(W, name)(*args)
    x.setflags(write=False)
    return x


def assert_quantize_rows(xb, fmt, codes, scales_linear):
    """GPU codes and linear scales of x equal the oracle's over every row (row chunks)."""
    T.assert_rows_equal(codes, lambda r0, r1: O.quantize(xb[r0:r1], fmt, O.LINEAR)[0], "codes")
    T.assert_rows_equal(scales_linear, lambda r0, r1: O.quantize(xb[r0:r1], fmt, O.LINEAR)[1],
                        "scales")


def quantize(xb, fmt, layout):
    c, s = mxq.mx_quantize(T.to_gpu(xb), fmt, layout)
    return T.u8(c), T.u8(s)


def qdq(xb, fmt, H=None):
    return T.bf16_bits(mxq.mx_qdq(T.to_gpu(xb), fmt, None if H is None else T.to_gpu(H)))


def assert_quantize_exact(xb, fmt, layout):
    c, s = quantize(xb, fmt, layout)
    rc, rs = O.quantize(xb, fmt, layout)
    np.testing.assert_array_equal(s, rs)
    np.testing.assert_array_equal(c, rc)


def guarded(nbytes):
    """A uint8 device buffer with GUARD canary bytes on both sides; returns (full, inner)."""
    full = torch.full((nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
    return full, full[GUARD:GUARD + nbytes]


def assert_guards(full, nbytes):
    f = full.cpu().numpy()
    assert (f[:GUARD] == CANARY).all() and (f[GUARD + nbytes:] == CANARY).all()


# ---------------------------------------------------------------------------------------------
# converters, exhaustively
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("fmt", FMTS)
def test_converter_sweep_bit_exact(fmt):
    """Every finite bf16 value at its own scale and at every larger scale (s in [-127, 125]):
    codes, scale bytes and QDQ outputs equal the oracle's."""
    xs = T.converter_sweep()
    assert_quantize_exact(xs, fmt, O.LINEAR)
    np.testing.assert_array_equal(qdq(xs, fmt), O.qdq(xs, fmt))


@pytest.mark.parametrize("fmt", FMTS)
def test_nan_and_inf_blocks(fmt):
    v = np.random.default_rng(3).standard_normal((4, 256)).astype(np.float32)
    v[0, 5], v[1, 40], v[2, 70], v[3, 255] = np.nan, np.inf, -np.inf, np.nan
    xb = W.to_bf16_bits(v)
    for layout in LAYOUTS:
        assert_quantize_exact(xb, fmt, layout)
    np.testing.assert_array_equal(qdq(xb, fmt), O.qdq(xb, fmt))


@pytest.mark.parametrize("fmt", FMTS)
def test_signed_zero_and_subnormal_blocks(fmt):
    v = np.zeros((2, 128), dtype=np.float32)
    v[0, 1::2] = -0.0
    v[1, :32] = -(2.0 ** -133)
    v[1, 32:64] = np.float32(2.0 ** -130) * np.arange(32)
    v[1, 64:] = -1e-38
    xb = W.to_bf16_bits(v)
    xb[0, 1::2] = 0x8000
    assert_quantize_exact(xb, fmt, O.LINEAR)
    np.testing.assert_array_equal(qdq(xb, fmt), O.qdq(xb, fmt))


# ---------------------------------------------------------------------------------------------
# non-rotated workloads
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("fmt", FMTS)
def test_mxfp8_linear_quant_workload_full_size(fmt, layout):
    """x[128, 4096] N(0,1) with 1% x50 outliers and an all-zero block per row."""
    assert_quantize_exact(W.mxfp8_linear_quant(), fmt, layout)


@pytest.mark.parametrize("fmt", FMTS)
def test_mxfp4_qdq_workload_small(fmt):
    np.testing.assert_array_equal(qdq(W.mxfp4_qdq_weight(384, 8192), fmt),
                                  O.qdq(W.mxfp4_qdq_weight(384, 8192), fmt))
    xa = W.mxfp4_qdq_activation(300, 8192)
    np.testing.assert_array_equal(qdq(xa, fmt), O.qdq(xa, fmt))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("which", ["weight", "activation"])
def test_mxfp4_qdq_workload_full_size(which, fmt):
    """The full tensors of the benchmark's step, x[8192, 8192] and x[4096, 8192]: every QDQ
    output equals the oracle's (MXFP4, the workload's format, and MXFP8), and
    QDQ(QDQ(x)) == QDQ(x) over the whole output."""
    xb = full_input("mxfp4_qdq_weight") if which == "weight" else full_input("mxfp4_qdq_activation")
    xg = T.to_gpu(xb)
    y = mxq.mx_qdq(xg, fmt)
    T.assert_rows_equal(T.bf16_bits(y), T.oracle_qdq_rows(xb, fmt), "QDQ")
    assert torch.equal(mxq.mx_qdq(y, fmt).view(torch.int16), y.view(torch.int16))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M", [1, 2, 127, 128, 129, 255])
@pytest.mark.parametrize("K", [32, 64, 96, 160, 416])
def test_edge_shapes_with_canaries(fmt, M, K):
    xb = W.mxfp8_linear_quant(M, K, stream=M * 1000 + K)
    x = T.to_gpu(xb)
    for layout in LAYOUTS:
        rows, cols = mxq.mx_scales_shape(M, K, layout)
        cb = mxq.code_bytes_per_row(fmt, K) * M
        cfull, codes = guarded(cb)
        sfull, scales = guarded(rows * cols)
        mxq.mx_quantize(x, fmt, layout, codes=codes, scales=scales)
        rc, rs = O.quantize(xb, fmt, layout)
        np.testing.assert_array_equal(T.u8(codes).reshape(rc.shape), rc)
        np.testing.assert_array_equal(T.u8(scales).reshape(rs.shape), rs)
        assert_guards(cfull, cb)
        assert_guards(sfull, rows * cols)
    yfull, ybytes = guarded(M * K * 2)
    mxq.mx_qdq(x, fmt, y=ybytes.view(torch.bfloat16).view(M, K))
    got = T.u8(ybytes).view(np.uint16).reshape(M, K)
    np.testing.assert_array_equal(got, O.qdq(xb, fmt))
    assert_guards(yfull, M * K * 2)


def test_non_default_stream_and_repeat_calls():
    xb = W.mxfp4_qdq_activation(256, 1024)
    x = T.to_gpu(xb)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        a = mxq.mx_qdq(x, mxq.E4M3)
        c1, s1 = mxq.mx_quantize(x, mxq.E2M1, mxq.SWIZZLED)
        c2, s2 = mxq.mx_quantize(x, mxq.E2M1, mxq.SWIZZLED)
    s.synchronize()
    np.testing.assert_array_equal(T.bf16_bits(a), O.qdq(xb, O.E4M3))
    assert torch.equal(c1, c2) and torch.equal(s1, s2)


@pytest.mark.parametrize("fmt", FMTS)
def test_qdq_idempotent_on_gpu(fmt):
    x = T.to_gpu(W.rotation_sweep_input("attn_in", 512, 8192))
    y = mxq.mx_qdq(x, fmt)
    assert torch.equal(mxq.mx_qdq(y, fmt).view(torch.int16), y.view(torch.int16))


# ---------------------------------------------------------------------------------------------
# dequantize stored codes + scales
# ---------------------------------------------------------------------------------------------
def dequantize(codes, scales, K, fmt, layout):
    y = mxq.mx_dequantize(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(), K,
                          fmt, layout)
    return T.bf16_bits(y)


@pytest.mark.parametrize("fmt", FMTS)
def test_dequantize_every_code_under_every_scale_byte(fmt):
    """Row r holds every code of the format under scale byte r (0..255): subnormal results,
    overflow to Inf, E8M0 NaN and E4M3 NaN codes included."""
    if fmt == O.E4M3:
        K = 256
        codes = np.tile(np.arange(256, dtype=np.uint8), (256, 1))
    else:
        K = 32
        nib = np.arange(32) % 16
        codes = np.tile((nib[0::2] | (nib[1::2] << 4)).astype(np.uint8), (256, 1))
    scales = np.repeat(np.arange(256, dtype=np.uint8), K // 32).reshape(256, K // 32)
    np.testing.assert_array_equal(dequantize(codes, scales, K, fmt, O.LINEAR),
                                  O.dequantize(codes, scales, K, fmt, O.LINEAR))


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (129, 416), (300, 4096), (1000, 2048)])
def test_dequantize_random_bytes_bit_exact(fmt, layout, M, K):
    rng = np.random.default_rng(M * 7 + K)
    codes = rng.integers(0, 256, (M, O.code_bytes_per_row(fmt, K)), dtype=np.uint8)
    scales = rng.integers(0, 256, O.scales_shape(M, K, layout), dtype=np.uint8)
    np.testing.assert_array_equal(dequantize(codes, scales, K, fmt, layout),
                                  O.dequantize(codes, scales, K, fmt, layout))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,K", [(1, 32), (127, 160), (255, 416)])
def test_dequantize_edge_shapes_with_canaries(fmt, M, K):
    xb = W.mxfp8_linear_quant(M, K, stream=M * 1000 + K + 1)
    for layout in LAYOUTS:
        c, s = mxq.mx_quantize(T.to_gpu(xb), fmt, layout)
        yfull, ybytes = guarded(M * K * 2)
        mxq.mx_dequantize(c, s, K, fmt, layout, y=ybytes.view(torch.bfloat16).view(M, K))
        got = T.u8(ybytes).view(np.uint16).reshape(M, K)
        np.testing.assert_array_equal(got, O.qdq(xb, fmt))
        assert_guards(yfull, M * K * 2)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("fmt", FMTS)
def test_dequantize_of_quantize_is_qdq_full_size(fmt, layout):
    """The MXFP4 QDQ weight workload x[8192, 8192]: the codes and scales of the quantize call
    (swizzle pads zero) and the bf16 output of dequantize(quantize(x)) equal the oracle's over
    the whole tensor, and the latter equals the GPU QDQ bit for bit."""
    xb = full_input("mxfp4_qdq_weight")
    x = T.to_gpu(xb)
    M, K = xb.shape
    c, s = mxq.mx_quantize(x, fmt, layout)
    y = mxq.mx_dequantize(c, s, K, fmt, layout)
    assert torch.equal(y.view(torch.int16), mxq.mx_qdq(x, fmt).view(torch.int16))
    s = T.u8(s)
    if layout == O.SWIZZLED:
        assert not T.swizzle_pads(s, M, K).any()
        s = T.unswizzle(s, M, K)
    assert_quantize_rows(xb, fmt, T.u8(c), s)
    T.assert_rows_equal(T.bf16_bits(y), T.oracle_qdq_rows(xb, fmt), "dequantize")


# ---------------------------------------------------------------------------------------------
# NVFP4 (16-element blocks, E4M3 scales under a global scale)
# ---------------------------------------------------------------------------------------------
def gs_of(xb) -> np.float32:
    """The usual global scale 448 * 6 / amax(x) (1 for an all-zero x: gs must be finite)."""
    amax = np.float32(np.abs(W.bf16_bits_to_float(xb)).max())
    return np.float32(448 * 6) / amax if amax > 0 else np.float32(1.0)


def gs_tensor(gs):
    return torch.tensor([float(gs)], dtype=torch.float32, device="cuda")


def nv_quantize(xb, gs, layout, H=None):
    c, s = mxq.mx_quantize_nvfp4(T.to_gpu(xb), gs_tensor(gs), layout,
                                 None if H is None else T.to_gpu(H))
    return T.u8(c), T.u8(s)


def nv_qdq(xb, gs, H=None):
    return T.bf16_bits(mxq.mx_qdq_nvfp4(T.to_gpu(xb), gs_tensor(gs),
                                        None if H is None else T.to_gpu(H)))


def assert_nvfp4_exact(xb, gs, H=None, layouts=LAYOUTS):
    for layout in layouts:
        c, s = nv_quantize(xb, gs, layout, H)
        rc, rs = O.nvfp4_quantize(xb, gs, layout, H_bits=H)
        np.testing.assert_array_equal(s, rs)
        np.testing.assert_array_equal(c, rc)
    np.testing.assert_array_equal(nv_qdq(xb, gs, H), O.nvfp4_qdq(xb, gs, H_bits=H))


@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (127, 160), (129, 416), (300, 4096), (64, 8192)])
def test_nvfp4_bit_exact(M, K):
    xb = W.mxfp4_qdq_activation(M, K) if K % 1024 == 0 else W.mxfp8_linear_quant(M, K, stream=M + K)
    for gs in (gs_of(xb), np.float32(1.0), np.float32(37.5)):
        assert_nvfp4_exact(xb, gs)


def test_nvfp4_special_underflow_and_saturation():
    v = np.random.default_rng(41).standard_normal((4, 256)).astype(np.float32)
    v[0, 5], v[1, 40], v[2, 70], v[3, 255] = np.nan, np.inf, -np.inf, np.nan
    v[3, :16] = 0.0
    v[3, 16:32] = -1e-30
    xb = W.to_bf16_bits(v)
    for gs in (np.float32(100.0), np.float32(1e-10), np.float32(6e6), np.float32(1e30)):
        assert_nvfp4_exact(xb, gs)


def test_nvfp4_every_scale_byte():
    """gs = 6 makes s_f the block abs-max itself, so the converter sweep (every finite bf16 at
    its own and every larger scale) reaches every E4M3 scale byte, saturation included."""
    xs = T.converter_sweep()
    assert_nvfp4_exact(xs, np.float32(6.0), layouts=[O.LINEAR])
    _, s = nv_quantize(xs, np.float32(6.0), O.LINEAR)
    assert set(np.unique(s)) >= set(range(0, 0x7F))


def test_nvfp4_full_size():
    """NVFP4 quantize (swizzled scales, pads zero) and QDQ of the weight x[8192, 8192]: codes,
    E4M3 scale bytes and bf16 outputs equal the oracle's over the whole tensor."""
    xb = full_input("mxfp4_qdq_weight")
    gs = gs_of(xb)
    x = T.to_gpu(xb)
    c, s = mxq.mx_quantize_nvfp4(x, gs_tensor(gs), mxq.SWIZZLED)
    y = mxq.mx_qdq_nvfp4(x, gs_tensor(gs))
    M, K = xb.shape
    s = T.u8(s)
    assert not T.swizzle_pads(s, M, 2 * K).any()
    ref = lambda r0, r1: O.nvfp4_quantize(xb[r0:r1], gs, O.LINEAR)
    T.assert_rows_equal(T.unswizzle(s, M, 2 * K), lambda r0, r1: ref(r0, r1)[1], "NVFP4 scales")
    T.assert_rows_equal(T.u8(c), lambda r0, r1: ref(r0, r1)[0], "NVFP4 codes")
    T.assert_rows_equal(T.bf16_bits(y), lambda r0, r1: O.nvfp4_qdq(xb[r0:r1], gs), "NVFP4 QDQ")


def nv_dequantize(codes, scales, K, gs, layout):
    y = mxq.mx_dequantize_nvfp4(torch.from_numpy(codes).cuda(), torch.from_numpy(scales).cuda(),
                                K, gs_tensor(gs), layout)
    return T.bf16_bits(y)


def test_nvfp4_dequantize_every_code_under_every_scale_byte():
    """Row r holds all 16 E2M1 codes in both of its blocks under E4M3 scale byte r (0..255:
    subnormal scales, the sign bit and the two NaN bytes included), for three global scales."""
    K = 32
    nib = np.arange(32) % 16
    codes = np.tile((nib[0::2] | (nib[1::2] << 4)).astype(np.uint8), (256, 1))
    scales = np.repeat(np.arange(256, dtype=np.uint8)[:, None], 2, axis=1)
    for gs in (np.float32(1.0), np.float32(0.3712), np.float32(2.0 ** -10 * 3)):
        np.testing.assert_array_equal(nv_dequantize(codes, scales, K, gs, O.LINEAR),
                                      O.nvfp4_dequantize(codes, scales, K, gs, O.LINEAR))


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("M,K", [(1, 32), (3, 96), (129, 416), (300, 4096), (1000, 2048)])
def test_nvfp4_dequantize_random_bytes_bit_exact(layout, M, K):
    rng = np.random.default_rng(M * 11 + K)
    codes = rng.integers(0, 256, (M, K // 2), dtype=np.uint8)
    scales = rng.integers(0, 256, O.nvfp4_scales_shape(M, K, layout), dtype=np.uint8)
    gs = np.float32(448 * 6 / 3.5)
    np.testing.assert_array_equal(nv_dequantize(codes, scales, K, gs, layout),
                                  O.nvfp4_dequantize(codes, scales, K, gs, layout))


@pytest.mark.parametrize("M,K", [(1, 32), (127, 160), (255, 416)])
def test_nvfp4_dequantize_edge_shapes_with_canaries(M, K):
    xb = W.mxfp8_linear_quant(M, K, stream=M * 1000 + K + 2)
    gs = gs_of(xb)
    for layout in LAYOUTS:
        c, s = mxq.mx_quantize_nvfp4(T.to_gpu(xb), gs_tensor(gs), layout)
        yfull, ybytes = guarded(M * K * 2)
        mxq.mx_dequantize_nvfp4(c, s, K, gs_tensor(gs), layout,
                                y=ybytes.view(torch.bfloat16).view(M, K))
        got = T.u8(ybytes).view(np.uint16).reshape(M, K)
        np.testing.assert_array_equal(got, O.nvfp4_qdq(xb, gs))
        assert_guards(yfull, M * K * 2)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_nvfp4_dequantize_of_quantize_is_qdq_full_size(layout):
    """x[8192, 8192] (the MXFP4 QDQ weight workload), plain and rotated (normalized Hadamard,
    g = 16): dequantize(quantize(x)) equals the GPU QDQ bit for bit over the whole tensor; the
    plain one also equals the oracle's QDQ over the whole tensor."""
    xb = full_input("mxfp4_qdq_weight")
    x = T.to_gpu(xb)
    gs = gs_of(xb)
    for H in (None, T.to_gpu(W.normalized_hadamard_bf16(16))):
        c, s = mxq.mx_quantize_nvfp4(x, gs_tensor(gs), layout, H)
        y = mxq.mx_dequantize_nvfp4(c, s, x.shape[1], gs_tensor(gs), layout)
        q = mxq.mx_qdq_nvfp4(x, gs_tensor(gs), H)
        assert torch.equal(y.view(torch.int16), q.view(torch.int16))
        if H is None:
            T.assert_rows_equal(T.bf16_bits(y), lambda r0, r1: O.nvfp4_qdq(xb[r0:r1], gs),
                                "NVFP4 dequantize")


@pytest.mark.parametrize("g", [16, 32, 64, 128])
def test_nvfp4_exact_rotations_bit_exact(g):
    """Identity and signed-permutation H make the rotation exact in fp32: the rotated NVFP4
    kernels then equal the oracle bit for bit."""
    xb = W.mxfp4_qdq_activation(200, 512)
    gs = gs_of(xb)
    assert_nvfp4_exact(xb, gs, rotation(g, "identity"))
    rng = np.random.default_rng(g)
    P = np.zeros((g, g))
    P[np.arange(g), rng.permutation(g)] = rng.choice([-1.0, 1.0], g)
    Hp = W.to_bf16_bits(P)
    assert_nvfp4_exact(xb, gs, Hp)
    # the signed permutation moves values across blocks: not the plain path's result
    assert not np.array_equal(O.nvfp4_qdq(xb, gs, H_bits=Hp), O.nvfp4_qdq(xb, gs))


@pytest.mark.parametrize("g", [16, 32, 64, 128])
def test_nvfp4_rotated_hadamard_rules(g):
    xb = W.rotate_quant_activation(300, 1024)
    H = rotation(g)
    gs = np.float32(448 * 6) / np.float32(np.abs(O.rotate(xb, H)).max())
    M, K = xb.shape
    for layout in LAYOUTS:
        c, s = nv_quantize(xb, gs, layout, H)
        if layout == O.SWIZZLED:
            assert not T.swizzle_pads(s, M, 2 * K).any()
            s = T.unswizzle(s, M, 2 * K)
        stats = T.check_rotated_nvfp4(xb, H, gs, c, s)
        assert stats["exempt_blocks"] <= 0.01 * stats["blocks"] + 2, stats
    stats = T.check_rotated_nvfp4_qdq(xb, H, gs, nv_qdq(xb, gs, H))
    assert stats["exempt_blocks"] <= 0.01 * stats["blocks"] + 2, stats


def test_nvfp4_rotated_full_size():
    """Rotate (normalized Hadamard, g = 16) + NVFP4 quantize, swizzled scales, and rotated NVFP4
    QDQ of the largest activation x[8192, 28672]: every block under the NVFP4 rules."""
    M, K = 8192, 28672
    xb = full_input("rotate_quant_activation", M, K)
    H = rotation(16)
    gs = np.float32(448 * 6 / 8.0)  # rotated N(0,1) values stay well below 8
    c, s = nv_quantize(xb, gs, O.SWIZZLED, H)
    assert not T.swizzle_pads(s, M, 2 * K).any()
    q = nv_qdq(xb, gs, H)
    st = T.check_rotated_multi(xb, H, nvfp4={gs: (c, T.unswizzle(s, M, 2 * K))},
                               nvfp4_qdq={gs: q})
    for v in st.values():
        assert v["exempt_blocks"] <= 0.01 * v["blocks"] + 2, st


# ---------------------------------------------------------------------------------------------
# grouped (MoE) quantize
# ---------------------------------------------------------------------------------------------
def grouped(xb, offsets, fmt, layout):
    c, s = mxq.mx_quantize_grouped(T.to_gpu(xb), torch.from_numpy(offsets).cuda(), fmt, layout)
    return T.u8(c), T.u8(s)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_moe_workload_full_size(layout):
    """128 experts, Zipf(1.1) token counts summing to 16384, rows [n_e, 2048], MXFP8."""
    xb, off = W.moe_quant()
    c, s = grouped(xb, off, O.E4M3, layout)
    rows = s.shape[0]
    rc, rs = O.quantize_grouped(xb, off, O.E4M3, layout, scale_rows=rows)
    np.testing.assert_array_equal(s, rs)
    np.testing.assert_array_equal(c, rc)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("counts", [[0, 1, 127, 128, 129, 0, 300, 5],
                                    [1000], [0, 0, 64], [128] * 6, [3] * 40])
def test_grouped_edge_counts(fmt, counts):
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    xb = W.mxfp8_linear_quant(int(off[-1]), 160, stream=len(counts))
    for layout in LAYOUTS:
        c, s = grouped(xb, off, fmt, layout)
        rc, rs = O.quantize_grouped(xb, off, fmt, layout, scale_rows=s.shape[0])
        np.testing.assert_array_equal(s, rs)
        np.testing.assert_array_equal(c, rc)


def nv_grouped(xb, offsets, gs, layout):
    c, s = mxq.mx_quantize_nvfp4_grouped(T.to_gpu(xb), torch.from_numpy(offsets).cuda(),
                                         torch.from_numpy(np.asarray(gs, np.float32)).cuda(),
                                         layout)
    return T.u8(c), T.u8(s)


def expert_global_scales(xb, off):
    """448 * 6 / amax of each expert's rows (1 for an expert without rows or all zeros)."""
    v = np.abs(W.bf16_bits_to_float(xb))
    gs = []
    for e in range(len(off) - 1):
        amax = np.float32(v[off[e]:off[e + 1]].max()) if off[e + 1] > off[e] else np.float32(0)
        gs.append(np.float32(448 * 6) / amax if amax > 0 else np.float32(1.0))
    return np.array(gs, np.float32)


@pytest.mark.parametrize("layout", LAYOUTS)
def test_nvfp4_moe_workload_full_size(layout):
    """The MoE workload (128 experts, Zipf(1.1) counts summing to 16384, rows [n_e, 2048]) in
    NVFP4 with one global scale per expert: bit-exact codes and scales, pads included."""
    xb, off = W.moe_quant()
    gs = expert_global_scales(xb, off)
    c, s = nv_grouped(xb, off, gs, layout)
    rc, rs = O.nvfp4_quantize_grouped(xb, off, gs, layout, scale_rows=s.shape[0])
    np.testing.assert_array_equal(s, rs)
    np.testing.assert_array_equal(c, rc)


@pytest.mark.parametrize("counts", [[0, 1, 127, 128, 129, 0, 300, 5],
                                    [1000], [0, 0, 64], [128] * 6, [3] * 40])
def test_nvfp4_grouped_edge_counts(counts):
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    for K in (160, 192):  # K/16 % 4 != 0 (partial last scale word) and == 0
        xb = W.mxfp8_linear_quant(int(off[-1]), K, stream=len(counts) + K)
        gs = expert_global_scales(xb, off) * np.float32(0.75)
        for layout in LAYOUTS:
            c, s = nv_grouped(xb, off, gs, layout)
            rc, rs = O.nvfp4_quantize_grouped(xb, off, gs, layout, scale_rows=s.shape[0])
            np.testing.assert_array_equal(s, rs)
            np.testing.assert_array_equal(c, rc)


def test_grouped_on_both_sides_of_the_row_table_limit():
    """MX grouped calls with swizzled scales run on the grid-stride kernel with a per-CTA table
    of its rows' padded-row shifts while the table fits (2048 entries), else on the
    contiguous-range kernel. K = 32 puts 258 rows in each CTA iteration: 300,000 rows stay
    within the table on a GB300 (2 iterations) and 1,300,000 rows exceed it (9); both formats
    against the oracle, and NVFP4 grouped (the contiguous-range kernel) at the same sizes."""
    for M in (300_000, 1_300_000):
        counts = W.moe_counts(E=96, tokens=M, stream=M % 1000)
        off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
        xb = W.mxfp8_linear_quant(M, 32, stream=7)
        for fmt in FMTS:
            c, s = grouped(xb, off, fmt, O.SWIZZLED)
            rc, rs = O.quantize_grouped(xb, off, fmt, O.SWIZZLED, scale_rows=s.shape[0])
            np.testing.assert_array_equal(s, rs)
            np.testing.assert_array_equal(c, rc)
        gs = expert_global_scales(xb, off)
        for layout in LAYOUTS:
            c, s = nv_grouped(xb, off, gs, layout)
            rc, rs = O.nvfp4_quantize_grouped(xb, off, gs, layout, scale_rows=s.shape[0])
            np.testing.assert_array_equal(s, rs)
            np.testing.assert_array_equal(c, rc)


@pytest.mark.parametrize("K", [8224, 28672])
def test_grouped_wide_rows(K):
    """Rows of more than 256 blocks (K = 8224: 257 blocks, the column wrap not a power of two;
    K = 28672: 896): each CTA iteration then spans at most two rows of the row table. 22 experts:
    Zipf counts with two empty experts inserted, both MX formats and NVFP4, both layouts."""
    counts = np.insert(W.moe_counts(E=20, tokens=600, stream=K % 97), [3, 11], 0)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    xb = W.mxfp8_linear_quant(int(off[-1]), K, stream=K)
    for layout in LAYOUTS:
        for fmt in FMTS:
            c, s = grouped(xb, off, fmt, layout)
            rc, rs = O.quantize_grouped(xb, off, fmt, layout, scale_rows=s.shape[0])
            np.testing.assert_array_equal(s, rs)
            np.testing.assert_array_equal(c, rc)
        gs = expert_global_scales(xb, off)
        c, s = nv_grouped(xb, off, gs, layout)
        rc, rs = O.nvfp4_quantize_grouped(xb, off, gs, layout, scale_rows=s.shape[0])
        np.testing.assert_array_equal(s, rs)
        np.testing.assert_array_equal(c, rc)


def test_grouped_maximum_expert_count():
    """1024 experts (the limit; the prologue's per-thread share of the expert scan is then
    full), random counts with many empty experts, MXFP8 and NVFP4, both layouts."""
    rng = np.random.default_rng(1024)
    counts = rng.integers(0, 6, 1024) * (rng.random(1024) < 0.6)
    off = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    xb = W.mxfp8_linear_quant(int(off[-1]), 96, stream=1024)
    gs = expert_global_scales(xb, off)
    for layout in LAYOUTS:
        c, s = grouped(xb, off, O.E4M3, layout)
        rc, rs = O.quantize_grouped(xb, off, O.E4M3, layout, scale_rows=s.shape[0])
        np.testing.assert_array_equal(s, rs)
        np.testing.assert_array_equal(c, rc)
        c, s = nv_grouped(xb, off, gs, layout)
        rc, rs = O.nvfp4_quantize_grouped(xb, off, gs, layout, scale_rows=s.shape[0])
        np.testing.assert_array_equal(s, rs)
        np.testing.assert_array_equal(c, rc)


def test_nvfp4_calls_capture_into_a_cuda_graph():
    """NVFP4 quantize (plain and rotated), QDQ, dequantize and grouped quantize captured in one
    CUDA graph replay bit-identically to eager calls."""
    xb = W.rotation_sweep_input("attn_in", 256, 1024)
    x = T.to_gpu(xb)
    H = T.to_gpu(rotation(16))
    gs = gs_tensor(gs_of(xb))
    xm, off = W.moe_quant(E=8, tokens=700, K=256)
    xg, offs = T.to_gpu(xm), torch.from_numpy(off).cuda()
    gse = torch.full((8,), 50.0, device="cuda")
    c, s = mxq.mx_quantize_nvfp4(x, gs, mxq.SWIZZLED)
    cr, sr = mxq.mx_quantize_nvfp4(x, gs, mxq.SWIZZLED, H)
    y, yd = torch.empty_like(x), torch.empty_like(x)
    cg, sg = mxq.mx_quantize_nvfp4_grouped(xg, offs, gse, mxq.SWIZZLED)
    K = x.shape[1]

    def calls():
        mxq.mx_quantize_nvfp4(x, gs, mxq.SWIZZLED, codes=c, scales=s)
        mxq.mx_quantize_nvfp4(x, gs, mxq.SWIZZLED, H, codes=cr, scales=sr)
        mxq.mx_qdq_nvfp4(x, gs, H, y=y)
        mxq.mx_dequantize_nvfp4(c, s, K, gs, mxq.SWIZZLED, y=yd)
        mxq.mx_quantize_nvfp4_grouped(xg, offs, gse, mxq.SWIZZLED, codes=cg, scales=sg)

    outs = (c, s, cr, sr, y, yd, cg, sg)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        calls()
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [t.clone() for t in outs]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        calls()
    for _ in range(2):
        for t in outs:
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for got, want in zip(outs, eager):
            assert torch.equal(got.view(torch.uint8), want.view(torch.uint8))
    np.testing.assert_array_equal(T.bf16_bits(yd), O.nvfp4_qdq(xb, gs_of(xb)))


@pytest.mark.parametrize("first", [0, 30])
def test_grouped_bad_offsets_stay_in_bounds(first):
    """Offsets that break the contract (decreasing, beyond M, first offset above 0 with rows
    before it) give unspecified values but no access outside the buffers (canaries intact) and
    no error from the device. K = 64: two scale columns, so the partial-word pad pass runs."""
    M, K, E = 200, 64, 4
    off = np.array([first, 150, 20, 500, 200], dtype=np.int64)
    x = T.to_gpu(W.mxfp8_linear_quant(M, K))
    rows, cols = mxq.mx_grouped_scales_shape(M, E, K, mxq.SWIZZLED)
    cfull, codes = guarded(M * K)
    sfull, scales = guarded(rows * cols)
    mxq.mx_quantize_grouped(x, torch.from_numpy(off).cuda(), mxq.E4M3, mxq.SWIZZLED, codes=codes,
                            scales=scales)
    torch.cuda.synchronize()
    assert_guards(cfull, M * K)
    assert_guards(sfull, rows * cols)
    rows, cols = mxq.mx_nvfp4_grouped_scales_shape(M, E, K, mxq.SWIZZLED)
    cfull, codes = guarded(M * K // 2)
    sfull, scales = guarded(rows * cols)
    mxq.mx_quantize_nvfp4_grouped(x, torch.from_numpy(off).cuda(),
                                  torch.ones(E, dtype=torch.float32, device="cuda"), mxq.SWIZZLED,
                                  codes=codes, scales=scales)
    torch.cuda.synchronize()
    assert_guards(cfull, M * K // 2)
    assert_guards(sfull, rows * cols)


# ---------------------------------------------------------------------------------------------
# rotated path
# ---------------------------------------------------------------------------------------------
def rotation(g, kind="hadamard"):
    if kind == "hadamard":
        return W.normalized_hadamard_bf16(g)
    if kind == "identity":
        return W.to_bf16_bits(np.eye(g))
    rng = np.random.default_rng(g)
    return W.to_bf16_bits(rng.standard_normal((g, g)) / np.sqrt(g))


@pytest.mark.parametrize("kind", ["hadamard", "random"])
@pytest.mark.parametrize("g", [16, 32, 64, 128])
def test_rotated_values_within_tolerance(g, kind):
    xb = W.rotate_quant_activation(300, 1024)
    H = rotation(g, kind)
    y = mxq.mx_rotate_debug(T.to_gpu(xb), T.to_gpu(H)).cpu().numpy()
    assert T.check_rotated_values(y, O.rotate(xb, H), g) <= 1.0


@pytest.mark.parametrize("g", [16, 32, 64, 128])
def test_identity_rotation_is_bit_exact(g):
    """x * I is exact in fp32: the rotated kernels then equal the plain path bit for bit."""
    xb = W.mxfp4_qdq_activation(200, 512)
    H = T.to_gpu(rotation(g, "identity"))
    x = T.to_gpu(xb)
    for fmt in FMTS:
        for layout in LAYOUTS:
            c, s = mxq.mx_rotate_quantize(x, H, fmt, layout)
            rc, rs = O.quantize(xb, fmt, layout)
            np.testing.assert_array_equal(T.u8(s), rs)
            np.testing.assert_array_equal(T.u8(c), rc)
        np.testing.assert_array_equal(T.bf16_bits(mxq.mx_qdq(x, fmt, H)), O.qdq(xb, fmt))


@pytest.mark.parametrize("K,g", [(96, 16), (96, 32), (160, 32), (192, 64), (416, 32)])
def test_identity_rotation_partial_column_tile(K, g):
    """K % 128 != 0 on the tensor-core kernel (M > 16): the last 128-column tile is partial, so
    its staged scales cover fewer than 4 (MX) / 8 (NVFP4) columns and the linear scale rows
    are not 4-byte aligned. With H = I the results equal the plain path bit for bit, both
    layouts, MX and NVFP4."""
    H = T.to_gpu(rotation(g, "identity"))
    for M in (129, 200):
        xb = W.mxfp8_linear_quant(M, K, stream=K + g)
        x = T.to_gpu(xb)
        for fmt in FMTS:
            for layout in LAYOUTS:
                c, s = mxq.mx_rotate_quantize(x, H, fmt, layout)
                rc, rs = O.quantize(xb, fmt, layout)
                np.testing.assert_array_equal(T.u8(s), rs)
                np.testing.assert_array_equal(T.u8(c), rc)
        gs = gs_of(xb)
        for layout in LAYOUTS:
            c, s = nv_quantize(xb, gs, layout, rotation(g, "identity"))
            rc, rs = O.nvfp4_quantize(xb, gs, layout)
            np.testing.assert_array_equal(s, rs)
            np.testing.assert_array_equal(c, rc)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,K", [(1, 8192), (16, 8192), (128, 1024), (300, 1024), (16, 28672)])
def test_rotate_quantize_rules(fmt, layout, M, K):
    """Fused rotate + quantize (g = 32 normalized Hadamard) on the activation workload."""
    xb = W.rotate_quant_activation(M, K)
    H = rotation(32)
    c, s = mxq.mx_rotate_quantize(T.to_gpu(xb), T.to_gpu(H), fmt, layout)
    c, s = T.u8(c), T.u8(s)
    if layout == O.SWIZZLED:
        assert not T.swizzle_pads(s, M, K).any()
        s = T.unswizzle(s, M, K)
    stats = T.check_rotated_codes(xb, H, fmt, c, s)
    assert stats["exempt_blocks"] <= 0.01 * stats["blocks"] + 2, stats


@pytest.mark.parametrize("kind", ["hadamard", "random"])
@pytest.mark.parametrize("g", [16, 32, 64, 128])
@pytest.mark.parametrize("fmt", FMTS)
def test_rotated_qdq_rules(fmt, g, kind):
    """Rotated QDQ on the decoder-layer input recipe (Student-t nu=5)."""
    xb = W.rotation_sweep_input("down_proj_in", 128, 2048)
    H = rotation(g, kind)
    out = qdq(xb, fmt, H)
    stats = T.check_rotated_qdq(xb, H, fmt, out)
    assert stats["exempt_blocks"] <= 0.01 * stats["blocks"] + 2, stats


def few_rows_K(g):
    """A K with a partial last 128-column tile where g allows one (K % g == 0)."""
    return {16: 288, 32: 288, 64: 320, 128: 384}[g]


@pytest.mark.parametrize("kind", ["hadamard", "random"])
@pytest.mark.parametrize("g", [16, 32, 64, 128])
@pytest.mark.parametrize("M", [1, 3, 16])
def test_few_rows_rotated_paths(M, g, kind):
    """Calls with at most 16 rows (decode-sized) run on the FMA kernel: rotated values within
    tolerance, rotate+quantize in both layouts (swizzled pads zero, canary bands intact) and
    rotated QDQ under the rules, for both MX formats."""
    K = few_rows_K(g)
    xb = W.rotate_quant_activation(M, K, stream=M * 1000 + g)
    H = rotation(g, kind)
    x, Hd = T.to_gpu(xb), T.to_gpu(H)
    y = mxq.mx_rotate_debug(x, Hd).cpu().numpy()
    assert T.check_rotated_values(y, O.rotate(xb, H), g) <= 1.0
    for fmt in FMTS:
        for layout in LAYOUTS:
            rows, cols = mxq.mx_scales_shape(M, K, layout)
            nc = M * O.code_bytes_per_row(fmt, K)
            cfull, codes = guarded(nc)
            sfull, scales = guarded(rows * cols)
            mxq.mx_rotate_quantize(x, Hd, fmt, layout, codes=codes, scales=scales)
            c = T.u8(codes).reshape(M, -1)
            s = T.u8(scales).reshape(rows, cols)
            assert_guards(cfull, nc)
            assert_guards(sfull, rows * cols)
            if layout == O.SWIZZLED:
                assert not T.swizzle_pads(s, M, K).any()
                s = T.unswizzle(s, M, K)
            stats = T.check_rotated_codes(xb, H, fmt, c, s)
            assert stats["exempt_blocks"] <= 0.01 * stats["blocks"] + 2, stats
        yfull, ybytes = guarded(M * K * 2)
        mxq.mx_qdq(x, fmt, Hd, y=ybytes.view(torch.bfloat16).view(M, K))
        assert_guards(yfull, M * K * 2)
        T.check_rotated_qdq(xb, H, fmt, T.u8(ybytes).view(np.uint16).reshape(M, K))


@pytest.mark.parametrize("g", [16, 32, 64, 128])
@pytest.mark.parametrize("M", [1, 5, 16])
def test_few_rows_identity_rotation_is_bit_exact(M, g):
    """x * I is exact in fp32 on the FMA kernel too: codes, scales (both layouts) and QDQ equal
    the plain path's oracle bit for bit, MX and NVFP4 (quantize and QDQ)."""
    K = few_rows_K(g)
    xb = W.mxfp8_linear_quant(M, K, stream=M * 100 + g)
    H = T.to_gpu(rotation(g, "identity"))
    x = T.to_gpu(xb)
    for fmt in FMTS:
        for layout in LAYOUTS:
            c, s = mxq.mx_rotate_quantize(x, H, fmt, layout)
            rc, rs = O.quantize(xb, fmt, layout)
            np.testing.assert_array_equal(T.u8(s), rs)
            np.testing.assert_array_equal(T.u8(c), rc)
        np.testing.assert_array_equal(T.bf16_bits(mxq.mx_qdq(x, fmt, H)), O.qdq(xb, fmt))
    gs = gs_of(xb)
    for layout in LAYOUTS:
        c, s = mxq.mx_quantize_nvfp4(x, gs_tensor(gs), layout, H)
        rc, rs = O.nvfp4_quantize(xb, gs, layout)
        np.testing.assert_array_equal(T.u8(s), rs)
        np.testing.assert_array_equal(T.u8(c), rc)
    np.testing.assert_array_equal(T.bf16_bits(mxq.mx_qdq_nvfp4(x, gs_tensor(gs), H)),
                                  O.nvfp4_qdq(xb, gs))


@pytest.mark.parametrize("g", [16, 32, 64, 128])
def test_few_rows_nvfp4_hadamard_rules(g):
    M, K = 7, few_rows_K(g)
    xb = W.rotate_quant_activation(M, K, stream=g + 3)
    H = rotation(g)
    gs = np.float32(448 * 6 / 8.0)
    for layout in LAYOUTS:
        c, s = nv_quantize(xb, gs, layout, H)
        if layout == O.SWIZZLED:
            s = T.unswizzle(s, M, 2 * K)
        stats = T.check_rotated_nvfp4(xb, H, gs, c, s)
        assert stats["exempt_blocks"] <= 0.01 * stats["blocks"] + 2, stats
    T.check_rotated_nvfp4_qdq(xb, H, gs, nv_qdq(xb, gs, H))


@pytest.mark.parametrize("g", [16, 32, 128])
@pytest.mark.parametrize("M", [5, 40])
def test_rotated_nan_and_inf_inputs(M, g):
    """NaN and +-Inf inputs on both rotation kernels (M = 5: the FMA kernel for g <= 64; M = 40
    and g = 128: the tensor-core kernel): every chunk holding one rotates to NaN/Inf values, its
    blocks get scale byte 0xFF with the fill codes (QDQ: 0x7FC0), exactly as in the oracle; the
    other chunks follow the rules."""
    K = 512
    v = np.random.default_rng(M * 10 + g).standard_normal((M, K)).astype(np.float32)
    v[0, 3], v[M - 1, 200], v[M // 2, 511] = np.nan, np.inf, -np.inf
    v[1, 130], v[1, 131] = np.inf, -np.inf
    xb = W.to_bf16_bits(v)
    H = rotation(g)
    x, Hd = T.to_gpu(xb), T.to_gpu(H)
    for fmt in FMTS:
        c, s = mxq.mx_rotate_quantize(x, Hd, fmt, mxq.LINEAR)
        c, s = T.u8(c), T.u8(s)
        _, rs = O.rotate_quantize(xb, H, fmt, O.LINEAR)
        special = rs == 255
        assert special.any() and (s[special] == 255).all() and (s[~special] != 255).all()
        stats = T.check_rotated_codes(xb, H, fmt, c, s)
        assert stats["exempt_blocks"] <= 0.01 * stats["blocks"] + 2, stats
        out = qdq(xb, fmt, H)
        ref = O.rotate_qdq(xb, H, fmt)
        nan_ref = np.repeat(special, 32, axis=1)
        np.testing.assert_array_equal(out[nan_ref], ref[nan_ref])
        T.check_rotated_qdq(xb, H, fmt, out)


@pytest.mark.parametrize("M,g", [(16, 32), (17, 32), (8, 64), (9, 64), (4, 128), (5, 128),
                                 (16, 16), (17, 16)])
def test_rotated_dispatch_boundary(M, g):
    """Both sides of the switch between the FMA kernel (M <= 16 and M * g <= 512) and the
    tensor-core kernel: rotate+quantize (both formats and layouts), rotated QDQ and rotated
    NVFP4 follow the oracle under the rules."""
    K = few_rows_K(g) + 2 * 128
    xb = W.rotate_quant_activation(M, K, stream=7 * M + g)
    H = rotation(g)
    x, Hd = T.to_gpu(xb), T.to_gpu(H)
    for fmt in FMTS:
        for layout in LAYOUTS:
            c, s = mxq.mx_rotate_quantize(x, Hd, fmt, layout)
            c, s = T.u8(c), T.u8(s)
            if layout == O.SWIZZLED:
                assert not T.swizzle_pads(s, M, K).any()
                s = T.unswizzle(s, M, K)
            stats = T.check_rotated_codes(xb, H, fmt, c, s)
            assert stats["exempt_blocks"] <= 0.01 * stats["blocks"] + 2, stats
        T.check_rotated_qdq(xb, H, fmt, qdq(xb, fmt, H))
    gs = np.float32(448 * 6 / 8.0)
    c, s = nv_quantize(xb, gs, O.SWIZZLED, H)
    stats = T.check_rotated_nvfp4(xb, H, gs, c, T.unswizzle(s, M, 2 * K))
    assert stats["exempt_blocks"] <= 0.01 * stats["blocks"] + 2, stats
    T.check_rotated_nvfp4_qdq(xb, H, gs, nv_qdq(xb, gs, H))


def test_random_shapes_every_entry_point():
    """Seeded random shapes (M from 1 to 300, K a random multiple of max(g, 32)): plain
    quantize, QDQ and dequantize of both formats and layouts and NVFP4 quantize / QDQ /
    dequantize bit-exact against the oracle; rotate+quantize and rotated QDQ under the rules."""
    rng = np.random.default_rng(2024)
    for case in range(16):
        M = int(rng.choice([1, 2, 7, 16, 17, 100, 129, 300]))
        g = int(rng.choice([16, 32, 64, 128]))
        K = int(rng.integers(1, 12)) * max(g, 32)
        xb = W.rotate_quant_activation(M, K, stream=1000 + case)
        x = T.to_gpu(xb)
        for fmt in FMTS:
            for layout in LAYOUTS:
                c, s = mxq.mx_quantize(x, fmt, layout)
                rc, rs = O.quantize(xb, fmt, layout)
                np.testing.assert_array_equal(T.u8(c), rc)
                np.testing.assert_array_equal(T.u8(s), rs)
                np.testing.assert_array_equal(T.bf16_bits(mxq.mx_dequantize(c, s, K, fmt, layout)),
                                              O.qdq(xb, fmt))
            np.testing.assert_array_equal(T.bf16_bits(mxq.mx_qdq(x, fmt)), O.qdq(xb, fmt))
        gs = gs_of(xb)
        assert_nvfp4_exact(xb, gs)
        c, s = mxq.mx_quantize_nvfp4(x, gs_tensor(gs), mxq.SWIZZLED)
        np.testing.assert_array_equal(
            T.bf16_bits(mxq.mx_dequantize_nvfp4(c, s, K, gs_tensor(gs), mxq.SWIZZLED)),
            O.nvfp4_qdq(xb, gs))
        H = rotation(g)
        fmt = FMTS[case % 2]
        c, s = mxq.mx_rotate_quantize(x, T.to_gpu(H), fmt, mxq.SWIZZLED)
        s = T.u8(s)
        assert not T.swizzle_pads(s, M, K).any()
        stats = T.check_rotated_codes(xb, H, fmt, T.u8(c), T.unswizzle(s, M, K))
        assert stats["exempt_blocks"] <= 0.01 * stats["blocks"] + 2, (M, K, g, stats)
        T.check_rotated_qdq(xb, H, fmt, qdq(xb, fmt, H))


def test_rotate_quantize_full_size_other_format_and_layout():
    """The largest activation of the rotate+quantize workload, x[8192, 28672], g = 32: MXFP8
    with swizzled scales and MXFP4 with linear scales (MXFP4 swizzled is the workload grid
    below), every block under the rules."""
    M, K = 8192, 28672
    xb = full_input("rotate_quant_activation", M, K)
    H = rotation(32)
    x, Hd = T.to_gpu(xb), T.to_gpu(H)
    c8, s8 = mxq.mx_rotate_quantize(x, Hd, mxq.E4M3, mxq.SWIZZLED)
    s8 = T.u8(s8)
    assert not T.swizzle_pads(s8, M, K).any()
    c4, s4 = mxq.mx_rotate_quantize(x, Hd, mxq.E2M1, mxq.LINEAR)
    st = T.check_rotated_multi(xb, H, codes={O.E4M3: (T.u8(c8), T.unswizzle(s8, M, K)),
                                             O.E2M1: (T.u8(c4), T.u8(s4))})
    for v in st.values():
        assert v["exempt_blocks"] <= 0.01 * v["blocks"] + 2, st


@pytest.mark.parametrize("N,K", W.WEIGHT_SHAPES)
def test_weight_rotate_quantize_full_size(N, K):
    """Weight-side rotate + quantize of the 70B layer weights (the same H as the activations),
    swizzled scales, both formats, g = 32 and g = 128: every block of the whole weight under
    the rules."""
    xb = W.weight_rotate_quant(N, K)
    x = T.to_gpu(xb)
    for g in (32, 128):
        H = rotation(g)
        outs = {}
        for fmt in FMTS:
            c, s = mxq.mx_rotate_quantize(x, T.to_gpu(H), fmt, mxq.SWIZZLED)
            s = T.u8(s)
            assert not T.swizzle_pads(s, N, K).any()
            outs[fmt] = (T.u8(c), T.unswizzle(s, N, K))
            del c
        st = T.check_rotated_multi(xb, H, codes=outs)
        for v in st.values():
            assert v["exempt_blocks"] <= 0.01 * v["blocks"] + 2, (g, st)


@pytest.mark.parametrize("K", W.ROTATE_QUANT_K)
@pytest.mark.parametrize("M", W.ROTATE_QUANT_M)
def test_rotate_quant_workload_grid(M, K):
    """The fused rotate + MXFP4 quantize workload at every one of its (M, K) sizes (g = 32
    normalized Hadamard, swizzled scales, rows padded to 128): every row under the rules,
    swizzle pads zero over the whole buffer."""
    xb = full_input("rotate_quant_activation", M, K)
    H = rotation(32)
    c, s = mxq.mx_rotate_quantize(T.to_gpu(xb), T.to_gpu(H), mxq.E2M1, mxq.SWIZZLED)
    s = T.u8(s)
    assert not T.swizzle_pads(s, M, K).any()
    stats = T.check_rotated_codes(xb, H, O.E2M1, T.u8(c), T.unswizzle(s, M, K))
    assert stats["exempt_blocks"] <= 0.01 * stats["blocks"] + 2, stats


@pytest.mark.parametrize("layer", [n for n, _, _ in W.ROTATION_SWEEP_LAYERS])
def test_rotation_sweep_full_size(layer):
    """The rotation-size sweep on each of the three decoder-layer inputs at full size: rotated
    QDQ for every g in {16, 32, 64, 128} and both formats, every block under the rules."""
    xb = W.rotation_sweep_input(layer)
    x = T.to_gpu(xb)
    for g in W.ROTATION_SWEEP_G:
        H = rotation(g)
        outs = {fmt: T.bf16_bits(mxq.mx_qdq(x, fmt, T.to_gpu(H))) for fmt in FMTS}
        st = T.check_rotated_multi(xb, H, qdq=outs)
        for v in st.values():
            assert v["exempt_blocks"] <= 0.01 * v["blocks"] + 2, (g, st)


def test_dependent_calls_keep_stream_order():
    """Every kernel is launched with programmatic stream serialization (it may be scheduled
    while the kernel before it finishes) and waits for that kernel before touching global
    memory. A chain of calls in which each reads what the one before wrote (and some overwrite
    what an earlier one read; GEMMs read codes written just before them and a QDQ reads a GEMM's
    output) gives the same bytes back to back, eagerly and in a CUDA graph, as with a
    synchronization after every call."""
    M, K = 4096, 8192
    x = T.to_gpu(W.rotation_sweep_input("attn_in", M, K))
    H = T.to_gpu(rotation(32))
    H128 = T.to_gpu(rotation(128))
    gs = torch.tensor([448.0 * 6 / 8.0], device="cuda")
    a, b, d = (torch.empty_like(x) for _ in range(3))
    c4, s4 = mxq.mx_rotate_quantize(x, H, mxq.E2M1, mxq.SWIZZLED)
    c8, s8 = mxq.mx_quantize(x, mxq.E4M3, mxq.LINEAR)
    cn, sn = mxq.mx_quantize_nvfp4(x, gs, mxq.SWIZZLED)
    small = torch.empty((8, K), dtype=torch.bfloat16, device="cuda")
    cs, ss = mxq.mx_rotate_quantize(x[:8], H, mxq.E2M1, mxq.SWIZZLED)
    # grouped calls: 8 experts of uneven sizes; the offsets are rewritten by a torch kernel in
    # the chain itself, so a grouped call's offset loads also depend on the launch before it
    counts = [700, 0, 1, 129, 2000, 300, 5, 961]
    off_src = torch.tensor(np.concatenate([[0], np.cumsum(counts)]), dtype=torch.int64,
                           device="cuda")
    offs = torch.zeros_like(off_src)
    gse = torch.full((len(counts),), 448.0 * 6 / 8.0, device="cuda")
    cg, sg = mxq.mx_quantize_grouped(x, off_src, mxq.E4M3, mxq.SWIZZLED)
    cgl, sgl = mxq.mx_quantize_grouped(x, off_src, mxq.E4M3, mxq.LINEAR)
    cng, sng = mxq.mx_quantize_nvfp4_grouped(x, off_src, gse, mxq.SWIZZLED)
    # GEMM consumers of codes written earlier in the chain; a QDQ then reads a GEMM's output
    cw, sw = mxq.mx_quantize(x[:512], mxq.E2M1, mxq.SWIZZLED)
    cw8, sw8 = mxq.mx_quantize(x[:256], mxq.E4M3, mxq.LINEAR)
    g1 = torch.empty((M, 512), dtype=torch.bfloat16, device="cuda")
    g2 = torch.empty_like(g1)
    g3 = torch.empty((M, 256), dtype=torch.bfloat16, device="cuda")
    outs = (a, b, d, c4, s4, c8, s8, cn, sn, small, cs, ss, offs, cg, sg, cgl, sgl, cng, sng,
            cw, sw, cw8, sw8, g1, g2, g3)

    def chain(sync):
        steps = [
            lambda: mxq.mx_qdq(x, mxq.E4M3, H128, y=a),
            lambda: mxq.mx_qdq(a, mxq.E2M1, y=b),
            lambda: mxq.mx_rotate_quantize(b, H, mxq.E2M1, mxq.SWIZZLED, codes=c4, scales=s4),
            lambda: mxq.mx_quantize(a[:512], mxq.E2M1, mxq.SWIZZLED, codes=cw, scales=sw),
            lambda: mxq.mx_gemm(c4, s4, cw, sw, K, mxq.E2M1, mxq.SWIZZLED, c=g1),
            lambda: mxq.mx_qdq(g1, mxq.E4M3, y=g2),
            lambda: mxq.mx_dequantize(c4, s4, K, mxq.E2M1, mxq.SWIZZLED, y=d),
            lambda: mxq.mx_qdq(d, mxq.E4M3, H, y=a),
            lambda: mxq.mx_quantize(a, mxq.E4M3, mxq.LINEAR, codes=c8, scales=s8),
            lambda: mxq.mx_quantize(d[:256], mxq.E4M3, mxq.LINEAR, codes=cw8, scales=sw8),
            lambda: mxq.mx_gemm(c8, s8, cw8, sw8, K, mxq.E4M3, mxq.LINEAR, c=g3),
            lambda: mxq.mx_dequantize(c8, s8, K, mxq.E4M3, mxq.LINEAR, y=b),
            lambda: mxq.mx_quantize_nvfp4(b, gs, mxq.SWIZZLED, codes=cn, scales=sn),
            lambda: mxq.mx_dequantize_nvfp4(cn, sn, K, gs, mxq.SWIZZLED, y=d),
            lambda: offs.copy_(off_src),
            lambda: mxq.mx_quantize_grouped(d, offs, mxq.E4M3, mxq.SWIZZLED, codes=cg, scales=sg),
            lambda: mxq.mx_quantize_grouped(d, offs, mxq.E4M3, mxq.LINEAR, codes=cgl, scales=sgl),
            lambda: mxq.mx_dequantize(cgl, sgl, K, mxq.E4M3, mxq.LINEAR, y=a),
            lambda: mxq.mx_quantize_nvfp4_grouped(a, offs, gse, mxq.SWIZZLED, codes=cng,
                                                  scales=sng),
            lambda: mxq.mx_qdq(d[:8], mxq.E2M1, H, y=small),
            lambda: mxq.mx_rotate_quantize(small, H, mxq.E2M1, mxq.SWIZZLED, codes=cs, scales=ss),
        ]
        for step in steps:
            step()
            if sync:
                torch.cuda.synchronize()

    chain(True)
    want = [t.clone() for t in outs]
    for t in outs:
        t.zero_()
    chain(False)
    torch.cuda.synchronize()
    for got, ref in zip(outs, want):
        assert torch.equal(got.view(torch.uint8), ref.view(torch.uint8))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        chain(False)
    for t in outs:
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    for got, ref in zip(outs, want):
        assert torch.equal(got.view(torch.uint8), ref.view(torch.uint8))
    assert mxq.mx_device_errors() == 0


def test_bounded_wait_gives_up_and_reports():
    """Failure detection without a fault: a wait that nothing completes (the tensor-core
    kernel's bounded-wait routine, 1 ms limit) gives up, the device error word reports it once
    (reading clears it), and the context still computes correct results afterwards."""
    assert mxq.mx_device_errors() == 0
    mxq.mx_selftest_bounded_wait(1_000_000)
    assert mxq.mx_device_errors() == 1
    assert mxq.mx_device_errors() == 0
    xb = W.rotate_quant_activation(256, 1024, stream=77)
    H = rotation(32, "identity")
    np.testing.assert_array_equal(qdq(xb, O.E2M1, H), O.qdq(xb, O.E2M1))
    assert mxq.mx_device_errors() == 0


def test_rotate_kernel_give_up_drains_and_reports():
    """Failure detection in the tensor-core kernel itself, without a fault: every mbarrier wait
    of a rotate+quantize call limited to 1 ns, 20 us and 1 ms (x[4096, 8192], 1024 tiles over
    the persistent CTAs) runs out while the pipeline is busy. Each call still ends (no role
    issues more work once its wait ran out, and loads, MMAs and stores in flight are waited
    for before tensor memory is freed), the error word reports the give-up at least for the
    1 ns limit, and afterwards the same context computes correct results."""
    assert mxq.mx_device_errors() == 0
    xb = W.rotate_quant_activation(4096, 8192, stream=79)
    x, H = T.to_gpu(xb), T.to_gpu(rotation(32))
    for limit in (1, 20_000, 1_000_000):
        mxq.mx_selftest_rotate_give_up(x, H, limit)
        errors = mxq.mx_device_errors()  # synchronizes: the call has ended
        assert errors in (0, 1)
        if limit == 1:
            assert errors == 1
    xs = W.rotate_quant_activation(256, 1024, stream=80)
    Hi = rotation(32, "identity")
    np.testing.assert_array_equal(qdq(xs, O.E2M1, Hi), O.qdq(xs, O.E2M1))
    c, s = mxq.mx_rotate_quantize(T.to_gpu(xs), T.to_gpu(Hi), mxq.E4M3, mxq.SWIZZLED)
    rc, rs = O.quantize(xs, O.E4M3, O.SWIZZLED)
    np.testing.assert_array_equal(T.u8(c), rc)
    np.testing.assert_array_equal(T.u8(s), rs)
    assert mxq.mx_device_errors() == 0


def test_calls_capture_into_a_cuda_graph():
    """The entry points allocate and synchronize nothing, so they can be captured in a CUDA
    graph (the CuTe QDQ page's requirement); replays equal eager calls bit for bit."""
    xb = W.rotation_sweep_input("attn_in", 512, 2048)
    x = T.to_gpu(xb)
    H = T.to_gpu(rotation(32))
    xm, off = W.moe_quant(E=8, tokens=700, K=256)
    xg, offs = T.to_gpu(xm), torch.from_numpy(off).cuda()
    # warm up on a side stream (first calls set kernel attributes), then capture
    y = torch.empty_like(x)
    yr = torch.empty_like(x)
    c, s = mxq.mx_rotate_quantize(x, H, mxq.E2M1, mxq.SWIZZLED)
    cg, sg = mxq.mx_quantize_grouped(xg, offs, mxq.E4M3, mxq.SWIZZLED)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        mxq.mx_qdq(x, mxq.E2M1, y=y)
        mxq.mx_qdq(x, mxq.E4M3, H, y=yr)
        mxq.mx_rotate_quantize(x, H, mxq.E2M1, mxq.SWIZZLED, codes=c, scales=s)
        mxq.mx_quantize_grouped(xg, offs, mxq.E4M3, mxq.SWIZZLED, codes=cg, scales=sg)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (y, yr, c, s, cg, sg)]
    for t in (y, yr, c, s, cg, sg):
        t.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        mxq.mx_qdq(x, mxq.E2M1, y=y)
        mxq.mx_qdq(x, mxq.E4M3, H, y=yr)
        mxq.mx_rotate_quantize(x, H, mxq.E2M1, mxq.SWIZZLED, codes=c, scales=s)
        mxq.mx_quantize_grouped(xg, offs, mxq.E4M3, mxq.SWIZZLED, codes=cg, scales=sg)
    for _ in range(2):
        for t in (y, yr, c, s, cg, sg):
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for got, want in zip((y, yr, c, s, cg, sg), eager):
            assert torch.equal(got.view(torch.uint8), want.view(torch.uint8))
    np.testing.assert_array_equal(T.bf16_bits(y), O.qdq(xb, O.E2M1))
