"""GPU parity of the block-scaled GEMM consumer (mx_gemm: C = alpha * dequant(A) @ dequant(B)^T,
bf16 out) against the oracle's definition (dequantize, then a float64 matmul), through the C ABI.

Tolerance, from the arithmetic: the operands are the bf16 dequantized values (exact for the
inputs used here), their products are exact in fp32, and the tensor cores add them in fp32 in an
order of their own; each of the K additions errs by at most 2^-23 of a partial sum, and a partial
sum is at most S = sum_k |a_k b_k|, so the fp32 value is within K * 2^-23 * |alpha| * S of the
exact one; rounding it to bf16 adds at most 2^-8 of its magnitude. Hence
|C_gpu - C_ref| <= 2^-8 |C_ref| + (1 + 2^-8) K 2^-23 |alpha| S (+ the smallest bf16 subnormal),
where S is taken exactly on the small shapes and bounded by ||a_i|| ||b_j|| (Cauchy-Schwarz) at
full size. Where one side of the product is an identity matrix each entry of C is one exact
product, so there C must equal the dequantized operand bit for bit (zero signs aside).
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
FMTS = [O.E2M1, O.E4M3]
LAYOUTS = [O.LINEAR, O.SWIZZLED]
GUARD = 4096
CANARY = 0x5A
BF16_MIN_SUB = 2.0 ** -133
# (M, N, K): one tile, ragged rows and columns (N % 8 == 0), several K steps and tiles (these
# take the kernel's 128 x 64 tiles; test_gemm_wide_tiles_ragged and the full-size tests its
# 128 x 256 tiles)
SHAPES = [(1, 8, 64), (3, 16, 128), (128, 128, 64), (129, 136, 192), (300, 264, 1024),
          (257, 520, 4096)]


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()
    yield
    assert mxq.mx_device_errors() == 0


def random_operand(rng, rows, K, fmt, layout, lo=120, hi=135):
    """Random MX codes (E4M3 NaN codes excluded) and scale bytes in [lo, hi) in the stored
    layout; swizzled pads hold random bytes too (never read)."""
    codes = rng.integers(0, 256, (rows, O.code_bytes_per_row(fmt, K)), dtype=np.uint8)
    if fmt == O.E4M3:
        codes[(codes & 0x7F) == 0x7F] ^= 0x01
    scales = rng.integers(lo, hi, O.scales_shape(rows, K, layout), dtype=np.uint8)
    return codes, scales


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def bf16_to_f64(t):
    return O.bf16_bits_to_double(T.bf16_bits(t))


def gemm_tolerance(C_ref, K, alpha, S):
    acc = K * 2.0 ** -23 * abs(alpha) * S
    return 2.0 ** -8 * np.abs(C_ref) + (1 + 2.0 ** -8) * acc + BF16_MIN_SUB


def assert_gemm_close(C_gpu, C_ref, tol, what):
    bad = ~(np.abs(C_gpu - C_ref) <= tol)
    if bad.any():
        i, j = np.argwhere(bad)[0]
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} entries out of tolerance; "
                             f"first [{i}, {j}] gpu {C_gpu[i, j]!r} ref {C_ref[i, j]!r} "
                             f"tol {tol[i, j]!r}")


def exact_S(a_codes, a_scales, b_codes, b_scales, K, fmt, layout):
    da = O.bf16_bits_to_double(O.dequantize(a_codes, a_scales, K, fmt, layout))
    db = O.bf16_bits_to_double(O.dequantize(b_codes, b_scales, K, fmt, layout))
    return np.abs(da) @ np.abs(db).T


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "x".join(map(str, s)))
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("fmt", FMTS)
def test_gemm_random_codes(fmt, layout, shape):
    M, N, K = shape
    rng = np.random.default_rng(M * 7 + N * 3 + K + 11 * fmt + layout)
    a, sa = random_operand(rng, M, K, fmt, layout)
    b, sb = random_operand(rng, N, K, fmt, layout)
    alpha = 1.0
    full = torch.full((M * N * 2 + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
    c = full[GUARD:GUARD + M * N * 2].view(torch.bfloat16).view(M, N)
    mxq.mx_gemm(dev(a), dev(sa), dev(b), dev(sb), K, fmt, layout, alpha, c=c)
    C_gpu = bf16_to_f64(c)
    C_ref = O.gemm(a, sa, b, sb, K, fmt, layout, alpha)
    S = exact_S(a, sa, b, sb, K, fmt, layout)
    assert_gemm_close(C_gpu, C_ref, gemm_tolerance(C_ref, K, alpha, S), "C")
    f = full.cpu().numpy()
    assert (f[:GUARD] == CANARY).all() and (f[GUARD + M * N * 2:] == CANARY).all()


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("fmt", FMTS)
def test_gemm_wide_tiles_ragged(fmt, layout):
    """A problem with enough 128 x 256 tiles to fill the SMs (so the kernel takes its wide
    tiles; most small shapes above take 128 x 64 tiles), ragged in M and N, inside canaries;
    random scale bytes partly outside the f16 window in one row block (bf16 operands there)."""
    M, N, K = 641, 7944, 256
    rng = np.random.default_rng(5 + fmt + 2 * layout)
    a, sa = random_operand(rng, M, K, fmt, layout)
    b, sb = random_operand(rng, N, K, fmt, layout)
    la = T.unswizzle(sa, M, K) if layout == O.SWIZZLED else sa
    la[300:310] = 150
    if layout == O.SWIZZLED:
        sa = swizzle(la, M, K)
    full = torch.full((M * N * 2 + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
    c = full[GUARD:GUARD + M * N * 2].view(torch.bfloat16).view(M, N)
    mxq.mx_gemm(dev(a), dev(sa), dev(b), dev(sb), K, fmt, layout, 0.75, c=c)
    C_ref = O.gemm(a, sa, b, sb, K, fmt, layout, 0.75)
    S = exact_S(a, sa, b, sb, K, fmt, layout)
    assert_gemm_close(bf16_to_f64(c), C_ref, gemm_tolerance(C_ref, K, 0.75, S), "C")
    f = full.cpu().numpy()
    assert (f[:GUARD] == CANARY).all() and (f[GUARD + M * N * 2:] == CANARY).all()


@pytest.mark.parametrize("alpha", [0.5, -3.0, 1.0 / 3.0])
@pytest.mark.parametrize("fmt", FMTS)
def test_gemm_alpha(fmt, alpha):
    M, N, K = 200, 136, 512
    rng = np.random.default_rng(int(abs(alpha) * 1000) + fmt)
    a, sa = random_operand(rng, M, K, fmt, O.SWIZZLED)
    b, sb = random_operand(rng, N, K, fmt, O.SWIZZLED)
    C_gpu = bf16_to_f64(mxq.mx_gemm(dev(a), dev(sa), dev(b), dev(sb), K, fmt, O.SWIZZLED, alpha))
    C_ref = O.gemm(a, sa, b, sb, K, fmt, O.SWIZZLED, alpha)
    S = exact_S(a, sa, b, sb, K, fmt, O.SWIZZLED)
    assert_gemm_close(C_gpu, C_ref, gemm_tolerance(C_ref, K, alpha, S), f"alpha {alpha}")


def identity_operand(n, fmt, layout):
    """Codes of the n x n identity (1.0 on the diagonal, 0 elsewhere) under scale byte 127."""
    one = 0x2 if fmt == O.E2M1 else 0x38
    codes = np.zeros((n, O.code_bytes_per_row(fmt, n)), dtype=np.uint8)
    for i in range(n):
        if fmt == O.E4M3:
            codes[i, i] = one
        else:
            codes[i, i // 2] = one << (4 * (i % 2))
    scales = np.full(O.scales_shape(n, n, layout), 127, dtype=np.uint8)
    return codes, scales


def zero_sign_free(bits):
    bits = bits.copy()
    bits[bits == 0x8000] = 0
    return bits


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("M,K", [(300, 1024), (128, 8192)])
def test_gemm_times_identity_is_the_dequantized_operand(fmt, layout, M, K):
    """A @ I^T and I @ B^T: each entry is one exact product, so C equals the oracle's
    dequantize of the other operand bit for bit. Scale bytes 0..239 (subnormal bf16 results
    included; no value overflows, since an infinity times a zero of the identity is NaN)."""
    rng = np.random.default_rng(K + M + fmt)
    a, sa = random_operand(rng, M, K, fmt, layout, lo=0, hi=240)
    ident, si = identity_operand(K, fmt, layout)
    want = zero_sign_free(O.dequantize(a, sa, K, fmt, layout))
    c1 = mxq.mx_gemm(dev(a), dev(sa), dev(ident), dev(si), K, fmt, layout)
    np.testing.assert_array_equal(zero_sign_free(T.bf16_bits(c1)), want)
    if M % 8 == 0:
        c2 = mxq.mx_gemm(dev(ident), dev(si), dev(a), dev(sa), K, fmt, layout)
        np.testing.assert_array_equal(zero_sign_free(T.bf16_bits(c2)), want.T)


# scale-byte windows in which every dequantized value is exact in f16 (the kernel then uses f16
# operands; outside, bf16 operands, with a second multiply above 2^15)
F16_WINDOW = {O.E2M1: (104, 140), O.E4M3: (112, 134)}


@pytest.mark.parametrize("where", ["inside", "edges", "below", "above", "some_rows"])
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("fmt", FMTS)
def test_gemm_scale_ranges(fmt, layout, where):
    """Scale bytes inside the f16 window, on its edges, below it, above it (X up to 32), and
    outside it in a few rows only (one CTA row block takes bf16 operands, the others f16)."""
    M, N, K = 300, 264, 640
    lo, hi = F16_WINDOW[fmt]
    kinds = ["inside", "edges", "below", "above", "some_rows"]
    rng = np.random.default_rng(100 * fmt + 10 * layout + kinds.index(where))
    ranges = {"inside": (lo, hi + 1), "edges": (lo, hi + 1), "below": (lo - 20, lo + 2),
              "above": (hi - 2, 160), "some_rows": (lo, hi + 1)}
    a, sa = random_operand(rng, M, K, fmt, layout, *ranges[where])
    b, sb = random_operand(rng, N, K, fmt, layout, *ranges[where])
    if where in ("edges", "some_rows"):
        la = T.unswizzle(sa, M, K) if layout == O.SWIZZLED else sa
        lb = T.unswizzle(sb, N, K) if layout == O.SWIZZLED else sb
        if where == "edges":
            la[::2, ::3] = lo
            la[1::2, ::3] = hi
            lb[::3, 1::2] = hi
        else:
            la[200:210] = rng.integers(hi + 1, hi + 20, la[200:210].shape)
        if layout == O.SWIZZLED:
            sa = swizzle(la, M, K)
            sb = swizzle(lb, N, K)
    C_gpu = bf16_to_f64(mxq.mx_gemm(dev(a), dev(sa), dev(b), dev(sb), K, fmt, layout))
    C_ref = O.gemm(a, sa, b, sb, K, fmt, layout)
    S = exact_S(a, sa, b, sb, K, fmt, layout)
    assert_gemm_close(C_gpu, C_ref, gemm_tolerance(C_ref, K, 1.0, S), where)


def swizzle(lin, rows, K):
    """Linear [rows, K/32] scale bytes -> the swizzled layout (pads 0), by the oracle's offset."""
    shape = O.scales_shape(rows, K, O.SWIZZLED)
    out = np.zeros(shape, dtype=np.uint8).reshape(-1)
    r, c = np.meshgrid(np.arange(rows), np.arange(K // 32), indexing="ij")
    off = np.vectorize(O.swizzled_offset)(r, c, shape[1])
    out[off.reshape(-1)] = lin.reshape(-1)
    return out.reshape(shape)


@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("fmt", FMTS)
def test_gemm_times_identity_inside_the_f16_window(fmt, layout):
    """The identity product with every scale byte inside the f16 window (f16 operands): C equals
    the oracle's dequantize bit for bit."""
    M, K = 256, 1024
    lo, hi = F16_WINDOW[fmt]
    rng = np.random.default_rng(77 + fmt + 3 * layout)
    a, sa = random_operand(rng, M, K, fmt, layout, lo=lo, hi=hi + 1)
    if layout == O.SWIZZLED:  # pads inside the window too, though never read
        sa[:] = np.where(sa == 0, lo, sa)
    ident, si = identity_operand(K, fmt, layout)
    want = zero_sign_free(O.dequantize(a, sa, K, fmt, layout))
    c1 = mxq.mx_gemm(dev(a), dev(sa), dev(ident), dev(si), K, fmt, layout)
    np.testing.assert_array_equal(zero_sign_free(T.bf16_bits(c1)), want)
    c2 = mxq.mx_gemm(dev(ident), dev(si), dev(a), dev(sa), K, fmt, layout)
    np.testing.assert_array_equal(zero_sign_free(T.bf16_bits(c2)), want.T)


def identity_operand_fast(n, fmt, layout):
    """identity_operand built with array indexing (n = 8192 in the wide-tile tests)."""
    codes = np.zeros((n, O.code_bytes_per_row(fmt, n)), dtype=np.uint8)
    i = np.arange(n)
    if fmt == O.E4M3:
        codes[i, i] = 0x38
    else:
        codes[i, i // 2] = np.where(i % 2 == 0, 0x02, 0x20)
    return codes, np.full(O.scales_shape(n, n, layout), 127, dtype=np.uint8)


@pytest.mark.parametrize("window", ["bf16", "f16"])
@pytest.mark.parametrize("layout", LAYOUTS)
@pytest.mark.parametrize("fmt", FMTS)
def test_gemm_times_identity_wide_tiles(fmt, layout, window):
    """The identity products at a size that takes the 128 x 256 tiles (A [640, 8192] against
    the 8192 x 8192 identity, both operand orders): bit-exact against the oracle's dequantize,
    with scale bytes 0..239 (bf16 operands) or inside the f16 window (f16 operands)."""
    M, K = 640, 8192
    rng = np.random.default_rng(11 + fmt + 2 * layout + (window == "f16"))
    lo, hi = (0, 240) if window == "bf16" else (F16_WINDOW[fmt][0], F16_WINDOW[fmt][1] + 1)
    a, sa = random_operand(rng, M, K, fmt, layout, lo=lo, hi=hi)
    if layout == O.SWIZZLED and window == "f16":
        sa[:] = np.where(sa == 0, lo, sa)
    ident, si = identity_operand_fast(K, fmt, layout)
    want = zero_sign_free(O.dequantize(a, sa, K, fmt, layout))
    ga, gsa, gi, gsi = dev(a), dev(sa), dev(ident), dev(si)
    c1 = mxq.mx_gemm(ga, gsa, gi, gsi, K, fmt, layout)
    np.testing.assert_array_equal(zero_sign_free(T.bf16_bits(c1)), want)
    c2 = mxq.mx_gemm(gi, gsi, ga, gsa, K, fmt, layout)
    np.testing.assert_array_equal(zero_sign_free(T.bf16_bits(c2)), want.T)


@pytest.mark.parametrize("fmt", FMTS)
def test_gemm_nan_scale_poisons_its_rows_and_columns(fmt):
    M, N, K = 160, 144, 256
    rng = np.random.default_rng(3 + fmt)
    a, sa = random_operand(rng, M, K, fmt, O.LINEAR)
    b, sb = random_operand(rng, N, K, fmt, O.LINEAR)
    sa[17, 3] = 255
    sb[130, 0] = 255
    C_gpu = bf16_to_f64(mxq.mx_gemm(dev(a), dev(sa), dev(b), dev(sb), K, fmt, O.LINEAR))
    nan = np.zeros((M, N), dtype=bool)
    nan[17, :] = True
    nan[:, 130] = True
    np.testing.assert_array_equal(np.isnan(C_gpu), nan)
    C_ref = O.gemm(a, sa, b, sb, K, fmt, O.LINEAR)
    assert np.isnan(C_ref[nan]).all()
    S = exact_S(a, sa, b, sb, K, fmt, O.LINEAR)
    tol = gemm_tolerance(C_ref, K, 1.0, S)
    assert_gemm_close(np.where(nan, 0, C_gpu), np.where(nan, 0, C_ref), np.where(nan, 1, tol), "C")


@pytest.mark.parametrize("limit_ns", [1, 20_000, 1_000_000])
def test_gemm_give_up_drains_and_reports(limit_ns):
    """Failure detection without a fault: the GEMM with every pipeline wait limited to a few
    ns .. 1 ms. Each call ends; the 1 ns call reports the give-up in the device error word;
    the same context then computes a GEMM equal (within tolerance) to the oracle's."""
    M, N, K = 2048, 4096, 4096
    rng = np.random.default_rng(limit_ns)
    a, sa = random_operand(rng, M, K, O.E2M1, O.SWIZZLED)
    b, sb = random_operand(rng, N, K, O.E2M1, O.SWIZZLED)
    ga, gsa, gb, gsb = dev(a), dev(sa), dev(b), dev(sb)
    assert mxq.mx_device_errors() == 0
    mxq.mx_selftest_gemm_give_up(ga, gsa, gb, gsb, K, O.E2M1, O.SWIZZLED, limit_ns)
    torch.cuda.synchronize()
    flags = mxq.mx_device_errors()
    if limit_ns == 1:
        assert flags == 1
    assert flags in (0, 1)
    # the context still computes: a small GEMM against the oracle
    m, n, k = 130, 264, 512
    a2, sa2 = random_operand(rng, m, k, O.E4M3, O.LINEAR)
    b2, sb2 = random_operand(rng, n, k, O.E4M3, O.LINEAR)
    C_gpu = bf16_to_f64(mxq.mx_gemm(dev(a2), dev(sa2), dev(b2), dev(sb2), k, O.E4M3, O.LINEAR))
    C_ref = O.gemm(a2, sa2, b2, sb2, k, O.E4M3, O.LINEAR)
    S = exact_S(a2, sa2, b2, sb2, k, O.E4M3, O.LINEAR)
    assert_gemm_close(C_gpu, C_ref, gemm_tolerance(C_ref, k, 1.0, S), "after give-up")
    assert mxq.mx_device_errors() == 0


def test_gemm_empty_calls():
    u = torch.zeros(1024, dtype=torch.uint8, device="cuda")
    c = mxq.mx_gemm(u[:0], u, u[:256].view(8, 32), u, 64, O.E2M1, O.LINEAR)
    assert c.shape == (0, 8)
    c = mxq.mx_gemm(u[:32].view(1, 32), u, u[:0], u, 64, O.E2M1, O.LINEAR)
    assert c.shape == (1, 0)


@pytest.mark.parametrize("fmt", FMTS)
def test_gemm_of_quantized_operands_in_a_graph(fmt):
    """The consumer on the quantizer's outputs (quantize activations and weights, then the GEMM)
    on a side stream and captured in a CUDA graph: the replay equals the eager run bit for bit,
    the codes equal the oracle's, and C is within tolerance of the oracle's GEMM of those codes."""
    M, N, K = 257, 392, 2048
    xa = W.mxfp4_qdq_activation(M, K)
    xw = W.mxfp4_qdq_weight(N, K)
    ga, gw = T.to_gpu(xa), T.to_gpu(xw)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ca, sa = mxq.mx_quantize(ga, fmt, O.SWIZZLED, stream=s)
        cw, sw = mxq.mx_quantize(gw, fmt, O.SWIZZLED, stream=s)
        c_eager = mxq.mx_gemm(ca, sa, cw, sw, K, fmt, O.SWIZZLED, 0.25, stream=s).clone()
    torch.cuda.current_stream().wait_stream(s)
    ref_a, ref_sa = O.quantize(xa, fmt, O.SWIZZLED)
    ref_w, ref_sw = O.quantize(xw, fmt, O.SWIZZLED)
    np.testing.assert_array_equal(T.u8(ca), ref_a)
    np.testing.assert_array_equal(T.u8(sa), ref_sa)
    np.testing.assert_array_equal(T.u8(cw), ref_w)
    np.testing.assert_array_equal(T.u8(sw), ref_sw)
    C_ref = O.gemm(ref_a, ref_sa, ref_w, ref_sw, K, fmt, O.SWIZZLED, 0.25)
    S = exact_S(ref_a, ref_sa, ref_w, ref_sw, K, fmt, O.SWIZZLED)
    assert_gemm_close(bf16_to_f64(c_eager), C_ref, gemm_tolerance(C_ref, K, 0.25, S), "eager")

    c = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        qa, qsa = mxq.mx_quantize(ga, fmt, O.SWIZZLED, stream=s)
        qw, qsw = mxq.mx_quantize(gw, fmt, O.SWIZZLED, stream=s)
        mxq.mx_gemm(qa, qsa, qw, qsw, K, fmt, O.SWIZZLED, 0.25, c=c, stream=s)
    for _ in range(3):
        c.fill_(0)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(c.view(torch.int16), c_eager.view(torch.int16))


# full-size layer shapes of the activation / weight workloads (Llama-2-70B-like)
FULL = [("o_proj", 4096, 8192, 8192), ("down_proj", 1024, 8192, 28672)]


@pytest.mark.parametrize("case", FULL, ids=lambda c: c[0])
@pytest.mark.parametrize("fmt", FMTS)
def test_gemm_full_size(fmt, case):
    """Every entry of C at full size: activations [M, K] and weights [N, K] quantized (codes
    checked against the oracle on sampled row ranges elsewhere; here their bytes are the
    oracle's by the quantizer's bit-exact tests), swizzled scales, alpha 1."""
    _, M, N, K = case
    xa = W.mxfp4_qdq_activation(M, K)
    xw = W.weight_rotate_quant(N, K)
    ca, sa = mxq.mx_quantize(T.to_gpu(xa), fmt, O.SWIZZLED)
    cw, sw = mxq.mx_quantize(T.to_gpu(xw), fmt, O.SWIZZLED)
    C_gpu = bf16_to_f64(mxq.mx_gemm(ca, sa, cw, sw, K, fmt, O.SWIZZLED))
    ref_a, ref_sa = O.quantize(xa, fmt, O.SWIZZLED)
    ref_w, ref_sw = O.quantize(xw, fmt, O.SWIZZLED)
    assert np.array_equal(T.u8(ca), ref_a) and np.array_equal(T.u8(cw), ref_w)
    assert np.array_equal(T.u8(sa), ref_sa) and np.array_equal(T.u8(sw), ref_sw)
    da = O.bf16_bits_to_double(O.dequantize(ref_a, ref_sa, K, fmt, O.SWIZZLED))
    db = O.bf16_bits_to_double(O.dequantize(ref_w, ref_sw, K, fmt, O.SWIZZLED))
    C_ref = da @ db.T
    S = np.outer(np.linalg.norm(da, axis=1), np.linalg.norm(db, axis=1))  # >= sum |a b|
    assert_gemm_close(C_gpu, C_ref, gemm_tolerance(C_ref, K, 1.0, S), "C")
    # the bound is loose at this K; the typical error must be far inside it
    assert np.median(np.abs(C_gpu - C_ref) / (np.abs(C_ref) + 1e-30)) < 2.0 ** -9
