"""GPU parity of the Hadamard-rotation path (rot_kind = ROT_HADAMARD: the streaming kernel with an
in-register fast Walsh-Hadamard transform) against the CPU oracle, through the C ABI.

The oracle rotates with the same bf16 matrix H by its definition (y = x_chunk * H in double),
so the rotated-path tolerance rules of mx_testlib apply unchanged: pre-quantization values
within 1e-5 of the chunk norm, codes different only next to rounding midpoints, scale bytes one
step off only next to the power of two that the step crosses. A matrix that is not a scaled
Sylvester Hadamard takes the kernel's dense fp32-FMA product instead; with H = I that product
is exact, so the results equal the plain path's bit for bit. With g = 128 the Hadamard-hinted
calls run on the tensor-core kernel (faster there), and the same tests hold for them.
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
HAD = mxq.ROT_HADAMARD
GUARD = 4096
CANARY = 0xA5
# ragged shapes per g: K a multiple of g (and of 32), M with partial warps and 128-row blocks
SHAPES = {16: [(1, 32), (3, 96), (129, 416), (300, 1024)],
          32: [(1, 32), (5, 160), (129, 416), (300, 1024)],
          64: [(1, 64), (3, 192), (129, 448), (300, 1024)],
          128: [(1, 128), (3, 384), (129, 640), (300, 1024)]}


@pytest.fixture(scope="module", autouse=True)
def built():
    __graft_entry__.build()
    yield
    assert mxq.mx_device_errors() == 0


def hadamard(g):
    return W.normalized_hadamard_bf16(g)


def guarded(nbytes):
    full = torch.full((nbytes + 2 * GUARD,), CANARY, dtype=torch.uint8, device="cuda")
    return full, full[GUARD:GUARD + nbytes]


def assert_guards(full, nbytes):
    f = full.cpu().numpy()
    assert (f[:GUARD] == CANARY).all() and (f[GUARD + nbytes:] == CANARY).all()


def within(stats):
    for v in (stats.values() if "blocks" not in stats else [stats]):
        assert v["exempt_blocks"] <= 0.01 * v["blocks"] + 2, stats


@pytest.mark.parametrize("g", [16, 32, 64, 128])
def test_hadamard_values_within_tolerance(g):
    """The fp32 values the Hadamard path quantizes (same device code, rotate_debug) agree with
    the oracle's x_chunk * H within 1e-5 of the chunk norm, on every shape."""
    H = hadamard(g)
    for M, K in SHAPES[g] + [(1000, 4096)]:
        xb = W.rotate_quant_activation(M, K, stream=g + 11)
        y = mxq.mx_rotate_debug(T.to_gpu(xb), T.to_gpu(H), rot_kind=HAD).cpu().numpy()
        assert T.check_rotated_values(y, O.rotate(xb, H), g) <= 1.0, (M, K)


@pytest.mark.parametrize("g", [16, 32, 64, 128])
def test_hadamard_rotate_quantize_and_qdq_rules(g):
    """Rotate + quantize (both formats, both layouts, swizzle pads zero, canary bands intact)
    and rotated QDQ on ragged shapes: every block under the rules."""
    H = hadamard(g)
    Hd = T.to_gpu(H)
    for M, K in SHAPES[g]:
        xb = W.rotate_quant_activation(M, K, stream=3 * g + M)
        x = T.to_gpu(xb)
        codes, qdqs = {}, {}
        for fmt in FMTS:
            for layout in LAYOUTS:
                rows, cols = mxq.mx_scales_shape(M, K, layout)
                nc = M * O.code_bytes_per_row(fmt, K)
                cfull, c = guarded(nc)
                sfull, s = guarded(rows * cols)
                mxq.mx_rotate_quantize(x, Hd, fmt, layout, codes=c, scales=s, rot_kind=HAD)
                c = T.u8(c).reshape(M, -1)
                s = T.u8(s).reshape(rows, cols)
                assert_guards(cfull, nc)
                assert_guards(sfull, rows * cols)
                if layout == O.SWIZZLED:
                    assert not T.swizzle_pads(s, M, K).any()
                    np.testing.assert_array_equal(T.unswizzle(s, M, K), codes[fmt][1])
                    np.testing.assert_array_equal(c, codes[fmt][0])
                else:
                    codes[fmt] = (c, s)
            yfull, ybytes = guarded(M * K * 2)
            mxq.mx_qdq(x, fmt, Hd, y=ybytes.view(torch.bfloat16).view(M, K), rot_kind=HAD)
            assert_guards(yfull, M * K * 2)
            qdqs[fmt] = T.u8(ybytes).view(np.uint16).reshape(M, K)
        within(T.check_rotated_multi(xb, H, codes=codes, qdq=qdqs))


@pytest.mark.parametrize("g", [16, 32, 64, 128])
def test_hadamard_nvfp4_rules(g):
    """Rotated NVFP4 quantize (both layouts) and QDQ on the Hadamard path under the NVFP4
    rules."""
    H = hadamard(g)
    Hd = T.to_gpu(H)
    gs = np.float32(448 * 6 / 8.0)
    gst = torch.tensor([float(gs)], device="cuda")
    for M, K in SHAPES[g]:
        xb = W.rotate_quant_activation(M, K, stream=5 * g + M)
        x = T.to_gpu(xb)
        c, s = mxq.mx_quantize_nvfp4(x, gst, mxq.SWIZZLED, Hd, rot_kind=HAD)
        s = T.u8(s)
        assert not T.swizzle_pads(s, M, 2 * K).any()
        cl, sl = mxq.mx_quantize_nvfp4(x, gst, mxq.LINEAR, Hd, rot_kind=HAD)
        np.testing.assert_array_equal(T.unswizzle(s, M, 2 * K), T.u8(sl))
        np.testing.assert_array_equal(T.u8(c), T.u8(cl))
        q = T.bf16_bits(mxq.mx_qdq_nvfp4(x, gst, Hd, rot_kind=HAD))
        within(T.check_rotated_multi(xb, H, nvfp4={gs: (T.u8(cl), T.u8(sl))},
                                     nvfp4_qdq={gs: q}))


@pytest.mark.parametrize("g", [16, 32, 64, 128])
def test_non_hadamard_matrix_takes_the_dense_product(g):
    """H that is not a scaled Sylvester matrix, passed with the Hadamard hint: the kernel sees
    it and computes the dense product. With H = I that product is exact in fp32, so codes,
    scales (both layouts) and QDQ equal the plain oracle's bit for bit (MX and NVFP4); a random
    H follows the rules; a Hadamard matrix with one entry's sign flipped too."""
    M, K = SHAPES[g][2]
    xb = W.mxfp8_linear_quant(M, K, stream=g + 77)
    x = T.to_gpu(xb)
    I = T.to_gpu(W.to_bf16_bits(np.eye(g)))
    for fmt in FMTS:
        for layout in LAYOUTS:
            c, s = mxq.mx_rotate_quantize(x, I, fmt, layout, rot_kind=HAD)
            rc, rs = O.quantize(xb, fmt, layout)
            np.testing.assert_array_equal(T.u8(s), rs)
            np.testing.assert_array_equal(T.u8(c), rc)
        np.testing.assert_array_equal(T.bf16_bits(mxq.mx_qdq(x, fmt, I, rot_kind=HAD)),
                                      O.qdq(xb, fmt))
    gs = np.float32(448 * 6) / np.float32(np.abs(W.bf16_bits_to_float(xb)).max())
    gst = torch.tensor([float(gs)], device="cuda")
    c, s = mxq.mx_quantize_nvfp4(x, gst, mxq.SWIZZLED, I, rot_kind=HAD)
    rc, rs = O.nvfp4_quantize(xb, gs, O.SWIZZLED)
    np.testing.assert_array_equal(T.u8(s), rs)
    np.testing.assert_array_equal(T.u8(c), rc)
    np.testing.assert_array_equal(T.bf16_bits(mxq.mx_qdq_nvfp4(x, gst, I, rot_kind=HAD)),
                                  O.nvfp4_qdq(xb, gs))
    rng = np.random.default_rng(g + 5)
    flipped = hadamard(g).copy()
    flipped[g // 2, g // 3] ^= 0x8000
    for Hn in (W.to_bf16_bits(rng.standard_normal((g, g)) / np.sqrt(g)), flipped):
        xr = W.rotate_quant_activation(M, K, stream=g + 78)
        xg, Hg = T.to_gpu(xr), T.to_gpu(Hn)
        y = mxq.mx_rotate_debug(xg, Hg, rot_kind=HAD).cpu().numpy()
        assert T.check_rotated_values(y, O.rotate(xr, Hn), g) <= 1.0
        codes = {fmt: (T.u8(mxq.mx_rotate_quantize(xg, Hg, fmt, mxq.LINEAR, rot_kind=HAD)[0]),
                       T.u8(mxq.mx_rotate_quantize(xg, Hg, fmt, mxq.LINEAR, rot_kind=HAD)[1]))
                 for fmt in FMTS}
        qdqs = {fmt: T.bf16_bits(mxq.mx_qdq(xg, fmt, Hg, rot_kind=HAD)) for fmt in FMTS}
        within(T.check_rotated_multi(xr, Hn, codes=codes, qdq=qdqs))


@pytest.mark.parametrize("g", [16, 32, 128])
def test_hadamard_nan_and_inf_inputs(g):
    """NaN and +-Inf inputs: every chunk holding one rotates to non-finite values, its blocks get
    scale byte 0xFF with the fill codes (QDQ 0x7FC0) as in the oracle; the rest follows the
    rules."""
    M, K = 40, 512
    v = np.random.default_rng(M * 10 + g).standard_normal((M, K)).astype(np.float32)
    v[0, 3], v[M - 1, 200], v[M // 2, 511] = np.nan, np.inf, -np.inf
    v[1, 130], v[1, 131] = np.inf, -np.inf
    xb = W.to_bf16_bits(v)
    H = hadamard(g)
    x, Hd = T.to_gpu(xb), T.to_gpu(H)
    for fmt in FMTS:
        c, s = mxq.mx_rotate_quantize(x, Hd, fmt, mxq.LINEAR, rot_kind=HAD)
        c, s = T.u8(c), T.u8(s)
        _, rs = O.rotate_quantize(xb, H, fmt, O.LINEAR)
        special = rs == 255
        assert special.any() and (s[special] == 255).all() and (s[~special] != 255).all()
        out = T.bf16_bits(mxq.mx_qdq(x, fmt, Hd, rot_kind=HAD))
        ref = O.rotate_qdq(xb, H, fmt)
        nan_ref = np.repeat(special, 32, axis=1)
        np.testing.assert_array_equal(out[nan_ref], ref[nan_ref])
        within(T.check_rotated_multi(xb, H, codes={fmt: (c, s)}, qdq={fmt: out}))


def test_hadamard_calls_keep_stream_order_and_capture():
    """Hadamard-path calls in a chain where each reads what the call before wrote (mixed with
    the tensor-core path and the plain kernels), back to back and in a CUDA graph, give the
    bytes of the same chain with a synchronization after every call."""
    M, K = 2048, 4096
    x = T.to_gpu(W.rotation_sweep_input("attn_in", M, K))
    H32, H128 = T.to_gpu(hadamard(32)), T.to_gpu(hadamard(128))
    a, b = torch.empty_like(x), torch.empty_like(x)
    c4, s4 = mxq.mx_rotate_quantize(x, H32, mxq.E2M1, mxq.SWIZZLED, rot_kind=HAD)
    c8, s8 = mxq.mx_rotate_quantize(x, H128, mxq.E4M3, mxq.LINEAR, rot_kind=HAD)
    outs = (a, b, c4, s4, c8, s8)

    def chain(sync):
        steps = [
            lambda: mxq.mx_qdq(x, mxq.E4M3, H128, y=a, rot_kind=HAD),
            lambda: mxq.mx_qdq(a, mxq.E2M1, H32, y=b),
            lambda: mxq.mx_rotate_quantize(b, H32, mxq.E2M1, mxq.SWIZZLED, codes=c4, scales=s4,
                                           rot_kind=HAD),
            lambda: mxq.mx_dequantize(c4, s4, K, mxq.E2M1, mxq.SWIZZLED, y=a),
            lambda: mxq.mx_rotate_quantize(a, H128, mxq.E4M3, mxq.LINEAR, codes=c8, scales=s8,
                                           rot_kind=HAD),
            lambda: mxq.mx_dequantize(c8, s8, K, mxq.E4M3, mxq.LINEAR, y=b),
            lambda: mxq.mx_qdq(b, mxq.E2M1, H128, y=a, rot_kind=HAD),
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


# ---------------------------------------------------------------------------------------------
# the workloads at full size, whole outputs
# ---------------------------------------------------------------------------------------------
@pytest.mark.parametrize("K", W.ROTATE_QUANT_K)
@pytest.mark.parametrize("M", W.ROTATE_QUANT_M)
def test_hadamard_rotate_quant_workload_grid(M, K):
    """The fused rotate + MXFP4 quantize workload (g = 32 normalized Hadamard, swizzled scales,
    rows padded to 128) at every (M, K) on the Hadamard path: every block under the rules."""
    xb = W.rotate_quant_activation(M, K)
    H = hadamard(32)
    c, s = mxq.mx_rotate_quantize(T.to_gpu(xb), T.to_gpu(H), mxq.E2M1, mxq.SWIZZLED, rot_kind=HAD)
    s = T.u8(s)
    assert not T.swizzle_pads(s, M, K).any()
    within(T.check_rotated_codes(xb, H, O.E2M1, T.u8(c), T.unswizzle(s, M, K)))


@pytest.mark.parametrize("layer", [n for n, _, _ in W.ROTATION_SWEEP_LAYERS])
def test_hadamard_rotation_sweep_full_size(layer):
    """The rotation-size sweep (every g, both formats, rotated QDQ) on each decoder-layer input
    at full size on the Hadamard path: every block under the rules."""
    xb = W.rotation_sweep_input(layer)
    x = T.to_gpu(xb)
    for g in W.ROTATION_SWEEP_G:
        H = hadamard(g)
        outs = {fmt: T.bf16_bits(mxq.mx_qdq(x, fmt, T.to_gpu(H), rot_kind=HAD)) for fmt in FMTS}
        within(T.check_rotated_multi(xb, H, qdq=outs))


def test_hadamard_weight_and_nvfp4_full_size():
    """The 70B weight [8192, 28672] rotate + quantize at g = 32 and 128 (both formats, swizzled)
    and rotate(g = 16) + NVFP4 quantize / QDQ of x[8192, 28672] on the Hadamard path."""
    N, K = 8192, 28672
    xb = W.weight_rotate_quant(N, K)
    x = T.to_gpu(xb)
    for g in (32, 128):
        H = hadamard(g)
        outs = {}
        for fmt in FMTS:
            c, s = mxq.mx_rotate_quantize(x, T.to_gpu(H), fmt, mxq.SWIZZLED, rot_kind=HAD)
            s = T.u8(s)
            assert not T.swizzle_pads(s, N, K).any()
            outs[fmt] = (T.u8(c), T.unswizzle(s, N, K))
        within(T.check_rotated_multi(xb, H, codes=outs))
    xa = W.rotate_quant_activation(8192, 28672)
    xg = T.to_gpu(xa)
    H = hadamard(16)
    gs = np.float32(448 * 6 / 8.0)
    gst = torch.tensor([float(gs)], device="cuda")
    c, s = mxq.mx_quantize_nvfp4(xg, gst, mxq.SWIZZLED, T.to_gpu(H), rot_kind=HAD)
    q = T.bf16_bits(mxq.mx_qdq_nvfp4(xg, gst, T.to_gpu(H), rot_kind=HAD))
    within(T.check_rotated_multi(xa, H, nvfp4={gs: (T.u8(c), T.unswizzle(T.u8(s), 8192, 2 * 28672))},
                                 nvfp4_qdq={gs: q}))


# (what, fmt, M, K, g, kernel ROT_AUTO must take)
AUTO_CASES = [
    ("codes", O.E2M1, 1, 8192, 32, "dense"),        # decode-sized: FMA kernel
    ("codes", O.E2M1, 1024, 8192, 32, "hadamard"),  # below 4096 rows
    ("codes", O.E2M1, 4096, 8192, 32, "dense"),     # 4-bit codes from 4096 rows
    ("codes", O.E4M3, 4096, 8192, 32, "dense"),     # wide output, M * K <= 3 * 2^25
    ("codes", O.E4M3, 4096, 32768, 64, "hadamard"),  # wide output above it
    ("qdq", O.E2M1, 4096, 8192, 16, "dense"),
    ("qdq", O.E4M3, 4096, 28672, 32, "hadamard"),
    ("codes", O.E2M1, 1024, 8192, 128, "dense"),    # g = 128: tensor cores
    ("nvfp4", None, 4096, 8192, 16, "dense"),
    ("nvfp4", None, 1024, 8192, 16, "hadamard"),
    ("quest", O.E2M1, 4096, 8192, 32, "dense"),
]


@pytest.mark.parametrize("case", AUTO_CASES, ids=lambda c: f"{c[0]}-{c[1]}-{c[2]}x{c[3]}-g{c[4]}")
def test_rot_auto_takes_the_faster_kernel_of_the_table(case):
    """ROT_AUTO gives exactly the output of the kernel its table names for the call. The two
    kernels round the rotation differently, so on these sizes their codes or QDQ outputs differ in
    a few blocks next to rounding midpoints; where they happen to agree the case still checks that
    ROT_AUTO computes a correct result."""
    what, fmt, M, K, g, want = case
    x = T.to_gpu(W.rotate_quant_activation(M, K, stream=g))
    H = T.to_gpu(W.normalized_hadamard_bf16(g))
    gs = torch.tensor([448.0 * 6.0 / 8.0], device="cuda")

    def run(rk):
        if what == "codes":
            c, s = mxq.mx_rotate_quantize(x, H, fmt, mxq.SWIZZLED, rot_kind=rk)
            return torch.cat([c.view(-1), s.view(-1)])
        if what == "quest":
            c, s = mxq.mx_rotate_quantize(x, H, fmt, mxq.SWIZZLED, rot_kind=rk, rounding=mxq.QUEST)
            return torch.cat([c.view(-1), s.view(-1)])
        if what == "qdq":
            return mxq.mx_qdq(x, fmt, H, rot_kind=rk).view(torch.uint8).view(-1)
        c, s = mxq.mx_quantize_nvfp4(x, gs, mxq.SWIZZLED, H, rot_kind=rk)
        return torch.cat([c.view(-1), s.view(-1)])

    auto = run(mxq.ROT_AUTO)
    ref = run(mxq.ROT_DENSE if want == "dense" else mxq.ROT_HADAMARD)
    assert torch.equal(auto, ref)
