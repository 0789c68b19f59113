"""Test helpers: device transfer of bf16 bit patterns, layout conversions written independently
of both the kernels and the oracle, exhaustive converter sweeps, and the tolerance rules for the
rotated path.

Rotated-path tolerance (the rotation is computed in fp32 on the tensor cores, the oracle in
double): for an element in rotation chunk c, tol = 1e-5 * ||y_ref chunk c||_2 (normwise relative,
the bound fp32 accumulation obeys). A code may differ from the oracle's only if the oracle's
scaled value t = y_ref / 2^s lies within tol / 2^s of the midpoint between the two codes' values
and the two values are neighbours on the grid. A block's scale byte may differ by one only if
the oracle's abs-max lies within the block's largest tol of a power of two; the block is then
re-quantized by the oracle under the GPU's scale and held to the same element rule.
"""

from __future__ import annotations

import concurrent.futures
import os

import numpy as np
import torch

import oracle as O
from mx_microscaling_quantize_gb300 import workloads as W


# ---------------------------------------------------------------------------------------------
# transfers
# ---------------------------------------------------------------------------------------------
def to_gpu(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).to(device).view(
        torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def u8(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


# ---------------------------------------------------------------------------------------------
# layouts
# ---------------------------------------------------------------------------------------------
def unswizzle(swz: np.ndarray, M: int, K: int) -> np.ndarray:
    """128x4 blocked scales -> linear [M, K/32] (pads dropped), by reshapes."""
    C = K // 32
    Cp = -(-C // 4) * 4
    R = -(-M // 128) * 128
    t = swz.reshape(R // 128, Cp // 4, 32, 4, 4)       # [rb, cb, r%32, r//32, c%4]
    t = t.transpose(0, 3, 2, 1, 4).reshape(R, Cp)       # row = rb*128 + (r//32)*32 + r%32
    return t[:M, :C]


def swizzle_pads(swz: np.ndarray, M: int, K: int) -> np.ndarray:
    """The pad bytes of a blocked scale buffer (rows >= M or columns >= K/32)."""
    C = K // 32
    Cp = -(-C // 4) * 4
    R = -(-M // 128) * 128
    t = swz.reshape(R // 128, Cp // 4, 32, 4, 4).transpose(0, 3, 2, 1, 4).reshape(R, Cp)
    mask = np.ones((R, Cp), dtype=bool)
    mask[:M, :C] = False
    return t[mask]


def unpack_codes(codes: np.ndarray, fmt: int) -> np.ndarray:
    """Per-element codes [M, K] from packed codes."""
    if fmt == O.E4M3:
        return codes
    out = np.empty((codes.shape[0], codes.shape[1] * 2), dtype=np.uint8)
    out[:, 0::2] = codes & 0xF
    out[:, 1::2] = codes >> 4
    return out


# ---------------------------------------------------------------------------------------------
# exhaustive converter sweep
# ---------------------------------------------------------------------------------------------
def finite_bf16() -> np.ndarray:
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    return b[((b >> 7) & 0xFF) != 0xFF]


def converter_sweep(K: int = 2048) -> np.ndarray:
    """bf16 bits [rows, K]: (1) one block per finite bf16 value v, holding v and zeros, so that
    every value sets its own scale; (2) for every anchor exponent A in [-133, 127], blocks
    [+-2^A, v_1..v_31] over every finite v with |v| <= 2^A, so that every value meets every
    scale at or above its own (all s in [-127, 125])."""
    fin = finite_bf16()
    mag = fin & 0x7FFF
    blocks = []
    own = np.zeros((fin.size, 32), dtype=np.uint16)
    own[:, 5] = fin
    blocks.append(own)
    for A in range(-133, 128):
        anchor = W.to_bf16_bits(np.array([2.0 ** A], dtype=np.float64).astype(np.float32))[0]
        if A < -126:  # 2^A is a bf16 subnormal; float32 holds it exactly too
            anchor = np.uint16(1 << (A + 133))
        vals = fin[mag <= anchor]
        n = -(-vals.size // 31)
        pad = np.zeros(n * 31, dtype=np.uint16)
        pad[:vals.size] = vals
        b = np.empty((n, 32), dtype=np.uint16)
        b[:, 0] = anchor | np.where(np.arange(n) % 2 == 1, 0x8000, 0).astype(np.uint16)
        b[:, 1:] = pad.reshape(n, 31)
        blocks.append(b)
    allb = np.concatenate(blocks)
    per_row = K // 32
    rows = -(-allb.shape[0] // per_row)
    out = np.zeros((rows * per_row, 32), dtype=np.uint16)
    out[:allb.shape[0]] = allb
    return out.reshape(rows, K)


# ---------------------------------------------------------------------------------------------
# whole outputs on all host cores: the oracle over row chunks in a thread pool (its ctypes calls
# and numpy's array operations run without the interpreter lock)
# ---------------------------------------------------------------------------------------------
THREADS = os.cpu_count() or 1


def rows_per_job(M: int, K: int, target_elems: int = 1 << 21) -> int:
    """Rows of one job: about target_elems elements, at least enough jobs for every thread."""
    by_size = max(1, target_elems // max(K, 1))
    by_threads = max(1, -(-M // (2 * THREADS)))
    return max(1, min(by_size, by_threads))


def map_row_chunks(fn, M: int, K: int, target_elems: int = 1 << 21) -> list:
    """fn(r0, r1) over consecutive row ranges covering [0, M); results in row order. An
    exception in any job is raised here."""
    step = rows_per_job(M, K, target_elems)
    ranges = [(r0, min(M, r0 + step)) for r0 in range(0, M, step)]
    if len(ranges) == 1:
        return [fn(*ranges[0])]
    with concurrent.futures.ThreadPoolExecutor(THREADS) as pool:
        return list(pool.map(lambda rr: fn(*rr), ranges))


def assert_rows_equal(got: np.ndarray, ref_fn, what: str = "output"):
    """got [M, ...] equals ref_fn(r0, r1) on every row range, element for element."""
    M = got.shape[0]
    width = int(np.prod(got.shape[1:])) if got.ndim > 1 else 1

    def job(r0, r1):
        ref = ref_fn(r0, r1)
        g = got[r0:r1]
        if not np.array_equal(g, ref.reshape(g.shape)):
            bad = np.argwhere(g != ref.reshape(g.shape))
            i = tuple(int(v) for v in bad[0])
            raise AssertionError(f"{what}: {len(bad)} elements differ from the oracle in rows "
                                 f"[{r0}, {r1}); first at {(i[0] + r0,) + i[1:]}: "
                                 f"got {g[i]} want {ref.reshape(g.shape)[i]}")
    map_row_chunks(job, M, width)


def oracle_qdq_rows(x_bits, fmt):
    """ref_fn for assert_rows_equal: the oracle's QDQ of rows [r0, r1) of x."""
    return lambda r0, r1: O.qdq(x_bits[r0:r1], fmt)


# ---------------------------------------------------------------------------------------------
# rotated-path tolerance rules
# ---------------------------------------------------------------------------------------------
def _grid(fmt):
    n = 16 if fmt == O.E2M1 else 256
    vals = np.array([O.decode(fmt, c) if not (fmt == O.E4M3 and (c & 0x7F) == 0x7F) else np.nan
                     for c in range(n)])
    return vals


_GRIDS = {}
_DQ_TABLES = {}


def grid_values(fmt) -> np.ndarray:
    if fmt not in _GRIDS:
        _GRIDS[fmt] = _grid(fmt)
    return _GRIDS[fmt]


def dequant_table(fmt, byte) -> np.ndarray:
    """bf16 bits of every code of the format dequantized under scale byte `byte` (oracle)."""
    key = (fmt, byte)
    if key not in _DQ_TABLES:
        n = 16 if fmt == O.E2M1 else 256
        _DQ_TABLES[key] = np.array([O.dequant_bf16(fmt, c, byte) for c in range(n)],
                                   dtype=np.uint16)
    return _DQ_TABLES[key]


def _neighbours(fmt, vals, a, b) -> bool:
    """Decoded values a, b are the same or adjacent points of the signed grid."""
    if a == b:
        return True
    grid = np.unique(vals[~np.isnan(vals)])
    ia = np.searchsorted(grid, a)
    ib = np.searchsorted(grid, b)
    return abs(int(ia) - int(ib)) == 1


def rotation_tolerance(y_ref: np.ndarray, g: int) -> np.ndarray:
    M, K = y_ref.shape
    cn = np.linalg.norm(y_ref.reshape(M, K // g, g), axis=2)
    return 1e-5 * np.repeat(cn, g, axis=1)


def check_rotated_values(y_gpu: np.ndarray, y_ref: np.ndarray, g: int) -> float:
    """Max of |y_gpu - y_ref| / tol; must be <= 1."""
    tol = rotation_tolerance(y_ref, g)
    err = np.abs(y_gpu.astype(np.float64) - y_ref)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(tol > 0, err / tol, np.where(err == 0, 0.0, np.inf))
    return float(r.max()) if r.size else 0.0


def _allowed_bytes(fmt, yb, tb, ref_byte):
    """Scale bytes the GPU may give a block: the oracle's, and one step off only where the
    oracle's abs-max lies within the block's tolerance of the power of two that the step
    crosses. amax in [2^k, 2^(k+1)) gives the oracle byte of exponent k; a GPU value within tol
    of it may fall below 2^k (one byte lower, only if amax is that close to 2^k) or reach
    2^(k+1) (one byte higher, only if amax is that close to 2^(k+1))."""
    amax = float(np.abs(yb).max())
    allowed = {ref_byte}
    if amax > 0:
        k = np.floor(np.log2(amax))
        tmax = float(tb.max())
        if amax - 2.0 ** k <= tmax:
            allowed.add(ref_byte - 1)
        if 2.0 ** (k + 1) - amax <= tmax:
            allowed.add(ref_byte + 1)
    return allowed


def _block_ok(fmt, vals, yb, tb, gpu_codes, gpu_byte, ref_byte,
              allowed=None) -> tuple[bool, int]:
    """Whether GPU codes + byte of one block satisfy the rules; returns (ok, #exempt codes).
    allowed: the scale bytes the GPU may give (default: the abs-max rule's)."""
    if allowed is None:
        allowed = _allowed_bytes(fmt, yb, tb, ref_byte)
    if gpu_byte not in allowed:
        return False, 0
    byte, rc = O.quantize_block(fmt, yb, forced_byte=gpu_byte)
    diff = np.nonzero(rc != gpu_codes)[0]
    scale = 2.0 ** (gpu_byte - 127)
    for i in diff:
        a, b = vals[rc[i]], vals[gpu_codes[i]]
        if not _neighbours(fmt, vals, a, b):
            return False, 0
        t = yb[i] / scale
        if abs(t - (a + b) / 2) > tb[i] / scale:
            return False, 0
    return True, len(diff)


def _codes_chunk(fmt, vals, y, tol, gc_packed, sg, r0):
    """Rules on one row chunk: y/tol the oracle's rotated values and tolerances, gc_packed and
    sg the GPU's codes and linear scales of the same rows."""
    n, K = y.shape
    rc, rs = O.quantize_values(y, fmt, O.LINEAR)
    gc = unpack_codes(gc_packed, fmt)
    rce = unpack_codes(rc, fmt)
    bad = np.nonzero((rs != sg) | (gc != rce).reshape(n, K // 32, 32).any(axis=2))
    exempt_codes = flips = 0
    for r, j in zip(*bad):
        sl = slice(32 * j, 32 * j + 32)
        ok, k = _block_ok(fmt, vals, y[r, sl], tol[r, sl], gc[r, sl], int(sg[r, j]), int(rs[r, j]))
        assert ok, (f"block (row {r0 + r}, block {j}) outside tolerance: gpu byte "
                    f"{sg[r, j]} ref byte {rs[r, j]}")
        exempt_codes += k
        flips += int(sg[r, j] != rs[r, j])
    return np.array([n * K // 32, len(bad[0]), exempt_codes, flips])


def _qdq_chunk(fmt, vals, y, tol, og, r0):
    """Rules for rotated QDQ on one row chunk: blocks that differ from the oracle must equal
    the dequantization of codes allowed by the rules under an allowed scale."""
    n, K = y.shape
    ref = O.qdq_values(y, fmt)
    bad = np.nonzero((ref != og).reshape(n, K // 32, 32).any(axis=2))
    for r, j in zip(*bad):
        sl = slice(32 * j, 32 * j + 32)
        yb, tb, ob = y[r, sl], tol[r, sl], og[r, sl]
        ref_byte, _ = O.quantize_block(fmt, yb)
        ok = False
        for b in sorted(_allowed_bytes(fmt, yb, tb, ref_byte)):
            # the GPU codes implied by its outputs under scale b
            _, rc = O.quantize_block(fmt, yb, forced_byte=b)
            table = dequant_table(fmt, b)
            codes = rc.copy()
            good = True
            for i in np.nonzero(table[rc] != ob)[0]:
                cands = [c for c in np.nonzero(table == ob[i])[0] if not np.isnan(vals[c])]
                if not cands:
                    good = False
                    break
                codes[i] = cands[0]
            if good and _block_ok(fmt, vals, yb, tb, codes, b, ref_byte)[0]:
                ok = True
                break
        assert ok, f"rotated QDQ block (row {r0 + r}, block {j}) outside tolerance"
    return np.array([n * K // 32, len(bad[0])])


def check_rotated_codes(x_bits, H_bits, fmt, codes_gpu, scales_gpu_linear):
    """Apply the rules to GPU codes/scales (linear layout) over every row (the oracle on row
    chunks, all host cores). Returns a dict of counts; raises AssertionError with the first
    offending block."""
    return check_rotated_multi(x_bits, H_bits, codes={fmt: (codes_gpu, scales_gpu_linear)})[fmt]


def check_rotated_qdq(x_bits, H_bits, fmt, out_gpu_bits):
    return check_rotated_multi(x_bits, H_bits, qdq={fmt: out_gpu_bits})[("qdq", fmt)]


def check_rotated_multi(x_bits, H_bits, codes=None, qdq=None, nvfp4=None, nvfp4_qdq=None):
    """Every rule check of one input and one rotation at once, each row chunk rotated once by
    the oracle: codes {fmt: (codes, linear scales)}, qdq {fmt: bf16 bits}, nvfp4 {gs: (codes,
    linear scales)}, nvfp4_qdq {gs: bf16 bits}. Returns {fmt: codes stats, ("qdq", fmt): ...,
    ("nvfp4", gs): ..., ("nvfp4_qdq", gs): ...}."""
    codes, qdq = codes or {}, qdq or {}
    nvfp4, nvfp4_qdq = nvfp4 or {}, nvfp4_qdq or {}
    x = np.ascontiguousarray(x_bits)
    M, K = x.shape
    g = H_bits.shape[0]
    for fmt in set(codes) | set(qdq):
        grid_values(fmt)

    def job(r0, r1):
        y = O.rotate(x[r0:r1], H_bits)
        tol = rotation_tolerance(y, g)
        out = {}
        for fmt, (c, s) in codes.items():
            out[fmt] = _codes_chunk(fmt, grid_values(fmt), y, tol, c[r0:r1], s[r0:r1], r0)
        for fmt, o in qdq.items():
            out[("qdq", fmt)] = _qdq_chunk(fmt, grid_values(fmt), y, tol, o[r0:r1], r0)
        for gs, (c, s) in nvfp4.items():
            out[("nvfp4", gs)] = _nvfp4_codes_chunk(y, tol, gs, c[r0:r1], s[r0:r1], r0)
        for gs, o in nvfp4_qdq.items():
            out[("nvfp4_qdq", gs)] = _nvfp4_qdq_chunk(y, tol, gs, o[r0:r1], r0)
        return out

    parts = map_row_chunks(job, M, K, target_elems=1 << 20)
    total = {k: sum(p[k] for p in parts) for k in parts[0]}
    stats = {}
    for k, v in total.items():
        if k in codes:
            stats[k] = {"blocks": int(v[0]), "exempt_blocks": int(v[1]),
                        "exempt_codes": int(v[2]), "scale_flips": int(v[3])}
        elif k[0] == "nvfp4":
            stats[k] = {"blocks": int(v[0]), "exempt_blocks": int(v[1]), "scale_flips": int(v[2])}
        else:
            stats[k] = {"blocks": int(v[0]), "exempt_blocks": int(v[1])}
    return stats


# ---------------------------------------------------------------------------------------------
# NVFP4: rotated-path tolerance rules (blocks of 16, E4M3 scale under the global scale gs)
# ---------------------------------------------------------------------------------------------
_E4M3_VALUES = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).float().numpy()
_E2M1_VALUES = np.array([O.decode(O.E2M1, c) for c in range(16)])


def e4m3_cast(v: np.ndarray) -> np.ndarray:
    """Non-negative fp32 values -> E4M3 bytes, nearest even, saturating at 448."""
    v = np.minimum(np.asarray(v, dtype=np.float32), np.float32(448.0))
    return torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def nvfp4_scale_candidates(amax: float, tb: float, gs: np.float32) -> set:
    """Scale bytes reachable by rounding s_f = amax' * (gs / 6) for amax' within tb of amax."""
    f = np.float32
    r6 = f(gs) / f(6.0)
    lo = f(max(amax - tb, 0.0)) * r6 * f(1 - 2.0 ** -22)
    hi = f(amax + tb) * r6 * f(1 + 2.0 ** -22)
    b_lo, b_hi = e4m3_cast(np.array([lo, hi]))
    return set(range(int(b_lo), int(b_hi) + 1))


def _nvfp4_block_ok(yb, tb, gs, gpu_codes, gpu_byte, ref_byte) -> tuple[bool, int]:
    f = np.float32
    if gpu_byte != ref_byte and gpu_byte not in nvfp4_scale_candidates(np.abs(yb).max(), tb.max(), gs):
        return False, 0
    s_dec = f(_E4M3_VALUES[gpu_byte])
    enc = f(gs) / s_dec if s_dec != 0 else f(0.0)
    t = yb.astype(np.float32) * enc
    _, rc = O.quantize_block(O.E2M1, t.astype(np.float64), forced_byte=127)
    diff = np.nonzero(rc != gpu_codes)[0]
    for i in diff:
        a, b = _E2M1_VALUES[rc[i]], _E2M1_VALUES[gpu_codes[i]]
        if not _neighbours(O.E2M1, _E2M1_VALUES, a, b):
            return False, 0
        slack = float(tb[i]) * float(enc) * 1.001 + 4 * float(np.spacing(np.float32(abs(t[i]))))
        if abs(float(t[i]) - (a + b) / 2) > slack:
            return False, 0
    return True, len(diff)


def _nvfp4_codes_chunk(y, tol, gs, gc_packed, sg, r0):
    n, K = y.shape
    rc, rs, _ = O.nvfp4_values(y, gs, O.LINEAR, qdq=False)
    gc, rce = unpack_codes(gc_packed, O.E2M1), unpack_codes(rc, O.E2M1)
    bad = np.nonzero((rs != sg) | (gc != rce).reshape(n, K // 16, 16).any(axis=2))
    flips = 0
    for r, j in zip(*bad):
        sl = slice(16 * j, 16 * j + 16)
        ok, _ = _nvfp4_block_ok(y[r, sl], tol[r, sl], gs, gc[r, sl], int(sg[r, j]), int(rs[r, j]))
        assert ok, (f"NVFP4 block (row {r0 + r}, block {j}) outside tolerance: gpu scale "
                    f"{sg[r, j]:#x} ref {rs[r, j]:#x}")
        flips += int(sg[r, j] != rs[r, j])
    return np.array([n * K // 16, len(bad[0]), flips])


def _nvfp4_qdq_chunk(y, tol, gs, og, r0):
    n, K = y.shape
    _, rs, ref = O.nvfp4_values(y, gs, O.LINEAR, codes=False)
    bad = np.nonzero((ref != og).reshape(n, K // 16, 16).any(axis=2))
    for r, j in zip(*bad):
        sl = slice(16 * j, 16 * j + 16)
        yb, tb, ob = y[r, sl], tol[r, sl], og[r, sl]
        ok = False
        for b in sorted(nvfp4_scale_candidates(np.abs(yb).max(), tb.max(), gs) | {int(rs[r, j])}):
            table = {c: O.nvfp4_dequant_bf16(c, b, float(gs)) for c in range(16)}
            codes = []
            for i in range(16):
                cands = [c for c in range(16) if table[c] == ob[i]]
                if not cands:
                    break
                codes.append(cands[0])
            if len(codes) == 16:
                # among codes with equal outputs (e.g. +0 / -0) any is fine: try the ref's first
                _, rc = O.nvfp4_block(yb.astype(np.float32), gs)
                codes = [int(rc[i]) if table[int(rc[i])] == ob[i] else codes[i] for i in range(16)]
                if _nvfp4_block_ok(yb, tb, gs, np.array(codes), b, int(rs[r, j]))[0]:
                    ok = True
                    break
        assert ok, f"rotated NVFP4 QDQ block (row {r0 + r}, block {j}) outside tolerance"
    return np.array([n * K // 16, len(bad[0])])


def check_rotated_nvfp4(x_bits, H_bits, gs, codes_gpu, scales_gpu_linear):
    return check_rotated_multi(x_bits, H_bits,
                               nvfp4={gs: (codes_gpu, scales_gpu_linear)})[("nvfp4", gs)]


def check_rotated_nvfp4_qdq(x_bits, H_bits, gs, out_gpu_bits):
    return check_rotated_multi(x_bits, H_bits, nvfp4_qdq={gs: out_gpu_bits})[("nvfp4_qdq", gs)]


# ---------------------------------------------------------------------------------------------
# Quest-like MXFP4 scale: the same element rules; the scale decision is a threshold on the clip
# point c = alpha * RMS instead of the abs-max
# ---------------------------------------------------------------------------------------------
# The kernel sums the squares in fp32 (after an exact power-of-two scaling) and multiplies by
# alpha^2 / 32 rounded to fp32: about 12 roundings of 2^-24 each on c^2, well inside 2^-20 on c.
QUEST_SUM_REL = 2.0 ** -20


def quest_clip(yb) -> float:
    yb = np.asarray(yb, dtype=np.float64)
    return O.quest_alpha() * float(np.sqrt(np.dot(yb, yb) / yb.size))


def quest_allowed_bytes(yb, tb, ref_byte):
    """The oracle's byte, and one step off only where c lies within its tolerance of the power
    of two that the step crosses (c in [2^k, 2^(k+1)) gives the oracle's byte). The tolerance:
    alpha / sqrt(32) times the 2-norm of the values' tolerances (c is that Lipschitz in the
    values) plus the kernel's relative error on the sum."""
    c = quest_clip(yb)
    allowed = {ref_byte}
    if c > 0:
        k = np.floor(np.log2(c))
        tc = O.quest_alpha() / np.sqrt(yb.size) * float(np.linalg.norm(tb)) + QUEST_SUM_REL * c
        if c - 2.0 ** k <= tc:
            allowed.add(ref_byte - 1)
        if 2.0 ** (k + 1) - c <= tc:
            allowed.add(ref_byte + 1)
    return allowed


def _quest_codes_chunk(vals, y, tol, gc_packed, sg, r0):
    n, K = y.shape
    rc, rs = O.quest_quantize_values(y, O.LINEAR)
    gc = unpack_codes(gc_packed, O.E2M1)
    rce = unpack_codes(rc, O.E2M1)
    bad = np.nonzero((rs != sg) | (gc != rce).reshape(n, K // 32, 32).any(axis=2))
    exempt_codes = flips = 0
    for r, j in zip(*bad):
        sl = slice(32 * j, 32 * j + 32)
        yb, tb = y[r, sl], tol[r, sl]
        ok, k = _block_ok(O.E2M1, vals, yb, tb, gc[r, sl], int(sg[r, j]), int(rs[r, j]),
                          quest_allowed_bytes(yb, tb, int(rs[r, j])))
        assert ok, (f"Quest block (row {r0 + r}, block {j}) outside tolerance: gpu byte "
                    f"{sg[r, j]} ref byte {rs[r, j]}")
        exempt_codes += k
        flips += int(sg[r, j] != rs[r, j])
    return np.array([n * K // 32, len(bad[0]), exempt_codes, flips])


def _quest_qdq_chunk(vals, y, tol, og, r0):
    n, K = y.shape
    ref = O.quest_qdq_values(y)
    bad = np.nonzero((ref != og).reshape(n, K // 32, 32).any(axis=2))
    for r, j in zip(*bad):
        sl = slice(32 * j, 32 * j + 32)
        yb, tb, ob = y[r, sl], tol[r, sl], og[r, sl]
        ref_byte = O.quest_scale_byte(yb)
        allowed = quest_allowed_bytes(yb, tb, ref_byte)
        ok = False
        for b in sorted(allowed):
            _, rc = O.quantize_block(O.E2M1, yb, forced_byte=b)
            table = dequant_table(O.E2M1, b)
            codes = rc.copy()
            good = True
            for i in np.nonzero(table[rc] != ob)[0]:
                cands = np.nonzero(table == ob[i])[0]
                if not len(cands):
                    good = False
                    break
                codes[i] = cands[0]
            if good and _block_ok(O.E2M1, vals, yb, tb, codes, b, ref_byte, allowed)[0]:
                ok = True
                break
        assert ok, f"Quest QDQ block (row {r0 + r}, block {j}) outside tolerance"
    return np.array([n * K // 32, len(bad[0])])


def check_quest(x_bits, H_bits=None, codes=None, qdq=None):
    """Quest-like MXFP4 outputs of x (rotated by H when given) against the oracle over every
    row: codes = (packed codes, linear scales), qdq = bf16 bits. Without H the values are the
    exact bf16 inputs (tolerance 0: only the kernel's fp32 sum can move a scale, and only next
    to a power of two). Returns {"codes": stats, "qdq": stats}."""
    x = np.ascontiguousarray(x_bits)
    M, K = x.shape
    vals = grid_values(O.E2M1)

    def job(r0, r1):
        if H_bits is None:
            y = O.bf16_bits_to_double(x[r0:r1])
            tol = np.zeros_like(y)
        else:
            y = O.rotate(x[r0:r1], H_bits)
            tol = rotation_tolerance(y, H_bits.shape[0])
        out = {}
        if codes is not None:
            out["codes"] = _quest_codes_chunk(vals, y, tol, codes[0][r0:r1], codes[1][r0:r1], r0)
        if qdq is not None:
            out["qdq"] = _quest_qdq_chunk(vals, y, tol, qdq[r0:r1], r0)
        return out

    parts = map_row_chunks(job, M, K, target_elems=1 << 20)
    stats = {}
    for k in parts[0]:
        v = sum(p[k] for p in parts)
        stats[k] = {"blocks": int(v[0]), "exempt_blocks": int(v[1])}
        if k == "codes":
            stats[k].update(exempt_codes=int(v[2]), scale_flips=int(v[3]))
    return stats
