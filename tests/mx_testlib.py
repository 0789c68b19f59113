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
# rotated-path tolerance rules
# ---------------------------------------------------------------------------------------------
def _grid(fmt):
    n = 16 if fmt == O.E2M1 else 256
    vals = np.array([O.decode(fmt, c) if not (fmt == O.E4M3 and (c & 0x7F) == 0x7F) else np.nan
                     for c in range(n)])
    return vals


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
    amax = np.abs(yb).max()
    allowed = {ref_byte}
    if amax > 0:
        k = np.floor(np.log2(amax))
        for p in (2.0 ** k, 2.0 ** (k + 1)):
            if abs(amax - p) <= tb.max():
                allowed |= {ref_byte - 1, ref_byte + 1}
    return allowed


def _block_ok(fmt, vals, yb, tb, gpu_codes, gpu_byte, ref_byte) -> tuple[bool, int]:
    """Whether GPU codes + byte of one block satisfy the rules; returns (ok, #exempt codes)."""
    if gpu_byte not in _allowed_bytes(fmt, yb, tb, ref_byte):
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


def check_rotated_codes(x_bits, H_bits, fmt, codes_gpu, scales_gpu_linear):
    """Apply the rules to GPU codes/scales (linear layout). Returns a dict of counts; raises
    AssertionError with the first offending block."""
    y = O.rotate(x_bits, H_bits)
    g = H_bits.shape[0]
    tol = rotation_tolerance(y, g)
    M, K = y.shape
    rc, rs = O.rotate_quantize(x_bits, H_bits, fmt, O.LINEAR)
    gc = unpack_codes(codes_gpu, fmt)
    rce = unpack_codes(rc, fmt)
    vals = _grid(fmt)
    bad_blocks = np.nonzero((rs != scales_gpu_linear) |
                            (gc != rce).reshape(M, K // 32, 32).any(axis=2))
    exempt_codes = 0
    flips = 0
    for r, j in zip(*bad_blocks):
        sl = slice(32 * j, 32 * j + 32)
        ok, n = _block_ok(fmt, vals, y[r, sl], tol[r, sl], gc[r, sl], int(scales_gpu_linear[r, j]),
                          int(rs[r, j]))
        assert ok, (f"block (row {r}, block {j}) outside tolerance: gpu byte "
                    f"{scales_gpu_linear[r, j]} ref byte {rs[r, j]}")
        exempt_codes += n
        flips += int(scales_gpu_linear[r, j] != rs[r, j])
    return {"blocks": M * K // 32, "exempt_blocks": len(bad_blocks[0]), "exempt_codes": exempt_codes,
            "scale_flips": flips}


def check_rotated_qdq(x_bits, H_bits, fmt, out_gpu_bits):
    """Rules for rotated QDQ: blocks that differ from the oracle must equal the dequantization of
    codes allowed by the rules under an allowed scale."""
    y = O.rotate(x_bits, H_bits)
    g = H_bits.shape[0]
    tol = rotation_tolerance(y, g)
    M, K = y.shape
    ref = O.rotate_qdq(x_bits, H_bits, fmt)
    _, rs = O.rotate_quantize(x_bits, H_bits, fmt, O.LINEAR)
    vals = _grid(fmt)
    bad = np.nonzero((ref != out_gpu_bits).reshape(M, K // 32, 32).any(axis=2))
    exempt = 0
    for r, j in zip(*bad):
        sl = slice(32 * j, 32 * j + 32)
        yb, tb, ob = y[r, sl], tol[r, sl], out_gpu_bits[r, sl]
        ok = False
        for b in sorted(_allowed_bytes(fmt, yb, tb, int(rs[r, j]))):
            # the GPU codes implied by its outputs under scale b
            _, rc = O.quantize_block(fmt, yb, forced_byte=b)
            codes = rc.copy()
            good = True
            for i in range(32):
                if O.dequant_bf16(fmt, int(rc[i]), b) == ob[i]:
                    continue
                cands = [c for c in range(len(vals)) if not np.isnan(vals[c])
                         and O.dequant_bf16(fmt, c, b) == ob[i]]
                if not cands:
                    good = False
                    break
                codes[i] = cands[0]
            if good and _block_ok(fmt, vals, yb, tb, codes, b, int(rs[r, j]))[0]:
                ok = True
                break
        assert ok, f"rotated QDQ block (row {r}, block {j}) outside tolerance"
        exempt += 1
    return {"blocks": M * K // 32, "exempt_blocks": exempt}


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


def check_rotated_nvfp4(x_bits, H_bits, gs, codes_gpu, scales_gpu_linear):
    y = O.rotate(x_bits, H_bits)
    tol = rotation_tolerance(y, H_bits.shape[0])
    M, K = y.shape
    rc, rs = O.nvfp4_quantize(x_bits, gs, O.LINEAR, H_bits=H_bits)
    gc, rce = unpack_codes(codes_gpu, O.E2M1), unpack_codes(rc, O.E2M1)
    bad = np.nonzero((rs != scales_gpu_linear) | (gc != rce).reshape(M, K // 16, 16).any(axis=2))
    flips = 0
    for r, j in zip(*bad):
        sl = slice(16 * j, 16 * j + 16)
        ok, _ = _nvfp4_block_ok(y[r, sl], tol[r, sl], gs, gc[r, sl], int(scales_gpu_linear[r, j]),
                                int(rs[r, j]))
        assert ok, (f"NVFP4 block (row {r}, block {j}) outside tolerance: gpu scale "
                    f"{scales_gpu_linear[r, j]:#x} ref {rs[r, j]:#x}")
        flips += int(scales_gpu_linear[r, j] != rs[r, j])
    return {"blocks": M * K // 16, "exempt_blocks": len(bad[0]), "scale_flips": flips}


def check_rotated_nvfp4_qdq(x_bits, H_bits, gs, out_gpu_bits):
    y = O.rotate(x_bits, H_bits)
    tol = rotation_tolerance(y, H_bits.shape[0])
    M, K = y.shape
    ref = O.nvfp4_qdq(x_bits, gs, H_bits=H_bits)
    _, rs = O.nvfp4_quantize(x_bits, gs, O.LINEAR, H_bits=H_bits)
    bad = np.nonzero((ref != out_gpu_bits).reshape(M, K // 16, 16).any(axis=2))
    for r, j in zip(*bad):
        sl = slice(16 * j, 16 * j + 16)
        yb, tb, ob = y[r, sl], tol[r, sl], out_gpu_bits[r, sl]
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
        assert ok, f"rotated NVFP4 QDQ block (row {r}, block {j}) outside tolerance"
    return {"blocks": M * K // 16, "exempt_blocks": len(bad[0])}
