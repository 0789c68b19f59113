"""Seeded synthetic inputs shaped like the workloads the MX pages describe.

This module only draws inputs: it holds none of the quantization arithmetic, and both the GPU
path's tests/benchmark and the CPU oracle consume exactly the same bf16 bit patterns from it.
Every generator is deterministic in its seed (numpy PCG64, one child stream per tensor) and
returns bf16 tensors as uint16 bit patterns (rounded to nearest-even from float32 by torch).

Workloads (shapes from the pages; value distributions chosen as weight-like / activation-like):
  * mxfp8_linear_quant: x[128, 4096] N(0,1), 1% of elements times 50, one all-zero 32-group per
    row (group (37*r) mod (K/32) of row r).
  * mxfp4_qdq: weight-like x[8192, 8192] Student-t(nu=4) * 0.02, and activation-like
    x[4096, 8192] N(0,1) whose columns 1029*i + 3 (i = 0..7) are times 100.
  * rotate_quant: activations x[M, K] N(0,1), M in {1,16,128,1024,8192}, K in {8192, 28672}
    (input widths of the Llama-3.1-70B layer shapes (8192,8192), (8192,57344), (28672,8192)
    named in the QuTLASS pull request's benchmark).
  * moe_quant: 128 experts, expert of each of 16384 tokens drawn from a Zipf(1.1) law over 128
    ranks mapped through a seeded permutation; rows [n_e, 2048] N(0,1) concatenated by expert.
  * rotation_sweep: one decoder layer's inputs at 4096 tokens: [4096, 8192] attention input,
    [4096, 8192] O-projection input, [4096, 28672] down-projection input, Student-t(nu=5).
  * weight_rotate_quant: weight-side rotate + quantize of the 70B layer weights [N, K] =
    (8192, 8192), (57344, 8192), (8192, 28672), N(0,1) * 0.02, drawn in 2048-row chunks with one
    child stream each so that any row range can be drawn alone.
The rotation matrix is an input too: the normalized Sylvester Hadamard H_g * g^-0.5 rounded to
bf16, the construction the QuTLASS benchmark loads at run time.
"""

from __future__ import annotations

import numpy as np
import torch

SEED_BASE = 1000
WORKLOADS = ("mxfp8_linear_quant", "mxfp4_qdq", "rotate_quant", "moe_quant", "rotation_sweep",
             "weight_rotate_quant")


def _rng(workload: str, stream: int = 0) -> np.random.Generator:
    idx = WORKLOADS.index(workload) + 1
    ss = np.random.SeedSequence([SEED_BASE + idx, stream])
    return np.random.Generator(np.random.PCG64(ss))


def to_bf16_bits(a) -> np.ndarray:
    """float array -> bf16 bit patterns (uint16), round to nearest even."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 (exact)."""
    return (np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def sylvester_hadamard(g: int) -> np.ndarray:
    """Unnormalized Sylvester Hadamard matrix of order g (a power of two), entries +-1."""
    assert g >= 1 and (g & (g - 1)) == 0
    h = np.ones((1, 1), dtype=np.float64)
    while h.shape[0] < g:
        h = np.block([[h, h], [h, -h]])
    return h


def normalized_hadamard_bf16(g: int) -> np.ndarray:
    """bf16 bits of H_g * g^-0.5, g x g row-major."""
    return to_bf16_bits(sylvester_hadamard(g) * g ** -0.5)


# ----------------------------------------------------------------------------------------------
# workloads (sizes are parameters so that tests can draw the same recipe at small scale)
# ----------------------------------------------------------------------------------------------
def mxfp8_linear_quant(M: int = 128, K: int = 4096, stream: int = 0) -> np.ndarray:
    rng = _rng("mxfp8_linear_quant", stream)
    x = rng.standard_normal((M, K), dtype=np.float32)
    outlier = rng.random((M, K)) < 0.01
    x[outlier] *= 50.0
    groups = K // 32
    for r in range(M):
        j = (37 * r) % groups
        x[r, 32 * j:32 * j + 32] = 0.0
    return to_bf16_bits(x)


def mxfp4_qdq_weight(M: int = 8192, K: int = 8192, stream: int = 0) -> np.ndarray:
    rng = _rng("mxfp4_qdq", 2 * stream)
    x = rng.standard_t(4.0, size=(M, K)) * 0.02
    return to_bf16_bits(x)


def mxfp4_qdq_activation(M: int = 4096, K: int = 8192, stream: int = 0) -> np.ndarray:
    rng = _rng("mxfp4_qdq", 2 * stream + 1)
    x = rng.standard_normal((M, K), dtype=np.float32)
    for i in range(8):
        c = 1029 * i + 3
        if c < K:
            x[:, c] *= 100.0
    return to_bf16_bits(x)


def rotate_quant_activation(M: int, K: int, stream: int = 0) -> np.ndarray:
    rng = _rng("rotate_quant", stream * 1_000_003 + M * 7 + K)
    return to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))


ROTATE_QUANT_M = (1, 16, 128, 1024, 8192)
ROTATE_QUANT_K = (8192, 28672)


def moe_counts(E: int = 128, tokens: int = 16384, stream: int = 0) -> np.ndarray:
    rng = _rng("moe_quant", 2 * stream)
    p = np.arange(1, E + 1, dtype=np.float64) ** -1.1
    p /= p.sum()
    rank = rng.choice(E, size=tokens, p=p)
    perm = rng.permutation(E)
    return np.bincount(perm[rank], minlength=E).astype(np.int64)


def moe_quant(E: int = 128, tokens: int = 16384, K: int = 2048, stream: int = 0):
    """-> (x bits [tokens, K], offsets int64 [E+1])."""
    counts = moe_counts(E, tokens, stream)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int64)
    rng = _rng("moe_quant", 2 * stream + 1)
    x = rng.standard_normal((tokens, K), dtype=np.float32)
    return to_bf16_bits(x), offsets


ROTATION_SWEEP_G = (16, 32, 64, 128)
ROTATION_SWEEP_LAYERS = (("attn_in", 4096, 8192), ("o_proj_in", 4096, 8192),
                         ("down_proj_in", 4096, 28672))


def rotation_sweep_input(name: str, M: int | None = None, K: int | None = None,
                         stream: int = 0) -> np.ndarray:
    idx = [n for n, _, _ in ROTATION_SWEEP_LAYERS].index(name)
    _, M0, K0 = ROTATION_SWEEP_LAYERS[idx]
    M = M0 if M is None else M
    K = K0 if K is None else K
    rng = _rng("rotation_sweep", 3 * stream + idx)
    return to_bf16_bits(rng.standard_t(5.0, size=(M, K)))


WEIGHT_SHAPES = ((8192, 8192), (57344, 8192), (8192, 28672))
WEIGHT_CHUNK_ROWS = 2048


def weight_rotate_quant(N: int, K: int, r0: int = 0, r1: int | None = None) -> np.ndarray:
    """Rows [r0, r1) of the weight-like [N, K] matrix N(0,1) * 0.02 (bf16 bits)."""
    r1 = N if r1 is None else r1
    assert 0 <= r0 <= r1 <= N
    out = np.empty((r1 - r0, K), dtype=np.uint16)
    for chunk in range(r0 // WEIGHT_CHUNK_ROWS, -(-r1 // WEIGHT_CHUNK_ROWS)):
        lo = chunk * WEIGHT_CHUNK_ROWS
        hi = min(lo + WEIGHT_CHUNK_ROWS, N)
        rng = _rng("weight_rotate_quant", (N * 1_000_003 + K) * 4096 + chunk)
        block = rng.standard_normal((hi - lo, K), dtype=np.float32) * np.float32(0.02)
        a, b = max(lo, r0), min(hi, r1)
        out[a - r0:b - r0] = to_bf16_bits(block[a - lo:b - lo])
    return out
