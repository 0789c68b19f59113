"""Library cross-check of the swizzled scale layout: a block-scaled GEMM (torch._scaled_mm with
E8M0 block scales, backed by cuBLAS) consumes the codes and 128x4-swizzled scales this library
writes, and must agree with dequantize-then-matmul (the test pattern of the QuTLASS pull
request, which compares its block-scaled GEMM against dequantized operands). Skipped when the
installed torch cannot run MXFP8 _scaled_mm on this GPU."""

import numpy as np
import pytest
import torch

import __graft_entry__
import mx_microscaling_quantize_gb300 as mxq
from mx_microscaling_quantize_gb300 import workloads as W
import mx_testlib as T

pytestmark = pytest.mark.gpu


def dequant_e4m3(codes_u8: torch.Tensor, scales_lin_u8: torch.Tensor) -> torch.Tensor:
    vals = codes_u8.view(torch.float8_e4m3fn).to(torch.float32)
    s = torch.ldexp(torch.ones_like(scales_lin_u8, dtype=torch.float32),
                    scales_lin_u8.to(torch.int32) - 127)
    return vals * s.repeat_interleave(32, dim=1)


def try_scaled_mm(a, b, sa, sb):
    attempts = [
        lambda: torch._scaled_mm(a, b.t(), scale_a=sa, scale_b=sb, out_dtype=torch.float32),
        lambda: torch._scaled_mm(a, b.t(), scale_a=sa, scale_b=sb, out_dtype=torch.bfloat16),
    ]
    errors = []
    for f in attempts:
        try:
            return f().float(), None
        except Exception as e:  # unsupported configuration in this torch build
            errors.append(f"{type(e).__name__}: {str(e)[:120]}")
    return None, "; ".join(errors)


def test_swizzled_scales_feed_a_block_scaled_gemm():
    __graft_entry__.build()
    M, N, K = 256, 384, 1024
    xa = T.to_gpu(W.mxfp4_qdq_activation(M, K))
    xb = T.to_gpu(W.rotation_sweep_input("attn_in", N, K))
    ca, sa_swz = mxq.mx_quantize(xa, mxq.E4M3, mxq.SWIZZLED)
    cb, sb_swz = mxq.mx_quantize(xb, mxq.E4M3, mxq.SWIZZLED)
    _, sa_lin = mxq.mx_quantize(xa, mxq.E4M3, mxq.LINEAR)
    _, sb_lin = mxq.mx_quantize(xb, mxq.E4M3, mxq.LINEAR)
    want = dequant_e4m3(ca, sa_lin) @ dequant_e4m3(cb, sb_lin).t()
    got, err = try_scaled_mm(ca.view(torch.float8_e4m3fn), cb.view(torch.float8_e4m3fn),
                             sa_swz.view(torch.float8_e8m0fnu).reshape(-1),
                             sb_swz.view(torch.float8_e8m0fnu).reshape(-1))
    if got is None:
        pytest.skip(f"MXFP8 _scaled_mm unavailable here: {err}")
    rel = (got - want).abs().max() / want.abs().max()
    assert rel < 1e-3, float(rel)
    # the same GEMM with the linear scales fed as if swizzled must NOT agree (the check has teeth)
    bad, _ = try_scaled_mm(ca.view(torch.float8_e4m3fn), cb.view(torch.float8_e4m3fn),
                           sa_lin.view(torch.float8_e8m0fnu).reshape(-1),
                           sb_lin.view(torch.float8_e8m0fnu).reshape(-1))
    if bad is not None:
        assert (bad - want).abs().max() / want.abs().max() > 1e-2
