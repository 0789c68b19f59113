"""OCP-MX block quantization (MXFP4 / MXFP8) on GB300: Python binding of libmxq.

Every function here has the name of the C entry point it calls (include/mxq.h) and does
argument marshalling only: it checks tensor device/dtype/shape, allocates outputs with torch
when the caller passes none, and hands raw device pointers and the current CUDA stream to the
library. All computation runs in the library's sm_103a kernels. If libmxq.so is missing the
calls raise; there is no fallback.
"""

from __future__ import annotations

import ctypes
import functools
import os

import torch

E2M1 = MXFP4 = 1
E4M3 = MXFP8 = 2
LINEAR = 0
SWIZZLED = 1
RNE = 0    # abs-max block scale
QUEST = 1  # Quest-like block scale (clip point alpha * RMS), MXFP4 only, not grouped
GROUP = 32
ROT_DENSE = 0     # any H: tensor-core product
ROT_HADAMARD = 1  # H = H[0][0] * Sylvester (stated by the caller, checked on the device)
ROT_AUTO = 2      # the same statement; the library takes the kernel measured faster for the call

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmxq.so")
_lib = None

EXPORTS = (
    "mx_status_string", "mx_scales_shape", "mx_grouped_scales_shape", "mx_quantize", "mx_qdq",
    "mx_rotate_quantize", "mx_quantize_grouped", "mx_dequantize", "mx_nvfp4_scales_shape",
    "mx_quantize_nvfp4", "mx_qdq_nvfp4", "mx_dequantize_nvfp4", "mx_nvfp4_grouped_scales_shape",
    "mx_quantize_nvfp4_grouped", "mx_rotate_debug", "mx_device_errors",
    "mx_selftest_bounded_wait", "mx_selftest_rotate_give_up", "mx_gemm",
    "mx_selftest_gemm_give_up",
)


class MXError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(message)
        self.status = status


def lib() -> ctypes.CDLL:
    """The loaded libmxq (ctypes handle with argument types set)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is not built; run `python -m mx_microscaling_quantize_gb300._build` "
            "(or __graft_entry__.build()) first")
    L = ctypes.CDLL(LIB_PATH)
    i32, i64, p = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
    pi64 = ctypes.POINTER(ctypes.c_int64)
    sigs = {
        "mx_status_string": (ctypes.c_char_p, [i32]),
        "mx_scales_shape": (i32, [i64, i64, i32, i32, pi64, pi64]),
        "mx_grouped_scales_shape": (i32, [i64, i32, i64, i32, i32, pi64, pi64]),
        "mx_quantize": (i32, [p, i64, i64, i32, i32, i32, i32, p, p, p]),
        "mx_qdq": (i32, [p, i64, i64, i32, i32, i32, p, i32, i32, p, p]),
        "mx_rotate_quantize": (i32, [p, i64, i64, p, i32, i32, i32, i32, i32, i32, p, p, p]),
        "mx_quantize_grouped": (i32, [p, p, i32, i64, i64, i32, i32, i32, i32, p, p, p]),
        "mx_dequantize": (i32, [p, p, i64, i64, i32, i32, i32, p, p]),
        "mx_nvfp4_scales_shape": (i32, [i64, i64, i32, pi64, pi64]),
        "mx_quantize_nvfp4": (i32, [p, i64, i64, p, i32, i32, p, i32, p, p, p]),
        "mx_qdq_nvfp4": (i32, [p, i64, i64, p, i32, i32, p, p, p]),
        "mx_dequantize_nvfp4": (i32, [p, p, i64, i64, p, i32, p, p]),
        "mx_nvfp4_grouped_scales_shape": (i32, [i64, i32, i64, i32, pi64, pi64]),
        "mx_quantize_nvfp4_grouped": (i32, [p, p, i32, i64, i64, p, i32, p, p, p]),
        "mx_rotate_debug": (i32, [p, i64, i64, p, i32, i32, p, p]),
        "mx_device_errors": (i32, [ctypes.POINTER(ctypes.c_int)]),
        "mx_selftest_bounded_wait": (i32, [i64, p]),
        "mx_selftest_rotate_give_up": (i32, [p, i64, i64, p, i32, p, p, i64, p]),
        "mx_gemm": (i32, [p, p, p, p, i64, i64, i64, i32, i32, i32, ctypes.c_float, p, p]),
        "mx_selftest_gemm_give_up": (i32, [p, p, p, p, i64, i64, i64, i32, i32, p, i64, p]),
    }
    for name, (res, args) in sigs.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    _lib = L
    return L


def mx_status_string(status: int) -> str:
    return lib().mx_status_string(status).decode()


def _check(status: int) -> None:
    if status != 0:
        raise MXError(status, mx_status_string(status))


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_ptr(stream, t: torch.Tensor) -> int:
    """The cudaStream_t to launch on: `stream` (a torch.cuda.Stream or a raw handle), or when
    None the current stream of t's device (read without building a Stream object, which costs
    microseconds per call)."""
    if stream is None:
        dev = t.get_device()
        if _raw_stream is not None:
            return _raw_stream(dev)
        return torch.cuda.current_stream(dev).cuda_stream
    return stream.cuda_stream if isinstance(stream, torch.cuda.Stream) else stream


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else t.data_ptr()


def _input(x: torch.Tensor, name: str = "x") -> tuple[int, int]:
    if not (isinstance(x, torch.Tensor) and x.is_cuda and x.dtype == torch.bfloat16):
        raise TypeError(f"{name} must be a CUDA bfloat16 tensor")
    if x.dim() != 2 or not x.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 2-D [M, K] tensor")
    return x.shape[0], x.shape[1]


def _rotation(H: torch.Tensor) -> int:
    if not (isinstance(H, torch.Tensor) and H.is_cuda and H.dtype == torch.bfloat16):
        raise TypeError("H must be a CUDA bfloat16 tensor")
    if H.dim() != 2 or H.shape[0] != H.shape[1] or not H.is_contiguous():
        raise ValueError("H must be a contiguous square [g, g] tensor")
    return H.shape[0]


def code_bytes_per_row(fmt: int, K: int) -> int:
    return K if fmt == E4M3 else K // 2


def _codes_out(codes, x, M, K, fmt):
    if codes is None:
        return torch.empty((M, code_bytes_per_row(fmt, K)), dtype=torch.uint8, device=x.device)
    if codes.numel() * codes.element_size() != M * code_bytes_per_row(fmt, K):
        raise ValueError("codes has the wrong size")
    return codes


def _scales_out(scales, x, rows, cols):
    if scales is None:
        return torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    if scales.numel() * scales.element_size() != rows * cols:
        raise ValueError("scales has the wrong size")
    return scales


@functools.lru_cache(maxsize=4096)
def mx_scales_shape(M: int, K: int, layout: int = LINEAR, group: int = GROUP) -> tuple[int, int]:
    r, c = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().mx_scales_shape(M, K, group, layout, ctypes.byref(r), ctypes.byref(c)))
    return r.value, c.value


@functools.lru_cache(maxsize=4096)
def mx_grouped_scales_shape(M_total: int, E: int, K: int, layout: int = SWIZZLED,
                            group: int = GROUP) -> tuple[int, int]:
    r, c = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().mx_grouped_scales_shape(M_total, E, K, group, layout, ctypes.byref(r),
                                         ctypes.byref(c)))
    return r.value, c.value


def mx_quantize(x, fmt, layout=LINEAR, *, codes=None, scales=None, group=GROUP, rounding=RNE,
                stream=None):
    """Block quantize bf16 [M, K] -> (codes uint8, E8M0 scales uint8)."""
    M, K = _input(x)
    codes = _codes_out(codes, x, M, K, fmt)
    scales = _scales_out(scales, x, *mx_scales_shape(M, K, layout, group))
    _check(lib().mx_quantize(_ptr(x), M, K, fmt, group, layout, rounding, _ptr(codes),
                             _ptr(scales), _stream_ptr(stream, x)))
    return codes, scales


def mx_qdq(x, fmt, H=None, *, y=None, group=GROUP, rounding=RNE, rot_kind=ROT_DENSE,
           stream=None):
    """Quantize-dequantize bf16 [M, K] -> bf16 [M, K]; with H, rotate each g-chunk first
    (rot_kind: ROT_DENSE, ROT_HADAMARD or ROT_AUTO)."""
    M, K = _input(x)
    g = _rotation(H) if H is not None else 0
    if y is None:
        y = torch.empty_like(x)
    _check(lib().mx_qdq(_ptr(x), M, K, fmt, group, rounding, _ptr(H), g, rot_kind, _ptr(y),
                        _stream_ptr(stream, x)))
    return y


def mx_rotate_quantize(x, H, fmt, layout=SWIZZLED, *, codes=None, scales=None, group=GROUP,
                       rounding=RNE, rot_kind=ROT_DENSE, stream=None):
    """Rotate each g-chunk by H, then block quantize -> (codes, scales)."""
    M, K = _input(x)
    g = _rotation(H)
    codes = _codes_out(codes, x, M, K, fmt)
    scales = _scales_out(scales, x, *mx_scales_shape(M, K, layout, group))
    _check(lib().mx_rotate_quantize(_ptr(x), M, K, _ptr(H), g, rot_kind, fmt, group, layout,
                                    rounding, _ptr(codes), _ptr(scales), _stream_ptr(stream, x)))
    return codes, scales


def mx_quantize_grouped(x, row_offsets, fmt, layout=SWIZZLED, *, codes=None, scales=None,
                        group=GROUP, rounding=RNE, stream=None):
    """Per-expert block quantize; row_offsets: CUDA int64 [E + 1]."""
    M, K = _input(x)
    if not (row_offsets.is_cuda and row_offsets.dtype == torch.int64 and row_offsets.dim() == 1
            and row_offsets.is_contiguous()):
        raise TypeError("row_offsets must be a contiguous CUDA int64 [E + 1] tensor")
    E = row_offsets.numel() - 1
    codes = _codes_out(codes, x, M, K, fmt)
    scales = _scales_out(scales, x, *mx_grouped_scales_shape(M, E, K, layout, group))
    _check(lib().mx_quantize_grouped(_ptr(x), _ptr(row_offsets), E, M, K, fmt, group, layout,
                                     rounding, _ptr(codes), _ptr(scales), _stream_ptr(stream, x)))
    return codes, scales


def mx_dequantize(codes, scales, K, fmt, layout=LINEAR, *, y=None, group=GROUP, stream=None):
    """Stored codes (uint8 [M, K or K/2]) and E8M0 scales -> bf16 [M, K]."""
    if not (isinstance(codes, torch.Tensor) and codes.is_cuda and codes.dim() == 2
            and codes.is_contiguous() and codes.element_size() == 1):
        raise TypeError("codes must be a contiguous CUDA 2-D tensor of bytes")
    if not (isinstance(scales, torch.Tensor) and scales.is_cuda and scales.is_contiguous()
            and scales.element_size() == 1):
        raise TypeError("scales must be a contiguous CUDA tensor of bytes")
    M = codes.shape[0]
    if codes.shape[1] != code_bytes_per_row(fmt, K):
        raise ValueError("codes has the wrong row length for K and fmt")
    rows, cols = mx_scales_shape(M, K, layout, group)
    if scales.numel() != rows * cols:
        raise ValueError("scales has the wrong size")
    if y is None:
        y = torch.empty((M, K), dtype=torch.bfloat16, device=codes.device)
    elif not (y.is_cuda and y.dtype == torch.bfloat16 and y.numel() == M * K
              and y.is_contiguous()):
        raise ValueError("y must be a contiguous CUDA bfloat16 tensor of M * K elements")
    _check(lib().mx_dequantize(_ptr(codes), _ptr(scales), M, K, fmt, group, layout, _ptr(y),
                               _stream_ptr(stream, codes)))
    return y


@functools.lru_cache(maxsize=4096)
def mx_nvfp4_scales_shape(M: int, K: int, layout: int = SWIZZLED) -> tuple[int, int]:
    r, c = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().mx_nvfp4_scales_shape(M, K, layout, ctypes.byref(r), ctypes.byref(c)))
    return r.value, c.value


def _global_scale(gs) -> None:
    if not (isinstance(gs, torch.Tensor) and gs.is_cuda and gs.dtype == torch.float32
            and gs.numel() == 1):
        raise TypeError("global_scale must be a CUDA float32 tensor of one element")


def mx_quantize_nvfp4(x, global_scale, layout=SWIZZLED, H=None, *, codes=None, scales=None,
                      rot_kind=ROT_DENSE, stream=None):
    """NVFP4 quantize (optionally rotating each g-chunk by H first) -> (codes, E4M3 scales)."""
    M, K = _input(x)
    _global_scale(global_scale)
    g = _rotation(H) if H is not None else 0
    codes = _codes_out(codes, x, M, K, E2M1)
    scales = _scales_out(scales, x, *mx_nvfp4_scales_shape(M, K, layout))
    _check(lib().mx_quantize_nvfp4(_ptr(x), M, K, _ptr(H), g, rot_kind, _ptr(global_scale),
                                   layout, _ptr(codes), _ptr(scales), _stream_ptr(stream, x)))
    return codes, scales


def mx_qdq_nvfp4(x, global_scale, H=None, *, y=None, rot_kind=ROT_DENSE, stream=None):
    """NVFP4 quantize-dequantize bf16 [M, K] -> bf16 [M, K] (optionally rotated)."""
    M, K = _input(x)
    _global_scale(global_scale)
    g = _rotation(H) if H is not None else 0
    if y is None:
        y = torch.empty_like(x)
    _check(lib().mx_qdq_nvfp4(_ptr(x), M, K, _ptr(H), g, rot_kind, _ptr(global_scale), _ptr(y),
                              _stream_ptr(stream, x)))
    return y


@functools.lru_cache(maxsize=4096)
def mx_nvfp4_grouped_scales_shape(M_total: int, E: int, K: int,
                                  layout: int = SWIZZLED) -> tuple[int, int]:
    r, c = ctypes.c_int64(), ctypes.c_int64()
    _check(lib().mx_nvfp4_grouped_scales_shape(M_total, E, K, layout, ctypes.byref(r),
                                               ctypes.byref(c)))
    return r.value, c.value


def mx_quantize_nvfp4_grouped(x, row_offsets, global_scales, layout=SWIZZLED, *, codes=None,
                              scales=None, stream=None):
    """Per-expert NVFP4 quantize; row_offsets: CUDA int64 [E + 1]; global_scales: CUDA fp32 [E]."""
    M, K = _input(x)
    if not (row_offsets.is_cuda and row_offsets.dtype == torch.int64 and row_offsets.dim() == 1
            and row_offsets.is_contiguous()):
        raise TypeError("row_offsets must be a contiguous CUDA int64 [E + 1] tensor")
    E = row_offsets.numel() - 1
    if not (isinstance(global_scales, torch.Tensor) and global_scales.is_cuda
            and global_scales.dtype == torch.float32 and global_scales.numel() == E
            and global_scales.is_contiguous()):
        raise TypeError("global_scales must be a contiguous CUDA float32 tensor of E elements")
    codes = _codes_out(codes, x, M, K, E2M1)
    scales = _scales_out(scales, x, *mx_nvfp4_grouped_scales_shape(M, E, K, layout))
    _check(lib().mx_quantize_nvfp4_grouped(_ptr(x), _ptr(row_offsets), E, M, K,
                                           _ptr(global_scales), layout, _ptr(codes),
                                           _ptr(scales), _stream_ptr(stream, x)))
    return codes, scales


def mx_dequantize_nvfp4(codes, scales, K, global_scale, layout=SWIZZLED, *, y=None,
                        stream=None):
    """Stored NVFP4 codes (uint8 [M, K/2]) and E4M3 scales -> bf16 [M, K]."""
    if not (isinstance(codes, torch.Tensor) and codes.is_cuda and codes.dim() == 2
            and codes.is_contiguous() and codes.element_size() == 1):
        raise TypeError("codes must be a contiguous CUDA 2-D tensor of bytes")
    if not (isinstance(scales, torch.Tensor) and scales.is_cuda and scales.is_contiguous()
            and scales.element_size() == 1):
        raise TypeError("scales must be a contiguous CUDA tensor of bytes")
    _global_scale(global_scale)
    M = codes.shape[0]
    if codes.shape[1] != K // 2:
        raise ValueError("codes has the wrong row length for K")
    rows, cols = mx_nvfp4_scales_shape(M, K, layout)
    if scales.numel() != rows * cols:
        raise ValueError("scales has the wrong size")
    if y is None:
        y = torch.empty((M, K), dtype=torch.bfloat16, device=codes.device)
    elif not (y.is_cuda and y.dtype == torch.bfloat16 and y.numel() == M * K
              and y.is_contiguous()):
        raise ValueError("y must be a contiguous CUDA bfloat16 tensor of M * K elements")
    _check(lib().mx_dequantize_nvfp4(_ptr(codes), _ptr(scales), M, K, _ptr(global_scale), layout,
                                     _ptr(y), _stream_ptr(stream, codes)))
    return y


def mx_rotate_debug(x, H, *, y=None, rot_kind=ROT_DENSE, stream=None):
    """The fp32 rotated values the rotated kernels quantize (diagnostics)."""
    M, K = _input(x)
    g = _rotation(H)
    if y is None:
        y = torch.empty((M, K), dtype=torch.float32, device=x.device)
    _check(lib().mx_rotate_debug(_ptr(x), M, K, _ptr(H), g, rot_kind, _ptr(y),
                                 _stream_ptr(stream, x)))
    return y


def mx_device_errors() -> int:
    """Synchronize and return (then clear) the device error word."""
    v = ctypes.c_int()
    _check(lib().mx_device_errors(ctypes.byref(v)))
    return v.value


def mx_selftest_bounded_wait(limit_ns: int = 1_000_000, *, stream=None, device: int = 0) -> None:
    """Run one bounded wait that nothing completes (it gives up after limit_ns and sets the
    device error word; read it with mx_device_errors())."""
    st = stream
    if st is None:
        st = _raw_stream(device) if _raw_stream is not None else torch.cuda.current_stream(device).cuda_stream
    elif isinstance(st, torch.cuda.Stream):
        st = st.cuda_stream
    _check(lib().mx_selftest_bounded_wait(limit_ns, st))


def mx_selftest_rotate_give_up(x, H, limit_ns: int, *, stream=None):
    """The tensor-core rotate + MXFP4 quantize (swizzled scales) with every wait of the kernel
    limited to limit_ns: waits run out while the pipeline is busy, the kernel stops issuing
    work, drains what is in flight and returns; the device error word reports it (read it with
    mx_device_errors()). Returns the (unspecified) codes and scales buffers."""
    M, K = _input(x)
    g = _rotation(H)
    codes = _codes_out(None, x, M, K, E2M1)
    scales = _scales_out(None, x, *mx_scales_shape(M, K, SWIZZLED))
    _check(lib().mx_selftest_rotate_give_up(_ptr(x), M, K, _ptr(H), g, _ptr(codes), _ptr(scales),
                                            limit_ns, _stream_ptr(stream, x)))
    return codes, scales


def _gemm_operands(a_codes, a_scales, b_codes, b_scales, K, fmt, c):
    for t in (a_codes, a_scales, b_codes, b_scales):
        if not (isinstance(t, torch.Tensor) and t.is_cuda and t.dtype == torch.uint8
                and t.is_contiguous()):
            raise TypeError("codes and scales must be contiguous CUDA uint8 tensors")
    M, N = a_codes.shape[0], b_codes.shape[0]
    if a_codes.numel() != M * code_bytes_per_row(fmt, K) or \
            b_codes.numel() != N * code_bytes_per_row(fmt, K):
        raise ValueError("codes do not match K and the format")
    if c is None:
        c = torch.empty((M, N), dtype=torch.bfloat16, device=a_codes.device)
    return M, N, c


def mx_selftest_gemm_give_up(a_codes, a_scales, b_codes, b_scales, K: int, fmt, layout, limit_ns: int,
                             *, stream=None):
    """mx_gemm with every pipeline wait of the kernel limited to limit_ns: the kernel stops
    issuing work, drains what is in flight and returns; the device error word reports it.
    Returns the (unspecified) C buffer."""
    M, N, c = _gemm_operands(a_codes, a_scales, b_codes, b_scales, K, fmt, None)
    _check(lib().mx_selftest_gemm_give_up(_ptr(a_codes), _ptr(a_scales), _ptr(b_codes),
                                          _ptr(b_scales), M, N, K, fmt, layout, _ptr(c), limit_ns,
                                          _stream_ptr(stream, a_codes)))
    return c


def mx_gemm(a_codes, a_scales, b_codes, b_scales, K: int, fmt, layout=SWIZZLED, alpha: float = 1.0,
            *, c=None, group=GROUP, stream=None):
    """C[M, N] = alpha * dequant(A) @ dequant(B)^T (bf16) from MX codes and E8M0 scales as
    mx_quantize returns them (A: [M, K/2 or K] codes, B: [N, ...])."""
    M, N, c = _gemm_operands(a_codes, a_scales, b_codes, b_scales, K, fmt, c)
    _check(lib().mx_gemm(_ptr(a_codes), _ptr(a_scales), _ptr(b_codes), _ptr(b_scales), M, N, K,
                         fmt, group, layout, alpha, _ptr(c), _stream_ptr(stream, a_codes)))
    return c
