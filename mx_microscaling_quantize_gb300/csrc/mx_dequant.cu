// mx_dequant.cu -- stored MX codes + E8M0 block scales -> bf16 (HBM-bound streaming kernel).
//
// Codes are a flat sequence of 32-element blocks (16 bytes per block for packed E2M1, 32 for
// E4M3) and the bf16 output a flat sequence of 64-byte blocks, so a persistent grid walks the
// blocks with a grid stride, consecutive threads on consecutive blocks, each thread loading
// its next block's codes and scale byte before converting the current one. A code pair is
// decoded exactly by the hardware paired converter to f16x2, widened, multiplied by 2^s in
// fp32 (exact: the product of a 2- or 4-bit significand and a power of two is an fp32 number
// whenever it is at least 2^-149 in magnitude, which covers every code down to 2^-9 * 2^-127)
// and rounded once to bf16, which is where subnormal results and overflow to infinity happen.
// Scale byte 0xFF (the E8M0 NaN) and E4M3 NaN codes give the bf16 NaN 0x7FC0.
// NVFP4 data is the same packed E2M1 stream with one E4M3 scale per 16 elements: a thread's
// 32-element chunk holds two blocks whose scale bytes are adjacent in both layouts; each block's
// factor is decode(scale) / gs (one IEEE division), applied like the MX power of two.
#include "mx_device.cuh"
#include "mx_launch.h"

namespace mxq {

namespace {

constexpr int kThreads = 256;

// 2 codes (one E2M1 byte, low nibble = lower K index) -> bf16x2 of code * sc
__device__ __forceinline__ uint32_t dq2_e2m1(uint32_t byte, float sc) {
  uint32_t r;
  asm("{\n\t.reg .b8 c;\n\t.reg .b16 a, b;\n\t.reg .b32 h;\n\t.reg .f32 f0, f1;\n\t"
      "cvt.u8.u32 c, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 h, c;\n\t"
      "mov.b32 {a, b}, h;\n\t"
      "cvt.f32.f16 f0, a;\n\tcvt.f32.f16 f1, b;\n\t"
      "mul.rn.f32 f0, f0, %2;\n\tmul.rn.f32 f1, f1, %2;\n\t"
      "cvt.rn.bf16x2.f32 %0, f1, f0;\n\t}"
      : "=r"(r)
      : "r"(byte), "f"(sc));
  return r;
}

// 2 codes (two E4M3 bytes, low byte = lower K index) -> bf16x2 of code * sc
__device__ __forceinline__ uint32_t dq2_e4m3(uint32_t pair, float sc) {
  uint32_t r;
  asm("{\n\t.reg .b16 c, a, b;\n\t.reg .b32 h;\n\t.reg .f32 f0, f1;\n\t"
      "cvt.u16.u32 c, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 h, c;\n\t"
      "mov.b32 {a, b}, h;\n\t"
      "cvt.f32.f16 f0, a;\n\tcvt.f32.f16 f1, b;\n\t"
      "mul.rn.f32 f0, f0, %2;\n\tmul.rn.f32 f1, f1, %2;\n\t"
      "cvt.rn.bf16x2.f32 %0, f1, f0;\n\t}"
      : "=r"(r)
      : "r"(pair), "f"(sc));
  return r;
}

// bf16 halves of w that are NaN replaced by 0x7FC0
__device__ __forceinline__ uint32_t canonical_nan2(uint32_t w) {
  const uint32_t nan = ((w & 0x7FFF7FFFu) + 0x007F007Fu) & 0x80008000u;  // |h| > 0x7F80
  const uint32_t m = (nan >> 15) * 0xFFFFu;
  return (w & ~m) | (kBf16NaNx2 & m);
}

template <int FMT>
struct CodeBlock {
  static constexpr int kWords = FMT == kFmtE4M3 ? 8 : 4;  // 32-bit words of codes per block
  uint32_t w[kWords];
  uint32_t scale;  // NVFP4: the two blocks' E4M3 bytes, first in the low byte
};

template <int FMT>
__device__ __forceinline__ void load_block(const uint8_t* codes, int64_t b, CodeBlock<FMT>& cb) {
  if (FMT == kFmtE4M3) load32B(codes + b * 32, cb.w);
  else load16B(codes + b * 16, cb.w);
}

// Iterations per warp whose codes are prefetched into L2 before pdl_wait. Measured on GB300
// (steady, back to back, x[8192, 8192]): 4 spans took E4M3 linear from 35.1 to 34.2 us and
// E2M1 swizzled from 28.4 to 28.0 us; 1 or 2 spans changed nothing measurable.
constexpr int kPrefetchSpans = 4;

// Minimum of one CTA per SM: the compiler may then use 55-79 registers (4 or 3 CTAs per SM
// instead of 5 at 48), which measured 5-8% faster back to back (E2M1 swizzled x[8192,8192]
// 29.6 -> 28.2 us, NVFP4 30.6 -> 28.2 us).
template <int FMT, bool SWZ>
__global__ void __launch_bounds__(kThreads, 1) mx_dequant_kernel(DequantArgs a) {
  pdl_launch_dependents();
  {
    // L2 prefetch (before pdl_wait: a hint, see prefetch_l2) of the codes of this warp's first
    // kPrefetchSpans iterations, 32 blocks each: 2 KiB (E2M1) or 4 KiB (E4M3) per warp.
    const int64_t nblk0 = a.M * (a.K >> 5);
    const int64_t w0 = (int64_t)blockIdx.x * kThreads + (threadIdx.x & ~31u);
    const int64_t ws = (int64_t)gridDim.x * kThreads;
    constexpr int kCodeBytes = FMT == kFmtE4M3 ? 32 : 16;
    if ((threadIdx.x & 31) == 0) {
#pragma unroll
      for (int d = 0; d < kPrefetchSpans; ++d) {
        const int64_t s0 = w0 + d * ws;
        if (s0 < nblk0) {
          const int64_t n = nblk0 - s0 < 32 ? nblk0 - s0 : 32;
          prefetch_l2(static_cast<const uint8_t*>(a.codes) + s0 * kCodeBytes,
                      (uint32_t)(n * kCodeBytes));
        }
      }
    }
  }
  pdl_wait();
  const uint8_t* codes = static_cast<const uint8_t*>(a.codes);
  const int64_t cblk = a.K >> 5;
  const int64_t nblk = a.M * cblk;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  int64_t b = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t row_step = stride / cblk, col_step = stride - row_step * cblk;
  int64_t row = b / cblk, col = b - row * cblk;  // advanced incrementally (swizzled scales)
  auto scale_at = [&](int64_t r, int64_t c, int64_t flat) -> uint32_t {
    if (FMT == kFmtNVFP4) {  // scale columns 2c and 2c + 1: adjacent bytes, 2-byte aligned
      const int64_t off = SWZ ? swizzled_offset(r, 2 * c, a.scale_cols) : 2 * flat;
      return load_u16(a.scales + off);
    }
    return load_u8(a.scales + (SWZ ? swizzled_offset(r, c, a.scale_cols) : flat));
  };
  const float gs = FMT == kFmtNVFP4 ? load_f32(a.gscale) : 0.0f;
  CodeBlock<FMT> cur, nxt;
  if (b < nblk) {
    load_block<FMT>(codes, b, cur);
    cur.scale = scale_at(row, col, b);
  }
  for (; b < nblk; b += stride) {
    col += col_step;
    row += row_step;
    if (col >= cblk) {
      col -= cblk;
      ++row;
    }
    const int64_t bn = b + stride;
    if (bn < nblk) {  // next block in flight while this one is converted
      load_block<FMT>(codes, bn, nxt);
      nxt.scale = scale_at(row, col, bn);
    }
    float sc0, sc1;  // factors of elements 0-15 and 16-31 (one MX scale: equal)
    if (FMT == kFmtNVFP4) {
      float d0, d1;
      e4m3x2_to_f32(cur.scale, d0, d1);
      sc0 = d0 == 0.0f ? 0.0f : __fdiv_rn(d0, gs);
      sc1 = d1 == 0.0f ? 0.0f : __fdiv_rn(d1, gs);
    } else {
      sc0 = sc1 = scale_of(cur.scale);
    }
    uint32_t o[16];
    uint32_t nan_codes = 0;
#pragma unroll
    for (int i = 0; i < CodeBlock<FMT>::kWords; ++i) {
      const uint32_t w = cur.w[i];
      if (FMT != kFmtE4M3) {
#pragma unroll
        for (int j = 0; j < 4; ++j) o[4 * i + j] = dq2_e2m1((w >> (8 * j)) & 0xFFu, i < 2 ? sc0 : sc1);
      } else {
        o[2 * i] = dq2_e4m3(w & 0xFFFFu, sc0);
        o[2 * i + 1] = dq2_e4m3(w >> 16, sc0);
        nan_codes |= (w & 0x7F7F7F7Fu) + 0x01010101u;  // a byte reaches 0x80 iff it is S.1111.111
      }
    }
    if (FMT == kFmtNVFP4) {
      const bool nan0 = (cur.scale & 0x7Fu) == 0x7Fu, nan1 = ((cur.scale >> 8) & 0x7Fu) == 0x7Fu;
      if (nan0 || nan1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) o[i] = (i < 8 ? nan0 : nan1) ? kBf16NaNx2 : o[i];
      }
    } else if (cur.scale == 255u) {
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i] = kBf16NaNx2;
    } else if (FMT == kFmtE4M3 && (nan_codes & 0x80808080u)) {
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i] = canonical_nan2(o[i]);
    }
    uint8_t* y = static_cast<uint8_t*>(a.y) + b * 64;
    store32B(y, o);
    store32B(y + 32, o + 8);
    cur = nxt;
  }
}

template <int FMT, bool SWZ>
cudaError_t launch_t(const DequantArgs& a, cudaStream_t stream) {
  const void* k = reinterpret_cast<const void*>(&mx_dequant_kernel<FMT, SWZ>);
  const int64_t need = (a.M * (a.K >> 5) + kThreads - 1) / kThreads;
  if (need <= 0) return cudaSuccess;
  const int resident = resident_ctas(k, kThreads, 0, 0);
  if (resident <= 0) return cudaErrorInvalidConfiguration;
  const int grid = (int)(need < resident ? need : resident);
  return launch_pdl(&mx_dequant_kernel<FMT, SWZ>, dim3(grid), dim3(kThreads), 0, stream, a);
}

}  // namespace

cudaError_t launch_dequant(int fmt, bool swizzled, const DequantArgs& a, cudaStream_t stream) {
  if (fmt == kFmtE2M1) {
    return swizzled ? launch_t<kFmtE2M1, true>(a, stream) : launch_t<kFmtE2M1, false>(a, stream);
  }
  if (fmt == kFmtNVFP4) {
    return swizzled ? launch_t<kFmtNVFP4, true>(a, stream) : launch_t<kFmtNVFP4, false>(a, stream);
  }
  return swizzled ? launch_t<kFmtE4M3, true>(a, stream) : launch_t<kFmtE4M3, false>(a, stream);
}

}  // namespace mxq
