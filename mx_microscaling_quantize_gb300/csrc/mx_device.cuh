// mx_device.cuh -- device arithmetic shared by the MX kernels (sm_103a).
//
// Block scale: for a block with abs-max amax (fp32 bits, sign cleared) the E8M0 byte is
// max(E - emax, 0) where E is amax's biased exponent: that is floor(log2 amax) - emax + 127
// clamped below at 0 (s = -127), and 0 for an all-zero block. E = 255 (Inf/NaN) gives 0xFF.
// Element codes come from the hardware's paired converters (round to nearest even, saturate
// to the largest finite value); the sign bit is OR-ed in from the input so that values that
// round to zero keep their sign.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace mxq {

constexpr int kFmtE2M1 = 1;
constexpr int kFmtE4M3 = 2;

template <int FMT>
struct FormatTraits;
template <>
struct FormatTraits<kFmtE2M1> {
  static constexpr uint32_t emax = 2;
};
template <>
struct FormatTraits<kFmtE4M3> {
  static constexpr uint32_t emax = 8;
};

// ------------------------------------------------------------------------------------------
// scales
// ------------------------------------------------------------------------------------------
template <int FMT>
__device__ __forceinline__ uint32_t scale_byte_from_amax_bits(uint32_t amax_f32_bits) {
  const uint32_t E = amax_f32_bits >> 23;
  const uint32_t emax = FormatTraits<FMT>::emax;
  return E == 255u ? 255u : (E > emax ? E - emax : 0u);
}

// 2^-(byte - 127) as fp32 (exact, normal for byte <= 253).
__device__ __forceinline__ float inv_scale_of(uint32_t byte) {
  const uint32_t b = byte > 253u ? 253u : byte;
  return __uint_as_float((254u - b) << 23);
}

// 2^(byte - 127) as fp32 (byte 0 -> 2^-127, an fp32 subnormal).
__device__ __forceinline__ float scale_of(uint32_t byte) {
  return byte ? __uint_as_float(byte << 23) : __uint_as_float(0x00400000u);
}

__device__ __forceinline__ uint32_t max_u16x2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.u16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ------------------------------------------------------------------------------------------
// element conversions (lo = lower K index = low nibble / low byte / low half)
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cvt_e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ uint32_t cvt_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float half_bits_to_f32(uint32_t h) {
  return __half2float(__ushort_as_half((unsigned short)h));
}

// one byte of two E2M1 codes -> two fp32 values (exact)
__device__ __forceinline__ void e2m1x2_to_f32(uint32_t byte, float& lo, float& hi) {
  uint32_t h2;
  asm("{\n\t.reg .b8 t;\n\tcvt.u8.u32 t, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, t;\n\t}"
      : "=r"(h2)
      : "r"(byte));
  lo = half_bits_to_f32(h2 & 0xFFFFu);
  hi = half_bits_to_f32(h2 >> 16);
}

// two E4M3 codes (low byte first) -> two fp32 values (exact)
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t pair, float& lo, float& hi) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)pair));
  lo = half_bits_to_f32(h2 & 0xFFFFu);
  hi = half_bits_to_f32(h2 >> 16);
}

// two fp32 -> packed bf16x2 (round to nearest even, subnormals kept)
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Sign bits of a bf16 pair placed where an E2M1 code byte / an E4M3 code pair keeps them.
__device__ __forceinline__ uint32_t e2m1_signs_of_bf16x2(uint32_t w) {
  return ((w >> 12) & 0x8u) | ((w >> 24) & 0x80u);
}
__device__ __forceinline__ uint32_t e4m3_signs_of_bf16x2(uint32_t w) {
  return ((w >> 8) & 0x80u) | ((w >> 16) & 0x8000u);
}
__device__ __forceinline__ uint32_t e2m1_signs_of_f32x2(float lo, float hi) {
  return ((__float_as_uint(lo) >> 28) & 0x8u) | ((__float_as_uint(hi) >> 24) & 0x80u);
}
__device__ __forceinline__ uint32_t e4m3_signs_of_f32x2(float lo, float hi) {
  return ((__float_as_uint(lo) >> 24) & 0x80u) | ((__float_as_uint(hi) >> 16) & 0x8000u);
}

// ------------------------------------------------------------------------------------------
// 8 bf16 elements (one 16-byte vector) -> codes / QDQ, given the block's scale.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t quant8_e2m1_bf16(const uint4& v, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t out = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t b = cvt_e2m1x2(bf16_lo(w[i]) * inv, bf16_hi(w[i]) * inv) | e2m1_signs_of_bf16x2(w[i]);
    out |= b << (8 * i);
  }
  return out;
}

__device__ __forceinline__ uint2 quant8_e4m3_bf16(const uint4& v, float inv) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
  uint32_t p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    p[i] = cvt_e4m3x2(bf16_lo(w[i]) * inv, bf16_hi(w[i]) * inv) | e4m3_signs_of_bf16x2(w[i]);
  }
  return make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
}

// dequantize 8 E2M1 codes (4 bytes) under scale `sc` -> 8 bf16
__device__ __forceinline__ uint4 dequant8_e2m1(uint32_t codes, float sc) {
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float lo, hi;
    e2m1x2_to_f32((codes >> (8 * i)) & 0xFFu, lo, hi);
    o[i] = pack_bf16x2(lo * sc, hi * sc);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// dequantize 8 E4M3 codes (8 bytes) under scale `sc` -> 8 bf16
__device__ __forceinline__ uint4 dequant8_e4m3(uint2 codes, float sc) {
  const uint32_t c[4] = {codes.x & 0xFFFFu, codes.x >> 16, codes.y & 0xFFFFu, codes.y >> 16};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float lo, hi;
    e4m3x2_to_f32(c[i], lo, hi);
    o[i] = pack_bf16x2(lo * sc, hi * sc);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// ------------------------------------------------------------------------------------------
// 8 fp32 elements -> codes (rotated path)
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t quant8_e2m1_f32(const float* y, float inv) {
  uint32_t out = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = y[2 * i], hi = y[2 * i + 1];
    uint32_t b = cvt_e2m1x2(lo * inv, hi * inv) | e2m1_signs_of_f32x2(lo, hi);
    out |= b << (8 * i);
  }
  return out;
}

__device__ __forceinline__ uint2 quant8_e4m3_f32(const float* y, float inv) {
  uint32_t p[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float lo = y[2 * i], hi = y[2 * i + 1];
    p[i] = cvt_e4m3x2(lo * inv, hi * inv) | e4m3_signs_of_f32x2(lo, hi);
  }
  return make_uint2(p[0] | (p[1] << 16), p[2] | (p[3] << 16));
}

constexpr uint32_t kE4M3NaNx4 = 0x7F7F7F7Fu;
constexpr uint32_t kBf16NaNx2 = 0x7FC07FC0u;

// Swizzled scale position of (r, c) inside one 128x4 tile.
__device__ __forceinline__ int swizzle_in_tile(int r, int c) {
  return (r & 31) * 16 + (r >> 5) * 4 + c;
}

}  // namespace mxq
