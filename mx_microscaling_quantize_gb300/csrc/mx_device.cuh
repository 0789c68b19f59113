// mx_device.cuh -- device arithmetic shared by the MX kernels (sm_103a).
//
// Block scale: for a block with abs-max amax (fp32 bits, sign cleared) the E8M0 byte is
// max(E - emax, 0) where E is amax's biased exponent: that is floor(log2 amax) - emax + 127
// clamped below at 0 (s = -127), and 0 for an all-zero block. E = 255 (Inf/NaN) gives 0xFF.
// Element codes come from the hardware's paired converters cvt.rn.satfinite.{e2m1x2,e4m3x2}:
// round to nearest even, saturate to the largest finite value, and keep the sign of values
// that round to zero (a property the exhaustive parity sweep checks against the oracle). The
// first source of a paired conversion lands in the upper nibble / byte / half, so the higher K
// index is passed first. Multiplying by 2^-s is exact (no overflow; an underflow only touches
// values far below half the smallest code).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace mxq {

constexpr int kFmtE2M1 = 1;
constexpr int kFmtE4M3 = 2;
constexpr int kFmtNVFP4 = 3;  // E2M1 elements, 16-element blocks, E4M3 scales, fp32 global scale
constexpr int kFmtE2M1Quest = 4;  // MXFP4 with the Quest-like scale (quest_byte_from_sum)

// MX formats with E2M1 elements (4-bit codes, two per byte) and E8M0 block scales.
template <int FMT>
__host__ __device__ constexpr bool mx_e2m1() {
  return FMT == kFmtE2M1 || FMT == kFmtE2M1Quest;
}

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
template <>
struct FormatTraits<kFmtNVFP4> {  // element format E2M1; the block scale is not a power of two
  static constexpr uint32_t emax = 2;
};
template <>
struct FormatTraits<kFmtE2M1Quest> {
  static constexpr uint32_t emax = 2;
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

// 2^-(byte - 127) as fp32, exact: normal for byte <= 253, the subnormal 2^-127 for 254 (reached
// only by the Quest-like scale; multiplying by it is exact wherever the product is normal). 255
// (NaN blocks, whose outputs are replaced) gives 2^-127 too.
__device__ __forceinline__ float inv_scale_of(uint32_t byte) {
  return byte >= 254u ? __uint_as_float(0x00400000u) : __uint_as_float((254u - byte) << 23);
}

// Quest-like block scale (QuTLASS page, feature list: "Quartet (i.e., Quest-like)"; the pages
// print no rule, so the reading is the MX rule with the block's clip point c in place of its
// abs-max): c = alpha * sqrt(sum v_i^2 / 32), alpha = 2.922475 the clip ratio minimising the
// E2M1 grid's mean squared error on a standard normal variable; byte = floor(log2 c) - 2 + 127
// clamped to [0, 254]; an all-zero block gives 0 and a block with a NaN or an infinity 0xFF.
// Every kernel first adds the plain squares of the block's values with fp32 FMAs in one fixed
// order (sq_sum); when that sum lies in [2^-80, 2^100] it is accurate to a few units in the last
// place (no overflow, and squares below 2^-126 are negligible against it) and decides the byte
// with e = 127. Otherwise (a NaN or an infinity, an overflow, a tiny block) the squares are
// summed again after an exact scaling by quest_prescale(E), E the abs-max's exponent field,
// which neither overflows nor loses bits for any finite input. The decision needs no square
// root: floor(log2 c) = (e - 127) + floor(floor(log2 p) / 2) for p = sum * alpha^2 / 32, the sum
// taken over the values times 2^(127 - e).
constexpr float kQuestBeta = (float)(2.922475 * 2.922475 / 32.0);  // alpha^2 / 32

// 2^(127 - e), e = E clamped to [1, 253] (normal): the block's largest scaled value lies in [1, 4)
// (below 1 only for a subnormal abs-max), so the scaled squares lie in [2^-46, 16).
__device__ __forceinline__ float quest_prescale(uint32_t E) {
  const uint32_t e = E < 1u ? 1u : (E > 253u ? 253u : E);
  return __uint_as_float((254u - e) << 23);
}

// The range in which the plain sum of squares decides the byte: [2^-80, 2^100] (NaN excluded).
__device__ __forceinline__ bool quest_sum_in_range(float sum_sq) {
  return __float_as_uint(sum_sq) - 0x17800000u <= 0x71800000u - 0x17800000u;
}

__device__ __forceinline__ uint32_t quest_byte_from_sum(float sum_scaled_sq, uint32_t E) {
  if (E == 255u) return 255u;
  if (sum_scaled_sq == 0.0f) return 0u;
  const int e = E < 1u ? 1 : (E > 253u ? 253 : (int)E);
  const float p = sum_scaled_sq * kQuestBeta;  // normal: in [2^-48, 2^8)
  const int lp = (int)(__float_as_uint(p) >> 23) - 127;  // floor(log2 p)
  const int b = e - 2 + (lp >> 1);                        // arithmetic shift: floor(lp / 2)
  return b < 0 ? 0u : (b > 254 ? 254u : (uint32_t)b);
}

// (lo, hi) <- (lo, hi) + (a, b)^2, one packed fp32 FMA per pair
__device__ __forceinline__ void fma_sq2(float& lo, float& hi, float a, float b) {
  asm("{\n\t.reg .b64 p, q;\n\tmov.b64 p, {%2, %3};\n\tmov.b64 q, {%0, %1};\n\t"
      "fma.rn.f32x2 q, p, p, q;\n\tmov.b64 {%0, %1}, q;\n\t}"
      : "+f"(lo), "+f"(hi)
      : "f"(a), "f"(b));
}

// 2^(byte - 127) as fp32 (byte 0 -> 2^-127, an fp32 subnormal).
__device__ __forceinline__ float scale_of(uint32_t byte) {
  return byte ? __uint_as_float(byte << 23) : __uint_as_float(0x00400000u);
}

// ------------------------------------------------------------------------------------------
// building blocks
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// (lo, hi) *= s with one packed fp32 multiply (exact here: s is a power of two)
__device__ __forceinline__ void mul2(float& lo, float& hi, float s) {
  asm("{\n\t.reg .b64 p, q;\n\tmov.b64 p, {%0, %1};\n\tmov.b64 q, {%2, %2};\n\t"
      "mul.rn.f32x2 p, p, q;\n\tmov.b64 {%0, %1}, p;\n\t}"
      : "+f"(lo), "+f"(hi)
      : "f"(s));
}

// max(|a|, |b|, |c|) in one instruction; NaN if any input is NaN.
__device__ __forceinline__ float absmax3(float a, float b, float c) {
  float d;
  asm("max.NaN.abs.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// abs-max of 16 fp32 values as sign-free fp32 bits; NaN propagates.
__device__ __forceinline__ uint32_t absmax_f32x16(const float* y) {
  // three-input tree: 16 -> 6 -> 2 -> 1 in 8 instructions
  float m[6];
#pragma unroll
  for (int i = 0; i < 5; ++i) m[i] = absmax3(y[3 * i], y[3 * i + 1], y[3 * i + 2]);
  m[5] = y[15];
  const float p = absmax3(m[0], m[1], m[2]), q = absmax3(m[3], m[4], m[5]);
  return __float_as_uint(absmax3(p, q, q)) & 0x7FFFFFFFu;
}

// abs-max of 32 fp32 values as sign-free fp32 bits; NaN propagates.
__device__ __forceinline__ uint32_t absmax_f32x32(const float* y) {
  // three-input tree: 32 -> 11 -> 4 -> 1 in 17 instructions
  float m[11];
#pragma unroll
  for (int i = 0; i < 10; ++i) m[i] = absmax3(y[3 * i], y[3 * i + 1], y[3 * i + 2]);
  m[10] = absmax3(y[30], y[31], y[31]);
  const float p0 = absmax3(m[0], m[1], m[2]), p1 = absmax3(m[3], m[4], m[5]);
  const float p2 = absmax3(m[6], m[7], m[8]), p3 = absmax3(m[9], m[10], m[10]);
  return __float_as_uint(absmax3(absmax3(p0, p1, p2), p3, p3)) & 0x7FFFFFFFu;
}

// Sum of the squares of n fp32 values (n % 4 == 0): four interleaved chains (value i goes to
// chain i % 4), then (c0 + c1) + (c2 + c3). Every kernel adds a 32-value block in this order.
template <int N>
__device__ __forceinline__ float sq_sum(const float* y) {
  float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
#pragma unroll
  for (int i = 0; i < N; i += 4) {
    fma_sq2(s0, s1, y[i], y[i + 1]);
    fma_sq2(s2, s3, y[i + 2], y[i + 3]);
  }
  return (s0 + s1) + (s2 + s3);
}

// The same sum with every value scaled by m first (exact: m is a power of two).
template <int N>
__device__ __forceinline__ float scaled_sq_sum(const float* y, float m) {
  float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
#pragma unroll
  for (int i = 0; i < N; i += 4) {
    float a = y[i], b = y[i + 1], c = y[i + 2], d = y[i + 3];
    mul2(a, b, m);
    mul2(c, d, m);
    fma_sq2(s0, s1, a, b);
    fma_sq2(s2, s3, c, d);
  }
  return (s0 + s1) + (s2 + s3);
}

// Quest-like scale byte of one block of 32 fp32 values, given their plain sum of squares.
__device__ __forceinline__ uint32_t quest_byte_f32x32(const float* y, float sum_sq) {
  if (quest_sum_in_range(sum_sq)) return quest_byte_from_sum(sum_sq, 127u);
  const uint32_t E = absmax_f32x32(y) >> 23;
  return quest_byte_from_sum(scaled_sq_sum<32>(y, quest_prescale(E)), E);
}
__device__ __forceinline__ uint32_t quest_byte_f32x32(const float* y) {
  return quest_byte_f32x32(y, sq_sum<32>(y));
}

// ------------------------------------------------------------------------------------------
// 8 scaled fp32 values t[0..8) (lower K index first) -> codes
// ------------------------------------------------------------------------------------------
// The four code bytes are widened and shifted into place; the vector form of mov from four
// 8-bit registers is not used (one kernel was seen to get zeros from it).
__device__ __forceinline__ uint32_t codes8_e2m1(const float* t) {
  uint32_t r = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t b;
    asm("{\n\t.reg .b8 c;\n\tcvt.rn.satfinite.e2m1x2.f32 c, %1, %2;\n\tcvt.u32.u8 %0, c;\n\t}"
        : "=r"(b)
        : "f"(t[2 * j + 1]), "f"(t[2 * j]));
    r |= b << (8 * j);
  }
  return r;
}

__device__ __forceinline__ uint2 codes8_e4m3(const float* t) {
  uint32_t a, b;
  asm("{\n\t.reg .b16 c0, c1, c2, c3;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 c0, %3, %2;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 c1, %5, %4;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 c2, %7, %6;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 c3, %9, %8;\n\t"
      "mov.b32 %0, {c0, c1};\n\tmov.b32 %1, {c2, c3};\n\t}"
      : "=r"(a), "=r"(b)
      : "f"(t[0]), "f"(t[1]), "f"(t[2]), "f"(t[3]), "f"(t[4]), "f"(t[5]), "f"(t[6]), "f"(t[7]));
  return make_uint2(a, b);
}

// ------------------------------------------------------------------------------------------
// QDQ of two scaled values (lo = lower K index): round to the grid with the hardware
// converter, decode exactly to f16x2, widen, multiply by the scale, round once to bf16x2.
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t qdq2_e2m1(float tlo, float thi, float sc) {
  uint32_t r;
  asm("{\n\t.reg .b8 c;\n\t.reg .b16 a, b;\n\t.reg .b32 h;\n\t.reg .f32 f0, f1;\n\t"
      "cvt.rn.satfinite.e2m1x2.f32 c, %2, %1;\n\t"
      "cvt.rn.f16x2.e2m1x2 h, c;\n\t"
      "mov.b32 {a, b}, h;\n\t"
      "cvt.f32.f16 f0, a;\n\tcvt.f32.f16 f1, b;\n\t"
      "mul.rn.f32 f0, f0, %3;\n\tmul.rn.f32 f1, f1, %3;\n\t"
      "cvt.rn.bf16x2.f32 %0, f1, f0;\n\t}"
      : "=r"(r)
      : "f"(tlo), "f"(thi), "f"(sc));
  return r;
}

__device__ __forceinline__ uint32_t qdq2_e4m3(float tlo, float thi, float sc) {
  uint32_t r;
  asm("{\n\t.reg .b16 c, a, b;\n\t.reg .b32 h;\n\t.reg .f32 f0, f1;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 c, %2, %1;\n\t"
      "cvt.rn.f16x2.e4m3x2 h, c;\n\t"
      "mov.b32 {a, b}, h;\n\t"
      "cvt.f32.f16 f0, a;\n\tcvt.f32.f16 f1, b;\n\t"
      "mul.rn.f32 f0, f0, %3;\n\tmul.rn.f32 f1, f1, %3;\n\t"
      "cvt.rn.bf16x2.f32 %0, f1, f0;\n\t}"
      : "=r"(r)
      : "f"(tlo), "f"(thi), "f"(sc));
  return r;
}

template <int FMT>
__device__ __forceinline__ uint32_t qdq2(float tlo, float thi, float sc) {
  return mx_e2m1<FMT>() ? qdq2_e2m1(tlo, thi, sc) : qdq2_e4m3(tlo, thi, sc);
}

constexpr uint32_t kE4M3NaNx4 = 0x7F7F7F7Fu;
constexpr uint32_t kBf16NaNx2 = 0x7FC07FC0u;

// Byte offset of scale (padded row pr, column c) in the 128x4 tiles (cp padded columns).
__device__ __forceinline__ int64_t swizzled_offset(int64_t pr, int64_t c, int64_t cp) {
  return ((pr >> 7) * (cp >> 2) + (c >> 2)) * 512 + (pr & 31) * 16 + ((pr >> 5) & 3) * 4 + (c & 3);
}

// Loads of kernel inputs. Every one is a coherent ld.global, never the non-coherent (.nc,
// __ldg) path: a kernel launched with programmatic stream serialization (see pdl_wait) runs
// while the kernel before it may still be writing what it reads, and .nc loads are defined
// only for data that stays unchanged for the whole life of the kernel (the compiler may also
// schedule them early). Each is an asm volatile, so it stays after pdl_wait in program order.
// 32-byte vector load, not kept in L1 (streamed once).
__device__ __forceinline__ void load32B(const void* p, uint32_t* r) {
  asm volatile("ld.global.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "l"(p));
}

__device__ __forceinline__ void load16B(const void* p, uint32_t* r) {
  asm volatile("ld.global.L1::no_allocate.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "l"(p));
}

// 16-byte vector load (kept in L1: small operands read by many threads, such as H)
__device__ __forceinline__ uint4 load_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

__device__ __forceinline__ float load_f32(const float* p) {
  float v;
  asm volatile("ld.global.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t load_u16(const void* p) {
  uint16_t v;
  asm volatile("ld.global.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ uint32_t load_u8(const void* p) {
  uint16_t v;
  asm volatile("ld.global.u8 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

__device__ __forceinline__ int64_t load_s64(const int64_t* p) {
  int64_t v;
  asm volatile("ld.global.s64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}

// 32-byte vector store, evict-first (written once, not re-read by this kernel).
__device__ __forceinline__ void store32B(void* p, const uint32_t* r) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// ------------------------------------------------------------------------------------------
// NVFP4 block scales. For a block of 16 values with abs-max amax under the global scale gs,
// every step is one fp32 operation rounded to nearest even, in this order:
//   s_f = amax * r6 (r6 = gs / 6);  sc = E4M3(s_f), saturating at 448;
//   enc = gs / decode(sc);  code_i = E2M1(v_i * enc);
//   QDQ: y_i = bf16(decode(code_i) * dq), dq = decode(sc) / gs;
// enc and dq are 0 when decode(sc) is 0. A block holding a NaN or an infinity gets scale byte
// 0x7F (the E4M3 NaN), codes 0 and QDQ outputs 0x7FC0 (the caller applies these fills).
// ------------------------------------------------------------------------------------------
struct NvScales {
  uint32_t bytes;  // E4M3 scale bytes of two consecutive blocks, the first in the low byte
  float enc[2];
  float dq[2];
  bool special[2];
};

// two E4M3 bytes (low byte first) -> exact fp32 values (every finite E4M3 value is an f16)
__device__ __forceinline__ void e4m3x2_to_f32(uint32_t pair, float& lo, float& hi) {
  asm("{\n\t.reg .b16 c, a, b;\n\t.reg .b32 h;\n\tcvt.u16.u32 c, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 h, c;\n\tmov.b32 {a, b}, h;\n\t"
      "cvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
      : "=f"(lo), "=f"(hi)
      : "r"(pair));
}

// amax0/amax1: sign-free fp32 bits of the two blocks' abs-max (Inf/NaN at or above 0x7F800000).
// Returns the two E4M3 scale bytes (first in the low byte; 0x7F for a block holding a NaN or an
// infinity) and sets the blocks' special flags.
__device__ __forceinline__ uint32_t nv_scale_pair(uint32_t amax0, uint32_t amax1, float r6,
                                                  bool* special) {
  const float s0 = __fmul_rn(__uint_as_float(amax0), r6);
  const float s1 = __fmul_rn(__uint_as_float(amax1), r6);
  uint32_t pair;
  asm("{\n\t.reg .b16 c;\n\tcvt.rn.satfinite.e4m3x2.f32 c, %1, %2;\n\tcvt.u32.u16 %0, c;\n\t}"
      : "=r"(pair)
      : "f"(s1), "f"(s0));
  special[0] = amax0 >= 0x7F800000u;
  special[1] = amax1 >= 0x7F800000u;
  if (special[0]) pair = (pair & 0xFF00u) | 0x007Fu;
  if (special[1]) pair = (pair & 0x00FFu) | 0x7F00u;
  return pair;
}

__device__ __forceinline__ NvScales nv_scales(uint32_t amax0, uint32_t amax1, float gs, float r6) {
  NvScales n;
  const uint32_t pair = nv_scale_pair(amax0, amax1, r6, n.special);
  float d0, d1;
  e4m3x2_to_f32(pair, d0, d1);
  n.enc[0] = d0 == 0.0f ? 0.0f : __fdiv_rn(gs, d0);
  n.enc[1] = d1 == 0.0f ? 0.0f : __fdiv_rn(gs, d1);
  n.dq[0] = d0 == 0.0f ? 0.0f : __fdiv_rn(d0, gs);
  n.dq[1] = d1 == 0.0f ? 0.0f : __fdiv_rn(d1, gs);
  n.bytes = pair;
  return n;
}

// The per-scale-byte factors of one global scale, for b in [0, 128): enc = gs / decode(b) and
// dq = decode(b) / gs (0 where decode(b) is 0), the same fp32 divisions nv_scales performs, so
// that a kernel can tabulate them once and look them up (nv_scales_tab) with identical results.
__device__ __forceinline__ void nv_factors_of_byte(uint32_t b, float gs, float& enc, float& dq) {
  float d, unused;
  e4m3x2_to_f32(b, d, unused);
  enc = d == 0.0f ? 0.0f : __fdiv_rn(gs, d);
  dq = d == 0.0f ? 0.0f : __fdiv_rn(d, gs);
}

// nv_scales with the factors looked up in tables t_enc / t_dq built by nv_factors_of_byte
// (indexed by the byte's low 7 bits; a special block's 0x7F reads the NaN entry, and its outputs
// are replaced by the caller anyway).
__device__ __forceinline__ NvScales nv_scales_tab(uint32_t amax0, uint32_t amax1, float r6,
                                                  const float* t_enc, const float* t_dq) {
  NvScales n;
  const uint32_t pair = nv_scale_pair(amax0, amax1, r6, n.special);
  n.enc[0] = t_enc[pair & 0x7Fu];
  n.enc[1] = t_enc[(pair >> 8) & 0x7Fu];
  n.dq[0] = t_dq[pair & 0x7Fu];
  n.dq[1] = t_dq[(pair >> 8) & 0x7Fu];
  n.bytes = pair;
  return n;
}

// ------------------------------------------------------------------------------------------
// One thread's 32 fp32 values (rotated values, lower K index first) -> output words.
// ------------------------------------------------------------------------------------------
// NVFP4: two 16-element blocks under the scales n (from nv_scales or nv_scales_tab). Writes 16
// words of bf16 QDQ output or 4 words of E2M1 codes; a NaN/Inf block gets 0x7FC0 / codes 0.
// Every lane of the warp must call it.
template <bool QDQ>
__device__ __forceinline__ void nv_block_f32(float* y, uint32_t* out, const NvScales& n) {
  const bool special = __any_sync(0xFFFFFFFFu, n.special[0] || n.special[1]);
#pragma unroll
  for (int i = 0; i < 16; ++i) mul2(y[2 * i], y[2 * i + 1], n.enc[i >> 3]);  // y <- y * enc
  if (QDQ) {
#pragma unroll
    for (int i = 0; i < 16; ++i) out[i] = qdq2_e2m1(y[2 * i], y[2 * i + 1], n.dq[i >> 3]);
    if (special) {
#pragma unroll
      for (int i = 0; i < 16; ++i) out[i] = n.special[i >> 3] ? kBf16NaNx2 : out[i];
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = codes8_e2m1(y + 8 * i);
    if (special) {
#pragma unroll
      for (int i = 0; i < 4; ++i) out[i] = n.special[i >> 1] ? 0u : out[i];
    }
  }
}

// Zeroes the pad bytes of a swizzled scale buffer of a plain (not grouped) call, spread over
// every thread of the grid (t0: this thread's index, nthr: the grid's threads): (A) in each of
// the M data rows, the bytes past column dcols of its last 4-byte word (only when dcols % 4 !=
// 0); (B) every 4-byte word of every pad row (rows M .. scale_rows - 1, as a flat list of
// (row, word) items so that a few wide pad rows do not serialize on a few threads).
__device__ __forceinline__ void zero_swizzled_pads(uint8_t* scales, int64_t M, int64_t dcols,
                                                   int64_t scale_rows, int64_t cp, int64_t t0,
                                                   int64_t nthr) {
  const int64_t cp4 = cp >> 2;
  if (dcols & 3) {
    const int64_t c4 = dcols & ~int64_t(3);
    for (int64_t r = t0; r < M; r += nthr) {
      uint8_t* run = scales + swizzled_offset(r, c4, cp);
      for (int64_t c = dcols; c < c4 + 4; ++c) run[c - c4] = 0;
    }
  }
  const int64_t pad_rows = scale_rows - M;
  for (int64_t i = t0; i < pad_rows * cp4; i += nthr) {
    const int64_t pr = M + i % pad_rows, c4 = (i / pad_rows) * 4;
    *reinterpret_cast<uint32_t*>(scales + swizzled_offset(pr, c4, cp)) = 0u;
  }
}

// Programmatic dependent launch. Every kernel of the library is launched with programmatic
// stream serialization (launch_pdl): its CTAs may be scheduled while the kernel before it on
// the stream is still finishing. Each kernel lets the next one be scheduled as soon as all of
// its own CTAs are running, and waits for the previous kernel to complete (with its memory
// visible) before its first global memory access, so stream order is kept; only set-up that
// touches nothing in global memory (shared memory, barriers, kernel parameters) runs earlier,
// and L2 prefetches of the first input bytes (prefetch_l2 below), which read no value.
// Without a programmatic dependency both instructions have no effect.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// L2 prefetch of [p, p + bytes) (p 16-byte aligned, bytes a multiple of 16, inside one
// allocation). A prefetch is a hint: it returns no data to the thread and has no effect on the
// values any load observes. The kernels issue it for their first input bytes BEFORE pdl_wait,
// while the previous kernel on the stream drains: L2 is the point of coherence of every SM of
// the device, so if that kernel still writes those bytes, its writes update the L2 lines and
// the loads issued after pdl_wait read the new values; they only find the lines on chip
// instead of waiting for DRAM. Measured on GB300, back to back: QDQ of x[8192, 8192]
// 43.4 -> 41.4 us, quantize 2-5% faster, rotate+quantize about 1.1 us less per launch.
__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// Swizzled scale position of (r, c) inside one 128x4 tile.
__device__ __forceinline__ int swizzle_in_tile(int r, int c) {
  return (r & 31) * 16 + (r >> 5) * 4 + c;
}

}  // namespace mxq
