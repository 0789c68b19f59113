// mx_oracle.cpp -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, double-precision CPU definition of OCP-MX block quantization, written to be
// checked by eye against its sources. Only the test suite, the smoke check and the benchmark's
// CPU-baseline leg may load it; the product library never does, and the two share no code.
//
// Sources for each step (pages cited by title and section):
//  * "[Transform] [Quantization] Add QuTLASS support to vLLM" (vllm PR 24440), feature list
//    "Multiple quantization schemes ... Abs-Max" and "Support for both NVFP4 and MXFP4": the
//    abs-max shared scale over a block; "Online rotations ... Rotation matrices loaded at runtime,
//    allowing any transformation ... Multiple rotation sizes (16/32/64/128)": the per-chunk
//    rotation y = x_chunk * H; review thread on vllm/_custom_ops.py (`xh_e2m1`, `xh_e8m0` with
//    `padded_rows, padded_cols`) and on vllm/qutlass_utils/utils.py (`to_blocked`): packed E2M1
//    codes, E8M0 scales and the padded blocked scale layout.
//  * "use cute-dsl to speedup mxfp QDQ" (intel/neural-compressor PR 2548), description: MXFP4 and
//    MXFP8 QDQ with group size 32 along K, K divisible by 32.
//  * prhub summary of vllm PR 47229, code snippet of mxfp8_utils.py: MXFP8_BLOCK_SIZE = 32,
//    E4M3 codes plus scales, linear scales viewed as [M, K/32] when not swizzled.
// The pages print no formula for the scale, no value grid and no rounding rule. The steps below
// take the plainest reading of the OCP MX formats that the pages name:
//   scale exponent s = floor(log2(amax)) - emax, clamped to [-127, 127], stored as s + 127;
//   element code = nearest member of the format's finite grid to x / 2^s, ties to the code
//   with an even mantissa, magnitudes above the grid maximum saturate to it, sign kept.
// The Quest-like MXFP4 scale (quest_scale_byte) is a further reading, stated where it is defined:
// the pages name the scheme but give no rule.
// Parity of this file is pinned by the CPU tests (format definitions, closed forms, brute force,
// torch's float8_e4m3fn casts, invariants); see tests/test_oracle_pins.py.

#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

namespace {

// ---------------------------------------------------------------------------------------------
// Element formats.  Format ids used by this file only: 1 = E2M1 (MXFP4), 2 = E4M3 (MXFP8).
// ---------------------------------------------------------------------------------------------
struct ElementFormat {
  int emax;          // exponent of the largest binade of the format
  int sign_bit;      // code bit that carries the sign
  int n_magnitudes;  // number of finite non-negative codes 0 .. n-1
  double magnitude[128];
};

// E2M1: 1 sign, 2 exponent bits (bias 1), 1 mantissa bit, no Inf/NaN.
ElementFormat make_e2m1() {
  ElementFormat f{};
  f.emax = 2;
  f.sign_bit = 0x8;
  f.n_magnitudes = 8;
  for (int c = 0; c < 8; ++c) {
    int e = (c >> 1) & 0x3;
    int m = c & 0x1;
    f.magnitude[c] = (e == 0) ? m * 0.5 : (1.0 + m / 2.0) * std::ldexp(1.0, e - 1);
  }
  return f;
}

// E4M3 ("fn" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no Inf, only
// S.1111.111 is NaN. Finite non-negative codes are 0x00 .. 0x7E.
ElementFormat make_e4m3() {
  ElementFormat f{};
  f.emax = 8;
  f.sign_bit = 0x80;
  f.n_magnitudes = 127;
  for (int c = 0; c < 127; ++c) {
    int e = (c >> 3) & 0xF;
    int m = c & 0x7;
    f.magnitude[c] = (e == 0) ? m * std::ldexp(1.0, -9) : (1.0 + m / 8.0) * std::ldexp(1.0, e - 7);
  }
  return f;
}

const ElementFormat kE2M1 = make_e2m1();
const ElementFormat kE4M3 = make_e4m3();

const ElementFormat* format_of(int fmt) {
  if (fmt == 1) return &kE2M1;
  if (fmt == 2) return &kE4M3;
  return nullptr;
}

// ---------------------------------------------------------------------------------------------
// bf16 <-> double.
// ---------------------------------------------------------------------------------------------
double bf16_to_double(uint16_t b) {
  int sign = b >> 15;
  int e = (b >> 7) & 0xFF;
  int m = b & 0x7F;
  double v;
  if (e == 0xFF) {
    v = (m != 0) ? NAN : INFINITY;
  } else if (e == 0) {
    v = std::ldexp((double)m, -133);  // subnormal: m * 2^-133
  } else {
    v = std::ldexp((double)(128 + m), e - 134);  // (1 + m/128) * 2^(e-127)
  }
  return sign ? -v : v;
}

// Encode a double that is exactly representable in bf16.
uint16_t bf16_bits_exact(double a_nonneg) {
  if (a_nonneg < std::ldexp(1.0, -126)) {
    return (uint16_t)(a_nonneg / std::ldexp(1.0, -133));  // subnormal mantissa (128 == 2^-126)
  }
  int ex;
  std::frexp(a_nonneg, &ex);  // a = f * 2^ex, f in [0.5, 1)
  int e = ex - 1;             // a in [2^e, 2^(e+1))
  int m = (int)(a_nonneg / std::ldexp(1.0, e - 7)) - 128;
  return (uint16_t)(((e + 127) << 7) | m);
}

// Round a double to bf16 once, to nearest, ties to even.
uint16_t double_to_bf16_rne(double v) {
  if (std::isnan(v)) return 0x7FC0;
  uint16_t sign = std::signbit(v) ? 0x8000 : 0;
  double a = std::fabs(v);
  if (a == 0.0) return sign;
  if (std::isinf(a)) return sign | 0x7F80;
  int ex;
  std::frexp(a, &ex);
  int e = ex - 1;
  int quantum_exp = (e < -126) ? -133 : e - 7;  // spacing of the bf16 grid around a
  double q = std::ldexp(a, -quantum_exp);       // exact
  double lower = std::floor(q);
  double frac = q - lower;
  double n = lower;
  if (frac > 0.5 || (frac == 0.5 && std::fmod(lower, 2.0) == 1.0)) n = lower + 1.0;
  double r = std::ldexp(n, quantum_exp);
  if (r >= std::ldexp(1.0, 128)) return sign | 0x7F80;
  return sign | bf16_bits_exact(r);
}

// ---------------------------------------------------------------------------------------------
// One MX block: shared scale + element codes.
// ---------------------------------------------------------------------------------------------

// Nearest grid member to |t| by exhaustive search; ties go to the even code. Magnitudes at or
// above the largest grid value saturate to it (done first: far above the grid the distances
// themselves round to equal doubles).
int nearest_magnitude_code(const ElementFormat& f, double abs_t) {
  if (abs_t >= f.magnitude[f.n_magnitudes - 1]) return f.n_magnitudes - 1;
  int best = 0;
  double best_err = std::fabs(f.magnitude[0] - abs_t);
  for (int c = 1; c < f.n_magnitudes; ++c) {
    double err = std::fabs(f.magnitude[c] - abs_t);
    if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
      best = c;
      best_err = err;
    }
  }
  return best;
}

// Shared scale byte of a block from its abs-max (finite amax only).
int scale_byte_from_amax(const ElementFormat& f, double amax) {
  if (amax == 0.0) return 0;  // all-zero block: smallest scale, all codes zero
  int ex;
  std::frexp(amax, &ex);
  int e = ex - 1;  // floor(log2(amax))
  int s = e - f.emax;
  if (s < -127) s = -127;
  if (s > 127) s = 127;
  return s + 127;
}

// Quantize one block of n values. forced_byte < 0: derive the scale from the block's abs-max;
// otherwise use the given E8M0 byte. Writes one unpacked code per value; returns the scale byte.
// A block holding a NaN or an infinity gets scale byte 0xFF (E8M0 NaN) and fill codes
// (E4M3: 0x7F, E2M1: 0x0); the pages leave this case open.
int quantize_block(const ElementFormat& f, const double* v, int n, int forced_byte, uint8_t* codes) {
  bool special = false;
  double amax = 0.0;
  for (int i = 0; i < n; ++i) {
    if (std::isnan(v[i]) || std::isinf(v[i])) special = true;
    else if (std::fabs(v[i]) > amax) amax = std::fabs(v[i]);
  }
  if (special && forced_byte < 0) {
    for (int i = 0; i < n; ++i) codes[i] = (f.sign_bit == 0x80) ? 0x7F : 0x0;
    return 0xFF;
  }
  int byte = (forced_byte >= 0) ? forced_byte : scale_byte_from_amax(f, amax);
  int s = byte - 127;
  for (int i = 0; i < n; ++i) {
    double t = std::ldexp(v[i], -s);  // exact
    int code = nearest_magnitude_code(f, std::fabs(t));
    if (std::signbit(t)) code |= f.sign_bit;
    codes[i] = (uint8_t)code;
  }
  return byte;
}

// ---------------------------------------------------------------------------------------------
// Quartet / "Quest-like" block scale for MXFP4. The QuTLASS page names the scheme (feature list,
// "Multiple quantization schemes": "Quartet (i.e., Quest-like)") and its call (review thread on
// vllm/_custom_ops.py: fusedQuantizeMxQuest(a, b, xh_e2m1, xh_e8m0) writes the E2M1 codes and
// E8M0 scales of the rotated input), but prints no rule. Reading taken: the shared scale follows
// the MX rule with the block's clip point c in place of its abs-max,
//   RMS = sqrt(sum_i v_i^2 / n),  c = alpha * RMS,
//   s = floor(log2 c) - emax(E2M1) clamped to [-127, 127], stored as s + 127 (c == 0: byte 0),
// where alpha is the clip ratio (clip point over standard deviation) that minimises the mean
// squared error of the E2M1 grid, stretched so that its largest value 6 sits at the clip point,
// on a standard normal variable (the Gaussian clipping of the QuEST method). The elements then
// follow quantize_block under that byte: values above 6 * 2^s saturate, which is the clipping.
// ---------------------------------------------------------------------------------------------
const double kQuestAlpha = 2.922475;  // the minimiser, to 7 significant digits

// Scale byte of a block of n finite values under the reading above.
int quest_scale_byte(const double* v, int n) {
  double sum_sq = 0.0;
  for (int i = 0; i < n; ++i) sum_sq += v[i] * v[i];
  const double c = kQuestAlpha * std::sqrt(sum_sq / n);
  if (c == 0.0) return 0;
  int ex;
  std::frexp(c, &ex);
  int s = (ex - 1) - kE2M1.emax;  // floor(log2 c) - emax
  if (s < -127) s = -127;
  if (s > 127) s = 127;
  return s + 127;
}

// quantize_block with the scale from quest_scale_byte (E2M1 elements). A block holding a NaN or
// an infinity gets byte 0xFF and codes 0, as in quantize_block.
int quantize_block_quest(const double* v, int n, uint8_t* codes) {
  for (int i = 0; i < n; ++i) {
    if (std::isnan(v[i]) || std::isinf(v[i])) return quantize_block(kE2M1, v, n, -1, codes);
  }
  return quantize_block(kE2M1, v, n, quest_scale_byte(v, n), codes);
}

// Scale schemes of the tensor operations below: 0 = abs-max (quantize_block), 1 = Quest-like
// (quantize_block_quest, E2M1 only).
int block_with_scheme(const ElementFormat& f, int scheme, const double* v, uint8_t* codes) {
  return scheme == 1 ? quantize_block_quest(v, 32, codes) : quantize_block(f, v, 32, -1, codes);
}

// Value of one code at scale 2^0. E4M3 S.1111.111 (0x7F, 0xFF) is the format's NaN.
double decode_code(const ElementFormat& f, int code) {
  int magnitude_code = code & (f.sign_bit - 1);
  if (magnitude_code >= f.n_magnitudes) return NAN;
  double mag = f.magnitude[magnitude_code];
  return (code & f.sign_bit) ? -mag : mag;
}

// Dequantize one code under an E8M0 scale byte, rounded to bf16 once.
uint16_t dequant_to_bf16(const ElementFormat& f, int code, int scale_byte) {
  if (scale_byte == 0xFF) return 0x7FC0;
  return double_to_bf16_rne(std::ldexp(decode_code(f, code), scale_byte - 127));
}

// ---------------------------------------------------------------------------------------------
// Scale layouts.
// ---------------------------------------------------------------------------------------------
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// 128x4 blocked layout consumed by block-scaled GEMMs: the [rows, cols] scale matrix is padded
// to [ceil(rows/128)*128, ceil(cols/4)*4] and cut into 128x4 tiles stored one after another in
// row-block-major order (512 bytes each). Inside a tile, scale (r, c) sits at
// (r % 32) * 16 + (r / 32) * 4 + c, with r in [0,128) and c in [0,4).
int64_t swizzled_offset(int64_t r, int64_t c, int64_t padded_cols) {
  int64_t tile = (r / 128) * (padded_cols / 4) + (c / 4);
  int64_t rr = r % 128;
  return tile * 512 + (rr % 32) * 16 + (rr / 32) * 4 + (c % 4);
}

// Quantize `rows` rows of `v` (doubles, row-major [rows, K]) whose first row is row `row0` of the
// scale matrix. layout 0 = linear [*, K/32], 1 = swizzled.
void quantize_rows(const ElementFormat& f, const double* v, int64_t rows, int64_t K, int64_t row0,
                   int layout, int64_t padded_cols, uint8_t* codes, uint8_t* scales,
                   int scheme = 0) {
  const int64_t groups = K / 32;
  uint8_t block_codes[32];
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t j = 0; j < groups; ++j) {
      int byte = block_with_scheme(f, scheme, v + r * K + j * 32, block_codes);
      if (layout == 0) {
        scales[(row0 + r) * groups + j] = (uint8_t)byte;
      } else {
        scales[swizzled_offset(row0 + r, j, padded_cols)] = (uint8_t)byte;
      }
      for (int i = 0; i < 32; ++i) {
        int64_t k = j * 32 + i;
        if (f.sign_bit == 0x80) {
          codes[r * K + k] = block_codes[i];
        } else {
          // two E2M1 codes per byte, the lower K index in the low nibble
          uint8_t& b = codes[r * (K / 2) + k / 2];
          if (k % 2 == 0) b = (uint8_t)((b & 0xF0) | block_codes[i]);
          else b = (uint8_t)((b & 0x0F) | (block_codes[i] << 4));
        }
      }
    }
  }
}

void qdq_rows(const ElementFormat& f, const double* v, int64_t rows, int64_t K, uint16_t* out,
              int scheme = 0) {
  uint8_t block_codes[32];
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t j = 0; j < K / 32; ++j) {
      int byte = block_with_scheme(f, scheme, v + r * K + j * 32, block_codes);
      for (int i = 0; i < 32; ++i) {
        out[r * K + j * 32 + i] = dequant_to_bf16(f, block_codes[i], byte);
      }
    }
  }
}

// Dequantize [rows, K] codes (E4M3: one byte each; E2M1: two per byte, the lower K index in the
// low nibble) under their block scales (linear [rows, K/32] or swizzled) into bf16.
void dequantize_rows(const ElementFormat& f, const uint8_t* codes, const uint8_t* scales,
                     int64_t rows, int64_t K, int layout, int64_t padded_cols, uint16_t* out) {
  const int64_t groups = K / 32;
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t j = 0; j < groups; ++j) {
      int byte = (layout == 0) ? scales[r * groups + j] : scales[swizzled_offset(r, j, padded_cols)];
      for (int i = 0; i < 32; ++i) {
        int64_t k = j * 32 + i;
        int code;
        if (f.sign_bit == 0x80) {
          code = codes[r * K + k];
        } else {
          uint8_t b = codes[r * (K / 2) + k / 2];
          code = (k % 2 == 0) ? (b & 0x0F) : (b >> 4);
        }
        out[r * K + k] = dequant_to_bf16(f, code, byte);
      }
    }
  }
}

std::vector<double> decode_rows(const uint16_t* x, int64_t rows, int64_t K) {
  std::vector<double> v((size_t)(rows * K));
  for (int64_t i = 0; i < rows * K; ++i) v[(size_t)i] = bf16_to_double(x[i]);
  return v;
}

// y = x_chunk * H for every g-element chunk along K; H is g x g row-major (H[i*g + j]).
// Every output y_j = sum over i = 0 .. g-1 of x_i * H[i][j], added in increasing i starting
// from 0: the loop takes input i in turn and adds x_i times row i of H to the whole chunk.
std::vector<double> rotate_rows(const uint16_t* x, int64_t rows, int64_t K, const uint16_t* H, int g) {
  std::vector<double> h((size_t)g * g);
  for (int i = 0; i < g * g; ++i) h[(size_t)i] = bf16_to_double(H[i]);
  std::vector<double> y((size_t)(rows * K), 0.0);
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t c0 = 0; c0 < K; c0 += g) {
      double* yc = y.data() + r * K + c0;
      for (int i = 0; i < g; ++i) {
        const double xi = bf16_to_double(x[r * K + c0 + i]);
        const double* hrow = h.data() + (size_t)i * g;
        for (int j = 0; j < g; ++j) yc[j] += xi * hrow[j];
      }
    }
  }
  return y;
}

// ---------------------------------------------------------------------------------------------
// NVFP4: E2M1 elements in blocks of 16 along K, one E4M3 scale per block under a per-tensor fp32
// global scale gs. The QuTLASS page names the format ("Support for both NVFP4 and MXFP4") and
// the call fusedQuantizeNv(a, H, global_scale) whose blocked scales are viewed as [-1, K/16]
// (review thread on benchmarks/kernels/bench_nvfp4_qutlass.py), but prints no scale rule. The
// reading taken is the usual two-level one, with every step an fp32 operation (round to nearest
// even), in this order:
//   r6 = gs / 6;  s_f = amax * r6;  sc = E4M3(s_f) (nearest even, saturating at 448);
//   enc = gs / decode(sc) (0 when decode(sc) == 0);  code_i = E2M1(v_i * enc);
//   QDQ: dq = decode(sc) / gs (0 when decode(sc) == 0);  y_i = bf16(decode(code_i) * dq).
// A block holding a NaN or an infinity gets scale byte 0x7F (the E4M3 NaN), codes 0 and QDQ
// outputs 0x7FC0. Values v_i are fp32 (bf16 inputs widen exactly; rotated values are rounded to
// fp32 once).
// ---------------------------------------------------------------------------------------------
int e4m3_code_of_nonneg(float v) { return nearest_magnitude_code(kE4M3, (double)v); }

// Quantize one block of n fp32 values; writes unpacked E2M1 codes, returns the E4M3 scale byte.
int nvfp4_block(const float* v, int n, float gs, uint8_t* codes) {
  bool special = false;
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    if (std::isnan(v[i]) || std::isinf(v[i])) special = true;
    else if (std::fabs(v[i]) > amax) amax = std::fabs(v[i]);
  }
  if (special) {
    for (int i = 0; i < n; ++i) codes[i] = 0;
    return 0x7F;
  }
  const float r6 = gs / 6.0f;
  const float s_f = amax * r6;
  const int sc = e4m3_code_of_nonneg(s_f);
  const float s_dec = (float)kE4M3.magnitude[sc];
  const float enc = (s_dec == 0.0f) ? 0.0f : gs / s_dec;
  for (int i = 0; i < n; ++i) {
    const float t = v[i] * enc;
    int code = nearest_magnitude_code(kE2M1, std::fabs((double)t));
    if (std::signbit(t)) code |= 0x8;
    codes[i] = (uint8_t)code;
  }
  return sc;
}

// decode(sc) is the signed E4M3 value of the scale byte (the quantizer only writes
// non-negative ones; stored data given to the dequantize may carry the sign bit).
uint16_t nvfp4_dequant_to_bf16(int code, int scale_byte, float gs) {
  if (scale_byte == 0x7F || scale_byte == 0xFF) return 0x7FC0;
  const float s_mag = (float)kE4M3.magnitude[scale_byte & 0x7F];
  const float s_dec = (scale_byte & 0x80) ? -s_mag : s_mag;
  const float dq = (s_dec == 0.0f) ? 0.0f : s_dec / gs;
  const float y = (float)decode_code(kE2M1, code) * dq;
  return double_to_bf16_rne((double)y);
}

// rows of fp32 values [rows, K] -> packed codes [rows, K/2], scales (linear [rows, K/16] or
// swizzled with padded_cols columns) and/or QDQ bf16 (either output may be null)
void nvfp4_rows(const float* v, int64_t rows, int64_t K, float gs, int layout, int64_t padded_cols,
                uint8_t* codes, uint8_t* scales, uint16_t* qdq) {
  const int64_t groups = K / 16;
  uint8_t bc[16];
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t j = 0; j < groups; ++j) {
      const int sc = nvfp4_block(v + r * K + j * 16, 16, gs, bc);
      if (scales) {
        if (layout == 0) scales[r * groups + j] = (uint8_t)sc;
        else scales[swizzled_offset(r, j, padded_cols)] = (uint8_t)sc;
      }
      for (int i = 0; i < 16; ++i) {
        const int64_t k = j * 16 + i;
        if (codes) {
          uint8_t& b = codes[r * (K / 2) + k / 2];
          if (k % 2 == 0) b = (uint8_t)((b & 0xF0) | bc[i]);
          else b = (uint8_t)((b & 0x0F) | (bc[i] << 4));
        }
        if (qdq) qdq[r * K + k] = nvfp4_dequant_to_bf16(bc[i], sc, gs);
      }
    }
  }
}

std::vector<float> bf16_rows_to_float(const uint16_t* x, int64_t n) {
  std::vector<float> v((size_t)n);
  for (int64_t i = 0; i < n; ++i) v[(size_t)i] = (float)bf16_to_double(x[i]);
  return v;
}

std::vector<float> doubles_to_float(const std::vector<double>& y) {
  std::vector<float> v(y.size());
  for (size_t i = 0; i < y.size(); ++i) v[i] = (float)y[i];
  return v;
}

}  // namespace

// ---------------------------------------------------------------------------------------------
// C interface (ctypes). All pointers are host memory owned by the caller.
// fmt: 1 = E2M1 (MXFP4), 2 = E4M3 (MXFP8). layout: 0 = linear, 1 = swizzled 128x4.
// ---------------------------------------------------------------------------------------------
extern "C" {

int mxo_emax(int fmt) { return format_of(fmt)->emax; }

double mxo_decode(int fmt, int code) { return decode_code(*format_of(fmt), code); }

double mxo_bf16_to_double(uint16_t b) { return bf16_to_double(b); }

uint16_t mxo_double_to_bf16(double v) { return double_to_bf16_rne(v); }

int mxo_scale_byte(int fmt, double amax) { return scale_byte_from_amax(*format_of(fmt), amax); }

int mxo_quantize_block(int fmt, const double* v, int n, int forced_byte, uint8_t* codes) {
  return quantize_block(*format_of(fmt), v, n, forced_byte, codes);
}

uint16_t mxo_dequant_bf16(int fmt, int code, int scale_byte) {
  return dequant_to_bf16(*format_of(fmt), code, scale_byte);
}

int64_t mxo_swizzled_offset(int64_t r, int64_t c, int64_t padded_cols) {
  return swizzled_offset(r, c, padded_cols);
}

// Scale matrix shape for an [M, K] input.
void mxo_scales_shape(int64_t M, int64_t K, int layout, int64_t* rows, int64_t* cols) {
  if (layout == 0) {
    *rows = M;
    *cols = K / 32;
  } else {
    *rows = ceil_div(M, 128) * 128;
    *cols = ceil_div(K / 32, 4) * 4;
  }
}

// codes: E4M3 [M, K] bytes, E2M1 [M, K/2] bytes. scales: see mxo_scales_shape (pads zeroed here).
void mxo_quantize(const uint16_t* x, int64_t M, int64_t K, int fmt, int layout, uint8_t* codes,
                  uint8_t* scales) {
  int64_t srows, scols;
  mxo_scales_shape(M, K, layout, &srows, &scols);
  std::memset(scales, 0, (size_t)(srows * scols));
  std::vector<double> v = decode_rows(x, M, K);
  quantize_rows(*format_of(fmt), v.data(), M, K, 0, layout, scols, codes, scales);
}

void mxo_qdq(const uint16_t* x, int64_t M, int64_t K, int fmt, uint16_t* out) {
  std::vector<double> v = decode_rows(x, M, K);
  qdq_rows(*format_of(fmt), v.data(), M, K, out);
}

// codes / scales as mxo_quantize writes them -> bf16 bits [M, K].
void mxo_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t M, int64_t K, int fmt,
                    int layout, uint16_t* out) {
  int64_t srows, scols;
  mxo_scales_shape(M, K, layout, &srows, &scols);
  dequantize_rows(*format_of(fmt), codes, scales, M, K, layout, scols, out);
}

void mxo_rotate(const uint16_t* x, int64_t M, int64_t K, const uint16_t* H, int g, double* y) {
  std::vector<double> v = rotate_rows(x, M, K, H, g);
  std::memcpy(y, v.data(), sizeof(double) * (size_t)(M * K));
}

void mxo_rotate_quantize(const uint16_t* x, int64_t M, int64_t K, const uint16_t* H, int g, int fmt,
                         int layout, uint8_t* codes, uint8_t* scales) {
  int64_t srows, scols;
  mxo_scales_shape(M, K, layout, &srows, &scols);
  std::memset(scales, 0, (size_t)(srows * scols));
  std::vector<double> y = rotate_rows(x, M, K, H, g);
  quantize_rows(*format_of(fmt), y.data(), M, K, 0, layout, scols, codes, scales);
}

void mxo_rotate_qdq(const uint16_t* x, int64_t M, int64_t K, const uint16_t* H, int g, int fmt,
                    uint16_t* out) {
  std::vector<double> y = rotate_rows(x, M, K, H, g);
  qdq_rows(*format_of(fmt), y.data(), M, K, out);
}

// Quantize / QDQ of values given as doubles, [M, K] row-major (the rotated values mxo_rotate
// returns, for instance): the same steps as mxo_quantize / mxo_qdq after the bf16 decode.
void mxo_quantize_values(const double* v, int64_t M, int64_t K, int fmt, int layout, uint8_t* codes,
                         uint8_t* scales) {
  int64_t srows, scols;
  mxo_scales_shape(M, K, layout, &srows, &scols);
  std::memset(scales, 0, (size_t)(srows * scols));
  quantize_rows(*format_of(fmt), v, M, K, 0, layout, scols, codes, scales);
}

void mxo_qdq_values(const double* v, int64_t M, int64_t K, int fmt, uint16_t* out) {
  qdq_rows(*format_of(fmt), v, M, K, out);
}

// Quest-like scale (see quest_scale_byte): the constant, the byte of one block of n finite
// values, one block's codes, and the tensor operations on float64 values [M, K] (bf16 inputs
// decoded, or the rotated values of mxo_rotate), E2M1 elements.
double mxo_quest_alpha() { return kQuestAlpha; }

int mxo_quest_scale_byte(const double* v, int n) { return quest_scale_byte(v, n); }

int mxo_quest_quantize_block(const double* v, int n, uint8_t* codes) {
  return quantize_block_quest(v, n, codes);
}

void mxo_quest_quantize_values(const double* v, int64_t M, int64_t K, int layout, uint8_t* codes,
                               uint8_t* scales) {
  int64_t srows, scols;
  mxo_scales_shape(M, K, layout, &srows, &scols);
  std::memset(scales, 0, (size_t)(srows * scols));
  quantize_rows(kE2M1, v, M, K, 0, layout, scols, codes, scales, 1);
}

void mxo_quest_qdq_values(const double* v, int64_t M, int64_t K, uint16_t* out) {
  qdq_rows(kE2M1, v, M, K, out, 1);
}

// Grouped (MoE) quantize: rows [offsets[e], offsets[e+1]) belong to expert e. Codes stay
// contiguous. Linear scales are [M_total, K/32]. Swizzled scales give every expert its own
// run of 128-row blocks: expert e starts at padded row P_e = sum_{e'<e} ceil(n_e'/128)*128.
// `scale_rows` is the number of rows of the scale buffer (all of it is written, pads zero).
void mxo_quantize_grouped(const uint16_t* x, const int64_t* offsets, int E, int64_t K, int fmt,
                          int layout, int64_t scale_rows, uint8_t* codes, uint8_t* scales) {
  const ElementFormat& f = *format_of(fmt);
  int64_t M_total = offsets[E];
  int64_t scols = (layout == 0) ? K / 32 : ceil_div(K / 32, 4) * 4;
  std::memset(scales, 0, (size_t)(scale_rows * scols));
  int64_t code_row_bytes = (fmt == 2) ? K : K / 2;
  int64_t padded_row = 0;
  for (int e = 0; e < E; ++e) {
    int64_t r0 = offsets[e];
    int64_t n = offsets[e + 1] - offsets[e];
    std::vector<double> v = decode_rows(x + r0 * K, n, K);
    int64_t scale_row0 = (layout == 0) ? r0 : padded_row;
    quantize_rows(f, v.data(), n, K, scale_row0, layout, scols, codes + r0 * code_row_bytes, scales);
    padded_row += ceil_div(n, 128) * 128;
  }
  (void)M_total;
}

// NVFP4 (see the reading above). Scale shapes: linear [M, K/16]; swizzled
// [ceil(M/128)*128, ceil(K/16/4)*4] (pads zeroed here). H may be null (no rotation).
void mxo_nvfp4_scales_shape(int64_t M, int64_t K, int layout, int64_t* rows, int64_t* cols) {
  if (layout == 0) {
    *rows = M;
    *cols = K / 16;
  } else {
    *rows = ceil_div(M, 128) * 128;
    *cols = ceil_div(K / 16, 4) * 4;
  }
}

int mxo_nvfp4_block(const float* v, int n, float gs, uint8_t* codes) {
  return nvfp4_block(v, n, gs, codes);
}

uint16_t mxo_nvfp4_dequant_bf16(int code, int scale_byte, float gs) {
  return nvfp4_dequant_to_bf16(code, scale_byte, gs);
}

void mxo_nvfp4_quantize(const uint16_t* x, int64_t M, int64_t K, const uint16_t* H, int g, float gs,
                        int layout, uint8_t* codes, uint8_t* scales) {
  int64_t srows, scols;
  mxo_nvfp4_scales_shape(M, K, layout, &srows, &scols);
  std::memset(scales, 0, (size_t)(srows * scols));
  std::memset(codes, 0, (size_t)(M * (K / 2)));
  std::vector<float> v = H ? doubles_to_float(rotate_rows(x, M, K, H, g)) : bf16_rows_to_float(x, M * K);
  nvfp4_rows(v.data(), M, K, gs, layout, scols, codes, scales, nullptr);
}

void mxo_nvfp4_qdq(const uint16_t* x, int64_t M, int64_t K, const uint16_t* H, int g, float gs,
                   uint16_t* out) {
  std::vector<float> v = H ? doubles_to_float(rotate_rows(x, M, K, H, g)) : bf16_rows_to_float(x, M * K);
  nvfp4_rows(v.data(), M, K, gs, 0, 0, nullptr, nullptr, out);
}

// NVFP4 of values given as doubles [M, K] (rotated values, for instance), each rounded to fp32
// once first; any of codes, scales, qdq may be null. Scales as mxo_nvfp4_quantize lays them out
// (pads zeroed here).
void mxo_nvfp4_values(const double* y, int64_t M, int64_t K, float gs, int layout, uint8_t* codes,
                      uint8_t* scales, uint16_t* qdq) {
  int64_t srows, scols;
  mxo_nvfp4_scales_shape(M, K, layout, &srows, &scols);
  if (scales) std::memset(scales, 0, (size_t)(srows * scols));
  if (codes) std::memset(codes, 0, (size_t)(M * (K / 2)));
  std::vector<float> v((size_t)(M * K));
  for (int64_t i = 0; i < M * K; ++i) v[(size_t)i] = (float)y[i];
  nvfp4_rows(v.data(), M, K, gs, layout, scols, codes, scales, qdq);
}

// Grouped (MoE) NVFP4 quantize: rows [offsets[e], offsets[e+1]) are expert e's input, quantized
// under that expert's own global scale gs[e]. Codes stay in row order. Linear scales are
// [M_total, K/16] in row order; swizzled scales give each expert its own run of 128-row tiles
// starting at padded row P_e = sum_{e' < e} ceil(n_e' / 128) * 128 (pads zero), as for the MX
// grouped layout.
void mxo_nvfp4_quantize_grouped(const uint16_t* x, const int64_t* offsets, int E, int64_t K,
                                const float* gs, int layout, int64_t scale_rows, uint8_t* codes,
                                uint8_t* scales) {
  int64_t srows, scols;
  mxo_nvfp4_scales_shape(0, K, layout, &srows, &scols);
  std::memset(scales, 0, (size_t)(scale_rows * scols));
  std::memset(codes, 0, (size_t)(offsets[E] * (K / 2)));
  int64_t padded_row = 0;
  for (int e = 0; e < E; ++e) {
    const int64_t r0 = offsets[e], n = offsets[e + 1] - offsets[e];
    std::vector<float> v = bf16_rows_to_float(x + r0 * K, n * K);
    const int64_t scale_row0 = (layout == 0) ? r0 : padded_row;
    nvfp4_rows(v.data(), n, K, gs[e], layout, scols, codes + r0 * (K / 2),
               scales + scale_row0 * scols, nullptr);
    padded_row += ceil_div(n, 128) * 128;
  }
}

// Stored NVFP4 data -> bf16: element k of row r is dequantized with the scale of its 16-element
// block (linear [M, K/16] or swizzled as mxo_nvfp4_scales_shape says).
void mxo_nvfp4_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t M, int64_t K,
                          float gs, int layout, uint16_t* y) {
  int64_t srows, scols;
  mxo_nvfp4_scales_shape(M, K, layout, &srows, &scols);
  for (int64_t r = 0; r < M; ++r) {
    for (int64_t k = 0; k < K; ++k) {
      const uint8_t b = codes[r * (K / 2) + k / 2];
      const int code = (k % 2 == 0) ? (b & 0x0F) : (b >> 4);
      const int64_t j = k / 16;
      const int sc = layout == 0 ? scales[r * (K / 16) + j] : scales[swizzled_offset(r, j, scols)];
      y[r * K + k] = nvfp4_dequant_to_bf16(code, sc, gs);
    }
  }
}

}  // extern "C"
