// mx_api.cu -- the extern "C" entry points declared in include/mxq.h: host-side validation,
// shape arithmetic and launch selection. No allocation, no synchronization, no device reads.
#include <climits>
#include <cstdint>

#include "mx_device.cuh"
#include "mx_launch.h"
#include "mxq.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
// x, y and codes are moved with 32-byte vector accesses
bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }
int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
bool valid_fmt(int fmt) { return fmt == MX_FMT_E2M1 || fmt == MX_FMT_E4M3; }
bool valid_layout(int layout) { return layout == MX_SCALES_LINEAR || layout == MX_SCALES_SWIZZLED; }
bool valid_g(int g) { return g == 16 || g == 32 || g == 64 || g == 128; }
bool valid_rot_kind(int k) {
  return k == MX_ROT_DENSE || k == MX_ROT_HADAMARD || k == MX_ROT_AUTO;
}
// Whether a rotated call runs on the Walsh-Hadamard kernel. MX_ROT_HADAMARD: always for g <= 64
// (for g = 128 its two shuffle stages made it 19-42% slower than the tensor-core kernel on every
// measured shape, so those calls run there, which takes any H). MX_ROT_AUTO: the kernel that
// measured faster on GB300 (steady, back to back) for the call's output and shape: the FMA kernel
// for decode-sized calls (M <= 16, M * g <= 512); the Walsh-Hadamard kernel below 4096 rows
// (x[1024, 8192] MXFP4 codes: 6.6 against 7.5 us); from 4096 rows the tensor cores for 4-bit codes
// (x[8192, 8192]: 29.7 against 31.0 us; x[8192, 28672]: 91.3 against 97.3) and, for the wider
// outputs (MXFP8 codes, bf16 QDQ), up to 3 * 2^25 elements (QDQ x[4096, 8192]: 22.6-23.0
// against 23.5-24.5; MXFP8 x[8192, 8192]: 34.1 against 34.8), the Walsh-Hadamard kernel above
// (QDQ x[4096, 28672]: 73.3-74.5 against 77.3-78.4; MXFP8 x[8192, 28672]: 112.3 against 115.6).
// wide_out: MXFP8 codes or QDQ.
bool use_fwht(int rot_kind, int g, bool wide_out, int64_t M, int64_t K) {
  if (g > 64 || rot_kind == MX_ROT_DENSE) return false;
  if (rot_kind == MX_ROT_HADAMARD) return true;
  if (M <= 16 && M * g <= 512) return false;
  if (M < 4096) return true;
  return wide_out && M * K > (int64_t(3) << 25);
}

// Kernel format id of an MX call: the Quest-like scale is its own instantiation of the kernels.
int kernel_fmt(int fmt, int rounding) {
  return rounding == MX_ROUND_QUEST ? mxq::kFmtE2M1Quest : fmt;
}

// Checks shared by every call on an [M, K] bf16 input. Returns MX_OK to go on; *empty is set
// when there is nothing to compute.
mx_status check_common(int64_t M, int64_t K, int fmt, int group, int rounding, bool* empty) {
  if (M < 0 || K < 0) return MX_ERR_SHAPE;
  if (group != 32) return MX_ERR_UNSUPPORTED;
  if (!valid_fmt(fmt)) return MX_ERR_UNSUPPORTED;
  if (rounding != MX_ROUND_RNE && !(rounding == MX_ROUND_QUEST && fmt == MX_FMT_E2M1)) {
    return MX_ERR_UNSUPPORTED;
  }
  if (K % 32 != 0) return MX_ERR_SHAPE;
  // element indices are formed in int64: keep M * K far from overflow
  if (K > 0 && M > (int64_t(1) << 40) / K) return MX_ERR_SHAPE;
  *empty = (M == 0 || K == 0);
  return MX_OK;
}

// the rotation kernels address rows and columns through a 2-D tensor map (32-bit coordinates)
bool fits_tensor_map(int64_t M, int64_t K) { return M <= INT32_MAX && K <= INT32_MAX; }

mx_status from_cuda(cudaError_t err) { return err == cudaSuccess ? MX_OK : MX_ERR_CUDA; }

mxq::RotArgs rot_args(const void* x, int64_t M, int64_t K, const void* H, void* out) {
  mxq::RotArgs a{};
  a.x = x;
  a.H = H;
  a.out = out;
  a.M = M;
  a.K = K;
  a.col_tiles = ceil_div(K, mxq::kTileCols);
  a.row_blocks = ceil_div(M, mxq::kTileRows);
  return a;
}

mxq::StreamArgs stream_args(const void* x, int64_t M, int64_t K, void* out) {
  mxq::StreamArgs a{};
  a.x = x;
  a.out = out;
  a.M = M;
  a.K = K;
  return a;
}

}  // namespace

extern "C" {

const char* mx_status_string(mx_status status) {
  switch (status) {
    case MX_OK: return "MX_OK";
    case MX_ERR_NULL: return "MX_ERR_NULL: a required pointer is NULL";
    case MX_ERR_SHAPE: return "MX_ERR_SHAPE: invalid size (negative, K % 32, K % g, experts)";
    case MX_ERR_ALIGN: return "MX_ERR_ALIGN: a buffer is misaligned (x, y, codes: 32 B; H, scales: 16 B)";
    case MX_ERR_UNSUPPORTED: return "MX_ERR_UNSUPPORTED: format, layout, rounding, group or g";
    case MX_ERR_CUDA: return "MX_ERR_CUDA: the CUDA runtime reported an error at launch";
    default: return "unknown mx_status";
  }
}

mx_status mx_scales_shape(int64_t M, int64_t K, int group, int layout, int64_t* rows,
                          int64_t* cols) {
  if (!rows || !cols) return MX_ERR_NULL;
  if (M < 0 || K < 0 || K % 32 != 0) return MX_ERR_SHAPE;
  if (group != 32 || !valid_layout(layout)) return MX_ERR_UNSUPPORTED;
  if (layout == MX_SCALES_LINEAR) {
    *rows = M;
    *cols = K / 32;
  } else {
    *rows = ceil_div(M, mxq::kTileRows) * mxq::kTileRows;
    *cols = ceil_div(K, mxq::kTileCols) * 4;
  }
  return MX_OK;
}

mx_status mx_grouped_scales_shape(int64_t M_total, int E, int64_t K, int group, int layout,
                                  int64_t* rows, int64_t* cols) {
  if (!rows || !cols) return MX_ERR_NULL;
  if (M_total < 0 || K < 0 || K % 32 != 0 || E < 1 || E > 1024) return MX_ERR_SHAPE;
  if (group != 32 || !valid_layout(layout)) return MX_ERR_UNSUPPORTED;
  if (layout == MX_SCALES_LINEAR) {
    *rows = M_total;
    *cols = K / 32;
  } else {
    *rows = (M_total + int64_t(mxq::kTileRows - 1) * E) / mxq::kTileRows * mxq::kTileRows;
    *cols = ceil_div(K, mxq::kTileCols) * 4;
  }
  return MX_OK;
}

mx_status mx_quantize(const void* x, int64_t M, int64_t K, int fmt, int group, int layout,
                      int rounding, void* codes, void* scales, void* stream) {
  bool empty = false;
  mx_status st = check_common(M, K, fmt, group, rounding, &empty);
  if (st != MX_OK) return st;
  if (!valid_layout(layout)) return MX_ERR_UNSUPPORTED;
  if (empty) return MX_OK;
  if (!x || !codes || !scales) return MX_ERR_NULL;
  if (!aligned32(x) || !aligned32(codes)) return MX_ERR_ALIGN;
  if (layout == MX_SCALES_SWIZZLED && !aligned16(scales)) return MX_ERR_ALIGN;
  mxq::StreamArgs a = stream_args(x, M, K, codes);
  a.scales = static_cast<uint8_t*>(scales);
  a.scale_cols = layout == MX_SCALES_LINEAR ? K / 32 : ceil_div(K, mxq::kTileCols) * 4;
  a.scale_rows = layout == MX_SCALES_LINEAR ? M : ceil_div(M, mxq::kTileRows) * mxq::kTileRows;
  return from_cuda(mxq::launch_stream(kernel_fmt(fmt, rounding), false, layout == MX_SCALES_SWIZZLED,
                                      false, a,
                                      static_cast<cudaStream_t>(stream)));
}

mx_status mx_qdq(const void* x, int64_t M, int64_t K, int fmt, int group, int rounding,
                 const void* H, int g, int rot_kind, void* y, void* stream) {
  bool empty = false;
  mx_status st = check_common(M, K, fmt, group, rounding, &empty);
  if (st != MX_OK) return st;
  if (H) {
    if (!valid_g(g) || !valid_rot_kind(rot_kind)) return MX_ERR_UNSUPPORTED;
    if (K % g != 0 || !fits_tensor_map(M, K)) return MX_ERR_SHAPE;
  }
  if (empty) return MX_OK;
  if (!x || !y) return MX_ERR_NULL;
  if (!aligned32(x) || !aligned32(y)) return MX_ERR_ALIGN;
  if (H) {
    if (!aligned16(H)) return MX_ERR_ALIGN;
    if (use_fwht(rot_kind, g, true, M, K)) {
      mxq::StreamArgs a = stream_args(x, M, K, y);
      a.H = H;
      return from_cuda(mxq::launch_hadamard(kernel_fmt(fmt, rounding), mxq::kRotQdq, false, g, a,
                                            static_cast<cudaStream_t>(stream)));
    }
    return from_cuda(mxq::launch_rotate(kernel_fmt(fmt, rounding), mxq::kRotQdq, false, g,
                                        rot_args(x, M, K, H, y),
                                        static_cast<cudaStream_t>(stream)));
  }
  return from_cuda(mxq::launch_stream(kernel_fmt(fmt, rounding), true, false, false,
                                      stream_args(x, M, K, y),
                                      static_cast<cudaStream_t>(stream)));
}

mx_status mx_dequantize(const void* codes, const void* scales, int64_t M, int64_t K, int fmt,
                        int group, int layout, void* y, void* stream) {
  bool empty = false;
  mx_status st = check_common(M, K, fmt, group, MX_ROUND_RNE, &empty);
  if (st != MX_OK) return st;
  if (!valid_layout(layout)) return MX_ERR_UNSUPPORTED;
  if (empty) return MX_OK;
  if (!codes || !scales || !y) return MX_ERR_NULL;
  if (!aligned32(codes) || !aligned32(y)) return MX_ERR_ALIGN;
  if (layout == MX_SCALES_SWIZZLED && !aligned16(scales)) return MX_ERR_ALIGN;
  mxq::DequantArgs a{};
  a.codes = codes;
  a.scales = static_cast<const uint8_t*>(scales);
  a.y = y;
  a.M = M;
  a.K = K;
  a.scale_cols = layout == MX_SCALES_LINEAR ? K / 32 : ceil_div(K, mxq::kTileCols) * 4;
  return from_cuda(mxq::launch_dequant(fmt, layout == MX_SCALES_SWIZZLED, a,
                                       static_cast<cudaStream_t>(stream)));
}

mx_status mx_rotate_quantize(const void* x, int64_t M, int64_t K, const void* H, int g,
                             int rot_kind, int fmt, int group, int layout, int rounding,
                             void* codes, void* scales, void* stream) {
  bool empty = false;
  mx_status st = check_common(M, K, fmt, group, rounding, &empty);
  if (st != MX_OK) return st;
  if (!valid_layout(layout) || !valid_g(g) || !valid_rot_kind(rot_kind)) return MX_ERR_UNSUPPORTED;
  if (K % g != 0 || !fits_tensor_map(M, K)) return MX_ERR_SHAPE;
  if (empty) return MX_OK;
  if (!x || !H || !codes || !scales) return MX_ERR_NULL;
  if (!aligned32(x) || !aligned32(codes)) return MX_ERR_ALIGN;
  if (layout == MX_SCALES_SWIZZLED && !aligned16(scales)) return MX_ERR_ALIGN;
  if (!aligned16(H)) return MX_ERR_ALIGN;
  if (use_fwht(rot_kind, g, fmt == MX_FMT_E4M3, M, K)) {
    mxq::StreamArgs a = stream_args(x, M, K, codes);
    a.scales = static_cast<uint8_t*>(scales);
    a.scale_cols = layout == MX_SCALES_LINEAR ? K / 32 : ceil_div(K, mxq::kTileCols) * 4;
    a.scale_rows = layout == MX_SCALES_LINEAR ? M : ceil_div(M, mxq::kTileRows) * mxq::kTileRows;
    a.H = H;
    return from_cuda(mxq::launch_hadamard(kernel_fmt(fmt, rounding), mxq::kRotCodes,
                                          layout == MX_SCALES_SWIZZLED, g, a,
                                          static_cast<cudaStream_t>(stream)));
  }
  mxq::RotArgs a = rot_args(x, M, K, H, codes);
  a.scales = static_cast<uint8_t*>(scales);
  a.scale_cols = layout == MX_SCALES_LINEAR ? K / 32 : a.col_tiles * 4;
  return from_cuda(mxq::launch_rotate(kernel_fmt(fmt, rounding), mxq::kRotCodes,
                                      layout == MX_SCALES_SWIZZLED, g, a,
                                      static_cast<cudaStream_t>(stream)));
}

mx_status mx_quantize_grouped(const void* x, const int64_t* row_offsets, int E, int64_t M_total,
                              int64_t K, int fmt, int group, int layout, int rounding,
                              void* codes, void* scales, void* stream) {
  bool empty = false;
  mx_status st = check_common(M_total, K, fmt, group, rounding, &empty);
  if (st != MX_OK) return st;
  if (rounding != MX_ROUND_RNE) return MX_ERR_UNSUPPORTED;  // no grouped Quest-like scale
  if (!valid_layout(layout)) return MX_ERR_UNSUPPORTED;
  if (E < 1 || E > 1024) return MX_ERR_SHAPE;
  int64_t srows = 0, scols = 0;
  st = mx_grouped_scales_shape(M_total, E, K, group, layout, &srows, &scols);
  if (st != MX_OK) return st;
  if (empty) return MX_OK;
  if (!row_offsets || !x || !codes || !scales) return MX_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(row_offsets) & 7u) return MX_ERR_ALIGN;
  if (!aligned32(x) || !aligned32(codes)) return MX_ERR_ALIGN;
  if (layout == MX_SCALES_SWIZZLED && !aligned16(scales)) return MX_ERR_ALIGN;
  mxq::StreamArgs a = stream_args(x, M_total, K, codes);
  a.scales = static_cast<uint8_t*>(scales);
  a.scale_cols = scols;
  a.scale_rows = srows;
  // Linear scales of a grouped call are [M_total, K/32] and the codes stay contiguous: exactly
  // the plain quantize of the whole x, which needs no expert offsets.
  const bool grouped = layout == MX_SCALES_SWIZZLED;
  if (grouped) {
    a.offsets = row_offsets;
    a.E = E;
  }
  return from_cuda(mxq::launch_stream(fmt, false, layout == MX_SCALES_SWIZZLED, grouped, a,
                                      static_cast<cudaStream_t>(stream)));
}

mx_status mx_nvfp4_scales_shape(int64_t M, int64_t K, int layout, int64_t* rows, int64_t* cols) {
  if (!rows || !cols) return MX_ERR_NULL;
  if (M < 0 || K < 0 || K % 32 != 0) return MX_ERR_SHAPE;
  if (!valid_layout(layout)) return MX_ERR_UNSUPPORTED;
  if (layout == MX_SCALES_LINEAR) {
    *rows = M;
    *cols = K / 16;
  } else {
    *rows = ceil_div(M, mxq::kTileRows) * mxq::kTileRows;
    *cols = ceil_div(K, 64) * 4;
  }
  return MX_OK;
}

namespace {

// Shared by the two NVFP4 calls: validation of x, H and the global scale. Returns MX_OK to go
// on; *empty is set when there is nothing to compute.
mx_status check_nvfp4(const void* x, int64_t M, int64_t K, const void* H, int g, int rot_kind,
                      const float* global_scale, bool* empty) {
  mx_status st = check_common(M, K, MX_FMT_E2M1, 32, MX_ROUND_RNE, empty);
  if (st != MX_OK) return st;
  if (H) {
    if (!valid_g(g) || !valid_rot_kind(rot_kind)) return MX_ERR_UNSUPPORTED;
    if (K % g != 0 || !fits_tensor_map(M, K)) return MX_ERR_SHAPE;
  }
  if (*empty) return MX_OK;
  if (!x || !global_scale) return MX_ERR_NULL;
  if (!aligned32(x) || (reinterpret_cast<uintptr_t>(global_scale) & 3u)) return MX_ERR_ALIGN;
  if (H && !aligned16(H)) return MX_ERR_ALIGN;
  return MX_OK;
}

}  // namespace

mx_status mx_quantize_nvfp4(const void* x, int64_t M, int64_t K, const void* H, int g,
                            int rot_kind, const float* global_scale, int layout, void* codes,
                            void* scales, void* stream) {
  if (!valid_layout(layout)) return MX_ERR_UNSUPPORTED;
  bool empty = false;
  mx_status st = check_nvfp4(x, M, K, H, g, rot_kind, global_scale, &empty);
  if (st != MX_OK || empty) return st;
  if (!codes || !scales) return MX_ERR_NULL;
  if (!aligned32(codes)) return MX_ERR_ALIGN;
  if (layout == MX_SCALES_SWIZZLED ? !aligned16(scales)
                                   : (reinterpret_cast<uintptr_t>(scales) & 1u) != 0) {
    return MX_ERR_ALIGN;
  }
  int64_t srows = 0, scols = 0;
  mx_nvfp4_scales_shape(M, K, layout, &srows, &scols);
  const bool swz = layout == MX_SCALES_SWIZZLED;
  if (H && use_fwht(rot_kind, g, false, M, K)) {
    mxq::StreamArgs a = stream_args(x, M, K, codes);
    a.scales = static_cast<uint8_t*>(scales);
    a.scale_cols = scols;
    a.scale_rows = srows;
    a.gscale = global_scale;
    a.H = H;
    return from_cuda(mxq::launch_hadamard(mxq::kFmtNVFP4, mxq::kRotCodes, swz, g, a,
                                          static_cast<cudaStream_t>(stream)));
  }
  if (H) {
    mxq::RotArgs a = rot_args(x, M, K, H, codes);
    a.scales = static_cast<uint8_t*>(scales);
    a.scale_cols = scols;
    a.gscale = global_scale;
    return from_cuda(mxq::launch_rotate(mxq::kFmtNVFP4, mxq::kRotCodes, swz, g, a,
                                        static_cast<cudaStream_t>(stream)));
  }
  mxq::StreamArgs a = stream_args(x, M, K, codes);
  a.scales = static_cast<uint8_t*>(scales);
  a.scale_cols = scols;
  a.scale_rows = srows;
  a.gscale = global_scale;
  return from_cuda(mxq::launch_stream(mxq::kFmtNVFP4, false, swz, false, a,
                                      static_cast<cudaStream_t>(stream)));
}

mx_status mx_qdq_nvfp4(const void* x, int64_t M, int64_t K, const void* H, int g, int rot_kind,
                       const float* global_scale, void* y, void* stream) {
  bool empty = false;
  mx_status st = check_nvfp4(x, M, K, H, g, rot_kind, global_scale, &empty);
  if (st != MX_OK || empty) return st;
  if (!y) return MX_ERR_NULL;
  if (!aligned32(y)) return MX_ERR_ALIGN;
  if (H && use_fwht(rot_kind, g, true, M, K)) {
    mxq::StreamArgs a = stream_args(x, M, K, y);
    a.gscale = global_scale;
    a.H = H;
    return from_cuda(mxq::launch_hadamard(mxq::kFmtNVFP4, mxq::kRotQdq, false, g, a,
                                          static_cast<cudaStream_t>(stream)));
  }
  if (H) {
    mxq::RotArgs a = rot_args(x, M, K, H, y);
    a.gscale = global_scale;
    return from_cuda(mxq::launch_rotate(mxq::kFmtNVFP4, mxq::kRotQdq, false, g, a,
                                        static_cast<cudaStream_t>(stream)));
  }
  mxq::StreamArgs a = stream_args(x, M, K, y);
  a.gscale = global_scale;
  return from_cuda(mxq::launch_stream(mxq::kFmtNVFP4, true, false, false, a,
                                      static_cast<cudaStream_t>(stream)));
}

mx_status mx_nvfp4_grouped_scales_shape(int64_t M_total, int E, int64_t K, int layout,
                                        int64_t* rows, int64_t* cols) {
  if (!rows || !cols) return MX_ERR_NULL;
  if (M_total < 0 || K < 0 || K % 32 != 0 || E < 1 || E > 1024) return MX_ERR_SHAPE;
  if (!valid_layout(layout)) return MX_ERR_UNSUPPORTED;
  if (layout == MX_SCALES_LINEAR) {
    *rows = M_total;
    *cols = K / 16;
  } else {
    *rows = (M_total + int64_t(mxq::kTileRows - 1) * E) / mxq::kTileRows * mxq::kTileRows;
    *cols = ceil_div(K, 64) * 4;
  }
  return MX_OK;
}

mx_status mx_quantize_nvfp4_grouped(const void* x, const int64_t* row_offsets, int E,
                                    int64_t M_total, int64_t K, const float* global_scales,
                                    int layout, void* codes, void* scales, void* stream) {
  bool empty = false;
  mx_status st = check_common(M_total, K, MX_FMT_E2M1, 32, MX_ROUND_RNE, &empty);
  if (st != MX_OK) return st;
  int64_t srows = 0, scols = 0;
  st = mx_nvfp4_grouped_scales_shape(M_total, E, K, layout, &srows, &scols);
  if (st != MX_OK) return st;
  if (empty) return MX_OK;
  if (!x || !row_offsets || !global_scales || !codes || !scales) return MX_ERR_NULL;
  if (reinterpret_cast<uintptr_t>(row_offsets) & 7u) return MX_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(global_scales) & 3u) return MX_ERR_ALIGN;
  if (!aligned32(x) || !aligned32(codes)) return MX_ERR_ALIGN;
  if (layout == MX_SCALES_SWIZZLED ? !aligned16(scales)
                                   : (reinterpret_cast<uintptr_t>(scales) & 1u) != 0) {
    return MX_ERR_ALIGN;
  }
  mxq::StreamArgs a = stream_args(x, M_total, K, codes);
  a.scales = static_cast<uint8_t*>(scales);
  a.scale_cols = scols;
  a.scale_rows = srows;
  a.offsets = row_offsets;
  a.E = E;
  a.gscale = global_scales;
  return from_cuda(mxq::launch_stream(mxq::kFmtNVFP4, false, layout == MX_SCALES_SWIZZLED, true,
                                      a, static_cast<cudaStream_t>(stream)));
}

mx_status mx_dequantize_nvfp4(const void* codes, const void* scales, int64_t M, int64_t K,
                              const float* global_scale, int layout, void* y, void* stream) {
  if (!valid_layout(layout)) return MX_ERR_UNSUPPORTED;
  bool empty = false;
  mx_status st = check_common(M, K, MX_FMT_E2M1, 32, MX_ROUND_RNE, &empty);
  if (st != MX_OK || empty) return st;
  if (!codes || !scales || !global_scale || !y) return MX_ERR_NULL;
  if (!aligned32(codes) || !aligned32(y)) return MX_ERR_ALIGN;
  if (reinterpret_cast<uintptr_t>(global_scale) & 3u) return MX_ERR_ALIGN;
  if (layout == MX_SCALES_SWIZZLED ? !aligned16(scales)
                                   : (reinterpret_cast<uintptr_t>(scales) & 1u) != 0) {
    return MX_ERR_ALIGN;
  }
  int64_t srows = 0, scols = 0;
  mx_nvfp4_scales_shape(M, K, layout, &srows, &scols);
  mxq::DequantArgs a{};
  a.codes = codes;
  a.scales = static_cast<const uint8_t*>(scales);
  a.y = y;
  a.M = M;
  a.K = K;
  a.scale_cols = scols;
  a.gscale = global_scale;
  return from_cuda(mxq::launch_dequant(mxq::kFmtNVFP4, layout == MX_SCALES_SWIZZLED, a,
                                       static_cast<cudaStream_t>(stream)));
}

mx_status mx_rotate_debug(const void* x, int64_t M, int64_t K, const void* H, int g, int rot_kind,
                          float* y_f32, void* stream) {
  bool empty = false;
  mx_status st = check_common(M, K, MX_FMT_E2M1, 32, MX_ROUND_RNE, &empty);
  if (st != MX_OK) return st;
  if (!valid_g(g) || !valid_rot_kind(rot_kind)) return MX_ERR_UNSUPPORTED;
  if (K % g != 0 || !fits_tensor_map(M, K)) return MX_ERR_SHAPE;
  if (empty) return MX_OK;
  if (!x || !H || !y_f32) return MX_ERR_NULL;
  if (!aligned32(x) || !aligned32(y_f32)) return MX_ERR_ALIGN;
  if (!aligned16(H)) return MX_ERR_ALIGN;
  if (use_fwht(rot_kind == MX_ROT_AUTO ? MX_ROT_HADAMARD : rot_kind, g, false, M, K)) {
    mxq::StreamArgs a = stream_args(x, M, K, y_f32);
    a.H = H;
    return from_cuda(mxq::launch_hadamard(MX_FMT_E2M1, mxq::kRotDebug, false, g, a,
                                          static_cast<cudaStream_t>(stream)));
  }
  return from_cuda(mxq::launch_rotate(MX_FMT_E2M1, mxq::kRotDebug, false, g,
                                      rot_args(x, M, K, H, y_f32),
                                      static_cast<cudaStream_t>(stream)));
}

namespace {
mx_status gemm_call(const void* a_codes, const void* a_scales, const void* b_codes,
                    const void* b_scales, int64_t M, int64_t N, int64_t K, int fmt, int group,
                    int layout, float alpha, void* c, unsigned long long wait_limit_ns,
                    void* stream) {
  if (M < 0 || N < 0 || K < 0) return MX_ERR_SHAPE;
  if (group != 32 || !valid_fmt(fmt) || !valid_layout(layout)) return MX_ERR_UNSUPPORTED;
  if (K == 0 || K % 64 != 0 || N % 8 != 0) return MX_ERR_SHAPE;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return MX_ERR_SHAPE;
  if (M > (int64_t(1) << 40) / K || N > (int64_t(1) << 40) / K) return MX_ERR_SHAPE;
  if (ceil_div(M, 128) > 65535) return MX_ERR_SHAPE;  // 128-row tiles on the grid's y axis
  if (M == 0 || N == 0) return MX_OK;
  if (!a_codes || !a_scales || !b_codes || !b_scales || !c) return MX_ERR_NULL;
  if (!aligned16(a_codes) || !aligned16(b_codes) || !aligned16(c)) return MX_ERR_ALIGN;
  if (layout == MX_SCALES_SWIZZLED && (!aligned16(a_scales) || !aligned16(b_scales))) {
    return MX_ERR_ALIGN;
  }
  if (((uintptr_t)a_scales | (uintptr_t)b_scales) & 1) return MX_ERR_ALIGN;  // 2-byte reads
  mxq::GemmArgs a{};
  a.a_codes = a_codes;
  a.a_scales = static_cast<const uint8_t*>(a_scales);
  a.b_codes = b_codes;
  a.b_scales = static_cast<const uint8_t*>(b_scales);
  a.c = c;
  a.M = M;
  a.N = N;
  a.K = K;
  a.a_scale_cols = a.b_scale_cols = layout == MX_SCALES_LINEAR ? K / 32 : ceil_div(K, mxq::kTileCols) * 4;
  a.alpha = alpha;
  a.wait_limit_ns = wait_limit_ns;
  cudaError_t err = mxq::device_error_word(&a.err);
  if (err != cudaSuccess) return from_cuda(err);
  return from_cuda(mxq::launch_gemm(fmt, layout == MX_SCALES_SWIZZLED, a,
                                    static_cast<cudaStream_t>(stream)));
}
}  // namespace

mx_status mx_gemm(const void* a_codes, const void* a_scales, const void* b_codes,
                  const void* b_scales, int64_t M, int64_t N, int64_t K, int fmt, int group,
                  int layout, float alpha, void* c, void* stream) {
  return gemm_call(a_codes, a_scales, b_codes, b_scales, M, N, K, fmt, group, layout, alpha, c,
                   2000000000ull, stream);
}

mx_status mx_selftest_gemm_give_up(const void* a_codes, const void* a_scales, const void* b_codes,
                                   const void* b_scales, int64_t M, int64_t N, int64_t K, int fmt,
                                   int layout, void* c, int64_t limit_ns, void* stream) {
  if (limit_ns <= 0 || limit_ns > 100000000) return MX_ERR_SHAPE;
  if (M == 0 || N == 0) return MX_ERR_SHAPE;  // a launch is the point
  return gemm_call(a_codes, a_scales, b_codes, b_scales, M, N, K, fmt, 32, layout, 1.0f, c,
                   (unsigned long long)limit_ns, stream);
}

mx_status mx_selftest_bounded_wait(int64_t limit_ns, void* stream) {
  if (limit_ns <= 0 || limit_ns > 100000000) return MX_ERR_SHAPE;
  return from_cuda(mxq::launch_wait_selftest((unsigned long long)limit_ns,
                                             static_cast<cudaStream_t>(stream)));
}

mx_status mx_selftest_rotate_give_up(const void* x, int64_t M, int64_t K, const void* H, int g,
                                     void* codes, void* scales, int64_t limit_ns, void* stream) {
  if (limit_ns <= 0 || limit_ns > 100000000) return MX_ERR_SHAPE;
  bool empty = false;
  mx_status st = check_common(M, K, MX_FMT_E2M1, 32, MX_ROUND_RNE, &empty);
  if (st != MX_OK) return st;
  if (!valid_g(g)) return MX_ERR_UNSUPPORTED;
  // the tensor-core kernel takes every call but the few-row ones (M <= 16 and M * g <= 512)
  if (K % g != 0 || !fits_tensor_map(M, K) || empty || (M <= 16 && M * g <= 512)) {
    return MX_ERR_SHAPE;
  }
  if (!x || !H || !codes || !scales) return MX_ERR_NULL;
  if (!aligned32(x) || !aligned32(codes) || !aligned16(scales) || !aligned16(H)) {
    return MX_ERR_ALIGN;
  }
  mxq::RotArgs a = rot_args(x, M, K, H, codes);
  a.scales = static_cast<uint8_t*>(scales);
  a.scale_cols = a.col_tiles * 4;
  a.wait_limit_ns = (unsigned long long)limit_ns;
  return from_cuda(mxq::launch_rotate(MX_FMT_E2M1, mxq::kRotCodes, true, g, a,
                                      static_cast<cudaStream_t>(stream)));
}

mx_status mx_device_errors(int* flags) {
  if (!flags) return MX_ERR_NULL;
  unsigned int v = 0;
  cudaError_t err = mxq::read_device_errors(&v);
  *flags = (int)v;
  return from_cuda(err);
}

}  // extern "C"
