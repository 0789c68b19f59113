// mx_launch.h -- host-side launch interface between the C ABI (mx_api.cu) and the kernels.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>
#include <utility>

namespace mxq {

// Launches `kernel` with programmatic stream serialization (see pdl_wait in mx_device.cuh).
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t err = cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
  if (err != cudaSuccess) (void)cudaGetLastError();  // reported here, not to a later caller
  return err;
}

// Work is cut into tiles of 128 rows x 128 elements along K; a tile's 4x128 block scales form
// exactly one 512-byte tile of the swizzled scale layout.
constexpr int kTileRows = 128;
constexpr int kTileCols = 128;

struct StreamArgs {
  const void* x;           // bf16 [M, K]
  void* out;               // codes (quantize) or bf16 [M, K] (QDQ)
  uint8_t* scales;         // quantize only
  int64_t M;               // rows of x (all experts when grouped)
  int64_t K;
  int64_t scale_cols;      // linear: K / 32; swizzled: col_tiles * 4
  int64_t scale_rows;      // rows of the scale buffer
  const int64_t* offsets;  // grouped only: device int64 [E + 1]
  int E;
  const float* gscale;     // NVFP4 only: device fp32 global scale (grouped: one per expert)
  const void* H;           // Hadamard-rotated calls only: bf16 [g, g] row-major
};

// fmt: 1 = E2M1, 2 = E4M3, 3 = NVFP4, 4 = E2M1 under the Quest-like scale (not grouped). qdq:
// write bf16 QDQ instead of codes + scales.
cudaError_t launch_stream(int fmt, bool qdq, bool swizzled, bool grouped, const StreamArgs& a,
                          cudaStream_t stream);

struct DequantArgs {
  const void* codes;      // E2M1 [M, K/2] or E4M3 [M, K] bytes
  const uint8_t* scales;  // linear [M, K/32] (NVFP4: [M, K/16]) or swizzled (scale_cols columns)
  void* y;                // bf16 [M, K]
  int64_t M;
  int64_t K;
  int64_t scale_cols;
  const float* gscale;    // NVFP4 only: device fp32 global scale
};

// fmt: 1 = E2M1, 2 = E4M3, 3 = NVFP4 (E2M1 codes, E4M3 scales per 16 elements).
cudaError_t launch_dequant(int fmt, bool swizzled, const DequantArgs& a, cudaStream_t stream);

enum RotOut { kRotCodes = 0, kRotQdq = 1, kRotDebug = 2 };

// Rotate + quantize / QDQ / debug values on the streaming layout with a fast Walsh-Hadamard
// transform (H stated to be H[0][0] * Sylvester; checked on the device, dense FMA product
// otherwise). fmt as launch_stream; out_kind a RotOut; a.H and g the rotation.
cudaError_t launch_hadamard(int fmt, int out_kind, bool swizzled, int g, const StreamArgs& a,
                            cudaStream_t stream);

struct RotArgs {
  const void* x;      // bf16 [M, K]
  const void* H;      // bf16 [g, g] row-major
  void* out;          // codes, bf16 QDQ, or fp32 rotated values
  uint8_t* scales;    // codes only
  int64_t M;
  int64_t K;
  int64_t col_tiles;
  int64_t row_blocks;
  int64_t scale_cols;
  const float* gscale;  // NVFP4 only: device fp32 global scale
  // Limit of each mbarrier wait in the tensor-core rotation kernel, ns; 0 = the default (2 s).
  // Only the give-up self-test sets it.
  unsigned long long wait_limit_ns;
};

cudaError_t launch_rotate(int fmt, int out_kind, bool swizzled, int g, const RotArgs& a,
                          cudaStream_t stream);

struct GemmArgs {
  const void* a_codes;      // A: E2M1 [M, K/2] or E4M3 [M, K] codes
  const uint8_t* a_scales;  // A's E8M0 scales, linear [M, K/32] or swizzled
  const void* b_codes;      // B: [N, K/2] or [N, K] codes
  const uint8_t* b_scales;
  void* c;                  // bf16 [M, N]
  int64_t M;
  int64_t N;
  int64_t K;
  int64_t a_scale_cols;     // columns of A's / B's scale matrix (linear: K/32; swizzled: padded)
  int64_t b_scale_cols;
  float alpha;
  unsigned int* err;        // device error word (device_error_word)
  unsigned long long wait_limit_ns;  // pipeline waits (drains always allow 2 s)
};

// Tensor map of a row-major [rows, cols] matrix of 1- or 2-byte elements, boxes of box_rows x
// box_cols, the given swizzle; loads read zeros out of bounds, stores drop what falls outside.
cudaError_t make_tensor_map_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                               CUtensorMapDataType type, int elem_bytes, int box_cols,
                               int box_rows, CUtensorMapSwizzle swizzle);

// C = alpha * dequant(A) * dequant(B)^T on the tensor cores (fmt: 1 = E2M1, 2 = E4M3).
cudaError_t launch_gemm(int fmt, bool swizzled, const GemmArgs& a, cudaStream_t stream);

// Device address of the current device's error word, for kernels outside the file that defines
// it (looked up once per device).
cudaError_t device_error_word(unsigned int** word);

// Reads and clears the device error word of the current device (synchronizes).
cudaError_t read_device_errors(unsigned int* flags);

// One wait on an mbarrier that nothing arrives at, given up after limit_ns (sets the error word).
cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream);

// Number of CTAs of `kernel` that fit on the current device at once: SMs x CTAs per SM from
// the kernel's registers and shared memory against the SM's limits, capped at max_per_sm when
// positive. Also raises the kernel's dynamic shared-memory limit when dyn_smem > 48 KiB.
// Cached per (device, kernel, threads, dyn_smem, max_per_sm).
int resident_ctas(const void* kernel, int threads, size_t dyn_smem, int max_per_sm);

}  // namespace mxq
