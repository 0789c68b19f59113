// mx_stream.cu -- block quantize / QDQ without rotation (HBM-bound streaming kernels).
//
// One persistent grid walks tiles of 128 rows x 128 elements. Each of the 256 threads of a CTA
// owns two whole 32-element blocks of a tile (rows r and r + 64, block column tid % 4): it reads
// each block with two 32-byte loads (a warp instruction covers 8 rows x 256 contiguous bytes and
// fills every sector it touches), takes the abs-max with packed bf16x2 abs-max instructions,
// derives the E8M0 byte from the exponent field once per block, converts in registers with the
// hardware paired converters and writes the block's codes (16 or 32 bytes) or its dequantized
// bf16 (two 32-byte stores). A tile's 4 x 128 block scales are exactly one 512-byte tile of the
// swizzled layout: they are gathered in shared memory and written as 32 x 16-byte stores.
// Grouped (MoE) calls map each 128-row block to its expert with a per-CTA prefix over the
// expert row counts.
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "mx_device.cuh"
#include "mx_launch.h"

namespace mxq {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxExperts = 1024;

__device__ __forceinline__ void load32B(const void* p, uint32_t* r) {
  asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "l"(p));
}

__device__ __forceinline__ void store32B(void* p, const uint32_t* r) {
  asm volatile("st.global.cs.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// abs-max of one block (16 bf16x2 words) as sign-free bf16 bits; NaN propagates.
__device__ __forceinline__ uint32_t absmax_block(const uint32_t* w) {
  uint32_t m[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[i]) : "r"(w[2 * i]), "r"(w[2 * i + 1]));
  }
#pragma unroll
  for (int h = 4; h >= 1; h >>= 1) {
#pragma unroll
    for (int i = 0; i < h; ++i) {
      asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[i]) : "r"(m[i]), "r"(m[i + h]));
    }
  }
  return max(m[0] & 0x7FFFu, (m[0] >> 16) & 0x7FFFu);
}

// Quantize (or QDQ) one block held in w[16]; writes codes / bf16 through `out` when `ok`.
// Returns the scale byte.
template <int FMT, bool QDQ>
__device__ __forceinline__ uint32_t block_kernel(const uint32_t* w, bool ok, void* out) {
  const uint32_t byte = scale_byte_from_amax_bits<FMT>(absmax_block(w) << 16);
  const float inv = inv_scale_of(byte);
  const bool special = __any_sync(0xFFFFFFFFu, byte == 255u);  // a NaN / Inf block in the warp
  if (QDQ) {
    const float sc = scale_of(byte);
    uint32_t o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float lo = bf16_lo(w[i]), hi = bf16_hi(w[i]);
      mul2(lo, hi, inv);
      o[i] = qdq2<FMT>(lo, hi, sc);
    }
    if (special && byte == 255u) {
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i] = kBf16NaNx2;
    }
    if (ok) {
      store32B(out, o);
      store32B(static_cast<uint8_t*>(out) + 32, o + 8);
    }
  } else {
    uint32_t c[8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float t[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        t[2 * i] = bf16_lo(w[4 * q + i]);
        t[2 * i + 1] = bf16_hi(w[4 * q + i]);
        mul2(t[2 * i], t[2 * i + 1], inv);
      }
      if (FMT == kFmtE2M1) {
        c[q] = codes8_e2m1(t);
      } else {
        const uint2 p = codes8_e4m3(t);
        c[2 * q] = p.x;
        c[2 * q + 1] = p.y;
      }
    }
    if (special && byte == 255u) {
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] = FMT == kFmtE2M1 ? 0u : kE4M3NaNx4;
    }
    if (ok) {
      if (FMT == kFmtE2M1) {
        __stcs(static_cast<uint4*>(out), make_uint4(c[0], c[1], c[2], c[3]));
      } else {
        store32B(out, c);
      }
    }
  }
  return byte;
}

template <int FMT, bool QDQ, bool SWZ, bool GROUPED>
__global__ void __launch_bounds__(kThreads) mx_stream_kernel(StreamArgs a) {
  __shared__ __align__(16) uint8_t s_scale[2][512];
  __shared__ int64_t s_off[GROUPED ? kMaxExperts + 1 : 1];     // clamped row offsets
  __shared__ int64_t s_prefix[GROUPED ? kMaxExperts + 1 : 1];  // 128-row blocks before expert e
  __shared__ int64_t s_warp[kThreads / 32];

  const int tid = threadIdx.x;
  const int bc = tid & 3;   // block column of the tile owned by this thread
  const int br = tid >> 2;  // tile rows br and br + 64
  const uint16_t* x = static_cast<const uint16_t*>(a.x);
  constexpr int kCodeBytes = QDQ ? 64 : (FMT == kFmtE2M1 ? 16 : 32);  // output bytes per block

  if (GROUPED) {
    // expert e owns ceil(n_e / 128) padded row blocks; s_prefix[e] = blocks of experts < e.
    int64_t nb[4];
    int64_t local = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = tid * 4 + j;
      nb[j] = 0;
      if (e < a.E) {
        int64_t lo = a.offsets[e], hi = a.offsets[e + 1];
        lo = lo < 0 ? 0 : (lo > a.M ? a.M : lo);
        hi = hi < lo ? lo : (hi > a.M ? a.M : hi);
        s_off[e] = lo;
        nb[j] = (hi - lo + kTileRows - 1) / kTileRows;
        local += nb[j];
      }
    }
    if (tid == 0) {
      const int64_t end = a.offsets[a.E];
      s_off[a.E] = end < 0 ? 0 : (end > a.M ? a.M : end);
    }
    int64_t incl = local;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int64_t o = __shfl_up_sync(0xFFFFFFFFu, incl, d);
      if ((tid & 31) >= d) incl += o;
    }
    if ((tid & 31) == 31) s_warp[tid >> 5] = incl;
    __syncthreads();
    int64_t before = 0;
    for (int w = 0; w < (tid >> 5); ++w) before += s_warp[w];
    int64_t run = before + incl - local;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = tid * 4 + j;
      if (e < a.E) s_prefix[e] = run;
      run += nb[j];
    }
    if (tid == kThreads - 1) s_prefix[a.E] = run;
    __syncthreads();
  }

  const int64_t n_tiles = a.row_blocks * a.col_tiles;
  int buf = 0;
  for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, buf ^= 1) {
    const int64_t rb = t / a.col_tiles;
    const int64_t cb = t - rb * a.col_tiles;
    int64_t row0;
    int64_t rows_valid;
    if (GROUPED) {
      if (rb >= s_prefix[a.E]) {
        row0 = 0;
        rows_valid = 0;  // padded rows past the last expert: zero scale tile only
      } else {
        // largest e with s_prefix[e] <= rb (prefixes are non-decreasing)
        int lo = 0, hi = a.E;
        while (hi - lo > 1) {
          const int mid = (lo + hi) >> 1;
          if (s_prefix[mid] <= rb) lo = mid;
          else hi = mid;
        }
        row0 = s_off[lo] + (rb - s_prefix[lo]) * kTileRows;
        const int64_t end = s_off[lo + 1] > s_off[lo] ? s_off[lo + 1] : s_off[lo];
        rows_valid = end - row0;
      }
    } else {
      row0 = rb * kTileRows;
      rows_valid = a.M - row0;
    }
    rows_valid = rows_valid > kTileRows ? kTileRows : (rows_valid < 0 ? 0 : rows_valid);
    const int64_t col = cb * kTileCols + bc * 32;
    const bool col_ok = col < a.K;

    // both blocks' loads in flight before any arithmetic
    uint32_t w[2][16];
    bool ok[2];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int r = br + 64 * j;
      ok[j] = col_ok && r < rows_valid;
      if (ok[j]) {
        const uint16_t* src = x + (row0 + r) * a.K + col;
        load32B(src, w[j]);
        load32B(src + 16, w[j] + 8);
      } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) w[j][i] = 0u;
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      const int r = br + 64 * j;
      const int64_t blk = ((row0 + r) * a.K + col) >> 5;  // block index in the flat input
      void* dst = static_cast<uint8_t*>(a.out) + blk * kCodeBytes;
      const uint32_t byte = block_kernel<FMT, QDQ>(w[j], ok[j], dst);
      if (!QDQ) {
        if (SWZ) {
          s_scale[buf][swizzle_in_tile(r, bc)] = (uint8_t)byte;  // pads: zero input -> 0
        } else if (ok[j]) {
          a.scales[(row0 + r) * a.scale_cols + cb * 4 + bc] = (uint8_t)byte;
        }
      }
    }
    if (SWZ && !QDQ) {
      __syncthreads();  // tile's scales complete; also orders reuse of s_scale[buf] two tiles on
      if (tid < 32) {
        uint4* dst = reinterpret_cast<uint4*>(a.scales + (rb * a.col_tiles + cb) * 512);
        dst[tid] = reinterpret_cast<const uint4*>(s_scale[buf])[tid];
      }
    }
  }
}

template <int FMT, bool QDQ, bool SWZ, bool GROUPED>
cudaError_t launch_t(const StreamArgs& a, cudaStream_t stream) {
  const void* k = reinterpret_cast<const void*>(&mx_stream_kernel<FMT, QDQ, SWZ, GROUPED>);
  const int64_t n_tiles = a.row_blocks * a.col_tiles;
  if (n_tiles <= 0) return cudaSuccess;
  const int resident = resident_ctas(k, kThreads, 0, 0);
  if (resident <= 0) return cudaErrorInvalidConfiguration;
  const int grid = (int)(n_tiles < resident ? n_tiles : resident);
  mx_stream_kernel<FMT, QDQ, SWZ, GROUPED><<<grid, kThreads, 0, stream>>>(a);
  return cudaGetLastError();
}

template <int FMT>
cudaError_t launch_fmt(bool qdq, bool swz, bool grouped, const StreamArgs& a, cudaStream_t st) {
  if (qdq) return launch_t<FMT, true, false, false>(a, st);
  if (grouped) {
    return swz ? launch_t<FMT, false, true, true>(a, st) : launch_t<FMT, false, false, true>(a, st);
  }
  return swz ? launch_t<FMT, false, true, false>(a, st) : launch_t<FMT, false, false, false>(a, st);
}

}  // namespace

cudaError_t launch_stream(int fmt, bool qdq, bool swizzled, bool grouped, const StreamArgs& a,
                          cudaStream_t stream) {
  if (fmt == kFmtE2M1) return launch_fmt<kFmtE2M1>(qdq, swizzled, grouped, a, stream);
  return launch_fmt<kFmtE4M3>(qdq, swizzled, grouped, a, stream);
}

int resident_ctas(const void* kernel, int threads, size_t dyn_smem, int max_per_sm) {
  // (device, kernel, block shape) -> SMs x CTAs per SM, computed once per process from the
  // kernel's registers and shared memory against the SM's limits.
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, int, size_t, int>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  const auto key = std::make_tuple(dev, kernel, threads, dyn_smem, max_per_sm);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int sms = 0, thr_sm = 0, regs_sm = 0, smem_sm = 0, smem_reserved = 0, blocks_sm = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&thr_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&smem_reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) !=
          cudaSuccess ||
      cudaDeviceGetAttribute(&blocks_sm, cudaDevAttrMaxBlocksPerMultiprocessor, dev) !=
          cudaSuccess) {
    return 0;
  }
  if (dyn_smem > 48 * 1024 &&
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dyn_smem) !=
          cudaSuccess) {
    return 0;
  }
  cudaFuncAttributes fa{};
  if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) return 0;
  const int warps = (threads + 31) / 32;
  const int regs_per_warp = ((fa.numRegs * 32 + 255) / 256) * 256;  // 256-register granules
  int per_sm = blocks_sm;
  per_sm = std::min(per_sm, thr_sm / (warps * 32));
  if (regs_per_warp > 0) per_sm = std::min(per_sm, regs_sm / (regs_per_warp * warps));
  const size_t smem_block = fa.sharedSizeBytes + dyn_smem + (size_t)smem_reserved;
  per_sm = std::min(per_sm, (int)((size_t)smem_sm / smem_block));
  if (max_per_sm > 0) per_sm = std::min(per_sm, max_per_sm);
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = sms * per_sm;
  return sms * per_sm;
}

}  // namespace mxq
