// mx_stream.cu -- block quantize / QDQ without rotation (HBM-bound streaming kernels).
//
// One persistent grid walks tiles of 128 rows x 128 elements. A CTA of 256 threads reads a
// tile as 2048 coalesced 16-byte vectors (a warp instruction covers 2 rows x 256 bytes, all
// eight loads of a thread are in flight together), finds each 32-element block's abs-max with
// packed bf16x2 abs-max instructions plus two shuffles across the block's 4 lanes,
// derives the E8M0 byte from the exponent field, converts in registers with the hardware
// paired converters and writes codes (or the dequantized bf16) with one coalesced store per
// vector. Swizzled scales of a tile are exactly one 512-byte tile of the 128x4 layout: they are
// gathered in shared memory and written as 32 x 16-byte stores. Grouped (MoE) calls map each
// 128-row block to its expert with a per-CTA prefix over the expert row counts.
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "mx_device.cuh"
#include "mx_launch.h"

namespace mxq {
namespace {

constexpr int kThreads = 256;
constexpr int kVecs = kTileRows * (kTileCols / 8) / kThreads;  // 16-byte vectors per thread: 8
constexpr int kMaxExperts = 1024;

__device__ __forceinline__ uint4 load_stream(const uint4* p) { return __ldcs(p); }

template <int FMT, bool QDQ, bool SWZ, bool GROUPED>
__global__ void __launch_bounds__(kThreads) mx_stream_kernel(StreamArgs a) {
  __shared__ __align__(16) uint8_t s_scale[2][512];
  __shared__ int64_t s_off[GROUPED ? kMaxExperts + 1 : 1];     // clamped row offsets
  __shared__ int64_t s_prefix[GROUPED ? kMaxExperts + 1 : 1];  // 128-row blocks before expert e
  __shared__ int64_t s_warp[kThreads / 32];

  const int tid = threadIdx.x;
  const int vec = tid & 15;  // 16-byte vector of the tile row
  const int rsub = tid >> 4;
  const int blk = vec >> 2;  // 32-element block of the tile row
  const uint4* x = static_cast<const uint4*>(a.x);

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
    const int64_t col = cb * kTileCols + vec * 8;
    const bool col_ok = col < a.K;

    uint4 v[kVecs];
#pragma unroll
    for (int i = 0; i < kVecs; ++i) {
      const int r = i * 16 + rsub;
      v[i] = make_uint4(0u, 0u, 0u, 0u);
      if (col_ok && r < rows_valid) v[i] = load_stream(x + (((row0 + r) * a.K + col) >> 3));
    }

#pragma unroll
    for (int i = 0; i < kVecs; ++i) {
      const int r = i * 16 + rsub;
      uint32_t m = absmax_bf16x8(v[i]);
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 1));
      m = max(m, __shfl_xor_sync(0xFFFFFFFFu, m, 2));
      const uint32_t byte = scale_byte_from_amax_bits<FMT>(m << 16);
      const bool ok = col_ok && r < rows_valid;
      const int64_t e0 = (row0 + r) * a.K + col;  // first element of this vector
      float t[8];
      scaled8_bf16(v[i], inv_scale_of(byte), t);
      const bool special = __any_sync(0xFFFFFFFFu, byte == 255u);  // a NaN / Inf block
      if (QDQ) {
        const float sc = scale_of(byte);
        uint4 o = make_uint4(qdq2<FMT>(t[0], t[1], sc), qdq2<FMT>(t[2], t[3], sc),
                             qdq2<FMT>(t[4], t[5], sc), qdq2<FMT>(t[6], t[7], sc));
        if (special && byte == 255u) o = make_uint4(kBf16NaNx2, kBf16NaNx2, kBf16NaNx2, kBf16NaNx2);
        if (ok) __stcs(static_cast<uint4*>(a.out) + (e0 >> 3), o);
      } else {
        if (FMT == kFmtE2M1) {
          uint32_t c = codes8_e2m1(t);
          if (special && byte == 255u) c = 0u;
          if (ok) __stcs(static_cast<unsigned int*>(a.out) + (e0 >> 3), c);
        } else {
          uint2 c = codes8_e4m3(t);
          if (special && byte == 255u) c = make_uint2(kE4M3NaNx4, kE4M3NaNx4);
          if (ok) __stcs(static_cast<uint2*>(a.out) + (e0 >> 3), c);
        }
        if ((vec & 3) == 0) {
          if (SWZ) {
            s_scale[buf][swizzle_in_tile(r, blk)] = (uint8_t)byte;  // pads: zero input -> 0
          } else if (ok) {
            a.scales[(row0 + r) * a.scale_cols + cb * 4 + blk] = (uint8_t)byte;
          }
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
