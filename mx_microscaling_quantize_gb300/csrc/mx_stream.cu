// mx_stream.cu -- block quantize / QDQ without rotation (HBM-bound streaming kernels).
//
// One persistent CTA per SM walks tiles of 128 rows x 128 elements. A producer warp streams
// tiles into a ring of shared-memory stages with bulk asynchronous copies (one cp.async.bulk
// per 256-byte row segment, completion counted in bytes on the stage's mbarrier), keeping up
// to kStages tiles (up to 6 x 32 KiB) in flight per SM. Sixteen consumer warps each own one
// 32-element block per tile (thread -> row 8w + lane%8, block column lane/8, so the eight
// lanes of a shared-memory phase read eight different rows: rows are padded to 272 bytes to
// spread them over all banks). A consumer takes the block's abs-max with packed bf16x2
// abs-max instructions, derives the E8M0 byte from the exponent field once per block,
// converts in registers with the hardware paired converters and writes the block's codes
// (16 or 32 bytes) or its dequantized bf16 (two 32-byte stores), then releases the stage on
// its empty mbarrier. A tile's 4 x 128 block scales are exactly one 512-byte tile of the
// swizzled layout: they are gathered in shared memory and written as 32 x 16-byte stores.
// Grouped (MoE) calls map each 128-row block to its expert with a per-CTA prefix over the
// expert row counts. Every mbarrier wait is bounded (2 s); a wait that runs out sets the
// device error word and the CTA stops waiting from then on.
#include <algorithm>
#include <map>
#include <mutex>
#include <tuple>

#include "mx_device.cuh"
#include "mx_launch.h"

namespace mxq {

__device__ unsigned int g_stream_errors;

namespace {

constexpr int kConsumerWarps = 16;                     // one 32-element block per thread
constexpr int kConsumers = kConsumerWarps * 32;         // 512
constexpr int kThreads = kConsumers + 32;               // + one producer warp
constexpr int kRowPitch = kTileCols * 2 + 16;           // 272 bytes per staged row
constexpr int kStageBytes = kTileRows * kRowPitch;      // 34816
constexpr int kMaxExperts = 1024;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s
constexpr uint32_t kErrWaitTimeout = 1u;

template <bool GROUPED>
struct StreamConfig {
  // stages in flight per SM (the grouped variant keeps 17 KiB of expert tables as well)
  static constexpr int kStages = GROUPED ? 5 : 6;
  static constexpr int kSmem = kStages * kStageBytes + 2 * 512 + 2 * kStages * 8;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred P;\n\tmbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Wait for the phase of the given parity. Gives up after kWaitLimitNs, and at once if this
// thread already gave up once (*failed); a give-up sets the device error word.
__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity, bool* failed) {
  if (mbar_try_wait(bar, parity) || *failed) return;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) {
      *failed = true;
      atomicOr(&g_stream_errors, kErrWaitTimeout);
      return;
    }
  }
}
// global -> shared bulk copy; completion is counted in bytes on `bar`
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                              uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void consumer_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
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

// Row range of tile t: first input row and number of valid rows (0..128); column block cb.
template <bool GROUPED>
__device__ __forceinline__ void tile_rows(const StreamArgs& a, int64_t rb, const int64_t* s_off,
                                          const int64_t* s_prefix, int64_t* row0,
                                          int64_t* rows_valid) {
  int64_t r0 = rb * kTileRows, n = a.M - r0;
  if (GROUPED) {
    if (rb >= s_prefix[a.E]) {
      r0 = 0;
      n = 0;  // padded rows past the last expert: zero scale tile only
    } else {
      // largest e with s_prefix[e] <= rb (prefixes are non-decreasing)
      int lo = 0, hi = a.E;
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (s_prefix[mid] <= rb) lo = mid;
        else hi = mid;
      }
      r0 = s_off[lo] + (rb - s_prefix[lo]) * kTileRows;
      const int64_t end = s_off[lo + 1] > s_off[lo] ? s_off[lo + 1] : s_off[lo];
      n = end - r0;
    }
  }
  *row0 = r0;
  *rows_valid = n > kTileRows ? kTileRows : (n < 0 ? 0 : n);
}

template <int FMT, bool QDQ, bool SWZ, bool GROUPED>
__global__ void __launch_bounds__(kThreads, 1) mx_stream_kernel(StreamArgs a) {
  constexpr int S = StreamConfig<GROUPED>::kStages;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* s_scale = smem + S * kStageBytes;                       // [2][512]
  uint64_t* full = reinterpret_cast<uint64_t*>(s_scale + 2 * 512);  // [S]
  uint64_t* empty = full + S;                                       // [S]
  __shared__ int64_t s_off[GROUPED ? kMaxExperts + 1 : 1];     // clamped row offsets
  __shared__ int64_t s_prefix[GROUPED ? kMaxExperts + 1 : 1];  // 128-row blocks before expert e
  __shared__ int64_t s_warp[8];

  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  constexpr int kCodeBytes = QDQ ? 64 : (FMT == kFmtE2M1 ? 16 : 32);  // output bytes per block

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (GROUPED && tid < 256) {
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
      if (lane >= d) incl += o;
    }
    if (lane == 31) s_warp[warp] = incl;
    asm volatile("bar.sync 2, 256;" ::: "memory");
    int64_t before = 0;
    for (int w = 0; w < warp; ++w) before += s_warp[w];
    int64_t run = before + incl - local;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = tid * 4 + j;
      if (e < a.E) s_prefix[e] = run;
      run += nb[j];
    }
    if (tid == 255) s_prefix[a.E] = run;
  }
  __syncthreads();

  const int64_t n_tiles = a.row_blocks * a.col_tiles;
  bool failed = false;
  if (warp == kConsumerWarps) {
    // ---------------- producer warp: tile rows -> shared-memory stage ----------------
    const uint8_t* x = static_cast<const uint8_t*>(a.x);
    int it = 0;
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
      const int s = it % S;
      if (it >= S) mbar_wait(smem_u32(empty + s), ((it / S) & 1) ^ 1, &failed);
      const int64_t rb = t / a.col_tiles, cb = t - rb * a.col_tiles;
      int64_t row0, rows;
      tile_rows<GROUPED>(a, rb, s_off, s_prefix, &row0, &rows);
      const int64_t kc = a.K - cb * kTileCols < kTileCols ? a.K - cb * kTileCols : kTileCols;
      const uint32_t bytes = (uint32_t)(kc * 2);
      if (lane == 0) mbar_arrive_expect_tx(smem_u32(full + s), (uint32_t)rows * bytes);
      __syncwarp();
      const uint32_t dst = smem_u32(smem + s * kStageBytes);
      for (int r = lane; r < rows; r += 32) {
        bulk_copy_g2s(dst + r * kRowPitch, x + ((row0 + r) * a.K + cb * kTileCols) * 2, bytes,
                      smem_u32(full + s));
      }
    }
    return;
  }

  // ---------------- consumer warps: one 32-element block per thread ----------------
  const int bc = lane >> 3;               // block column of the tile
  const int r = warp * 8 + (lane & 7);    // tile row
  int it = 0;
  for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
    const int s = it % S;
    const int64_t rb = t / a.col_tiles, cb = t - rb * a.col_tiles;
    int64_t row0, rows;
    tile_rows<GROUPED>(a, rb, s_off, s_prefix, &row0, &rows);
    const int64_t col = cb * kTileCols + bc * 32;
    const bool ok = r < rows && col < a.K;
    mbar_wait(smem_u32(full + s), (it / S) & 1, &failed);
    uint32_t w[16];
    if (ok) {
      const uint4* src = reinterpret_cast<const uint4*>(smem + s * kStageBytes + r * kRowPitch +
                                                        bc * 64);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 q = src[k];
        w[4 * k] = q.x;
        w[4 * k + 1] = q.y;
        w[4 * k + 2] = q.z;
        w[4 * k + 3] = q.w;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) w[i] = 0u;  // pads: zero block -> scale byte 0
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(empty + s));  // this warp is done with the stage

    const int64_t blk = ((row0 + r) * a.K + col) >> 5;  // block index in the flat input
    void* dst = static_cast<uint8_t*>(a.out) + blk * kCodeBytes;
    const uint32_t byte = block_kernel<FMT, QDQ>(w, ok, dst);
    if (!QDQ) {
      uint8_t* tile_scales = s_scale + (it & 1) * 512;
      if (SWZ) {
        tile_scales[swizzle_in_tile(r, bc)] = (uint8_t)byte;
      } else if (ok) {
        a.scales[(row0 + r) * a.scale_cols + cb * 4 + bc] = (uint8_t)byte;
      }
      if (SWZ) {
        consumer_sync();  // tile's scales complete; also orders reuse two tiles on
        if (warp == 0) {
          uint4* d = reinterpret_cast<uint4*>(a.scales + (rb * a.col_tiles + cb) * 512);
          d[lane] = reinterpret_cast<const uint4*>(tile_scales)[lane];
        }
      }
    }
  }
}

template <int FMT, bool QDQ, bool SWZ, bool GROUPED>
cudaError_t launch_t(const StreamArgs& a, cudaStream_t stream) {
  auto kern = mx_stream_kernel<FMT, QDQ, SWZ, GROUPED>;
  const void* k = reinterpret_cast<const void*>(kern);
  constexpr int smem = StreamConfig<GROUPED>::kSmem;
  const int64_t n_tiles = a.row_blocks * a.col_tiles;
  if (n_tiles <= 0) return cudaSuccess;
  const int resident = resident_ctas(k, kThreads, smem, 1);
  if (resident <= 0) return cudaErrorInvalidConfiguration;
  const int grid = (int)(n_tiles < resident ? n_tiles : resident);
  kern<<<grid, kThreads, smem, stream>>>(a);
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

cudaError_t read_stream_errors(unsigned int* flags) {
  cudaError_t err = cudaMemcpyFromSymbol(flags, g_stream_errors, sizeof(unsigned int));
  if (err != cudaSuccess) return err;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_stream_errors, &zero, sizeof(unsigned int));
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
