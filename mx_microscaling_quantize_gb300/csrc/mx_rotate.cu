// mx_rotate.cu -- fused rotate + block quantize on the 5th-generation tensor cores.
//
// The rotation multiplies every g-element chunk along K by a runtime-loaded g x g bf16 matrix
// H (QuTLASS pull request, feature list: "Rotation matrices loaded at runtime, allowing any
// transformation", sizes 16/32/64/128). For a tile of 128 rows x 128 elements that is
// 128/g independent products [128 x g] * [g x g], issued as tcgen05.mma (kind::f16, bf16
// operands, fp32 accumulation) by one thread, with both operands in shared memory and the
// 128 x 128 fp32 result in tensor memory (TMEM). The epilogue reads TMEM with tcgen05.ld so
// that thread r holds row r of the tile, i.e. four whole 32-element blocks, and quantizes
// them in registers.
//
// Shared-memory operand layout (no swizzle, K-major "core matrices" of 8 rows x 16 bytes):
//   A (x tile):  element (r, c) at (c / 8) * kALbo + r * 16 + (c % 8) * 2, so a thread that
//                loaded 16 bytes (8 elements) of row r stores them with one 16-byte store;
//                kALbo = 128 * 16 + 16 keeps those stores free of bank conflicts.
//                Descriptor: leading (K-direction) byte offset kALbo, stride (8-row) 128.
//   B (H^T):     element (n, k) = H[k][n] at (k / 8) * (g * 16) + n * 16 + (k % 8) * 2.
//                Descriptor: leading byte offset g * 16, stride 128.
// Per tile: registers -> A (st.shared), fence.proxy.async, barrier, one thread issues the
// MMAs and commits to an mbarrier, every thread prefetches the next tile into registers,
// waits on the mbarrier (bounded), reads TMEM, quantizes and stores.
#include "mx_device.cuh"
#include "mx_launch.h"

namespace mxq {

__device__ unsigned int g_device_errors;

namespace {

constexpr int kThreads = 128;
constexpr int kALbo = kTileRows * 16 + 16;       // 2064
constexpr int kASmem = (kTileCols / 8) * kALbo;  // 33024
constexpr int kTmemCols = 128;
constexpr int kMaxCtasPerSm = 512 / kTmemCols;  // TMEM columns per SM / columns per CTA
constexpr uint32_t kErrWaitTimeout = 1u;
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s

// ------------------------------------------------------------------------------------------
// PTX wrappers
// ------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void tmem_alloc(uint32_t slot_addr, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot_addr),
               "r"(ncols));
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols));
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_init(uint32_t addr, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(addr), "r"(count));
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t addr, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred P;\n\tmbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(done)
      : "r"(addr), "r"(parity)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
// Wait for the mbarrier phase with the given parity; give up after kWaitLimitNs.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t addr, uint32_t parity) {
  if (mbar_try_wait(addr, parity)) return true;
  const unsigned long long t0 = global_ns();
  while (!mbar_try_wait(addr, parity)) {
    if (global_ns() - t0 > kWaitLimitNs) return false;
  }
  return true;
}

// Shared-memory matrix descriptor, no swizzle: start, leading and stride byte offsets (all
// multiples of 16), bit 46 set (descriptor version of the 5th-generation tensor core).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
         ((uint64_t)(sbo >> 4) << 32) | (1ull << 46);
}

// Instruction descriptor, kind::f16: fp32 accumulator (bits 4-5 = 1), A and B bf16 (bits 7-9
// and 10-12 = 1), both K-major, N >> 3 at bits 17-22, M >> 4 at bits 24-28.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                         uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void mma_commit(uint32_t mbar_addr) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          mbar_addr)
      : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float* y) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, "
      "%28, %29, %30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) y[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, const uint4& v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y),
               "r"(v.z), "r"(v.w)
               : "memory");
}

// ------------------------------------------------------------------------------------------
// kernel
// ------------------------------------------------------------------------------------------
template <int G>
constexpr int smem_bytes() {
  return kASmem + G * G * 2 + 16 + 2 * 512;
}
// Dynamic shared memory requested per CTA: at least 56 KiB so that no more than four CTAs
// share an SM (four x 128 TMEM columns = the SM's 512), whatever g is.
template <int G>
constexpr int smem_request() {
  return smem_bytes<G>() > 56 * 1024 ? smem_bytes<G>() : 56 * 1024;
}

template <int FMT, int OUT, bool SWZ, int G>
__global__ void __launch_bounds__(kThreads) mx_rotate_kernel(RotArgs a) {
  extern __shared__ __align__(1024) uint8_t smem[];
  uint8_t* sA = smem;
  uint8_t* sB = smem + kASmem;
  uint64_t* mbar = reinterpret_cast<uint64_t*>(sB + G * G * 2);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mbar + 1);
  uint8_t* s_scale = reinterpret_cast<uint8_t*>(mbar + 2);  // [2][512]

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const uint4* x = static_cast<const uint4*>(a.x);
  const uint16_t* H = static_cast<const uint16_t*>(a.H);

  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (tid == 0) mbar_init(smem_u32(mbar), 1);
  // B = H^T in K-major core-matrix layout (coalesced reads of H's rows).
  for (int idx = tid; idx < G * G; idx += kThreads) {
    const int k = idx / G, n = idx % G;
    *reinterpret_cast<uint16_t*>(sB + (k / 8) * (G * 16) + n * 16 + (k % 8) * 2) = H[idx];
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sA_u32 = smem_u32(sA);
  const uint32_t sB_u32 = smem_u32(sB);
  const uint32_t mbar_u32 = smem_u32(mbar);
  constexpr uint32_t idesc = idesc_bf16_f32(kTileRows, G);

  const int lvec = tid & 15;  // loader: 16-byte vector of the row
  const int lrow = tid >> 4;  // loader: rows lrow + 8 i
  const int64_t n_tiles = a.row_blocks * a.col_tiles;

  uint4 v[16];
  auto load_tile = [&](int64_t t) {
    const int64_t rb = t / a.col_tiles;
    const int64_t cb = t - rb * a.col_tiles;
    const int64_t row0 = rb * kTileRows;
    const int64_t col = cb * kTileCols + lvec * 8;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int64_t row = row0 + i * 8 + lrow;
      v[i] = make_uint4(0u, 0u, 0u, 0u);
      if (row < a.M && col < a.K) v[i] = __ldcs(x + ((row * a.K + col) >> 3));
    }
  };

  int64_t t = blockIdx.x;
  if (t < n_tiles) load_tile(t);
  uint32_t phase = 0;
  int buf = 0;
  int64_t prev_tile = -1;
  for (; t < n_tiles; t += gridDim.x) {
    const int64_t rb = t / a.col_tiles;
    const int64_t cb = t - rb * a.col_tiles;
    const int64_t row0 = rb * kTileRows;
    const int64_t kc64 = a.K - cb * kTileCols;
    const int kc = kc64 > kTileCols ? kTileCols : (int)kc64;  // valid columns (multiple of 32, g)
    const bool row_ok = row0 + tid < a.M;

#pragma unroll
    for (int i = 0; i < 16; ++i) st_shared_v4(sA_u32 + lvec * kALbo + (i * 8 + lrow) * 16, v[i]);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (SWZ && OUT == kRotCodes && prev_tile >= 0 && tid < 32) {
      uint4* dst = reinterpret_cast<uint4*>(a.scales + prev_tile * 512);
      dst[tid] = reinterpret_cast<const uint4*>(s_scale + (buf ^ 1) * 512)[tid];
    }
    if (tid == 0) {
      for (int j = 0; j < kc / G; ++j) {
#pragma unroll
        for (int s = 0; s < G / 16; ++s) {
          const uint64_t ad = smem_desc(sA_u32 + (j * (G / 8) + 2 * s) * kALbo, kALbo, 128);
          const uint64_t bd = smem_desc(sB_u32 + (2 * s) * (G * 16), G * 16, 128);
          mma_bf16(tmem + (uint32_t)(j * G), ad, bd, idesc, s > 0 ? 1u : 0u);
        }
      }
      mma_commit(mbar_u32);
    }
    __syncwarp();
    if (t + gridDim.x < n_tiles) load_tile(t + gridDim.x);
    const bool timed_out = !mbar_wait_bounded(mbar_u32, phase);
    // the give-up decision is taken by the whole CTA so that no thread skips a barrier
    if (__syncthreads_or(timed_out)) {
      if (tid == 0) atomicOr(&g_device_errors, kErrWaitTimeout);
      break;
    }
    phase ^= 1u;
    tc_fence_after();

    const uint32_t lane_base = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll 1
    for (int q = 0; q < 4; ++q) {
      if (q * 32 >= kc) {
        if (SWZ && OUT == kRotCodes) s_scale[buf * 512 + swizzle_in_tile(tid, q)] = 0;
        continue;
      }
      float y[32];
      tmem_ld32(lane_base + (uint32_t)(q * 32), y);
      const int64_t e0 = (row0 + tid) * a.K + cb * kTileCols + q * 32;  // first element
      if (OUT == kRotDebug) {
        if (row_ok) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + e0);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            dst[i] = make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
          }
        }
        continue;
      }
      const uint32_t byte = scale_byte_from_amax_bits<FMT>(absmax_f32x32(y));
      const bool special = __any_sync(0xFFFFFFFFu, byte == 255u);  // a NaN / Inf block
      {
        const float inv = inv_scale_of(byte);
#pragma unroll
        for (int i = 0; i < 16; ++i) mul2(y[2 * i], y[2 * i + 1], inv);  // y <- y / 2^s
      }
      if (OUT == kRotQdq) {
        const float sc = scale_of(byte);
        uint4 o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float* t = y + 8 * i;
          o[i] = make_uint4(qdq2<FMT>(t[0], t[1], sc), qdq2<FMT>(t[2], t[3], sc),
                            qdq2<FMT>(t[4], t[5], sc), qdq2<FMT>(t[6], t[7], sc));
          if (special && byte == 255u) {
            o[i] = make_uint4(kBf16NaNx2, kBf16NaNx2, kBf16NaNx2, kBf16NaNx2);
          }
        }
        if (row_ok) {
          uint4* dst = static_cast<uint4*>(a.out) + (e0 >> 3);
#pragma unroll
          for (int i = 0; i < 4; ++i) __stcs(dst + i, o[i]);
        }
      } else {
        if (FMT == kFmtE2M1) {
          uint4 c = make_uint4(codes8_e2m1(y), codes8_e2m1(y + 8), codes8_e2m1(y + 16),
                               codes8_e2m1(y + 24));
          if (special && byte == 255u) c = make_uint4(0u, 0u, 0u, 0u);
          if (row_ok) {
            __stcs(reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) + (e0 >> 1)), c);
          }
        } else {
          uint2 c[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            c[i] = codes8_e4m3(y + 8 * i);
            if (special && byte == 255u) c[i] = make_uint2(kE4M3NaNx4, kE4M3NaNx4);
          }
          if (row_ok) {
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(a.out) + e0);
            __stcs(dst, make_uint4(c[0].x, c[0].y, c[1].x, c[1].y));
            __stcs(dst + 1, make_uint4(c[2].x, c[2].y, c[3].x, c[3].y));
          }
        }
        if (SWZ) {
          s_scale[buf * 512 + swizzle_in_tile(tid, q)] = (uint8_t)byte;  // pad rows: 0
        } else if (row_ok) {
          a.scales[(row0 + tid) * a.scale_cols + cb * 4 + q] = (uint8_t)byte;
        }
      }
    }
    tc_fence_before();
    prev_tile = t;
    buf ^= 1;
  }
  __syncthreads();
  if (SWZ && OUT == kRotCodes && prev_tile >= 0 && tid < 32) {
    uint4* dst = reinterpret_cast<uint4*>(a.scales + prev_tile * 512);
    dst[tid] = reinterpret_cast<const uint4*>(s_scale + (buf ^ 1) * 512)[tid];
  }
  tc_fence_after();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

template <int FMT, int OUT, bool SWZ, int G>
cudaError_t launch_t(const RotArgs& a, cudaStream_t stream) {
  auto kern = mx_rotate_kernel<FMT, OUT, SWZ, G>;
  const void* k = reinterpret_cast<const void*>(kern);
  constexpr int smem = smem_request<G>();
  const int64_t n_tiles = a.row_blocks * a.col_tiles;
  if (n_tiles <= 0) return cudaSuccess;
  const int resident = resident_ctas(k, kThreads, smem, kMaxCtasPerSm);
  if (resident <= 0) return cudaErrorInvalidConfiguration;
  const int grid = (int)(n_tiles < resident ? n_tiles : resident);
  kern<<<grid, kThreads, smem, stream>>>(a);
  return cudaGetLastError();
}

template <int FMT, int OUT, bool SWZ>
cudaError_t launch_g(int g, const RotArgs& a, cudaStream_t st) {
  switch (g) {
    case 16: return launch_t<FMT, OUT, SWZ, 16>(a, st);
    case 32: return launch_t<FMT, OUT, SWZ, 32>(a, st);
    case 64: return launch_t<FMT, OUT, SWZ, 64>(a, st);
    default: return launch_t<FMT, OUT, SWZ, 128>(a, st);
  }
}

template <int FMT>
cudaError_t launch_fmt(int out_kind, bool swz, int g, const RotArgs& a, cudaStream_t st) {
  if (out_kind == kRotQdq) return launch_g<FMT, kRotQdq, false>(g, a, st);
  return swz ? launch_g<FMT, kRotCodes, true>(g, a, st) : launch_g<FMT, kRotCodes, false>(g, a, st);
}

}  // namespace

cudaError_t launch_rotate(int fmt, int out_kind, bool swizzled, int g, const RotArgs& a,
                          cudaStream_t stream) {
  if (out_kind == kRotDebug) return launch_g<kFmtE2M1, kRotDebug, false>(g, a, stream);
  if (fmt == kFmtE2M1) return launch_fmt<kFmtE2M1>(out_kind, swizzled, g, a, stream);
  return launch_fmt<kFmtE4M3>(out_kind, swizzled, g, a, stream);
}

cudaError_t read_device_errors(unsigned int* flags) {
  cudaError_t err = cudaDeviceSynchronize();
  if (err != cudaSuccess) return err;
  err = cudaMemcpyFromSymbol(flags, g_device_errors, sizeof(unsigned int));
  if (err != cudaSuccess) return err;
  const unsigned int zero = 0;
  return cudaMemcpyToSymbol(g_device_errors, &zero, sizeof(unsigned int));
}

}  // namespace mxq
