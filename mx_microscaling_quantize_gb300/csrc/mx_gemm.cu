// mx_gemm.cu -- block-scaled GEMM consumer of the library's MX codes and scales on the
// 5th-generation tensor cores:
//   C[M, N] = alpha * dequant(A)[M, K] * dequant(B)[N, K]^T   (bf16 out, fp32 accumulation),
// A and B given as MX codes (E2M1 packed two per byte, or E4M3) with their E8M0 block scales in
// the linear or the 128x4 blocked layout, as mx_quantize writes them. This is the consumer the
// QuTLASS pull request tests its quantizer against (review thread on the MXFP4 test:
// matmul_mxf4_bf16_tn(a_e2m1, b_e2m1, a_e8m0, b_e8m0, alpha) compared with the matmul of the
// dequantized operands).
//
// Each CTA computes one 128 x 128 tile of C, K in steps of 64:
//   warps 0..7   producers: each K step they read the tile's A and B codes (16 or 32 bytes of
//                codes per 32-element block) and their scale bytes from global memory and write
//                the dequantized values decode(code) * 2^(byte - 127), rounded once to bf16 (exact
//                for every E2M1 code and for E4M3 codes unless the product falls below the bf16
//                range), into a stage of shared memory: A and B as 128 rows x 64 bf16, K-major,
//                in the 128-byte swizzled layout (16-byte chunk c of row r at chunk c ^ (r % 8)),
//                the form a tensor-core shared-memory descriptor reads;
//   warp 8       allocates 128 tensor-memory columns and, from one lane, issues per stage four
//                tcgen05.mma kind::f16 (M = 128, N = 128, K = 16, bf16 x bf16 -> fp32 in tensor
//                memory) and commits them to the stage's "empty" barrier;
//   warps 8..11  epilogue: tcgen05.ld of the accumulator (warp w reads lanes 32 (w % 4) .. +31,
//                the tile's rows), times alpha, rounded to bf16, 16-byte stores.
// Three stages in flight; two CTAs per SM. Every mbarrier wait is bounded as in the rotation
// kernel: a wait that runs out sets the device error word and its role stops issuing work, and
// the MMA thread waits for its MMAs before the tensor memory is freed.
#include "mx_device.cuh"
#include "mx_launch.h"
#include "mx_tcgen05.cuh"

namespace mxq {

namespace {

using namespace tc;

constexpr int kBM = 128, kBN = 128, kBK = 64;
constexpr int kStages = 3;
constexpr int kOperandBytes = kBM * kBK * 2;  // 16 KiB of bf16 per operand and stage
constexpr int kGemmStageBytes = 2 * kOperandBytes;
constexpr int kProducerWarps = 8;
constexpr int kGemmThreads = (kProducerWarps + 4) * 32;
constexpr int kChunksPerThread = 2 * kBM * (kBK / 8) / (kProducerWarps * 32);  // 8
constexpr unsigned long long kGemmWaitNs = 2000000000ull;  // 2 s
constexpr int kGemmSmem = 1024 + kStages * kGemmStageBytes + (2 * kStages + 1) * 8 + 16;

// Eight codes (8 E2M1 nibbles in a 32-bit word, lower K first; or 8 E4M3 bytes in two words)
// under the E8M0 byte `sb` -> 8 bf16 (4 words), each decode(code) * 2^(sb - 127) rounded once.
// Scale byte 0xFF (E8M0 NaN) gives the bf16 NaN 0x7FC0, as the dequantize kernel does.
template <int FMT>
__device__ __forceinline__ uint4 dequant8(uint32_t w0, uint32_t w1, uint32_t sb) {
  const float sc = scale_of(sb);
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t h;  // two codes decoded exactly to f16x2 (lower K in the low half)
    if (FMT == kFmtE2M1) {
      const uint32_t byte = (w0 >> (8 * i)) & 0xFFu;
      asm("{\n\t.reg .b8 c;\n\tcvt.u8.u32 c, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, c;\n\t}"
          : "=r"(h)
          : "r"(byte));
    } else {
      const uint32_t pair = ((i < 2 ? w0 : w1) >> (16 * (i & 1))) & 0xFFFFu;
      asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
          : "=r"(h)
          : "r"(pair));
    }
    float lo, hi;
    asm("{\n\t.reg .b16 a, b;\n\tmov.b32 {a, b}, %2;\n\tcvt.f32.f16 %0, a;\n\tcvt.f32.f16 %1, b;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(h));
    lo *= sc;  // exact: a power of two times a code value, inside the fp32 range
    hi *= sc;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(o[i]) : "f"(hi), "f"(lo));
  }
  if (sb == 255u) return make_uint4(kBf16NaNx2, kBf16NaNx2, kBf16NaNx2, kBf16NaNx2);
  return make_uint4(o[0], o[1], o[2], o[3]);
}

template <int FMT, bool SWZ>
__global__ void __launch_bounds__(kGemmThreads, 2) mx_gemm_kernel(GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kGemmStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* acc_full = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(acc_full + 1);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t m0 = (int64_t)blockIdx.y * kBM, n0 = (int64_t)blockIdx.x * kBN;
  const int nk = (int)(a.K / kBK);
  constexpr int kCodeBytesPer8 = FMT == kFmtE2M1 ? 4 : 8;  // code bytes of 8 elements
  const int64_t code_row = FMT == kFmtE2M1 ? a.K / 2 : a.K;

  pdl_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(full + s), kProducerWarps);
      mbar_init(smem_u32(empty + s), 1);
    }
    mbar_init(smem_u32(acc_full), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_wait();  // also: the kernel before may still hold this SM's tensor memory until then
  if (warp == kProducerWarps) {
    tmem_alloc(smem_u32(tmem_slot), kBN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool failed = false;

  if (warp < kProducerWarps) {
    // ---------------- producers ----------------
    // chunk q in [0, 2048): operand q / 1024 (A, B), row (q % 1024) / 8, 8 elements
    // 8 (q % 8) .. +7 of the K step; this thread takes q = tid + 256 j.
    uint32_t w0[kChunksPerThread], w1[kChunksPerThread], sb[kChunksPerThread];
    auto load_step = [&](int kk) {
#pragma unroll
      for (int j = 0; j < kChunksPerThread; ++j) {
        const int q = tid + 256 * j;
        const bool is_b = q >= 1024;
        const int r = (q & 1023) >> 3, c = q & 7;
        const int64_t row = (is_b ? n0 : m0) + r;
        const int64_t rows = is_b ? a.N : a.M;
        w0[j] = 0u;
        w1[j] = 0u;
        sb[j] = 0u;
        if (row < rows) {
          const int64_t k = (int64_t)kk * kBK + 8 * c;
          const uint8_t* codes = static_cast<const uint8_t*>(is_b ? a.b_codes : a.a_codes) +
                                 row * code_row + k * kCodeBytesPer8 / 8;
          if (FMT == kFmtE2M1) {
            w0[j] = load_u32(codes);
          } else {
            const uint2 v = load_u64(codes);
            w0[j] = v.x;
            w1[j] = v.y;
          }
          const int64_t scols = is_b ? a.b_scale_cols : a.a_scale_cols;
          const int64_t kb = k >> 5;
          const uint8_t* sc = is_b ? a.b_scales : a.a_scales;
          sb[j] = load_u8(sc + (SWZ ? swizzled_offset(row, kb, scols) : row * scols + kb));
        }
      }
    };
    load_step(0);
    for (int kk = 0; kk < nk; ++kk) {
      const int s = kk % kStages;
      if (kk >= kStages) {
        mbar_wait(smem_u32(empty + s), ((kk / kStages) & 1) ^ 1, &failed, kGemmWaitNs, a.err);
        failed = __any_sync(0xFFFFFFFFu, failed);  // the warp leaves together (__syncwarp below)
      }
      if (failed) break;
      uint8_t* stage = smem + s * kGemmStageBytes;
#pragma unroll
      for (int j = 0; j < kChunksPerThread; ++j) {
        const int q = tid + 256 * j;
        const int r = (q & 1023) >> 3, c = q & 7;
        const uint4 v = dequant8<FMT>(w0[j], w1[j], sb[j]);
        *reinterpret_cast<uint4*>(stage + (q >= 1024 ? kOperandBytes : 0) + r * 128 +
                                  ((c ^ (r & 7)) << 4)) = v;
      }
      if (kk + 1 < nk) load_step(kk + 1);  // next step's codes in flight during the wait
      fence_proxy_async_smem();            // the writes are visible to the tensor cores
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(full + s));
    }
  } else if (warp == kProducerWarps && lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc = idesc_bf16_f32(kBM, kBN);
    for (int kk = 0; kk < nk; ++kk) {
      const int s = kk % kStages;
      mbar_wait(smem_u32(full + s), (kk / kStages) & 1, &failed, kGemmWaitNs, a.err);
      if (failed) break;
      tc_fence_after();
      const uint32_t sa = smem_u32(smem + s * kGemmStageBytes), sbb = sa + kOperandBytes;
#pragma unroll
      for (int k16 = 0; k16 < kBK / 16; ++k16) {
        mma_bf16(tmem, desc_sw128(sa + 32 * k16), desc_sw128(sbb + 32 * k16), idesc,
                 (kk > 0 || k16 > 0) ? 1u : 0u);
      }
      mma_commit(smem_u32(empty + s));  // stage free once these MMAs have read it
    }
    mma_commit(smem_u32(acc_full));  // tracks every MMA issued above
  }
  if (warp >= kProducerWarps) {
    // ---------------- epilogue ----------------
    bool efailed = false;
    mbar_wait(smem_u32(acc_full), 0, &efailed, kGemmWaitNs, a.err);
    efailed = __any_sync(0xFFFFFFFFu, efailed || failed);
    tc_fence_after();
    const int quarter = warp & 3;
    const int64_t row = m0 + quarter * 32 + lane;
#pragma unroll 1
    for (int cb = 0; cb < kBN / 32; ++cb) {
      float y[32];
      if (!efailed) tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(cb * 32), y);
      if (efailed || row >= a.M) continue;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int64_t col = n0 + cb * 32 + g * 8;
        if (col >= a.N) break;
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
              : "=r"(o[i])
              : "f"(a.alpha * y[g * 8 + 2 * i + 1]), "f"(a.alpha * y[g * 8 + 2 * i]));
        }
        *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.c) + row * a.N + col) =
            make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kProducerWarps) tmem_dealloc(tmem, kBN);
}

template <int FMT, bool SWZ>
cudaError_t launch_t(const GemmArgs& a, cudaStream_t stream) {
  const void* k = reinterpret_cast<const void*>(&mx_gemm_kernel<FMT, SWZ>);
  if (resident_ctas(k, kGemmThreads, kGemmSmem, 0) <= 0) return cudaErrorInvalidConfiguration;
  const dim3 grid((unsigned)((a.N + kBN - 1) / kBN), (unsigned)((a.M + kBM - 1) / kBM));
  return launch_pdl(&mx_gemm_kernel<FMT, SWZ>, grid, dim3(kGemmThreads), kGemmSmem, stream, a);
}

}  // namespace

cudaError_t launch_gemm(int fmt, bool swizzled, const GemmArgs& a, cudaStream_t stream) {
  if (fmt == kFmtE2M1) {
    return swizzled ? launch_t<kFmtE2M1, true>(a, stream) : launch_t<kFmtE2M1, false>(a, stream);
  }
  return swizzled ? launch_t<kFmtE4M3, true>(a, stream) : launch_t<kFmtE4M3, false>(a, stream);
}

}  // namespace mxq
