// mx_hadamard.cu -- rotate + block quantize / QDQ when the rotation is a scaled Hadamard matrix:
// an in-register fast Walsh-Hadamard transform on the streaming kernel's layout.
//
// The rotation of the QuTLASS pull request (feature list: rotation matrices loaded at run time,
// sizes 16/32/64/128; benchmark review thread: hadamard(g) * g^-0.5 in the activation dtype)
// multiplies every g-element chunk along K by H. When H = c * S_g, with S_g the Sylvester
// Hadamard matrix of order g (entries (-1)^popcount(i & j)) and c = H[0][0], the product is
// y_j = c * sum_i (-1)^popcount(i & j) x_i: log2(g) butterfly stages of additions and
// subtractions, then one multiplication by c, all in fp32. The caller states that H has this
// form (MX_ROT_HADAMARD); every CTA checks it on the bf16 bit patterns of H and, where it does
// not hold, computes the dense product sum_i x_i H[i][j] with fp32 FMAs instead (increasing i),
// so the results are the rotation's for any H, only slower.
//
// Layout: as in mx_stream.cu, the input is a flat sequence of 32-element blocks, a persistent
// grid walks them with a grid stride and consecutive threads own consecutive blocks (a warp moves
// 2 KiB of contiguous input) and each thread loads its next block before working on the current
// one. A chunk never
// crosses a row (K % g == 0) and starts at a multiple of g in the flat order, so a g = 16 or 32
// chunk lies inside one thread's block and a g = 64 / 128 chunk spans 2 / 4 consecutive lanes,
// whose butterfly stages exchange values with shuffles. The loop's trip count is the same for
// every lane of a warp (lanes past the end compute on zeros and store nothing), so the shuffles
// always have the whole warp. After the rotation the block's fp32 values take the same
// quantization steps as in the tensor-core kernel; for the MX formats the factor c is folded
// into the power-of-two scaling (exact, see mx_hadamard_block).
#include "mx_device.cuh"
#include "mx_launch.h"

namespace mxq {

namespace {

constexpr int kThreads = 256;

// bf16 bits of c * S_g[i][j]: the sign of c flipped where popcount(i & j) is odd.
__device__ __forceinline__ uint32_t scaled_sylvester_bits(uint32_t c_bits, int i, int j) {
  return c_bits ^ ((uint32_t)(__popc(i & j) & 1) << 15);
}

// Whether H (bf16 [G, G], row-major, 16-byte aligned) equals H[0][0] * S_G bit for bit. Every
// thread of the block gets the answer.
template <int G>
__device__ __forceinline__ bool is_scaled_sylvester(const uint16_t* H, uint32_t c_bits) {
  bool ok = true;
  for (int v = threadIdx.x; v < G * G / 8; v += kThreads) {
    const uint4 q = load_v4(H + 8 * v);  // entries 8v .. 8v + 7 of row (8v) / G
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    const int i = (8 * v) / G, j0 = (8 * v) % G;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const uint32_t h = (w[k >> 1] >> (16 * (k & 1))) & 0xFFFFu;
      ok = ok && h == scaled_sylvester_bits(c_bits, i, j0 + k);
    }
  }
  return __syncthreads_and(ok) != 0;
}

// (a0, a1) <- (a0 + b0, a1 + b1) and (b0, b1) <- (a0 - b0, a1 - b1) with packed fp32 operations
// (each element rounded once, as the scalar operations would).
__device__ __forceinline__ void addsub2(float& a0, float& a1, float& b0, float& b1) {
  asm("{\n\t.reg .b64 a, b, s, d;\n\tmov.b64 a, {%0, %1};\n\tmov.b64 b, {%2, %3};\n\t"
      "add.rn.f32x2 s, a, b;\n\tsub.rn.f32x2 d, a, b;\n\tmov.b64 {%0, %1}, s;\n\t"
      "mov.b64 {%2, %3}, d;\n\t}"
      : "+f"(a0), "+f"(a1), "+f"(b0), "+f"(b1));
}

// v <- S_G v over every G-chunk of the warp's values (unnormalized fast Walsh-Hadamard
// transform). Stage h pairs the elements i and i + h of a chunk ((i & h) == 0) into
// (v_i + v_{i+h}, v_i - v_{i+h}); stage 1 pairs neighbours (scalar), stages h >= 2 take two
// neighbouring pairs at once (packed). Stages inside a thread first; for G = 64 / 128 the element
// index i = 32 * (lane within the chunk) + t, so stage h = 32 / 64 pairs lane bit 1 / 2: the
// lower lane keeps its value plus its partner's, the upper lane its partner's minus its own.
template <int G>
__device__ __forceinline__ void fwht(float* v, int lane) {
  constexpr int kIn = G < 32 ? G : 32;
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float a = v[i], b = v[i + 1];
    v[i] = a + b;
    v[i + 1] = a - b;
  }
#pragma unroll
  for (int h = 2; h < kIn; h <<= 1) {
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
      if ((i & h) == 0) addsub2(v[i], v[i + 1], v[i + h], v[i + h + 1]);
    }
  }
#pragma unroll
  for (int d = 1; d < G / 32; d <<= 1) {
    const float sgn = (lane & d) ? -1.0f : 1.0f;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const float p = __shfl_xor_sync(0xFFFFFFFFu, v[i], d);
      v[i] = fmaf(sgn, v[i], p);  // exact product by +-1, one rounding
    }
  }
}

// y_j = sum_i x_i H[i][j] over each G-chunk in fp32 FMAs, increasing i (any H). The thread's 32
// values go through its row of the warp's staging area s_w (32 rows of 33 floats), so that only
// the accumulators stay in registers and a G = 64 / 128 chunk reads the values of the lanes
// holding its other parts. Rows of H are read through L1 with 16-byte loads. Only runs when H
// is not a scaled Sylvester matrix.
template <int G>
__device__ __forceinline__ void dense_rotate(float* v, const uint16_t* H, int lane, float* s_w) {
  float* mine = s_w + lane * 33;
#pragma unroll
  for (int t = 0; t < 32; ++t) mine[t] = v[t];
  __syncwarp();
  float acc[32];
#pragma unroll
  for (int j = 0; j < 32; ++j) acc[j] = 0.0f;
  if constexpr (G <= 32) {
#pragma unroll 1
    for (int i = 0; i < G; ++i) {
#pragma unroll
      for (int j0 = 0; j0 < G; j0 += 8) {
        const uint4 q = load_v4(H + i * G + j0);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const float h = (jj & 1) ? bf16_hi(w[jj >> 1]) : bf16_lo(w[jj >> 1]);
#pragma unroll
          for (int k = 0; k < 32; k += G) acc[k + j0 + jj] = fmaf(mine[k + i], h, acc[k + j0 + jj]);
        }
      }
    }
  } else {
    constexpr int kLanes = G / 32;
    const int first = lane & ~(kLanes - 1), part = lane & (kLanes - 1);
#pragma unroll 1
    for (int i = 0; i < G; ++i) {  // input i of the chunk: lane first + i / 32, value i % 32
      const float xi = s_w[(first + (i >> 5)) * 33 + (i & 31)];
      const uint16_t* hrow = H + i * G + part * 32;
#pragma unroll
      for (int j0 = 0; j0 < 32; j0 += 8) {
        const uint4 q = load_v4(hrow + j0);
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const float h = (jj & 1) ? bf16_hi(w[jj >> 1]) : bf16_lo(w[jj >> 1]);
          acc[j0 + jj] = fmaf(xi, h, acc[j0 + jj]);
        }
      }
    }
  }
  __syncwarp();  // every lane has read the staging area before it is written again
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] = acc[j];
}

// MX block of the unscaled transform s (y = c * s): returns the E8M0 byte and writes the QDQ
// output or the codes. The abs-max of y is |c| * max |s_j| rounded once (rounding is monotonic
// and symmetric, so this is max_j |fl(c s_j)|), and the values are scaled by q = c * 2^-s in one
// multiplication: fl(s_j q) = fl(c s_j) * 2^-s exactly while q is a normal number (the scaling
// by a power of two is exact); otherwise the two multiplications are done in turn.
// The Quest-like scale (FMT kFmtE2M1Quest) takes the sum of the squares of y as c^2 times that of
// s (one rounding more than summing the squares of y itself); where that product leaves the
// plain-sum range, y = c * s is formed and the scaled sum of quest_byte_f32x32 taken instead.
template <int FMT, bool QDQ>
__device__ __forceinline__ uint32_t mx_hadamard_block(float* v, float c, uint32_t* out) {
  uint32_t byte;
  bool c_applied = false;  // v already holds y = c * s
  if constexpr (FMT == kFmtE2M1Quest) {
    const float sum = __fmul_rn(__fmul_rn(c, c), sq_sum<32>(v));
    if (quest_sum_in_range(sum)) {
      byte = quest_byte_from_sum(sum, 127u);
    } else {
#pragma unroll
      for (int i = 0; i < 16; ++i) mul2(v[2 * i], v[2 * i + 1], c);
      c_applied = true;
      const uint32_t E = absmax_f32x32(v) >> 23;
      byte = quest_byte_from_sum(scaled_sq_sum<32>(v, quest_prescale(E)), E);
    }
  } else {
    const float amax_s = __uint_as_float(absmax_f32x32(v));
    const float amax = __fmul_rn(fabsf(c), amax_s);
    byte = scale_byte_from_amax_bits<FMT>(__float_as_uint(amax) & 0x7FFFFFFFu);
  }
  const bool special = __any_sync(0xFFFFFFFFu, byte == 255u);
  const float inv = inv_scale_of(byte);
  const float q = c_applied ? inv : __fmul_rn(c, inv);
  if (c_applied || fabsf(q) >= 1.17549435e-38f || c == 0.0f) {  // one exact step
#pragma unroll
    for (int i = 0; i < 16; ++i) mul2(v[2 * i], v[2 * i + 1], q);
  } else {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      mul2(v[2 * i], v[2 * i + 1], c);
      mul2(v[2 * i], v[2 * i + 1], inv);
    }
  }
  if (QDQ) {
    const float sc = scale_of(byte);
#pragma unroll
    for (int i = 0; i < 16; ++i) out[i] = qdq2<FMT>(v[2 * i], v[2 * i + 1], sc);
  } else if (mx_e2m1<FMT>()) {
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = codes8_e2m1(v + 8 * i);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint2 cc = codes8_e4m3(v + 8 * i);
      out[2 * i] = cc.x;
      out[2 * i + 1] = cc.y;
    }
  }
  if (special && byte == 255u) {
    const uint32_t fill = QDQ ? kBf16NaNx2 : (mx_e2m1<FMT>() ? 0u : kE4M3NaNx4);
#pragma unroll
    for (int i = 0; i < (QDQ ? 16 : (mx_e2m1<FMT>() ? 4 : 8)); ++i) out[i] = fill;
  }
  return byte;
}

// CTAs per SM the register budget is set for: QDQ (two 32-byte stores per block, the widest
// epilogue) 2, which measured 6-8% faster than 3 (its 80-register build spills); codes 3, 5-10%
// faster than 2 (rotated MXFP8 x[8192, 28672]: 115.2 -> 109.1 us).
template <int OUT>
__host__ __device__ constexpr int hadamard_min_ctas() {
  return OUT == kRotQdq ? 2 : 3;
}

template <int FMT, int OUT, bool SWZ, int G>
__global__ void __launch_bounds__(kThreads, hadamard_min_ctas<OUT>())
    mx_hadamard_kernel(StreamArgs a) {
  constexpr bool kNv = FMT == kFmtNVFP4;
  constexpr bool kQdq = OUT == kRotQdq;
  // output bytes per 32-element block: QDQ bf16 64, E4M3 codes 32, E2M1 codes 16, debug fp32 128
  constexpr int kOutBytes = OUT == kRotDebug ? 128 : (kQdq ? 64 : (FMT == kFmtE4M3 ? 32 : 16));
  __shared__ float s_dense[kThreads / 32][32 * 33];  // dense_rotate's staging, one area per warp
  const int tid = threadIdx.x, lane = tid & 31;
  const uint8_t* x = static_cast<const uint8_t*>(a.x);
  const uint16_t* H = static_cast<const uint16_t*>(a.H);
  const int64_t cblk = a.K >> 5;  // blocks per row
  const int64_t nblk = a.M * cblk;
  const int64_t stride = (int64_t)gridDim.x * kThreads;
  pdl_launch_dependents();
  if (lane == 0) {  // the warp's first 2 KiB into L2 (a hint, see prefetch_l2)
    const int64_t s0 = (int64_t)blockIdx.x * kThreads + (tid & ~31);
    if (s0 < nblk) prefetch_l2(x + s0 * 64, (uint32_t)((nblk - s0 < 32 ? nblk - s0 : 32) * 64));
  }
  pdl_wait();

  // the warp's blocks: wb + lane for wb = the warp's first block, + stride, ... (the same
  // number of iterations for every lane)
  int64_t wb = (int64_t)blockIdx.x * kThreads + (tid & ~31);
  int64_t b = wb + lane;
  uint32_t cur[16], nxt[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) cur[i] = 0u;
  if (b < nblk) {  // in flight while H is checked
    load32B(x + b * 64, cur);
    load32B(x + b * 64 + 32, cur + 8);
  }
  const uint32_t c_bits = load_u16(H);
  const float c = __uint_as_float(c_bits << 16);
  const bool hadamard = is_scaled_sylvester<G>(H, c_bits);
  const float cm = hadamard ? c : 1.0f;  // the dense product already holds the rotated values
  float gs = 0.0f, r6 = 0.0f;
  if (kNv && OUT != kRotDebug) {
    gs = load_f32(a.gscale);
    r6 = __fdiv_rn(gs, 6.0f);
  }
  const int64_t row_step = stride / cblk, col_step = stride - row_step * cblk;
  int64_t row = b / cblk, col = b - row * cblk;  // advanced incrementally below

  for (; wb < nblk; wb += stride, b += stride) {
    const bool valid = b < nblk;
    const int64_t bn = b + stride;
#pragma unroll
    for (int i = 0; i < 16; ++i) nxt[i] = 0u;
    if (bn < nblk) {  // next block in flight while this one is converted
      load32B(x + bn * 64, nxt);
      load32B(x + bn * 64 + 32, nxt + 8);
    }
    float v[32];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      v[2 * i] = bf16_lo(cur[i]);
      v[2 * i + 1] = bf16_hi(cur[i]);
    }
    if (hadamard) {
      fwht<G>(v, lane);
    } else {
      dense_rotate<G>(v, H, lane, s_dense[tid >> 5]);
    }
    uint8_t* dst = static_cast<uint8_t*>(a.out) + b * kOutBytes;
    if constexpr (OUT == kRotDebug) {
#pragma unroll
      for (int i = 0; i < 16; ++i) mul2(v[2 * i], v[2 * i + 1], cm);
      if (valid) {
        float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
        for (int i = 0; i < 8; ++i) d4[i] = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
      }
    } else {
      uint32_t o[16];
      uint32_t byte;
      if constexpr (kNv) {
#pragma unroll
        for (int i = 0; i < 16; ++i) mul2(v[2 * i], v[2 * i + 1], cm);
        const NvScales n = nv_scales(absmax_f32x16(v), absmax_f32x16(v + 16), gs, r6);
        nv_block_f32<kQdq>(v, o, n);
        byte = n.bytes;
      } else {
        byte = mx_hadamard_block<FMT, kQdq>(v, cm, o);
      }
      if (valid) {
        if (kQdq) {
          store32B(dst, o);
          store32B(dst + 32, o + 8);
        } else if (FMT == kFmtE4M3) {
          store32B(dst, o);
        } else {
          __stcs(reinterpret_cast<uint4*>(dst), make_uint4(o[0], o[1], o[2], o[3]));
        }
        if (!kQdq) {
          // linear: flat block order; swizzled: the block's row / column in the 128x4 tiles.
          // NVFP4: two scale bytes (blocks 2 col and 2 col + 1), adjacent in both layouts.
          if (kNv) {
            const int64_t off = SWZ ? swizzled_offset(row, 2 * col, a.scale_cols) : 2 * b;
            *reinterpret_cast<uint16_t*>(a.scales + off) = (uint16_t)byte;
          } else {
            const int64_t off = SWZ ? swizzled_offset(row, col, a.scale_cols) : b;
            a.scales[off] = (uint8_t)byte;
          }
        }
      }
    }
#pragma unroll
    for (int i = 0; i < 16; ++i) cur[i] = nxt[i];
    col += col_step;
    row += row_step;
    if (col >= cblk) {
      col -= cblk;
      ++row;
    }
  }
  if (SWZ && OUT == kRotCodes) {
    zero_swizzled_pads(a.scales, a.M, kNv ? 2 * cblk : cblk, a.scale_rows, a.scale_cols,
                       (int64_t)blockIdx.x * kThreads + tid, stride);
  }
}

template <int FMT, int OUT, bool SWZ, int G>
cudaError_t launch_t(const StreamArgs& a, cudaStream_t stream) {
  const void* k = reinterpret_cast<const void*>(&mx_hadamard_kernel<FMT, OUT, SWZ, G>);
  const int64_t nblk = a.M * (a.K >> 5);
  int64_t need = (nblk + kThreads - 1) / kThreads;
  if (SWZ && OUT == kRotCodes) {  // enough threads for the pad items as well
    const int64_t pad_need = ((a.scale_rows - a.M) * (a.scale_cols / 4) + kThreads - 1) / kThreads;
    if (pad_need > need) need = pad_need;
  }
  if (need <= 0) return cudaSuccess;
  const int resident = resident_ctas(k, kThreads, 0, 0);
  if (resident <= 0) return cudaErrorInvalidConfiguration;
  const int grid = (int)(need < resident ? need : resident);
  return launch_pdl(&mx_hadamard_kernel<FMT, OUT, SWZ, G>, dim3(grid), dim3(kThreads), 0, stream,
                    a);
}

template <int FMT, int OUT, bool SWZ>
cudaError_t launch_g(int g, const StreamArgs& a, cudaStream_t st) {
  switch (g) {
    case 16: return launch_t<FMT, OUT, SWZ, 16>(a, st);
    case 32: return launch_t<FMT, OUT, SWZ, 32>(a, st);
    case 64: return launch_t<FMT, OUT, SWZ, 64>(a, st);
    default: return cudaErrorInvalidValue;  // g = 128 calls run on the tensor-core kernel
  }
}

template <int FMT>
cudaError_t launch_fmt(int out_kind, bool swz, int g, const StreamArgs& a, cudaStream_t st) {
  if (out_kind == kRotQdq) return launch_g<FMT, kRotQdq, false>(g, a, st);
  return swz ? launch_g<FMT, kRotCodes, true>(g, a, st) : launch_g<FMT, kRotCodes, false>(g, a, st);
}

}  // namespace

cudaError_t launch_hadamard(int fmt, int out_kind, bool swizzled, int g, const StreamArgs& a,
                            cudaStream_t stream) {
  if (out_kind == kRotDebug) return launch_g<kFmtE2M1, kRotDebug, false>(g, a, stream);
  if (fmt == kFmtE2M1) return launch_fmt<kFmtE2M1>(out_kind, swizzled, g, a, stream);
  if (fmt == kFmtE2M1Quest) return launch_fmt<kFmtE2M1Quest>(out_kind, swizzled, g, a, stream);
  if (fmt == kFmtNVFP4) return launch_fmt<kFmtNVFP4>(out_kind, swizzled, g, a, stream);
  return launch_fmt<kFmtE4M3>(out_kind, swizzled, g, a, stream);
}

}  // namespace mxq
