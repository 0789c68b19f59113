// mx_stream.cu -- block quantize / QDQ without rotation (HBM-bound streaming kernel).
//
// The input [M, K] is contiguous and K % 32 == 0, so it is a flat sequence of 32-element
// blocks; codes and QDQ outputs are flat sequences too, and linear scales are indexed by the
// flat block number. A persistent grid walks the blocks with a grid stride (grouped calls: one
// contiguous range per CTA): consecutive threads own consecutive blocks (a warp moves 2 KiB of
// contiguous input with 32-byte vector loads), and each thread loads its next block before
// working on the current one. A thread
// takes the block's abs-max with packed bf16x2 abs-max instructions, derives the E8M0 byte
// from the exponent field, converts in registers with the hardware paired converters, and
// writes the block's codes (16 or 32 bytes) or dequantized bf16 (two 32-byte stores) and its
// scale byte: at the flat block index (linear) or at its place in the 128x4 tiles (swizzled;
// the row/column of the block are advanced incrementally, grouped calls map the row to its
// expert's padded row). After the main loop a pass spread over the whole grid writes zeros
// into the pad bytes.
// NVFP4 (E2M1 codes, one E4M3 scale per 16 elements under an fp32 global scale) runs on the
// same kernel: a thread's 32 elements are two NVFP4 blocks; so does MXFP4 under the Quest-like
// scale (FMT kFmtE2M1Quest: the scale from the block's sum of squares instead of its abs-max).
// Grouped MX calls with swizzled scales take a grid-stride kernel with a per-CTA table of row
// shifts (mx_grouped_table_kernel, below) while that table fits.
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

// Sum of the squares of one block held in w[16] (bf16 pairs), each value scaled by m, in the
// order of sq_sum<32> (element i of the block to chain i % 4); the values are widened on the fly.
__device__ __forceinline__ float sq_sum_bf16x32(const uint32_t* w, float m) {
  float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    float a = bf16_lo(w[i]), b = bf16_hi(w[i]), c = bf16_lo(w[i + 1]), d = bf16_hi(w[i + 1]);
    mul2(a, b, m);
    mul2(c, d, m);
    fma_sq2(s0, s1, a, b);
    fma_sq2(s2, s3, c, d);
  }
  return (s0 + s1) + (s2 + s3);
}

// Quest-like scale byte of one block held in w[16], with the arithmetic and the order of
// quest_byte_f32x32 on the widened values (the plain sum is the scaled one with m = 1).
__device__ __forceinline__ uint32_t quest_byte_bf16x32(const uint32_t* w) {
  const float s = sq_sum_bf16x32(w, 1.0f);
  if (quest_sum_in_range(s)) return quest_byte_from_sum(s, 127u);
  const uint32_t E = (absmax_block(w) << 16) >> 23;
  return quest_byte_from_sum(sq_sum_bf16x32(w, quest_prescale(E)), E);
}

// Quantize (or QDQ) one block held in w[16]; writes codes / bf16 through `out` when `ok`.
// Returns the scale byte.
template <int FMT, bool QDQ>
__device__ __forceinline__ uint32_t block_kernel(const uint32_t* w, bool ok, void* out) {
  const uint32_t byte = FMT == kFmtE2M1Quest ? quest_byte_bf16x32(w)
                                             : scale_byte_from_amax_bits<FMT>(absmax_block(w) << 16);
  const float inv = inv_scale_of(byte);
  const bool special = __any_sync(__activemask(), byte == 255u);  // a NaN / Inf block nearby
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
      if (mx_e2m1<FMT>()) {
        c[q] = codes8_e2m1(t);
      } else {
        const uint2 p = codes8_e4m3(t);
        c[2 * q] = p.x;
        c[2 * q + 1] = p.y;
      }
    }
    if (special && byte == 255u) {
#pragma unroll
      for (int i = 0; i < 8; ++i) c[i] = mx_e2m1<FMT>() ? 0u : kE4M3NaNx4;
    }
    if (ok) {
      if (mx_e2m1<FMT>()) {
        __stcs(static_cast<uint4*>(out), make_uint4(c[0], c[1], c[2], c[3]));
      } else {
        store32B(out, c);
      }
    }
  }
  return byte;
}

// abs-max of 8 bf16x2 words (one 16-element block) as sign-free bf16 bits; NaN propagates.
__device__ __forceinline__ uint32_t absmax_words8(const uint32_t* w) {
  uint32_t m[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[i]) : "r"(w[2 * i]), "r"(w[2 * i + 1]));
  }
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[0]) : "r"(m[0]), "r"(m[2]));
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[1]) : "r"(m[1]), "r"(m[3]));
  asm("max.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(m[0]) : "r"(m[0]), "r"(m[1]));
  return max(m[0] & 0x7FFFu, (m[0] >> 16) & 0x7FFFu);
}

// NVFP4: the 32 values in w[16] are two 16-element blocks. Writes their codes (16 bytes) or
// QDQ bf16 (64 bytes) through `out`; returns the two E4M3 scale bytes (first in the low byte).
template <bool QDQ>
__device__ __forceinline__ uint32_t nv_block_kernel(const uint32_t* w, void* out, float gs,
                                                    float r6) {
  const NvScales n = nv_scales(absmax_words8(w) << 16, absmax_words8(w + 8) << 16, gs, r6);
  const bool special = __any_sync(__activemask(), n.special[0] || n.special[1]);
  if (QDQ) {
    uint32_t o[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      float lo = bf16_lo(w[i]), hi = bf16_hi(w[i]);
      mul2(lo, hi, n.enc[i >> 3]);
      o[i] = qdq2_e2m1(lo, hi, n.dq[i >> 3]);
    }
    if (special) {
#pragma unroll
      for (int i = 0; i < 16; ++i) o[i] = n.special[i >> 3] ? kBf16NaNx2 : o[i];
    }
    store32B(out, o);
    store32B(static_cast<uint8_t*>(out) + 32, o + 8);
  } else {
    uint32_t c[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      float t[8];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        t[2 * i] = bf16_lo(w[4 * q + i]);
        t[2 * i + 1] = bf16_hi(w[4 * q + i]);
        mul2(t[2 * i], t[2 * i + 1], n.enc[q >> 1]);
      }
      c[q] = codes8_e2m1(t);
    }
    if (special) {
#pragma unroll
      for (int q = 0; q < 4; ++q) c[q] = n.special[q >> 1] ? 0u : c[q];
    }
    __stcs(static_cast<uint4*>(out), make_uint4(c[0], c[1], c[2], c[3]));
  }
  return n.bytes;
}

// largest e in [0, n) with v[e] <= key (v[0] <= key assumed)
__device__ __forceinline__ int last_not_above(const int64_t* v, int n, int64_t key) {
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (v[mid] <= key) lo = mid;
    else hi = mid;
  }
  return lo;
}

// Pad bytes of a grouped call's swizzled scale buffer, spread evenly over every thread of the
// grid (s_off: clamped first row of each expert and the end; s_prow: first padded scale row of
// each expert and the total):
//  (A) in each data row, the bytes past the last data column of its last 4-byte word (only when
//      the data columns are not a multiple of 4);
//  (B) the rows past the last expert's padded range: whole 128-row blocks, whose tiles form one
//      contiguous byte range at the end of the buffer (tiles are row-block-major), zeroed with
//      16-byte stores;
//  (C) the pad rows inside each expert's last 128-row block (those at or past its row count):
//      one warp per (expert, 4-byte word of the row) task, 4-byte stores into one tile.
// Runs after the main loop. Its cost is the work of the warps that get a task, so the inner
// pad rows are split into short per-warp tasks with 32-bit index arithmetic inside a tile:
// measured 0.5-0.6 us less per call than one thread per pad row writing the row's words in a
// loop (x[16384, 2048], 128 experts), and faster than running the same pass before the main
// loop, where it delays the loop's loads.
template <bool kNv>
__device__ __forceinline__ void zero_grouped_pads(const StreamArgs& a, const int64_t* s_off,
                                                  const int64_t* s_prow, int64_t cblk) {
  const int64_t cp = a.scale_cols, cp4 = cp >> 2;
  const int64_t dcols = kNv ? 2 * cblk : cblk;  // scale columns holding data
  const int64_t nthr = (int64_t)gridDim.x * kThreads;
  const int64_t t0 = (int64_t)blockIdx.x * kThreads + threadIdx.x;
  const int64_t used = s_prow[a.E] < a.scale_rows ? s_prow[a.E] : a.scale_rows;
  if (dcols & 3) {  // (A)
    const int64_t c4 = dcols & ~int64_t(3);
    for (int64_t r = t0; r < a.M; r += nthr) {
      const int ex = last_not_above(s_off, a.E, r);
      if (r < s_off[ex] || r >= s_off[ex + 1]) continue;  // rows outside every expert
      const int64_t pr = s_prow[ex] + (r - s_off[ex]);
      if (pr >= a.scale_rows) continue;
      uint8_t* run = a.scales + swizzled_offset(pr, c4, cp);
      for (int64_t c = dcols; c < c4 + 4; ++c) run[c - c4] = 0;
    }
  }
  uint4* tail = reinterpret_cast<uint4*>(a.scales + used * cp);  // (B)
  const int64_t tail_vecs = (a.scale_rows - used) * cp / 16;
  for (int64_t i = t0; i < tail_vecs; i += nthr) tail[i] = make_uint4(0u, 0u, 0u, 0u);
  // (C) one warp per (expert, 4-byte word) task; lane l takes rows l, l + 32, ... of the
  // expert's last 128-row block, whose word sits in one 512-byte tile
  const int lane = (int)(threadIdx.x & 31);
  const int64_t nwarps = (int64_t)gridDim.x * (kThreads / 32);
  const int64_t tasks = (int64_t)a.E * cp4;
  for (int64_t t = (int64_t)blockIdx.x * (kThreads / 32) + (threadIdx.x >> 5); t < tasks;
       t += nwarps) {
    int ex;
    int64_t w;
    if (tasks <= 0xFFFFFFFFll) {
      ex = (int)((uint32_t)t % (uint32_t)a.E);
      w = (uint32_t)t / (uint32_t)a.E;
    } else {
      ex = (int)(t % a.E);
      w = t / a.E;
    }
    const int64_t n = s_off[ex + 1] > s_off[ex] ? s_off[ex + 1] - s_off[ex] : 0;
    if (n == 0) continue;
    const int64_t last = s_prow[ex + 1] - kTileRows;  // first row of the last block (>= 0)
    const int64_t first_pad = s_prow[ex] + n;
    uint8_t* tile = a.scales + ((last >> 7) * cp4 + w) * 512;
#pragma unroll
    for (int k = lane; k < kTileRows; k += 32) {
      const int64_t pr = last + k;
      if (pr >= first_pad && pr < used) {
        *reinterpret_cast<uint32_t*>(tile + (k & 31) * 16 + (k >> 5) * 4) = 0u;
      }
    }
  }
}

// Register budget per instantiation (the grid is sized from the resulting occupancy): QDQ
// kernels are given room for more registers (66, 3 CTAs per SM), which measured 2-3% faster
// than the 50-register, 4-CTA build (x[8192,8192] 44.9 -> 44.0 us, x[4096,8192] 22.8 -> 22.1 us
// back to back); quantize kernels keep <= 64 registers and 4 CTAs per SM; grouped NVFP4 needs
// 78 and 3 CTAs (forcing 64 spills and measured 14% slower), and so does the Quest-like
// quantize (its sum of squares and scaled fallback spilled 40-132 bytes at 64).
template <int FMT, bool QDQ, bool GROUPED>
__host__ __device__ constexpr int stream_min_ctas() {
  return QDQ ? 1 : (((GROUPED && FMT == kFmtNVFP4) || FMT == kFmtE2M1Quest) ? 3 : 4);
}

// First blocks of each warp prefetched into L2 before pdl_wait: one 2 KiB span (the warp's
// first 32 blocks) per warp for the 4-CTA quantize builds, two spans (its first two iterations)
// for the 3-CTA builds (QDQ, grouped NVFP4), i.e. 64-96 KiB per SM. Measured on GB300 (steady,
// back to back): one span per warp took QDQ of x[8192, 8192] from 43.4 to 42.0 us and two
// to 41.4 us, while the quantize builds were fastest with one (E4M3 linear x[8192, 8192]
// 31.7 -> 30.3 us; two: 30.6 us); more in-flight prefetch competes with the previous kernel.
template <int FMT, bool QDQ, bool GROUPED>
__host__ __device__ constexpr int stream_prefetch_spans() {
  return stream_min_ctas<FMT, QDQ, GROUPED>() == 4 ? 1 : 2;
}

template <int FMT, bool QDQ, bool SWZ, bool GROUPED>
__global__ void __launch_bounds__(kThreads, stream_min_ctas<FMT, QDQ, GROUPED>())
    mx_stream_kernel(StreamArgs a) {
  __shared__ int64_t s_off[GROUPED ? kMaxExperts + 1 : 1];   // clamped first row of expert e
  __shared__ int64_t s_prow[GROUPED ? kMaxExperts + 1 : 1];  // first padded scale row of e
  __shared__ int64_t s_warp[kThreads / 32];
  constexpr bool kNv = FMT == kFmtNVFP4;
  __shared__ float s_gs[GROUPED && kNv ? kMaxExperts : 1];  // NVFP4 grouped: gs of expert e
  const int tid = threadIdx.x;
  constexpr int kCodeBytes = QDQ ? 64 : (FMT == kFmtE4M3 ? 32 : 16);  // output bytes per block
  pdl_launch_dependents();
  {
    // L2 prefetch of this warp's first blocks (before pdl_wait: a hint, see prefetch_l2),
    // laid out as the block walk below assigns them
    const int64_t nblk0 = a.M * (a.K >> 5);
    int64_t w0, wend, wstride;
    if (GROUPED) {
      const int64_t per = ((nblk0 + gridDim.x - 1) / gridDim.x + kThreads - 1) / kThreads * kThreads;
      w0 = (int64_t)blockIdx.x * per + (tid & ~31);
      wend = (int64_t)(blockIdx.x + 1) * per < nblk0 ? (int64_t)(blockIdx.x + 1) * per : nblk0;
      wstride = kThreads;
    } else {
      w0 = (int64_t)blockIdx.x * kThreads + (tid & ~31);
      wend = nblk0;
      wstride = (int64_t)gridDim.x * kThreads;
    }
    if ((tid & 31) == 0) {
#pragma unroll
      for (int d = 0; d < stream_prefetch_spans<FMT, QDQ, GROUPED>(); ++d) {
        const int64_t s0 = w0 + d * wstride;
        if (s0 < wend) {
          const int64_t n = wend - s0 < 32 ? wend - s0 : 32;
          prefetch_l2(static_cast<const uint8_t*>(a.x) + s0 * 64, (uint32_t)(n * 64));
        }
      }
    }
  }
  pdl_wait();
  float gs = 0.0f, r6 = 0.0f;  // NVFP4 global scale and gs / 6 (grouped: of the current expert)
  if (kNv && !GROUPED) {
    gs = load_f32(a.gscale);
    r6 = __fdiv_rn(gs, 6.0f);
  }

  const uint8_t* x = static_cast<const uint8_t*>(a.x);
  const int64_t cblk = a.K >> 5;  // blocks per row
  const int64_t nblk = a.M * cblk;
  // Plain calls walk the blocks with a grid stride. Grouped calls give each CTA one contiguous
  // range, so that a thread's row advances by only kThreads / (K/32) rows per step and its
  // expert can be tracked incrementally instead of searched for every block.
  int64_t b, b_end, stride;
  if (GROUPED) {
    const int64_t per_cta = ((nblk + gridDim.x - 1) / gridDim.x + kThreads - 1) / kThreads * kThreads;
    b = (int64_t)blockIdx.x * per_cta + tid;
    b_end = (int64_t)(blockIdx.x + 1) * per_cta < nblk ? (int64_t)(blockIdx.x + 1) * per_cta : nblk;
    stride = kThreads;
  } else {
    b = (int64_t)blockIdx.x * kThreads + tid;
    b_end = nblk;
    stride = (int64_t)gridDim.x * kThreads;
  }
  const int64_t row_step = stride / cblk, col_step = stride - row_step * cblk;
  int64_t row = b / cblk, col = b - row * cblk;  // advanced incrementally below
  uint32_t cur[16], nxt[16];
  if (b < b_end) {  // the first block's load is in flight during the grouped prologue
    load32B(x + b * 64, cur);
    load32B(x + b * 64 + 32, cur + 8);
  }
  if (GROUPED) {
    // expert e owns ceil(n_e / 128) * 128 padded scale rows; s_prow is their prefix sum
    int64_t nb[4];
    int64_t local = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = tid * 4 + j;
      nb[j] = 0;
      if (e < a.E) {
        int64_t lo = load_s64(a.offsets + e), hi = load_s64(a.offsets + e + 1);
        if (kNv) s_gs[e] = load_f32(a.gscale + e);
        lo = lo < 0 ? 0 : (lo > a.M ? a.M : lo);
        hi = hi < lo ? lo : (hi > a.M ? a.M : hi);
        s_off[e] = lo;
        nb[j] = (hi - lo + kTileRows - 1) / kTileRows * kTileRows;
        local += nb[j];
      }
    }
    if (tid == 0) {
      const int64_t end = load_s64(a.offsets + a.E);
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
    int64_t run = incl - local;
    for (int w = 0; w < (tid >> 5); ++w) run += s_warp[w];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = tid * 4 + j;
      if (e < a.E) s_prow[e] = run;
      run += nb[j];
    }
    if (tid == kThreads - 1) s_prow[a.E] = run;
    __syncthreads();
  }

  // Grouped: the expert of `row` and, in registers, its first row, end row and first padded
  // scale row (and NVFP4 global scale); reloaded from shared memory only when `row` leaves it.
  int e = GROUPED ? last_not_above(s_off, a.E, row) : 0;
  int64_t e_lo = 0, e_hi = 0, e_prow = 0;
  if (GROUPED) {
    e_lo = s_off[e];
    e_hi = s_off[e + 1];
    e_prow = s_prow[e];
    if (kNv) {
      gs = s_gs[e];
      r6 = __fdiv_rn(gs, 6.0f);
    }
  }
  for (; b < b_end; b += stride) {
    const int64_t bn = b + stride;
    if (bn < b_end) {  // next block in flight while this one is converted
      load32B(x + bn * 64, nxt);
      load32B(x + bn * 64 + 32, nxt + 8);
    }
    if (GROUPED && row >= e_hi && e + 1 < a.E) {  // rows only grow within a thread
      do {
        ++e;
      } while (e + 1 < a.E && row >= s_off[e + 1]);
      e_lo = s_off[e];
      e_hi = s_off[e + 1];
      e_prow = s_prow[e];
      if (kNv) {
        gs = s_gs[e];
        r6 = __fdiv_rn(gs, 6.0f);
      }
    }
    uint32_t byte;
    if constexpr (kNv) {
      byte = nv_block_kernel<QDQ>(cur, static_cast<uint8_t*>(a.out) + b * kCodeBytes, gs, r6);
    } else {
      byte = block_kernel<FMT, QDQ>(cur, true, static_cast<uint8_t*>(a.out) + b * kCodeBytes);
    }
    if (!QDQ) {
      // scale position: linear = flat block order; swizzled = the row's (padded) tile row.
      // NVFP4: two scale bytes, blocks 2 * col and 2 * col + 1, adjacent in both layouts.
      int64_t pr = row;
      bool ok = true;
      if (GROUPED && SWZ) {
        pr = e_prow + (row - e_lo);
        ok = row >= e_lo && row < e_hi && pr < a.scale_rows;
      }
      if (kNv) {
        const int64_t off = SWZ ? swizzled_offset(pr, 2 * col, a.scale_cols) : 2 * b;
        if (ok) *reinterpret_cast<uint16_t*>(a.scales + off) = (uint16_t)byte;
      } else {
        const int64_t off = SWZ ? swizzled_offset(pr, col, a.scale_cols) : b;
        if (ok) a.scales[off] = (uint8_t)byte;
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

  if (SWZ && !QDQ && GROUPED) zero_grouped_pads<kNv>(a, s_off, s_prow, cblk);
  if (SWZ && !QDQ && !GROUPED) {  // grouped calls write their pad bytes with zero_grouped_pads
    zero_swizzled_pads(a.scales, a.M, kNv ? 2 * cblk : cblk, a.scale_rows, a.scale_cols,
                       (int64_t)blockIdx.x * kThreads + tid, (int64_t)gridDim.x * kThreads);
  }
}

// Grouped MX quantize with swizzled scales, walked like the plain kernel (grid stride). Codes and
// scale bytes of MX formats do not depend on the expert; only the padded scale row does:
// pr = row + shift(row), shift = (first padded row of the row's expert) - (its first row). The
// rows a CTA visits follow from its block indices alone (iteration i covers the rows of blocks
// f0 + i * stride .. + 255, at most kThreads / (K/32) + 2 of them), so once the expert offsets
// are in shared memory the CTA resolves all its rows' shifts into a table, one search per row,
// spread over its threads. The offsets are copied asynchronously during the first iteration, whose
// scale byte waits in a register until the table is built. The host takes this kernel when the
// table fits (kRowTable entries) and the contiguous-range kernel otherwise.
constexpr int kRowTable = 2048;
constexpr int64_t kNoRow = INT64_MIN;  // a row outside every expert: its scale byte is not written

__device__ __forceinline__ void cp_async_8(void* smem_dst, const void* gmem_src) {
  const uint32_t d = static_cast<uint32_t>(__cvta_generic_to_shared(smem_dst));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(d), "l"(gmem_src) : "memory");
}

template <int FMT>
__global__ void __launch_bounds__(kThreads, stream_min_ctas<FMT, false, true>())
    mx_grouped_table_kernel(StreamArgs a) {
  __shared__ int64_t s_raw[kMaxExperts + 1];   // the offsets as given
  __shared__ int64_t s_off[kMaxExperts + 1];   // clamped first row of expert e
  __shared__ int64_t s_prow[kMaxExperts + 1];  // first padded scale row of e
  __shared__ int64_t s_warp[kThreads / 32];
  __shared__ int64_t s_shift[kRowTable];       // shift of row (f_i / cblk + k) at i * rpi + k
  constexpr int kCodeBytes = FMT == kFmtE4M3 ? 32 : 16;
  const int tid = threadIdx.x;
  // the host takes this kernel only when every block index fits in 31 bits
  const int cblk = (int)(a.K >> 5);
  const int nblk = (int)(a.M * cblk);
  const int stride = (int)gridDim.x * kThreads;
  const int f0 = (int)blockIdx.x * kThreads;  // the CTA's first block
  pdl_launch_dependents();
  // L2 prefetch (a hint) of this warp's span in iterations d0 .. d1 of the walk
  auto prefetch_spans = [&](int d0, int d1) {
    if ((tid & 31) != 0) return;
    for (int d = d0; d <= d1; ++d) {
      const int64_t s0 = (int64_t)f0 + (tid & ~31) + (int64_t)d * stride;
      if (s0 < nblk) {
        const int64_t n = nblk - s0 < 32 ? nblk - s0 : 32;
        prefetch_l2(static_cast<const uint8_t*>(a.x) + s0 * 64, (uint32_t)(n * 64));
      }
    }
  };
  prefetch_spans(0, 0);
  pdl_wait();
  for (int e = tid; e <= a.E; e += kThreads) cp_async_8(&s_raw[e], a.offsets + e);
  asm volatile("cp.async.commit_group;" ::: "memory");

  const uint8_t* x = static_cast<const uint8_t*>(a.x);
  uint8_t* out = static_cast<uint8_t*>(a.out);
  const int row_step = stride / cblk, col_step = stride - row_step * cblk;
  int b = f0 + tid;
  int row = b / cblk, col = b - row * cblk;  // this thread's block, advanced incrementally
  int fcol = f0 - (f0 / cblk) * cblk;        // column of the CTA's first block of the iteration
  int k = row - f0 / cblk;                   // row - the row of that block: the table column
  const int rpi = kThreads / cblk + 2;       // table entries per iteration
  uint32_t cur[16], nxt[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) nxt[i] = 0u;

  // iteration 0: codes now, the scale byte once the table is built
  const bool have0 = b < nblk;
  uint32_t byte0 = 0;
  if (have0) {
    load32B(x + (int64_t)b * 64, cur);
    load32B(x + (int64_t)b * 64 + 32, cur + 8);
    if (b + stride < nblk) {
      load32B(x + ((int64_t)b + stride) * 64, nxt);
      load32B(x + ((int64_t)b + stride) * 64 + 32, nxt + 8);
    }
    byte0 = block_kernel<FMT, false>(cur, true, out + (int64_t)b * kCodeBytes);
  }

  // The prologue below stops every warp for a while with one block of loads in flight; the
  // spans of iterations 2 and 3 go to L2 meanwhile (x[16384, 2048], 128 experts: 18.5 -> 17.4
  // us back to back; iterations 2 .. 4: 17.7).
  prefetch_spans(2, 3);
  // expert tables: clamped offsets, padded first rows (prefix sum of ceil(n_e / 128) * 128)
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  {
    int64_t nb[4];
    int64_t local = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = tid * 4 + j;
      nb[j] = 0;
      if (e < a.E) {
        int64_t lo = s_raw[e], hi = s_raw[e + 1];
        lo = lo < 0 ? 0 : (lo > a.M ? a.M : lo);
        hi = hi < lo ? lo : (hi > a.M ? a.M : hi);
        s_off[e] = lo;
        nb[j] = (hi - lo + kTileRows - 1) / kTileRows * kTileRows;
        local += nb[j];
      }
    }
    if (tid == 0) {
      const int64_t end = s_raw[a.E];
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
    int64_t run = incl - local;
    for (int w = 0; w < (tid >> 5); ++w) run += s_warp[w];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int e = tid * 4 + j;
      if (e < a.E) s_prow[e] = run;
      run += nb[j];
    }
    if (tid == kThreads - 1) s_prow[a.E] = run;
    __syncthreads();
  }
  // the row table of this CTA's iterations
  {
    const int iters = f0 < nblk ? (nblk - f0 + stride - 1) / stride : 0;
    const int entries = iters * rpi;
    for (int t = tid; t < entries; t += kThreads) {
      const int it = t / rpi;
      const int64_t r = (int64_t)((f0 + (int64_t)it * stride) / cblk) + (t - it * rpi);
      int64_t shift = kNoRow;
      if (r < a.M) {
        const int e = last_not_above(s_off, a.E, r);
        if (r >= s_off[e] && r < s_off[e + 1]) shift = s_prow[e] - s_off[e];
      }
      s_shift[t] = shift;
    }
    __syncthreads();
  }

  const int64_t* shift_row = s_shift;  // the table's row of the current iteration
  if (have0) {
    const int64_t shift = shift_row[k];
    const int64_t pr = row + shift;
    if (shift != kNoRow && pr >= 0 && pr < a.scale_rows) {
      a.scales[swizzled_offset(pr, col, a.scale_cols)] = (uint8_t)byte0;
    }
  }
  for (b += stride; b < nblk; b += stride) {
    // advance to this iteration: the thread's block and the CTA's first block move by stride
    col += col_step;
    row += row_step;
    fcol += col_step;
    if (col >= cblk) {
      col -= cblk;
      ++row;
      ++k;
    }
    if (fcol >= cblk) {
      fcol -= cblk;
      --k;
    }
    shift_row += rpi;
#pragma unroll
    for (int i = 0; i < 16; ++i) cur[i] = nxt[i];
    const int bn = b + stride;
    if (bn < nblk) {
      load32B(x + (int64_t)bn * 64, nxt);
      load32B(x + (int64_t)bn * 64 + 32, nxt + 8);
    }
    const uint32_t byte = block_kernel<FMT, false>(cur, true, out + (int64_t)b * kCodeBytes);
    const int64_t shift = shift_row[k];
    const int64_t pr = row + shift;
    if (shift != kNoRow && pr >= 0 && pr < a.scale_rows) {
      a.scales[swizzled_offset(pr, col, a.scale_cols)] = (uint8_t)byte;
    }
  }
  zero_grouped_pads<false>(a, s_off, s_prow, a.K >> 5);
}

// Table entries the grouped-table kernel needs per CTA with `grid` CTAs (its largest CTA).
inline int64_t row_table_entries(const StreamArgs& a, int64_t grid) {
  const int64_t cblk = a.K >> 5, nblk = a.M * cblk, stride = grid * kThreads;
  return (nblk + stride - 1) / stride * (kThreads / cblk + 2);
}

template <int FMT, bool QDQ, bool SWZ, bool GROUPED>
cudaError_t launch_t(const StreamArgs& a, cudaStream_t stream) {
  const void* k = reinterpret_cast<const void*>(&mx_stream_kernel<FMT, QDQ, SWZ, GROUPED>);
  const int64_t nblk = a.M * (a.K >> 5);
  int64_t need = (nblk + kThreads - 1) / kThreads;
  if (SWZ && !QDQ) {  // enough threads for the pad items as well (see the kernel's pad pass)
    const int64_t cp4 = a.scale_cols / 4;
    const int64_t items = GROUPED ? a.scale_rows : (a.scale_rows - a.M) * cp4;
    const int64_t pad_need = (items + kThreads - 1) / kThreads;
    if (pad_need > need) need = pad_need;
  }
  if (need <= 0) return cudaSuccess;
  if constexpr (GROUPED && SWZ && !QDQ && FMT != kFmtNVFP4) {
    const void* kt = reinterpret_cast<const void*>(&mx_grouped_table_kernel<FMT>);
    const int resident_t = resident_ctas(kt, kThreads, 0, 0);
    if (resident_t <= 0) return cudaErrorInvalidConfiguration;
    const int grid_t = (int)(need < resident_t ? need : resident_t);
    const int64_t nblk = a.M * (a.K >> 5);
    if (row_table_entries(a, grid_t) <= kRowTable &&
        nblk + (int64_t)grid_t * kThreads < ((int64_t)1 << 31)) {
      return launch_pdl(&mx_grouped_table_kernel<FMT>, dim3(grid_t), dim3(kThreads), 0, stream, a);
    }
  }
  const int resident = resident_ctas(k, kThreads, 0, 0);
  if (resident <= 0) return cudaErrorInvalidConfiguration;
  const int grid = (int)(need < resident ? need : resident);
  return launch_pdl(&mx_stream_kernel<FMT, QDQ, SWZ, GROUPED>, dim3(grid), dim3(kThreads), 0,
                    stream, a);
}

template <int FMT>
cudaError_t launch_fmt(bool qdq, bool swz, bool grouped, const StreamArgs& a, cudaStream_t st) {
  if (qdq) return launch_t<FMT, true, false, false>(a, st);
  if (grouped) {
    if constexpr (FMT == kFmtE2M1Quest) {
      return cudaErrorInvalidValue;  // no grouped variant of the Quest-like scale
    } else if constexpr (FMT == kFmtNVFP4) {
      return swz ? launch_t<FMT, false, true, true>(a, st) : launch_t<FMT, false, false, true>(a, st);
    } else {  // MX grouped calls with linear scales run as plain calls (mx_api.cu)
      return swz ? launch_t<FMT, false, true, true>(a, st) : cudaErrorInvalidValue;
    }
  }
  return swz ? launch_t<FMT, false, true, false>(a, st) : launch_t<FMT, false, false, false>(a, st);
}

}  // namespace

cudaError_t launch_stream(int fmt, bool qdq, bool swizzled, bool grouped, const StreamArgs& a,
                          cudaStream_t stream) {
  if (fmt == kFmtE2M1) return launch_fmt<kFmtE2M1>(qdq, swizzled, grouped, a, stream);
  if (fmt == kFmtE2M1Quest) return launch_fmt<kFmtE2M1Quest>(qdq, swizzled, grouped, a, stream);
  if (fmt == kFmtNVFP4) return launch_fmt<kFmtNVFP4>(qdq, swizzled, grouped, a, stream);
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
