// mx_gemm.cu -- block-scaled GEMM consumer of the library's MX codes and scales on the
// 5th-generation tensor cores:
//   C[M, N] = alpha * dequant(A)[M, K] * dequant(B)[N, K]^T   (bf16 out, fp32 accumulation),
// A and B given as MX codes (E2M1 packed two per byte, or E4M3) with their E8M0 block scales in
// the linear or the 128x4 blocked layout, as mx_quantize writes them. This is the consumer the
// QuTLASS pull request tests its quantizer against (review thread on the MXFP4 test:
// matmul_mxf4_bf16_tn(a_e2m1, b_e2m1, a_e8m0, b_e8m0, alpha) compared with the matmul of the
// dequantized operands).
//
// Each CTA computes one 128 x 256 tile of C, K in steps of 64 (warp numbers for the default of
// one converter thread per row, MX_GEMM_SPLIT 1; with 2, two threads share a row, one block
// each, and there are twice as many converter warps):
//   warp 12      one thread loads the raw codes with the tensor-memory accelerator, 128 code
//                bytes of each of A's 128 and B's 256 rows per stage (4 steps of E2M1, 2 of
//                E4M3: one full line per row), 128-byte swizzled so that threads reading their
//                own rows hit distinct banks, into a ring of two stages;
//   warps 0..3   A converters, one thread per row of A (warp w: rows 32 w .. +31): the step's 64
//                codes and two scale bytes -> 64 values decode(code) * 2^(byte - 127) (rounded
//                once to bf16; exact for every E2M1 code and for E4M3 unless below the bf16
//                range), written straight into tensor memory (tcgen05.st; row i in lane i, two
//                values per column), the form in which the MMA reads its A operand;
//   warps 4..11  B converters, one thread per row of B: the same values written to shared
//                memory as 256 rows x 128 bytes, K-major, 128-byte swizzled (16-byte chunk c of
//                row r at chunk c ^ (r % 8)), the layout a shared-memory descriptor reads;
//   warp 13      allocates the tensor memory (accumulator: 256 fp32 columns; A: four stages of
//                32 columns) and, from one lane, issues per step four tcgen05.mma kind::f16
//                (M = 128, N = 256, K = 16, A from tensor memory, B from shared memory,
//                f16 or bf16 products summed in fp32) and commits them to the step's "empty"
//                barrier;
//   warps 0..7   epilogue: tcgen05.ld of the accumulator (warp w: rows 32 (w % 4) .. +31,
//                columns 128 (w / 4) .. +127), times alpha, rounded to bf16, staged in shared
//                memory and written with tensor-map stores.
// Operand type. When every scale byte of the CTA's rows lies in the window where every value
// decode(code) * 2^X (X = byte - 127) is exact in f16 (E2M1: X in [-23, 13]; E4M3: [-15, 7]),
// the operands are f16: two codes take one hardware conversion to f16x2 (exact) and one f16x2
// multiply by 2^X (exact). Otherwise they are bf16: the f16 patterns are moved to bf16 position
// (the values times 2^-112, still exact), then one bf16x2 multiply by 2^(X + 112) (rounded
// once) and a second one only when X > 15 (2^(X + 112) is then beyond the bf16 range). In the
// window both give the same operand values, so the choice changes no product. The converters
// check the window over the CTA's scale bytes before the first step (one CTA-wide vote).
// Scale bytes are read by each converter from global memory two steps ahead.
// Every mbarrier wait is bounded (pipeline waits by GemmArgs::wait_limit_ns, 2 s unless a
// self-test sets it shorter): a wait that runs out sets the device error word and its role
// stops issuing work; the loads in flight and the MMAs issued are waited for (always with the
// 2 s limit) before the CTA frees its tensor memory and exits.
#include "mx_device.cuh"
#include "mx_launch.h"
#include "mx_tcgen05.cuh"

namespace mxq {

namespace {

using namespace tc;

constexpr int kBM = 128, kBK = 64;
constexpr int kRawStages = 2;   // raw code stages (tensor-memory-accelerator ring)
constexpr int kOpStages = 4;    // operand stages (A in tensor memory, B in shared memory)
// Converter threads per row of wide tiles (each taking 2 / split of the step's two 32-element
// blocks); narrow tiles always use two (their CTAs are few, so more warps per CTA pay).
#ifndef MX_GEMM_SPLIT
#define MX_GEMM_SPLIT 1
#endif
constexpr uint32_t kAStageCols = kBK / 2;     // bf16 pairs of a 64-wide K step

// Everything that depends on the tile's width BN (columns of C, rows of B): 256 for large
// problems, 64 when 128 x 256 tiles would not fill the SMs (two CTAs per SM then).
template <int BN>
struct Tile {
  static constexpr int kSplit = BN <= 64 ? 2 : MX_GEMM_SPLIT;  // converter threads per row
  static constexpr int kBlocksPerThread = 2 / kSplit;
  static constexpr int kAWarps = 4 * kSplit;
  static constexpr int kBRowWarps = BN / 32;  // warps covering B's rows once
  static constexpr int kBWarps = kBRowWarps * kSplit, kConvWarps = kAWarps + kBWarps;
  static constexpr int kTmaWarp = kConvWarps, kMmaWarp = kConvWarps + 1;
  static constexpr int kThreads = (kConvWarps + 2) * 32;
  // epilogue: 4 lane quarters x column slices of the accumulator, one converter warp each
  static constexpr int kEpiWarps = kConvWarps >= 16 ? 16 : (kConvWarps >= 8 && BN >= 128 ? 8 : 4);
  static constexpr int kEpiCols = BN / (kEpiWarps / 4);
  static constexpr uint32_t kAccCols = BN;  // fp32 accumulator columns
  static constexpr uint32_t kTmemCols = BN + kOpStages * kAStageCols <= 256 ? 256 : 512;
  static constexpr int kBOpBytes = BN * kBK * 2;  // bf16 of one B stage (32 or 8 KiB)
  static constexpr int kMinCtas = 1;
  static_assert(kEpiWarps <= kConvWarps, "the epilogue runs on converter warps");
  static_assert(kEpiCols % 32 == 0, "32-column accumulator loads");
  static_assert((BN / 64) * kBM * 128 <= kOpStages * kBOpBytes, "C staging fits the B stages");
};
constexpr unsigned long long kGemmWaitNs = 2000000000ull;  // 2 s

// A raw stage holds 128 code bytes of each row (kSteps K steps: 4 of E2M1, 2 of E4M3), so that
// every row of a box is one full 128-byte line; rows 128-byte swizzled (16-byte chunk q of row
// r at q ^ (r % 8)).
template <int FMT, int BN>
struct RawLayout {
  static constexpr int kRowBytes = FMT == kFmtE2M1 ? 32 : 64;  // code bytes of a row per step
  static constexpr int kPitch = 128;                           // code bytes of a row per stage
  static constexpr int kSteps = kPitch / kRowBytes;
  static constexpr int kABytes = kBM * kPitch;
  static constexpr int kStageBytes = (kBM + BN) * kPitch;      // 48 or 24 KiB
};

template <int FMT, int BN>
constexpr int gemm_smem() {
  return 1024 + kOpStages * Tile<BN>::kBOpBytes + kRawStages * RawLayout<FMT, BN>::kStageBytes +
         (2 * kRawStages + 2 * kOpStages + 1) * 8 + 16;  // + tmem slot, vote
}

__device__ __forceinline__ uint32_t hmul2_bf16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// f16x2 pattern of two code values (exact: each normal or zero with the low 7 mantissa bits
// zero) -> bf16x2 pattern of the same values times 2^-112: exponent and top mantissa bits move
// down three places into bf16 position, the signs stay.
__device__ __forceinline__ uint32_t f16x2_to_bf16x2_lowered(uint32_t h) {
  return ((h >> 3) & 0x0FFF0FFFu) | (h & 0x80008000u);
}

// Per 32-element block with scale byte sb: f1 = 2^(min(X, 15) + 112) in both bf16 halves and,
// when X > 15, f2 = 2^(X - 15) (bf16 NaN for the E8M0 NaN byte 0xFF), X = sb - 127.
struct BlockFactors {
  uint32_t f1, f2;
  bool big;
};
__device__ __forceinline__ BlockFactors block_factors(uint32_t sb) {
  BlockFactors f;
  f.f1 = ((min(sb, 142u) + 112u) << 7) * 0x00010001u;
  f.big = sb > 142u;
  f.f2 = sb == 255u ? kBf16NaNx2 : ((sb - 15u) << 7) * 0x00010001u;
  return f;
}

// One block of a row (32 codes, raw[]: E2M1 4 words, E4M3 8 words, lower K first) under the
// scale byte sb -> 16 bf16x2 words, lower K in the low half.
template <int FMT>
__device__ __forceinline__ void convert_block(const uint32_t* raw, uint32_t sb, uint32_t* out) {
  const BlockFactors b = block_factors(sb);
  if (FMT == kFmtE2M1) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        uint32_t h;
        asm("{\n\t.reg .b8 c;\n\tcvt.u8.u32 c, %1;\n\tcvt.rn.f16x2.e2m1x2 %0, c;\n\t}"
            : "=r"(h)
            : "r"(raw[j] >> (8 * t)));
        out[4 * j + t] = hmul2_bf16(f16x2_to_bf16x2_lowered(h), b.f1);
      }
    }
  } else {
    uint32_t nan = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t w = raw[j];
      nan |= (w & 0x7F7F7F7Fu) + 0x01010101u;  // a byte reaches 0x80 iff it is S.1111.111
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        uint32_t h;
        asm("{\n\t.reg .b16 c;\n\tcvt.u16.u32 c, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, c;\n\t}"
            : "=r"(h)
            : "r"(w >> (16 * t)));
        out[2 * j + t] = hmul2_bf16(f16x2_to_bf16x2_lowered(h), b.f1);
      }
    }
    if (nan & 0x80808080u) {  // E4M3 NaN codes: their values are the bf16 NaN
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t n = ((raw[j] & 0x7F7F7F7Fu) + 0x01010101u) & 0x80808080u;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const uint32_t lo = (n >> (16 * t + 7)) & 1u, hi = (n >> (16 * t + 15)) & 1u;
          uint32_t v = out[2 * j + t];
          if (lo) v = (v & 0xFFFF0000u) | 0x7FC0u;
          if (hi) v = (v & 0x0000FFFFu) | 0x7FC00000u;
          out[2 * j + t] = v;
        }
      }
    }
  }
  if (b.big) {
#pragma unroll
    for (int i = 0; i < 16; ++i) out[i] = hmul2_bf16(out[i], b.f2);
  }
}

// Scale-byte window in which every value decode(code) * 2^(byte - 127) is exact in f16.
template <int FMT>
struct F16Window {
  static constexpr uint32_t kLo = FMT == kFmtE2M1 ? 104u : 112u;  // X >= -23 / -15
  static constexpr uint32_t kHi = FMT == kFmtE2M1 ? 140u : 134u;  // X <= 13 / 7
};

__device__ __forceinline__ uint32_t hmul2_f16(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// 2^(sb - 127) as f16 in both halves, sb inside the window (2^-23 .. 2^-15 are subnormal).
__device__ __forceinline__ uint32_t f16_pow2x2(uint32_t sb) {
  const int x = (int)sb - 127;
  const uint32_t h = x >= -14 ? (uint32_t)(x + 15) << 10 : 1u << (x + 24);
  return h * 0x00010001u;
}

// The f16 form of convert_block, scale byte inside the window: values exact.
template <int FMT>
__device__ __forceinline__ void convert_block_f16(const uint32_t* raw, uint32_t sb, uint32_t* out) {
  const uint32_t m = f16_pow2x2(sb);
  if (FMT == kFmtE2M1) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      uint32_t h[4];
      asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\tmov.b32 {c0, c1, c2, c3}, %4;\n\t"
          "cvt.rn.f16x2.e2m1x2 %0, c0;\n\tcvt.rn.f16x2.e2m1x2 %1, c1;\n\t"
          "cvt.rn.f16x2.e2m1x2 %2, c2;\n\tcvt.rn.f16x2.e2m1x2 %3, c3;\n\t}"
          : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
          : "r"(raw[j]));
#pragma unroll
      for (int t = 0; t < 4; ++t) out[4 * j + t] = hmul2_f16(h[t], m);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t h[2];
      asm("{\n\t.reg .b16 c0, c1;\n\tmov.b32 {c0, c1}, %2;\n\t"
          "cvt.rn.f16x2.e4m3x2 %0, c0;\n\tcvt.rn.f16x2.e4m3x2 %1, c1;\n\t}"
          : "=r"(h[0]), "=r"(h[1])
          : "r"(raw[j]));
      out[2 * j] = hmul2_f16(h[0], m);
      out[2 * j + 1] = hmul2_f16(h[1], m);
    }
  }
}

// Whether any byte of w lies outside [lo, hi] (lo <= 128, hi >= 127): a byte b < lo borrows
// into its top bit in w - lo * 0x01010101 while its own top bit is clear ("has a byte less
// than n", exact for n <= 128 as an existence test), and b > hi is 255 - b < 255 - hi, the
// same test on ~w. Bytes of rows or blocks that do not exist are passed as lo.
struct ByteWindow {
  uint32_t lo_n, hi_n, bad = 0u;
  __device__ __forceinline__ ByteWindow(uint32_t lo, uint32_t hi)
      : lo_n(lo * 0x01010101u), hi_n((255u - hi) * 0x01010101u) {}
  __device__ __forceinline__ void add(uint32_t w) {
    bad |= ((w - lo_n) & ~w) | ((~w - hi_n) & w);
  }
  __device__ __forceinline__ bool inside() const { return (bad & 0x80808080u) == 0u; }
};

__device__ __forceinline__ uint32_t load_scale_pair(const uint8_t* p) {
  uint16_t v;
  asm volatile("ld.global.u16 %0, [%1];" : "=h"(v) : "l"(p));
  return v;
}

// Shared-memory carve-up and per-CTA constants of one GEMM CTA.
template <int FMT>
struct GemmCta {
  uint8_t* bop;       // kOpStages x Tile::kBOpBytes: B operand stages
  uint8_t* raw;       // kRawStages x RawLayout::kStageBytes: raw code stages
  uint64_t* raw_full;
  uint64_t* raw_empty;
  uint64_t* op_full;
  uint64_t* op_empty;
  uint64_t* acc_full;
  uint32_t tmem;
  int64_t m0, n0;
  int nk;
};

__device__ __forceinline__ uint4 load_scale_chunk(const uint8_t* p) {  // 16-byte aligned
  uint4 v;
  asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Whether every scale byte of this converter's share of the CTA's rows (A: one block of 128
// rows; B: the one or two blocks its rows lie in) lies inside [lo, hi]. Swizzled: the nthreads
// threads of a row block share its contiguous tiles (t: the thread's index within the block,
// row0 its first row); linear: thread (row, part 0) takes the row (grow), the others nothing. Rows past M / N, and the padding columns of
// the swizzled layout, are not looked at.
template <bool SWZ>
__device__ __forceinline__ bool scales_inside(const GemmArgs& a, bool is_a, int t, int nthreads,
                                              int64_t row0, int64_t grow, int part, uint32_t lo,
                                              uint32_t hi) {
  ByteWindow br(lo, hi);
  const uint8_t* sc = is_a ? a.a_scales : a.b_scales;
  const int64_t scols = is_a ? a.a_scale_cols : a.b_scale_cols;
  const int64_t rows = is_a ? a.M : a.N;
  const uint32_t fill = lo * 0x01010101u;
  if (SWZ) {
    // the 128-row block's 512-byte tiles are contiguous: chunk i (16 bytes) of the block holds
    // rows q, q + 32, q + 64, q + 96 (q = i % 32) of tile i / 32, 4 blocks each
    const int u = t;
    if (row0 < rows) {
      const int64_t ctiles = scols >> 2;
      const int kb_last = (int)((a.K / 32) & 3);  // 2 when the last tile holds 2 pad columns
      const uint8_t* base = sc + (row0 >> 7) * ctiles * 512;
#pragma unroll 8
      for (int64_t i = u; i < ctiles * 32; i += nthreads) {
        const uint4 v = load_scale_chunk(base + i * 16);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        const bool last = i / 32 == ctiles - 1 && kb_last != 0;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          uint32_t x = row0 + (i & 31) + 32 * g < rows ? w[g] : fill;
          if (last) x = (x & 0x0000FFFFu) | (fill & 0xFFFF0000u);
          br.add(x);
        }
      }
    }
  } else if (grow < rows && part == 0) {
    const uint8_t* p = sc + grow * scols;
    if ((scols & 15) == 0 && (reinterpret_cast<uintptr_t>(p) & 15) == 0) {
#pragma unroll 8
      for (int64_t i = 0; i < scols; i += 16) {
        const uint4 v = load_scale_chunk(p + i);
        br.add(v.x);
        br.add(v.y);
        br.add(v.z);
        br.add(v.w);
      }
    } else {
      for (int64_t i = 0; i < scols; i += 2) br.add(load_scale_pair(p + i) * 0x00010001u);
    }
  }
  return br.inside();
}

// Raw code loads (one thread of warp kTmaWarp): runs from the start, independent of the operand
// type, so that the first stages are in flight while the converters vote.
template <int FMT, int BN>
__device__ __forceinline__ void gemm_loads(const CUtensorMap& amap, const CUtensorMap& bmap,
                                           const GemmArgs& a, const GemmCta<FMT>& c) {
  using R = RawLayout<FMT, BN>;
  const int nk = c.nk;
  bool failed = false;
  const int nstages = (nk + R::kSteps - 1) / R::kSteps;
  int issued = 0;
  for (int rs = 0; rs < nstages; ++rs) {
    const int s = rs % kRawStages;
    if (rs >= kRawStages) {
      mbar_wait(smem_u32(c.raw_empty + s), ((rs / kRawStages) & 1) ^ 1, &failed,
                a.wait_limit_ns, a.err);
    }
    if (failed) break;
    const uint32_t dst = smem_u32(c.raw + s * R::kStageBytes);
    mbar_arrive_expect_tx(smem_u32(c.raw_full + s), R::kStageBytes);
    tma_load_box(dst, &amap, rs * R::kPitch, (int)c.m0, smem_u32(c.raw_full + s));
    tma_load_box(dst + R::kABytes, &bmap, rs * R::kPitch, (int)c.n0, smem_u32(c.raw_full + s));
    issued = rs + 1;
  }
  // loads still in flight land before the CTA's shared memory goes away
  bool drain_failed = false;
  for (int rs = issued > kRawStages ? issued - kRawStages : 0; rs < issued; ++rs) {
    mbar_wait(smem_u32(c.raw_full + rs % kRawStages), (rs / kRawStages) & 1, &drain_failed,
              kGemmWaitNs, a.err);
  }
}

template <int FMT, bool SWZ, bool F16, int BN>
__device__ __forceinline__ void gemm_roles(const CUtensorMap& cmap, const GemmArgs& a,
                                           const GemmCta<FMT>& c) {
  using R = RawLayout<FMT, BN>;
  using T = Tile<BN>;
  constexpr int kSplit = T::kSplit, kBlocksPerThread = T::kBlocksPerThread, kAWarps = T::kAWarps;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t tmem = c.tmem;
  const int nk = c.nk;
  bool failed = false;

  if (warp < T::kConvWarps) {
    // ---------------- converters: blocks part * kBlocksPerThread .. of row r ----------------
    const bool is_a = warp < kAWarps;
    const int wq = is_a ? warp : warp - kAWarps;
    const int row_warps = is_a ? 4 : T::kBRowWarps;
    const int r = (wq % row_warps) * 32 + lane;  // A: lane quarter = warp % 4
    const int part = wq / row_warps;
    const int64_t grow = (is_a ? c.m0 : c.n0) + r;
    const bool valid = grow < (is_a ? a.M : a.N);
    // narrow tiles (small M): a warp whose rows all lie past M (N) converts nothing; the MMA
    // then reads stale operand rows, which only reach rows (columns) of C that are not stored.
    // Wide tiles convert every row (the test costs them registers and 7 %).
    const bool live = BN > 64 || grow - lane < (is_a ? a.M : a.N);
    const uint8_t* sc = is_a ? a.a_scales : a.b_scales;
    const int64_t scols = is_a ? a.a_scale_cols : a.b_scale_cols;
    // scale bytes of blocks 2 kk + part * kBlocksPerThread ..: linear row-major, or bytes
    // (2 kk + ..) % 4 of the row's 4-byte slot in the 512-byte tile holding blocks 4t .. 4t + 3
    // (t = kk / 2)
    const uint8_t* sbase =
        SWZ ? sc + ((grow >> 7) * (scols >> 2)) * 512 + (grow & 31) * 16 + ((grow >> 5) & 3) * 4 +
                  part * kBlocksPerThread
            : sc + grow * scols + part * kBlocksPerThread;
    auto scale_at = [&](int kk) -> uint32_t {
      if (!valid || kk >= nk) return kBlocksPerThread == 2 ? 0x7F7Fu : 0x7Fu;
      const uint8_t* p = SWZ ? sbase + (int64_t)(kk >> 1) * 512 + (kk & 1) * 2
                             : sbase + 2 * (int64_t)kk;
      return kBlocksPerThread == 2 ? load_scale_pair(p) : load_u8(p);
    };
    constexpr int kPartBytes = R::kRowBytes / kSplit;  // code bytes this thread converts
    constexpr int kBlockWords = R::kRowBytes / 8;      // 32-bit words of codes of one block
    const uint32_t raw_row = (is_a ? 0u : (uint32_t)R::kABytes) + (uint32_t)r * R::kPitch;
    // one step; returns false once a wait has run out (warp-uniform)
    auto step = [&](int kk, uint32_t sb) -> bool {
      const int rs = kk / R::kSteps, sub = kk % R::kSteps;  // raw stage, step within it
      const int sr = rs % kRawStages, so = kk % kOpStages;
      if (sub == 0) {
        mbar_wait(smem_u32(c.raw_full + sr), (rs / kRawStages) & 1, &failed, a.wait_limit_ns,
                  a.err);
        failed = __any_sync(0xFFFFFFFFu, failed);
        if (failed) return false;
      }
      uint32_t out[16 * kBlocksPerThread];
      if (live) {
        uint32_t w[kPartBytes / 4];
        const uint8_t* row = c.raw + sr * R::kStageBytes + raw_row;
#pragma unroll
        for (int j = 0; j < kPartBytes / 16; ++j) {
          const int q = sub * (R::kRowBytes / 16) + part * (kPartBytes / 16) + j;
          const uint4 v = *reinterpret_cast<const uint4*>(row + ((q ^ (r & 7)) * 16));  // 128-B swizzle
          w[4 * j] = v.x;
          w[4 * j + 1] = v.y;
          w[4 * j + 2] = v.z;
          w[4 * j + 3] = v.w;
        }
#pragma unroll
        for (int i = 0; i < kBlocksPerThread; ++i) {
          const uint32_t b = (sb >> (8 * i)) & 0xFFu;
          if (F16) {
            convert_block_f16<FMT>(w + i * kBlockWords, b, out + 16 * i);
          } else {
            convert_block<FMT>(w + i * kBlockWords, b, out + 16 * i);
          }
        }
      }
      if (sub == R::kSteps - 1 || kk == nk - 1) {  // the stage's raw bytes are consumed
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(c.raw_empty + sr));
      }
      if (kk >= kOpStages) {
        mbar_wait(smem_u32(c.op_empty + so), ((kk / kOpStages) & 1) ^ 1, &failed,
                  a.wait_limit_ns, a.err);
        failed = __any_sync(0xFFFFFFFFu, failed);
        if (failed) return false;
      }
      if (!live) {
        // nothing to store
      } else if (is_a) {
        const uint32_t ta = tmem + ((uint32_t)((warp & 3) * 32) << 16) + T::kAccCols +
                            so * kAStageCols + part * (kAStageCols / kSplit);
        if (kBlocksPerThread == 2) {
          tmem_st32_async(ta, out);
        } else {
          tmem_st16_async(ta, out);
        }
        tmem_wait_st();
        tc_fence_before();
      } else {
        uint8_t* dst = c.bop + so * T::kBOpBytes + r * 128;
#pragma unroll
        for (int j = 0; j < 8 / kSplit; ++j) {
          const int q = part * (8 / kSplit) + j;
          *reinterpret_cast<uint4*>(dst + ((q ^ (r & 7)) << 4)) =
              make_uint4(out[4 * j], out[4 * j + 1], out[4 * j + 2], out[4 * j + 3]);
        }
        fence_proxy_async_smem();  // visible to the tensor cores
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(c.op_full + so));
      return true;
    };
    // two steps per iteration, each with its own scale register, reloaded right after its use
    // for the step two later (no register move waits on a load in flight)
    uint32_t sc0 = scale_at(0), sc1 = scale_at(1);
    for (int kk = 0; kk < nk; kk += 2) {
      if (!step(kk, sc0)) break;
      sc0 = scale_at(kk + 2);
      if (kk + 1 >= nk) break;
      if (!step(kk + 1, sc1)) break;
      sc1 = scale_at(kk + 3);
    }
  } else if (warp == T::kMmaWarp && lane == 0) {
    // ---------------- MMA issuer ----------------
    constexpr uint32_t idesc = F16 ? idesc_f16_f32(kBM, BN) : idesc_bf16_f32(kBM, BN);
    for (int kk = 0; kk < nk; ++kk) {
      const int s = kk % kOpStages;
      mbar_wait(smem_u32(c.op_full + s), (kk / kOpStages) & 1, &failed, a.wait_limit_ns, a.err);
      if (failed) break;
      tc_fence_after();
      const uint32_t b0 = smem_u32(c.bop + s * T::kBOpBytes);
#pragma unroll
      for (int k16 = 0; k16 < kBK / 16; ++k16) {
        mma_bf16_ts(tmem, tmem + T::kAccCols + s * kAStageCols + k16 * 8, desc_sw128(b0 + 32 * k16),
                    idesc, (kk > 0 || k16 > 0) ? 1u : 0u);
      }
      mma_commit(smem_u32(c.op_empty + s));  // stage free once these MMAs have read it
    }
    mma_commit(smem_u32(c.acc_full));  // tracks every MMA issued above
    bool drain_failed = false;         // the MMAs complete before the tensor memory is freed
    mbar_wait(smem_u32(c.acc_full), 0, &drain_failed, kGemmWaitNs, a.err);
  }

  if (warp < T::kEpiWarps) {
    // ---------------- epilogue ----------------
    // The bf16 tile is staged in the (now idle) B operand stages as 64-column boxes of
    // 128 rows x 128 bytes, 128-byte swizzled (16-byte chunk q of row r at q ^ (r % 8)), and
    // written with tensor-map stores, which drop what lies past M and N.
    bool efailed = failed;
    mbar_wait(smem_u32(c.acc_full), 0, &efailed, a.wait_limit_ns, a.err);
    efailed = __any_sync(0xFFFFFFFFu, efailed);
    tc_fence_after();
    const int quarter = warp & 3;
    const uint32_t col0 = (uint32_t)(warp >> 2) * T::kEpiCols;
    const int r = quarter * 32 + lane;  // row of the tile
#pragma unroll 1
    for (int cb = 0; cb < T::kEpiCols / 32; ++cb) {
      if (efailed) break;
      float y[32];
      tmem_ld32(tmem + ((uint32_t)(quarter * 32) << 16) + col0 + cb * 32, y);
      const uint32_t col = col0 + cb * 32;  // first of 32 columns: half of a 64-column box
      uint8_t* box = c.bop + (col / 64) * (kBM * 128) + r * 128;
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          asm("cvt.rn.bf16x2.f32 %0, %1, %2;"
              : "=r"(o[i])
              : "f"(a.alpha * y[g * 8 + 2 * i + 1]), "f"(a.alpha * y[g * 8 + 2 * i]));
        }
        const int q = (int)((col % 64) / 8) + g;
        *reinterpret_cast<uint4*>(box + ((q ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
      }
    }
    fence_proxy_async_smem();  // the staged tile is visible to the tensor-map stores
    asm volatile("bar.sync 2, %0;" ::"n"(T::kEpiWarps * 32) : "memory");
    if (warp == 0 && lane == 0 && !efailed) {
#pragma unroll 1
      for (int bx = 0; bx < BN / 64 && c.n0 + bx * 64 < a.N; ++bx) {  // boxes inside N only
        tma_store_box(&cmap, (int)c.n0 + bx * 64, (int)c.m0,
                      smem_u32(c.bop + bx * (kBM * 128)));
      }
      bulk_commit_group();
      bulk_wait_read_all();  // the staging is read before the CTA's shared memory goes away
    }
  }
}

template <int FMT, bool SWZ, int BN>
__global__ void __launch_bounds__(Tile<BN>::kThreads, Tile<BN>::kMinCtas)
    mx_gemm_kernel(const __grid_constant__ CUtensorMap amap,
                   const __grid_constant__ CUtensorMap bmap,
                   const __grid_constant__ CUtensorMap cmap, GemmArgs a) {
  using R = RawLayout<FMT, BN>;
  using T = Tile<BN>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  GemmCta<FMT> c;
  c.bop = smem;
  c.raw = smem + kOpStages * T::kBOpBytes;
  c.raw_full = reinterpret_cast<uint64_t*>(c.raw + kRawStages * R::kStageBytes);
  c.raw_empty = c.raw_full + kRawStages;
  c.op_full = c.raw_empty + kRawStages;
  c.op_empty = c.op_full + kOpStages;
  c.acc_full = c.op_empty + kOpStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(c.acc_full + 1);
  uint32_t* outside = tmem_slot + 1;  // count of converters with a scale byte outside the window
  const int tid = threadIdx.x, warp = tid >> 5;
  c.m0 = (int64_t)blockIdx.y * kBM;
  c.n0 = (int64_t)blockIdx.x * BN;
  c.nk = (int)(a.K / kBK);

  pdl_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < kRawStages; ++s) {
      mbar_init(smem_u32(c.raw_full + s), 1);
      mbar_init(smem_u32(c.raw_empty + s), T::kConvWarps);
    }
    for (int s = 0; s < kOpStages; ++s) {
      mbar_init(smem_u32(c.op_full + s), T::kConvWarps);
      mbar_init(smem_u32(c.op_empty + s), 1);
    }
    mbar_init(smem_u32(c.acc_full), 1);
    *outside = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  pdl_wait();  // inputs written by the kernel before; its tensor memory freed
  if (warp == T::kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), T::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();  // barriers initialised, tensor memory allocated
  tc_fence_after();
  c.tmem = *tmem_slot;
  if (warp == T::kTmaWarp) {
    if ((tid & 31) == 0) gemm_loads<FMT, BN>(amap, bmap, a, c);
  } else {
    if (warp < T::kConvWarps) {  // f16 window vote over the CTA's scale bytes
      constexpr int kAWarps = T::kAWarps;
      const bool is_a = warp < kAWarps;
      const int wq = is_a ? warp : warp - kAWarps;
      const int row_warps = is_a ? 4 : T::kBRowWarps;
      const int r = (wq % row_warps) * 32 + (tid & 31);
      const int part = wq / row_warps;
      // swizzled: the 128-row blocks holding the CTA's rows (A: one; B: one or two), each
      // shared by nthr threads
      const int nblocks = is_a ? 1 : (BN + 127) / 128;
      const int nthr = (is_a ? kAWarps * 32 : T::kBWarps * 32) / nblocks;
      const int bt = is_a ? tid : tid - kAWarps * 32;
      const int64_t row0 = ((is_a ? c.m0 : c.n0) >> 7 << 7) + (bt / nthr) * 128;
      const bool in = scales_inside<SWZ>(a, is_a, bt % nthr, nthr, row0,
                                         (is_a ? c.m0 : c.n0) + r, part, F16Window<FMT>::kLo,
                                         F16Window<FMT>::kHi);
      if (!__all_sync(0xFFFFFFFFu, in) && (tid & 31) == 0) atomicAdd(outside, 1u);
    }
    // converters and the MMA warp (the load warp is already running)
    asm volatile("bar.sync 1, %0;" ::"n"((T::kConvWarps + 1) * 32) : "memory");
    if (*outside == 0) {
      gemm_roles<FMT, SWZ, true, BN>(cmap, a, c);
    } else {
      gemm_roles<FMT, SWZ, false, BN>(cmap, a, c);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == T::kMmaWarp) tmem_dealloc(c.tmem, T::kTmemCols);
}

template <int FMT, bool SWZ, int BN>
cudaError_t launch_tile(const GemmArgs& a, cudaStream_t stream) {
  using R = RawLayout<FMT, BN>;
  using T = Tile<BN>;
  const void* k = reinterpret_cast<const void*>(&mx_gemm_kernel<FMT, SWZ, BN>);
  constexpr int smem = gemm_smem<FMT, BN>();
  if (resident_ctas(k, T::kThreads, smem, T::kMinCtas) <= 0) return cudaErrorInvalidConfiguration;
  const int64_t code_row = FMT == kFmtE2M1 ? a.K / 2 : a.K;
  const CUtensorMapSwizzle swz = CU_TENSOR_MAP_SWIZZLE_128B;
  CUtensorMap amap, bmap;
  cudaError_t err = make_tensor_map_2d(&amap, a.a_codes, a.M, code_row,
                                       CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, R::kPitch, kBM, swz);
  if (err != cudaSuccess) return err;
  err = make_tensor_map_2d(&bmap, a.b_codes, a.N, code_row, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1,
                           R::kPitch, BN, swz);
  if (err != cudaSuccess) return err;
  CUtensorMap cmap;  // C: bf16 [M, N], boxes of 128 rows x 64 columns
  err = make_tensor_map_2d(&cmap, a.c, a.M, a.N, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, 64, kBM,
                           swz);
  if (err != cudaSuccess) return err;
  const dim3 grid((unsigned)((a.N + BN - 1) / BN), (unsigned)((a.M + kBM - 1) / kBM));
  return launch_pdl(&mx_gemm_kernel<FMT, SWZ, BN>, grid, dim3(T::kThreads), smem, stream, amap,
                    bmap, cmap, a);
}

// 128 x 256 tiles, or 128 x 64 tiles when the 128 x 256 tiles would leave SMs idle and the
// narrow tiles fit in one wave (narrow tiles beyond one wave measured 2x slower at M = 512).
template <int FMT, bool SWZ>
cudaError_t launch_t(const GemmArgs& a, cudaStream_t stream) {
  const void* k = reinterpret_cast<const void*>(&mx_gemm_kernel<FMT, SWZ, 256>);
  const int sms = resident_ctas(k, Tile<256>::kThreads, gemm_smem<FMT, 256>(), 1);
  const void* kn = reinterpret_cast<const void*>(&mx_gemm_kernel<FMT, SWZ, 64>);
  const int narrow_slots = resident_ctas(kn, Tile<64>::kThreads, gemm_smem<FMT, 64>(), 4);
  const int64_t row_tiles = (a.M + kBM - 1) / kBM;
  const int64_t wide_tiles = row_tiles * ((a.N + 255) / 256);
  const int64_t narrow_tiles = row_tiles * ((a.N + 63) / 64);
  if (sms > 0 && wide_tiles < sms && narrow_tiles <= narrow_slots) {
    return launch_tile<FMT, SWZ, 64>(a, stream);
  }
  return launch_tile<FMT, SWZ, 256>(a, stream);
}

}  // namespace

cudaError_t launch_gemm(int fmt, bool swizzled, const GemmArgs& a, cudaStream_t stream) {
  if (fmt == kFmtE2M1) {
    return swizzled ? launch_t<kFmtE2M1, true>(a, stream) : launch_t<kFmtE2M1, false>(a, stream);
  }
  return swizzled ? launch_t<kFmtE4M3, true>(a, stream) : launch_t<kFmtE4M3, false>(a, stream);
}

}  // namespace mxq
