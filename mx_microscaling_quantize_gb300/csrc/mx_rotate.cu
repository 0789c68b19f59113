// mx_rotate.cu -- fused rotate + block quantize on the 5th-generation tensor cores.
//
// The rotation multiplies every g-element chunk along K by a runtime-loaded g x g bf16 matrix
// H (QuTLASS pull request, feature list: "Rotation matrices loaded at runtime, allowing any
// transformation", sizes 16/32/64/128). For a tile of 128 rows x 128 elements that is 128/g
// independent products [128 x g] * [g x g]: tcgen05.mma (kind::f16, bf16 operands, fp32
// accumulation in tensor memory), M = 128, N = g, K = 16 per instruction.
//
// One persistent CTA per SM, warp-specialized:
//   warp 0       TMA producer: two 2-D boxes of 128 rows x 64 elements per tile, 128-byte
//                swizzle, into a ring of kStages shared-memory stages (mbarrier complete_tx);
//   warp 1       allocates 512 TMEM columns (four 128-column fp32 accumulators) and, from one
//                lane, issues the tile's MMAs and commits them to the stage's "empty" barrier
//                and to the accumulator's "full" barrier;
//   warps 2..17  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lanes
//                32*(w%4) .. +31, i.e. tile rows; the four warps of a quarter take one
//                32-column block each), abs-max, E8M0 scale, conversion, stores; then they
//                free the accumulator for the MMA four tiles on. Outputs and scales (both
//                layouts) are staged per tile in shared memory and written back with TMA /
//                bulk stores (linear scales: one store per tile row); NVFP4 factors come from
//                per-CTA tables of all 128 scale bytes.
// Loads, MMAs and the epilogue of different tiles overlap; each CTA prefetches its first two
// tiles into L2 before waiting for the kernel before it on the stream. Operands: A (the x tile) in the
// K-major 128-byte-swizzled layout the TMA writes (8-row groups 1024 bytes apart); B = H^T in
// the K-major no-swizzle core-matrix layout, written once per CTA:
//   element (n, k) = H[k][n] at (k / 8) * (g * 16) + n * 16 + (k % 8) * 2.
// Every mbarrier wait is bounded (2 s); a wait that runs out sets the device error word and
// the thread stops waiting from then on. A role whose wait ran out stops issuing work: the
// producer issues no more loads, the MMA thread no more MMAs, and the epilogue warps (the whole
// warp, since tcgen05.ld is warp-collective) skip their tensor-memory reads and stores while
// still taking part in every epilogue barrier. Before the block deallocates tensor memory and
// exits, the producer waits for its loads still in flight, the MMA thread for its last commit
// and the storing thread for its bulk stores. Calls with very few rows go to a plain FMA kernel
// instead (mx_rotate_small_kernel, below), which is faster at those sizes.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "mx_device.cuh"
#include "mx_launch.h"
#include "mx_tcgen05.cuh"

namespace mxq {

__device__ unsigned int g_device_errors;

namespace {

using namespace tc;

constexpr int kAcc = 4;  // fp32 accumulators in TMEM (128 columns each)
constexpr int kBoxCols = 64;                  // bf16 per 128-byte swizzled row
constexpr int kBoxBytes = kTileRows * 128;    // 16 KiB
constexpr int kStageBytes = 2 * kBoxBytes;    // 128 rows x 128 elements
constexpr int kEpiWarps = 16;
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = (2 + kEpiWarps) * 32;  // producer, MMA, epilogue
constexpr int kTmemCols = 128 * kAcc;             // all 512 columns of the SM
constexpr unsigned long long kWaitLimitNs = 2000000000ull;  // 2 s
// Tiles per CTA prefetched into L2 before pdl_wait (64 KiB per SM). Measured on GB300 (steady,
// back to back, rotate+quantize E2M1 g = 32): 1.0-1.2 us less per launch with 2 tiles
// (x[4096, 8192] 18.1 -> 17.0 us, x[8192, 8192] 30.6 -> 29.6 us); 1, 3 and 4 tiles gained
// less on most shapes, all 6 ring stages nothing (they compete with the previous kernel).
constexpr int kPrefetchTiles = 2;

// Bounded mbarrier wait of this file's kernels: gives up after limit_ns (kWaitLimitNs by
// default), and at once once this thread has given up before (*failed); a give-up sets the
// device error word.
__device__ __forceinline__ void mbar_wait(uint32_t bar, uint32_t parity, bool* failed,
                                          unsigned long long limit_ns = kWaitLimitNs) {
  tc::mbar_wait(bar, parity, failed, limit_ns, &g_device_errors);
}

// L2 policy for data touched once (inputs read once, outputs written once): evict first.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 2-D tensor-map load of one box into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(bar), "l"(l2_evict_first_policy())
      : "memory");
}

// L2 prefetch of one box through the tensor map (a hint that reads no value; see prefetch_l2).
__device__ __forceinline__ void tma_prefetch_2d(const CUtensorMap* map, int x, int y) {
  asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" ::"l"(
                   reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y)
               : "memory");
}
// 2-D tensor-map store of one box from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const CUtensorMap* map, int x, int y, uint32_t src) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%1, %2}], [%3], %4;"
      ::"l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(src), "l"(l2_evict_first_policy())
      : "memory");
}
// shared -> global bulk copy in the current bulk group (16-byte aligned, size % 16 == 0)
__device__ __forceinline__ void bulk_store_s2g(void* dst, uint32_t src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
               "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// all committed bulk store groups but the most recent one have finished reading shared memory
__device__ __forceinline__ void bulk_wait_read_all_but_one() {
  asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory");
}
// all committed bulk stores have completed, their global writes included (the kernel ends
// after this, so a dependent kernel that stops waiting at its pdl_wait sees every output)
__device__ __forceinline__ void bulk_wait_all() {
  asm volatile("cp.async.bulk.wait_group 0;" ::: "memory");
}

// Both 64-column boxes of tile t (128 rows x 128 columns) into one ring stage.
__device__ __forceinline__ void load_tile(const RotArgs& a, const CUtensorMap* map, uint32_t dst,
                                          uint32_t bar, int64_t t) {
  const int64_t rb = t / a.col_tiles, cb = t - rb * a.col_tiles;
  mbar_arrive_expect_tx(bar, kStageBytes);
  tma_load_2d(dst, map, (int)(cb * kTileCols), (int)(rb * kTileRows), bar);
  tma_load_2d(dst + kBoxBytes, map, (int)(cb * kTileCols + kBoxCols), (int)(rb * kTileRows), bar);
}

__device__ __forceinline__ void epilogue_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}

// ------------------------------------------------------------------------------------------
// one 32-element block of rotated values -> its output bytes and scale byte
// ------------------------------------------------------------------------------------------
// Output bytes per block: QDQ 64 (bf16), E4M3 codes 32, E2M1 codes 16.
template <int FMT, int OUT>
__host__ __device__ constexpr int block_out_words() {
  return OUT == kRotQdq ? 16 : (FMT == kFmtE4M3 ? 8 : 4);
}

// NVFP4 (two 16-element blocks per 32 values): returns both E4M3 scale bytes, low byte first.
// The factors gs / decode(scale) and decode(scale) / gs come from per-CTA tables of all 128
// scale bytes (t_enc, t_dq: the same divisions, done once): two IEEE divisions per block in the
// epilogue kept rotate+quantize NVFP4 at 107 us on x[8192, 28672] (g = 16, back to back)
// against 93 us for MXFP4; with the tables it takes 94 us.
template <int OUT>
__device__ __forceinline__ uint32_t nv_block_outputs(float* y, uint32_t* out, float r6,
                                                     const float* t_enc, const float* t_dq) {
  const NvScales n = nv_scales_tab(absmax_f32x16(y), absmax_f32x16(y + 16), r6, t_enc, t_dq);
  const bool special = __any_sync(0xFFFFFFFFu, n.special[0] || n.special[1]);
#pragma unroll
  for (int i = 0; i < 16; ++i) mul2(y[2 * i], y[2 * i + 1], n.enc[i >> 3]);  // y <- y * enc
  if (OUT == kRotQdq) {
#pragma unroll
    for (int i = 0; i < 16; ++i) out[i] = qdq2_e2m1(y[2 * i], y[2 * i + 1], n.dq[i >> 3]);
    if (special) {
#pragma unroll
      for (int i = 0; i < 16; ++i) out[i] = n.special[i >> 3] ? kBf16NaNx2 : out[i];
    }
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = codes8_e2m1(y + 8 * i);
    if (special) {
#pragma unroll
      for (int i = 0; i < 4; ++i) out[i] = n.special[i >> 1] ? 0u : out[i];
    }
  }
  return n.bytes;
}

template <int FMT, int OUT>
__device__ __forceinline__ uint32_t block_outputs(float* y, uint32_t* out) {
  const uint32_t byte = FMT == kFmtE2M1Quest ? quest_byte_f32x32(y)
                                             : scale_byte_from_amax_bits<FMT>(absmax_f32x32(y));
  const bool special = __any_sync(0xFFFFFFFFu, byte == 255u);  // a NaN / Inf block in the warp
  const float inv = inv_scale_of(byte);
#pragma unroll
  for (int i = 0; i < 16; ++i) mul2(y[2 * i], y[2 * i + 1], inv);  // y <- y / 2^s
  if (OUT == kRotQdq) {
    const float sc = scale_of(byte);
#pragma unroll
    for (int i = 0; i < 16; ++i) out[i] = qdq2<FMT>(y[2 * i], y[2 * i + 1], sc);
  } else if (mx_e2m1<FMT>()) {
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = codes8_e2m1(y + 8 * i);
  } else {
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint2 c = codes8_e4m3(y + 8 * i);
      out[2 * i] = c.x;
      out[2 * i + 1] = c.y;
    }
  }
  if (special && byte == 255u) {
    const uint32_t fill = OUT == kRotQdq ? kBf16NaNx2 : (mx_e2m1<FMT>() ? 0u : kE4M3NaNx4);
#pragma unroll
    for (int i = 0; i < block_out_words<FMT, OUT>(); ++i) out[i] = fill;
  }
  return byte;
}

// shared-memory stages in flight: as many 32 KiB tiles as fit beside H^T and the output tile
template <int FMT, int G, int OUT>
__host__ __device__ constexpr int stages() {
  return OUT == kRotQdq ? 4 : ((G == 128 || OUT == kRotDebug || FMT == kFmtE4M3) ? 5 : 6);
}
// Output tile staged in shared memory and written back with TMA: 128 rows of 128 bf16 (QDQ),
// 128 E4M3 bytes or 64 E2M1 bytes. Two such buffers alternate between tiles.
template <int FMT, int OUT>
__host__ __device__ constexpr int out_stage_bytes() {
  return OUT == kRotDebug ? 0 : kTileRows * block_out_words<FMT, OUT>() * 4 * 4;
}
// Scales staged per 128x128 tile when codes are written: swizzled, one 512-byte 128x4 tile
// (4 scale columns) for the MX formats, two for NVFP4 (8 scale columns of 16-element blocks);
// linear, the same bytes as 128 rows of 4 (MX) or 8 (NVFP4) consecutive scale bytes.
template <int FMT, int OUT>
__host__ __device__ constexpr int scale_stage_bytes() {
  return OUT != kRotCodes ? 0 : (FMT == kFmtNVFP4 ? 1024 : 512);
}
// NVFP4: tables of the two per-scale-byte factors (128 fp32 each).
template <int FMT, int OUT>
__host__ __device__ constexpr int nv_table_bytes() {
  return (FMT == kFmtNVFP4 && OUT != kRotDebug) ? 2 * 128 * 4 : 0;
}
template <int FMT, int G, int OUT>
__host__ __device__ constexpr int smem_request() {
  // 1 KiB of slack for aligning the stage ring to 1024 bytes
  return 1024 + stages<FMT, G, OUT>() * kStageBytes + 2 * out_stage_bytes<FMT, OUT>() + G * G * 2 +
         2 * scale_stage_bytes<FMT, OUT>() + nv_table_bytes<FMT, OUT>() +
         (2 * stages<FMT, G, OUT>() + 2 * kAcc + 1) * 8 + 16;
}
constexpr int kMaxSmemPerCta = 232448;  // opt-in dynamic shared memory limit of the SM

template <int FMT, int OUT, bool SWZ, int G>
__global__ void __launch_bounds__(kThreads, 1)
    mx_rotate_kernel(const __grid_constant__ CUtensorMap tmap, const __grid_constant__ CUtensorMap ymap,
                     RotArgs a) {
  constexpr int kStages = stages<FMT, G, OUT>();
  static_assert(smem_request<FMT, G, OUT>() <= kMaxSmemPerCta, "shared memory budget");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;                                  // kStages x (two swizzled boxes)
  uint8_t* sOut = smem + kStages * kStageBytes;        // [2] output tiles, written back by TMA
  uint8_t* sB = sOut + 2 * out_stage_bytes<FMT, OUT>();  // H^T, core-matrix layout
  uint8_t* s_scale = sB + G * G * 2;  // [2][scale_stage_bytes] staged scales of a tile
  float* t_enc = reinterpret_cast<float*>(s_scale + 2 * scale_stage_bytes<FMT, OUT>());  // NVFP4
  float* t_dq = t_enc + 128;
  uint64_t* full = reinterpret_cast<uint64_t*>(s_scale + 2 * scale_stage_bytes<FMT, OUT>() +
                                               nv_table_bytes<FMT, OUT>());
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + kAcc;
  uint64_t* h_ready = tempty + kAcc;  // B = H^T staged
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(h_ready + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t n_tiles = a.row_blocks * a.col_tiles;
  const uint32_t sA_u32 = smem_u32(sA), sB_u32 = smem_u32(sB);
  // Thread 0 initializes the barriers and is also the TMA producer: it fills the first stages
  // of the ring at once (they wait for nothing), so that the first loads are in flight while
  // the block allocates tensor memory and stages H.
  pdl_launch_dependents();
  int first_loads = 0;
  if (tid == 0) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmap)) : "memory");
    if (OUT != kRotDebug) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&ymap)) : "memory");
    }
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_u32(full + s), 1);
      mbar_init(smem_u32(empty + s), 1);
    }
    for (int b = 0; b < kAcc; ++b) {
      mbar_init(smem_u32(tfull + b), 1);
      mbar_init(smem_u32(tempty + b), kEpiWarps);
    }
    mbar_init(smem_u32(h_ready), kEpiWarps);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    // This CTA's first kPrefetchTiles tiles are prefetched into L2 before pdl_wait (a hint),
    // so that its first loads after the wait find them on chip.
    int pf = 0;
    for (int64_t t = blockIdx.x; t < n_tiles && pf < kPrefetchTiles; t += gridDim.x, ++pf) {
      const int64_t rb = t / a.col_tiles, cb = t - rb * a.col_tiles;
      tma_prefetch_2d(&tmap, (int)(cb * kTileCols), (int)(rb * kTileRows));
      tma_prefetch_2d(&tmap, (int)(cb * kTileCols + kBoxCols), (int)(rb * kTileRows));
    }
  }
  // Everything above touches only shared memory, kernel parameters and L2 prefetch hints; x,
  // H, the outputs and tensor memory are used only once the kernel before this one on the
  // stream has completed.
  pdl_wait();
  if (tid == 0) {
    for (int64_t t = blockIdx.x; t < n_tiles && first_loads < kStages; t += gridDim.x) {
      load_tile(a, &tmap, sA_u32 + first_loads * kStageBytes, smem_u32(full + first_loads), t);
      ++first_loads;
    }
  }
  // The epilogue warps stage B = H^T one 16-byte core-matrix row at a time: row c of the
  // layout (k-group c / G, column n = c % G) holds H[8 (c / G) + t][n], t = 0..7, and sits at
  // byte 16 c, so consecutive threads write consecutive 16 bytes (no bank conflicts). Its eight
  // 2-byte loads (consecutive threads: consecutive columns of a row of H) are issued before
  // the block-wide barrier; the packing, the shared-memory writes and the arrival on h_ready
  // (initialized by thread 0) come after it.
  constexpr int kChunks = G * G / 8;
  constexpr int kPer = (kChunks + kEpiThreads - 1) / kEpiThreads;
  uint32_t hv[kPer][8];
  if (warp >= 2) {
    const uint16_t* H = static_cast<const uint16_t*>(a.H);
    const int et = tid - 64;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int c = et + i * kEpiThreads;
      if (c < kChunks) {
        const int k0 = (c / G) * 8, n = c % G;
#pragma unroll
        for (int t = 0; t < 8; ++t) hv[i][t] = load_u16(H + (k0 + t) * G + n);
      }
    }
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp >= 2) {
    const int et = tid - 64;
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
      const int c = et + i * kEpiThreads;
      if (c < kChunks) {
        uint32_t w[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) w[t] = hv[i][2 * t] | (hv[i][2 * t + 1] << 16);
        *reinterpret_cast<uint4*>(sB + c * 16) = make_uint4(w[0], w[1], w[2], w[3]);
      }
    }
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(smem_u32(h_ready));
  }
  const uint32_t tmem = *tmem_slot;
  bool failed = false;
  const unsigned long long limit = a.wait_limit_ns ? a.wait_limit_ns : kWaitLimitNs;

  if (warp == 0) {
    // ---------------- TMA producer ----------------
    if (lane == 0) {
      int issued = first_loads;  // the first stages were issued before the block-wide barrier
      for (int64_t t = blockIdx.x + (int64_t)issued * gridDim.x; t < n_tiles; t += gridDim.x) {
        const int s = issued % kStages;
        mbar_wait(smem_u32(empty + s), ((issued / kStages) & 1) ^ 1, &failed, limit);
        if (failed) break;
        load_tile(a, &tmap, sA_u32 + s * kStageBytes, smem_u32(full + s), t);
        ++issued;
      }
      // Every load issued has landed before the block can exit: wait for the most recent load
      // of each stage (the earlier ones were consumed before their stage was refilled). After
      // a normal run these phases completed long ago and the waits return at once.
      bool drain_failed = false;
      for (int i = issued > kStages ? issued - kStages : 0; i < issued; ++i) {
        mbar_wait(smem_u32(full + i % kStages), (i / kStages) & 1, &drain_failed);
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer ----------------
    if (lane == 0) {
      constexpr uint32_t idesc = idesc_bf16_f32(kTileRows, G);
      mbar_wait(smem_u32(h_ready), 0, &failed, limit);
      int it = 0;
      for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
        const int s = it % kStages, acc = it % kAcc;
        const int64_t cb = t % a.col_tiles;
        const int64_t kc64 = a.K - cb * kTileCols;
        const int kc = kc64 > kTileCols ? kTileCols : (int)kc64;  // multiple of 32 and of g
        mbar_wait(smem_u32(full + s), (it / kStages) & 1, &failed, limit);
        if (it >= kAcc) mbar_wait(smem_u32(tempty + acc), ((it / kAcc) & 1) ^ 1, &failed, limit);
        if (failed) break;
        tc_fence_after();
        for (int j = 0; j < kc / G; ++j) {
#pragma unroll
          for (int ks = 0; ks < G / 16; ++ks) {
            const int col = j * G + ks * 16;  // first K column of this MMA in the tile
            const uint32_t a_addr = sA_u32 + s * kStageBytes + (col / kBoxCols) * kBoxBytes +
                                    (col % kBoxCols) * 2;
            const uint64_t bd = desc_noswizzle(sB_u32 + 2 * ks * (G * 16), G * 16, 128);
            mma_bf16(tmem + (uint32_t)(acc * 128 + j * G), desc_sw128(a_addr), bd, idesc,
                     ks > 0 ? 1u : 0u);
          }
        }
        mma_commit(smem_u32(empty + s));   // stage free once these MMAs have read it
        mma_commit(smem_u32(tfull + acc));  // accumulator ready
      }
      // `it` tiles were committed; the last commit tracks every MMA this thread issued, so its
      // completion means no MMA still reads shared memory or writes tensor memory.
      if (it > 0) {
        bool drain_failed = false;
        mbar_wait(smem_u32(tfull + (it - 1) % kAcc), ((it - 1) / kAcc) & 1, &drain_failed);
      }
    }
  } else {
    // ---------------- epilogue warps ----------------
    // Thread (quad, lane) owns tile row r = 32 * quad + lane and, in warp quarter q, the
    // 32-column block q. Each tile: read the block's fp32 values from TMEM, free the
    // accumulator, convert, write the block's output bytes into the staged output tile, then
    // one thread writes the tile (and the swizzled scale tile) back with TMA / bulk stores.
    const int e = warp - 2;
    const int quad = warp & 3;          // TMEM lanes 32*quad .. +31 = tile rows
    const int q = e >> 2;               // the 32-column block of the tile this warp converts
    const int r = quad * 32 + lane;     // tile row of this thread
    const uint32_t lane_base = tmem + ((uint32_t)(quad * 32) << 16);
    constexpr int kWords = block_out_words<FMT, OUT>();
    constexpr bool kNv = FMT == kFmtNVFP4;
    float gs = 0.0f, r6 = 0.0f;  // NVFP4 global scale and gs / 6
    if (kNv && OUT != kRotDebug) {
      gs = load_f32(a.gscale);
      r6 = __fdiv_rn(gs, 6.0f);
      if (tid - 64 < 128) nv_factors_of_byte((uint32_t)(tid - 64), gs, t_enc[tid - 64], t_dq[tid - 64]);
      epilogue_sync();  // the factor tables are complete
    }
    int it = 0;
    for (int64_t t = blockIdx.x; t < n_tiles; t += gridDim.x, ++it) {
      const int acc = it % kAcc;
      const int64_t rb = t / a.col_tiles, cb = t - rb * a.col_tiles;
      const int64_t row0 = rb * kTileRows;
      const int64_t kc64 = a.K - cb * kTileCols;
      const int kc = kc64 > kTileCols ? kTileCols : (int)kc64;
      const bool row_ok = row0 + r < a.M;
      const bool active = q * 32 < kc;  // this warp's 32 columns exist in the tile
      mbar_wait(smem_u32(tfull + acc), (it / kAcc) & 1, &failed, limit);
      // tcgen05.ld is warp-collective: once any lane's wait ran out, the whole warp skips it
      failed = __any_sync(0xFFFFFFFFu, failed);
      const bool work = active && !failed;
      tc_fence_after();
      float y[32];
      if (work) tmem_ld32(lane_base + (uint32_t)(acc * 128 + q * 32), y);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_u32(tempty + acc));  // accumulator free for tile it + kAcc
      if (OUT == kRotDebug) {
        if (work && row_ok) {
          float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) +
                                                  (row0 + r) * a.K + cb * kTileCols + q * 32);
#pragma unroll
          for (int i = 0; i < 8; ++i) dst[i] = make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
        }
        continue;
      }
      uint32_t o[kWords];
      uint32_t byte = 0;  // pad rows / columns of the swizzled scale tile stay zero
      if (work) {
        if constexpr (kNv) byte = nv_block_outputs<OUT>(y, o, r6, t_enc, t_dq);
        else byte = block_outputs<FMT, OUT>(y, o);
      }
      // staged tiles alternate; the stores issued two tiles ago (same buffers) have read them
      uint8_t* out_tile = sOut + (it & 1) * out_stage_bytes<FMT, OUT>();
      uint8_t* scale_tile = s_scale + (it & 1) * scale_stage_bytes<FMT, OUT>();
      if (e == 0 && lane == 0) bulk_wait_read_all_but_one();
      epilogue_sync();
      if (work) {
        if (OUT == kRotQdq) {
          // two 128-byte-swizzled boxes of 64 bf16 per row: chunk c of row r at c ^ (r % 8)
          uint8_t* row = out_tile + (q >> 1) * kBoxBytes + r * 128;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int c = (q & 1) * 4 + k;
            *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4)) =
                make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
          }
        } else if (FMT == kFmtE4M3) {
          // one 128-byte-swizzled box of 128 code bytes per row
          uint8_t* row = out_tile + r * 128;
#pragma unroll
          for (int k = 0; k < 2; ++k) {
            const int c = 2 * q + k;
            *reinterpret_cast<uint4*>(row + ((c ^ (r & 7)) << 4)) =
                make_uint4(o[4 * k], o[4 * k + 1], o[4 * k + 2], o[4 * k + 3]);
          }
        } else {
          // one 64-byte-swizzled box of 64 code bytes per row: chunk c at c ^ ((r / 2) % 4)
          *reinterpret_cast<uint4*>(out_tile + r * 64 + ((q ^ ((r >> 1) & 3)) << 4)) =
              make_uint4(o[0], o[1], o[2], o[3]);
        }
      }
      if (OUT == kRotCodes && SWZ) {
        if (kNv) {  // scale columns 2q, 2q + 1: 128x4 tile q / 2, adjacent bytes
          *reinterpret_cast<uint16_t*>(scale_tile + (q >> 1) * 512 +
                                       swizzle_in_tile(r, (2 * q) & 3)) = (uint16_t)byte;
        } else {
          scale_tile[swizzle_in_tile(r, q)] = (uint8_t)byte;
        }
      } else if (OUT == kRotCodes && work) {  // linear: the tile's scales of row r, in order
        if (kNv) *reinterpret_cast<uint16_t*>(scale_tile + r * 8 + 2 * q) = (uint16_t)byte;
        else scale_tile[r * 4 + q] = (uint8_t)byte;
      }
      fence_proxy_async_smem();
      epilogue_sync();
      if (OUT == kRotCodes && !SWZ && q == 0 && row_ok && !failed) {
        // Linear scales: one thread per tile row writes the row's scale bytes of this tile
        // (4 MX / 8 NVFP4 bytes, fewer in a partial last column tile) with one store when the
        // destination allows it, instead of one 1- or 2-byte store per 32-element block.
        // Measured on GB300 (x[8192, 28672], back to back): MXFP4 g = 32 151 -> 94 us, MXFP8
        // 146 -> 119 us, NVFP4 g = 16 159 -> 105 us, each now as fast as its swizzled layout.
        constexpr int kRowBytes = kNv ? 8 : 4;
        const int nbytes = (kc / 32) * (kNv ? 2 : 1);
        uint8_t* dst = a.scales + (row0 + r) * a.scale_cols + cb * kRowBytes;
        const uint8_t* src = scale_tile + r * kRowBytes;
        const uintptr_t addr = reinterpret_cast<uintptr_t>(dst);
        if (nbytes == kRowBytes && (addr & (kRowBytes - 1)) == 0) {
          if (kNv) *reinterpret_cast<uint2*>(dst) = *reinterpret_cast<const uint2*>(src);
          else *reinterpret_cast<uint32_t*>(dst) = *reinterpret_cast<const uint32_t*>(src);
        } else if (kNv) {  // NVFP4 linear scales are 2-byte aligned
          for (int i = 0; i < nbytes; i += 2) {
            *reinterpret_cast<uint16_t*>(dst + i) = *reinterpret_cast<const uint16_t*>(src + i);
          }
        } else {
          for (int i = 0; i < nbytes; ++i) dst[i] = src[i];
        }
      }
      if (e == 0 && lane == 0 && !failed) {
        const uint32_t src = smem_u32(out_tile);
        if (OUT == kRotQdq) {  // rows >= M and columns >= K are dropped by the TMA
          tma_store_2d(&ymap, (int)(cb * kTileCols), (int)row0, src);
          if (kc > kBoxCols) tma_store_2d(&ymap, (int)(cb * kTileCols + kBoxCols), (int)row0, src + kBoxBytes);
        } else if (FMT == kFmtE4M3) {
          tma_store_2d(&ymap, (int)(cb * kTileCols), (int)row0, src);
        } else {
          tma_store_2d(&ymap, (int)(cb * kTileCols / 2), (int)row0, src);
        }
        if (OUT == kRotCodes && SWZ) {
          if (kNv) {  // 128x4 tiles 2 cb and 2 cb + 1 of row block rb (the second may not exist)
            const int64_t per_rb = a.scale_cols / 4, first = 2 * cb;
            const uint32_t bytes = first + 1 < per_rb ? 1024u : 512u;
            bulk_store_s2g(a.scales + (rb * per_rb + first) * 512, smem_u32(scale_tile), bytes);
          } else {
            bulk_store_s2g(a.scales + t * 512, smem_u32(scale_tile), 512);
          }
        }
        bulk_commit();
      }
    }
  }
  if (OUT != kRotDebug && warp == 2 && lane == 0) bulk_wait_all();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// ------------------------------------------------------------------------------------------
// Few rows (M <= kSmallRows, M * g <= kSmallWork): the same rotation and quantization with
// plain fp32 FMAs, one CTA per 128-column tile, x and H staged in shared memory. At these
// sizes the tensor-core kernel's fixed latency chain (tensor memory allocation, TMA load, MMA,
// tensor-memory read, TMA store) is most of a call, while the arithmetic is a few thousand
// FMAs per thread. Thread (r, cg) computes columns
// 8 cg .. 8 cg + 7 of the tile for row r, y_j = sum_i x[r][c0 + i] * H[i][j - c0] with c0 the
// start of the column's g-chunk, accumulated in fp32 in increasing i; the four threads of a
// 32-element block (two of a 16-element NVFP4 block) combine their abs-max with shuffles. The
// CTA writes the tile's swizzled scale tile(s) whole (pad rows zero) from shared memory.
// ------------------------------------------------------------------------------------------
constexpr int kSmallRows = 16;
constexpr int kSmallThreads = kSmallRows * 16;
// The FMA kernel takes a call when M <= kSmallRows and M * g <= kSmallWork: measured in CUDA
// graphs on GB300 it is then faster than the tensor-core kernel (M = 1: 1.7 vs 3.7 us at
// g = 32, 3.4 vs 4.3 us at g = 128), while at M = 16, g = 128 its 8 g FMAs per thread make it
// slower (4.8 vs 4.3 us at K = 8192, 7.8 vs 5.3 us at K = 28672).
constexpr int kSmallWork = 512;

// abs-max of 8 fp32 values as sign-free fp32 bits; NaN propagates.
__device__ __forceinline__ uint32_t absmax_f32x8(const float* y) {
  float m[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    asm("max.NaN.xorsign.abs.f32 %0, %1, %2;" : "=f"(m[i]) : "f"(y[2 * i]), "f"(y[2 * i + 1]));
  }
  asm("max.NaN.xorsign.abs.f32 %0, %1, %2;" : "=f"(m[0]) : "f"(m[0]), "f"(m[2]));
  asm("max.NaN.xorsign.abs.f32 %0, %1, %2;" : "=f"(m[1]) : "f"(m[1]), "f"(m[3]));
  asm("max.NaN.xorsign.abs.f32 %0, %1, %2;" : "=f"(m[0]) : "f"(m[0]), "f"(m[1]));
  return __float_as_uint(m[0]) & 0x7FFFFFFFu;
}

template <int FMT, int OUT, bool SWZ, int G>
__global__ void __launch_bounds__(kSmallThreads)
    mx_rotate_small_kernel(RotArgs a) {
  constexpr bool kNv = FMT == kFmtNVFP4;
  constexpr int kScaleTiles = kNv ? 2 : 1;  // 128x4 scale tiles per 128 columns
  constexpr int kHv = (G * G / 8 + kSmallThreads - 1) / kSmallThreads;  // 16-byte H loads
  __shared__ __align__(16) uint16_t s_h[G * G];                        // H, row-major
  __shared__ __align__(16) uint16_t s_x[kSmallRows * kTileCols];        // the tile's rows of x
  __shared__ __align__(16) uint8_t s_scale[SWZ && OUT == kRotCodes ? kScaleTiles * 512 : 16];
  const int tid = threadIdx.x, r = tid >> 4, cg = tid & 15;
  const int64_t cb = blockIdx.x;
  const int64_t col = cb * kTileCols + cg * 8;
  const bool ok = r < a.M && col < a.K;
  pdl_launch_dependents();
  pdl_wait();

  // stage H and x[r][col .. col + 7] (every 16-byte load issued before one barrier)
  uint4 hreg[kHv];
#pragma unroll
  for (int i = 0; i < kHv; ++i) {
    const int v = tid + i * kSmallThreads;
    if (v < G * G / 8) hreg[i] = load_v4(static_cast<const uint4*>(a.H) + v);
  }
  uint4 xv = make_uint4(0u, 0u, 0u, 0u);
  if (ok) xv = load_v4(static_cast<const uint16_t*>(a.x) + r * a.K + col);
#pragma unroll
  for (int i = 0; i < kHv; ++i) {
    const int v = tid + i * kSmallThreads;
    if (v < G * G / 8) reinterpret_cast<uint4*>(s_h)[v] = hreg[i];
  }
  reinterpret_cast<uint4*>(s_x)[tid] = xv;  // row r, columns 8 cg .. 8 cg + 7 of the tile
  if (SWZ && OUT == kRotCodes) {
    for (int i = tid; i < kScaleTiles * 128; i += kSmallThreads) {
      reinterpret_cast<uint32_t*>(s_scale)[i] = 0u;
    }
  }
  __syncthreads();

  // rotation: 8 outputs of row r, chunk start c0 = col - jj0 (inside the tile: G divides 128)
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
  if (ok) {
    const int jj0 = (int)(col % G);
    const uint16_t* xr = s_x + r * kTileCols + cg * 8 - jj0;
#pragma unroll 4
    for (int i0 = 0; i0 < G; i0 += 8) {
      const uint4 xq = *reinterpret_cast<const uint4*>(xr + i0);
      const uint32_t xw[4] = {xq.x, xq.y, xq.z, xq.w};
#pragma unroll
      for (int ii = 0; ii < 8; ++ii) {
        const float xi = (ii & 1) ? bf16_hi(xw[ii >> 1]) : bf16_lo(xw[ii >> 1]);
        const uint4 hq = *reinterpret_cast<const uint4*>(s_h + (i0 + ii) * G + jj0);
        const uint32_t hw[4] = {hq.x, hq.y, hq.z, hq.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[2 * j] = fmaf(xi, bf16_lo(hw[j]), acc[2 * j]);
          acc[2 * j + 1] = fmaf(xi, bf16_hi(hw[j]), acc[2 * j + 1]);
        }
      }
    }
  }

  if (OUT == kRotDebug) {
    if (ok) {
      float4* dst = reinterpret_cast<float4*>(static_cast<float*>(a.out) + r * a.K + col);
      dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
    return;
  }

  // block scale: abs-max over the 4 threads of a 32-element block (2 of a 16-element block);
  // the Quest-like scale adds the 4 threads' scaled sums of squares as well
  uint32_t amax = absmax_f32x8(acc);
  amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
  if (!kNv) amax = max(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
  uint32_t quest_byte = 0;
  if constexpr (FMT == kFmtE2M1Quest) {  // the plain sum first, the scaled one where needed
    float sum = sq_sum<8>(acc);
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 1);
    sum += __shfl_xor_sync(0xFFFFFFFFu, sum, 2);
    const bool plain = quest_sum_in_range(sum);
    quest_byte = quest_byte_from_sum(sum, 127u);
    if (__any_sync(0xFFFFFFFFu, !plain)) {  // every lane takes part in the shuffles
      const uint32_t E = amax >> 23;
      float scaled = scaled_sq_sum<8>(acc, quest_prescale(E));
      scaled += __shfl_xor_sync(0xFFFFFFFFu, scaled, 1);
      scaled += __shfl_xor_sync(0xFFFFFFFFu, scaled, 2);
      if (!plain) quest_byte = quest_byte_from_sum(scaled, E);
    }
  }
  uint32_t byte;
  uint32_t o[4];
  if constexpr (kNv) {
    const float gs = load_f32(a.gscale);
    const float r6 = __fdiv_rn(gs, 6.0f);
    const NvScales n = nv_scales(amax, amax, gs, r6);
    byte = n.bytes & 0xFFu;
#pragma unroll
    for (int i = 0; i < 4; ++i) mul2(acc[2 * i], acc[2 * i + 1], n.enc[0]);
    if (OUT == kRotQdq) {
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = n.special[0] ? kBf16NaNx2 : qdq2_e2m1(acc[2 * i], acc[2 * i + 1], n.dq[0]);
    } else {
      o[0] = n.special[0] ? 0u : codes8_e2m1(acc);
    }
  } else {
    byte = FMT == kFmtE2M1Quest ? quest_byte : scale_byte_from_amax_bits<FMT>(amax);
    const float inv = inv_scale_of(byte);
#pragma unroll
    for (int i = 0; i < 4; ++i) mul2(acc[2 * i], acc[2 * i + 1], inv);
    if (OUT == kRotQdq) {
      const float sc = scale_of(byte);
#pragma unroll
      for (int i = 0; i < 4; ++i) o[i] = qdq2<FMT>(acc[2 * i], acc[2 * i + 1], sc);
      if (byte == 255u) {
#pragma unroll
        for (int i = 0; i < 4; ++i) o[i] = kBf16NaNx2;
      }
    } else if (mx_e2m1<FMT>()) {
      o[0] = byte == 255u ? 0u : codes8_e2m1(acc);
    } else {
      const uint2 c = codes8_e4m3(acc);
      o[0] = byte == 255u ? kE4M3NaNx4 : c.x;
      o[1] = byte == 255u ? kE4M3NaNx4 : c.y;
    }
  }

  // element outputs
  if (ok) {
    if (OUT == kRotQdq) {
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.out) + r * a.K + col) =
          make_uint4(o[0], o[1], o[2], o[3]);
    } else if (FMT == kFmtE4M3) {
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(a.out) + r * a.K + col) = make_uint2(o[0], o[1]);
    } else {
      *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(a.out) + r * (a.K / 2) + col / 2) = o[0];
    }
  }
  if (OUT != kRotCodes) return;

  // scales: one thread per block writes its byte
  const int per_block = kNv ? 2 : 4;  // threads per scale block
  const int sc_col = cg / per_block;  // scale column within the tile
  const bool writer = ok && (cg % per_block) == 0;
  if (!SWZ) {
    if (writer) a.scales[r * a.scale_cols + cb * (kNv ? 8 : 4) + sc_col] = (uint8_t)byte;
    return;
  }
  __syncthreads();  // the staged tile(s) are zero
  if (writer) s_scale[(sc_col >> 2) * 512 + swizzle_in_tile(r, sc_col & 3)] = (uint8_t)byte;
  __syncthreads();
  const int64_t per_rb = a.scale_cols / 4;  // 128x4 tiles per row block
  const int64_t first = cb * kScaleTiles;
  const int words = (first + kScaleTiles <= per_rb ? kScaleTiles : 1) * 32;  // 16-byte words
  if (tid < words) {
    reinterpret_cast<uint4*>(a.scales + first * 512)[tid] = reinterpret_cast<const uint4*>(s_scale)[tid];
  }
}

// Self-test of the bounded wait: one thread waits on an mbarrier that nothing ever arrives at,
// with the kernels' wait routine and a short limit; the wait gives up and sets the device error
// word, and the kernel returns.
__global__ void mx_wait_selftest_kernel(unsigned long long limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    bool failed = false;
    mbar_wait(smem_u32(&bar), 0, &failed, limit_ns);
  }
}

// ------------------------------------------------------------------------------------------
// host side
// ------------------------------------------------------------------------------------------
// Tensor map of a row-major [rows, cols] matrix, boxes of kTileRows x box_cols.
cudaError_t make_tensor_map(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                            CUtensorMapDataType type, int elem_bytes, int box_cols,
                            CUtensorMapSwizzle swizzle) {
  return make_tensor_map_2d(map, base, rows, cols, type, elem_bytes, box_cols, kTileRows, swizzle);
}

template <int FMT, int OUT, bool SWZ, int G>
cudaError_t launch_t(const RotArgs& a, cudaStream_t stream) {
  if (a.M <= kSmallRows && a.M * G <= kSmallWork) {  // few rows: the FMA kernel
    if (a.col_tiles <= 0) return cudaSuccess;
    return launch_pdl(&mx_rotate_small_kernel<FMT, OUT, SWZ, G>, dim3((unsigned)a.col_tiles),
                      dim3(kSmallThreads), 0, stream, a);
  }
  auto kern = mx_rotate_kernel<FMT, OUT, SWZ, G>;
  const void* k = reinterpret_cast<const void*>(kern);
  constexpr int smem = smem_request<FMT, G, OUT>();
  const int64_t n_tiles = a.row_blocks * a.col_tiles;
  if (n_tiles <= 0) return cudaSuccess;
  CUtensorMap map, ymap;
  cudaError_t err = make_tensor_map(&map, a.x, a.M, a.K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                                    kBoxCols, CU_TENSOR_MAP_SWIZZLE_128B);
  if (err != cudaSuccess) return err;
  if (OUT == kRotQdq) {  // bf16 [M, K]
    err = make_tensor_map(&ymap, a.out, a.M, a.K, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, kBoxCols,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  } else if (OUT == kRotCodes && FMT == kFmtE4M3) {  // E4M3 bytes [M, K]
    err = make_tensor_map(&ymap, a.out, a.M, a.K, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 128,
                          CU_TENSOR_MAP_SWIZZLE_128B);
  } else if (OUT == kRotCodes) {  // E2M1 bytes [M, K / 2]
    err = make_tensor_map(&ymap, a.out, a.M, a.K / 2, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, 64,
                          CU_TENSOR_MAP_SWIZZLE_64B);
  } else {
    ymap = map;  // unused
  }
  if (err != cudaSuccess) return err;
  const int resident = resident_ctas(k, kThreads, smem, 1);
  if (resident <= 0) return cudaErrorInvalidConfiguration;
  const int grid = (int)(n_tiles < resident ? n_tiles : resident);
  return launch_pdl(kern, dim3(grid), dim3(kThreads), smem, stream, map, ymap, a);
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

// Tensor map of a row-major [rows, cols] matrix of 1- or 2-byte elements, boxes of box_rows x
// box_cols, the given swizzle; loads read zeros out of bounds, stores drop what falls outside.
cudaError_t make_tensor_map_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                               CUtensorMapDataType type, int elem_bytes, int box_cols,
                               int box_rows, CUtensorMapSwizzle swizzle) {
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess) {
      encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
  });
  if (!encode) return cudaErrorNotSupported;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * elem_bytes};
  const cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  const cuuint32_t elem_strides[2] = {1, 1};
  const CUresult r = encode(map, type, 2, const_cast<void*>(base), dims, strides, box, elem_strides,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}


cudaError_t launch_rotate(int fmt, int out_kind, bool swizzled, int g, const RotArgs& a,
                          cudaStream_t stream) {
  if (out_kind == kRotDebug) return launch_g<kFmtE2M1, kRotDebug, false>(g, a, stream);
  if (fmt == kFmtE2M1) return launch_fmt<kFmtE2M1>(out_kind, swizzled, g, a, stream);
  if (fmt == kFmtE2M1Quest) return launch_fmt<kFmtE2M1Quest>(out_kind, swizzled, g, a, stream);
  if (fmt == kFmtNVFP4) return launch_fmt<kFmtNVFP4>(out_kind, swizzled, g, a, stream);
  return launch_fmt<kFmtE4M3>(out_kind, swizzled, g, a, stream);
}

cudaError_t launch_wait_selftest(unsigned long long limit_ns, cudaStream_t stream) {
  mx_wait_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
  return cudaGetLastError();
}

cudaError_t device_error_word(unsigned int** word) {
  static std::mutex mu;
  static unsigned int* cache[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void* p = nullptr;
    err = cudaGetSymbolAddress(&p, g_device_errors);
    if (err != cudaSuccess) return err;
    cache[dev] = static_cast<unsigned int*>(p);
  }
  *word = cache[dev];
  return cudaSuccess;
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
