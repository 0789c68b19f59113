/*
 * mxq.h -- C ABI of libmxq: OCP-MX block quantization (MXFP4 / MXFP8) on one GB300 GPU.
 *
 * What the library computes (sources are the pages this library restates):
 *  - "[Transform] [Quantization] Add QuTLASS support to vLLM" (vllm PR 24440), feature list:
 *    abs-max block scales ("Multiple quantization schemes ... Abs-Max"), the MXFP4 format,
 *    "Fused transform + quantization + scale computation", rotation matrices "loaded at
 *    runtime, allowing any transformation", rotation sizes 16/32/64/128; review thread on
 *    vllm/_custom_ops.py (`fusedQuantizeMx(a, b, ...)` returning packed E2M1 codes and E8M0
 *    scales of shape `padded_rows x padded_cols`) and on vllm/qutlass_utils/utils.py
 *    (`to_blocked`: the blocked scale layout block-scaled GEMMs consume).
 *  - "use cute-dsl to speedup mxfp QDQ" (intel/neural-compressor PR 2548), Description:
 *    MXFP4 / MXFP8 QDQ on contiguous input, group size 32, K divisible by 32, CUDA-Graph use.
 *  - prhub summary of vllm PR 47229, code snippet of mxfp8_utils.py: MXFP8 (E4M3) quantize
 *    with MXFP8_BLOCK_SIZE = 32 returning codes and scales, scales viewed as [M, K/32] when not
 *    swizzled, or in the swizzled layout when `is_sf_swizzled_layout`.
 *
 * Arithmetic (the pages name the formats but print no formula; this is the OCP MX reading):
 *  For every block of 32 consecutive elements along K of a bf16 row-major [M, K] matrix:
 *    amax = max |v_i|;  s = clamp(floor(log2 amax) - emax, -127, 127)  (emax = 2 for E2M1,
 *    8 for E4M3; an all-zero block gets s = -127);  E8M0 scale byte = s + 127;
 *    code_i = v_i / 2^s rounded to nearest-even on the element grid, saturating at the largest
 *    finite magnitude (6 for E2M1, 448 for E4M3), sign kept (also for zero);
 *    QDQ output_i = bf16_round_nearest_even(decode(code_i) * 2^s).
 *  A block holding a NaN or an infinity gets scale byte 0xFF; its codes are 0x7F (E4M3) or
 *  0x0 (E2M1) and its QDQ outputs are the bf16 NaN 0x7FC0.
 *
 * Conventions for every entry point:
 *  - Pointers named x, y, codes, scales, H, row_offsets are DEVICE memory owned by the caller;
 *    the library never allocates, frees or synchronizes, and never reads device memory on the
 *    host. Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default stream) and is
 *    asynchronous.
 *  - Validation happens on the host before any launch; on error nothing is launched and the
 *    status says why. After the launch, a launch failure maps to MX_ERR_CUDA.
 *  - x, y and codes must be 32-byte aligned, H and swizzled scales 16-byte aligned; rows
 *    are contiguous.
 *  - M == 0 or K == 0 is a valid empty call: nothing is launched, MX_OK is returned.
 *  - Layouts: E4M3 codes are [M, K] bytes (float8_e4m3fn). E2M1 codes are [M, K/2] bytes, two
 *    codes per byte, the lower K index in the low nibble. Linear scales are [M, K/32] bytes,
 *    row-major. Swizzled scales are [ceil(M/128)*128, ceil(K/128)*4] bytes: the scale matrix is
 *    padded with zero bytes and cut into 128x4 tiles of 512 bytes, stored row-block-major; scale
 *    (r, c) of a tile sits at byte (r % 32) * 16 + (r / 32) * 4 + c. Every byte, pads
 *    included, is written by each call.
 */
#ifndef MXQ_H
#define MXQ_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int mx_status;

/* status codes */
#define MX_OK 0
#define MX_ERR_NULL 1        /* a required pointer is NULL */
#define MX_ERR_SHAPE 2       /* negative size, K % 32 != 0, K % g != 0, bad expert count */
#define MX_ERR_ALIGN 3       /* misaligned pointer (x, y, codes: 32 B; H, scales: 16 B) */
#define MX_ERR_UNSUPPORTED 4 /* unknown format / layout / rounding, group != 32, bad g */
#define MX_ERR_CUDA 5        /* the CUDA runtime reported an error at launch */

/* element formats */
#define MX_FMT_E2M1 1 /* MXFP4: 1 sign, 2 exponent, 1 mantissa bit */
#define MX_FMT_E4M3 2 /* MXFP8: 1 sign, 4 exponent, 3 mantissa bits ("fn": max 448, no Inf) */

/* scale layouts */
#define MX_SCALES_LINEAR 0   /* [M, K/32] row-major */
#define MX_SCALES_SWIZZLED 1 /* 128x4 blocked tiles, padded (see above) */

/*
 * Rounding schemes (argument `rounding`): how the block scale is chosen. The elements are always
 * rounded to nearest even with saturation under the chosen scale.
 *  MX_ROUND_RNE: the abs-max scale above (the QuTLASS feature list's "Abs-Max" scheme).
 *  MX_ROUND_QUEST: the Quartet / "Quest-like" scale (QuTLASS feature list: "Multiple
 *    quantization schemes ... Quartet (i.e., Quest-like)"; the review thread on
 *    vllm/_custom_ops.py names its call fusedQuantizeMxQuest(a, b, xh_e2m1, xh_e8m0)). MXFP4
 *    (MX_FMT_E2M1) only; not for grouped calls. The pages print no rule; the reading is the
 *    rule above with the block's clip point c in place of amax:
 *      c = alpha * sqrt(sum_i v_i^2 / 32),  s = clamp(floor(log2 c) - 2, -127, 127),
 *    alpha = 2.922475, the ratio of clip point to standard deviation that minimises the mean
 *    squared error of the E2M1 grid (its largest value 6 at the clip point) on a normally
 *    distributed input; values above 6 * 2^s saturate (the clipping). An all-zero block gets
 *    byte 0, a block with a NaN or an infinity 0xFF as above. The sum of squares is formed in
 *    fp32 after an exact power-of-two scaling (no overflow or underflow for any finite input),
 *    so s can differ from the real-number rule only where c lies within about 2^-20 relative of
 *    a power of two.
 */
#define MX_ROUND_RNE 0
#define MX_ROUND_QUEST 1

/*
 * Rotation kinds (argument rot_kind of the rotating calls; ignored where H is NULL).
 *  MX_ROT_DENSE: H is any bf16 [g, g] matrix; the product runs on the tensor cores (calls
 *    with at most 16 rows and M * g <= 512: fp32 FMAs).
 *  MX_ROT_HADAMARD: the caller states that H = c * S_g, where S_g is the Sylvester Hadamard
 *    matrix of order g (S_1 = [1], S_2n = [[S_n, S_n], [S_n, -S_n]], entry (i, j) =
 *    (-1)^popcount(i & j)) and c = H[0][0], e.g. the normalized hadamard(g) * g^-0.5 rounded
 *    to bf16. For g <= 64 the product is then a fast Walsh-Hadamard transform in registers
 *    (log2 g butterfly stages in fp32, then a multiplication by c) on the streaming kernel.
 *    Every CTA checks the statement on the bit patterns of H on the device; where it does not
 *    hold the call computes sum_i x_i H[i][j] with fp32 FMAs instead, so the results are
 *    correct for any H (only slower). For g = 128 the call runs as MX_ROT_DENSE (faster
 *    there).
 *  MX_ROT_AUTO: the same statement as MX_ROT_HADAMARD; the library takes whichever of the two
 *    kernels measured faster on GB300 for the call: the fp32-FMA kernel for decode-sized calls
 *    (M <= 16, M * g <= 512) and the tensor cores for g = 128; otherwise the Walsh-Hadamard
 *    kernel below 4096 rows, and from 4096 rows the tensor cores for 4-bit codes (MXFP4, NVFP4)
 *    and for MXFP8 codes or QDQ outputs while M * K <= 3 * 2^25, the Walsh-Hadamard kernel above.
 *    mx_rotate_debug treats it as MX_ROT_HADAMARD.
 * The kinds compute the same rotation up to fp32 rounding (well inside the 1e-5 normwise
 * tolerance of the rotated path).
 */
#define MX_ROT_DENSE 0
#define MX_ROT_HADAMARD 1
#define MX_ROT_AUTO 2

/* Text of a status code (static storage). */
const char* mx_status_string(mx_status status);

/*
 * Shape of the scale matrix for an [M, K] input: linear [M, K/32]; swizzled
 * [ceil(M/128)*128, ceil(K/128)*4]. Host only, launches nothing.
 * Errors: MX_ERR_NULL (rows or cols NULL), MX_ERR_SHAPE (M < 0, K < 0, K % 32),
 * MX_ERR_UNSUPPORTED (group != 32, unknown layout).
 */
mx_status mx_scales_shape(int64_t M, int64_t K, int group, int layout, int64_t* rows,
                          int64_t* cols);

/*
 * Block quantize (pages: fusedQuantizeMx without the rotation; mxfp8_quantize).
 * x: bf16 [M, K]. codes: see layouts. scales: per `layout`. fmt: MX_FMT_*. group: must be 32.
 * rounding: MX_ROUND_RNE, or MX_ROUND_QUEST with MX_FMT_E2M1. Errors: see conventions.
 */
mx_status mx_quantize(const void* x, int64_t M, int64_t K, int fmt, int group, int layout,
                      int rounding, void* codes, void* scales, void* stream);

/*
 * QDQ: quantize then dequantize, bf16 in, bf16 out (pages: mxfp4_qdq / mxfp8_qdq).
 * If H is not NULL, every g-element chunk along K is first rotated, y_chunk = x_chunk * H
 * (H: bf16 [g, g] row-major device matrix, g in {16, 32, 64, 128}, K % g == 0, rot_kind an
 * MX_ROT_* value), and the rotated values are quantized; the output stays in the rotated
 * basis. If H is NULL, g and rot_kind are ignored. y: bf16 [M, K], must not overlap x.
 * rounding as in mx_quantize.
 */
mx_status mx_qdq(const void* x, int64_t M, int64_t K, int fmt, int group, int rounding,
                 const void* H, int g, int rot_kind, void* y, void* stream);

/*
 * Dequantize stored MX data to bf16 (pages: the QuTLASS review thread on vLLM's MXFP4 test,
 * which dequantizes packed E2M1 codes with their E8M0 scales, `_dq_fp4(b_e2m1, b_e8m0, ...)`,
 * before a reference matmul; the dequantize half of mxfp4_qdq / mxfp8_qdq).
 * y_i = bf16_round_nearest_even(decode(code_i) * 2^(scale_byte - 127)) for every element, so
 * mx_dequantize(mx_quantize(x)) == mx_qdq(x) bit for bit. Any code and scale byte is accepted:
 * scale byte 0xFF (E8M0 NaN) and E4M3 codes S.1111.111 give the bf16 NaN 0x7FC0, products
 * above the bf16 range give +-Inf, tiny products round to bf16 subnormals or signed zero.
 * codes: E2M1 [M, K/2] or E4M3 [M, K] bytes (32-byte aligned), laid out as mx_quantize writes
 * them. scales: linear [M, K/32] or swizzled (16-byte aligned) as returned by
 * mx_scales_shape(); pad bytes are not read. y: bf16 [M, K] (32-byte aligned), must not
 * overlap the inputs. Errors: see conventions.
 */
mx_status mx_dequantize(const void* codes, const void* scales, int64_t M, int64_t K, int fmt,
                        int group, int layout, void* y, void* stream);

/*
 * Fused rotate + quantize (pages: fusedQuantizeMx(a, b) with b the runtime-loaded rotation).
 * y_chunk = x_chunk * H for every g-chunk along K (bf16 products, fp32 accumulation; see
 * MX_ROT_* for how), then the block quantization above on the fp32 rotated values.
 * H: bf16 [g, g] row-major, g in {16, 32, 64, 128}, K % g == 0. rot_kind: MX_ROT_*. Other
 * arguments as mx_quantize.
 */
mx_status mx_rotate_quantize(const void* x, int64_t M, int64_t K, const void* H, int g,
                             int rot_kind, int fmt, int group, int layout, int rounding,
                             void* codes, void* scales, void* stream);

/*
 * Scale-matrix shape for a grouped call with E experts and M_total rows: linear
 * [M_total, K/32]; swizzled [R, ceil(K/128)*4] with R = floor((M_total + 127*E) / 128) * 128,
 * an upper bound of sum_e ceil(n_e/128)*128 valid for any split of M_total rows.
 */
mx_status mx_grouped_scales_shape(int64_t M_total, int E, int64_t K, int group, int layout,
                                  int64_t* rows, int64_t* cols);

/*
 * Grouped (MoE expert) quantize. Rows [row_offsets[e], row_offsets[e+1]) of x belong to
 * expert e (row_offsets: DEVICE int64 [E+1], row_offsets[0] = 0, row_offsets[E] = M_total,
 * non-decreasing). Codes stay contiguous as for mx_quantize on the whole x. Linear scales are
 * [M_total, K/32]: the call is then mx_quantize on the whole x and does not read row_offsets.
 * Swizzled scales give each expert its own run of 128-row tiles: expert e's
 * rows start at padded row P_e = sum_{e' < e} ceil(n_e'/128) * 128; the buffer has
 * mx_grouped_scales_shape() rows and all of it is written (rows past the last expert: zero).
 * 1 <= E <= 1024. Offsets that break the contract give unspecified values but every access
 * stays inside x, codes and scales. rounding: MX_ROUND_RNE (MX_ROUND_QUEST: MX_ERR_UNSUPPORTED).
 */
mx_status mx_quantize_grouped(const void* x, const int64_t* row_offsets, int E, int64_t M_total,
                              int64_t K, int fmt, int group, int layout, int rounding,
                              void* codes, void* scales, void* stream);

/*
 * NVFP4 (pages: the QuTLASS feature list, "Support for both NVFP4 and MXFP4", and its review
 * thread on benchmarks/kernels/bench_nvfp4_qutlass.py: fusedQuantizeNv(a, H, global_scale)
 * returning E2M1 codes and blocked scales viewed as [-1, K/16]). E2M1 codes in blocks of 16
 * along K, one E4M3 scale byte per block, under a per-tensor fp32 global scale gs. The pages
 * print no scale rule; the reading is the usual two-level one, every step one fp32 operation
 * rounded to nearest even, in this order, per block with abs-max amax:
 *   s_f = amax * (gs / 6);  scale byte = E4M3(s_f), saturating at 448;
 *   enc = gs / decode(scale);  code_i = E2M1(v_i * enc)  (enc = 0 when decode(scale) == 0);
 *   QDQ: y_i = bf16(decode(code_i) * (decode(scale) / gs))  (0 factor likewise).
 * A block holding a NaN or an infinity gets scale byte 0x7F, codes 0 and QDQ outputs 0x7FC0.
 * With H (bf16 [g, g], g in {16, 32, 64, 128}, K % g == 0) every g-chunk is first rotated,
 * y_chunk = x_chunk * H (fp32 accumulation; rot_kind as in mx_rotate_quantize, ignored without
 * H), as in mx_rotate_quantize.
 * global_scale: DEVICE pointer to one fp32 value, 4-byte aligned, read by the kernel (so it may
 * come from an earlier kernel on the same stream); it must be positive and finite, and
 * gs / 2^-9 must not overflow fp32 (gs < 1.7e38 * 2^-9), else results are unspecified.
 * K % 32 == 0. Codes: [M, K/2] bytes (32-byte aligned), the lower K index in the low nibble.
 * Scales: linear [M, K/16] (2-byte aligned) or swizzled [ceil(M/128)*128, ceil(K/64)*4]
 * (16-byte aligned; 128x4 tiles as for the MX scales, pads zero), see mx_nvfp4_scales_shape.
 */
mx_status mx_nvfp4_scales_shape(int64_t M, int64_t K, int layout, int64_t* rows, int64_t* cols);

mx_status mx_quantize_nvfp4(const void* x, int64_t M, int64_t K, const void* H, int g,
                            int rot_kind, const float* global_scale, int layout, void* codes,
                            void* scales, void* stream);

/* NVFP4 QDQ (see above): bf16 y [M, K], 32-byte aligned, must not overlap x. */
mx_status mx_qdq_nvfp4(const void* x, int64_t M, int64_t K, const void* H, int g, int rot_kind,
                       const float* global_scale, void* y, void* stream);

/*
 * Grouped (MoE expert) NVFP4 quantize: rows [row_offsets[e], row_offsets[e+1]) of x are expert
 * e's input and are quantized as by mx_quantize_nvfp4 (no rotation) under that expert's own
 * global scale global_scales[e] (DEVICE fp32 [E], 4-byte aligned, each positive and finite;
 * pass E equal values for one shared scale). row_offsets: DEVICE int64 [E+1] with the contract
 * of mx_quantize_grouped. Codes stay contiguous [M_total, K/2]. Linear scales are
 * [M_total, K/16] (2-byte aligned); swizzled scales give each expert its own run of 128-row
 * tiles starting at padded row P_e = sum_{e' < e} ceil(n_e'/128) * 128, in a buffer of
 * mx_nvfp4_grouped_scales_shape() bytes that is written whole (pads zero; 16-byte aligned).
 * 1 <= E <= 1024, K % 32 == 0.
 */
mx_status mx_nvfp4_grouped_scales_shape(int64_t M_total, int E, int64_t K, int layout,
                                        int64_t* rows, int64_t* cols);

mx_status mx_quantize_nvfp4_grouped(const void* x, const int64_t* row_offsets, int E,
                                    int64_t M_total, int64_t K, const float* global_scales,
                                    int layout, void* codes, void* scales, void* stream);

/*
 * NVFP4 dequantize (the dequantize half of NVFP4 QDQ; see the NVFP4 reading above):
 * y_i = bf16(decode(code_i) * (decode(scale) / gs)) with each 16-element block's E4M3 scale
 * byte decoded as a signed E4M3 value (0 factor when it decodes to zero), every step one fp32
 * operation rounded to nearest even, so mx_dequantize_nvfp4(mx_quantize_nvfp4(x)) ==
 * mx_qdq_nvfp4(x) bit for bit (same H, same gs). Scale bytes 0x7F / 0xFF (the E4M3 NaN) give
 * 0x7FC0 for their block. codes: [M, K/2] bytes (32-byte aligned). scales: linear [M, K/16]
 * (2-byte aligned) or swizzled as mx_nvfp4_scales_shape() (16-byte aligned; pads not read).
 * global_scale: DEVICE pointer to one positive finite fp32 value (4-byte aligned). y: bf16
 * [M, K] (32-byte aligned), must not overlap the inputs. K % 32 == 0. Errors: see conventions.
 */
mx_status mx_dequantize_nvfp4(const void* codes, const void* scales, int64_t M, int64_t K,
                              const float* global_scale, int layout, void* y, void* stream);

/*
 * Block-scaled GEMM consumer (pages: the QuTLASS review thread on vLLM's MXFP4 test, which runs
 * matmul_mxf4_bf16_tn(a_e2m1, b_e2m1, a_e8m0, b_e8m0, alpha) on the quantizer's outputs and
 * compares it with the matmul of the dequantized operands `_dq_fp4(...)`):
 *   C[i][j] = alpha * sum_k dequant(A)[i][k] * dequant(B)[j][k]   ("TN": both K-major),
 * dequant as in mx_dequantize (decode(code) * 2^(scale_byte - 127) rounded to bf16 once: exact
 * for every E2M1 value and for E4M3 unless below the bf16 range), products exact, sums in fp32
 * on the tensor cores, C rounded to bf16 once. A: codes [M, K/2] (E2M1) or [M, K] (E4M3) with
 * scales [M, K/32] (linear) or the 128x4 blocked layout of mx_scales_shape(M, K) (swizzled), as
 * mx_quantize writes them; B likewise with N rows; both in the same fmt and layout. C: bf16
 * [M, N] row-major, must not overlap the inputs. K % 64 == 0 (K > 0), N % 8 == 0; codes and C
 * 16-byte aligned, linear scales 2-byte aligned, swizzled scales 16-byte aligned. A scale byte
 * 0xFF makes its 32 values NaN.
 * M <= 8,388,480 (65,535 tiles of 128 rows). M == 0 or N == 0 is a no-op returning MX_OK.
 * Errors: see conventions; K not a positive multiple of 64, N % 8 or M too large ->
 * MX_ERR_SHAPE.
 */
mx_status mx_gemm(const void* a_codes, const void* a_scales, const void* b_codes,
                  const void* b_scales, int64_t M, int64_t N, int64_t K, int fmt, int group,
                  int layout, float alpha, void* c, void* stream);

/*
 * Diagnostics: the rotated values y = x_chunk * H exactly as mx_rotate_quantize computes them
 * before quantization with the same rot_kind (same device code), written as fp32 [M, K] to
 * y_f32 (device, 32-byte aligned).
 */
mx_status mx_rotate_debug(const void* x, int64_t M, int64_t K, const void* H, int g, int rot_kind,
                          float* y_f32, void* stream);

/*
 * Device-side error word of the current device: bit 0 set if a kernel gave up waiting for
 * its tensor-core work to complete (a bounded wait ran out; its outputs are then invalid).
 * Synchronizes the device, returns the word in *flags and clears it.
 */
mx_status mx_device_errors(int* flags);

/*
 * Failure-detection self-test (no counterpart on the pages): launches one thread that waits on
 * an mbarrier nothing ever arrives at, with the same bounded-wait routine the tensor-core
 * kernel uses for every wait, given up after limit_ns nanoseconds (1 .. 100,000,000). The wait
 * gives up, sets bit 0 of the device error word (read it with mx_device_errors) and the kernel
 * returns; the context stays usable. Errors: MX_ERR_SHAPE (limit out of range), MX_ERR_CUDA.
 */
mx_status mx_selftest_bounded_wait(int64_t limit_ns, void* stream);

/*
 * Give-up self-test of the tensor-core rotation kernel (no counterpart on the pages): the call
 * mx_rotate_quantize(x, M, K, H, g, MX_FMT_E2M1, 32, MX_SCALES_SWIZZLED, MX_ROUND_RNE, codes,
 * scales, stream) makes, with every mbarrier wait of the kernel limited to limit_ns
 * nanoseconds (1 .. 100,000,000) instead of 2 s, so that waits run out while the pipeline is
 * busy. A role whose wait ran out stops issuing work, and the kernel still waits for its loads,
 * MMAs and stores in flight before it frees tensor memory and exits: the call ends, the device
 * error word reports the give-up (mx_device_errors) and the context stays usable. codes and
 * scales then hold unspecified bytes. Shapes as mx_rotate_quantize, except that calls the
 * few-row kernel would take (M <= 16 and M * g <= 512) and empty calls are MX_ERR_SHAPE.
 * Errors: MX_ERR_SHAPE (limit or shape), MX_ERR_NULL, MX_ERR_ALIGN, MX_ERR_UNSUPPORTED (g),
 * MX_ERR_CUDA.
 */
mx_status mx_selftest_rotate_give_up(const void* x, int64_t M, int64_t K, const void* H, int g,
                                     void* codes, void* scales, int64_t limit_ns, void* stream);

/*
 * Give-up self-test of the GEMM kernel (no counterpart on the pages): the call
 * mx_gemm(a_codes, a_scales, b_codes, b_scales, M, N, K, fmt, 32, layout, 1.0f, c, stream)
 * makes, with every pipeline wait of the kernel limited to limit_ns nanoseconds
 * (1 .. 100,000,000) instead of 2 s. A role whose wait ran out stops issuing work; the loads in
 * flight and the MMAs issued are still waited for (2 s) before the kernel frees its tensor
 * memory and exits: the call ends, the device error word reports the give-up
 * (mx_device_errors) and the context stays usable. c then holds unspecified bytes. Shapes and
 * errors as mx_gemm, except that M == 0 or N == 0 is MX_ERR_SHAPE.
 */
mx_status mx_selftest_gemm_give_up(const void* a_codes, const void* a_scales, const void* b_codes,
                                   const void* b_scales, int64_t M, int64_t N, int64_t K, int fmt,
                                   int layout, void* c, int64_t limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MXQ_H */
