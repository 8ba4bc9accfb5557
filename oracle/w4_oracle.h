/*
 * w4_oracle.h -- the CPU oracle for the symmetric group-wise INT4
 * weight-only projection (W4A16).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the timed
 * CPU baseline of the benchmark may load this library.  The product path
 * (the CUDA library and its binding) never calls it, and the two share no
 * code, header, table or constant.
 *
 * What it computes follows "Building a Custom LLM Inference Runtime for
 * Qwen2.5-Coder-7B on NVIDIA H100 Hopper Architecture", section "Technical
 * Specifications and Hardware Alignment": weights are signed 4-bit integers,
 * symmetric (no zero point), in groups of 128 along K with one FP16 scale per
 * group; activations stay FP16 (same page, "The INT8 vs. FP16 Activation
 * Trade-off", Path B).  Plain FP64 arithmetic, k ascending, one final
 * IEEE-754 binary16 round-to-nearest-even.
 *
 * Every function here is pinned by tests against things other than itself
 * (IEEE-754 binary16 tables, exhaustive enumeration, exact rational brute
 * force, closed forms, symmetries, a library float64 matmul); see the
 * oracle's tests.
 */
#ifndef W4_ORACLE_H
#define W4_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* IEEE 754-2008 binary16: the value of bit pattern h, exactly, as a double
 * (NaN patterns give a NaN, 0x7C00/0xFC00 give +/-inf). */
double w4o_double_from_half(uint16_t h);

/* IEEE 754-2008 binary16 rounding of v, round-to-nearest, ties-to-even;
 * |v| >= 65520 gives +/-inf, NaN gives 0x7E00 (sign kept). */
uint16_t w4o_half_from_double(double v);

/* y[m,n] = half_rne( sum_{k=0}^{K-1} x[m,k] * q[n,k] * s[n, k/128] )
 * evaluated in FP64 with k ascending.
 *   x   : fp16 bit patterns, [M, K] row-major
 *   q   : int8 in [-8, 7],   [N, K] row-major (unpacked, one value per byte)
 *   s   : fp16 bit patterns, [N, K/128] row-major
 *   y   : fp16 bit patterns, [M, N] row-major (written)
 *   acc : optional [M, N] FP64 sums before rounding (written if non-NULL)
 * Returns 0, or -1 for K % 128 != 0 / negative sizes / NULL pointers,
 * -2 for a q outside [-8, 7].  Rows n are spread over `nthreads` threads
 * (<= 0: one thread). */
int w4o_linear(const uint16_t* x, const int8_t* q, const uint16_t* s,
               int64_t M, int64_t N, int64_t K,
               uint16_t* y, double* acc, int nthreads);

/* bfloat16 (the upper 16 bits of IEEE 754 binary32): the exact value of bit
 * pattern b, and the round-to-nearest, ties-to-even bfloat16 of v
 * (|v| >= 255.5 * 2^120 gives +/-inf, NaN gives 0x7FC0 with the sign kept).
 * For the BF16-activation variant of the projection (x and y in bfloat16
 * instead of binary16, weights and scales unchanged). */
double w4o_double_from_bf16(uint16_t b);
uint16_t w4o_bf16_from_double(double v);

/* w4o_linear with the activation type chosen: act 0 = binary16 x and y,
 * act 1 = bfloat16 x and y (scales stay binary16).  Same FP64 sum, k
 * ascending, one final rounding to the output type.  -1 for a bad act. */
int w4o_linear_act(const uint16_t* x, int act, const int8_t* q, const uint16_t* s,
                   int64_t M, int64_t N, int64_t K,
                   uint16_t* y, double* acc, int nthreads);

/* Path A of the pages ("Building a Custom LLM Inference Runtime ...", "3. The
 * INT8 vs. FP16 Activation Trade-off"; "The Architecture of Modern Inference
 * ...", "3. The Performance Paradox"): activations quantised to INT8 and
 * integer dot products.  The pages give no quantisation details; the
 * reading taken: per-token symmetric absmax, in IEEE binary32,
 * sx = max|x| / 127, xq = rne(x / sx) clamped to +-127 (the integer
 * decision in the GPU's precision), then
 * y = half_rne(sum_g s * sx * sum_{k in g} xq * q) with exact integer group
 * sums and FP64 scaling.  w4o_quantize_x8 exposes the quantisation. */
void w4o_quantize_x8(const uint16_t* x, int64_t M, int64_t K, int8_t* xq, float* sx);
int w4o_linear_q8(const uint16_t* x, const int8_t* q, const uint16_t* s,
                  int64_t M, int64_t N, int64_t K, uint16_t* y, double* acc);

/* The packed device layout, written out plainly from its definition
 * (the layout is a design of this library, not of the pages; the pages only
 * say that the nibbles are shuffled for the byte-permute datapath:
 * "The .nanoqwen File Format and Safety Protocols", ValueShuffle).
 *
 * Tiles of 16 rows x 128 K; tile (band b, group g) at byte
 * (b * (K/128) + g) * 1056.  With u = q + 8 (offset binary), the 32-bit word
 * of warp lane L (L = 4*r + c, r in 0..7, c in 0..3) and k16-step j (0..7)
 * sits at byte (j < 4 ? 0 : 512) + 16*L + 4*(j % 4) of the tile, little
 * endian, and holds in nibble i (bits 4i..4i+3):
 *   i=0: u[r][16j+4c]    i=1: u[r+8][16j+4c]
 *   i=2: u[r][16j+4c+2]  i=3: u[r+8][16j+4c+2]
 *   i=4: u[r][16j+4c+1]  i=5: u[r+8][16j+4c+1]
 *   i=6: u[r][16j+4c+3]  i=7: u[r+8][16j+4c+3]
 * (rows relative to the band, k relative to the group).  Bytes
 * 1024 + 4p .. 1024 + 4p + 3 (p = 0..7) hold the fp16 scales of rows p
 * (low half) and p + 8 (high half).  Rows n >= N are padding: u = 8, scale 0.
 * dst must hold ceil(N/16) * (K/128) * 1056 bytes.  Returns 0, -1 on bad
 * arguments, -2 on a q outside [-8, 7]. */
int w4o_pack_layout(const int8_t* q, const uint16_t* s, int64_t N, int64_t K,
                    uint8_t* dst);

#ifdef __cplusplus
}
#endif
#endif
