/*
 * q4_oracle.h -- CPU oracle for the GGUF Q4_0 weight-only-quantized linear layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This is a plain, slow, single-purpose restatement of
 * what the Q4_0 path computes, used to check the CUDA library.  Only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg may load it.  It
 * shares no code, header, table or constant with the CUDA library, and the CUDA
 * library never calls it.
 *
 * Source of the method: the GeekNews write-up of the Rust/Burn port of
 * "Voxtral Mini 4B Realtime" (es.news.hada.io/topic?id=26595, section
 * "Arquitectura") names the weight format of the quantized inference path as
 * GGUF Q4_0, run through custom GPU shaders, and section "Soluciones técnicas"
 * keeps the 1.5 GiB embedding table as Q4 rows looked up per token.  The pages do
 * not print the block layout; the layout below is the public GGUF Q4_0 format:
 *
 *   block of 32 weights = 18 bytes
 *     bytes [0,2)  : scale d, IEEE binary16, little-endian
 *     bytes [2,18) : qs[16]; element j (0..15) is the low nibble of qs[j],
 *                    element j+16 is the high nibble of qs[j]
 *   decoded weight  w = (q - 8) * d
 *
 * A weight matrix W with N outputs and reduction length K (K % 32 == 0) is N
 * rows of K/32 consecutive blocks, rows contiguous (row stride 18*K/32 bytes).
 *
 * Status codes returned here use the same numbering as the library's C ABI so
 * that tests can compare them; they are restated, not included.
 */
#ifndef Q4_ORACLE_H
#define Q4_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define Q4O_OK 0
#define Q4O_ERR_INVALID_ARG 1
#define Q4O_ERR_NONFINITE 4
#define Q4O_ERR_ID_OUT_OF_RANGE 5

/* IEEE binary16 <-> binary32, written from the format definition. */
float q4o_half_to_float(uint16_t h);
uint16_t q4o_float_to_half_rne(float f);

/* Decode one 18-byte block into 32 fp32 weights, w = (q - 8) * d, computed as one
 * fp32 multiply of the small integer (q - 8) by d (always exact). */
void q4o_decode_block(const uint8_t* blk, float* out32);

/* Quantize one block of 32 fp32 weights (reading of the quantizer: the pages do
 * not give one).  Returns Q4O_OK, or Q4O_ERR_NONFINITE for a block holding a
 * NaN/Inf or whose scale overflows binary16; such a block is written as d = +0
 * and all codes 8. */
int q4o_quantize_block(const float* x32, uint8_t* blk);

/* Row-wise forms.  k must be a positive multiple of 32.  Returns Q4O_OK or
 * Q4O_ERR_INVALID_ARG; q4o_quantize returns Q4O_ERR_NONFINITE if any block was
 * non-finite (all other blocks are still written) and counts them. */
int q4o_quantize(const float* w, int64_t n, int64_t k, uint8_t* blocks, int64_t* n_bad);
int q4o_dequant_rows(const uint8_t* blocks, int64_t n_rows, int64_t k, float* out);

/* Y[m][i] = sum_k W^[i][k] * X[m][k] in fp64, in increasing k, over the exactly
 * decoded weights and the exact fp32 inputs; S[m][i] = sum_k |W^[i][k] X[m][k]|.
 * X is row-major with leading dimension ldx; Y and S have leading dimension ldy.
 * Rows i are split over nthreads POSIX threads (results do not depend on it). */
int q4o_matmul(const uint8_t* W, int64_t n, int64_t k, const float* X, int64_t m,
               int64_t ldx, double* Y, double* S, int64_t ldy, int nthreads);

/* out[b][:] = decode(row ids[b]); an id outside [0, vocab) gives a row of +0.0
 * and makes the call return Q4O_ERR_ID_OUT_OF_RANGE (other rows are written). */
int q4o_embed_gather(const uint8_t* table, int64_t vocab, int64_t k, const int32_t* ids,
                     int64_t n_ids, float* out);

/* Y = W^ X as q4o_matmul, with X given in fp64 (an input that is itself the
 * exact result of an earlier fp64 step, e.g. the gated FFN activation). */
int q4o_matmul_f64(const uint8_t* W, int64_t n, int64_t k, const double* X, int64_t m,
                   int64_t ldx, double* Y, double* S, int64_t ldy, int nthreads);

/* Gated FFN activation between the decoder's w1/w3 and w2 linears.  READING:
 * the pages name the decoder (GeekNews "Arquitectura") but no activation; the
 * plainest reading for this Mistral-family decoder is the SiLU-gated unit:
 *   out[i] = a[i] * sigmoid(a[i]) * b[i],  sigmoid(t) = 1 / (1 + exp(-t)),
 * in fp64, a = the w1 rows' output, b = the w3 rows' output. */
void q4o_swiglu(const double* a, const double* b, int64_t n, double* out);

/* Index of the largest y[i] (the greedy next token over the output head's
 * logits); the lowest index among equal maxima; NaN entries are ignored.
 * Returns -1 when n <= 0 or every entry is NaN. */
int64_t q4o_argmax(const double* y, int64_t n);

/* Q4 x Q8 integer path (READING: the usual companion of GGUF Q4_0; details
 * are this library's).  q4o_quantize_q8: x [k] (k % 32 == 0) -> int8 codes q
 * [k] and fp32 scales d [k/32]: amax = max |x_j| per block, d = amax / 127,
 * q_j = round-half-away(x_j / d) clamped to +-127 (fp32 IEEE division);
 * amax == 0 -> d = +0, q = 0; a non-finite element -> d = NaN, q = 0.
 * q4o_matmul_q8: Y[m][n] = sum_b d_w * d_x * sum_j (q_w - 8) q_x per row of X
 * (integer sums exact, the rest fp64), S the sum of the block terms'
 * magnitudes.  Return Q4O_OK or Q4O_ERR_INVALID_ARG. */
int q4o_quantize_q8(const float* x, int64_t k, int8_t* q, float* d);
int q4o_matmul_q8(const uint8_t* W, int64_t n, int64_t k, const float* X, int64_t m,
                  int64_t ldx, double* Y, double* S, int64_t ldy);

/* Repacked tile layout of a Q4_0 matrix (this library's GPU-native layout;
 * the pages name only the GGUF format).  Definition, for k % 256 == 0:
 *   rows are taken in groups of 16 (the last group padded with rows whose
 *   blocks have d = +0 and every code 8), k in slices of 256 (8 blocks);
 *   tile (G, t) = rows 16G..16G+15 x blocks 8t..8t+7 is 2304 bytes at offset
 *   (G * (k/256) + t) * 2304.  Inside a tile, with g = 0..7 and hr = 0 for row
 *   16G + g, hr = 1 for row 16G + g + 8:
 *     scales: bytes [32g + 4b + 2hr, +2) hold the binary16 d of that row's
 *       block 8t + b, little-endian;
 *     codes: the tile's 256 columns are 16 steps of 16 (column c = 16s + i);
 *       lane L = 4g + (i % 8) / 2 of step s owns a little-endian 32-bit word
 *       at 256 + 512 (s / 4) + 16L + 4 (s % 4), whose nibble
 *       m = hr + 2 (i / 8) + 4 (i % 2) (bits 4m..4m+3) holds the code of
 *       column c.  So a byte of a word holds rows g (low nibble) and g + 8
 *       (high nibble) of one column, and the word holds a lane's four columns
 *       2(i%8/2) + {0, 1, 8, 9} of the step: the operand order of a 16 x 16
 *       row-major tensor-core A fragment.
 * q4o_repack_bytes gives the size; q4o_repack / q4o_unrepack convert (the
 * padding rows are dropped by q4o_unrepack).  Return Q4O_OK or
 * Q4O_ERR_INVALID_ARG. */
int64_t q4o_repack_bytes(int64_t n, int64_t k);
int q4o_repack(const uint8_t* W, int64_t n, int64_t k, uint8_t* R);
int q4o_unrepack(const uint8_t* R, int64_t n, int64_t k, uint8_t* W);

#ifdef __cplusplus
}
#endif
#endif
