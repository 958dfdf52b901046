/*
 * oracle.h -- plain, slow, single-threaded CPU oracle for the block-quantized
 * weight GEMV  y[M,N] = x[M,K] . W[N,K]^T  and its grouped per-expert form.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load or call this library. The product path
 * (the CUDA library) never does, and shares no code, header, table or constant
 * generator with it.
 *
 * Everything here is written from the definitions, in the order the pages and
 * the number-format definitions give them; nothing is blocked, fused or
 * reordered. Floating-point dequantization is fp32 with round-to-nearest-even
 * (compiled with -ffp-contract=off); dot products accumulate in fp64.
 *
 * Canonical (input) byte layouts, one per format; all multi-byte fields are
 * little-endian:
 *   Q8_0  34 B per 32 values : fp16 d | 32 x int8 q
 *   Q4_K 144 B per 256 values: fp16 d | fp16 dmin | 12 B scales | 128 B quants
 *         scales = 96-bit LSB-first bitstream of sixteen 6-bit fields,
 *         fields 0..7 = sub-block scales sc_j, fields 8..15 = sub-block mins m_j;
 *         quant byte b: low nibble = element 2b, high nibble = element 2b+1
 *   Q5_K 176 B per 256 values: fp16 d | fp16 dmin | 12 B scales | 32 B qh | 128 B qs
 *         scales exactly as Q4_K; qs exactly as Q4_K's quants (low 4 bits);
 *         qh = 256-bit LSB-first bitstream, bit e = 5th bit (value 16) of element e;
 *         q = lo | hi << 4 in 0..31
 *   Q6_K 210 B per 256 values: 128 B ql | 64 B qh | 16 x int8 scales | fp16 d
 *         ql byte b: low nibble = low 4 bits of element 2b, high = of 2b+1;
 *         qh byte b: bits 2i..2i+1 = high 2 bits of element 4b+i (i = 0..3)
 *   NVFP4 per matrix: codes [rows][K/2] (element 2i in the low nibble of byte i)
 *         | E4M3 block scales [rows][K/16] | fp32 tensor scale
 *   FP8_ROW per matrix: E4M3 codes [rows][K] | fp32 row scales [rows]
 *   IQ4_XS per matrix: 136-byte blocks of 256 values [rows][K/256] | codebook C,
 *         16 x int8. Block: fp16 d | u16 sh | 4 B sl | 128 B indices. Scale of
 *         32-value sub-block j: ls_j = (sl byte j/2, nibble j%2) | (sh bits 2j..2j+1)
 *         << 4, in 0..63; index byte b: low nibble = element 2b, high = 2b+1.
 *         The pages fix the block size (136 B / 256) and that a weight is a
 *         codebook entry; the field order, the signed scale ls - 32 and the
 *         caller-supplied codebook are this reading (no GGUF layout is printed).
 * A stacked tower of E experts is E such matrices back to back (for the
 * K-quants this is the same bytes as one [E*N, K] matrix).
 */
#ifndef QMV_ORACLE_H
#define QMV_ORACLE_H
#include <stdint.h>
#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { OR_Q8_0 = 1, OR_Q4_K = 2, OR_Q6_K = 3, OR_NVFP4 = 4, OR_FP8_ROW = 5, OR_Q5_K = 6, OR_IQ4_XS = 7 };

/* scalar number formats */
float or_fp16_to_f32(uint16_t h);
uint16_t or_f32_to_fp16(float f);
float or_bf16_to_f32(uint16_t b);
float or_e4m3_to_f32(uint8_t c);
uint8_t or_f32_to_e4m3(float f);
float or_e2m1_to_f32(uint8_t c);
uint8_t or_f32_to_e2m1(float f);

/* sizes */
int64_t or_block_values(int fmt);
int64_t or_canon_bytes(int fmt, int64_t rows, int64_t K);

/* encoders: synthetic-data generation only (not on the hot path) */
int or_encode(int fmt, const float* W, int64_t rows, int64_t K, float tensor_scale,
              uint8_t* canon);
/* the codebook formats (IQ4_XS): the matrix's codebook C (16 x int8) is an input */
int or_encode_cb(int fmt, const float* W, int64_t rows, int64_t K, const int8_t* codebook,
                 uint8_t* canon);

/* BlockToFloat: canonical bytes of `rows` rows -> fp32 W[rows][K] */
int or_block_to_float(int fmt, const uint8_t* canon, int64_t rows, int64_t K, float* W);

/* y[m][n] = sum_k (double)W[n][k] * (double)x[m][k];  den[m][n] = sum_k |W x| */
void or_gemv_f64(const float* W, int64_t N, int64_t K, const uint16_t* x_bf16, int64_t M,
                 double* y, double* den);

/* sorted distinct expert ids of ids[n]; returns the count */
int64_t or_unique_experts(const int32_t* ids, int64_t n, int32_t* out);

/* NVFP4 activation quantizer for the W4A4 route */
void or_quant_act_nvfp4(const uint16_t* x_bf16, int64_t M, int64_t K, float x_scale,
                        uint8_t* codes, uint8_t* scales);

/* W4A4: y[m][n] = sum_k dq(quant_act(x))[m][k] * W[n][k] in fp64, W = BlockToFloat of
 * the NVFP4 weights [N][K]; den = sum |terms| */
void or_w4a4_f64(const uint16_t* x_bf16, int64_t M, int64_t K, float x_scale, const float* W, int64_t N,
                 double* y, double* den);

/* SwiGLU: h = silu(g) * u, silu(g) = g / (1 + exp(-g)), fp64 elementwise */
void or_swiglu_f64(const double* g, const double* u, int64_t n, double* h);

#ifdef __cplusplus
}
#endif
#endif
