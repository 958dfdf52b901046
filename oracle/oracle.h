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
 *   IQ3_S, IQ2_S per tower: the grid G (a table of the format, caller-supplied:
 *         IQ3_S 512 entries x 4 uint8 magnitudes, IQ2_S 1024 x 8), then the blocks
 *         of all rows [rows][K/256]. A group of 4 (IQ3_S) or 8 (IQ2_S) consecutive
 *         weights is one grid entry with one sign bit per weight:
 *         w = (d * (2 sc + 1)) * G[idx][i] * (sign ? -1 : +1)   (exact).
 *         IQ3_S 110 B: fp16 d | 64 B idx bits 0..7 of group i (elements 4i..4i+3) |
 *           8 B: bit i = idx bit 8 of group i | 32 B: bit e = sign of element e |
 *           4 B: nibble j (byte j/2, low nibble for even j) = sc of 32-value sub-block j
 *         IQ2_S 82 B: fp16 d | 32 B idx bits 0..7 of group i (elements 8i..8i+7) |
 *           32 B: byte i bit k = sign of element 8i+k | 8 B: bits 2i..2i+1 = idx bits
 *           8..9 of group i | 8 B: nibble k = sc of 16-value sub-block k
 *         The pages fix the block sizes (110 and 82 B / 256), the group widths (four
 *         gathers per group of four for IQ3_S; 1,024 entries of 8 weights for IQ2_S)
 *         and the sign bits; field order, the odd scale 2 sc + 1 and the caller-
 *         supplied grid are this reading (no grid values are printed).
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

enum { OR_Q8_0 = 1, OR_Q4_K = 2, OR_Q6_K = 3, OR_NVFP4 = 4, OR_FP8_ROW = 5, OR_Q5_K = 6, OR_IQ4_XS = 7,
       OR_IQ3_S = 8, OR_IQ2_S = 9 };

/* scalar number formats */
float or_fp16_to_f32(uint16_t h);
uint16_t or_f32_to_fp16(float f);
float or_bf16_to_f32(uint16_t b);
uint16_t or_f64_to_bf16(double v);
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
/* the codebook formats: IQ4_XS takes the matrix's codebook C (16 x int8); IQ3_S and
 * IQ2_S take the grid G (512 x 4 / 1024 x 8 uint8 magnitudes) */
int or_encode_cb(int fmt, const float* W, int64_t rows, int64_t K, const void* codebook,
                 uint8_t* canon);
/* grid bytes of a grid format (0 for the others) */
int64_t or_grid_bytes(int fmt);

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

/* int8-dot lever: x quantized to int8 per 32 values (d = amax / 127, q = rint(x / d));
 * y = sum_k W[n][k] d q_k in fp64 against BlockToFloat W [N][K]; den = sum |terms| */
void or_quant_act_q8(const uint16_t* x_bf16, int64_t M, int64_t K, int8_t* codes, float* scales);
void or_int8dot_f64(const uint16_t* x_bf16, int64_t M, int64_t K, const float* W, int64_t N, double* y,
                    double* den);

/* SwiGLU: h = silu(g) * u, silu(g) = g / (1 + exp(-g)), fp64 elementwise */
void or_swiglu_f64(const double* g, const double* u, int64_t n, double* h);

#ifdef __cplusplus
}
#endif
#endif
