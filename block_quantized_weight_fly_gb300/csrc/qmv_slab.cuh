// qmv_slab.cuh -- per-format decode + tensor-core inner product of one slab
// (128 rows x 256 values of packed weights, already in shared memory).
//
// A consumer warp w owns rows 16w .. 16w+15 of the slab. The inner product runs
// on mma.sync m16n8k16 with the weight rows as the 16-row A operand; the weights
// are decoded in registers straight into A fragments:
//   Q4_K, Q6_K -> bf16: masks alone turn element pairs into exact bf16 values
//                      {q, q'} x 2^-133 .. 2^-127 through bf16's linear (subnormal and
//                      first normal) range; x is scaled by a power of two so that
//                      every product lands at one scale (see the Q4_K and Q6_K notes).
//   Q5_K, Q8_0 -> bf16: one AND-OR per two fields gives {128 + q, 128 + q'} exactly
//                      (element pairs at fields (p, p+4) of each 32-bit word); the
//                      +128 offset is removed with the per-block term through X = sum x.
//   NVFP4, FP8 -> f16: hardware cvt of FP4/FP8 pairs to f16x2 (exact).
//   IQ4_XS     -> f16: a byte-permute lookup of the 16-entry codebook, placed under
//                      the f16 pattern of 1024 ({1152 + C[q], 1152 + C[q']} exactly).
//   IQ3_S, IQ2_S -> f16: an 8-byte shared-memory load of the grid entry (f16
//                      magnitudes), signs applied with one multiply and one AND-XOR.
// Products of these small exact values with the activations are exact and the
// tensor core accumulates in fp32.
//
// The 8 columns of the mma output are used in one of two ways:
//   M = 1 ("unit columns"): column n holds the partial sum of one unit (sub-block
//     or block) of the slab. A thread's B registers carry activations only for its
//     own unit, zero elsewhere, so one accumulator collects the partial sums of 8
//     units at once and each block scale is applied once per slab.
//   M = 2..8 ("token columns"): column n is token n; each unit gets its own MMA
//     chain started from zero.
//
// One accumulation order for every M (so that row m of an M-row call equals the
// one-row call on x[m] bit for bit). The units of a slab are split among the four
// threads t of an mma quad exactly as the unit columns place them: quad position t
// owns the units of chunks 2t and 2t+1 (Q4_K, Q5_K, Q8_0, FP8, IQ4_XS, IQ3_S: units
// 2t, 2t+1; Q6_K, IQ2_S units 4t .. 4t+3; NVFP4 blocks 4t .. 4t+3). Per output
// (row, token):
//   * every unit sum is the same MMA chain over the same operands in both forms
//     (in the unit-column form the other columns only add exact zeros);
//   * c_t = the format's combination of position t's unit sums with their scales
//     (the *_comb functions below, written with explicit roundings so that the
//     compiler cannot contract them differently in the two forms);
//   * A_t = the fp32 sum of c_t over the slabs of a piece, in k order;
//   * the piece value is (A_0 + A_1) + (A_2 + A_3).
// How pieces are formed and added up is the stream kernel's part (qmv_stream.cu).
// The unit-column form adds a thread's own c_t (it is quad position t) and the
// quad's four sums are joined with two shuffles; the token-column form keeps the
// four sums A_0..A_3 of each of its outputs.
#pragma once
#include <cstdint>
#include "qmv_layout.cuh"

namespace qmv {

constexpr int kXStride = 576;          // bytes per token row of a stage's x slice (512 + 64 pad)
constexpr int kXZero = 512;            // M = 1: the pad after x row 0 holds zeros ...
constexpr int kXZeroBytes = 64;        // ... (64 bytes, written once per kernel)
constexpr int kTblStride = 17;         // float2 entries per row of a warp's scale table
constexpr uint32_t kOnesBf16 = 0x3F803F80u;

// ---------------------------------------------------------------------------
// helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_bf16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void mma_f16(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                        uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint32_t lds32(const void* p) { return *reinterpret_cast<const uint32_t*>(p); }
__device__ __forceinline__ uint2 lds64(const void* p) { return *reinterpret_cast<const uint2*>(p); }
__device__ __forceinline__ uint4 lds128v(const void* p) { return *reinterpret_cast<const uint4*>(p); }

__device__ __forceinline__ void load8(const uint8_t* p, uint32_t* w) {    // 32 bytes, 16-B aligned
  const uint4 a = lds128v(p), b = lds128v(p + 16);
  w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
}
__device__ __forceinline__ void load16(const uint8_t* p, uint32_t* w) {   // 64 bytes, 16-B aligned
  load8(p, w);
  load8(p + 32, w + 8);
}
// (a & m) | o as one three-input logic op
__device__ __forceinline__ uint32_t and_or(uint32_t a, uint32_t m, uint32_t o) {
  uint32_t d;
  asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(d) : "r"(a), "r"(m), "r"(o));
  return d;
}
// two 4-bit fields at nibbles (p, p+4) -> bf16x2 {128 + lo, 128 + hi}
__device__ __forceinline__ uint32_t nib_pair(uint32_t w, int p) {
  return and_or(p ? (w >> (4 * p)) : w, 0x000F000Fu, 0x43004300u);
}
// two 2-bit fields at bits (2k, 2k + 16) -> bf16x2 {128 + lo, 128 + hi}
__device__ __forceinline__ uint32_t bit2_pair(uint32_t w, int k) {
  return and_or(k ? (w >> (2 * k)) : w, 0x00030003u, 0x43004300u);
}
// the low 6 bits of v as an exact fp32
__device__ __forceinline__ float u6f(uint32_t v) {
  return __uint_as_float(and_or(v, 63u, 0x4B000000u)) - 8388608.0f;
}
// the two fp16 values of a 32-bit word as fp32 (exact)
__device__ __forceinline__ float2 h2x2f(uint32_t v) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}
// FP8 E4M3 pair (low 16 bits) -> f16x2, exact
__device__ __forceinline__ uint32_t e4m3x2_f16(uint32_t two) {
  uint32_t r;
  const unsigned short v = (unsigned short)(two & 0xFFFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(v));
  return r;
}
// the four E2M1 pairs of a word (bytes 0..3) -> four f16x2, exact. The bytes are
// taken as the low bytes of the word's 16-bit halves and of those of word >> 8, so
// one shift serves all four conversions.
__device__ __forceinline__ void e2m1x4_f16(uint32_t w, uint32_t* p) {
  asm("{ .reg .b16 l, h, l8, h8; .reg .b8 b0, b1, b2, b3; .reg .b32 s;\n\t"
      "shr.b32 s, %4, 8;\n\t"
      "mov.b32 {l, h}, %4;\n\t"
      "mov.b32 {l8, h8}, s;\n\t"
      "cvt.u8.u16 b0, l;\n\t"
      "cvt.u8.u16 b1, l8;\n\t"
      "cvt.u8.u16 b2, h;\n\t"
      "cvt.u8.u16 b3, h8;\n\t"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n\t"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n\t"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n\t"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n\t}"
      : "=r"(p[0]), "=r"(p[1]), "=r"(p[2]), "=r"(p[3])
      : "r"(w));
}
// the two E4M3 pairs of a word (halves 0, 1) -> two f16x2, exact
__device__ __forceinline__ void e4m3x4_f16(uint32_t w, uint32_t* p) {
  asm("{ .reg .b16 l, h;\n\t"
      "mov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\t"
      "cvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(p[0]), "=r"(p[1])
      : "r"(w));
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// bf16x2 activations -> f16x2 (round to nearest; exact for |x| in fp16's normal range)
__device__ __forceinline__ uint32_t bf16x2_to_f16x2(uint32_t w) {
  uint32_t r;
  const float lo = __uint_as_float(w << 16), hi = __uint_as_float(w & 0xFFFF0000u);
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// a small non-negative integer (< 2^23) -> exact fp32, without I2F
__device__ __forceinline__ float u2f_small(uint32_t v) {
  return __uint_as_float(v | 0x4B000000u) - 8388608.0f;
}
__device__ __forceinline__ float i8f(uint32_t byte) {   // signed int8 -> fp32
  return __uint_as_float(((byte & 0xFFu) ^ 0x80u) | 0x4B000000u) - 8388736.0f;
}
// keep v if this thread's unit is the current one, else zero (sparse unit-column B)
__device__ __forceinline__ uint32_t sel(bool mine, uint32_t v) { return mine ? v : 0u; }
// Sparse unit-column B from shared memory: the thread's own activations for the
// sub-block it owns, the zero pad for every other sub-block (one address select
// per load instead of one select per register).
__device__ __forceinline__ uint4 ldx128(const uint8_t* xs, bool mine, uint32_t off) {
  return lds128v(xs + (mine ? off : (uint32_t)kXZero));
}
__device__ __forceinline__ uint2 ldx64(const uint8_t* xs, bool mine, uint32_t off) {
  return lds64(xs + (mine ? off : (uint32_t)kXZero));
}

template <int FMT, int MT>
struct Slab;

// ---------------------------------------------------------------------------
// Canonical combinations c_t of one quad position's unit sums (shared by both
// forms; explicit roundings, no contraction)
// ---------------------------------------------------------------------------
// Q4_K and Q5_K over two 32-value sub-blocks: a_i D_i - b_i X_i
__device__ __forceinline__ float kq_comb(float a0, float a1, float b0, float b1, float D0, float D1, float X0,
                                         float X1) {
  return __fmaf_rn(a0, D0, __fmaf_rn(a1, D1, -__fmaf_rn(b0, X0, __fmul_rn(b1, X1))));
}
// Q8_0: sum q x of one 32-value chunk = lo + 16 hi - 2304 X (fields taken as 128 + nibble)
__device__ __forceinline__ float q80_part(float lo, float hi, float X) {
  return __fmaf_rn(-2304.0f, X, __fmaf_rn(16.0f, hi, lo));
}
__device__ __forceinline__ float q80_comb(float d0, float d1, float lo0, float hi0, float X0, float lo1, float hi1,
                                          float X1) {
  return __fmaf_rn(d0, q80_part(lo0, hi0, X0), __fmul_rn(d1, q80_part(lo1, hi1, X1)));
}
// Q6_K: one 16-value unit folded into v; a66 = d sc 2^66, m32 = -32 d sc
__device__ __forceinline__ float q6k_step(float v, float a66, float m32, float lo, float hi, float X) {
  return __fmaf_rn(a66, __fadd_rn(lo, hi), __fmaf_rn(m32, X, v));
}
__device__ __forceinline__ float q6k_a66(float a) { return __fmul_rn(a, 7.3786976294838206e19f); }  // exact
__device__ __forceinline__ float q6k_m32(float a) { return __fmul_rn(-32.0f, a); }                 // exact
// NVFP4: four 16-value blocks with their E4M3 scales
__device__ __forceinline__ float nv_comb(float s0, float s1, float s2, float s3, float B0, float B1, float B2,
                                         float B3) {
  return __fmaf_rn(s0, B0, __fmaf_rn(s1, B1, __fmaf_rn(s2, B2, __fmul_rn(s3, B3))));
}
// FP8: two chunk sums (the row scale multiplies the row's total)
__device__ __forceinline__ float fp8_comb(float D0, float D1) { return __fadd_rn(D0, D1); }
// IQ3_S over two 32-value chunks, IQ2_S over four 16-value units (no offset term)
__device__ __forceinline__ float grid_comb(float a0, float a1, float D0, float D1) {
  return __fmaf_rn(a0, D0, __fmul_rn(a1, D1));
}
__device__ __forceinline__ float grid16_comb(float a0, float a1, float a2, float a3, float D0, float D1, float D2,
                                             float D3) {
  return __fmaf_rn(a3, D3, __fmaf_rn(a2, D2, __fmaf_rn(a1, D1, __fmul_rn(a0, D0))));
}
// IQ4_XS over two 32-value chunks: a_i (D_i - 1152 X_i), D_i over 1152 + C[q]
__device__ __forceinline__ float iq4_comb(float a0, float a1, float D0, float D1, float X0, float X1) {
  return __fmaf_rn(a0, __fmaf_rn(-1152.0f, X0, D0), __fmul_rn(a1, __fmaf_rn(-1152.0f, X1, D1)));
}
// the piece value from the four quad positions' sums
__device__ __forceinline__ float quad_join(float a0, float a1, float a2, float a3) {
  return __fadd_rn(__fadd_rn(a0, a1), __fadd_rn(a2, a3));
}
// the token-column form adds c into A_t of output e
__device__ __forceinline__ void tc_add(float (&a)[4][4], int t, int e, float c) { a[t][e] = __fadd_rn(a[t][e], c); }

// ============================================================================
// Q4_K. w = a_j q - b_j (a_j = d sc_j, b_j = dmin m_j, sub-block j = 32 values).
// Decoded through bf16's linear range: the bit patterns 0..255 of a bf16 are
// exactly the values 0..255 x 2^-133 (subnormals and the first normal binade), so a
// word masked with 0x000F000F gives {q, q'} x 2^-133 and masked with 0x00F000F0
// gives {q, q'} x 2^-129 -- no shift for two of the four pairs and no offset. The
// activations are scaled by 2^67 (low-nibble pairs) or 2^63 (high-nibble pairs)
// with one exact bf16x2 multiply each, so every product is q x 2^-66: a normal fp32
// value for 2^-60 <= |x| < 2^61 (the tensor core keeps subnormal bf16 operands
// exactly). The sum is rescaled by 2^66 through a_j.
// ============================================================================
__device__ __forceinline__ uint32_t bmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
constexpr uint32_t kX67 = 0x61006100u;   // bf16x2 {2^67, 2^67}
constexpr uint32_t kX63 = 0x5F005F00u;   // bf16x2 {2^63, 2^63}
constexpr uint32_t kX71 = 0x63006300u;   // bf16x2 {2^71, 2^71}
constexpr uint32_t kX69 = 0x62006200u;   // bf16x2 {2^69, 2^69}
constexpr uint32_t kX65 = 0x60006000u;   // bf16x2 {2^65, 2^65}

// sc_j, m_j of sub-blocks 2t, 2t+1 of a header (12 consecutive stream bits each):
// from the header words in registers, or from a record in shared memory (the scale
// stream starts at byte 4, the fields at stream bits 12t (sc) and 48 + 12t (m), each
// pair taken from two aligned words with one funnel shift)
__device__ __forceinline__ void q4k_fields(const uint4 hd, int t, uint32_t* s, uint32_t* m) {
  const uint64_t lo = ((uint64_t)hd.z << 32) | hd.y, hi = ((uint64_t)hd.w << 32) | hd.z;
  *s = (uint32_t)(lo >> (12 * t));
  *m = (uint32_t)(hi >> (16 + 12 * t));
}
__device__ __forceinline__ void q4k_fields_rec(const uint8_t* rec, int t, uint32_t* s, uint32_t* m) {
  const uint32_t* sw = reinterpret_cast<const uint32_t*>(rec + 4);
  const int bs = 12 * t, bm = 48 + 12 * t;
  *s = __funnelshift_r(sw[bs >> 5], sw[(bs >> 5) + 1], bs & 31);
  *m = __funnelshift_r(sw[bm >> 5], sw[(bm >> 5) + 1], bm & 31);
}
// Q4_K: a_j x 2^66 and b_j (all products exact)
__device__ __forceinline__ void q4k_scales_lin(uint32_t dw, uint32_t s, uint32_t m, float* a, float* b) {
  const float2 dd = h2x2f(dw);
  const float d66 = __fmul_rn(dd.x, 7.3786976294838206e19f);      // d x 2^66
  a[0] = __fmul_rn(d66, u6f(s));
  a[1] = __fmul_rn(d66, u6f(s >> 6));
  b[0] = __fmul_rn(dd.y, u6f(m));
  b[1] = __fmul_rn(dd.y, u6f(m >> 6));
}
// Q5_K (fields taken as 128 + q): a_j and c_j = 128 a_j + b_j (exact)
__device__ __forceinline__ void q5k_scales(uint32_t dw, uint32_t s, uint32_t m, float* a, float* c) {
  const float2 dd = h2x2f(dw);
  a[0] = __fmul_rn(dd.x, u6f(s));
  a[1] = __fmul_rn(dd.x, u6f(s >> 6));
  c[0] = __fmaf_rn(128.0f, a[0], __fmul_rn(dd.y, u6f(m)));
  c[1] = __fmaf_rn(128.0f, a[1], __fmul_rn(dd.y, u6f(m >> 6)));
}

// the sub-block sums of one Q4_K chunk of rows (g, g+8): words wa, wb (thread t's
// 8 elements of each row), activations b (the same 8 positions, unscaled bf16)
__device__ __forceinline__ void q4k_chunk_mma(float* d, uint32_t wa, uint32_t wb, const uint4 b) {
  const uint32_t ha = wa >> 8, hb = wb >> 8;
  mma_bf16(d, wa & 0x000F000Fu, wb & 0x000F000Fu, wa & 0x00F000F0u, wb & 0x00F000F0u, bmul2(b.x, kX67),
           bmul2(b.y, kX63));
  mma_bf16(d, ha & 0x000F000Fu, hb & 0x000F000Fu, ha & 0x00F000F0u, hb & 0x00F000F0u, bmul2(b.z, kX67),
           bmul2(b.w, kX63));
}
__device__ __forceinline__ void ones_mma(float* xx, const uint4 b) {
  mma_bf16(xx, kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, b.x, b.y);
  mma_bf16(xx, kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, b.z, b.w);
}

template <>
struct Slab<F_Q4_K, 1> {
  // unit j = chunk j in column j: even chunks accumulate in dE, odd ones in dO, so
  // thread t's units 2t, 2t+1 are dE column 2t and dO column 2t+1
  __device__ static void run(const uint8_t* st, const uint8_t*, const uint8_t* xs, int, int w, int lane,
                             float2*, float* acc) {
    const int g = lane >> 2, t = lane & 3;
    const uint8_t* rA = st + (16 * w + g) * 144;
    const uint8_t* rB = rA + 8 * 144;
    const uint32_t xo = 64 * g + 16 * t;                     // unit g = chunk g of token 0
    uint32_t WA[8], WB[8];
    load8(rA + q4k_word_off(t, 0), WA);
    load8(rB + q4k_word_off(t, 0), WB);
    float dE[4] = {0.f, 0.f, 0.f, 0.f}, dO[4] = {0.f, 0.f, 0.f, 0.f}, xx[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) q4k_chunk_mma((j & 1) ? dO : dE, WA[j], WB[j], ldx128(xs, g == j, xo));
    ones_mma(xx, lds128v(xs + xo));
    uint32_t s, m;
    float aA[2], bA[2], aB[2], bB[2];
    q4k_fields_rec(rA, t, &s, &m);
    q4k_scales_lin(lds32(rA), s, m, aA, bA);
    q4k_fields_rec(rB, t, &s, &m);
    q4k_scales_lin(lds32(rB), s, m, aB, bB);
    acc[0] = __fadd_rn(acc[0], kq_comb(aA[0], aA[1], bA[0], bA[1], dE[0], dO[1], xx[0], xx[1]));
    acc[1] = __fadd_rn(acc[1], kq_comb(aB[0], aB[1], bB[0], bB[1], dE[2], dO[3], xx[2], xx[3]));
  }
};

template <>
struct Slab<F_Q4_K, 8> {
  __device__ static void run(const uint8_t* st, const uint8_t*, const uint8_t* xs, int R, int w, int lane,
                             float2* tbl, float (&a)[4][4]) {
    const int g = lane >> 2, tq = lane & 3;
    {   // scale table of the warp's 16 rows: lane -> (row lane/2, sub-blocks 4h..4h+3)
      const int rl = lane >> 1, h = lane & 1;
      const uint4 hd = lds128v(st + (16 * w + rl) * 144);
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        uint32_t s, m;
        float sa[2], sb[2];
        q4k_fields(hd, 2 * h + p, &s, &m);
        q4k_scales_lin(hd.x, s, m, sa, sb);
        tbl[rl * kTblStride + 4 * h + 2 * p] = make_float2(sa[0], sb[0]);
        tbl[rl * kTblStride + 4 * h + 2 * p + 1] = make_float2(sa[1], sb[1]);
      }
    }
    __syncwarp();
    const uint8_t* wA = st + (16 * w + g) * 144 + q4k_word_off(tq, 0);
    const uint8_t* wB = wA + 8 * 144;
    const bool has_x = g < R;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      // the words of chunks 2t, 2t+1 only (fewer live registers than the whole slab's)
      const uint2 WA = lds64(wA + 8 * t), WB = lds64(wB + 8 * t);
      float dd[2][4], xx[2][4];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
#pragma unroll
        for (int e = 0; e < 4; ++e) dd[q][e] = xx[q][e] = 0.f;
        const int j = 2 * t + q;
        const uint4 xv = has_x ? lds128v(xs + 64 * j + 16 * tq) : make_uint4(0u, 0u, 0u, 0u);
        q4k_chunk_mma(dd[q], q ? WA.y : WA.x, q ? WB.y : WB.x, xv);
        ones_mma(xx[q], xv);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = (e < 2) ? g : g + 8;
        const float2 s0 = tbl[row * kTblStride + 2 * t], s1 = tbl[row * kTblStride + 2 * t + 1];
        tc_add(a, t, e, kq_comb(s0.x, s1.x, s0.y, s1.y, dd[0][e], dd[1][e], xx[0][e], xx[1][e]));
      }
    }
    __syncwarp();
  }
};

// ============================================================================
// Q5_K. The Q4_K header (d, dmin, scale stream) with q = 0..31 taken as the exact
// bf16 value A = 128 + q; the pairs come from the 5-bit words plus the chunk's
// nibble word (packed layout: qmv_layout.cuh). sum w x = a_j D_j - c_j X_j with
// D_j = sum A x and c_j = 128 a_j + b_j.
// ============================================================================
// the four pairs {128 + q(8t+2p), 128 + q(8t+2p+1)} of a thread's 5-bit word v;
// u = the chunk's nibble word already shifted right by 4t
__device__ __forceinline__ void q5k_quad(uint32_t v, uint32_t u, uint32_t* a) {
  a[0] = and_or(v, 0x001F001Fu, 0x43004300u);
  a[1] = and_or(v >> 5, 0x001F001Fu, 0x43004300u);
  a[2] = and_or(v >> 10, 0x001F001Fu, 0x43004300u);
  a[3] = and_or(v >> 11, 0x00100010u, and_or(u, 0x000F000Fu, 0x43004300u));
}
__device__ __forceinline__ void q5k_chunk_mma(float* d, const uint32_t* pa, const uint32_t* pb, const uint4 b) {
  mma_bf16(d, pa[0], pb[0], pa[1], pb[1], b.x, b.y);
  mma_bf16(d, pa[2], pb[2], pa[3], pb[3], b.z, b.w);
}

template <>
struct Slab<F_Q5_K, 1> {
  __device__ static void run(const uint8_t* st, const uint8_t*, const uint8_t* xs, int, int w, int lane,
                             float2*, float* acc) {
    const int g = lane >> 2, t = lane & 3;
    const uint8_t* rA = st + (16 * w + g) * 176;
    const uint8_t* rB = rA + 8 * 176;
    const uint32_t xo = 64 * g + 16 * t;                     // unit g = chunk g of token 0
    uint32_t WA[8], WB[8], UA[8], UB[8];
    load8(rA + q5k_word_off(t, 0), WA);
    load8(rB + q5k_word_off(t, 0), WB);
    load8(rA + q5k_nib_off(0), UA);
    load8(rB + q5k_nib_off(0), UB);
    const int us = 4 * t;
    float dE[4] = {0.f, 0.f, 0.f, 0.f}, dO[4] = {0.f, 0.f, 0.f, 0.f}, xx[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t pa[4], pb[4];
      q5k_quad(WA[j], UA[j] >> us, pa);
      q5k_quad(WB[j], UB[j] >> us, pb);
      q5k_chunk_mma((j & 1) ? dO : dE, pa, pb, ldx128(xs, g == j, xo));
    }
    ones_mma(xx, lds128v(xs + xo));
    uint32_t s, m;
    float aA[2], cA[2], aB[2], cB[2];
    q4k_fields_rec(rA, t, &s, &m);
    q5k_scales(lds32(rA), s, m, aA, cA);
    q4k_fields_rec(rB, t, &s, &m);
    q5k_scales(lds32(rB), s, m, aB, cB);
    acc[0] = __fadd_rn(acc[0], kq_comb(aA[0], aA[1], cA[0], cA[1], dE[0], dO[1], xx[0], xx[1]));
    acc[1] = __fadd_rn(acc[1], kq_comb(aB[0], aB[1], cB[0], cB[1], dE[2], dO[3], xx[2], xx[3]));
  }
};

template <>
struct Slab<F_Q5_K, 8> {
  __device__ static void run(const uint8_t* st, const uint8_t*, const uint8_t* xs, int R, int w, int lane,
                             float2* tbl, float (&a)[4][4]) {
    const int g = lane >> 2, tq = lane & 3;
    {   // scale table of the warp's 16 rows: lane -> (row lane/2, sub-blocks 4h..4h+3)
      const int rl = lane >> 1, h = lane & 1;
      const uint4 hd = lds128v(st + (16 * w + rl) * 176);
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        uint32_t s, m;
        float sa[2], sc[2];
        q4k_fields(hd, 2 * h + p, &s, &m);
        q5k_scales(hd.x, s, m, sa, sc);
        tbl[rl * kTblStride + 4 * h + 2 * p] = make_float2(sa[0], sc[0]);
        tbl[rl * kTblStride + 4 * h + 2 * p + 1] = make_float2(sa[1], sc[1]);
      }
    }
    __syncwarp();
    const uint8_t* rA = st + (16 * w + g) * 176;
    const uint8_t* rB = rA + 8 * 176;
    const int us = 4 * tq;
    const bool has_x = g < R;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      // the 5-bit and nibble words of chunks 2t, 2t+1 only (fewer live registers)
      const uint2 wa = lds64(rA + q5k_word_off(tq, 2 * t)), wb = lds64(rB + q5k_word_off(tq, 2 * t));
      const uint2 ua = lds64(rA + q5k_nib_off(2 * t)), ub = lds64(rB + q5k_nib_off(2 * t));
      const uint32_t WA[2] = {wa.x, wa.y}, WB[2] = {wb.x, wb.y};
      const uint32_t UA[2] = {ua.x, ua.y}, UB[2] = {ub.x, ub.y};
      float dd[2][4], xx[2][4];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
#pragma unroll
        for (int e = 0; e < 4; ++e) dd[q][e] = xx[q][e] = 0.f;
        const int j = 2 * t + q;
        uint32_t pa[4], pb[4];
        q5k_quad(WA[q], UA[q] >> us, pa);
        q5k_quad(WB[q], UB[q] >> us, pb);
        const uint4 xv = has_x ? lds128v(xs + 64 * j + 16 * tq) : make_uint4(0u, 0u, 0u, 0u);
        q5k_chunk_mma(dd[q], pa, pb, xv);
        ones_mma(xx[q], xv);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int row = (e < 2) ? g : g + 8;
        const float2 s0 = tbl[row * kTblStride + 2 * t], s1 = tbl[row * kTblStride + 2 * t + 1];
        tc_add(a, t, e, kq_comb(s0.x, s1.x, s0.y, s1.y, dd[0][e], dd[1][e], xx[0][e], xx[1][e]));
      }
    }
    __syncwarp();
  }
};

// ============================================================================
// Q8_0. q = u - 128 with u = 16 uh + ul; lo / hi over (128 + ul) / (128 + uh):
// sum q x = lo + 16 hi - 2304 X; w = d q (d per 32-value chunk).
// ============================================================================
__device__ __forceinline__ void q80_chunk_mma(float* lo, float* hi, uint2 wa, uint2 wb, const uint4 b) {
  mma_bf16(lo, nib_pair(wa.x, 0), nib_pair(wb.x, 0), nib_pair(wa.x, 1), nib_pair(wb.x, 1), b.x, b.y);
  mma_bf16(hi, nib_pair(wa.x, 2), nib_pair(wb.x, 2), nib_pair(wa.x, 3), nib_pair(wb.x, 3), b.x, b.y);
  mma_bf16(lo, nib_pair(wa.y, 0), nib_pair(wb.y, 0), nib_pair(wa.y, 1), nib_pair(wb.y, 1), b.z, b.w);
  mma_bf16(hi, nib_pair(wa.y, 2), nib_pair(wb.y, 2), nib_pair(wa.y, 3), nib_pair(wb.y, 3), b.z, b.w);
}

template <>
struct Slab<F_Q8_0, 1> {
  // unit j = chunk j in column j of the single lo / hi / X accumulators
  __device__ static void run(const uint8_t* st, const uint8_t*, const uint8_t* xs, int, int w, int lane,
                             float2*, float* acc) {
    const int g = lane >> 2, t = lane & 3;
    const uint8_t* rA = st + (16 * w + g) * 272;
    const uint8_t* rB = rA + 8 * 272;
    const uint32_t xo = 64 * g + 16 * t;
    uint32_t WA[16], WB[16];
    load16(rA + q80_word_off(t, 0), WA);
    load16(rB + q80_word_off(t, 0), WB);
    float lo[4] = {0.f, 0.f, 0.f, 0.f}, hi[4] = {0.f, 0.f, 0.f, 0.f}, xx[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j)
      q80_chunk_mma(lo, hi, make_uint2(WA[2 * j], WA[2 * j + 1]), make_uint2(WB[2 * j], WB[2 * j + 1]),
                    ldx128(xs, g == j, xo));
    ones_mma(xx, lds128v(xs + xo));
    const float2 da = h2x2f(lds32(rA + 4 * t)), db = h2x2f(lds32(rB + 4 * t));     // d of chunks 2t, 2t+1
    acc[0] = __fadd_rn(acc[0], q80_comb(da.x, da.y, lo[0], hi[0], xx[0], lo[1], hi[1], xx[1]));
    acc[1] = __fadd_rn(acc[1], q80_comb(db.x, db.y, lo[2], hi[2], xx[2], lo[3], hi[3], xx[3]));
  }
};

template <>
struct Slab<F_Q8_0, 8> {
  __device__ static void run(const uint8_t* st, const uint8_t*, const uint8_t* xs, int R, int w, int lane,
                             float2*, float (&a)[4][4]) {
    const int g = lane >> 2, tq = lane & 3;
    const uint8_t* rA = st + (16 * w + g) * 272;
    const uint8_t* rB = rA + 8 * 272;
    const bool has_x = g < R;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      // the words of chunks 2t, 2t+1 only (fewer live registers than the whole slab's)
      const uint4 WA = lds128v(rA + q80_word_off(tq, 2 * t)), WB = lds128v(rB + q80_word_off(tq, 2 * t));
      float lo[2][4], hi[2][4], xx[2][4];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
#pragma unroll
        for (int e = 0; e < 4; ++e) lo[q][e] = hi[q][e] = xx[q][e] = 0.f;
        const int j = 2 * t + q;
        const uint4 xv = has_x ? lds128v(xs + 64 * j + 16 * tq) : make_uint4(0u, 0u, 0u, 0u);
        q80_chunk_mma(lo[q], hi[q], q ? make_uint2(WA.z, WA.w) : make_uint2(WA.x, WA.y),
                      q ? make_uint2(WB.z, WB.w) : make_uint2(WB.x, WB.y), xv);
        ones_mma(xx[q], xv);
      }
      const float2 da = h2x2f(lds32(rA + 4 * t)), db = h2x2f(lds32(rB + 4 * t));   // d of chunks 2t, 2t+1
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 d = (e < 2) ? da : db;
        tc_add(a, t, e, q80_comb(d.x, d.y, lo[0][e], hi[0][e], xx[0][e], lo[1][e], hi[1][e], xx[1][e]));
      }
    }
    __syncwarp();
  }
};

// ============================================================================
// Q6_K. q = ql + 16 qh, w = a_u (q - 32), a_u = d sc_u per 16-value unit u = 2j + s
// (chunk j, half s). Through bf16's linear range: the low nibbles of pair p of an
// ql word sit at nibbles (p, p+4), their 2-bit highs at bits (2k, 2k+16) of the
// thread's qh word (k = p), so masks alone give exact bf16 values {v, v'} x
// 2^(s - 133): s = 0, 4 for nibble pairs 0, 1 (pairs 2, 3 after one shift by 8) and
// s = 0, 2, 4, 6 for the 2-bit pairs. x is scaled per k position to bring every
// product to (lo + 16 hi) x 2^-66, so the lo and hi MMAs add into sums of one scale:
// lo gets x 2^67 | 2^63, hi x 2^71 | 2^69 (pairs 0, 1) and x 2^67 | 2^65 (pairs 2, 3).
// Exact for |x| < 2^56. sum w x = a_u 2^66 (lo + hi) - 32 a_u X.
// ============================================================================
__device__ __forceinline__ void q6k_linear_mma(float* lo, float* hi, uint32_t la, uint32_t lb, uint32_t ha,
                                               uint32_t hb, int s2, uint2 xv) {
  if (s2 == 0) {
    mma_bf16(lo, la & 0x000F000Fu, lb & 0x000F000Fu, la & 0x00F000F0u, lb & 0x00F000F0u, bmul2(xv.x, kX67),
             bmul2(xv.y, kX63));
    mma_bf16(hi, ha & 0x00030003u, hb & 0x00030003u, ha & 0x000C000Cu, hb & 0x000C000Cu, bmul2(xv.x, kX71),
             bmul2(xv.y, kX69));
  } else {
    const uint32_t la8 = la >> 8, lb8 = lb >> 8;
    mma_bf16(lo, la8 & 0x000F000Fu, lb8 & 0x000F000Fu, la8 & 0x00F000F0u, lb8 & 0x00F000F0u, bmul2(xv.x, kX67),
             bmul2(xv.y, kX63));
    mma_bf16(hi, ha & 0x00300030u, hb & 0x00300030u, ha & 0x00C000C0u, hb & 0x00C000C0u, bmul2(xv.x, kX67),
             bmul2(xv.y, kX65));
  }
}
__device__ __forceinline__ void ones_mma64(float* xx, const uint2 b) {
  mma_bf16(xx, kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, b.x, b.y);
}

template <>
struct Slab<F_Q6_K, 1> {
  // Unit u = 2j + s sits in accumulator group j & 1, column 2(j >> 1) + s, so thread
  // t's columns 2t, 2t+1 hold the units of chunks 2t (group 0) and 2t+1 (group 1):
  // units 4t .. 4t+3. Thread (g', t) carries the activations of the unit in column g'.
  __device__ static void run(const uint8_t* st, const uint8_t* dplane, const uint8_t* xs, int, int w,
                             int lane, float2*, float* acc) {
    const int g = lane >> 2, t = lane & 3;
    const int rowA = 16 * w + g, rowB = rowA + 8;
    const uint8_t* rA = st + rowA * 208;
    const uint8_t* rB = st + rowB * 208;
    const int hsh = 8 * (t & 1);
    // column g of group q: chunk 2(g >> 1) + q, half g & 1
    const uint2 x0 = lds64(xs + 128 * (g >> 1) + 32 * (g & 1) + 8 * t);
    const uint2 x1 = lds64(xs + 128 * (g >> 1) + 64 + 32 * (g & 1) + 8 * t);
    uint32_t LA[8], LB[8], HA[8], HB[8];
    load8(rA + q6k_ql_word_off(t, 0), LA);
    load8(rB + q6k_ql_word_off(t, 0), LB);
    load8(rA + q6k_qh_word_off(t >> 1, 0), HA);
    load8(rB + q6k_qh_word_off(t >> 1, 0), HB);
    float lo[2][4], hi[2][4], xx[2][4];
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e) lo[q][e] = hi[q][e] = xx[q][e] = 0.f;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t ha = HA[j] >> hsh, hb = HB[j] >> hsh;
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        const uint2 xv = ldx64(xs, (2 * (j >> 1) + s2) == g, 64 * j + 32 * s2 + 8 * t);
        q6k_linear_mma(lo[j & 1], hi[j & 1], LA[j], LB[j], ha, hb, s2, xv);
      }
    }
    ones_mma64(xx[0], x0);
    ones_mma64(xx[1], x1);
    const float dA = h2f(*reinterpret_cast<const unsigned short*>(dplane + 2 * rowA));
    const float dB = h2f(*reinterpret_cast<const unsigned short*>(dplane + 2 * rowB));
    const uint32_t scA = lds32(rA + 192 + 4 * t), scB = lds32(rB + 192 + 4 * t);   // units 4t .. 4t+3
    float vA = 0.f, vB = 0.f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int k = 2 * q + e;
        const float aa = __fmul_rn(dA, i8f(scA >> (8 * k))), ab = __fmul_rn(dB, i8f(scB >> (8 * k)));
        vA = q6k_step(vA, q6k_a66(aa), q6k_m32(aa), lo[q][e], hi[q][e], xx[q][e]);
        vB = q6k_step(vB, q6k_a66(ab), q6k_m32(ab), lo[q][2 + e], hi[q][2 + e], xx[q][2 + e]);
      }
    }
    acc[0] = __fadd_rn(acc[0], vA);
    acc[1] = __fadd_rn(acc[1], vB);
  }
};

template <>
struct Slab<F_Q6_K, 8> {
  __device__ static void run(const uint8_t* st, const uint8_t* dplane, const uint8_t* xs, int R, int w,
                             int lane, float2* tbl, float (&a)[4][4]) {
    const int g = lane >> 2, tq = lane & 3;
    {   // scale table of the warp's 16 rows: lane -> (row lane/2, units 8h..8h+7)
      const int rl = lane >> 1, h = lane & 1;
      const int row = 16 * w + rl;
      const float d = h2f(*reinterpret_cast<const unsigned short*>(dplane + 2 * row));
      const uint2 sv = lds64(st + row * 208 + 192 + 8 * h);
      const uint32_t sw[2] = {sv.x, sv.y};
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const float av = __fmul_rn(d, i8f(sw[jj >> 2] >> (8 * (jj & 3))));
        tbl[rl * kTblStride + 8 * h + jj] = make_float2(q6k_a66(av), q6k_m32(av));
      }
    }
    __syncwarp();
    const uint8_t* rA = st + (16 * w + g) * 208;
    const uint8_t* rB = rA + 8 * 208;
    const int hsh = 8 * (tq & 1);
    const bool has_x = g < R;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      // the words of chunks 2t, 2t+1 only (fewer live registers than the whole slab's)
      const uint2 la2 = lds64(rA + q6k_ql_word_off(tq, 2 * t)), lb2 = lds64(rB + q6k_ql_word_off(tq, 2 * t));
      const uint2 ha2 = lds64(rA + q6k_qh_word_off(tq >> 1, 2 * t)), hb2 = lds64(rB + q6k_qh_word_off(tq >> 1, 2 * t));
      float v[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int j = 2 * t + q;
        const uint32_t la = q ? la2.y : la2.x, lb = q ? lb2.y : lb2.x;
        const uint32_t ha = (q ? ha2.y : ha2.x) >> hsh, hb = (q ? hb2.y : hb2.x) >> hsh;
#pragma unroll
        for (int s2 = 0; s2 < 2; ++s2) {
          const int u = 2 * j + s2;
          const uint2 xv = has_x ? lds64(xs + 64 * j + 32 * s2 + 8 * tq) : make_uint2(0u, 0u);
          float lo[4] = {0.f, 0.f, 0.f, 0.f}, hi[4] = {0.f, 0.f, 0.f, 0.f}, xx[4] = {0.f, 0.f, 0.f, 0.f};
          q6k_linear_mma(lo, hi, la, lb, ha, hb, s2, xv);
          ones_mma64(xx, xv);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 s = tbl[((e < 2) ? g : g + 8) * kTblStride + u];
            v[e] = q6k_step(v[e], s.x, s.y, lo[e], hi[e], xx[e]);
          }
        }
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) tc_add(a, t, e, v[e]);
    }
    __syncwarp();
  }
};

// ============================================================================
// NVFP4. The codes go to the MMA as plain e2m1 values (f16) and each 16-value
// block's E4M3 scale multiplies the block sum in fp32; s_T in the epilogue.
// The codes of row r, K chunk j sit in the tensor-core tile at
// (r/8)*1024 + j*128 + (r%8)*16 (thread t reads word t: elements 8t..8t+7, all of
// block t/2 of the chunk); the scales of the row's four blocks of K step ks are one
// 32-bit word of plane B at ks*512 + 16*(r%32) + 4*(r/32). The blocks of chunks 2t,
// 2t+1 (blocks 4t .. 4t+3) are K step t.
// ============================================================================
__device__ __forceinline__ uint32_t nv_code_word_addr_off(int r, int t) { return (r >> 3) * 1024 + (r & 7) * 16 + 4 * t; }
__device__ __forceinline__ uint32_t nv_scale_word_off(int r, int ks) {
  return 512 * ks + 16 * (r & 31) + 4 * (r >> 5);
}

// M = 1: block-separated unit columns. Chunk j's two blocks land in columns
// 2(j/2) and 2(j/2) + 1 of accumulator set j%2, so each of a row's 16 blocks in the
// slab keeps its own output slot. Column c is fed by lanes (c, t): x of chunk pair
// c/2, and only from the lanes whose k positions hold block c%2 of the chunk
// (t/2 == c%2); other lanes feed 0. Lane (g, t) ends with blocks 4t..4t+3 of rows g
// and g + 8: dE columns 2t, 2t+1 (chunk 2t) and dO columns 2t, 2t+1 (chunk 2t+1).
template <>
struct Slab<F_NVFP4, 1> {
  __device__ static void run(const uint8_t* st, const uint8_t* sf, const uint8_t* xs, int, int w, int lane,
                             float2*, float* acc) {
    const int g = lane >> 2, t = lane & 3;
    const int rA = 16 * w + g, rB = rA + 8;
    const int jp = g >> 1;                           // the chunk pair this lane's column serves
    const bool feeds = ((t >> 1) == (g & 1));
    uint32_t xe[4], xo[4];
    {
      const uint4 a = lds128v(xs + 128 * jp + 16 * t);
      const uint4 b = lds128v(xs + 128 * jp + 64 + 16 * t);
      xe[0] = feeds ? bf16x2_to_f16x2(a.x) : 0u;
      xe[1] = feeds ? bf16x2_to_f16x2(a.y) : 0u;
      xe[2] = feeds ? bf16x2_to_f16x2(a.z) : 0u;
      xe[3] = feeds ? bf16x2_to_f16x2(a.w) : 0u;
      xo[0] = feeds ? bf16x2_to_f16x2(b.x) : 0u;
      xo[1] = feeds ? bf16x2_to_f16x2(b.y) : 0u;
      xo[2] = feeds ? bf16x2_to_f16x2(b.z) : 0u;
      xo[3] = feeds ? bf16x2_to_f16x2(b.w) : 0u;
    }
    uint32_t CA[8], CB[8];
    {
      const uint8_t* ca = st + nv_code_word_addr_off(rA, t);
      const uint8_t* cb = st + nv_code_word_addr_off(rB, t);
#pragma unroll
      for (int j = 0; j < 8; ++j) { CA[j] = lds32(ca + 128 * j); CB[j] = lds32(cb + 128 * j); }
    }
    float dE[4] = {0.f, 0.f, 0.f, 0.f}, dO[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      // the B operand is x only in the chunk pair this lane's column serves: zeroed by a
      // multiply with an f16x2 {1, 1} / {0, 0} mask on the FMA pipe (x is finite),
      // which keeps the ALU pipe for the decode
      const uint32_t mk = ((j >> 1) == jp) ? 0x3C003C00u : 0u;
      const uint32_t* xv = (j & 1) ? xo : xe;
      float* d = (j & 1) ? dO : dE;
      uint32_t pa[4], pb[4];
      e2m1x4_f16(CA[j], pa);
      e2m1x4_f16(CB[j], pb);
      mma_f16(d, pa[0], pb[0], pa[1], pb[1], hmul2(xv[0], mk), hmul2(xv[1], mk));
      mma_f16(d, pa[2], pb[2], pa[3], pb[3], hmul2(xv[2], mk), hmul2(xv[3], mk));
    }
    uint32_t hA[2], hB[2];
    e4m3x4_f16(lds32(sf + nv_scale_word_off(rA, t)), hA);
    e4m3x4_f16(lds32(sf + nv_scale_word_off(rB, t)), hB);
    const float2 a01 = h2x2f(hA[0]), a23 = h2x2f(hA[1]);
    const float2 b01 = h2x2f(hB[0]), b23 = h2x2f(hB[1]);
    acc[0] = __fadd_rn(acc[0], nv_comb(a01.x, a01.y, a23.x, a23.y, dE[0], dE[1], dO[0], dO[1]));
    acc[1] = __fadd_rn(acc[1], nv_comb(b01.x, b01.y, b23.x, b23.y, dE[2], dE[3], dO[2], dO[3]));
  }
};

// M > 1: token columns; each block of a chunk has its own MMA chain, whose B operand
// keeps x only on the lanes holding that block (t/2 == block), as in the unit columns.
template <>
struct Slab<F_NVFP4, 8> {
  __device__ static void run(const uint8_t* st, const uint8_t* sf, const uint8_t* xs, int R, int w, int lane,
                             float2*, float (&a)[4][4]) {
    const int g = lane >> 2, tq = lane & 3;
    const int rA = 16 * w + g, rB = rA + 8;
    const bool has_x = g < R;
    const uint8_t* ca = st + nv_code_word_addr_off(rA, tq);
    const uint8_t* cb = st + nv_code_word_addr_off(rB, tq);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      float D[2][2][4];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int j = 2 * t + q;
        // x already f16 (converted per stage)
        const uint4 xv = has_x ? lds128v(xs + 64 * j + 16 * tq) : make_uint4(0u, 0u, 0u, 0u);
        uint32_t pa[4], pb[4];
        e2m1x4_f16(lds32(ca + 128 * j), pa);
        e2m1x4_f16(lds32(cb + 128 * j), pb);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          const bool on = (tq >> 1) == b;
          const uint4 xb = on ? xv : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
          for (int e = 0; e < 4; ++e) D[q][b][e] = 0.f;
          mma_f16(D[q][b], pa[0], pb[0], pa[1], pb[1], xb.x, xb.y);
          mma_f16(D[q][b], pa[2], pb[2], pa[3], pb[3], xb.z, xb.w);
        }
      }
      uint32_t hA[2], hB[2];
      e4m3x4_f16(lds32(sf + nv_scale_word_off(rA, t)), hA);
      e4m3x4_f16(lds32(sf + nv_scale_word_off(rB, t)), hB);
      const float2 a01 = h2x2f(hA[0]), a23 = h2x2f(hA[1]);
      const float2 b01 = h2x2f(hB[0]), b23 = h2x2f(hB[1]);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 s01 = (e < 2) ? a01 : b01, s23 = (e < 2) ? a23 : b23;
        tc_add(a, t, e, nv_comb(s01.x, s01.y, s23.x, s23.y, D[0][0][e], D[0][1][e], D[1][0][e], D[1][1][e]));
      }
    }
  }
};

// ============================================================================
// FP8 row-scaled. A = e4m3 in f16 (exact), B = x in f16; s_row in the epilogue.
// The thread's 8 values of chunk j are bytes 8(t&1).. of 16-byte vector 2j + t/2.
// ============================================================================
__device__ __forceinline__ void fp8_chunk_mma(float* d, uint2 ca, uint2 cb, uint32_t x0, uint32_t x1, uint32_t x2,
                                              uint32_t x3) {
  uint32_t a0[2], b0[2], a1[2], b1[2];
  e4m3x4_f16(ca.x, a0);
  e4m3x4_f16(cb.x, b0);
  e4m3x4_f16(ca.y, a1);
  e4m3x4_f16(cb.y, b1);
  mma_f16(d, a0[0], b0[0], a0[1], b0[1], x0, x1);
  mma_f16(d, a1[0], b1[0], a1[1], b1[1], x2, x3);
}

template <>
struct Slab<F_FP8, 1> {
  // unit j = chunk j in column j: thread t's units 2t, 2t+1 are dE column 2t and dO
  // column 2t+1
  __device__ static void run(const uint8_t* st, const uint8_t*, const uint8_t* xs, int, int w, int lane,
                             float2*, float* acc) {
    const int g = lane >> 2, t = lane & 3;
    const int rowA = 16 * w + g, rowB = rowA + 8;
    const uint8_t* rA = st + rowA * 256 + 8 * (t & 1);
    const uint8_t* rB = st + rowB * 256 + 8 * (t & 1);
    const uint4 xr = lds128v(xs + 64 * g + 16 * t);
    const uint32_t x0 = bf16x2_to_f16x2(xr.x), x1 = bf16x2_to_f16x2(xr.y);
    const uint32_t x2 = bf16x2_to_f16x2(xr.z), x3 = bf16x2_to_f16x2(xr.w);
    float dE[4] = {0.f, 0.f, 0.f, 0.f}, dO[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int v = 2 * j + (t >> 1);
      const bool mine = (g == j);
      fp8_chunk_mma((j & 1) ? dO : dE, lds64(rA + fp8_v_off(v, rowA & 7)), lds64(rB + fp8_v_off(v, rowB & 7)),
                    sel(mine, x0), sel(mine, x1), sel(mine, x2), sel(mine, x3));
    }
    acc[0] = __fadd_rn(acc[0], fp8_comb(dE[0], dO[1]));
    acc[1] = __fadd_rn(acc[1], fp8_comb(dE[2], dO[3]));
  }
};

template <>
struct Slab<F_FP8, 8> {
  __device__ static void run(const uint8_t* st, const uint8_t*, const uint8_t* xs, int R, int w, int lane,
                             float2*, float (&a)[4][4]) {
    const int g = lane >> 2, tq = lane & 3;
    const int rowA = 16 * w + g, rowB = rowA + 8;
    const uint8_t* rA = st + rowA * 256 + 8 * (tq & 1);
    const uint8_t* rB = st + rowB * 256 + 8 * (tq & 1);
    const bool has_x = g < R;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      float D[2][4];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int j = 2 * t + q;
        const int v = 2 * j + (tq >> 1);
        // x already f16 (converted per stage)
        const uint4 xv = has_x ? lds128v(xs + 64 * j + 16 * tq) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int e = 0; e < 4; ++e) D[q][e] = 0.f;
        fp8_chunk_mma(D[q], lds64(rA + fp8_v_off(v, rowA & 7)), lds64(rB + fp8_v_off(v, rowB & 7)), xv.x, xv.y,
                      xv.z, xv.w);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) tc_add(a, t, e, fp8_comb(D[0][e], D[1][e]));
    }
  }
};

// ============================================================================
// IQ4_XS. A weight is the matrix's codebook entry C[q] (16 x int8) times the
// sub-block scale a_j = d (ls_j - 32) of its 32-value chunk. The decode is a
// lookup in registers: the table bytes C + 128 sit in four registers; one prmt
// picks the bytes of indices 0..7 and one those of indices 8..15 (three selector
// bits each), and a third, driven by the top bit of each index, selects between
// them. One more prmt per pair places two table bytes b under the f16 pattern 0x64
// (1024 + b), so each A register holds {1152 + C[q], 1152 + C[q']} exactly. x goes
// to the MMA in f16; sum C x = D - 1152 X with X = sum x.
// ============================================================================
constexpr uint32_t kOnesF16 = 0x3C003C00u;

__device__ __forceinline__ void iq4_table(const uint8_t* cbp, uint32_t (&T)[4]) {
  const uint4 c = lds128v(cbp);
  T[0] = c.x ^ 0x80808080u;
  T[1] = c.y ^ 0x80808080u;
  T[2] = c.z ^ 0x80808080u;
  T[3] = c.w ^ 0x80808080u;
}
// the table bytes of the four indices in the low 16 bits of s (index i at nibble i)
__device__ __forceinline__ uint32_t iq4_look4(uint32_t s, const uint32_t (&T)[4]) {
  const uint32_t s7 = s & 0x7777u;
  const uint32_t lo = __byte_perm(T[0], T[1], s7), hi = __byte_perm(T[2], T[3], s7);
  const uint32_t m = __byte_perm(0x0000FF00u, 0u, (s >> 3) & 0x1111u);   // 0xFF where index >= 8
  return (lo & ~m) | (hi & m);
}
// word w (elements 0..7 at nibbles 0..7) -> the A registers {e0,e1}, {e2,e3}, {e4,e5}, {e6,e7}
__device__ __forceinline__ void iq4_word(uint32_t w, const uint32_t (&T)[4], uint32_t* p) {
  const uint32_t v0 = iq4_look4(w, T), v1 = iq4_look4(w >> 16, T);
  p[0] = __byte_perm(v0, 0x64646464u, 0x4140);
  p[1] = __byte_perm(v0, 0x64646464u, 0x4342);
  p[2] = __byte_perm(v1, 0x64646464u, 0x4140);
  p[3] = __byte_perm(v1, 0x64646464u, 0x4342);
}
__device__ __forceinline__ void iq4_chunk_mma(float* d, uint32_t wa, uint32_t wb, const uint32_t (&T)[4],
                                              uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3) {
  uint32_t pa[4], pb[4];
  iq4_word(wa, T, pa);
  iq4_word(wb, T, pb);
  mma_f16(d, pa[0], pb[0], pa[1], pb[1], x0, x1);
  mma_f16(d, pa[2], pb[2], pa[3], pb[3], x2, x3);
}
__device__ __forceinline__ void ones_mma_f16(float* xx, uint32_t x0, uint32_t x1, uint32_t x2, uint32_t x3) {
  mma_f16(xx, kOnesF16, kOnesF16, kOnesF16, kOnesF16, x0, x1);
  mma_f16(xx, kOnesF16, kOnesF16, kOnesF16, kOnesF16, x2, x3);
}
// a_j = d (ls_j - 32) of chunks 2t, 2t+1 from a row's scale fields (fp16 d, u16 sh, u32 sl)
__device__ __forceinline__ void iq4_scales(const uint8_t* sf, int t, float* a) {
  const uint2 v = lds64(sf);
  const float d = h2f(v.x);
  const uint32_t sh = (v.x >> 16) >> (4 * t), sl = v.y >> (8 * t);
  a[0] = __fmul_rn(d, (float)((int)((sl & 15u) | ((sh & 3u) << 4)) - 32));
  a[1] = __fmul_rn(d, (float)((int)(((sl >> 4) & 15u) | (((sh >> 2) & 3u) << 4)) - 32));
}

template <>
struct Slab<F_IQ4_XS, 1> {
  // unit j = chunk j in column j: even chunks accumulate in dE, odd ones in dO, so
  // position t's units 2t, 2t+1 are dE column 2t and dO column 2t+1
  __device__ static void run(const uint8_t* st, const uint8_t* pb, const uint8_t* xs, int, int w, int lane,
                             float2*, float* acc) {
    const int g = lane >> 2, t = lane & 3;
    const int rowA = 16 * w + g, rowB = rowA + 8;   // both at rotation g (row & 7)
    const uint8_t* rA = st + rowA * 128;
    const uint8_t* rB = st + rowB * 128;
    uint32_t T[4];
    iq4_table(pb + 128 * 8, T);
    const uint4 xr = lds128v(xs + 64 * g + 16 * t);   // the lane's unit: chunk g, elements 8t..8t+7
    const uint32_t x0 = bf16x2_to_f16x2(xr.x), x1 = bf16x2_to_f16x2(xr.y);
    const uint32_t x2 = bf16x2_to_f16x2(xr.z), x3 = bf16x2_to_f16x2(xr.w);
    const uint4 a0 = lds128v(rA + 16 * ((2 * t) ^ g)), a1 = lds128v(rA + 16 * ((2 * t + 1) ^ g));
    const uint4 b0 = lds128v(rB + 16 * ((2 * t) ^ g)), b1 = lds128v(rB + 16 * ((2 * t + 1) ^ g));
    const uint32_t WA[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const uint32_t WB[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    float dE[4] = {0.f, 0.f, 0.f, 0.f}, dO[4] = {0.f, 0.f, 0.f, 0.f}, xx[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      // B is x only in the column of chunk j: an f16x2 {1, 1} / {0, 0} mask multiply on
      // the FMA pipe (x is finite), which keeps the ALU pipe for the lookups
      const uint32_t mk = (g == j) ? kOnesF16 : 0u;
      iq4_chunk_mma((j & 1) ? dO : dE, WA[j], WB[j], T, hmul2(x0, mk), hmul2(x1, mk), hmul2(x2, mk),
                    hmul2(x3, mk));
    }
    ones_mma_f16(xx, x0, x1, x2, x3);
    float aA[2], aB[2];
    iq4_scales(pb + rowA * 8, t, aA);
    iq4_scales(pb + rowB * 8, t, aB);
    acc[0] = __fadd_rn(acc[0], iq4_comb(aA[0], aA[1], dE[0], dO[1], xx[0], xx[1]));
    acc[1] = __fadd_rn(acc[1], iq4_comb(aB[0], aB[1], dE[2], dO[3], xx[2], xx[3]));
  }
};

template <>
struct Slab<F_IQ4_XS, 8> {
  __device__ static void run(const uint8_t* st, const uint8_t* pb, const uint8_t* xs, int R, int w, int lane,
                             float2*, float (&a)[4][4]) {
    const int g = lane >> 2, tq = lane & 3;
    const int rowA = 16 * w + g, rowB = rowA + 8;
    const uint8_t* rA = st + rowA * 128;
    const uint8_t* rB = st + rowB * 128;
    const bool has_x = g < R;
    uint32_t T[4];
    iq4_table(pb + 128 * 8, T);
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      // the words of chunks 2t, 2t+1: vector 2tq + (t >> 1) (rotated by g), words 2(t & 1), +1
      const int v = (2 * tq + (t >> 1)) ^ g;
      const uint2 WA = lds64(rA + 16 * v + 8 * (t & 1)), WB = lds64(rB + 16 * v + 8 * (t & 1));
      float D[2][4], X[2][4];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
#pragma unroll
        for (int e = 0; e < 4; ++e) D[q][e] = X[q][e] = 0.f;
        const int j = 2 * t + q;
        // x already f16 (converted per stage)
        const uint4 xv = has_x ? lds128v(xs + 64 * j + 16 * tq) : make_uint4(0u, 0u, 0u, 0u);
        iq4_chunk_mma(D[q], q ? WA.y : WA.x, q ? WB.y : WB.x, T, xv.x, xv.y, xv.z, xv.w);
        ones_mma_f16(X[q], xv.x, xv.y, xv.z, xv.w);
      }
      float sA[2], sB[2];
      iq4_scales(pb + rowA * 8, t, sA);
      iq4_scales(pb + rowB * 8, t, sB);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float* sc = (e < 2) ? sA : sB;
        tc_add(a, t, e, iq4_comb(sc[0], sc[1], D[0][e], D[1][e], X[0][e], X[1][e]));
      }
    }
  }
};

// ============================================================================
// IQ3_S, IQ2_S. A group of weights is one entry of the format's grid, kept in shared
// memory as f16 magnitudes, with one sign bit per weight: w = a G[idx][i] (+-), a =
// d (2 sc + 1) per 32 (IQ3_S) / 16 (IQ2_S) values. The MMA of slot m = 2j + s (chunk
// j, half s) covers elements 32j + 16s + 4t .. +3 in thread t: one IQ3_S group, half
// an IQ2_S group. Its four magnitudes are one 8-byte shared-memory load (two f16
// pairs); its four sign bits are spread onto the pairs' sign bits with one multiply
// each (no carries: the two shifted copies of the nibble do not overlap) and applied
// with one AND-XOR. x goes to the MMA in f16.
// ============================================================================
__device__ __forceinline__ uint32_t lds16(const void* p) { return *reinterpret_cast<const unsigned short*>(p); }

// the two A registers of a slot: grid entry bytes at e (4 f16), sign nibble nib
__device__ __forceinline__ void grid_slot(const uint8_t* e, uint32_t nib, uint32_t& p01, uint32_t& p23) {
  const uint2 v = lds64(e);
  p01 = v.x ^ ((nib * 0x40008000u) & 0x80008000u);   // sign bits 0, 1 -> bits 15, 31
  p23 = v.y ^ ((nib * 0x10002000u) & 0x80008000u);   // sign bits 2, 3 -> bits 15, 31
}
// index low byte m of a 16-byte vector (4 words), compile-time m
__device__ __forceinline__ uint32_t byte_of(const uint32_t (&Q)[4], int m) { return (Q[m >> 2] >> (8 * (m & 3))) & 0xFFu; }

template <>
struct Slab<F_IQ3_S, 1> {
  // unit j = chunk j in column j: even chunks accumulate in dE, odd ones in dO, so
  // position t's units 2t, 2t+1 are dE column 2t and dO column 2t+1
  __device__ static void run(const uint8_t* st, const uint8_t* pb, const uint8_t* xs, int, int w, int lane,
                             float2* gtab, float* acc) {
    const int g = lane >> 2, t = lane & 3;
    const uint8_t* G = reinterpret_cast<const uint8_t*>(gtab);   // 512 entries x 4 f16 (8 B)
    const int rowA = 16 * w + g, rowB = rowA + 8;
    const uint8_t* rA = st + rowA * 96;
    const uint8_t* rB = st + rowB * 96;
    const uint8_t* bA = pb + rowA * 14;
    const uint8_t* bB = pb + rowB * 14;
    // the lane's unit: chunk g, elements 16s + 4t .. +3 (s = 0, 1)
    const uint2 xa = lds64(xs + 64 * g + 8 * t), xb = lds64(xs + 64 * g + 32 + 8 * t);
    const uint32_t x0 = bf16x2_to_f16x2(xa.x), x1 = bf16x2_to_f16x2(xa.y);
    const uint32_t x2 = bf16x2_to_f16x2(xb.x), x3 = bf16x2_to_f16x2(xb.y);
    const uint4 qa = lds128v(rA + 16 * t), qb = lds128v(rB + 16 * t);
    const uint32_t QA[4] = {qa.x, qa.y, qa.z, qa.w}, QB[4] = {qb.x, qb.y, qb.z, qb.w};
    const uint2 sA = lds64(rA + 64 + 8 * t), sB = lds64(rB + 64 + 8 * t);
    const uint32_t hA = lds16(bA + 6 + 2 * t), hB = lds16(bB + 6 + 2 * t);
    float dE[4] = {0.f, 0.f, 0.f, 0.f}, dO[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const int j = m >> 1, sh = m & 1;
      const uint32_t mk = (g == j) ? kOnesF16 : 0u;
      const uint32_t iA = byte_of(QA, m) | (((hA >> m) & 1u) << 8), iB = byte_of(QB, m) | (((hB >> m) & 1u) << 8);
      const uint32_t nA = ((m < 8 ? sA.x : sA.y) >> (4 * (m & 7))) & 15u;
      const uint32_t nB = ((m < 8 ? sB.x : sB.y) >> (4 * (m & 7))) & 15u;
      uint32_t a01, a23, b01, b23;
      grid_slot(G + 8 * iA, nA, a01, a23);
      grid_slot(G + 8 * iB, nB, b01, b23);
      mma_f16((j & 1) ? dO : dE, a01, b01, a23, b23, hmul2(sh ? x2 : x0, mk), hmul2(sh ? x3 : x1, mk));
    }
    const float dA = h2f(lds16(bA)), dB = h2f(lds16(bB));
    const uint32_t cA = bA[2 + t], cB = bB[2 + t];                  // scales of chunks 2t, 2t+1
    const float aA0 = __fmul_rn(dA, (float)(2 * (int)(cA & 15u) + 1)), aA1 = __fmul_rn(dA, (float)(2 * (int)(cA >> 4) + 1));
    const float aB0 = __fmul_rn(dB, (float)(2 * (int)(cB & 15u) + 1)), aB1 = __fmul_rn(dB, (float)(2 * (int)(cB >> 4) + 1));
    acc[0] = __fadd_rn(acc[0], grid_comb(aA0, aA1, dE[0], dO[1]));
    acc[1] = __fadd_rn(acc[1], grid_comb(aB0, aB1, dE[2], dO[3]));
  }
};

template <>
struct Slab<F_IQ3_S, 8> {
  __device__ static void run(const uint8_t* st, const uint8_t* pb, const uint8_t* xs, int R, int w, int lane,
                             float2* gtab, float (&a)[4][4]) {
    const int g = lane >> 2, tq = lane & 3;
    const uint8_t* G = reinterpret_cast<const uint8_t*>(gtab);
    const int rowA = 16 * w + g, rowB = rowA + 8;
    const uint8_t* rA = st + rowA * 96;
    const uint8_t* rB = st + rowB * 96;
    const uint8_t* bA = pb + rowA * 14;
    const uint8_t* bB = pb + rowB * 14;
    const bool has_x = g < R;
    const uint4 qa = lds128v(rA + 16 * tq), qb = lds128v(rB + 16 * tq);
    const uint32_t QA[4] = {qa.x, qa.y, qa.z, qa.w}, QB[4] = {qb.x, qb.y, qb.z, qb.w};
    const uint2 sA = lds64(rA + 64 + 8 * tq), sB = lds64(rB + 64 + 8 * tq);
    const uint32_t hA = lds16(bA + 6 + 2 * tq), hB = lds16(bB + 6 + 2 * tq);
    const float dA = h2f(lds16(bA)), dB = h2f(lds16(bB));
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      float D[2][4];
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int j = 2 * t + q;
#pragma unroll
        for (int e = 0; e < 4; ++e) D[q][e] = 0.f;
#pragma unroll
        for (int sh = 0; sh < 2; ++sh) {
          const int m = 2 * j + sh;
          // x already f16 (converted per stage)
          const uint2 xv = has_x ? lds64(xs + 64 * j + 32 * sh + 8 * tq) : make_uint2(0u, 0u);
          const uint32_t iA = byte_of(QA, m) | (((hA >> m) & 1u) << 8), iB = byte_of(QB, m) | (((hB >> m) & 1u) << 8);
          const uint32_t nA = ((m < 8 ? sA.x : sA.y) >> (4 * (m & 7))) & 15u;
          const uint32_t nB = ((m < 8 ? sB.x : sB.y) >> (4 * (m & 7))) & 15u;
          uint32_t a01, a23, b01, b23;
          grid_slot(G + 8 * iA, nA, a01, a23);
          grid_slot(G + 8 * iB, nB, b01, b23);
          mma_f16(D[q], a01, b01, a23, b23, xv.x, xv.y);
        }
      }
      const uint32_t cA = bA[2 + t], cB = bB[2 + t];
      const float sA0 = __fmul_rn(dA, (float)(2 * (int)(cA & 15u) + 1)), sA1 = __fmul_rn(dA, (float)(2 * (int)(cA >> 4) + 1));
      const float sB0 = __fmul_rn(dB, (float)(2 * (int)(cB & 15u) + 1)), sB1 = __fmul_rn(dB, (float)(2 * (int)(cB >> 4) + 1));
#pragma unroll
      for (int e = 0; e < 4; ++e)
        tc_add(a, t, e, (e < 2) ? grid_comb(sA0, sA1, D[0][e], D[1][e]) : grid_comb(sB0, sB1, D[0][e], D[1][e]));
    }
  }
};

template <>
struct Slab<F_IQ2_S, 1> {
  // Unit u = 2j + s (16 values) sits in accumulator group j & 1, column 2(j >> 1) + s
  // (as Q6_K): position t's columns 2t, 2t+1 hold units 4t .. 4t+3. Thread (g', t)
  // carries the activations of the unit in column g'.
  __device__ static void run(const uint8_t* st, const uint8_t* pb, const uint8_t* xs, int, int w, int lane,
                             float2* gtab, float* acc) {
    const int g = lane >> 2, t = lane & 3, p = t >> 1;
    const uint8_t* G = reinterpret_cast<const uint8_t*>(gtab) + 8 * (t & 1);   // 1024 entries x 8 f16 (16 B)
    const int rowA = 16 * w + g, rowB = rowA + 8;
    const uint8_t* rA = st + rowA * 64;
    const uint8_t* rB = st + rowB * 64;
    const uint8_t* bA = pb + rowA * 18;
    const uint8_t* bB = pb + rowB * 18;
    // column g of group q: chunk 2(g >> 1) + q, half g & 1, elements 4t .. 4t+3
    const uint2 xa = lds64(xs + 128 * (g >> 1) + 32 * (g & 1) + 8 * t);
    const uint2 xb = lds64(xs + 128 * (g >> 1) + 64 + 32 * (g & 1) + 8 * t);
    const uint32_t x0 = bf16x2_to_f16x2(xa.x), x1 = bf16x2_to_f16x2(xa.y);
    const uint32_t x2 = bf16x2_to_f16x2(xb.x), x3 = bf16x2_to_f16x2(xb.y);
    const uint4 qa = lds128v(rA + 16 * p), qb = lds128v(rB + 16 * p);
    const uint32_t QA[4] = {qa.x, qa.y, qa.z, qa.w}, QB[4] = {qb.x, qb.y, qb.z, qb.w};
    const uint2 sA = lds64(rA + 32 + 8 * t), sB = lds64(rB + 32 + 8 * t);
    const uint32_t hA = lds16(bA + 10 + 4 * p) | (lds16(bA + 12 + 4 * p) << 16);
    const uint32_t hB = lds16(bB + 10 + 4 * p) | (lds16(bB + 12 + 4 * p) << 16);
    float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int m = 0; m < 16; ++m) {
      const int j = m >> 1, sh = m & 1;
      const uint32_t mk = ((2 * (j >> 1) + sh) == g) ? kOnesF16 : 0u;
      const uint32_t iA = byte_of(QA, m) | (((hA >> (2 * m)) & 3u) << 8), iB = byte_of(QB, m) | (((hB >> (2 * m)) & 3u) << 8);
      const uint32_t nA = ((m < 8 ? sA.x : sA.y) >> (4 * (m & 7))) & 15u;
      const uint32_t nB = ((m < 8 ? sB.x : sB.y) >> (4 * (m & 7))) & 15u;
      uint32_t a01, a23, b01, b23;
      grid_slot(G + 16 * iA, nA, a01, a23);
      grid_slot(G + 16 * iB, nB, b01, b23);
      mma_f16((j & 1) ? d1 : d0, a01, b01, a23, b23, hmul2((j & 1) ? x2 : x0, mk), hmul2((j & 1) ? x3 : x1, mk));
    }
    const float dA = h2f(lds16(bA)), dB = h2f(lds16(bB));
    const uint32_t cA = lds16(bA + 2 + 2 * t), cB = lds16(bB + 2 + 2 * t);   // scales of units 4t .. 4t+3
    float aA[4], aB[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      aA[k] = __fmul_rn(dA, (float)(2 * (int)((cA >> (4 * k)) & 15u) + 1));
      aB[k] = __fmul_rn(dB, (float)(2 * (int)((cB >> (4 * k)) & 15u) + 1));
    }
    acc[0] = __fadd_rn(acc[0], grid16_comb(aA[0], aA[1], aA[2], aA[3], d0[0], d0[1], d1[0], d1[1]));
    acc[1] = __fadd_rn(acc[1], grid16_comb(aB[0], aB[1], aB[2], aB[3], d0[2], d0[3], d1[2], d1[3]));
  }
};

template <>
struct Slab<F_IQ2_S, 8> {
  __device__ static void run(const uint8_t* st, const uint8_t* pb, const uint8_t* xs, int R, int w, int lane,
                             float2* gtab, float (&a)[4][4]) {
    const int g = lane >> 2, tq = lane & 3, p = tq >> 1;
    const uint8_t* G = reinterpret_cast<const uint8_t*>(gtab) + 8 * (tq & 1);
    const int rowA = 16 * w + g, rowB = rowA + 8;
    const uint8_t* rA = st + rowA * 64;
    const uint8_t* rB = st + rowB * 64;
    const uint8_t* bA = pb + rowA * 18;
    const uint8_t* bB = pb + rowB * 18;
    const bool has_x = g < R;
    const uint4 qa = lds128v(rA + 16 * p), qb = lds128v(rB + 16 * p);
    const uint32_t QA[4] = {qa.x, qa.y, qa.z, qa.w}, QB[4] = {qb.x, qb.y, qb.z, qb.w};
    const uint2 sA = lds64(rA + 32 + 8 * tq), sB = lds64(rB + 32 + 8 * tq);
    const uint32_t hA = lds16(bA + 10 + 4 * p) | (lds16(bA + 12 + 4 * p) << 16);
    const uint32_t hB = lds16(bB + 10 + 4 * p) | (lds16(bB + 12 + 4 * p) << 16);
    const float dA = h2f(lds16(bA)), dB = h2f(lds16(bB));
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      float D[4][4];            // units 4t .. 4t+3 = slots m = 4t .. 4t+3
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int m = 4 * t + k, j = m >> 1, sh = m & 1;
#pragma unroll
        for (int e = 0; e < 4; ++e) D[k][e] = 0.f;
        // x already f16 (converted per stage)
        const uint2 xv = has_x ? lds64(xs + 64 * j + 32 * sh + 8 * tq) : make_uint2(0u, 0u);
        const uint32_t iA = byte_of(QA, m) | (((hA >> (2 * m)) & 3u) << 8), iB = byte_of(QB, m) | (((hB >> (2 * m)) & 3u) << 8);
        const uint32_t nA = ((m < 8 ? sA.x : sA.y) >> (4 * (m & 7))) & 15u;
        const uint32_t nB = ((m < 8 ? sB.x : sB.y) >> (4 * (m & 7))) & 15u;
        uint32_t a01, a23, b01, b23;
        grid_slot(G + 16 * iA, nA, a01, a23);
        grid_slot(G + 16 * iB, nB, b01, b23);
        mma_f16(D[k], a01, b01, a23, b23, xv.x, xv.y);
      }
      const uint32_t cA = lds16(bA + 2 + 2 * t), cB = lds16(bB + 2 + 2 * t);
      float sA4[4], sB4[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        sA4[k] = __fmul_rn(dA, (float)(2 * (int)((cA >> (4 * k)) & 15u) + 1));
        sB4[k] = __fmul_rn(dB, (float)(2 * (int)((cB >> (4 * k)) & 15u) + 1));
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float* sc = (e < 2) ? sA4 : sB4;
        tc_add(a, t, e, grid16_comb(sc[0], sc[1], sc[2], sc[3], D[0][e], D[1][e], D[2][e], D[3][e]));
      }
    }
  }
};

}  // namespace qmv
