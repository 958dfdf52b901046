// qmv_slab.cuh -- per-format decode + tensor-core inner product of one slab
// (128 rows x 256 values of packed weights, already in shared memory).
//
// A consumer warp w owns rows 16w .. 16w+15 of the slab. The inner product runs
// on mma.sync m16n8k16 with the weight rows as the 16-row A operand; the weights
// are decoded in registers straight into A fragments:
//   K-quants -> bf16:  one AND-OR per two 4-bit fields gives {128 + q_lo, 128 + q_hi}
//                      exactly (the packed layout stores element pairs at nibbles
//                      (p, p+4) of each 32-bit word); the +128 offset is removed with
//                      the per-block min term through X = sum x.
//   NVFP4, FP8 -> f16: hardware cvt of FP4/FP8 pairs to f16x2 (exact); for NVFP4 the
//                      E4M3 block scale is multiplied in with one exact f16x2 multiply.
// Products of these small exact values with the activations are exact and the
// tensor core accumulates in fp32.
//
// The 8 columns of the mma output are used in one of two ways:
//   M = 1 ("unit columns"): column n holds the partial sum of sub-block (unit) n
//     of the slab. A thread's B registers carry activations only for its own unit,
//     zero elsewhere, so one accumulator collects all 8 units' partial sums at once
//     and each block scale is applied once per slab. A thread (g, t) ends with the
//     partial sums of rows g, g+8 over units 2t, 2t+1; the four threads of a quad
//     are added at the end of the row tile.
//   M = 2..8 ("token columns"): column n is token n; each 32-value sub-block gets
//     its own accumulator and its scale is applied per sub-block. Thread (g, t)
//     holds rows g, g+8 x tokens 2t, 2t+1.
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

// ============================================================================
// Q4_K. w = a_j q - b_j (a_j = d sc_j, b_j = dmin m_j, sub-block j = 32 values);
// with A = 128 + q: sum w x = a_j D_j - c_j X_j, c_j = 128 a_j + b_j.
// ============================================================================
__device__ __forceinline__ void q4k_pair_scales(const uint4 hd, int t, float* a, float* c) {
  // sc_j, m_j of sub-blocks j = 2t, 2t+1 (12 consecutive bits each)
  const float2 dd = h2x2f(hd.x);
  const uint64_t lo = ((uint64_t)hd.z << 32) | hd.y, hi = ((uint64_t)hd.w << 32) | hd.z;
  const uint32_t s = (uint32_t)(lo >> (12 * t)), m = (uint32_t)(hi >> (16 + 12 * t));
  a[0] = dd.x * u6f(s);
  a[1] = dd.x * u6f(s >> 6);
  c[0] = fmaf(128.0f, a[0], dd.y * u6f(m));
  c[1] = fmaf(128.0f, a[1], dd.y * u6f(m >> 6));
}
// the same from a record in shared memory: the scale stream starts at byte 4 and
// the fields of sub-blocks 2t, 2t+1 sit at stream bits 12t (sc) and 48 + 12t (m);
// each pair is taken from two aligned 32-bit words with one funnel shift
__device__ __forceinline__ void q4k_pair_scales_rec(const uint8_t* rec, int t, float* a, float* c) {
  const uint32_t* sw = reinterpret_cast<const uint32_t*>(rec + 4);
  const int bs = 12 * t, bm = 48 + 12 * t;
  const uint32_t s = __funnelshift_r(sw[bs >> 5], sw[(bs >> 5) + 1], bs & 31);
  const uint32_t m = __funnelshift_r(sw[bm >> 5], sw[(bm >> 5) + 1], bm & 31);
  const float2 dd = h2x2f(*reinterpret_cast<const uint32_t*>(rec));
  a[0] = dd.x * u6f(s);
  a[1] = dd.x * u6f(s >> 6);
  c[0] = fmaf(128.0f, a[0], dd.y * u6f(m));
  c[1] = fmaf(128.0f, a[1], dd.y * u6f(m >> 6));
}

// M = 1 decodes through bf16's linear range instead: the bit patterns 0..255 of a
// bf16 are exactly the values 0..255 x 2^-133 (subnormals and the first normal
// binade), so a word masked with 0x000F000F gives {q, q'} x 2^-133 and masked with
// 0x00F000F0 gives {q, q'} x 2^-129 -- no shift for two of the four pairs and no
// +128 offset. The activations are scaled by 2^67 (low-nibble pairs) or 2^63
// (high-nibble pairs) with one exact bf16x2 multiply each, so every product is
// q x 2^-66: a normal fp32 value for 2^-60 <= |x| < 2^61 (the tensor core keeps
// subnormal bf16 operands exactly). The sum is rescaled by 2^66 through a_j.
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
// a_j x 2^66 and b_j for sub-blocks 2t, 2t+1 of a record in shared memory
__device__ __forceinline__ void q4k_pair_scales_lin_rec(const uint8_t* rec, int t, float* a, float* b) {
  const uint32_t* sw = reinterpret_cast<const uint32_t*>(rec + 4);
  const int bs = 12 * t, bm = 48 + 12 * t;
  const uint32_t s = __funnelshift_r(sw[bs >> 5], sw[(bs >> 5) + 1], bs & 31);
  const uint32_t m = __funnelshift_r(sw[bm >> 5], sw[(bm >> 5) + 1], bm & 31);
  const float2 dd = h2x2f(*reinterpret_cast<const uint32_t*>(rec));
  const float d66 = dd.x * 7.3786976294838206e19f;      // d x 2^66 (exact)
  a[0] = d66 * u6f(s);
  a[1] = d66 * u6f(s >> 6);
  b[0] = dd.y * u6f(m);
  b[1] = dd.y * u6f(m >> 6);
}

template <>
struct Slab<F_Q4_K, 1> {
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
    for (int j = 0; j < 8; ++j) {
      const uint32_t wa = WA[j], wb = WB[j], ha = wa >> 8, hb = wb >> 8;
      const uint4 b = ldx128(xs, g == j, xo);
      float* d = (j & 1) ? dO : dE;
      mma_bf16(d, wa & 0x000F000Fu, wb & 0x000F000Fu, wa & 0x00F000F0u, wb & 0x00F000F0u, bmul2(b.x, kX67),
               bmul2(b.y, kX63));
      mma_bf16(d, ha & 0x000F000Fu, hb & 0x000F000Fu, ha & 0x00F000F0u, hb & 0x00F000F0u, bmul2(b.z, kX67),
               bmul2(b.w, kX63));
    }
    const uint4 xv = lds128v(xs + xo);
    mma_bf16(xx, kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, xv.x, xv.y);
    mma_bf16(xx, kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, xv.z, xv.w);
    float aA[2], bA[2], aB[2], bB[2];
    q4k_pair_scales_lin_rec(rA, t, aA, bA);
    q4k_pair_scales_lin_rec(rB, t, aB, bB);
    acc[0] += fmaf(aA[0], dE[0] + dO[0], fmaf(aA[1], dE[1] + dO[1], -fmaf(bA[0], xx[0], bA[1] * xx[1])));
    acc[1] += fmaf(aB[0], dE[2] + dO[2], fmaf(aB[1], dE[3] + dO[3], -fmaf(bB[0], xx[2], bB[1] * xx[3])));
  }
};

// the same from the header words in registers (the M > 1 scale tables)
__device__ __forceinline__ void q4k_pair_scales_lin(const uint4 hd, int t, float* a, float* b) {
  const float2 dd = h2x2f(hd.x);
  const uint64_t lo = ((uint64_t)hd.z << 32) | hd.y, hi = ((uint64_t)hd.w << 32) | hd.z;
  const uint32_t s = (uint32_t)(lo >> (12 * t)), m = (uint32_t)(hi >> (16 + 12 * t));
  const float d66 = dd.x * 7.3786976294838206e19f;      // d x 2^66 (exact)
  a[0] = d66 * u6f(s);
  a[1] = d66 * u6f(s >> 6);
  b[0] = dd.y * u6f(m);
  b[1] = dd.y * u6f(m >> 6);
}

template <>
struct Slab<F_Q4_K, 8> {
  __device__ static void run(const uint8_t* st, const uint8_t*, const uint8_t* xs, int R, int w, int lane,
                             float2* tbl, float* acc) {
    const int g = lane >> 2, t = lane & 3;
    {   // scale table of the warp's 16 rows: lane -> (row lane/2, sub-blocks 4h..4h+3)
      const int rl = lane >> 1, h = lane & 1;
      const uint4 hd = lds128v(st + (16 * w + rl) * 144);
      float a[2], b[2];
      q4k_pair_scales_lin(hd, 2 * h, a, b);
      tbl[rl * kTblStride + 4 * h + 0] = make_float2(a[0], b[0]);
      tbl[rl * kTblStride + 4 * h + 1] = make_float2(a[1], b[1]);
      q4k_pair_scales_lin(hd, 2 * h + 1, a, b);
      tbl[rl * kTblStride + 4 * h + 2] = make_float2(a[0], b[0]);
      tbl[rl * kTblStride + 4 * h + 3] = make_float2(a[1], b[1]);
    }
    __syncwarp();
    uint32_t WA[8], WB[8];
    load8(st + (16 * w + g) * 144 + q4k_word_off(t, 0), WA);
    load8(st + (16 * w + g + 8) * 144 + q4k_word_off(t, 0), WB);
    const bool has_x = g < R;
#pragma unroll
    for (int j0 = 0; j0 < 8; j0 += 4) {
      float dd[4][4], xx[4][4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) dd[q][e] = xx[q][e] = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = j0 + q;
        const uint32_t wa = WA[j], wb = WB[j], ha = wa >> 8, hb = wb >> 8;
        const uint4 xv = has_x ? lds128v(xs + 64 * j + 16 * t) : make_uint4(0u, 0u, 0u, 0u);
        mma_bf16(dd[q], wa & 0x000F000Fu, wb & 0x000F000Fu, wa & 0x00F000F0u, wb & 0x00F000F0u,
                 bmul2(xv.x, kX67), bmul2(xv.y, kX63));
        mma_bf16(xx[q], kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, xv.x, xv.y);
        mma_bf16(dd[q], ha & 0x000F000Fu, hb & 0x000F000Fu, ha & 0x00F000F0u, hb & 0x00F000F0u,
                 bmul2(xv.z, kX67), bmul2(xv.w, kX63));
        mma_bf16(xx[q], kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, xv.z, xv.w);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 sA = tbl[g * kTblStride + j0 + q], sB = tbl[(g + 8) * kTblStride + j0 + q];
        acc[0] = fmaf(sA.x, dd[q][0], fmaf(-sA.y, xx[q][0], acc[0]));
        acc[1] = fmaf(sA.x, dd[q][1], fmaf(-sA.y, xx[q][1], acc[1]));
        acc[2] = fmaf(sB.x, dd[q][2], fmaf(-sB.y, xx[q][2], acc[2]));
        acc[3] = fmaf(sB.x, dd[q][3], fmaf(-sB.y, xx[q][3], acc[3]));
      }
    }
    __syncwarp();
  }
};

// ============================================================================
// Q5_K. The Q4_K scheme with q = 0..31: A = 128 + q is still exact in bf16, the
// header (d, dmin, scale stream) is Q4_K's, and the pairs come from the 5-bit
// words plus the chunk's nibble word (packed layout: qmv_layout.cuh).
// ============================================================================
// the four pairs {128 + q(8t+2p), 128 + q(8t+2p+1)} of a thread's 5-bit word v;
// u = the chunk's nibble word already shifted right by 4t
__device__ __forceinline__ void q5k_quad(uint32_t v, uint32_t u, uint32_t* a) {
  a[0] = and_or(v, 0x001F001Fu, 0x43004300u);
  a[1] = and_or(v >> 5, 0x001F001Fu, 0x43004300u);
  a[2] = and_or(v >> 10, 0x001F001Fu, 0x43004300u);
  a[3] = and_or(v >> 11, 0x00100010u, and_or(u, 0x000F000Fu, 0x43004300u));
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
      const uint4 b = ldx128(xs, g == j, xo);
      float* d = (j & 1) ? dO : dE;
      mma_bf16(d, pa[0], pb[0], pa[1], pb[1], b.x, b.y);
      mma_bf16(d, pa[2], pb[2], pa[3], pb[3], b.z, b.w);
    }
    const uint4 xv = lds128v(xs + xo);
    mma_bf16(xx, kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, xv.x, xv.y);
    mma_bf16(xx, kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, xv.z, xv.w);
    float aA[2], cA[2], aB[2], cB[2];
    q4k_pair_scales_rec(rA, t, aA, cA);
    q4k_pair_scales_rec(rB, t, aB, cB);
    acc[0] += fmaf(aA[0], dE[0] + dO[0], fmaf(aA[1], dE[1] + dO[1], -fmaf(cA[0], xx[0], cA[1] * xx[1])));
    acc[1] += fmaf(aB[0], dE[2] + dO[2], fmaf(aB[1], dE[3] + dO[3], -fmaf(cB[0], xx[2], cB[1] * xx[3])));
  }
};

template <>
struct Slab<F_Q5_K, 8> {
  __device__ static void run(const uint8_t* st, const uint8_t*, const uint8_t* xs, int R, int w, int lane,
                             float2* tbl, float* acc) {
    const int g = lane >> 2, t = lane & 3;
    {   // scale table of the warp's 16 rows: lane -> (row lane/2, sub-blocks 4h..4h+3)
      const int rl = lane >> 1, h = lane & 1;
      const uint4 hd = lds128v(st + (16 * w + rl) * 176);
      float a[2], c[2];
      q4k_pair_scales(hd, 2 * h, a, c);
      tbl[rl * kTblStride + 4 * h + 0] = make_float2(a[0], c[0]);
      tbl[rl * kTblStride + 4 * h + 1] = make_float2(a[1], c[1]);
      q4k_pair_scales(hd, 2 * h + 1, a, c);
      tbl[rl * kTblStride + 4 * h + 2] = make_float2(a[0], c[0]);
      tbl[rl * kTblStride + 4 * h + 3] = make_float2(a[1], c[1]);
    }
    __syncwarp();
    const uint8_t* rA = st + (16 * w + g) * 176;
    const uint8_t* rB = rA + 8 * 176;
    uint32_t WA[8], WB[8];
    load8(rA + q5k_word_off(t, 0), WA);
    load8(rB + q5k_word_off(t, 0), WB);
    const int us = 4 * t;
    const bool has_x = g < R;
#pragma unroll
    for (int j0 = 0; j0 < 8; j0 += 4) {
      // the nibble words of these four chunks only (fewer live registers)
      const uint4 ua = lds128v(rA + q5k_nib_off(j0)), ub = lds128v(rB + q5k_nib_off(j0));
      const uint32_t UA[4] = {ua.x, ua.y, ua.z, ua.w}, UB[4] = {ub.x, ub.y, ub.z, ub.w};
      float dd[4][4], xx[4][4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) dd[q][e] = xx[q][e] = 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int j = j0 + q;
        uint32_t pa[4], pb[4];
        q5k_quad(WA[j], UA[q] >> us, pa);
        q5k_quad(WB[j], UB[q] >> us, pb);
        const uint4 xv = has_x ? lds128v(xs + 64 * j + 16 * t) : make_uint4(0u, 0u, 0u, 0u);
        mma_bf16(dd[q], pa[0], pb[0], pa[1], pb[1], xv.x, xv.y);
        mma_bf16(xx[q], kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, xv.x, xv.y);
        mma_bf16(dd[q], pa[2], pb[2], pa[3], pb[3], xv.z, xv.w);
        mma_bf16(xx[q], kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, xv.z, xv.w);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 sA = tbl[g * kTblStride + j0 + q], sB = tbl[(g + 8) * kTblStride + j0 + q];
        acc[0] = fmaf(sA.x, dd[q][0], fmaf(-sA.y, xx[q][0], acc[0]));
        acc[1] = fmaf(sA.x, dd[q][1], fmaf(-sA.y, xx[q][1], acc[1]));
        acc[2] = fmaf(sB.x, dd[q][2], fmaf(-sB.y, xx[q][2], acc[2]));
        acc[3] = fmaf(sB.x, dd[q][3], fmaf(-sB.y, xx[q][3], acc[3]));
      }
    }
    __syncwarp();
  }
};

// ============================================================================
// Q8_0. q = u - 128 with u = 16 uh + ul; D_lo / D_hi over (128 + ul) / (128 + uh):
// sum q x = D_lo + 16 D_hi - 2304 X; w = d q (d per 32-value chunk).
// ============================================================================
template <>
struct Slab<F_Q8_0, 1> {
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
    for (int j = 0; j < 8; ++j) {
      const uint2 wa = make_uint2(WA[2 * j], WA[2 * j + 1]), wb = make_uint2(WB[2 * j], WB[2 * j + 1]);
      const uint4 bv = ldx128(xs, g == j, xo);
      const uint32_t b0 = bv.x, b1 = bv.y, b2 = bv.z, b3 = bv.w;
      mma_bf16(lo, nib_pair(wa.x, 0), nib_pair(wb.x, 0), nib_pair(wa.x, 1), nib_pair(wb.x, 1), b0, b1);
      mma_bf16(hi, nib_pair(wa.x, 2), nib_pair(wb.x, 2), nib_pair(wa.x, 3), nib_pair(wb.x, 3), b0, b1);
      mma_bf16(lo, nib_pair(wa.y, 0), nib_pair(wb.y, 0), nib_pair(wa.y, 1), nib_pair(wb.y, 1), b2, b3);
      mma_bf16(hi, nib_pair(wa.y, 2), nib_pair(wb.y, 2), nib_pair(wa.y, 3), nib_pair(wb.y, 3), b2, b3);
    }
    const uint4 xv = lds128v(xs + xo);
    mma_bf16(xx, kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, xv.x, xv.y);
    mma_bf16(xx, kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, xv.z, xv.w);
    const uint32_t dA = lds32(rA + 4 * t), dB = lds32(rB + 4 * t);     // d of chunks 2t, 2t+1
    const float2 da = h2x2f(dA), db = h2x2f(dB);
    const float a0 = da.x, a1 = da.y, b0 = db.x, b1 = db.y;
    acc[0] += fmaf(a0, fmaf(16.f, hi[0], lo[0]) - 2304.f * xx[0], a1 * (fmaf(16.f, hi[1], lo[1]) - 2304.f * xx[1]));
    acc[1] += fmaf(b0, fmaf(16.f, hi[2], lo[2]) - 2304.f * xx[2], b1 * (fmaf(16.f, hi[3], lo[3]) - 2304.f * xx[3]));
  }
};

template <>
struct Slab<F_Q8_0, 8> {
  __device__ static void run(const uint8_t* st, const uint8_t*, const uint8_t* xs, int R, int w, int lane,
                             float2* tbl, float* acc) {
    const int g = lane >> 2, t = lane & 3;
    {
      const int rl = lane >> 1, h = lane & 1;
      const uint2 dv = lds64(st + (16 * w + rl) * 272 + 8 * h);
      const uint32_t dw[2] = {dv.x, dv.y};
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const float d = h2f(dw[jj >> 1] >> (16 * (jj & 1)));
        tbl[rl * kTblStride + 4 * h + jj] = make_float2(d, 2304.0f * d);
      }
    }
    __syncwarp();
    uint32_t WA[16], WB[16];
    load16(st + (16 * w + g) * 272 + q80_word_off(t, 0), WA);
    load16(st + (16 * w + g + 8) * 272 + q80_word_off(t, 0), WB);
    const bool has_x = g < R;
#pragma unroll
    for (int j0 = 0; j0 < 8; j0 += 2) {
      float lo[2][4], hi[2][4], xx[2][4];
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) lo[q][e] = hi[q][e] = xx[q][e] = 0.f;
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const int j = j0 + q;
        const uint2 wa = make_uint2(WA[2 * j], WA[2 * j + 1]), wb = make_uint2(WB[2 * j], WB[2 * j + 1]);
        const uint4 xv = has_x ? lds128v(xs + 64 * j + 16 * t) : make_uint4(0u, 0u, 0u, 0u);
        mma_bf16(lo[q], nib_pair(wa.x, 0), nib_pair(wb.x, 0), nib_pair(wa.x, 1), nib_pair(wb.x, 1), xv.x, xv.y);
        mma_bf16(hi[q], nib_pair(wa.x, 2), nib_pair(wb.x, 2), nib_pair(wa.x, 3), nib_pair(wb.x, 3), xv.x, xv.y);
        mma_bf16(xx[q], kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, xv.x, xv.y);
        mma_bf16(lo[q], nib_pair(wa.y, 0), nib_pair(wb.y, 0), nib_pair(wa.y, 1), nib_pair(wb.y, 1), xv.z, xv.w);
        mma_bf16(hi[q], nib_pair(wa.y, 2), nib_pair(wb.y, 2), nib_pair(wa.y, 3), nib_pair(wb.y, 3), xv.z, xv.w);
        mma_bf16(xx[q], kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, xv.z, xv.w);
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        const float2 sA = tbl[g * kTblStride + j0 + q], sB = tbl[(g + 8) * kTblStride + j0 + q];
        acc[0] = fmaf(sA.x, fmaf(16.f, hi[q][0], lo[q][0]), fmaf(-sA.y, xx[q][0], acc[0]));
        acc[1] = fmaf(sA.x, fmaf(16.f, hi[q][1], lo[q][1]), fmaf(-sA.y, xx[q][1], acc[1]));
        acc[2] = fmaf(sB.x, fmaf(16.f, hi[q][2], lo[q][2]), fmaf(-sB.y, xx[q][2], acc[2]));
        acc[3] = fmaf(sB.x, fmaf(16.f, hi[q][3], lo[q][3]), fmaf(-sB.y, xx[q][3], acc[3]));
      }
    }
    __syncwarp();
  }
};

// ============================================================================
// Q6_K. q = ql + 16 qh, w = a_u (q - 32), a_u = d sc_u per 16-value sub-block u;
// sum w x = a_u (D_lo + 16 D_hi - 2208 X). k-step s of chunk j covers sub-block
// u = 2j + s; the thread's slots hold elements 16s + 4t .. 16s + 4t + 3 of chunk j.
// ============================================================================
// Q6_K through bf16's linear range: the low nibbles of pair p of an ql word sit at
// nibbles (p, p+4), their 2-bit highs at bits (2k, 2k+16) of the thread's qh word (k = p),
// so masks alone give exact bf16 values {v, v'} x 2^(s - 133): s = 0, 4 for nibble pairs
// 0, 1 (pairs 2, 3 after one shift by 8) and s = 0, 2, 4, 6 for the 2-bit pairs. x is
// scaled per k position to bring every product to (lo + 16 hi) x 2^-66, so the lo and hi
// MMAs add into sums of one scale: lo gets x 2^67 | 2^63, hi x 2^71 | 2^69 (pairs 0, 1)
// and x 2^67 | 2^65 (pairs 2, 3). Exact for |x| < 2^56.
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

template <>
struct Slab<F_Q6_K, 1> {
  // 16 units (sub-blocks): units 0..7 -> accumulator group 0, 8..15 -> group 1,
  // column n = u % 8. Thread (g', t) carries activations for units g' and g' + 8.
  __device__ static void run(const uint8_t* st, const uint8_t* dplane, const uint8_t* xs, int, int w,
                             int lane, float2*, float* acc) {
    const int g = lane >> 2, t = lane & 3;
    const int rowA = 16 * w + g, rowB = rowA + 8;
    const uint8_t* rA = st + rowA * 208;
    const uint8_t* rB = st + rowB * 208;
    const int hsh = 8 * (t & 1);
    // unit g' = 2j' + s': chunk j' = g'/2, s' = g' & 1; unit g' + 8: chunk j' + 4
    const uint2 x0 = lds64(xs + 64 * (g >> 1) + 32 * (g & 1) + 8 * t);
    const uint2 x1 = lds64(xs + 64 * ((g >> 1) + 4) + 32 * (g & 1) + 8 * t);
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
      const uint32_t la = LA[j], lb = LB[j];
      const uint32_t ha = HA[j] >> hsh;
      const uint32_t hb = HB[j] >> hsh;
      const int grp = j >> 2;
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        const int u = 2 * j + s2;
        const uint2 xv = ldx64(xs, (u & 7) == g, 32 * u + 8 * t);
        q6k_linear_mma(lo[grp], hi[grp], la, lb, ha, hb, s2, xv);
      }
    }
    mma_bf16(xx[0], kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, x0.x, x0.y);
    mma_bf16(xx[1], kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, x1.x, x1.y);
    // this thread's columns 2t, 2t+1 -> units {2t, 2t+1} (group 0), {8+2t, 9+2t} (group 1)
    const float dA = h2f(*reinterpret_cast<const unsigned short*>(dplane + 2 * rowA));
    const float dB = h2f(*reinterpret_cast<const unsigned short*>(dplane + 2 * rowB));
    const uint32_t sA0 = *reinterpret_cast<const unsigned short*>(rA + 192 + 2 * t);
    const uint32_t sA1 = *reinterpret_cast<const unsigned short*>(rA + 200 + 2 * t);
    const uint32_t sB0 = *reinterpret_cast<const unsigned short*>(rB + 192 + 2 * t);
    const uint32_t sB1 = *reinterpret_cast<const unsigned short*>(rB + 200 + 2 * t);
    float vA = 0.f, vB = 0.f;
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const uint32_t scA = q ? sA1 : sA0, scB = q ? sB1 : sB0;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const float aa = dA * i8f(scA >> (8 * e)), ab = dB * i8f(scB >> (8 * e));
        // sum (q - 32) x = 2^66 (lo + hi) - 32 sum x
        vA = fmaf(aa * 7.3786976294838206e19f, lo[q][e] + hi[q][e], fmaf(-32.f * aa, xx[q][e], vA));
        vB = fmaf(ab * 7.3786976294838206e19f, lo[q][2 + e] + hi[q][2 + e], fmaf(-32.f * ab, xx[q][2 + e], vB));
      }
    }
    acc[0] += vA;
    acc[1] += vB;
  }
};

template <>
struct Slab<F_Q6_K, 8> {
  __device__ static void run(const uint8_t* st, const uint8_t* dplane, const uint8_t* xs, int R, int w,
                             int lane, float2* tbl, float* acc) {
    const int g = lane >> 2, t = lane & 3;
    {
      const int rl = lane >> 1, h = lane & 1;
      const int row = 16 * w + rl;
      const float d = h2f(*reinterpret_cast<const unsigned short*>(dplane + 2 * row));
      const uint2 sv = lds64(st + row * 208 + 192 + 8 * h);
      const uint32_t sw[2] = {sv.x, sv.y};
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const float a = d * i8f(sw[jj >> 2] >> (8 * (jj & 3)));
        tbl[rl * kTblStride + 8 * h + jj] = make_float2(a * 7.3786976294838206e19f, 32.0f * a);
      }
    }
    __syncwarp();
    const uint8_t* rA = st + (16 * w + g) * 208;
    const uint8_t* rB = rA + 8 * 208;
    const int hsh = 8 * (t & 1);
    const bool has_x = g < R;
    uint32_t LA[8], LB[8], HA[8], HB[8];
    load8(rA + q6k_ql_word_off(t, 0), LA);
    load8(rB + q6k_ql_word_off(t, 0), LB);
    load8(rA + q6k_qh_word_off(t >> 1, 0), HA);
    load8(rB + q6k_qh_word_off(t >> 1, 0), HB);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t la = LA[j], lb = LB[j];
      const uint32_t ha = HA[j] >> hsh;
      const uint32_t hb = HB[j] >> hsh;
      float lo[2][4], hi[2][4], xx[2][4];
#pragma unroll
      for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) lo[q][e] = hi[q][e] = xx[q][e] = 0.f;
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        const uint2 xv = has_x ? lds64(xs + 64 * j + 32 * s2 + 8 * t) : make_uint2(0u, 0u);
        q6k_linear_mma(lo[s2], hi[s2], la, lb, ha, hb, s2, xv);
        mma_bf16(xx[s2], kOnesBf16, kOnesBf16, kOnesBf16, kOnesBf16, xv.x, xv.y);
      }
#pragma unroll
      for (int s2 = 0; s2 < 2; ++s2) {
        const float2 sA = tbl[g * kTblStride + 2 * j + s2], sB = tbl[(g + 8) * kTblStride + 2 * j + s2];
        acc[0] = fmaf(sA.x, lo[s2][0] + hi[s2][0], fmaf(-sA.y, xx[s2][0], acc[0]));
        acc[1] = fmaf(sA.x, lo[s2][1] + hi[s2][1], fmaf(-sA.y, xx[s2][1], acc[1]));
        acc[2] = fmaf(sB.x, lo[s2][2] + hi[s2][2], fmaf(-sB.y, xx[s2][2], acc[2]));
        acc[3] = fmaf(sB.x, lo[s2][3] + hi[s2][3], fmaf(-sB.y, xx[s2][3], acc[3]));
      }
    }
    __syncwarp();
  }
};

// ============================================================================
// NVFP4. A = e2m1(c) * s_b in f16 (exact), B = x in f16; s_T in the epilogue.
// The codes of row r, K chunk j sit in the tensor-core tile at
// (r/8)*1024 + j*128 + (r%8)*16 (thread t reads word t: elements 8t..8t+7); the
// scales of the row's four blocks of K step ks are one 32-bit word of plane B at
// ks*512 + 16*(r%32) + 4*(r/32); chunk j uses block 2(j%2) + t/2 of step j/2.
// ============================================================================
__device__ __forceinline__ void nv_load(const uint8_t* st, const uint8_t* sf, int r, int t, uint32_t* C,
                                        uint32_t* S) {
  const uint8_t* c = st + (r >> 3) * 1024 + (r & 7) * 16 + 4 * t;
#pragma unroll
  for (int j = 0; j < 8; ++j) C[j] = lds32(c + 128 * j);
  const uint8_t* s = sf + 16 * (r & 31) + 4 * (r >> 5);
#pragma unroll
  for (int ks = 0; ks < 4; ++ks) S[ks] = lds32(s + 512 * ks);
}
// the E4M3 scale byte of chunk j for thread t
__device__ __forceinline__ uint32_t nv_sbyte(const uint32_t* S, int j, int t) {
  return (S[j >> 1] >> (8 * (2 * (j & 1) + (t >> 1)))) & 0xFFu;
}
__device__ __forceinline__ void nv_frag(uint32_t code_word, uint32_t sbyte, uint32_t* p) {
  const uint32_t s = e4m3x2_f16(sbyte | (sbyte << 8));
  e2m1x4_f16(code_word, p);
  p[0] = hmul2(p[0], s);
  p[1] = hmul2(p[1], s);
  p[2] = hmul2(p[2], s);
  p[3] = hmul2(p[3], s);
}

// M = 1: block-separated unit columns. Chunk j's two 16-value blocks land in
// columns 2(j/2) and 2(j/2) + 1 of accumulator set j%2, so each of a row's 16
// blocks in the slab keeps its own output slot; the codes go to the MMA as plain
// e2m1 values and each block's E4M3 scale multiplies its sum once, after the MMAs.
// Column c is fed by lanes (c, t): x of chunk pair c/2, and only from the lanes
// whose k positions hold block c%2 of the chunk (t/2 == c%2); other lanes feed 0.
// Lane (g, t) ends with blocks 4t..4t+3 of rows g and g + 8 -- K step t of the
// scale plane, one 32-bit word per row.
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
      const uint8_t* ca = st + (rA >> 3) * 1024 + (rA & 7) * 16 + 4 * t;
      const uint8_t* cb = st + (rB >> 3) * 1024 + (rB & 7) * 16 + 4 * t;
#pragma unroll
      for (int j = 0; j < 8; ++j) { CA[j] = lds32(ca + 128 * j); CB[j] = lds32(cb + 128 * j); }
    }
    float dE[4] = {0.f, 0.f, 0.f, 0.f}, dO[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const uint32_t wa = CA[j], wb = CB[j];
      // the B operand is x only in the chunk pair this lane's column serves: zeroed by a
      // multiply with an f16x2 {1, 1} / {0, 0} mask on the FMA pipe (x is finite),
      // which keeps the ALU pipe for the decode
      const uint32_t mk = ((j >> 1) == jp) ? 0x3C003C00u : 0u;
      const uint32_t* xv = (j & 1) ? xo : xe;
      float* d = (j & 1) ? dO : dE;
      uint32_t pa[4], pb[4];
      e2m1x4_f16(wa, pa);
      e2m1x4_f16(wb, pb);
      mma_f16(d, pa[0], pb[0], pa[1], pb[1], hmul2(xv[0], mk), hmul2(xv[1], mk));
      mma_f16(d, pa[2], pb[2], pa[3], pb[3], hmul2(xv[2], mk), hmul2(xv[3], mk));
    }
    const uint32_t sA = lds32(sf + 512 * t + 16 * (rA & 31) + 4 * (rA >> 5));
    const uint32_t sB = lds32(sf + 512 * t + 16 * (rB & 31) + 4 * (rB >> 5));
    uint32_t hA[2], hB[2];
    e4m3x4_f16(sA, hA);
    e4m3x4_f16(sB, hB);
    const float2 a01 = h2x2f(hA[0]), a23 = h2x2f(hA[1]);
    const float2 b01 = h2x2f(hB[0]), b23 = h2x2f(hB[1]);
    acc[0] += fmaf(a01.x, dE[0], fmaf(a01.y, dE[1], fmaf(a23.x, dO[0], a23.y * dO[1])));
    acc[1] += fmaf(b01.x, dE[2], fmaf(b01.y, dE[3], fmaf(b23.x, dO[2], b23.y * dO[3])));
  }
};

template <>
struct Slab<F_NVFP4, 8> {
  __device__ static void run(const uint8_t* st, const uint8_t* sf, const uint8_t* xs, int R, int w, int lane,
                             float2*, float* acc) {
    const int g = lane >> 2, t = lane & 3;
    const bool has_x = g < R;
    uint32_t CA[8], CB[8], SA[4], SB[4];
    nv_load(st, sf, 16 * w + g, t, CA, SA);
    nv_load(st, sf, 16 * w + g + 8, t, CB, SB);
    float dO[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      uint32_t pa[4], pb[4];
      nv_frag(CA[j], nv_sbyte(SA, j, t), pa);
      nv_frag(CB[j], nv_sbyte(SB, j, t), pb);
      uint4 xv = has_x ? lds128v(xs + 64 * j + 16 * t) : make_uint4(0u, 0u, 0u, 0u);
      float* d = (j & 1) ? dO : acc;
      mma_f16(d, pa[0], pb[0], pa[1], pb[1], xv.x, xv.y);     // x already f16 (converted per stage)
      mma_f16(d, pa[2], pb[2], pa[3], pb[3], xv.z, xv.w);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] += dO[e];
  }
};

// ============================================================================
// FP8 row-scaled. A = e4m3 in f16 (exact), B = x in f16; s_row in the epilogue.
// The thread's 8 values of chunk j are bytes 8(t&1).. of 16-byte vector 2j + t/2.
// ============================================================================
template <>
struct Slab<F_FP8, 1> {
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
      const uint2 ca = lds64(rA + fp8_v_off(v, rowA & 7)), cb = lds64(rB + fp8_v_off(v, rowB & 7));
      const bool mine = (g == j);
      float* d = (j & 1) ? dO : dE;
      uint32_t a0[2], b0[2], a1[2], b1[2];
      e4m3x4_f16(ca.x, a0);
      e4m3x4_f16(cb.x, b0);
      e4m3x4_f16(ca.y, a1);
      e4m3x4_f16(cb.y, b1);
      mma_f16(d, a0[0], b0[0], a0[1], b0[1], sel(mine, x0), sel(mine, x1));
      mma_f16(d, a1[0], b1[0], a1[1], b1[1], sel(mine, x2), sel(mine, x3));
    }
    acc[0] += (dE[0] + dO[0]) + (dE[1] + dO[1]);
    acc[1] += (dE[2] + dO[2]) + (dE[3] + dO[3]);
  }
};

template <>
struct Slab<F_FP8, 8> {
  __device__ static void run(const uint8_t* st, const uint8_t*, const uint8_t* xs, int R, int w, int lane,
                             float2*, float* acc) {
    const int g = lane >> 2, t = lane & 3;
    const int rowA = 16 * w + g, rowB = rowA + 8;
    const uint8_t* rA = st + rowA * 256 + 8 * (t & 1);
    const uint8_t* rB = st + rowB * 256 + 8 * (t & 1);
    const bool has_x = g < R;
    float dO[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int v = 2 * j + (t >> 1);
      const uint2 ca = lds64(rA + fp8_v_off(v, rowA & 7)), cb = lds64(rB + fp8_v_off(v, rowB & 7));
      const uint4 xv = has_x ? lds128v(xs + 64 * j + 16 * t) : make_uint4(0u, 0u, 0u, 0u);
      float* d = (j & 1) ? dO : acc;
      uint32_t a0[2], b0[2], a1[2], b1[2];
      e4m3x4_f16(ca.x, a0);
      e4m3x4_f16(cb.x, b0);
      e4m3x4_f16(ca.y, a1);
      e4m3x4_f16(cb.y, b1);
      mma_f16(d, a0[0], b0[0], a0[1], b0[1], xv.x, xv.y);     // x already f16 (converted per stage)
      mma_f16(d, a1[0], b1[0], a1[1], b1[1], xv.z, xv.w);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) acc[e] += dO[e];
  }
};

}  // namespace qmv
