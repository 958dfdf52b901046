// qmv_layout.cuh -- device ("packed") layout of block-quantized weights and the
// scalar decoders shared by the pack, dequant and GEMV kernels.
//
// Layout of one [N, K] matrix (one expert): k-group major. K is cut into groups
// of 256 values (the last group is zero-padded if K is not a multiple of 256);
// rows are padded to n_pad = a multiple of 128 with zero blocks. For every
// k-group g there is a plane of n_pad row records:
//
//   Q4_K : record = the canonical 144-byte superblock (d, dmin, 12 B scales, 128 B nibbles)
//   NVFP4: record = 16 B of E4M3 block scales | 128 B of E2M1 codes          (144 B)
//   Q8_0 : record = 8 fp16 d | 8 x 32 int8 quants                             (272 B)
//   Q6_K : record = 128 B ql | 64 B qh | 16 B int8 scales                     (208 B)
//          plus a second plane of n_pad fp16 d                                (2 B)
//   FP8  : record = 256 E4M3 codes, its 16-byte vectors rotated by (row & 7)  (256 B)
//
// so the bytes of (any row range) x (one k-group) are one contiguous span per
// plane: one bulk copy moves a 128-row x 256-value slab into shared memory. The
// bytes are the canonical bytes, regrouped; the bytes streamed per value equal
// the canonical block size. Records of 144, 208 and 272 bytes are odd multiples
// of 16, so 8 consecutive rows read at the same offset hit 8 different 16-byte
// bank groups; the 256-byte FP8 record gets the same property from its rotation.
//
// This regrouping is the planar-repack idea ("A 320B MoE on a free Kaggle TPU",
// "The 110 GB claim, checked against the tensor index": blocks split into dense
// planes with the matrix row on the lane axis) and the word-shadow idea of padding
// blocks to aligned words ("vllm.cpp #3030", "Budget on the 32 GB P150"), laid out
// for 128-bit loads and TMA bulk copies.
//
// Per expert, after its planes, an "extras" area holds the NVFP4 tensor scale
// (fp32) or the FP8 row scales (fp32 [n_pad]). A 256-byte header precedes the first
// expert.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_fp16.h>

namespace qmv {

constexpr int kSlabRows = 128;
constexpr int kSlabK = 256;
constexpr int kChunk = 32;           // values per lane chunk
constexpr int kChunksPerSlab = 8;
constexpr int kHeaderBytes = 256;
constexpr uint32_t kMagic = 0x31564D51u;  // "QMV1"
constexpr uint32_t kVersion = 2;

enum Fmt { F_Q8_0 = 1, F_Q4_K = 2, F_Q6_K = 3, F_NVFP4 = 4, F_FP8 = 5 };

struct PackedHeader {                 // first 256 bytes of a packed buffer
  uint32_t magic, version, fmt, reserved;
  int64_t N, K, E;
  int64_t expert_bytes, plane_bytes;
};

__host__ __device__ inline int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

// Granule of K the packed layout serves.
__host__ __device__ inline int64_t k_granule(int fmt) {
  return (fmt == F_Q4_K || fmt == F_Q6_K) ? 256 : (fmt == F_NVFP4 ? 16 : 32);
}

// bytes of one row record of plane A (per 256 values)
__host__ __device__ inline int rec_bytes(int fmt) {
  switch (fmt) {
    case F_Q8_0: return 272;
    case F_Q4_K: return 144;
    case F_Q6_K: return 208;
    case F_NVFP4: return 144;
    case F_FP8: return 256;
    default: return 0;
  }
}

struct Layout {
  int fmt;
  int rec;              // plane-A record bytes
  int64_t N, K, E;
  int64_t row_tiles;    // n_pad / 128
  int64_t n_pad;        // N rounded up to 128
  int64_t k_groups;     // ceil(K / 256)
  int64_t plane_a;      // bytes of one k-group's plane A (n_pad * rec)
  int64_t plane_b;      // bytes of one k-group's plane B (Q6_K d: n_pad * 2), else 0
  int64_t group_bytes;  // plane_a + plane_b
  int64_t extras;       // per-expert extras bytes (aligned to 256)
  int64_t expert_bytes; // bytes per expert (aligned to 256)
  int64_t total;        // header + E * expert_bytes
};

__host__ __device__ inline bool make_layout(int fmt, int64_t N, int64_t K, int64_t E, Layout* L) {
  if (fmt < F_Q8_0 || fmt > F_FP8 || N <= 0 || K <= 0 || E <= 0) return false;
  if (K % k_granule(fmt) != 0 || K % 32 != 0) return false;
  L->fmt = fmt;
  L->rec = rec_bytes(fmt);
  L->N = N; L->K = K; L->E = E;
  L->row_tiles = (N + kSlabRows - 1) / kSlabRows;
  L->n_pad = L->row_tiles * kSlabRows;
  L->k_groups = (K + kSlabK - 1) / kSlabK;
  L->plane_a = L->n_pad * L->rec;
  L->plane_b = (fmt == F_Q6_K) ? L->n_pad * 2 : 0;
  L->group_bytes = L->plane_a + L->plane_b;
  int64_t ex = 0;
  if (fmt == F_NVFP4) ex = 256;
  if (fmt == F_FP8) ex = align_up(L->n_pad * 4, 256);
  L->extras = ex;
  L->expert_bytes = align_up(L->k_groups * L->group_bytes + ex, 256);
  L->total = kHeaderBytes + E * L->expert_bytes;
  return true;
}

__host__ __device__ inline int64_t canon_matrix_bytes(int fmt, int64_t N, int64_t K) {
  switch (fmt) {
    case F_Q8_0: return N * (K / 32) * 34;
    case F_Q4_K: return N * (K / 256) * 144;
    case F_Q6_K: return N * (K / 256) * 210;
    case F_NVFP4: return N * (K / 2) + N * (K / 16) + 4;
    case F_FP8: return N * K + N * 4;
    default: return 0;
  }
}

// ---- record-internal offsets --------------------------------------------------
// Q8_0: d of chunk c at 2c; 16-byte vector h (0,1) of chunk c at 16 + 32c + 16h
__host__ __device__ inline int q80_q_off(int c, int h) { return 16 + 32 * c + 16 * h; }
// Q4_K: header at 0, 16 nibble bytes of chunk c at 16 + 16c
__host__ __device__ inline int q4k_q_off(int c) { return 16 + 16 * c; }
// NVFP4: scales at 0 (byte b = block b of 16 values), codes of chunk c at 16 + 16c
__host__ __device__ inline int nv_q_off(int c) { return 16 + 16 * c; }
// Q6_K: ql of chunk c at 16c, qh of chunk c at 128 + 8c, scales at 192
__host__ __device__ inline int q6k_ql_off(int c) { return 16 * c; }
__host__ __device__ inline int q6k_qh_off(int c) { return 128 + 8 * c; }
// FP8: 16-byte vector v (0..15) of row r sits at 16 * (v ^ (r & 7))
__host__ __device__ inline int fp8_v_off(int v, int r) { return 16 * (v ^ (r & 7)); }

// ---- scalar decoders (exact) -------------------------------------------------
__device__ __forceinline__ float h2f(uint32_t h) {
  return __half2float(__ushort_as_half((unsigned short)(h & 0xFFFFu)));
}
__device__ __forceinline__ float bf2f(uint32_t b) { return __uint_as_float((b & 0xFFFFu) << 16); }

// E4M3 -> fp32 (exact): hardware cvt to f16, then f16 -> f32
__device__ __forceinline__ float e4m3f(uint32_t c) {
  uint32_t h2;
  unsigned short v = (unsigned short)(c & 0xFFu);
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(v));
  return h2f(h2);
}
// E2M1 -> fp32 (exact); magnitudes times two {0,1,2,3,4,6,8,12} are the nibbles of 0xC8643210
__device__ __forceinline__ float e2m1f(uint32_t c) {
  uint32_t m2 = (0xC8643210u >> (4 * (c & 7))) & 15u;
  float v = (float)m2 * 0.5f;
  return (c & 8) ? -v : v;
}

// Q4_K 6-bit field f (0..15) of the 96-bit little-endian scale stream in header
// words s1..s3 (header bytes 4..15)
__device__ __forceinline__ uint32_t q4k_field(uint32_t s1, uint32_t s2, uint32_t s3, int f) {
  const int bit = 6 * f;
  const uint64_t lo = ((uint64_t)s2 << 32) | s1;
  const uint64_t hi = ((uint64_t)s3 << 32) | s2;
  const uint64_t src = (bit < 32) ? lo : hi;
  const int sh = (bit < 32) ? bit : bit - 32;
  return (uint32_t)(src >> sh) & 63u;
}

}  // namespace qmv
