// qmv_layout.cuh -- device ("packed") layout of block-quantized weights and the
// scalar decoders shared by the pack, dequant and GEMV kernels.
//
// Layout of one [N, K] matrix (one expert): k-group major. K is cut into groups
// of 256 values (the last group is zero-padded if K is not a multiple of 256);
// rows are padded to n_pad = a multiple of 128 with zero blocks. For every
// k-group g there is a plane of n_pad row records:
//
//   Q4_K : record = the canonical 144-byte superblock (d, dmin, 12 B scales, 128 B nibbles)
//   Q5_K : record = the 16-byte header (d, dmin, 12 B scales) | 128 B of 5-bit words |
//          32 B of nibble words (below)                                      (176 B)
//   NVFP4: plane A = E2M1 codes, 128 B per row, in tensor-core tiles (below)  (128 B)
//          plus a plane B of E4M3 block scales, 16 B per row, in the tile layout
//          the tensor memory copy of block scale factors takes                 (16 B)
//   Q8_0 : record = 8 fp16 d | 8 x 32 int8 quants                             (272 B)
//   Q6_K : record = 128 B ql | 64 B qh | 16 B int8 scales                     (208 B)
//          plus a second plane of n_pad fp16 d                                (2 B)
//   FP8  : record = 256 E4M3 codes, its 16-byte vectors rotated by (row & 7)  (256 B)
//   IQ4_XS: record = 128 B of codebook indices, thread-major 16-byte vectors rotated
//          by (row & 7) (below)                                              (128 B)
//          plus a plane B per 128-row tile: the rows' 8-byte scale fields (fp16 d,
//          u16 sh, u32 sl, canonical order), then the matrix's 16-byte codebook, so
//          that every slab copy brings its codebook along         (128 x 8 + 16 B)
//   IQ3_S: record = 64 B of index low bytes, then 32 B of sign bits, both
//          thread-major (below)                                               (96 B)
//          plus a plane B of 14 B per row: fp16 d, the 4 bytes of 4-bit scales, the
//          index bits 8 as one u16 per thread                                 (14 B)
//   IQ2_S: record = 32 B of index low bytes (per thread pair), then 32 B of sign
//          bits (per thread)                                                  (64 B)
//          plus a plane B of 18 B per row: fp16 d, the 8 bytes of 4-bit scales, the
//          index bits 8..9 as one u32 per thread pair                         (18 B)
//   The grid of IQ3_S / IQ2_S (one table per tower) is stored once, as f16 values,
//   between the header and the first expert (the "prefix").
//
// so the bytes of (any row range) x (one k-group) are one contiguous span per
// plane: one bulk copy moves a 128-row x 256-value slab into shared memory. The
// bytes are the canonical bytes, regrouped (and, inside some 32-bit words, their
// nibbles permuted -- see below); the bytes streamed per value equal the
// canonical block size.
//
// Nibble order inside 32-bit quant words. The kernels turn two 4-bit fields into
// two exact bf16 values with one AND-OR against the bf16 pattern of 128.0:
// ((word >> 4p) & 0x000F000F) | 0x43004300 = {128 + field(p), 128 + field(p+4)}.
// So each word stores the fields of consecutive element pairs at nibbles (p, p+4):
//   Q4_K : word w of a 32-value chunk = elements 8w..8w+7; element 8w+2p -> nibble p,
//          element 8w+2p+1 -> nibble p+4                              (p = 0..3)
//   Q5_K : 5-bit fields, decoded by the same AND-OR with mask 0x001F001F. Word w of a
//          chunk (its elements 8w..8w+7): the pairs (8w+2p, 8w+2p+1), p = 0..2, as
//          5-bit fields at bits (5p, 16+5p); bits 15 and 31 = the fifth bits of
//          elements 8w+6 and 8w+7. The low nibbles of those two elements sit in the
//          chunk's shared nibble word, at nibbles w and w+4. So a pair costs one
//          shift and one AND-OR, the last pair two of each; the record holds the
//          canonical 176 bytes' information in 176 bytes.
//   Q8_0 : byte u = q XOR 0x80 (0..255, the code plus 128); word w = elements 4w..4w+3:
//          low nibbles of elements (4w, 4w+1) -> nibbles (0, 4), of (4w+2, 4w+3) ->
//          (1, 5); high nibbles of (4w, 4w+1) -> (2, 6), of (4w+2, 4w+3) -> (3, 7)
//   Q6_K : ql word w of a chunk = low nibbles of elements {4w..4w+3, 16+4w..16+4w+3}
//          as pairs (4w,4w+1) -> (0,4), (4w+2,4w+3) -> (1,5), (16+4w,..) -> (2,6),
//          (16+4w+2,..) -> (3,7); qh word h (h = 0, 1) of a chunk: for element pairs of
//          quad w = 2h + s (s = 0, 1), pair k's 2-bit highs sit at bits
//          8s + 2k, 8s + 2k + 16 (k indexes the same four pairs as the ql word)
// NVFP4 and FP8 codes keep their canonical order (element 2i in the low nibble or
// byte), which the hardware FP4/FP8 -> f16x2 conversions consume directly.
// IQ4_XS: word t of chunk j = the canonical index bytes of elements 8t..8t+7 (element
// 8t+i at nibble i, unchanged); the 16-byte vector v = 2t + (j >> 2) of the record
// holds the words of chunks 4(j >> 2) .. +3 of thread t, stored at 16 (v ^ (row & 7)).
// IQ3_S, IQ2_S: the MMA (chunk j, half s) of thread t covers elements 32j + 16s + 4t
// .. +3, which is one IQ3_S group (8j + 4s + t) and half (t & 1) of one IQ2_S group
// (4j + 2s + (t >> 1)). Slot m = 2j + s of a thread: index low byte at 16t + m (IQ3_S)
// or 16(t >> 1) + m (IQ2_S); its four sign bits at bits 4m .. 4m+3 of the thread's
// 64-bit sign word (IQ3_S at 64 + 8t, IQ2_S at 32 + 8t); the index bit 8 at bit m of
// the thread's u16 in plane B (IQ3_S), bits 8..9 at bits 2m, 2m+1 of the thread
// pair's u32 (IQ2_S).
//
// NVFP4 tiles. The codes of a 128-row tile of a k-group (16 KB) are stored as the
// K-major "core matrices" of the 5th-generation tensor core: 8 rows x 16 bytes (32
// codes) each, 128 contiguous bytes; core (row group r/8, K chunk kc) at
// (r/8)*1024 + kc*128, row r%8 at +16*(r%8). So the same 16 KB serve a tcgen05.mma
// operand directly (leading byte offset 128, stride byte offset 1024) and the GEMV
// decoder. The block scales of the tile (2 KB) are four 512-byte blocks, one per
// 64-value K step: the scale of 16-value block kb (0..3) of row r at
// 16*(r%32) + 4*(r/32) + kb -- the 32 x 16-byte layout that tcgen05.cp.32x128b.warpx4
// replicates into the four lane quadrants of tensor memory.
//
// Records of 144, 176, 208 and 272 bytes are odd multiples of 16, so 8 consecutive rows
// read at the same offset hit 8 different 16-byte bank groups; the 256-byte FP8
// record gets the same property from its rotation.
//
// This regrouping is the planar-repack idea ("A 320B MoE on a free Kaggle TPU",
// "The 110 GB claim, checked against the tensor index": blocks split into dense
// planes with the matrix row on the lane axis) and the word-shadow idea of padding
// blocks to aligned words ("feat(BACKEND-TENSTORRENT-KEEPQUANT): the 27B arm — on-core
// decode residency, TT grouped keep-quant GEMM, e2e gate", "Budget on the 32 GB
// P150"), laid out for 128-bit loads and TMA bulk copies.
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
constexpr uint32_t kVersion = 5;

enum Fmt { F_Q8_0 = 1, F_Q4_K = 2, F_Q6_K = 3, F_NVFP4 = 4, F_FP8 = 5, F_Q5_K = 6, F_IQ4_XS = 7,
           F_IQ3_S = 8, F_IQ2_S = 9 };
constexpr int F_LAST = F_IQ2_S;
__host__ __device__ constexpr bool is_grid_fmt(int fmt) { return fmt == F_IQ3_S || fmt == F_IQ2_S; }
// grid entries and weights per entry (IQ3_S 512 x 4, IQ2_S 1024 x 8)
__host__ __device__ constexpr int grid_entries(int fmt) { return fmt == F_IQ3_S ? 512 : (fmt == F_IQ2_S ? 1024 : 0); }
__host__ __device__ constexpr int grid_width(int fmt) { return fmt == F_IQ3_S ? 4 : (fmt == F_IQ2_S ? 8 : 0); }
// plane B bytes per row of the grid formats
__host__ __device__ constexpr int grid_brow(int fmt) { return fmt == F_IQ3_S ? 14 : 18; }
// IQ4_XS plane B per 128-row tile: 8 bytes of scale fields per row, then the codebook
constexpr int kIq4TileB = 128 * 8 + 16;

struct PackedHeader {                 // first 256 bytes of a packed buffer
  uint32_t magic, version, fmt, reserved;
  int64_t N, K, E;
  int64_t expert_bytes, plane_bytes;
};

__host__ __device__ inline int64_t align_up(int64_t v, int64_t a) { return (v + a - 1) / a * a; }

// Granule of K the packed layout serves.
__host__ __device__ inline int64_t k_granule(int fmt) {
  return (fmt == F_Q4_K || fmt == F_Q5_K || fmt == F_Q6_K || fmt >= F_IQ4_XS) ? 256 : (fmt == F_NVFP4 ? 16 : 32);
}

// bytes of one row record of plane A (per 256 values)
__host__ __device__ inline int rec_bytes(int fmt) {
  switch (fmt) {
    case F_Q8_0: return 272;
    case F_Q4_K: return 144;
    case F_Q5_K: return 176;
    case F_Q6_K: return 208;
    case F_NVFP4: return 128;
    case F_FP8: return 256;
    case F_IQ4_XS: return 128;
    case F_IQ3_S: return 96;
    case F_IQ2_S: return 64;
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
  int64_t plane_b;      // bytes of one k-group's plane B (Q6_K d: n_pad * 2; NVFP4 scales: n_pad * 16;
                        // IQ4_XS: row_tiles * (128 * 8 + 16)), else 0
  int64_t group_bytes;  // plane_a + plane_b
  int64_t extras;       // per-expert extras bytes (aligned to 256)
  int64_t expert_bytes; // bytes per expert (aligned to 256)
  int64_t prefix;       // the grid formats' f16 grid after the header, else 0 (256-aligned)
  int64_t base;         // offset of expert 0 = header + prefix
  int64_t total;        // header + prefix + E * expert_bytes
};

__host__ __device__ inline bool make_layout(int fmt, int64_t N, int64_t K, int64_t E, Layout* L) {
  if (fmt < F_Q8_0 || fmt > F_LAST || N <= 0 || K <= 0 || E <= 0) return false;
  if (K % k_granule(fmt) != 0 || K % 32 != 0) return false;
  L->fmt = fmt;
  L->rec = rec_bytes(fmt);
  L->N = N; L->K = K; L->E = E;
  L->row_tiles = (N + kSlabRows - 1) / kSlabRows;
  L->n_pad = L->row_tiles * kSlabRows;
  L->k_groups = (K + kSlabK - 1) / kSlabK;
  L->plane_a = L->n_pad * L->rec;
  L->plane_b = (fmt == F_Q6_K)     ? L->n_pad * 2
               : (fmt == F_NVFP4)  ? L->n_pad * 16
               : (fmt == F_IQ4_XS) ? L->row_tiles * kIq4TileB
               : is_grid_fmt(fmt)  ? L->n_pad * grid_brow(fmt)
                                   : 0;
  L->group_bytes = L->plane_a + L->plane_b;
  int64_t ex = 0;
  if (fmt == F_NVFP4) ex = 256;
  if (fmt == F_FP8) ex = align_up(L->n_pad * 4, 256);
  L->extras = ex;
  L->expert_bytes = align_up(L->k_groups * L->group_bytes + ex, 256);
  L->prefix = is_grid_fmt(fmt) ? align_up((int64_t)grid_entries(fmt) * grid_width(fmt) * 2, 256) : 0;
  L->base = kHeaderBytes + L->prefix;
  L->total = L->base + E * L->expert_bytes;
  return true;
}

__host__ __device__ inline int64_t canon_matrix_bytes(int fmt, int64_t N, int64_t K) {
  switch (fmt) {
    case F_Q8_0: return N * (K / 32) * 34;
    case F_Q4_K: return N * (K / 256) * 144;
    case F_Q5_K: return N * (K / 256) * 176;
    case F_Q6_K: return N * (K / 256) * 210;
    case F_NVFP4: return N * (K / 2) + N * (K / 16) + 4;
    case F_FP8: return N * K + N * 4;
    case F_IQ4_XS: return N * (K / 256) * 136 + 16;
    case F_IQ3_S: return N * (K / 256) * 110;     // per matrix; a tower adds the grid once
    case F_IQ2_S: return N * (K / 256) * 82;
    default: return 0;
  }
}

// ---- record-internal offsets --------------------------------------------------
// Quant words are stored thread-major: the consumer thread t (t = 0..3) of an mma
// quad reads, for every 32-value chunk j of the k-group, the same 4 (or 8) bytes;
// those bytes of all 8 chunks are contiguous, so one or two 128-bit loads fetch them.
//   Q4_K        : word t of chunk j (its elements 8t..8t+7) at 16 + 32t + 4j
//   Q5_K        : 5-bit word t of chunk j at 16 + 32t + 4j; nibble word of chunk j at 144 + 4j
//   Q8_0        : words 2t, 2t+1 of chunk j (elements 8t..8t+7) at 16 + 64t + 8j
//   Q6_K        : ql word t of chunk j at 32t + 4j; qh word h of chunk j at 128 + 32h + 4j
__host__ __device__ inline int q4k_word_off(int t, int j) { return 16 + 32 * t + 4 * j; }
__host__ __device__ inline int q5k_word_off(int t, int j) { return 16 + 32 * t + 4 * j; }
__host__ __device__ inline int q5k_nib_off(int j) { return 144 + 4 * j; }
// NVFP4: byte offset (within plane A of a k-group) of code word wd (0..3) of K chunk kc
// (0..7) of row n, and (within plane B) of the scale of 16-value block b (0..15)
__host__ __device__ inline int64_t nv_code_off(int64_t n, int kc, int wd) {
  return (n >> 7) * 16384 + ((n & 127) >> 3) * 1024 + kc * 128 + (n & 7) * 16 + 4 * wd;
}
__host__ __device__ inline int64_t nv_scale_off(int64_t n, int b) {
  return (n >> 7) * 2048 + (b >> 2) * 512 + 16 * (n & 31) + 4 * ((n & 127) >> 5) + (b & 3);
}
__host__ __device__ inline int q80_word_off(int t, int j) { return 16 + 64 * t + 8 * j; }
__host__ __device__ inline int q6k_ql_word_off(int t, int j) { return 32 * t + 4 * j; }
__host__ __device__ inline int q6k_qh_word_off(int h, int j) { return 128 + 32 * h + 4 * j; }
// FP8: 16-byte vector v (0..15) of row r sits at 16 * (v ^ (r & 7))
__host__ __device__ inline int fp8_v_off(int v, int r) { return 16 * (v ^ (r & 7)); }
// IQ4_XS: index word t of chunk j of row r, and the offset (within the k-group's plane
// B) of row n's scale fields and of the codebook copy of its tile
__host__ __device__ inline int iq4_word_off(int t, int j, int r) {
  return 16 * ((2 * t + (j >> 2)) ^ (r & 7)) + 4 * (j & 3);
}
__host__ __device__ inline int64_t iq4_scale_off(int64_t n) { return (n >> 7) * kIq4TileB + (n & 127) * 8; }
__host__ __device__ inline int64_t iq4_codebook_off(int64_t n) { return (n >> 7) * kIq4TileB + 128 * 8; }

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

// ---- nibble permutations of the packed words (see the comment at the top) ---
// canonical nibble n (element 8w+n of a Q4_K word) -> packed nibble position
__host__ __device__ inline int q4k_pos(int n) { return (n & 1) ? (n >> 1) + 4 : (n >> 1); }
__host__ __device__ inline uint32_t q4k_permute(uint32_t w) {
  uint32_t o = 0;
  for (int n = 0; n < 8; ++n) o |= ((w >> (4 * n)) & 15u) << (4 * q4k_pos(n));
  return o;
}
__host__ __device__ inline uint32_t q4k_unpermute(uint32_t w) {
  uint32_t o = 0;
  for (int n = 0; n < 8; ++n) o |= ((w >> (4 * q4k_pos(n))) & 15u) << (4 * n);
  return o;
}
// Q8_0 word of 4 signed codes (byte i = element 4w+i) -> packed word
__host__ __device__ inline uint32_t q80_permute(uint32_t w) {
  uint32_t u = w ^ 0x80808080u, o = 0;
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = (u >> (8 * i)) & 15u, hi = (u >> (8 * i + 4)) & 15u;
    const int pl = (i >> 1) + 4 * (i & 1);        // low nibbles: pairs (0,4), (1,5)
    const int ph = 2 + (i >> 1) + 4 * (i & 1);    // high nibbles: pairs (2,6), (3,7)
    o |= lo << (4 * pl);
    o |= hi << (4 * ph);
  }
  return o;
}
__host__ __device__ inline uint32_t q80_unpermute(uint32_t w) {   // -> canonical signed bytes
  uint32_t o = 0;
  for (int i = 0; i < 4; ++i) {
    const int pl = (i >> 1) + 4 * (i & 1);
    const int ph = 2 + (i >> 1) + 4 * (i & 1);
    const uint32_t u = ((w >> (4 * pl)) & 15u) | (((w >> (4 * ph)) & 15u) << 4);
    o |= (u ^ 0x80u) << (8 * i);
  }
  return o;
}
// Q5_K: the 5-bit word of elements 8w..8w+7 (q[i] = element 8w+i, 0..31) and its
// part of the chunk's nibble word (nibbles w, w+4)
__host__ __device__ inline uint32_t q5k_word(const uint32_t* q) {
  uint32_t v = 0;
  for (int p = 0; p < 3; ++p) v |= (q[2 * p] << (5 * p)) | (q[2 * p + 1] << (16 + 5 * p));
  return v | ((q[6] >> 4) << 15) | ((q[7] >> 4) << 31);
}
__host__ __device__ inline uint32_t q5k_nibs(const uint32_t* q, int w) {
  return ((q[6] & 15u) << (4 * w)) | ((q[7] & 15u) << (16 + 4 * w));
}
// ... and back: element 8w+i of a word and its nibble word
__host__ __device__ inline uint32_t q5k_elem(uint32_t v, uint32_t u, int w, int i) {
  if (i < 6) return (v >> ((i & 1) * 16 + 5 * (i >> 1))) & 31u;
  const int h = (i & 1) * 16;
  return ((u >> (h + 4 * w)) & 15u) | (((v >> (15 + h)) & 1u) << 4);
}
// Q6_K: element e (0..31) of a chunk -> (ql word, nibble) and (qh word, bit)
__host__ __device__ inline void q6k_pos(int e, int* lw, int* ln, int* hw, int* hb) {
  const int half = e >> 4, r = e & 15;           // sub-block of 16 within the chunk
  const int w = r >> 2, q = r & 3;               // quad w of the sub-block, element q
  const int k = 2 * half + (q >> 1);             // pair index within the word (0..3)
  *lw = w;
  *ln = (q & 1) ? k + 4 : k;
  *hw = w >> 1;
  *hb = 8 * (w & 1) + 2 * k + ((q & 1) ? 16 : 0);
}

}  // namespace qmv
