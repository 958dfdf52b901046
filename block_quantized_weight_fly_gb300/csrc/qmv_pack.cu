// qmv_pack.cu -- load-phase kernels: canonical -> packed repack, BlockToFloat on the
// packed layout, the synthetic-data quantizers, and the NVFP4 activation quantizer.
//
// None of these is on the per-token GEMV path except the activation quantizer
// of the W4A4 prefill route.
#include <cuda_fp16.h>
#include "qmv_internal.h"

namespace qmv {

// ---------------------------------------------------------------------------
// canonical -> packed. One thread per (expert, row < N, 32-value chunk); the
// buffer is zero-filled first, which also writes every padding row, padding
// chunk and alignment gap.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void copy_bytes(uint8_t* dst, const uint8_t* src, int n) {
  for (int i = 0; i < n; ++i) dst[i] = src[i];
}
// little-endian 32-bit load from a byte address of any alignment
__device__ __forceinline__ uint32_t load_u32(const uint8_t* p) {
  return (uint32_t)p[0] | ((uint32_t)p[1] << 8) | ((uint32_t)p[2] << 16) | ((uint32_t)p[3] << 24);
}

__device__ __forceinline__ uint8_t* group_plane(const Layout& L, uint8_t* base, int64_t e, int64_t g) {
  return base + L.base + e * L.expert_bytes + g * L.group_bytes;
}

__global__ void pack_kernel(Layout L, const uint8_t* __restrict__ canon, uint8_t* __restrict__ dst) {
  const int64_t chunks = L.K / kChunk;
  const int64_t total = L.E * L.N * chunks;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx == 0) {
    PackedHeader* h = reinterpret_cast<PackedHeader*>(dst);
    h->magic = kMagic; h->version = kVersion; h->fmt = (uint32_t)L.fmt; h->reserved = 0;
    h->N = L.N; h->K = L.K; h->E = L.E;
    h->expert_bytes = L.expert_bytes; h->plane_bytes = L.group_bytes;
  }
  if (idx >= total) return;
  const int64_t c = idx % chunks;
  const int64_t rest = idx / chunks;
  const int64_t n = rest % L.N;
  const int64_t e = rest / L.N;
  const int64_t g = c / kChunksPerSlab;
  const int cl = (int)(c % kChunksPerSlab);
  uint8_t* plane = group_plane(L, dst, e, g);
  uint8_t* rec = plane + n * L.rec;
  uint8_t* extras = dst + L.base + e * L.expert_bytes + L.k_groups * L.group_bytes;
  const int64_t row = e * L.N + n;          // row of the stacked tower
  switch (L.fmt) {
    case F_Q8_0: {
      const uint8_t* src = canon + (row * chunks + c) * 34;
      copy_bytes(rec + 2 * cl, src, 2);
      for (int wd = 0; wd < 8; ++wd)
        *reinterpret_cast<uint32_t*>(rec + q80_word_off(wd >> 1, cl) + 4 * (wd & 1)) =
            q80_permute(load_u32(src + 2 + 4 * wd));
    } break;
    case F_Q4_K: {
      const uint8_t* blk = canon + (row * (L.K / 256) + g) * 144;
      for (int wd = 0; wd < 4; ++wd)
        *reinterpret_cast<uint32_t*>(rec + q4k_word_off(wd, cl)) = q4k_permute(load_u32(blk + 16 + 16 * cl + 4 * wd));
      if (cl == 0) copy_bytes(rec, blk, 16);
    } break;
    case F_Q5_K: {
      const uint8_t* blk = canon + (row * (L.K / 256) + g) * 176;
      uint32_t nibs = 0u;
      for (int wd = 0; wd < 4; ++wd) {
        uint32_t q[8];
        for (int i = 0; i < 8; ++i) {
          const int ce = 32 * cl + 8 * wd + i;            // element within the superblock
          q[i] = ((blk[48 + (ce >> 1)] >> (4 * (ce & 1))) & 15u) | (((blk[16 + (ce >> 3)] >> (ce & 7)) & 1u) << 4);
        }
        *reinterpret_cast<uint32_t*>(rec + q5k_word_off(wd, cl)) = q5k_word(q);
        nibs |= q5k_nibs(q, wd);
      }
      *reinterpret_cast<uint32_t*>(rec + q5k_nib_off(cl)) = nibs;
      if (cl == 0) copy_bytes(rec, blk, 16);
    } break;
    case F_Q6_K: {
      const uint8_t* blk = canon + (row * (L.K / 256) + g) * 210;
      uint32_t lw[4] = {0u, 0u, 0u, 0u}, hw[2] = {0u, 0u};
      for (int e = 0; e < 32; ++e) {
        const int ce = 32 * cl + e;                       // element within the superblock
        const uint32_t lo = (blk[ce >> 1] >> (4 * (ce & 1))) & 15u;
        const uint32_t hi = (blk[128 + (ce >> 2)] >> (2 * (ce & 3))) & 3u;
        int a, b, c2, d2;
        q6k_pos(e, &a, &b, &c2, &d2);
        lw[a] |= lo << (4 * b);
        hw[c2] |= hi << d2;
      }
      for (int i = 0; i < 4; ++i) *reinterpret_cast<uint32_t*>(rec + q6k_ql_word_off(i, cl)) = lw[i];
      for (int h = 0; h < 2; ++h) *reinterpret_cast<uint32_t*>(rec + q6k_qh_word_off(h, cl)) = hw[h];
      if (cl == 0) {
        copy_bytes(rec + 192, blk + 192, 16);
        copy_bytes(plane + L.plane_a + 2 * n, blk + 208, 2);
      }
    } break;
    case F_NVFP4: {
      const uint8_t* ce = canon + e * canon_matrix_bytes(F_NVFP4, L.N, L.K);
      for (int wd = 0; wd < 4; ++wd)
        *reinterpret_cast<uint32_t*>(plane + nv_code_off(n, cl, wd)) = load_u32(ce + n * (L.K / 2) + c * 16 + 4 * wd);
      const uint8_t* sc = ce + L.N * (L.K / 2) + n * (L.K / 16) + 2 * c;
      plane[L.plane_a + nv_scale_off(n, 2 * cl)] = sc[0];
      plane[L.plane_a + nv_scale_off(n, 2 * cl + 1)] = sc[1];
      if (n == 0 && c == 0) copy_bytes(extras, ce + L.N * (L.K / 2) + L.N * (L.K / 16), 4);
    } break;
    case F_FP8: {
      const uint8_t* ce = canon + e * canon_matrix_bytes(F_FP8, L.N, L.K);
      const int r = (int)(n & 7);
      copy_bytes(rec + fp8_v_off(2 * cl, r), ce + n * L.K + 32 * c, 16);
      copy_bytes(rec + fp8_v_off(2 * cl + 1, r), ce + n * L.K + 32 * c + 16, 16);
      if (c == 0) copy_bytes(extras + 4 * n, ce + L.N * L.K + 4 * n, 4);
    } break;
    case F_IQ4_XS: {
      const uint8_t* ce = canon + e * canon_matrix_bytes(F_IQ4_XS, L.N, L.K);
      const uint8_t* blk = ce + (n * (L.K / 256) + g) * 136;
      const int r = (int)(n & 7);
      for (int wd = 0; wd < 4; ++wd)
        *reinterpret_cast<uint32_t*>(rec + iq4_word_off(wd, cl, r)) = load_u32(blk + 8 + 16 * cl + 4 * wd);
      if (cl == 0) copy_bytes(plane + L.plane_a + iq4_scale_off(n), blk, 8);
      // every 128-row tile's plane B ends with the matrix's codebook
      if (cl == 0 && (n & 127) == 0)
        copy_bytes(plane + L.plane_a + iq4_codebook_off(n), ce + L.N * (L.K / 256) * 136, 16);
    } break;
    case F_IQ3_S: {
      // chunk cl of the block: groups 8cl .. 8cl+7; thread t's slots m = 2cl + s hold group 8cl + 4s + t
      const uint8_t* blk = canon + grid_entries(F_IQ3_S) * 4 + (row * (L.K / 256) + g) * 110;
      for (int t = 0; t < 4; ++t)
        for (int sh = 0; sh < 2; ++sh) {
          const int gr = 8 * cl + 4 * sh + t, m = 2 * cl + sh;
          rec[16 * t + m] = blk[2 + gr];
          const uint32_t sg = (blk[74 + gr / 2] >> (4 * (gr & 1))) & 15u;   // elements 4gr..4gr+3
          rec[64 + 8 * t + m / 2] |= (uint8_t)(sg << (4 * (m & 1)));
        }
      if (cl == 0) {   // plane B of the row: d, scales, and every slot's index bit 8
        uint8_t* pb = plane + L.plane_a + n * 14;
        copy_bytes(pb, blk, 2);
        copy_bytes(pb + 2, blk + 106, 4);
        for (int t = 0; t < 4; ++t) {
          uint32_t h = 0u;
          for (int m = 0; m < 16; ++m) {
            const int gr = 8 * (m >> 1) + 4 * (m & 1) + t;
            h |= ((uint32_t)(blk[66 + gr / 8] >> (gr & 7)) & 1u) << m;
          }
          pb[6 + 2 * t] = (uint8_t)h;
          pb[7 + 2 * t] = (uint8_t)(h >> 8);
        }
      }
    } break;
    case F_IQ2_S: {
      // chunk cl: groups 4cl .. 4cl+3; pair p's slots m = 2cl + s hold group 4cl + 2s + p, and
      // thread t's sign slot m holds half (t & 1) of that group (t >> 1 = p)
      const uint8_t* blk = canon + grid_entries(F_IQ2_S) * 8 + (row * (L.K / 256) + g) * 82;
      for (int p = 0; p < 2; ++p)
        for (int sh = 0; sh < 2; ++sh) {
          const int gr = 4 * cl + 2 * sh + p, m = 2 * cl + sh;
          rec[16 * p + m] = blk[2 + gr];
          for (int hf = 0; hf < 2; ++hf) {
            const int t = 2 * p + hf;
            const uint32_t sg = (blk[34 + gr] >> (4 * hf)) & 15u;
            rec[32 + 8 * t + m / 2] |= (uint8_t)(sg << (4 * (m & 1)));
          }
        }
      if (cl == 0) {   // plane B of the row: d, scales, and every slot's index bits 8..9
        uint8_t* pb = plane + L.plane_a + n * 18;
        copy_bytes(pb, blk, 2);
        copy_bytes(pb + 2, blk + 74, 8);
        for (int p = 0; p < 2; ++p) {
          uint32_t h = 0u;
          for (int m = 0; m < 16; ++m) {
            const int gr = 4 * (m >> 1) + 2 * (m & 1) + p;
            h |= ((uint32_t)(blk[66 + gr / 4] >> (2 * (gr & 3))) & 3u) << (2 * m);
          }
          for (int i = 0; i < 4; ++i) pb[10 + 4 * p + i] = (uint8_t)(h >> (8 * i));
        }
      }
    } break;
  }
}

// the grid formats' table (canonical uint8 magnitudes at the front of the stream) ->
// f16 values in the packed prefix
__global__ void pack_grid_kernel(int n, const uint8_t* __restrict__ canon, uint8_t* __restrict__ dst) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) reinterpret_cast<__half*>(dst + kHeaderBytes)[i] = __ushort2half_rn((unsigned short)canon[i]);
}

cudaError_t launch_pack(const Layout& L, const uint8_t* canon, uint8_t* dst, cudaStream_t s) {
  cudaError_t err = cudaMemsetAsync(dst, 0, (size_t)L.total, s);
  if (err != cudaSuccess) return err;
  const int64_t total = L.E * L.N * (L.K / kChunk);
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  pack_kernel<<<(unsigned)blocks, threads, 0, s>>>(L, canon, dst);
  if (is_grid_fmt(L.fmt)) {
    const int n = grid_entries(L.fmt) * grid_width(L.fmt);
    pack_grid_kernel<<<(n + threads - 1) / threads, threads, 0, s>>>(n, canon, dst);
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// BlockToFloat on the packed layout. One thread per (tower row, chunk); the
// op order is the canonical one and every product is rounded on its own
// (__fmul_rn / __fsub_rn keep the compiler from fusing them).
// ---------------------------------------------------------------------------
__device__ bool header_ok(const uint8_t* packed, const Layout& L) {
  const PackedHeader* h = reinterpret_cast<const PackedHeader*>(packed);
  return h->magic == kMagic && h->version == kVersion && h->fmt == (uint32_t)L.fmt &&
         h->N == L.N && h->K == L.K && h->E == L.E && h->expert_bytes == L.expert_bytes;
}

__global__ void dequant_kernel(Layout L, const uint8_t* __restrict__ packed, int64_t row0,
                               int64_t rows, float* __restrict__ out, unsigned* status) {
  const int64_t chunks = L.K / kChunk;
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (!header_ok(packed, L)) {
    if (idx == 0) atomicOr(status, kStatHeader);
    return;
  }
  if (idx >= rows * chunks) return;
  const int64_t c = idx % chunks;
  const int64_t row = row0 + idx / chunks;
  const int64_t e = row / L.N, n = row % L.N;
  const int64_t g = c / kChunksPerSlab;
  const int cl = (int)(c % kChunksPerSlab);
  const uint8_t* plane = packed + L.base + e * L.expert_bytes + g * L.group_bytes;
  const uint8_t* rec = plane + n * L.rec;
  const uint8_t* extras = packed + L.base + e * L.expert_bytes + L.k_groups * L.group_bytes;
  float* o = out + (row - row0) * L.K + c * kChunk;
  switch (L.fmt) {
    case F_Q8_0: {
      float d = h2f(*reinterpret_cast<const uint16_t*>(rec + 2 * cl));
      for (int wd = 0; wd < 8; ++wd) {
        const uint32_t cw = q80_unpermute(
            *reinterpret_cast<const uint32_t*>(rec + q80_word_off(wd >> 1, cl) + 4 * (wd & 1)));
        for (int i = 0; i < 4; ++i) o[4 * wd + i] = __fmul_rn(d, (float)(int8_t)((cw >> (8 * i)) & 0xFFu));
      }
    } break;
    case F_Q4_K: {
      const uint32_t* hd = reinterpret_cast<const uint32_t*>(rec);
      float d = h2f(hd[0]), dmin = h2f(hd[0] >> 16);
      uint32_t sc = q4k_field(hd[1], hd[2], hd[3], cl), m = q4k_field(hd[1], hd[2], hd[3], 8 + cl);
      float a = __fmul_rn(d, (float)sc), b = __fmul_rn(dmin, (float)m);
      for (int wd = 0; wd < 4; ++wd) {
        const uint32_t cw = q4k_unpermute(*reinterpret_cast<const uint32_t*>(rec + q4k_word_off(wd, cl)));
        for (int i = 0; i < 8; ++i) o[8 * wd + i] = __fsub_rn(__fmul_rn(a, (float)((cw >> (4 * i)) & 15u)), b);
      }
    } break;
    case F_Q5_K: {
      const uint32_t* hd = reinterpret_cast<const uint32_t*>(rec);
      float d = h2f(hd[0]), dmin = h2f(hd[0] >> 16);
      uint32_t sc = q4k_field(hd[1], hd[2], hd[3], cl), m = q4k_field(hd[1], hd[2], hd[3], 8 + cl);
      float a = __fmul_rn(d, (float)sc), b = __fmul_rn(dmin, (float)m);
      const uint32_t u = *reinterpret_cast<const uint32_t*>(rec + q5k_nib_off(cl));
      for (int wd = 0; wd < 4; ++wd) {
        const uint32_t v = *reinterpret_cast<const uint32_t*>(rec + q5k_word_off(wd, cl));
        for (int i = 0; i < 8; ++i) o[8 * wd + i] = __fsub_rn(__fmul_rn(a, (float)q5k_elem(v, u, wd, i)), b);
      }
    } break;
    case F_Q6_K: {
      uint32_t lw[4], hw[2];
      for (int i = 0; i < 4; ++i) lw[i] = *reinterpret_cast<const uint32_t*>(rec + q6k_ql_word_off(i, cl));
      for (int h = 0; h < 2; ++h) hw[h] = *reinterpret_cast<const uint32_t*>(rec + q6k_qh_word_off(h, cl));
      const int8_t* sc = reinterpret_cast<const int8_t*>(rec + 192);
      float d = h2f(*reinterpret_cast<const uint16_t*>(plane + L.plane_a + 2 * n));
      for (int i = 0; i < 32; ++i) {
        int a, b, c2, d2;
        q6k_pos(i, &a, &b, &c2, &d2);
        const int lo = (int)((lw[a] >> (4 * b)) & 15u);
        const int hi = (int)((hw[c2] >> d2) & 3u);
        const int qq = lo | (hi << 4);
        const float as = __fmul_rn(d, (float)sc[2 * cl + (i >> 4)]);
        o[i] = __fmul_rn(as, (float)(qq - 32));
      }
    } break;
    case F_NVFP4: {
      const float sT = *reinterpret_cast<const float*>(extras);
      for (int i = 0; i < 32; ++i) {
        const uint32_t cw = *reinterpret_cast<const uint32_t*>(plane + nv_code_off(n, cl, i >> 3));
        uint32_t code = (cw >> (4 * (i & 7))) & 15u;
        float p = __fmul_rn(e2m1f(code), e4m3f(plane[L.plane_a + nv_scale_off(n, 2 * cl + (i >> 4))]));
        o[i] = __fmul_rn(p, sT);
      }
    } break;
    case F_FP8: {
      const int r = (int)(n & 7);
      const uint8_t* c0 = rec + fp8_v_off(2 * cl, r);
      const uint8_t* c1 = rec + fp8_v_off(2 * cl + 1, r);
      const float s = reinterpret_cast<const float*>(extras)[n];
      for (int i = 0; i < 16; ++i) o[i] = __fmul_rn(e4m3f(c0[i]), s);
      for (int i = 0; i < 16; ++i) o[16 + i] = __fmul_rn(e4m3f(c1[i]), s);
    } break;
    case F_IQ4_XS: {
      const uint8_t* sf = plane + L.plane_a + iq4_scale_off(n);
      const int8_t* cb = reinterpret_cast<const int8_t*>(plane + L.plane_a + iq4_codebook_off(n));
      const float d = h2f(*reinterpret_cast<const uint16_t*>(sf));
      const uint32_t sh = *reinterpret_cast<const uint16_t*>(sf + 2);
      const uint32_t sl = *reinterpret_cast<const uint32_t*>(sf + 4);
      const int ls = (int)(((sl >> (4 * cl)) & 15u) | (((sh >> (2 * cl)) & 3u) << 4));
      const float a = __fmul_rn(d, (float)(ls - 32));
      const int r = (int)(n & 7);
      for (int wd = 0; wd < 4; ++wd) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(rec + iq4_word_off(wd, cl, r));
        for (int i = 0; i < 8; ++i) o[8 * wd + i] = __fmul_rn(a, (float)cb[(w >> (4 * i)) & 15u]);
      }
    } break;
    case F_IQ3_S:
    case F_IQ2_S: {
      // w = (d (2 sc + 1)) (+-G[idx][i]); G from the packed prefix (f16, exact)
      const bool iq3 = L.fmt == F_IQ3_S;
      const __half* G = reinterpret_cast<const __half*>(packed + kHeaderBytes);
      const uint8_t* pb = plane + L.plane_a + n * grid_brow(L.fmt);
      const float d = h2f((uint32_t)pb[0] | ((uint32_t)pb[1] << 8));
      for (int sh = 0; sh < 2; ++sh) {
        const int m = 2 * cl + sh;
        const int k = iq3 ? cl : m;                              // sub-block of 32 / 16 values
        const int sc = (pb[2 + k / 2] >> (4 * (k & 1))) & 15;
        const float a = __fmul_rn(d, (float)(2 * sc + 1));
        for (int t = 0; t < 4; ++t) {
          int idx, gw, off;
          if (iq3) {
            const int hb = (pb[6 + 2 * t + m / 8] >> (m & 7)) & 1;
            idx = rec[16 * t + m] | (hb << 8);
            gw = 4;
            off = 0;
          } else {
            const int p = t >> 1;
            const int hb = (pb[10 + 4 * p + (2 * m) / 8] >> ((2 * m) & 7)) & 3;
            idx = rec[16 * p + m] | (hb << 8);
            gw = 8;
            off = 4 * (t & 1);
          }
          const uint32_t sg = (rec[(iq3 ? 64 : 32) + 8 * t + m / 2] >> (4 * (m & 1))) & 15u;
          for (int i = 0; i < 4; ++i) {
            const float mg = __half2float(G[idx * gw + off + i]);
            o[16 * sh + 4 * t + i] = __fmul_rn(a, ((sg >> i) & 1u) ? -mg : mg);
          }
        }
      }
    } break;
  }
}

cudaError_t launch_dequant(const Layout& L, const uint8_t* packed, int64_t row0, int64_t rows,
                           float* out, unsigned* status, cudaStream_t s) {
  const int64_t total = rows * (L.K / kChunk);
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  if (blocks == 0) return cudaSuccess;
  dequant_kernel<<<(unsigned)blocks, threads, 0, s>>>(L, packed, row0, rows, out, status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Quantizers for synthetic data. fp32 arithmetic with every operation rounded
// on its own, in the order written; round-to-nearest-even everywhere.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t f2h_bits(float f) {
  return (uint32_t)__half_as_ushort(__float2half_rn(f));
}
__device__ __forceinline__ uint32_t f2e4m3(float f) {   // RNE, saturate to +-448
  unsigned short v;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(v) : "f"(0.0f), "f"(f));
  return v & 0xFFu;
}
__device__ __forceinline__ uint32_t f2e2m1(float f) {   // RNE, saturate to +-6
  uint32_t v;
  asm("{ .reg .b8 t; cvt.rn.satfinite.e2m1x2.f32 t, %1, %2; cvt.u32.u8 %0, t; }"
      : "=r"(v) : "f"(0.0f), "f"(f));
  return v & 0xFu;
}
__device__ __forceinline__ float clampf(float v, float lo, float hi) { return fminf(fmaxf(v, lo), hi); }

__global__ void quant_q8_0_kernel(const float* __restrict__ W, int64_t nblk, uint8_t* __restrict__ out) {
  int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nblk) return;
  const float* x = W + b * 32;
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const uint32_t d = f2h_bits(__fdiv_rn(amax, 127.0f));
  const float dd = h2f(d);
  // assemble the 34-byte block in registers, then store it byte by byte
  uint32_t words[9];
  words[0] = d;
  for (int i = 1; i < 9; ++i) words[i] = 0u;
  for (int i = 0; i < 32; ++i) {
    const float q = (dd == 0.0f) ? 0.0f : clampf(rintf(__fdiv_rn(x[i], dd)), -127.0f, 127.0f);
    const uint32_t byte = (uint32_t)((int)q) & 0xFFu;
    const int pos = 2 + i;
    words[pos >> 2] |= byte << (8 * (pos & 3));
  }
  uint8_t* o = out + b * 34;
  for (int i = 0; i < 34; ++i) o[i] = (uint8_t)(words[i >> 2] >> (8 * (i & 3)));
}

__global__ void quant_q4_k_kernel(const float* __restrict__ W, int64_t nblk, uint8_t* __restrict__ out) {
  int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nblk) return;
  const float* x = W + b * 256;
  uint8_t* o = out + b * 144;
  float s[8], mn[8], smax = 0.0f, mmax = 0.0f;
  for (int j = 0; j < 8; ++j) {
    float lo = 0.0f, hi = x[32 * j];
    for (int i = 0; i < 32; ++i) {
      float v = x[32 * j + i];
      lo = fminf(lo, v);
      hi = fmaxf(hi, v);
    }
    s[j] = __fdiv_rn(__fsub_rn(hi, lo), 15.0f);
    mn[j] = -lo;
    smax = fmaxf(smax, s[j]);
    mmax = fmaxf(mmax, mn[j]);
  }
  uint32_t d = f2h_bits(__fdiv_rn(smax, 63.0f)), dmin = f2h_bits(__fdiv_rn(mmax, 63.0f));
  float dd = h2f(d), dm = h2f(dmin);
  uint32_t sw[3] = {0u, 0u, 0u};
  uint32_t sc[8], mq[8];
  for (int j = 0; j < 8; ++j) {
    sc[j] = (dd == 0.0f) ? 0u : (uint32_t)clampf(rintf(__fdiv_rn(s[j], dd)), 0.0f, 63.0f);
    mq[j] = (dm == 0.0f) ? 0u : (uint32_t)clampf(rintf(__fdiv_rn(mn[j], dm)), 0.0f, 63.0f);
  }
  for (int f = 0; f < 16; ++f) {
    uint32_t v = f < 8 ? sc[f] : mq[f - 8];
    for (int bit = 0; bit < 6; ++bit) {
      int pos = 6 * f + bit;
      sw[pos >> 5] |= ((v >> bit) & 1u) << (pos & 31);
    }
  }
  o[0] = (uint8_t)d; o[1] = (uint8_t)(d >> 8); o[2] = (uint8_t)dmin; o[3] = (uint8_t)(dmin >> 8);
  for (int i = 0; i < 12; ++i) o[4 + i] = (uint8_t)(sw[i >> 2] >> (8 * (i & 3)));
  for (int j = 0; j < 8; ++j) {
    float den = __fmul_rn(dd, (float)sc[j]);
    float off = __fmul_rn(dm, (float)mq[j]);
    for (int i = 0; i < 32; i += 2) {
      uint32_t q2[2];
      for (int u = 0; u < 2; ++u) {
        float num = __fadd_rn(x[32 * j + i + u], off);
        q2[u] = (den == 0.0f) ? 0u : (uint32_t)clampf(rintf(__fdiv_rn(num, den)), 0.0f, 15.0f);
      }
      o[16 + (32 * j + i) / 2] = (uint8_t)(q2[0] | (q2[1] << 4));
    }
  }
}

// Q5_K: the Q4_K quantizer with 32 levels; fifth bits at 16 + e/8, nibbles at 48 + e/2
__global__ void quant_q5_k_kernel(const float* __restrict__ W, int64_t nblk, uint8_t* __restrict__ out) {
  int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nblk) return;
  const float* x = W + b * 256;
  uint8_t* o = out + b * 176;
  float s[8], mn[8], smax = 0.0f, mmax = 0.0f;
  for (int j = 0; j < 8; ++j) {
    float lo = 0.0f, hi = x[32 * j];
    for (int i = 0; i < 32; ++i) {
      float v = x[32 * j + i];
      lo = fminf(lo, v);
      hi = fmaxf(hi, v);
    }
    s[j] = __fdiv_rn(__fsub_rn(hi, lo), 31.0f);
    mn[j] = -lo;
    smax = fmaxf(smax, s[j]);
    mmax = fmaxf(mmax, mn[j]);
  }
  uint32_t d = f2h_bits(__fdiv_rn(smax, 63.0f)), dmin = f2h_bits(__fdiv_rn(mmax, 63.0f));
  float dd = h2f(d), dm = h2f(dmin);
  uint32_t sw[3] = {0u, 0u, 0u};
  uint32_t sc[8], mq[8];
  for (int j = 0; j < 8; ++j) {
    sc[j] = (dd == 0.0f) ? 0u : (uint32_t)clampf(rintf(__fdiv_rn(s[j], dd)), 0.0f, 63.0f);
    mq[j] = (dm == 0.0f) ? 0u : (uint32_t)clampf(rintf(__fdiv_rn(mn[j], dm)), 0.0f, 63.0f);
  }
  for (int f = 0; f < 16; ++f) {
    uint32_t v = f < 8 ? sc[f] : mq[f - 8];
    for (int bit = 0; bit < 6; ++bit) {
      int pos = 6 * f + bit;
      sw[pos >> 5] |= ((v >> bit) & 1u) << (pos & 31);
    }
  }
  o[0] = (uint8_t)d; o[1] = (uint8_t)(d >> 8); o[2] = (uint8_t)dmin; o[3] = (uint8_t)(dmin >> 8);
  for (int i = 0; i < 12; ++i) o[4 + i] = (uint8_t)(sw[i >> 2] >> (8 * (i & 3)));
  for (int j = 0; j < 8; ++j) {
    float den = __fmul_rn(dd, (float)sc[j]);
    float off = __fmul_rn(dm, (float)mq[j]);
    uint32_t hb = 0u;                                   // fifth bits of the sub-block
    for (int i = 0; i < 32; i += 2) {
      uint32_t q2[2];
      for (int u = 0; u < 2; ++u) {
        float num = __fadd_rn(x[32 * j + i + u], off);
        q2[u] = (den == 0.0f) ? 0u : (uint32_t)clampf(rintf(__fdiv_rn(num, den)), 0.0f, 31.0f);
        hb |= (q2[u] >> 4) << (i + u);
      }
      o[48 + (32 * j + i) / 2] = (uint8_t)((q2[0] & 15u) | ((q2[1] & 15u) << 4));
    }
    for (int i = 0; i < 4; ++i) o[16 + 4 * j + i] = (uint8_t)(hb >> (8 * i));
  }
}

__global__ void quant_q6_k_kernel(const float* __restrict__ W, int64_t nblk, uint8_t* __restrict__ out) {
  int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nblk) return;
  const float* x = W + b * 256;
  uint8_t* o = out + b * 210;
  float s[16], smax = 0.0f;
  for (int j = 0; j < 16; ++j) {
    float amax = 0.0f;
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[16 * j + i]));
    s[j] = __fdiv_rn(amax, 32.0f);
    smax = fmaxf(smax, s[j]);
  }
  uint32_t d = f2h_bits(__fdiv_rn(smax, 127.0f));
  float dd = h2f(d);
  for (int i = 0; i < 192; ++i) o[i] = 0;
  for (int j = 0; j < 16; ++j) {
    int sc = (dd == 0.0f) ? 0 : (int)clampf(rintf(__fdiv_rn(s[j], dd)), -128.0f, 127.0f);
    o[192 + j] = (uint8_t)(int8_t)sc;
    float den = __fmul_rn(dd, (float)sc);
    for (int i = 0; i < 16; ++i) {
      int e = 16 * j + i;
      int q = (den == 0.0f) ? 0 : (int)clampf(rintf(__fdiv_rn(x[e], den)), -32.0f, 31.0f);
      int u = q + 32;
      o[e >> 1] |= (uint8_t)((u & 15) << (4 * (e & 1)));
      o[128 + (e >> 2)] |= (uint8_t)(((u >> 4) & 3) << (2 * (e & 3)));
    }
  }
  o[208] = (uint8_t)d; o[209] = (uint8_t)(d >> 8);
}

// NVFP4: one thread per 16-value block of row-major W[rows][K]
__global__ void quant_nvfp4_kernel(const float* __restrict__ W, int64_t rows, int64_t K, float sT,
                                   uint8_t* __restrict__ out) {
  int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t bpr = K / 16;
  if (b >= rows * bpr) return;
  const int64_t r = b / bpr, kb = b % bpr;
  const float* x = W + r * K + kb * 16;
  float amax = 0.0f;
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  float t = __fmul_rn(6.0f, sT);
  uint32_t sb = (t > 0.0f) ? f2e4m3(__fdiv_rn(amax, t)) : 0u;
  out[rows * (K / 2) + r * bpr + kb] = (uint8_t)sb;
  float den = __fmul_rn(e4m3f(sb), sT);
  uint8_t* codes = out + r * (K / 2) + kb * 8;
  for (int i = 0; i < 16; i += 2) {
    uint32_t c0 = (den == 0.0f) ? 0u : f2e2m1(__fdiv_rn(x[i], den));
    uint32_t c1 = (den == 0.0f) ? 0u : f2e2m1(__fdiv_rn(x[i + 1], den));
    codes[i >> 1] = (uint8_t)(c0 | (c1 << 4));
  }
  if (b == 0) *reinterpret_cast<float*>(out + rows * (K / 2) + rows * bpr) = sT;
}

// FP8 row-scaled: one block per row
__global__ void quant_fp8_kernel(const float* __restrict__ W, int64_t rows, int64_t K,
                                 uint8_t* __restrict__ out) {
  const int64_t r = blockIdx.x;
  const float* x = W + r * K;
  __shared__ float red[32];
  float amax = 0.0f;
  for (int64_t k = threadIdx.x; k < K; k += blockDim.x) amax = fmaxf(amax, fabsf(x[k]));
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.0f;
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float s = __fdiv_rn(red[0], 448.0f);
  for (int64_t k = threadIdx.x; k < K; k += blockDim.x)
    out[r * K + k] = (uint8_t)((s == 0.0f) ? 0u : f2e4m3(__fdiv_rn(x[k], s)));
  if (threadIdx.x == 0) *reinterpret_cast<float*>(out + rows * K + 4 * r) = s;
}

// IQ4_XS: sub-block j gets the signed scale s_j that maps its element of largest
// magnitude onto the codebook entry of largest magnitude (the first such entry);
// d = max_j |s_j| / 31 in fp16; ls_j = clamp(rint(s_j / d) + 32, 0, 63); each element
// takes the entry c nearest to it, |w - a_j C[c]| with a_j = d (ls_j - 32), ties to
// the lower index. Block 0's thread also writes the codebook after the blocks.
__global__ void quant_iq4_xs_kernel(const float* __restrict__ W, int64_t nblk, Codebook16 cb,
                                    uint8_t* __restrict__ out) {
  int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b == 0)
    for (int i = 0; i < 16; ++i) out[nblk * 136 + i] = (uint8_t)cb.v[i];
  if (b >= nblk) return;
  const float* x = W + b * 256;
  int cm = 0;
  for (int c = 1; c < 16; ++c)
    if (abs((int)cb.v[c]) > abs((int)cb.v[cm])) cm = c;
  float s[8], smax = 0.0f;
  for (int j = 0; j < 8; ++j) {
    int em = 0;
    for (int i = 1; i < 32; ++i)
      if (fabsf(x[32 * j + i]) > fabsf(x[32 * j + em])) em = i;
    s[j] = (cb.v[cm] != 0) ? __fdiv_rn(x[32 * j + em], (float)cb.v[cm]) : 0.0f;
    if (fabsf(s[j]) > smax) smax = fabsf(s[j]);
  }
  const uint32_t dh = f2h_bits(__fdiv_rn(smax, 31.0f));
  const float d = h2f(dh);
  uint32_t words[34];
  for (int i = 0; i < 34; ++i) words[i] = 0u;
  uint32_t sh = 0u;
  for (int j = 0; j < 8; ++j) {
    int ls = 32;
    if (d > 0.0f) ls = (int)clampf(__fadd_rn(rintf(__fdiv_rn(s[j], d)), 32.0f), 0.0f, 63.0f);
    sh |= (uint32_t)((ls >> 4) & 3) << (2 * j);
    words[1] |= (uint32_t)(ls & 15) << (4 * j);
    const float a = __fmul_rn(d, (float)(ls - 32));
    for (int i = 0; i < 32; ++i) {
      const float v = x[32 * j + i];
      int best = 0;
      float be = fabsf(__fsub_rn(v, __fmul_rn(a, (float)cb.v[0])));
      for (int c = 1; c < 16; ++c) {
        const float e = fabsf(__fsub_rn(v, __fmul_rn(a, (float)cb.v[c])));
        if (e < be) { be = e; best = c; }
      }
      const int e = 32 * j + i;                     // nibble e of the 128 index bytes
      words[2 + (e >> 3)] |= (uint32_t)best << (4 * (e & 7));
    }
  }
  words[0] = dh | (sh << 16);
  uint8_t* o = out + b * 136;
  for (int i = 0; i < 136; ++i) o[i] = (uint8_t)(words[i >> 2] >> (8 * (i & 3)));
}

// IQ3_S / IQ2_S: per sub-block (32 / 16 values) s = amax / gmax, gmax = the largest
// magnitude in the grid; d = max s / 31 in fp16; sc = clamp(rint((s / d - 1) / 2), 0, 15),
// a = d (2 sc + 1); per group (4 / 8 weights) the signs of its weights and the grid
// entry nearest to their magnitudes, sum_i (|w_i| - a G[c][i])^2 in fp32 in i order,
// ties to the lower index. One thread per block; G (uint8) is in global memory.
template <int FMT>
__global__ void quant_grid_kernel(const float* __restrict__ W, int64_t nblk, const uint8_t* __restrict__ G,
                                  int gmax, uint8_t* __restrict__ out) {
  constexpr bool kIq3 = FMT == F_IQ3_S;
  constexpr int gw = kIq3 ? 4 : 8, ne = kIq3 ? 512 : 1024, sbs = kIq3 ? 32 : 16, bb = kIq3 ? 110 : 82;
  constexpr int nsb = 256 / sbs;
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nblk) return;
  const float* x = W + b * 256;
  // the block is assembled in 32-bit words, then stored byte by byte
  uint32_t wd[(bb + 3) / 4];
  for (int i = 0; i < (bb + 3) / 4; ++i) wd[i] = 0u;
  auto put = [&](int byte, uint32_t v) { wd[byte >> 2] |= (v & 0xFFu) << (8 * (byte & 3)); };
  float s[nsb], smax = 0.0f;
  for (int k = 0; k < nsb; ++k) {
    float amax = 0.0f;
    for (int i = 0; i < sbs; ++i)
      if (fabsf(x[k * sbs + i]) > amax) amax = fabsf(x[k * sbs + i]);
    s[k] = (gmax > 0) ? __fdiv_rn(amax, (float)gmax) : 0.0f;
    if (s[k] > smax) smax = s[k];
  }
  const uint32_t dh = f2h_bits(__fdiv_rn(smax, 31.0f));
  const float d = h2f(dh);
  put(0, dh);
  put(1, dh >> 8);
  for (int k = 0; k < nsb; ++k) {
    int sc = 0;
    if (d > 0.0f) sc = (int)clampf(rintf(__fdiv_rn(__fsub_rn(__fdiv_rn(s[k], d), 1.0f), 2.0f)), 0.0f, 15.0f);
    put((kIq3 ? 106 : 74) + k / 2, (uint32_t)sc << (4 * (k & 1)));
    const float a = __fmul_rn(d, (float)(2 * sc + 1));
    for (int g = k * sbs / gw; g < (k + 1) * sbs / gw; ++g) {
      const float* xg = x + g * gw;
      float m[gw];
      for (int i = 0; i < gw; ++i) m[i] = fabsf(xg[i]);
      int best = 0;
      float be = 0.0f;
      for (int c = 0; c < ne; ++c) {
        float e = 0.0f;
        for (int i = 0; i < gw; ++i) {
          const float t = __fsub_rn(m[i], __fmul_rn(a, (float)G[c * gw + i]));
          e = __fadd_rn(e, __fmul_rn(t, t));
        }
        if (c == 0 || e < be) { be = e; best = c; }
      }
      put(2 + g, (uint32_t)best);
      if (kIq3) put(66 + g / 8, (uint32_t)((best >> 8) & 1) << (g & 7));
      else put(66 + g / 4, (uint32_t)((best >> 8) & 3) << (2 * (g & 3)));
      for (int i = 0; i < gw; ++i)
        if (xg[i] < 0.0f) {
          if (kIq3) put(74 + (g * 4 + i) / 8, 1u << ((g * 4 + i) & 7));
          else put(34 + g, 1u << i);
        }
    }
  }
  uint8_t* o = out + b * bb;
  for (int i = 0; i < bb; ++i) o[i] = (uint8_t)(wd[i >> 2] >> (8 * (i & 3)));
}

cudaError_t launch_quantize_codebook(int fmt, const float* W, int64_t rows, int64_t K, const uint8_t* codebook,
                                     uint8_t* canon, cudaStream_t s) {
  const int threads = 128;
  const int64_t n = rows * (K / 256);
  if (fmt == F_IQ4_XS) {
    Codebook16 cb;
    for (int i = 0; i < 16; ++i) cb.v[i] = (int8_t)codebook[i];
    quant_iq4_xs_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, s>>>(W, n, cb, canon);
    return cudaGetLastError();
  }
  if (!is_grid_fmt(fmt)) return cudaErrorInvalidValue;
  // the grid goes first in the stream (and is what the kernel reads)
  const size_t gb = (size_t)grid_entries(fmt) * grid_width(fmt);
  int gmax = 0;
  for (size_t i = 0; i < gb; ++i) gmax = codebook[i] > gmax ? codebook[i] : gmax;
  cudaError_t err = cudaMemcpyAsync(canon, codebook, gb, cudaMemcpyHostToDevice, s);
  if (err != cudaSuccess) return err;
  if (fmt == F_IQ3_S)
    quant_grid_kernel<F_IQ3_S><<<(unsigned)((n + threads - 1) / threads), threads, 0, s>>>(W, n, canon, gmax, canon + gb);
  else
    quant_grid_kernel<F_IQ2_S><<<(unsigned)((n + threads - 1) / threads), threads, 0, s>>>(W, n, canon, gmax, canon + gb);
  return cudaGetLastError();
}

cudaError_t launch_quantize(int fmt, const float* W, int64_t rows, int64_t K, float ts,
                            uint8_t* canon, cudaStream_t s) {
  const int threads = 128;
  switch (fmt) {
    case F_Q8_0: {
      int64_t n = rows * (K / 32);
      quant_q8_0_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, s>>>(W, n, canon);
    } break;
    case F_Q4_K: {
      int64_t n = rows * (K / 256);
      quant_q4_k_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, s>>>(W, n, canon);
    } break;
    case F_Q5_K: {
      int64_t n = rows * (K / 256);
      quant_q5_k_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, s>>>(W, n, canon);
    } break;
    case F_Q6_K: {
      int64_t n = rows * (K / 256);
      quant_q6_k_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, s>>>(W, n, canon);
    } break;
    case F_NVFP4: {
      int64_t n = rows * (K / 16);
      quant_nvfp4_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, s>>>(W, rows, K, ts, canon);
    } break;
    case F_FP8:
      quant_fp8_kernel<<<(unsigned)rows, 256, 0, s>>>(W, rows, K, canon);
      break;
    default:
      return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// NVFP4 activation quantizer: one thread per 16-value block of x[M][K].
// s_b = e4m3(amax_b / (6 x_scale)); zero block scale -> zero codes;
// else codes = e2m1(x / (s_b x_scale)).
// ---------------------------------------------------------------------------
// one 16-value block: the E4M3 scale and the 16 E2M1 codes (element i at nibble i)
__device__ __forceinline__ uint32_t quant_block16(const uint16_t* src16, float xs, uint32_t* packed) {
  const uint4* src = reinterpret_cast<const uint4*>(src16);
  uint4 v0 = src[0], v1 = src[1];
  uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
  float xv[16];
  float amax = 0.0f;
  for (int i = 0; i < 8; ++i) {
    xv[2 * i] = bf2f(w[i]);
    xv[2 * i + 1] = bf2f(w[i] >> 16);
    amax = fmaxf(amax, fmaxf(fabsf(xv[2 * i]), fabsf(xv[2 * i + 1])));
  }
  const float t = __fmul_rn(6.0f, xs);
  const uint32_t sb = (t > 0.0f) ? f2e4m3(__fdiv_rn(amax, t)) : 0u;
  packed[0] = packed[1] = 0u;
  if (sb != 0u) {
    const float den = __fmul_rn(e4m3f(sb), xs);
    for (int i = 0; i < 16; ++i) packed[i >> 3] |= f2e2m1(__fdiv_rn(xv[i], den)) << (4 * (i & 7));
  }
  return sb;
}

__global__ void quant_act_kernel(const uint16_t* __restrict__ x, float xs, uint8_t* __restrict__ codes,
                                 uint8_t* __restrict__ scales, int64_t M, int64_t K) {
  int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t bpr = K / 16;
  if (b >= M * bpr) return;
  const int64_t m = b / bpr, kb = b % bpr;
  uint32_t packed[2];
  scales[m * bpr + kb] = (uint8_t)quant_block16(x + m * K + kb * 16, xs, packed);
  uint2* dst = reinterpret_cast<uint2*>(codes + m * (K / 2) + kb * 8);
  *dst = make_uint2(packed[0], packed[1]);
}

// The same quantizer writing the tensor-core tiles of the W4A4 GEMM's activation
// operand: per k-group a plane of m_pad rows x 128 B of codes (core-matrix tiles,
// as the NVFP4 weight planes) followed by m_pad x 16 B of scales (tcgen05.cp tile
// layout). Rows m >= M (padding up to a multiple of 128) get zero codes and scales.
// One thread per row and 32-value chunk (two blocks), rows fastest across the
// threads: a warp's code stores cover whole 128-byte lines of the core-matrix tiles.
__global__ void quant_act_tiled_kernel(const uint16_t* __restrict__ x, float xs, uint8_t* __restrict__ planes,
                                       int64_t M, int64_t m_pad, int64_t K) {
  // the GEMM launched next may start its prologue and weight copies now; it reads
  // these planes only after its grid-dependency wait
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t cpr = K / 32;                      // 32-value chunks per row
  if (b >= m_pad * cpr) return;
  const int64_t m = b % m_pad, kc = b / m_pad;
  uint32_t packed[4] = {0u, 0u, 0u, 0u};
  uint32_t s0 = 0u, s1 = 0u;
  if (m < M) {
    s0 = quant_block16(x + m * K + kc * 32, xs, packed);
    s1 = quant_block16(x + m * K + kc * 32 + 16, xs, packed + 2);
  }
  uint8_t* plane = planes + (kc / 8) * (m_pad * 144);
  const int c = (int)(kc % 8);                    // chunk within the k-group: blocks 2c, 2c+1
  *reinterpret_cast<uint4*>(plane + nv_code_off(m, c, 0)) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
  *reinterpret_cast<uint16_t*>(plane + m_pad * 128 + nv_scale_off(m, 2 * c)) = (uint16_t)(s0 | (s1 << 8));
}

cudaError_t launch_quant_act_tiled(const uint16_t* x, float xs, uint8_t* planes, int M, int64_t m_pad, int64_t K,
                                   cudaStream_t s) {
  const int64_t total = m_pad * (K / 32);
  const int threads = 256;
  quant_act_tiled_kernel<<<(unsigned)((total + threads - 1) / threads), threads, 0, s>>>(x, xs, planes, M, m_pad, K);
  return cudaGetLastError();
}

cudaError_t launch_quant_act(const uint16_t* x, float xs, uint8_t* codes, uint8_t* scales, int M,
                             int64_t K, cudaStream_t s) {
  const int64_t n = (int64_t)M * (K / 16);
  const int threads = 128;
  if (n == 0) return cudaSuccess;
  quant_act_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, s>>>(x, xs, codes, scales, M, K);
  return cudaGetLastError();
}

}  // namespace qmv
