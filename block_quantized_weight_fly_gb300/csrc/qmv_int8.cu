// qmv_int8.cu -- the int8-dot variant of the decode GEMV: the activation is quantized
// to int8 per 32 values (d = amax / 127, q = rint(x / d) clamped to +-127) and each
// 32-value block's product is an integer dot of the weight codes with those codes
// (dp4a, exact in int32), scaled in fp32 by the weight block's scale and d. The lever
// the keep-quant issue books as the repayment of its slow decode ("feat(BACKEND-
// TENSTORRENT-KEEPQUANT) ...", "Scope", its "Out of scope" line and the accepted-cost
// note). Served for Q8_0 and Q4_K (w = d sc q - dmin m: the min term takes the sum of
// the block's x codes), reading the same packed layout as the mma.sync GEMV.
//
// Two launches: the activation quantizer (one thread per 32-value block, fp32 ops
// rounded one at a time, bit-exact with the oracle), then the GEMV: one warp per
// weight row, all M rows of x, the lanes of a warp on the eight 32-value chunks of a
// k-group (four lanes per chunk, eight values each), every weight byte read once.
#include "qmv_internal.h"

namespace qmv {

namespace {

__device__ __forceinline__ int dp4a_s8(uint32_t a, uint32_t b, int c) {
  int r;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

// x (bf16 [M][K]) -> int8 codes [M][K] and fp32 block scales [M][K/32]
__global__ void quant_q8_kernel(const uint16_t* __restrict__ x, int64_t nblk, int8_t* __restrict__ codes,
                                float* __restrict__ scales) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  asm volatile("griddepcontrol.wait;" ::: "memory");     // x may come from the kernel before
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nblk) return;
  const uint4* src = reinterpret_cast<const uint4*>(x + b * 32);
  float xv[32];
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint4 v = src[i];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      xv[8 * i + 2 * k] = bf2f(w[k]);
      xv[8 * i + 2 * k + 1] = bf2f(w[k] >> 16);
    }
  }
#pragma unroll
  for (int i = 0; i < 32; ++i)
    if (fabsf(xv[i]) > amax) amax = fabsf(xv[i]);
  const float d = __fdiv_rn(amax, 127.0f);
  uint32_t out[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) out[i] = 0u;
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int q = (d == 0.0f) ? 0 : (int)fminf(fmaxf(rintf(__fdiv_rn(xv[i], d)), -127.0f), 127.0f);
    out[i >> 2] |= ((uint32_t)q & 0xFFu) << (8 * (i & 3));
  }
  uint4* dst = reinterpret_cast<uint4*>(codes + b * 32);
  dst[0] = make_uint4(out[0], out[1], out[2], out[3]);
  dst[1] = make_uint4(out[4], out[5], out[6], out[7]);
  scales[b] = d;
}

// Q8_0 packed word pair of thread t, chunk j (elements 8t..8t+7) -> the eight signed codes
// in element order. In a packed word the low nibbles of elements (0, 1) sit at nibbles
// (0, 4), of (2, 3) at (1, 5), the high nibbles at (2, 6) and (3, 7) (codes XOR 0x80):
// A = w & 0x0F0F0F0F holds lo(e0), hi(e0), lo(e1), hi(e1) in its bytes, B = w >> 4 the same
// for e2, e3; byte 0 of A | A >> 4 is then e0's code, byte 2 e1's.
__device__ __forceinline__ uint32_t q80_codes4(uint32_t w) {
  const uint32_t a = w & 0x0F0F0F0Fu, b = (w >> 4) & 0x0F0F0F0Fu;
  const uint32_t ca = a | (a >> 4), cb = b | (b >> 4);
  return __byte_perm(ca, cb, 0x6420) ^ 0x80808080u;
}

// One warp per weight row n (all MT rows of x): lanes (j, t) = (lane / 4, lane % 4) take
// the eight values 8t..8t+7 of chunk j of every k-group.
template <int FMT, int MT>
__global__ void __launch_bounds__(256, 4) int8dot_kernel(Layout L, const uint8_t* __restrict__ packed,
                                                      const int8_t* __restrict__ codes,
                                                      const float* __restrict__ xsc, float* __restrict__ y,
                                                      int M, unsigned* status) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int lane = threadIdx.x & 31;
  const int64_t n = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const PackedHeader* h = reinterpret_cast<const PackedHeader*>(packed);
  if (!(h->magic == kMagic && h->version == kVersion && h->fmt == (uint32_t)L.fmt && h->N == L.N &&
        h->K == L.K && h->E == 1 && h->expert_bytes == L.expert_bytes)) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, kStatHeader);
    return;
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");      // the quantized x of the pre-pass
  if (n >= L.N) return;
  const int j = lane >> 2, t = lane & 3;
  float acc[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) acc[m] = 0.f;
  const int64_t G = L.k_groups;
#pragma unroll 4
  for (int64_t g = 0; g < G; ++g) {
    const uint8_t* rec = packed + L.base + g * L.group_bytes + n * L.rec;
    const int64_t kx = g * 256 + 32 * j + 8 * t;           // first of this lane's 8 values
    if constexpr (FMT == F_Q8_0) {
      if (kx >= L.K) continue;                             // the chunks past K in a ragged last group
      const uint2 w = *reinterpret_cast<const uint2*>(rec + q80_word_off(t, j));
      const float dw = h2f(*reinterpret_cast<const uint16_t*>(rec + 2 * j));
      const uint32_t c0 = q80_codes4(w.x), c1 = q80_codes4(w.y);
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m >= M) break;
        const uint2 xq = *reinterpret_cast<const uint2*>(codes + (int64_t)m * L.K + kx);
        const int s = dp4a_s8(c1, xq.y, dp4a_s8(c0, xq.x, 0));
        const float dx = xsc[(int64_t)m * (L.K / 32) + kx / 32];
        acc[m] = __fmaf_rn(__fmul_rn(dw, dx), (float)s, acc[m]);
      }
    } else {   // Q4_K
      const uint32_t w = *reinterpret_cast<const uint32_t*>(rec + q4k_word_off(t, j));
      const uint4 hd = *reinterpret_cast<const uint4*>(rec);
      const float d = h2f(hd.x), dmin = h2f(hd.x >> 16);
      const float a = __fmul_rn(d, (float)q4k_field(hd.y, hd.z, hd.w, j));
      const float c = __fmul_rn(dmin, (float)q4k_field(hd.y, hd.z, hd.w, 8 + j));
      // nibble k of the packed word holds element {0, 2, 4, 6, 1, 3, 5, 7}[k]: the low
      // nibbles are elements 0, 4, 1, 5 and the high ones 2, 6, 3, 7, in byte order
      const uint32_t lo = w & 0x0F0F0F0Fu, hi = (w >> 4) & 0x0F0F0F0Fu;
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m >= M) break;
        const uint2 xq = *reinterpret_cast<const uint2*>(codes + (int64_t)m * L.K + kx);
        const uint32_t xlo = __byte_perm(xq.x, xq.y, 0x5140), xhi = __byte_perm(xq.x, xq.y, 0x7362);
        const int s = dp4a_s8(hi, xhi, dp4a_s8(lo, xlo, 0));
        const int sx = dp4a_s8(0x01010101u, xq.y, dp4a_s8(0x01010101u, xq.x, 0));
        const float dx = xsc[(int64_t)m * (L.K / 32) + kx / 32];
        acc[m] = __fmaf_rn(__fmul_rn(a, dx), (float)s, __fmaf_rn(-__fmul_rn(c, dx), (float)sx, acc[m]));
      }
    }
  }
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    float v = acc[m];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0 && m < M) y[(int64_t)m * L.N + n] = v;
  }
}

}  // namespace

int64_t int8dot_workspace_bytes(int M, int64_t K) { return align_up((int64_t)M * K, 256) + align_up((int64_t)M * (K / 32) * 4, 256); }

cudaError_t launch_int8dot(const Layout& L, const uint8_t* packed, const uint16_t* x, float* y, int M, uint8_t* ws,
                           unsigned* status, cudaStream_t s) {
  int8_t* codes = reinterpret_cast<int8_t*>(ws);
  float* xsc = reinterpret_cast<float*>(ws + align_up((int64_t)M * L.K, 256));
  const int64_t nblk = (int64_t)M * (L.K / 32);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((nblk + 127) / 128));
  cfg.blockDim = dim3(128);
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t err = cudaLaunchKernelEx(&cfg, quant_q8_kernel, x, nblk, codes, xsc);
  if (err != cudaSuccess) return err;
  cfg.gridDim = dim3((unsigned)((L.N + 7) / 8));
  cfg.blockDim = dim3(256);
  if (L.fmt == F_Q8_0)
    err = M <= 1 ? cudaLaunchKernelEx(&cfg, int8dot_kernel<F_Q8_0, 1>, L, packed, (const int8_t*)codes,
                                      (const float*)xsc, y, M, status)
                 : cudaLaunchKernelEx(&cfg, int8dot_kernel<F_Q8_0, 8>, L, packed, (const int8_t*)codes,
                                      (const float*)xsc, y, M, status);
  else if (L.fmt == F_Q4_K)
    err = M <= 1 ? cudaLaunchKernelEx(&cfg, int8dot_kernel<F_Q4_K, 1>, L, packed, (const int8_t*)codes,
                                      (const float*)xsc, y, M, status)
                 : cudaLaunchKernelEx(&cfg, int8dot_kernel<F_Q4_K, 8>, L, packed, (const int8_t*)codes,
                                      (const float*)xsc, y, M, status);
  else
    return cudaErrorInvalidValue;
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace qmv
