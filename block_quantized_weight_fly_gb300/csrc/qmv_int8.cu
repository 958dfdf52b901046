// qmv_int8.cu -- the int8-dot variant of the decode GEMV: the activation is quantized
// to int8 per 32 values (d = amax / 127, q = rint(x / d) clamped to +-127) and each
// 32-value block's product is an integer dot of the weight codes with those codes
// (dp4a, exact in int32), scaled in fp32 by the weight block's scale and d. The lever
// the keep-quant issue books as the repayment of its slow decode ("feat(BACKEND-
// TENSTORRENT-KEEPQUANT) ...", "Scope", its "Out of scope" line and the accepted-cost
// note). Served for Q8_0 and Q4_K (w = d sc q - dmin m: the min term takes the sum of
// the block's x codes), reading the same packed layout as the mma.sync GEMV.
//
// Two launches, chained by programmatic dependent launch:
//  - the activation quantizer: one thread per 32-value block, fp32 operations rounded
//    one at a time (bit-exact with the oracle). Codes go to the workspace the way the
//    packed weights hold their words, so that a lane fetches its codes with one or two
//    16-byte loads and needs no byte shuffle: per row of x and 256-value k-group,
//    slice t (values 8t .. 8t+7) of chunk j at byte 64t + 8j, Q8_0 in element order,
//    Q4_K in the nibble order of a packed Q4_K word (low nibbles: elements 0, 4, 1, 5;
//    high nibbles: 2, 6, 3, 7 of the slice). Rows are Kp = 256 x (k-groups) bytes
//    apart; the block scales [M][Kp/32] follow;
//  - the GEMV: one warp per weight row, all M rows of x. A k-group's record is read
//    with one 16-byte load per lane (Q4_K: 8 lanes per group, 4 groups per warp step;
//    Q8_0: 16 lanes, 2 groups), so a warp has several k-groups' bytes in flight.
//    Lane sums are joined by a fixed butterfly at the end (the same for every M).
#include "qmv_internal.h"

namespace qmv {

namespace {

__device__ __forceinline__ int dp4a_s8(uint32_t a, uint32_t b, int c) {
  int r;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(c));
  return r;
}

__device__ __forceinline__ uint4 ldg128(const uint8_t* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

// byte position, within its 8-value slice, of element p of the slice
template <int FMT>
__device__ __forceinline__ int slice_pos(int p) {
  if constexpr (FMT == F_Q4_K) return ((p & 1) << 1 | (p >> 2)) + (((p >> 1) & 1) << 2);
  return p;
}

// x (bf16 [M][K]) -> int8 codes [M][Kp] and fp32 block scales [M][Kp/32] (order above)
template <int FMT>
__global__ void quant_q8_kernel(const uint16_t* __restrict__ x, int64_t nblk, int64_t kb, int64_t kp,
                                int8_t* __restrict__ codes, float* __restrict__ scales) {
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
    const int pos = 8 * (i >> 3) + slice_pos<FMT>(i & 7);
    out[pos >> 2] |= ((uint32_t)q & 0xFFu) << (8 * (pos & 3));
  }
  const int64_t m = b / kb, blk = b % kb, g = blk >> 3;
  const int j = (int)(blk & 7);
  int8_t* dst = codes + m * kp + g * 256 + 8 * j;
#pragma unroll
  for (int t = 0; t < 4; ++t) *reinterpret_cast<uint2*>(dst + 64 * t) = make_uint2(out[2 * t], out[2 * t + 1]);
  scales[m * (kp / 32) + blk] = d;
}

// Q8_0 packed word (elements 4i .. 4i+3 of a slice, offset-binary nibbles) -> the four
// signed codes in element order. In a packed word the low nibbles of elements (0, 1)
// sit at nibbles (0, 4), of (2, 3) at (1, 5), the high nibbles at (2, 6) and (3, 7):
// A = w & 0x0F0F0F0F holds lo(e0), hi(e0), lo(e1), hi(e1) in its bytes, B = w >> 4 the
// same for e2, e3; byte 0 of A | A >> 4 is then e0's offset code, byte 2 e1's.
__device__ __forceinline__ uint32_t q80_codes4(uint32_t w) {
  const uint32_t a = w & 0x0F0F0F0Fu, b = (w >> 4) & 0x0F0F0F0Fu;
  const uint32_t ca = a | (a >> 4), cb = b | (b >> 4);
  return __byte_perm(ca, cb, 0x6420) ^ 0x80808080u;
}

// exact int -> fp32 for |v| < 2^22 (one integer add and one subtraction of 1.5 x 2^23)
__device__ __forceinline__ float i2f_small(int v) { return __int_as_float(v + 0x4B400000) - 12582912.0f; }
__device__ __forceinline__ float u6f(uint32_t v) { return __uint_as_float((v & 63u) | 0x4B000000u) - 8388608.0f; }

// One warp per weight row n (all MT rows of x). Lane l takes k-group slot l / LPG of
// each warp step (LPG lanes per group) and 16-byte piece p = l % LPG of that group's
// record:
//   Q4_K (LPG 8): bytes 16 + 16p = word t = p / 2 of chunks j0 .. j0+3, j0 = 4 (p % 2)
//     (elements 8t .. 8t+7 of each chunk); the 16-byte header by every lane;
//   Q8_0 (LPG 16): bytes 16 + 16p = words 2t, 2t+1 (t = p / 4) of chunks j0, j0+1,
//     j0 = 2 (p % 4); their fp16 d from header bytes 4 (p % 4).
template <int FMT, int MT>
__global__ void __launch_bounds__(256) int8dot_kernel(Layout L, const uint8_t* __restrict__ packed,
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
  constexpr int LPG = (FMT == F_Q4_K) ? 8 : 16;
  constexpr int GPS = 32 / LPG;                           // k-groups per warp step
  const int gs = lane / LPG, p = lane % LPG;
  float acc[MT];
#pragma unroll
  for (int m = 0; m < MT; ++m) acc[m] = 0.f;
  const int64_t G = L.k_groups, KB = L.K / 32, Kp = G * 256, KBp = G * 8;
  const uint8_t* rec0 = packed + L.base + n * L.rec;
  // one warp step: this lane's piece of k-group g
  auto step = [&](const int64_t g) {
    const uint8_t* rec = rec0 + g * L.group_bytes;
    if constexpr (FMT == F_Q4_K) {
      const int t = p >> 1;
      const uint4 w = ldg128(rec + 16 + 16 * p);
      const uint4 hd = ldg128(rec);
      // sc of chunks j0.. at bits 0, 6, 12, 18 of sw; their m at the same bits of mw
      const uint32_t sw = (p & 1) ? __funnelshift_r(hd.y, hd.z, 24) : hd.y;
      const uint32_t mw = (p & 1) ? (hd.w >> 8) : __funnelshift_r(hd.z, hd.w, 16);
      const float d = h2f(hd.x), dmin = h2f(hd.x >> 16);
      const uint32_t W[4] = {w.x, w.y, w.z, w.w};
      const int j0 = 4 * (p & 1);
      float a[4], cm[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        a[c] = __fmul_rn(d, u6f(sw >> (6 * c)));
        cm[c] = __fmul_rn(dmin, u6f(mw >> (6 * c)));
      }
#pragma unroll
      for (int m = 0; m < MT; ++m) {
        if (m >= M) break;
        const int8_t* xg = codes + m * Kp + g * 256 + 64 * t + 8 * j0;          // chunks j0 .. j0+3
        const uint4 xa = *reinterpret_cast<const uint4*>(xg), xb = *reinterpret_cast<const uint4*>(xg + 16);
        const float4 dx4 = *reinterpret_cast<const float4*>(xsc + m * KBp + g * 8 + j0);
        const uint32_t XL[4] = {xa.x, xa.z, xb.x, xb.z}, XH[4] = {xa.y, xa.w, xb.y, xb.w};
        const float DX[4] = {dx4.x, dx4.y, dx4.z, dx4.w};
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t lo = W[c] & 0x0F0F0F0Fu, hi = (W[c] >> 4) & 0x0F0F0F0Fu;
          const int s = dp4a_s8(hi, XH[c], dp4a_s8(lo, XL[c], 0));
          const int sx = dp4a_s8(0x01010101u, XH[c], dp4a_s8(0x01010101u, XL[c], 0));
          acc[m] = __fmaf_rn(__fmul_rn(a[c], DX[c]), i2f_small(s),
                             __fmaf_rn(-__fmul_rn(cm[c], DX[c]), i2f_small(sx), acc[m]));
        }
      }
    } else {   // Q8_0
      const int t = p >> 2;
      const uint4 w = ldg128(rec + 16 + 16 * p);
      const uint32_t dw = *reinterpret_cast<const uint32_t*>(rec + 4 * (p & 3));
#pragma unroll
      for (int c = 0; c < 2; ++c) {
        const int j = 2 * (p & 3) + c;
        const int64_t blk = g * 8 + j;
        if (blk >= KB) continue;      // a ragged last group: its codes and scales past K were never written
        const uint32_t c0 = q80_codes4(c ? w.z : w.x), c1 = q80_codes4(c ? w.w : w.y);
        const float dwj = h2f(c ? (dw >> 16) : dw);
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          if (m >= M) break;
          const uint2 xq = *reinterpret_cast<const uint2*>(codes + m * Kp + g * 256 + 64 * t + 8 * j);
          const float dx = xsc[m * KBp + blk];
          const int sv = dp4a_s8(c1, xq.y, dp4a_s8(c0, xq.x, 0));
          acc[m] = __fmaf_rn(__fmul_rn(dwj, dx), i2f_small(sv), acc[m]);
        }
      }
    }
  };
  // whole warp steps without a guard (so that the unrolled steps' loads can be issued
  // ahead of their arithmetic), then the ragged last step
  constexpr int kUnroll = MT == 1 ? 4 : 2;
  int64_t g0 = 0;
#pragma unroll kUnroll
  for (; g0 + GPS <= G; g0 += GPS) step(g0 + gs);
  if (g0 + gs < G) step(g0 + gs);
#pragma unroll
  for (int m = 0; m < MT; ++m) {
    float v = acc[m];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0 && m < M) y[(int64_t)m * L.N + n] = v;
  }
}

template <int FMT>
cudaError_t launch_int8dot_t(const Layout& L, const uint8_t* packed, const uint16_t* x, float* y, int M,
                             uint8_t* ws, unsigned* status, cudaStream_t s) {
  const int64_t kp = L.k_groups * 256;
  int8_t* codes = reinterpret_cast<int8_t*>(ws);
  float* xsc = reinterpret_cast<float*>(ws + align_up((int64_t)M * kp, 256));
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
  cudaError_t err = cudaLaunchKernelEx(&cfg, quant_q8_kernel<FMT>, x, nblk, L.K / 32, kp, codes, xsc);
  if (err != cudaSuccess) return err;
  cfg.gridDim = dim3((unsigned)((L.N + 7) / 8));
  cfg.blockDim = dim3(256);
  err = M <= 1 ? cudaLaunchKernelEx(&cfg, int8dot_kernel<FMT, 1>, L, packed, (const int8_t*)codes,
                                    (const float*)xsc, y, M, status)
               : cudaLaunchKernelEx(&cfg, int8dot_kernel<FMT, 8>, L, packed, (const int8_t*)codes,
                                    (const float*)xsc, y, M, status);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

int64_t int8dot_workspace_bytes(int M, int64_t K) {
  const int64_t kp = align_up(K, 256);
  return align_up((int64_t)M * kp, 256) + align_up((int64_t)M * (kp / 32) * 4, 256);
}

cudaError_t launch_int8dot(const Layout& L, const uint8_t* packed, const uint16_t* x, float* y, int M, uint8_t* ws,
                           unsigned* status, cudaStream_t s) {
  if (L.fmt == F_Q8_0) return launch_int8dot_t<F_Q8_0>(L, packed, x, y, M, ws, status, s);
  if (L.fmt == F_Q4_K) return launch_int8dot_t<F_Q4_K>(L, packed, x, y, M, ws, status, s);
  return cudaErrorInvalidValue;
}

}  // namespace qmv
