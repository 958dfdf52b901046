// qmv_w4a4.cu -- NVFP4 W4A4 prefill GEMM on the 5th-generation tensor cores:
//   y[m][n] = x_scale * s_T * sum_b s_b(x) s_b(W) sum_i e2m1(x) e2m1(W)
// with the activation quantized to NVFP4 first ("I Built a Custom Blackwell Kernel
// for Qwen3.8-27B", "What the custom path actually does": W4A4 tensor-core kernels
// after quantising the activation, for prefill).
//
// One CTA computes a 128-token x NT-row tile (NT = 256 or 128) over all of K:
//  * warp 0, one lane: streams, per 256-value k-group, the activation tile (16 KB
//    of codes + 2 KB of scales, written by the tiled activation quantizer) and the
//    weight tile (NT/128 x (16 KB + 2 KB) of the packed NVFP4 planes) into a ring
//    of shared-memory stages with cp.async.bulk; full/empty mbarriers;
//  * warp 1: allocates tensor memory (the fp32 accumulator: 128 lanes x NT
//    columns, plus the block-scale columns); one lane copies each 64-value K step's
//    block scales from shared to tensor memory (tcgen05.cp.32x128b.warpx4) and
//    issues tcgen05.mma kind::mxf4nvf4.block_scale.scale_vec::4X (M=128, N=NT,
//    K=64, E2M1 x E2M1 with UE4M3 scales per 16 values); tcgen05.commit releases
//    the stage when its MMAs have read it;
//  * warps 2..5: read the accumulator (tcgen05.ld, each warp its lane quadrant),
//    apply x_scale * s_T and store y.
// The operand tiles are exactly the packed bytes (K-major core matrices, leading
// byte offset 128, stride byte offset 1024), so no shared-memory relayout is done.
// Every wait is bounded; on expiry the CTA latches QMV_ETIMEOUT, still commits a
// final barrier (so no MMA is in flight when tensor memory is freed) and returns.
#include "qmv_internal.h"

namespace qmv {

namespace {

constexpr int kW4Threads = 192;
constexpr unsigned long long kW4TimeoutNs = 1000000000ull;
constexpr int kTileBytes = 16384 + 2048;   // codes + scales of a 128-row tile of a k-group

__device__ __forceinline__ uint32_t su32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }
__device__ __forceinline__ unsigned long long gtimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile("{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
               : "=r"(ok) : "r"(su32(b)), "r"(parity) : "memory");
  return ok != 0;
}
__device__ __forceinline__ bool wait_bounded(uint64_t* b, uint32_t parity) {
  if (try_wait(b, parity)) return true;
  const unsigned long long t0 = gtimer();
  for (uint32_t it = 1;; ++it) {
    if (try_wait(b, parity)) return true;
    if ((it & 63u) == 0 && gtimer() - t0 > kW4TimeoutNs) return false;
  }
}
__device__ __forceinline__ void bulk(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   su32(dst)), "l"(src), "r"(bytes), "r"(su32(bar))
               : "memory");
}
// shared-memory matrix descriptor: start, leading and stride byte offsets (>> 4),
// descriptor version 1, no swizzle
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         ((uint64_t)1 << 46);
}

struct W4Params {
  Layout L;
  const uint8_t* packed;
  const uint8_t* act;        // activation planes: per k-group m_pad*128 B codes + m_pad*16 B scales
  float* y;
  float scale;               // x_scale * s_T is formed on the device (s_T in the packed extras)
  int M;
  int64_t m_pad;
  int m_tiles;
  int stages;
  int stage_bytes;
  unsigned* status;
};

template <int NT>
__global__ void __launch_bounds__(kW4Threads, 1) w4a4_kernel(const W4Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr int kTiles = NT / 128;
  const Layout& L = p.L;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + 8;
  uint64_t* done = empty + 8;
  volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(smem + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 260);
  uint8_t* stage0 = smem + 1024;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = (int)(blockIdx.x % p.m_tiles), n_tile = (int)(blockIdx.x / p.m_tiles);
  const int G = (int)L.k_groups;

  if (threadIdx.x == 0) {
    const PackedHeader* h = reinterpret_cast<const PackedHeader*>(p.packed);
    const bool bad = !(h->magic == kMagic && h->version == kVersion && h->fmt == (uint32_t)F_NVFP4 &&
                       h->N == L.N && h->K == L.K && h->E == 1 && h->expert_bytes == L.expert_bytes);
    if (bad) atomicOr(p.status, kStatHeader);
    *abort_flag = bad ? 1 : 0;
    for (int i = 0; i < p.stages; ++i) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&full[i])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&empty[i])));
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(done)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    // the accumulator (NT columns) and two buffers of block-scale columns; 512
    // columns, so one CTA per SM holds them (the shared memory use allows no more)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(su32((const void*)tslot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tslot;
  const bool bad_header = *abort_flag != 0;

  const int64_t act_plane = p.m_pad * 144;
  if (warp == 0) {
    // ------------------------------ producer --------------------------------
    if (lane == 0 && !bad_header) {
      const uint32_t bytes = (uint32_t)(kTileBytes * (1 + kTiles));
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      for (int kg = 0; kg < G; ++kg) {
        if (kg >= p.stages && !wait_bounded(&empty[stage], phase ^ 1u)) {
          atomicOr(p.status, kStatTimeout);
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        uint8_t* st = stage0 + stage * p.stage_bytes;
        const uint8_t* ap = p.act + kg * act_plane;
        const uint8_t* wp = p.packed + kHeaderBytes + kg * L.group_bytes;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(&full[stage])), "r"(bytes)
                     : "memory");
        bulk(st, ap + (int64_t)m_tile * 16384, 16384, &full[stage]);
        bulk(st + 16384, ap + p.m_pad * 128 + (int64_t)m_tile * 2048, 2048, &full[stage]);
        bulk(st + kTileBytes, wp + (int64_t)n_tile * kTiles * 16384, 16384 * kTiles, &full[stage]);
        bulk(st + kTileBytes + 16384 * kTiles, wp + L.plane_a + (int64_t)n_tile * kTiles * 2048, 2048 * kTiles,
             &full[stage]);
        ++issued;
        if (++stage == p.stages) { stage = 0; phase ^= 1u; }
      }
      // copies still in flight land before the CTA can exit
      for (int j = (issued > p.stages ? issued - p.stages : 0); j < issued; ++j)
        (void)wait_bounded(&full[j % p.stages], (uint32_t)((j / p.stages) & 1));
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      // kind::mxf4nvf4 instruction descriptor: A, B E2M1 (1) at bits 7 and 10,
      // K-major, N / 8 at bit 17, UE4M3 scales (bit 23 clear), M / 16 at bit 24
      const uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(NT >> 3) << 17) | ((128u >> 4) << 24);
      int stage = 0;
      uint32_t phase = 0;
      for (int kg = 0; kg < G && !bad_header; ++kg) {
        if (!wait_bounded(&full[stage], phase)) {
          atomicOr(p.status, kStatTimeout);
          *abort_flag = 1;
          break;
        }
        if (*abort_flag) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint8_t* st = stage0 + stage * p.stage_bytes;
        const uint32_t a_codes = su32(st), a_sf = su32(st + 16384);
        const uint32_t b_codes = su32(st + kTileBytes), b_sf = su32(st + kTileBytes + 16384 * kTiles);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          // block-scale columns: buffer (kg & 1), step ks: A 4 columns, B 4 per 128 rows
          const uint32_t sfa = tmem + 256 + (uint32_t)((kg & 1) * 48 + ks * 12);
          const uint32_t sfb = sfa + 4;
          asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(sfa),
                       "l"(sdesc(a_sf + 512 * ks, 128, 128)));
#pragma unroll
          for (int h = 0; h < kTiles; ++h)
            asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(sfb + 4 * h),
                         "l"(sdesc(b_sf + 2048 * h + 512 * ks, 128, 128)));
          const uint64_t ad = sdesc(a_codes + 256 * ks, 128, 1024);
          const uint64_t bd = sdesc(b_codes + 256 * ks, 128, 1024);
          const uint32_t acc = (kg > 0 || ks > 0) ? 1u : 0u;
          asm volatile(
              "{ .reg .pred p; setp.ne.b32 p, %6, 0;\n"
              "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p; }"
              ::"r"(tmem), "l"(ad), "l"(bd), "r"(idesc), "r"(sfa), "r"(sfb), "r"(acc)
              : "memory");
        }
        // the stage is free once these MMAs (and copies) have read it
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                         su32(&empty[stage]))
                     : "memory");
        if (++stage == p.stages) { stage = 0; phase ^= 1u; }
      }
      // always: arrives when every MMA issued above has completed
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(done))
                   : "memory");
    }
  } else {
    // ------------------------------ epilogue --------------------------------
    const bool ok = wait_bounded(done, 0u);
    if (!ok) atomicOr(p.status, kStatTimeout);
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if (ok && !*abort_flag) {
      const int q = warp & 3;                              // this warp's lane quadrant
      const int64_t m = (int64_t)m_tile * 128 + 32 * q + lane;
      const float sT = *reinterpret_cast<const float*>(p.packed + kHeaderBytes + L.k_groups * L.group_bytes);
      const float scale = p.scale * sT;
#pragma unroll 1
      for (int c0 = 0; c0 < NT; c0 += 32) {
        uint32_t r[32];
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
            "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
            : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
              "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
              "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
              "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
              "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
            : "r"(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)c0));
        asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
        const int64_t n0 = (int64_t)n_tile * NT + c0;
        if (m < p.M) {
          float* yr = p.y + m * L.N + n0;
          if (n0 + 32 <= L.N && (L.N & 3) == 0) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              *reinterpret_cast<float4*>(yr + j) =
                  make_float4(__uint_as_float(r[j]) * scale, __uint_as_float(r[j + 1]) * scale,
                              __uint_as_float(r[j + 2]) * scale, __uint_as_float(r[j + 3]) * scale);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (n0 + j < L.N) yr[j] = __uint_as_float(r[j]) * scale;
          }
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    // no MMA may still write the accumulator when it is freed
    if (lane == 0) (void)wait_bounded(done, 0u);
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
  }
}

template <int NT>
cudaError_t launch_nt(W4Params p, int grid, cudaStream_t s) {
  int dev = 0, smem_max = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (err != cudaSuccess) return err;
  p.stage_bytes = kTileBytes * (1 + NT / 128);
  p.stages = (smem_max - 1024) / p.stage_bytes;
  if (p.stages > 8) p.stages = 8;
  if (p.stages < 2) return cudaErrorInvalidConfiguration;
  const int smem = 1024 + p.stages * p.stage_bytes;
  static int opted[64] = {0};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (opted[dev] < smem) {
    err = cudaFuncSetAttribute(w4a4_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    opted[dev] = smem;
  }
  w4a4_kernel<NT><<<grid, kW4Threads, smem, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_w4a4(const Layout& L, const uint8_t* packed, const uint8_t* act_planes, float x_scale,
                        float* y, int M, int64_t m_pad, unsigned* status, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  W4Params p;
  p.L = L;
  p.packed = packed;
  p.act = act_planes;
  p.y = y;
  p.scale = x_scale;
  p.M = M;
  p.m_pad = m_pad;
  p.m_tiles = (int)(m_pad / 128);
  p.status = status;
  p.stages = 0;
  p.stage_bytes = 0;
  // 256-row weight tiles when they give at least one CTA per SM, else 128-row ones
  const int64_t tiles256 = (L.n_pad % 256 == 0) ? (L.n_pad / 256) * p.m_tiles : 0;
  if (tiles256 >= sms) return launch_nt<256>(p, (int)tiles256, s);
  return launch_nt<128>(p, (int)((L.n_pad / 128) * p.m_tiles), s);
}

}  // namespace qmv
