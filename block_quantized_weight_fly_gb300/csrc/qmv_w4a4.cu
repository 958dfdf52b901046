// qmv_w4a4.cu -- NVFP4 W4A4 prefill GEMM on the 5th-generation tensor cores:
//   y[m][n] = x_scale * s_T * sum_b s_b(x) s_b(W) sum_i e2m1(x) e2m1(W)
// with the activation quantized to NVFP4 first ("I Built a Custom Blackwell Kernel
// for Qwen3.8-27B", "What the custom path actually does": W4A4 tensor-core kernels
// after quantising the activation, for prefill).
//
// Work: output tiles of 128 tokens x NT weight rows (NT = 256, or 128 when N is not
// a multiple of 256), each a sum over K's 256-value k-groups. The grid (at most one
// CTA per SM) is split into one group of CTAs per 128-token tile; each group cuts
// the same (weight tile, k-group) sequence into equal contiguous ranges, so every
// SM gets the same tensor work whatever the tile count, and the CTAs of different
// groups with the same rank stream the same weight tiles at about the same time
// (one HBM read serves all token tiles). A tile split between CTAs is finished by the CTA holding
// its first k-group (that part is the last of its range, so every stage buffer is
// free by then). The other parts are each their CTA's first part: the CTA stores
// its fp32 partial sums in its own slot of the workspace and raises its flag with a
// release store. The finishing CTA acquires its peers' flags, pulls their slots into
// the free stage buffers with bulk copies, adds them in CTA order and clears the
// flags (all flags are zero again after a call).
//
// One CTA (320 threads):
//  * warp 0, one lane: streams each unit's operands -- the activation tile (16 KB of
//    codes + 2 KB of block scales, written by the tiled activation quantizer) and the
//    weight tile (NT/128 x (16 KB + 2 KB) of the packed NVFP4 planes) -- into a ring
//    of shared-memory stages with cp.async.bulk; full/empty mbarriers. The weight
//    copies of the first stages go out before the grid-dependency wait (they do not
//    depend on the quantizer that runs just before), the activation copies after it;
//  * warp 1: allocates tensor memory (the fp32 accumulator, NT columns, plus two
//    buffers of block-scale columns); one lane copies each 64-value K step's block
//    scales from shared to tensor memory (tcgen05.cp.32x128b.warpx4) and issues
//    tcgen05.mma kind::mxf4nvf4.block_scale.scale_vec::4X (M=128, N=NT, K=64, E2M1 x
//    E2M1 with UE4M3 scales per 16 values); tcgen05.commit releases each stage and,
//    after a part's last k-group, signals the epilogue;
//  * warps 2..9: read the accumulator (tcgen05.ld; two warps per 32-lane quadrant,
//    each a quarter of every column half, 16 columns at a time, the next load
//    issued before the stores of the last), hand it back to the MMA warp as soon
//    as every column is read, and write each row's 64-byte pieces: y (scaled by
//    x_scale * s_T), or the partial sums, or y after adding the peers' partial
//    sums. The eight epilogue warps take every abort decision together, after a
//    named barrier.
// The operand tiles are exactly the packed bytes (K-major core matrices, leading
// byte offset 128, stride byte offset 1024), so no shared-memory relayout is done.
// Every wait is bounded; on expiry the CTA latches QMV_ETIMEOUT and stops. The MMA
// lane always commits a final barrier, which warp 1 waits for before freeing tensor
// memory, so no MMA is in flight when it is freed.
#include "qmv_internal.h"

namespace qmv {

namespace {

constexpr int kW4Threads = 320;            // producer, MMA issuer, 8 epilogue warps
constexpr unsigned long long kW4TimeoutNs = 1000000000ull;
constexpr int kTileBytes = 16384 + 2048;   // codes + scales of a 128-row tile of a k-group
constexpr int kMaxW4Stages = 8;
constexpr int kStageOff = 1024;             // control block, then the stages

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
__device__ __forceinline__ void arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
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
__device__ __forceinline__ uint32_t ld_acquire(const unsigned* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(unsigned* p, uint32_t v) {
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void st_relaxed(unsigned* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// 16 consecutive accumulator columns of this warp's 32 lanes (lane = row), and the
// wait for every load issued so far
__device__ __forceinline__ void tld16(uint32_t* r, uint32_t taddr) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
// the eight epilogue warps (256 threads) meet at named barrier 1
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

struct W4Params {
  Layout L;
  const uint8_t* packed;
  const uint8_t* act;        // activation planes: per k-group m_pad*128 B codes + m_pad*16 B scales
  float* y;
  float* partials;           // per CTA a slot: [2 column halves][128 rows][NT/2 columns] fp32
  unsigned* flags;           // per CTA: 1 while its slot holds a published part
  float scale;               // x_scale (times s_T, read from the packed extras on the device)
  int M;
  int64_t m_pad;
  int m_tiles;
  int units;                 // units of one token tile's group: weight tiles x k-groups
  int stages;
  int stage_bytes;
  unsigned* status;
};

// first unit of CTA i's range (units * gridDim < 2^31 is checked on the host)
__device__ __forceinline__ int range_start(int i, int units, int P) {
  const int q = units / P, r = units % P;
  return i * q + (i * r) / P;
}

template <int NT>
__global__ void __launch_bounds__(kW4Threads, 1) w4a4_kernel(const W4Params p) {
  extern __shared__ __align__(1024) uint8_t smem[];
  constexpr int kTiles = NT / 128;
  const Layout& L = p.L;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxW4Stages;
  uint64_t* acc_full = empty + kMaxW4Stages;     // MMA lane -> epilogue: a part's sums are complete
  uint64_t* acc_free = acc_full + 1;             // epilogue -> MMA lane: the accumulator was read
  uint64_t* done = acc_free + 1;                 // every MMA of the CTA has completed
  uint64_t* pbar = done + 1;                     // peers' partial sums copied into the stages
  volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(smem + 512);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 516);
  volatile int* epi_abort = reinterpret_cast<volatile int*>(smem + 520);   // written by the epilogue leader only
  uint8_t* stage0 = smem + kStageOff;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = (int)L.k_groups;
  const int P = (int)gridDim.x;
  const int c = (int)blockIdx.x;
  const int m_tile = c % p.m_tiles;           // this CTA's token tile
  const int Pg = P / p.m_tiles;                // CTAs per token tile (the grid is a multiple)
  const int j = c / p.m_tiles;                 // rank within the group; peers are j + 1, ...
  const int u0 = range_start(j, p.units, Pg), u1 = range_start(j + 1, p.units, Pg);

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
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(acc_full)));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 8;" ::"r"(su32(acc_free)));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(done)));
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(pbar)));
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
      const int n = u1 - u0;
      const int first = n < p.stages ? n : p.stages;
      // the weights of the first round of stages (independent of the quantizer)
      for (int i = 0; i < first; ++i) {
        const int u = u0 + i, kg = u % G, n_tile = u / G;
        uint8_t* st = stage0 + i * p.stage_bytes;
        const uint8_t* wp = p.packed + kHeaderBytes + kg * L.group_bytes;
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(&full[i])), "r"(bytes)
                     : "memory");
        bulk(st + kTileBytes, wp + (int64_t)n_tile * kTiles * 16384, 16384 * kTiles, &full[i]);
        bulk(st + kTileBytes + 16384 * kTiles, wp + L.plane_a + (int64_t)n_tile * kTiles * 2048, 2048 * kTiles,
             &full[i]);
      }
      asm volatile("griddepcontrol.wait;" ::: "memory");     // the activation planes
      int stage = 0;
      uint32_t phase = 0;
      int issued = 0;
      for (int i = 0; i < n; ++i) {
        const int u = u0 + i, kg = u % G, n_tile = u / G;
        uint8_t* st = stage0 + stage * p.stage_bytes;
        if (i >= p.stages) {   // a later round: the stage's previous unit must be consumed
          if (!wait_bounded(&empty[stage], phase ^ 1u)) {
            atomicOr(p.status, kStatTimeout);
            *abort_flag = 1;
            break;
          }
          if (*abort_flag) break;
          const uint8_t* wp = p.packed + kHeaderBytes + kg * L.group_bytes;
          asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(&full[stage])),
                       "r"(bytes)
                       : "memory");
          bulk(st + kTileBytes, wp + (int64_t)n_tile * kTiles * 16384, 16384 * kTiles, &full[stage]);
          bulk(st + kTileBytes + 16384 * kTiles, wp + L.plane_a + (int64_t)n_tile * kTiles * 2048,
               2048 * kTiles, &full[stage]);
        }
        const uint8_t* ap = p.act + kg * act_plane;
        bulk(st, ap + (int64_t)m_tile * 16384, 16384, &full[stage]);
        bulk(st + 16384, ap + p.m_pad * 128 + (int64_t)m_tile * 2048, 2048, &full[stage]);
        issued = i + 1;
        if (++stage == p.stages) { stage = 0; phase ^= 1u; }
      }
      // copies still in flight land before the CTA can exit (every stage of the first
      // round got its activation copies above: the loop cannot stop before it)
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
      int part = 0;
      for (int u = u0; u < u1 && !bad_header; ++u) {
        const int kg = u % G;
        const bool part_start = (u == u0) || (kg == 0);
        const bool part_end = (u == u1 - 1) || (kg == G - 1);
        bool ok = true;
        // a new part overwrites the accumulator: the epilogue must have read the last one
        if (part_start && part > 0) ok = wait_bounded(acc_free, (uint32_t)((part - 1) & 1));
        if (ok) ok = wait_bounded(&full[stage], phase);
        if (!ok) {
          atomicOr(p.status, kStatTimeout);
          *abort_flag = 1;
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
          const uint32_t acc = (!part_start || ks > 0) ? 1u : 0u;
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
        if (part_end) {
          asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                           su32(acc_full))
                       : "memory");
          ++part;
        }
        if (++stage == p.stages) { stage = 0; phase ^= 1u; }
      }
      // always: arrives when every MMA issued above has completed
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(done))
                   : "memory");
    }
  } else {
    // ------------------------------ epilogue --------------------------------
    constexpr int kHalf = 128 * (NT / 2);               // fp32 words of one column half of a slot
    const int q = warp & 3;                              // this warp's lane quadrant: rows 32q .. 32q+31
    const int grp = (warp - 2) >> 2;                     // which quarter of each column half
    const bool leader = threadIdx.x == 64;               // the first epilogue thread
    const int row = 32 * q + lane;                       // this thread's row of the tile
    const float sT = *reinterpret_cast<const float*>(p.packed + kHeaderBytes + L.k_groups * L.group_bytes);
    const float scale = p.scale * sT;
    const bool vec_ok = (L.N & 3) == 0;
    float* slot = p.partials + (int64_t)c * (2 * kHalf);
    // Any warp may raise the CTA's abort flag at any time; the epilogue warps act on
    // one snapshot of it, taken by the leader between two barriers, so all four take
    // the same branch and none is left waiting at a barrier.
    auto decide_abort = [&]() -> bool {
      epi_sync();
      if (leader) *epi_abort = *abort_flag;
      epi_sync();
      return *epi_abort != 0;
    };
    int part = 0;
    for (int pu0 = u0; pu0 < u1;) {
      const int t = pu0 / G;
      const int pu1 = ((t + 1) * G < u1) ? (t + 1) * G : u1;
      const bool head = (pu0 % G) == 0;                  // holds the tile's first k-group
      const bool whole = head && (pu1 - pu0 == G);
      const int n_tile = t;
      // the peers of a finishing part: the next CTAs, whose ranges start in this tile
      int npeer = 0;
      if (head && !whole)
        while (j + 1 + npeer < Pg && range_start(j + 1 + npeer, p.units, Pg) < (t + 1) * G) ++npeer;
      const bool staged = npeer * kHalf * 4 <= p.stages * p.stage_bytes;
      if (bad_header || !wait_bounded(acc_full, (uint32_t)(part & 1))) {
        if (!bad_header) atomicOr(p.status, kStatTimeout);
        *abort_flag = 1;
      }
      if (head && !whole && leader && !*abort_flag) {
        // the peers published before their ranges moved on; acquire their flags, then
        // let the copy engine read their slots (every stage buffer is free: this is the
        // CTA's last part and its MMAs have completed)
        for (int k = 0; k < npeer; ++k) {
          const unsigned* f = p.flags + c + (1 + k) * p.m_tiles;
          bool got = ld_acquire(f) != 0u;
          const unsigned long long t0 = gtimer();
          while (!got && gtimer() - t0 <= kW4TimeoutNs) got = ld_acquire(f) != 0u;
          if (!got) { atomicOr(p.status, kStatTimeout); *abort_flag = 1; break; }
        }
        asm volatile("fence.proxy.async.global;" ::: "memory");
      }
      if (decide_abort()) break;
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      int h = 0;
      // one 16-column chunk of row `row` of the part, in registers: four 16-byte pieces
      auto store_chunk = [&](const uint32_t* r, int c0) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int col = c0 + 4 * i;                                 // column of the tile
          const int hw = row * (NT / 2) + (col - h * (NT / 2));       // word within a slot half
          float4 v = make_float4(__uint_as_float(r[4 * i]), __uint_as_float(r[4 * i + 1]),
                                 __uint_as_float(r[4 * i + 2]), __uint_as_float(r[4 * i + 3]));
          if (!head) {                                                // another CTA finishes it
            *reinterpret_cast<float4*>(slot + h * kHalf + hw) = v;
            continue;
          }
          for (int k = 0; k < npeer; ++k) {                           // the peers' parts, in order
            const float4 x = staged ? *reinterpret_cast<const float4*>(stage0 + 4 * (k * kHalf + hw))
                                    : __ldcg(reinterpret_cast<const float4*>(
                                          p.partials + (int64_t)(c + (1 + k) * p.m_tiles) * (2 * kHalf) + h * kHalf + hw));
            v.x += x.x; v.y += x.y; v.z += x.z; v.w += x.w;
          }
          const int64_t m = (int64_t)m_tile * 128 + row;
          const int64_t n0 = (int64_t)n_tile * NT + col;
          if (m >= p.M) continue;
          float* yr = p.y + m * L.N + n0;
          if (vec_ok && n0 + 4 <= L.N) {
            *reinterpret_cast<float4*>(yr) = make_float4(v.x * scale, v.y * scale, v.z * scale, v.w * scale);
          } else {
            const float e4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
              if (n0 + e < L.N) yr[e] = e4[e] * scale;
          }
        }
      };
      for (h = 0; h < 2; ++h) {
        if (head && !whole && staged) {
          if (leader) {
            asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(pbar)),
                         "r"((uint32_t)(npeer * kHalf * 4))
                         : "memory");
            for (int k = 0; k < npeer; ++k)
              bulk(stage0 + k * kHalf * 4, p.partials + (int64_t)(c + (1 + k) * p.m_tiles) * (2 * kHalf) + h * kHalf,
                   (uint32_t)(kHalf * 4), pbar);
          }
          if (!wait_bounded(pbar, (uint32_t)h)) { atomicOr(p.status, kStatTimeout); *abort_flag = 1; }
          if (decide_abort()) break;
        }
        // This warp's quarter of the half, 16 columns at a time, each load issued
        // before the previous chunk's stores so that its latency overlaps them.
        constexpr int kQ = NT / 4;                       // columns per warp per half
        const int cbase = h * (NT / 2) + grp * kQ;
        const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16);
        uint32_t ra[16], rb[16];
        tld16(ra, tq + (uint32_t)cbase);
#pragma unroll 1
        for (int cc = 0; cc < kQ; cc += 32) {
          const int c0 = cbase + cc;
          tld_wait();
          tld16(rb, tq + (uint32_t)(c0 + 16));
          store_chunk(ra, c0);
          tld_wait();
          if (h == 1 && cc + 32 == kQ) {
            // every column of this part is in registers now: the MMA lane may overwrite it
            asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
            __syncwarp();
            if (lane == 0) arrive(acc_free);
          }
          if (cc + 32 < kQ) tld16(ra, tq + (uint32_t)(c0 + 32));
          store_chunk(rb, c0 + 16);
        }
        // the next half's copies overwrite the stage buffers only after every thread read them
        if (head && !whole && staged) epi_sync();
      }
      if (decide_abort()) break;
      if (!head) {
        // publish: every epilogue thread's stores of this slot before the flag
        epi_sync();
        if (leader) st_release(p.flags + c, 1u);
      } else if (!whole) {
        epi_sync();
        if (leader)
          for (int k = 0; k < npeer; ++k) st_relaxed(p.flags + c + (1 + k) * p.m_tiles, 0u);
      }
      ++part;
      pu0 = pu1;
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
  p.stages = (smem_max - kStageOff) / p.stage_bytes;
  if (p.stages > kMaxW4Stages) p.stages = kMaxW4Stages;
  if (p.stages < 2) return cudaErrorInvalidConfiguration;
  const int smem = kStageOff + p.stages * p.stage_bytes;
  static int opted[64] = {0};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (opted[dev] < smem) {
    err = cudaFuncSetAttribute(w4a4_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    opted[dev] = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kW4Threads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  // The grid has at most one CTA per SM, so all its CTAs are resident together once
  // the kernels before it have left (a finishing CTA's bounded wait on its peers'
  // partial sums ends). Programmatic serialization lets the prologue and the first
  // weight copies overlap the activation quantizer launched just before.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, w4a4_kernel<NT>, p);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace

// per SM: a slot of 128 x 256 fp32 partial sums; then one flag word per SM
int64_t w4a4_partials_bytes(int sms) { return (int64_t)sms * 128 * 256 * 4 + align_up((int64_t)sms * 4, 256); }

cudaError_t launch_w4a4(const Layout& L, const uint8_t* packed, const uint8_t* act_planes, uint8_t* partials,
                        float x_scale, float* y, int M, int64_t m_pad, unsigned* status, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  W4Params p;
  p.L = L;
  p.packed = packed;
  p.act = act_planes;
  p.partials = reinterpret_cast<float*>(partials);
  p.flags = reinterpret_cast<unsigned*>(partials + (int64_t)sms * 128 * 256 * 4);
  p.y = y;
  p.scale = x_scale;
  p.M = M;
  p.m_pad = m_pad;
  p.m_tiles = (int)(m_pad / 128);
  p.status = status;
  p.stages = 0;
  p.stage_bytes = 0;
  // 256-row weight tiles when N allows them, else 128-row ones
  const bool wide = (L.n_pad % 256) == 0;
  const int64_t units = (L.n_pad / (wide ? 256 : 128)) * L.k_groups;   // per token tile
  if (units <= 0 || units * (int64_t)sms >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  // one group of CTAs per token tile, all resident at once (one CTA per SM)
  int64_t per = sms / p.m_tiles;
  if (per < 1) return cudaErrorInvalidValue;            // more token tiles than SMs
  if (per > units) per = units;
  p.units = (int)units;
  const int grid = (int)(per * p.m_tiles);
  return wide ? launch_nt<256>(p, grid, s) : launch_nt<128>(p, grid, s);
}

}  // namespace qmv
