// qmv_kq.cu -- K-quant (Q4_K, Q5_K) prefill GEMM on the 5th-generation tensor cores:
//   y[m][n] = sum_k x[m][k] w[n][k],  w = d sc_j q - dmin m_j  (per 256-value superblock kb
// of row n and 32-value sub-block j), for M in the hundreds to thousands of tokens, with
// each weight slab streamed from HBM once per call instead of once per 8 tokens (the
// re-streaming that made prefill slow on the Tenstorrent card: "Qwen3.8-27B on one
// Tenstorrent P150", "3. Porting the 9B stack to 27B geometry", its prefill fixes; the
// per-sub-block factored form of
// the decode kernels: "I Built a Custom Blackwell Kernel for Qwen3.8-27B", "What the
// custom path actually does").
//
// Arithmetic. Per superblock the sum splits into
//   D1[n][m] = sum_k (sc_j q)[n][k] 2^-14 * x[m][k]          (f16 x f16, fp32 accumulator)
//   D2[n][m] = sum_j m_j[n] (xs_hi[m][j] + xs_lo[m][j])      (f16 x f16, fp32 accumulator)
//   y[m][n] += (d[n] 2^14) D1[n][m] - dmin[n] D2[n][m]       (fp32, per superblock)
// where xs = the fp32 sum of x over the sub-block, split into two f16 (hi + lo, 2^-22
// relative). Q6_K (w = d sc_u (q - 32) per 16-value unit u, sc_u int8) has no min
// term; sc_u (q - 32) needs up to 12 significant bits, one more than f16 holds, so the
// scale is split, sc_u = 16 sh_u + sl_u (sh_u = sc_u >> 4, sl_u = sc_u & 15), and each K
// step takes two MMAs into D1: A = (q - 32) 16 sh_u (|.| <= 4096, 9 significant bits)
// and A = (q - 32) sl_u (|.| <= 480); both exact, y[m][n] += d[n] D1[n][m]. sc_j q <= 63 * 15 = 945 (Q5_K: 63 * 31 = 1953) and m_j <= 63 are exact in
// f16; the decoder makes sc_j q 2^-14 with one mask (the field lands in f16's subnormal
// range: q 2^-24, or q 2^-20 for a Q4_K high nibble) and one f16 multiply by sc_j 2^10
// (2^6), so every product is exact and only the fp32 accumulations round. x is taken in f16 (exact for bf16
// values of magnitude 2^-14 .. 65504; smaller ones keep an absolute error below 2^-25).
//
// Work: output tiles of 128 weight rows x 128 tokens, each a sum over K's superblocks;
// units = (tile, superblock), tiles ordered token tile fastest (the four token tiles
// of a weight tile follow each other, so its weights come from L2 after the first).
// The grid (one CTA per SM) cuts the unit sequence into equal contiguous ranges; a tile
// split between CTAs is finished by the CTA holding its first superblock (the last part
// of that CTA's range), which adds the peers' published fp32 partial tiles (a
// workspace slot per CTA, a flag raised with a release store) in CTA order.
//
// One CTA (448 threads):
//  * warp 0, one lane: after the grid-dependency wait (the activation tiles come from
//    the pre-pass launched just before), bulk-copies per superblock the x sub-block-sum
//    tile (4 KB) and the four 64-value K steps of the x tile (16 KB each) into rings;
//  * warps 2..5, one thread per weight row: load the row's 144-byte Q4_K (176-byte Q5_K) record of the
//    superblock from global memory (the next unit's is loaded while the current one is
//    decoded), write the mins tile row (m_j as f16, twice) and (d 2^14, dmin), then
//    decode each K step into the decoded-weight ring (K-major core matrices);
//  * warp 1: allocates 512 tensor-memory columns -- two buffers of (D1: 128 columns,
//    D2: 128 columns) -- and one lane issues per K step four tcgen05.mma kind::f16
//    (M = 128 rows, N = 128 tokens, K = 16) into D1 of the unit's buffer, then one for
//    D2; commits release the ring slots and hand the buffer to the epilogue;
//  * warps 6..13: two warps per lane quadrant, 64 tokens each: per superblock read D1
//    and D2 (tcgen05.ld) and fold them into the fp32 tile kept in registers; at the end
//    of a part store y, or publish the partial tile, or add the peers' and store y.
// Every wait is bounded; on expiry the CTA latches QMV_ETIMEOUT and stops. The MMA lane
// always commits a final barrier, which warp 1 waits for before freeing tensor memory.
#include "qmv_internal.h"

namespace qmv {

namespace {

constexpr int kKqThreads = 448;
constexpr unsigned long long kKqTimeoutNs = 1000000000ull;
constexpr int kKqCtrl = 1024;
constexpr int kXSlots = 8;                     // x K-step tiles: 128 tokens x 64 f16
constexpr int kASlots = 4;                     // decoded weight K-step tiles: 128 rows x 64 f16
constexpr int kSSlots = 3;                     // per superblock: sums tile | mins tile | row scales
constexpr int kStepBytes = 16384;
constexpr int kSumsOff = 0, kMinsOff = 4096, kSclOff = 8192, kSBytes = 9216;
constexpr int kXOff = kKqCtrl;
constexpr int kAOff = kXOff + kXSlots * kStepBytes;
constexpr int kSOff = kAOff + kASlots * kStepBytes;
constexpr int kKqSmem = kSOff + kSSlots * kSBytes;     // 225280 bytes
constexpr int kSlotWords = 128 * 128;                  // fp32 words of a partial tile

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
    if ((it & 63u) == 0 && gtimer() - t0 > kKqTimeoutNs) return false;
  }
}
// lane 0 waits, the warp learns the outcome
__device__ __forceinline__ bool warp_wait(uint64_t* b, uint32_t parity, int lane) {
  int ok = 1;
  if (lane == 0) ok = wait_bounded(b, parity) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}
__device__ __forceinline__ void arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   su32(dst)), "l"(src), "r"(bytes), "r"(su32(bar))
               : "memory");
}
__device__ __forceinline__ void commit(uint64_t* b) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(su32(b))
               : "memory");
}
// shared-memory matrix descriptor: start, leading and stride byte offsets (>> 4),
// descriptor version 1, no swizzle
__device__ __forceinline__ uint64_t sdesc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) | ((uint64_t)(sbo >> 4) << 32) |
         ((uint64_t)1 << 46);
}
__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{ .reg .pred p; setp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
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
__device__ __forceinline__ uint4 ldg_nc(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// a small exact value v (f16-representable) in both halves of an f16x2
__device__ __forceinline__ uint32_t f16x2_dup(float v) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %1;" : "=r"(r) : "f"(v));
  return r;
}
__device__ __forceinline__ void tld16(uint32_t* r, uint32_t taddr) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// 32-bit word w of a packed record (byte offset o, a compile-time constant after unrolling)
template <int NV>
__device__ __forceinline__ uint32_t rec_word(const uint4 (&cur)[NV], int o) {
  const uint4 cv = cur[o >> 4];
  const int e = (o & 15) >> 2;
  return e == 0 ? cv.x : e == 1 ? cv.y : e == 2 ? cv.z : cv.w;
}

// The eight values (elements 8t..8t+7 of sub-block j) of one packed word as sc_j q 2^-14
// in f16 pairs: each pair masked into f16's subnormal range (q 2^-24, or q 2^-20 for a
// Q4_K high nibble) and multiplied by sc_j 2^10 (2^6), exact.
template <int FMT, int NV>
__device__ __forceinline__ uint4 kq_decode_word(const uint4 (&cur)[NV], int t, int j, uint32_t S, uint32_t S16) {
  uint4 out;
  if constexpr (FMT == F_Q4_K) {
    // nibbles (p, p+4) = elements (8t+2p, 8t+2p+1)
    const uint32_t w = rec_word(cur, 16 + 32 * t + 4 * j), w8 = w >> 8;
    out.x = hmul2(w & 0x000F000Fu, S);
    out.y = hmul2(w & 0x00F000F0u, S16);
    out.z = hmul2(w8 & 0x000F000Fu, S);
    out.w = hmul2(w8 & 0x00F000F0u, S16);
  } else {
    // Q5_K: pairs p = 0..2 as 5-bit fields at bits (5p, 16+5p); the last pair's low
    // nibbles in the sub-block's nibble word (nibbles t, t+4), fifth bits at 15, 31
    (void)S16;
    const uint32_t v = rec_word(cur, 16 + 32 * t + 4 * j), u = rec_word(cur, 144 + 4 * j);
    out.x = hmul2(v & 0x001F001Fu, S);
    out.y = hmul2((v >> 5) & 0x001F001Fu, S);
    out.z = hmul2((v >> 10) & 0x001F001Fu, S);
    out.w = hmul2(((u >> (4 * t)) & 0x000F000Fu) | ((v >> 11) & 0x00100010u), S);
  }
  return out;
}

// Q6_K: the f16 values q - 32 of elements (8g .. 8g+7) of the 64-value K step s of a
// packed record (ql word t of chunk j at 32t + 4j, qh word h at 128 + 32h + 4j; see
// qmv_layout.cuh), as four f16 pairs
template <int NV>
__device__ __forceinline__ void q6k_step_pairs(const uint4 (&cur)[NV], int s, int g, uint32_t* v) {
  const int j = 2 * s + (g >> 2);           // chunk
  const int half = (g & 3) >> 1;            // 16-value half of the chunk
  const int w0 = 2 * (g & 1);               // the two quads of 4 elements: w0, w0 + 1
  const uint32_t qh = rec_word(cur, 128 + 32 * (w0 >> 1) + 4 * j);
#pragma unroll
  for (int qd = 0; qd < 2; ++qd) {
    const int w = w0 + qd;
    const uint32_t ql = rec_word(cur, 32 * w + 4 * j);
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
      const int k = 2 * half + pr;          // pair index within the words
      const uint32_t lo = (ql >> (4 * k)) & 0x000F000Fu;
      const uint32_t hi = (qh >> (8 * (w & 1) + 2 * k)) & 0x00030003u;
      const uint32_t p = lo | (hi << 4) | 0x64006400u;                 // {1024 + q, 1024 + q'}
      uint32_t r;
      asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(p), "r"(0x64206420u));   // - 1056: {q - 32, q' - 32}
      v[2 * qd + pr] = r;
    }
  }
}

struct KqParams {
  Layout L;
  const uint8_t* packed;
  const uint8_t* xt;         // x tiles: [m_tile][K step] 16 KB each
  const uint8_t* sums;       // x sub-block-sum tiles: [m_tile][superblock] 4 KB each
  float* y;
  float* partials;           // per CTA a 128 x 128 fp32 slot
  unsigned* flags;           // per CTA: 1 while its slot holds a published part
  int M;
  int m_tiles;
  int units;                 // weight tiles x token tiles x superblocks
  unsigned* status;
};

__device__ __forceinline__ int range_start(int i, int units, int P) {
  const int q = units / P, r = units % P;
  return i * q + (i * r) / P;
}

template <int FMT>
__global__ void __launch_bounds__(kKqThreads, 1) kq_kernel(const KqParams p) {
  constexpr bool kQ6 = FMT == F_Q6_K;
  constexpr int kRec = (FMT == F_Q5_K) ? 176 : kQ6 ? 208 : 144;   // record bytes per row and superblock
  constexpr int kAPerStep = kQ6 ? 2 : 1;                    // decoded weight tiles per K step
  constexpr int kRecV = kRec / 16;
  extern __shared__ __align__(1024) uint8_t smem[];
  const Layout& L = p.L;
  uint64_t* x_full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* x_empty = x_full + kXSlots;
  uint64_t* a_full = x_empty + kXSlots;      // decoders -> MMA (4 warp arrivals)
  uint64_t* a_empty = a_full + kASlots;      // MMA commit -> decoders
  uint64_t* sx_full = a_empty + kASlots;     // sums tile landed (producer, tx)
  uint64_t* sd_full = sx_full + kSSlots;     // mins tile and row scales written (4 warp arrivals)
  uint64_t* s_empty = sd_full + kSSlots;     // MMA commit + 8 epilogue warps
  uint64_t* acc_full = s_empty + kSSlots;    // [2] MMA -> epilogue
  uint64_t* acc_free = acc_full + 2;         // [2] epilogue (8 warps) -> MMA
  uint64_t* done = acc_free + 2;
  volatile uint32_t* tslot = reinterpret_cast<volatile uint32_t*>(smem + 512);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + 516);
  volatile int* epi_abort = reinterpret_cast<volatile int*>(smem + 520);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int KB = (int)L.k_groups;
  const int KS = 4 * KB;
  const int P = (int)gridDim.x;
  const int c = (int)blockIdx.x;
  const int u0 = range_start(c, p.units, P), u1 = range_start(c + 1, p.units, P);
  const int n = u1 - u0;

  if (threadIdx.x == 0) {
    const PackedHeader* h = reinterpret_cast<const PackedHeader*>(p.packed);
    const bool bad = !(h->magic == kMagic && h->version == kVersion && h->fmt == (uint32_t)FMT &&
                       h->N == L.N && h->K == L.K && h->E == 1 && h->expert_bytes == L.expert_bytes);
    if (bad) atomicOr(p.status, kStatHeader);
    *abort_flag = bad ? 1 : 0;
    for (int i = 0; i < kXSlots; ++i) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&x_full[i])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&x_empty[i])));
    }
    for (int i = 0; i < kASlots; ++i) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(su32(&a_full[i])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&a_empty[i])));
    }
    for (int i = 0; i < kSSlots; ++i) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&sx_full[i])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 4;" ::"r"(su32(&sd_full[i])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 9;" ::"r"(su32(&s_empty[i])));
    }
    for (int i = 0; i < 2; ++i) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(&acc_full[i])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 8;" ::"r"(su32(&acc_free[i])));
    }
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(su32(done)));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;" ::"r"(su32((const void*)tslot)));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tslot;
  const bool bad_header = *abort_flag != 0;
  uint8_t* xring = smem + kXOff;
  uint8_t* aring = smem + kAOff;
  uint8_t* sring = smem + kSOff;

  if (warp == 0) {
    // ------------------------------ producer --------------------------------
    if (lane == 0 && !bad_header) {
      asm volatile("griddepcontrol.wait;" ::: "memory");      // the x tiles of the pre-pass
      int xs = 0, ss = 0, xi = 0;
      uint32_t xph = 0, sph = 0;
      int si = 0;
      for (int i = 0; i < n; ++i) {
        const int u = u0 + i, kb = u % KB, mt = (u / KB) % p.m_tiles;
        if (si >= kSSlots && !wait_bounded(&s_empty[ss], sph ^ 1u)) {
          atomicOr(p.status, kStatTimeout);
          *abort_flag = 1;
        }
        if (*abort_flag) break;
        expect_tx(&sx_full[ss], 4096u);
        bulk(sring + ss * kSBytes + kSumsOff, p.sums + ((int64_t)mt * KB + kb) * 4096, 4096u, &sx_full[ss]);
        ++si;
        if (++ss == kSSlots) { ss = 0; sph ^= 1u; }
        bool stop = false;
        for (int s = 0; s < 4; ++s) {
          if (xi >= kXSlots && !wait_bounded(&x_empty[xs], xph ^ 1u)) {
            atomicOr(p.status, kStatTimeout);
            *abort_flag = 1;
          }
          if (*abort_flag) { stop = true; break; }
          expect_tx(&x_full[xs], (uint32_t)kStepBytes);
          bulk(xring + xs * kStepBytes, p.xt + ((int64_t)mt * KS + 4 * kb + s) * kStepBytes, (uint32_t)kStepBytes,
               &x_full[xs]);
          ++xi;
          if (++xs == kXSlots) { xs = 0; xph ^= 1u; }
        }
        if (stop) break;
      }
      // copies still in flight land before the CTA can exit
      for (int j = (xi > kXSlots ? xi - kXSlots : 0); j < xi; ++j)
        (void)wait_bounded(&x_full[j % kXSlots], (uint32_t)((j / kXSlots) & 1));
      for (int j = (si > kSSlots ? si - kSSlots : 0); j < si; ++j)
        (void)wait_bounded(&sx_full[j % kSSlots], (uint32_t)((j / kSSlots) & 1));
    }
  } else if (warp == 1) {
    // ------------------------------ MMA issuer ------------------------------
    if (lane == 0) {
      // kind::f16: fp32 D (bit 4), f16 A and B, both K-major, N = 128 (bit 17), M = 128 (bit 24)
      const uint32_t idesc = (1u << 4) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
      int xs = 0, as = 0, ss = 0;
      uint32_t xph = 0, aph = 0, sph = 0;
      for (int i = 0; i < n && !bad_header; ++i) {
        const int b = i & 1;
        const uint32_t d1 = tmem + (uint32_t)(b * 256), d2 = d1 + 128u;
        bool ok = true;
        if (i >= 2) ok = wait_bounded(&acc_free[b], (uint32_t)((i / 2 - 1) & 1));
        for (int s = 0; s < 4 && ok; ++s) {
          ok = wait_bounded(&x_full[xs], xph);
          const uint32_t xa = su32(xring + xs * kStepBytes);
          for (int h = 0; h < kAPerStep && ok; ++h) {
            ok = wait_bounded(&a_full[as], aph);
            if (!ok || *abort_flag) break;
            asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
            const uint32_t aa = su32(aring + as * kStepBytes);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_f16(d1, sdesc(aa + 256 * k, 128, 1024), sdesc(xa + 256 * k, 128, 1024), idesc,
                      (s | k | h) ? 1u : 0u);
            commit(&a_empty[as]);
            if (++as == kASlots) { as = 0; aph ^= 1u; }
          }
          if (!ok || *abort_flag) break;
          commit(&x_empty[xs]);
          if (++xs == kXSlots) { xs = 0; xph ^= 1u; }
        }
        if (ok) ok = wait_bounded(&sx_full[ss], sph) && wait_bounded(&sd_full[ss], sph);
        if (!ok) {
          atomicOr(p.status, kStatTimeout);
          *abort_flag = 1;
        }
        if (*abort_flag) break;
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t sb = su32(sring + ss * kSBytes);
        if (!kQ6) mma_f16(d2, sdesc(sb + kMinsOff, 128, 256), sdesc(sb + kSumsOff, 128, 256), idesc, 0u);
        commit(&s_empty[ss]);
        commit(&acc_full[b]);
        if (++ss == kSSlots) { ss = 0; sph ^= 1u; }
      }
      commit(done);      // arrives when every MMA issued above has completed
    }
  } else if (warp < 6) {
    // ------------------------------ decoders --------------------------------
    const int r = threadIdx.x - 64;                         // weight row of the tile
    uint4 nxt[kRecV];
    uint32_t nxt_d = 0u;                                    // Q6_K: the row's fp16 d (plane B)
    auto load_rec = [&](int u) {
      const int kb = u % KB, nt = (u / KB) / p.m_tiles;
      const uint8_t* plane = p.packed + kHeaderBytes + (int64_t)kb * L.group_bytes;
      const uint8_t* rec = plane + ((int64_t)nt * 128 + r) * kRec;
#pragma unroll
      for (int v = 0; v < kRecV; ++v) nxt[v] = ldg_nc(rec + 16 * v);
      if constexpr (kQ6) nxt_d = __ldg(reinterpret_cast<const unsigned short*>(plane + L.plane_a) + (nt * 128 + r));
    };
    if (n > 0 && !bad_header) load_rec(u0);
    int as = 0, ss = 0, ai = 0;
    uint32_t aph = 0, sph = 0;
    for (int i = 0; i < n && !bad_header; ++i) {
      uint4 cur[kRecV];
#pragma unroll
      for (int v = 0; v < kRecV; ++v) cur[v] = nxt[v];
      const uint32_t cur_d = nxt_d;
      if (i + 1 < n) load_rec(u0 + i + 1);
      const uint32_t hw[4] = {cur[0].x, cur[0].y, cur[0].z, cur[0].w};
      const float d = kQ6 ? h2f(cur_d) : h2f(hw[0]), dmin = kQ6 ? 0.0f : h2f(hw[0] >> 16);
      // mins tile row r and the row scales
      if (i >= kSSlots && !warp_wait(&s_empty[ss], sph ^ 1u, lane)) {
        if (lane == 0) { atomicOr(p.status, kStatTimeout); *abort_flag = 1; }
        break;
      }
      if (__shfl_sync(0xffffffffu, *abort_flag, 0)) break;   // one decision per warp
      {
        uint8_t* sl = sring + ss * kSBytes;
        if constexpr (!kQ6) {
          uint32_t mh[4];
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const uint32_t m0 = q4k_field(hw[1], hw[2], hw[3], 8 + 2 * jj);
            const uint32_t m1 = q4k_field(hw[1], hw[2], hw[3], 9 + 2 * jj);
            asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(mh[jj]) : "f"((float)m1), "f"((float)m0));
          }
          const uint4 mv = make_uint4(mh[0], mh[1], mh[2], mh[3]);
          const int ro = (r >> 3) * 256 + (r & 7) * 16;
          *reinterpret_cast<uint4*>(sl + kMinsOff + ro) = mv;          // columns 0..7:  m_0..m_7
          *reinterpret_cast<uint4*>(sl + kMinsOff + ro + 128) = mv;    // columns 8..15: m_0..m_7
        }
        // the row scales: Q4_K / Q5_K (d 2^14, dmin); Q6_K (d, 0)
        *reinterpret_cast<float2*>(sl + kSclOff + 8 * r) = make_float2(kQ6 ? d : d * 16384.0f, dmin);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) arrive(&sd_full[ss]);
        if (++ss == kSSlots) { ss = 0; sph ^= 1u; }
      }
      bool stop = false;
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        if (ai >= kASlots && !warp_wait(&a_empty[as], aph ^ 1u, lane)) {
          if (lane == 0) { atomicOr(p.status, kStatTimeout); *abort_flag = 1; }
          stop = true;
          break;
        }
        if (__shfl_sync(0xffffffffu, *abort_flag, 0)) { stop = true; break; }
        if constexpr (kQ6) {
          // two tiles per K step, slots as and as2: (q - 32) 16 sh_u, then (q - 32) sl_u;
          // the second slot is waited for here too, so each pair of values is decoded once
          const int as2 = (as + 1 == kASlots) ? 0 : as + 1;
          const uint32_t aph2 = (as + 1 == kASlots) ? (aph ^ 1u) : aph;
          if (ai + 1 >= kASlots && !warp_wait(&a_empty[as2], aph2 ^ 1u, lane)) {
            if (lane == 0) { atomicOr(p.status, kStatTimeout); *abort_flag = 1; }
            stop = true;
            break;
          }
          if (__shfl_sync(0xffffffffu, *abort_flag, 0)) { stop = true; break; }
          uint8_t* at1 = aring + as * kStepBytes + (r >> 3) * 1024 + (r & 7) * 16;
          uint8_t* at2 = aring + as2 * kStepBytes + (r >> 3) * 1024 + (r & 7) * 16;
#pragma unroll
          for (int g = 0; g < 8; ++g) {
            uint32_t v[4];
            q6k_step_pairs(cur, s, g, v);
            const int u = 4 * s + (g >> 1);                        // 16-value unit of the superblock
            const int sc = (int)(int8_t)(rec_word(cur, 192 + (u & ~3)) >> (8 * (u & 3)));
            const uint32_t S1 = f16x2_dup((float)(16 * (sc >> 4))), S2 = f16x2_dup((float)(sc & 15));
            *reinterpret_cast<uint4*>(at1 + g * 128) =
                make_uint4(hmul2(v[0], S1), hmul2(v[1], S1), hmul2(v[2], S1), hmul2(v[3], S1));
            *reinterpret_cast<uint4*>(at2 + g * 128) =
                make_uint4(hmul2(v[0], S2), hmul2(v[1], S2), hmul2(v[2], S2), hmul2(v[3], S2));
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) { arrive(&a_full[as]); arrive(&a_full[as2]); }
          ai += 2;
          for (int h = 0; h < 2; ++h)
            if (++as == kASlots) { as = 0; aph ^= 1u; }
        } else {
          uint8_t* at = aring + as * kStepBytes + (r >> 3) * 1024 + (r & 7) * 16;
#pragma unroll
          for (int jj = 0; jj < 2; ++jj) {
            const int j = 2 * s + jj;                              // sub-block (32 values)
            const float sc = (float)q4k_field(hw[1], hw[2], hw[3], j);
            const uint32_t S = f16x2_dup(sc * 1024.0f), S16 = f16x2_dup(sc * 64.0f);
#pragma unroll
            for (int t = 0; t < 4; ++t)                             // word t: elements 8t..8t+7
              *reinterpret_cast<uint4*>(at + (4 * jj + t) * 128) = kq_decode_word<FMT>(cur, t, j, S, S16);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) arrive(&a_full[as]);
          ++ai;
          if (++as == kASlots) { as = 0; aph ^= 1u; }
        }
      }
      if (stop) break;
    }
  } else {
    // ------------------------------ epilogue --------------------------------
    const int q = warp & 3;                                  // lane quadrant: tile rows 32q .. 32q+31
    const int hf = (warp - 6) >> 2;                          // tokens 64 hf .. 64 hf + 63
    const bool leader = threadIdx.x == 192;
    const int row = 32 * q + lane;
    const uint32_t tq = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(64 * hf);
    float* slot = p.partials + (int64_t)c * kSlotWords;
    auto decide_abort = [&]() -> bool {
      epi_sync();
      if (leader) *epi_abort = *abort_flag;
      epi_sync();
      return *epi_abort != 0;
    };
    int ss = 0;
    uint32_t sph = 0;
    int i = 0;
    bool quit = bad_header;
    for (int pu0 = u0; pu0 < u1 && !quit;) {
      const int t = pu0 / KB;
      const int pu1 = ((t + 1) * KB < u1) ? (t + 1) * KB : u1;
      const bool head = (pu0 % KB) == 0;
      const bool whole = head && (pu1 - pu0 == KB);
      const int mt = t % p.m_tiles, nt = t / p.m_tiles;
      int npeer = 0;
      if (head && !whole)
        while (c + 1 + npeer < P && range_start(c + 1 + npeer, p.units, P) < (t + 1) * KB) ++npeer;
      float acc[64];
#pragma unroll
      for (int e = 0; e < 64; ++e) acc[e] = 0.f;
      for (int u = pu0; u < pu1; ++u, ++i) {
        const int b = i & 1;
        if (!wait_bounded(&acc_full[b], (uint32_t)((i / 2) & 1)) || !wait_bounded(&sd_full[ss], sph)) {
          atomicOr(p.status, kStatTimeout);
          *abort_flag = 1;
        }
        if (decide_abort()) { quit = true; break; }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const float2 sc = *reinterpret_cast<const float2*>(sring + ss * kSBytes + kSclOff + 8 * row);
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t r1[16], r2[16];
          tld16(r1, tq + (uint32_t)(b * 256 + 16 * cc));
          if constexpr (!kQ6) tld16(r2, tq + (uint32_t)(b * 256 + 128 + 16 * cc));
          tld_wait();
#pragma unroll
          for (int e = 0; e < 16; ++e) {
            if constexpr (kQ6)
              acc[16 * cc + e] = fmaf(sc.x, __uint_as_float(r1[e]), acc[16 * cc + e]);
            else
              acc[16 * cc + e] =
                  fmaf(sc.x, __uint_as_float(r1[e]), fmaf(-sc.y, __uint_as_float(r2[e]), acc[16 * cc + e]));
          }
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncwarp();
        if (lane == 0) { arrive(&acc_free[b]); arrive(&s_empty[ss]); }
        if (++ss == kSSlots) { ss = 0; sph ^= 1u; }
      }
      if (quit) break;
      float* srow = slot + row * 128 + 64 * hf;
      if (!head) {
        // publish this part; a later CTA finishes the tile
#pragma unroll
        for (int e = 0; e < 64; e += 4)
          *reinterpret_cast<float4*>(srow + e) = make_float4(acc[e], acc[e + 1], acc[e + 2], acc[e + 3]);
        __threadfence();
        epi_sync();
        if (leader) st_release(p.flags + c, 1u);
      } else {
        if (!whole) {
          if (leader) {
            for (int k = 0; k < npeer; ++k) {
              const unsigned* f = p.flags + c + 1 + k;
              bool got = ld_acquire(f) != 0u;
              const unsigned long long t0 = gtimer();
              while (!got && gtimer() - t0 <= kKqTimeoutNs) got = ld_acquire(f) != 0u;
              if (!got) { atomicOr(p.status, kStatTimeout); *abort_flag = 1; break; }
            }
          }
          if (decide_abort()) break;
          for (int k = 0; k < npeer; ++k) {
            const float* prow = p.partials + (int64_t)(c + 1 + k) * kSlotWords + row * 128 + 64 * hf;
#pragma unroll
            for (int e = 0; e < 64; e += 4) {
              const float4 v = __ldcg(reinterpret_cast<const float4*>(prow + e));
              acc[e] += v.x; acc[e + 1] += v.y; acc[e + 2] += v.z; acc[e + 3] += v.w;
            }
          }
          epi_sync();
          if (leader)
            for (int k = 0; k < npeer; ++k) st_relaxed(p.flags + c + 1 + k, 0u);
        }
        const int64_t nrow = (int64_t)nt * 128 + row;
        if (nrow < L.N) {
#pragma unroll
          for (int e = 0; e < 64; ++e) {
            const int64_t m = (int64_t)mt * 128 + 64 * hf + e;
            if (m < p.M) p.y[m * L.N + nrow] = acc[e];
          }
        }
      }
      pu0 = pu1;
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (warp == 1) {
    if (lane == 0) (void)wait_bounded(done, 0u);
    __syncwarp();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;" ::"r"(tmem));
  }
}

// ---------------------------------------------------------------------------
// pre-pass: x (bf16 [M][K]) -> f16 K-step tiles and sub-block-sum tiles
// ---------------------------------------------------------------------------
__global__ void kq_act_kernel(const uint16_t* __restrict__ x, uint8_t* __restrict__ xt, uint8_t* __restrict__ sums,
                              int64_t M, int64_t m_pad, int64_t K) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t nsub = K / 32;
  if (b >= m_pad * nsub) return;
  const int64_t m = b % m_pad, jg = b / m_pad;        // token, global sub-block
  const int64_t mt = m / 128;
  const int r = (int)(m % 128);
  const int64_t KS = K / 64, KB = K / 256;
  uint4 v[4] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u),
                make_uint4(0u, 0u, 0u, 0u)};
  if (m < M) {
    const uint4* src = reinterpret_cast<const uint4*>(x + m * K + 32 * jg);
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = __ldg(src + i);
  }
  float sum = 0.f;
  uint8_t* tile = xt + (mt * KS + jg / 2) * kStepBytes + (r >> 3) * 1024 + (r & 7) * 16;
  const int cm0 = 4 * (int)(jg & 1);                 // first core-matrix column of this sub-block
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t w[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
    uint32_t h[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float lo = __uint_as_float(w[k] << 16), hi = __uint_as_float(w[k] & 0xFFFF0000u);
      sum += lo;
      sum += hi;
      asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h[k]) : "f"(hi), "f"(lo));
    }
    *reinterpret_cast<uint4*>(tile + (cm0 + i) * 128) = make_uint4(h[0], h[1], h[2], h[3]);
  }
  const __half shi = __float2half_rn(sum);
  const __half slo = __float2half_rn(sum - __half2float(shi));
  const int kb = (int)(jg / 8), j = (int)(jg % 8);
  uint8_t* st = sums + (mt * KB + kb) * 4096 + (r >> 3) * 256 + (r & 7) * 16 + 2 * j;
  *reinterpret_cast<__half*>(st) = shi;             // column j
  *reinterpret_cast<__half*>(st + 128) = slo;       // column 8 + j
}

}  // namespace

int64_t kq_workspace_bytes(int64_t m_pad, int64_t K, int sms) {
  const int64_t xt = m_pad * K * 2;
  const int64_t sm = (m_pad / 128) * (K / 256) * 4096;
  return xt + sm + (int64_t)sms * kSlotWords * 4 + align_up((int64_t)sms * 4, 256);
}

cudaError_t launch_kq(const Layout& L, const uint8_t* packed, const uint16_t* x, float* y, int M, uint8_t* ws,
                      unsigned* status, cudaStream_t s) {
  int dev = 0, sms = 0, smem_max = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (err != cudaSuccess) return err;
  if (smem_max < kKqSmem) return cudaErrorInvalidConfiguration;
  const int64_t m_pad = align_up(M, 128);
  const int64_t m_tiles = m_pad / 128;
  const int64_t units = L.row_tiles * m_tiles * L.k_groups;
  if (units <= 0 || units * (int64_t)sms >= ((int64_t)1 << 31)) return cudaErrorInvalidValue;
  KqParams p;
  p.L = L;
  p.packed = packed;
  p.xt = ws;
  p.sums = ws + m_pad * L.K * 2;
  p.partials = reinterpret_cast<float*>(ws + m_pad * L.K * 2 + m_tiles * L.k_groups * 4096);
  p.flags = reinterpret_cast<unsigned*>(reinterpret_cast<uint8_t*>(p.partials) + (int64_t)sms * kSlotWords * 4);
  p.y = y;
  p.M = M;
  p.m_tiles = (int)m_tiles;
  p.units = (int)units;
  p.status = status;
  // the pre-pass: one thread per (token, 32-value sub-block), tokens fastest
  const int64_t total = m_pad * (L.K / 32);
  kq_act_kernel<<<(unsigned)((total + 255) / 256), 256, 0, s>>>(x, ws, const_cast<uint8_t*>(p.sums), M, m_pad, L.K);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  static int opted[64] = {0};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!opted[dev]) {
    err = cudaFuncSetAttribute(kq_kernel<F_Q4_K>, cudaFuncAttributeMaxDynamicSharedMemorySize, kKqSmem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(kq_kernel<F_Q5_K>, cudaFuncAttributeMaxDynamicSharedMemorySize, kKqSmem);
    if (err != cudaSuccess) return err;
    err = cudaFuncSetAttribute(kq_kernel<F_Q6_K>, cudaFuncAttributeMaxDynamicSharedMemorySize, kKqSmem);
    if (err != cudaSuccess) return err;
    opted[dev] = 1;
  }
  const int grid = (int)(units < sms ? units : sms);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kKqThreads);
  cfg.dynamicSmemBytes = (size_t)kKqSmem;
  cfg.stream = s;
  // At most one CTA per SM (its shared memory allows no more), so every CTA is
  // resident once the kernels before it have left: a finishing CTA's bounded wait on
  // its peers' partial tiles ends. The prologue overlaps the pre-pass.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = (L.fmt == F_Q5_K)   ? cudaLaunchKernelEx(&cfg, kq_kernel<F_Q5_K>, p)
        : (L.fmt == F_Q6_K) ? cudaLaunchKernelEx(&cfg, kq_kernel<F_Q6_K>, p)
                            : cudaLaunchKernelEx(&cfg, kq_kernel<F_Q4_K>, p);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

}  // namespace qmv
