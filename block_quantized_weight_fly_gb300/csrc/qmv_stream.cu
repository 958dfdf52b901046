// qmv_stream.cu -- the decode GEMV: y[M,N] = x[M,K] . W[N,K]^T with W packed
// (one matrix), and its grouped per-expert form over a stacked tower.
//
// Batch-1 decode is bound by weight delivery: the bytes read divided by the
// bandwidth set the ceiling ("Qwen3.8-27B on one Tenstorrent P150", section
// "Measuring the ceiling": removing arithmetic changed nothing, removing weight
// reads halved latency). So the kernel is built around streaming the packed
// weights from HBM exactly once per call for all M rows of x:
//
//  * persistent grid, one CTA per SM; the work is the list of slabs
//    (segment, 128-row tile, 256-value k-group) in tile-major order, cut into
//    equal contiguous ranges, one per CTA (split-K at slab granularity);
//  * warp 0 is a producer: one elected lane streams each slab (and the matching
//    256-value slice of every x row routed to it) into a ring of shared-memory
//    stages with cp.async.bulk, completion tracked by mbarriers; no multicast;
//  * warps 1..8 are consumers: warp w decodes 32-value chunk w of the slab for
//    its 128 rows (lane = row, four passes), the decode is in registers and the
//    inner product is factored per block: y += scale * sum(q * x) (- min * sum x);
//  * at the end of a row tile the warps' partial sums are added in shared
//    memory in a fixed order. A tile split between CTAs is finished by the CTA
//    that holds its first k-groups: the others publish their partial sums and a
//    flag, and it adds them in CTA order -- deterministic, no float atomics.
//
// Grouped form: the distinct routed experts are found on the device (sorted,
// each expert once, "A 320B MoE on a free Kaggle TPU", "The decode kernel's
// cost is not 'distinct experts'"); each becomes a segment whose slabs are
// streamed once and dotted with every x row routed to it.
//
// Every wait (mbarrier, peer flag) is bounded in time; on expiry the CTA latches
// QMV_ETIMEOUT in the device status word and stops.
#include <cuda_fp16.h>
#include "qmv_internal.h"

namespace qmv {

constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (1 + kConsumerWarps);
constexpr int kMaxStages = 16;
constexpr int kMaxSeg = 64;
constexpr unsigned long long kTimeoutNs = 1000000000ull;   // 1 s

struct Seg {
  int expert;
  int R;            // rows of x routed to this expert (<= 8)
  int xrow[8];
  int yrow[8];
};

// ---------------------------------------------------------------------------
// PTX helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(b)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t* b, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity)
      : "memory");
  return ok != 0;
}
// bounded wait on phase `parity`; false (and the status latched) on timeout
__device__ __forceinline__ bool mbar_wait(uint64_t* b, uint32_t parity, unsigned* status) {
  if (mbar_try_wait(b, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(b, parity)) return true;
    if ((it & 63u) == 0 && globaltimer() - t0 > kTimeoutNs) {
      atomicOr(status, kStatTimeout);
      return false;
    }
  }
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
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
__device__ __forceinline__ uint4 lds128(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// ---------------------------------------------------------------------------
// per-format chunk dot products: one row, one 32-value chunk, one x row.
// xf: the 32 x values (fp32, exact bf16). Returns the chunk's contribution.
// ---------------------------------------------------------------------------
template <int FMT>
struct ChunkDot;

template <>
struct ChunkDot<F_Q4_K> {
  // w = (d sc) q - dmin m  =>  contribution = (d sc) sum(q x) - (dmin m) sum(x)
  __device__ static float run(const uint8_t* rec, const uint8_t*, int row, int w, const float* xf,
                              float xsum) {
    (void)row;
    const uint4 hd = lds128(rec);
    const uint4 q = lds128(rec + q4k_q_off(w));
    const float d = h2f(hd.x), dmin = h2f(hd.x >> 16);
    const float a = d * (float)q4k_field(hd.y, hd.z, hd.w, w);
    const float b = dmin * (float)q4k_field(hd.y, hd.z, hd.w, 8 + w);
    const uint32_t qw[4] = {q.x, q.y, q.z, q.w};
    float s = 0.0f;
#pragma unroll
    for (int u = 0; u < 4; ++u)
#pragma unroll
      for (int v = 0; v < 8; ++v) s = fmaf((float)((qw[u] >> (4 * v)) & 15u), xf[8 * u + v], s);
    return fmaf(a, s, -b * xsum);
  }
};

template <>
struct ChunkDot<F_Q8_0> {
  __device__ static float run(const uint8_t* rec, const uint8_t*, int row, int w, const float* xf,
                              float) {
    (void)row;
    const float d = h2f(*reinterpret_cast<const unsigned short*>(rec + 2 * w));
    const uint4 q0 = lds128(rec + q80_q_off(w, 0));
    const uint4 q1 = lds128(rec + q80_q_off(w, 1));
    const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
    float s = 0.0f;
#pragma unroll
    for (int u = 0; u < 8; ++u)
#pragma unroll
      for (int v = 0; v < 4; ++v)
        s = fmaf((float)(int)(int8_t)((qw[u] >> (8 * v)) & 0xFFu), xf[4 * u + v], s);
    return d * s;
  }
};

template <>
struct ChunkDot<F_Q6_K> {
  // w = (d sc_j) (q - 32), sc_j per 16 values
  __device__ static float run(const uint8_t* rec, const uint8_t* dplane, int row, int w,
                              const float* xf, float) {
    const uint4 ql = lds128(rec + q6k_ql_off(w));
    const uint2 qh = *reinterpret_cast<const uint2*>(rec + q6k_qh_off(w));
    const int sc0 = (int)(int8_t)rec[192 + 2 * w], sc1 = (int)(int8_t)rec[192 + 2 * w + 1];
    const float d = h2f(*reinterpret_cast<const unsigned short*>(dplane + 2 * row));
    const uint32_t lw[4] = {ql.x, ql.y, ql.z, ql.w};
    const uint32_t hw[2] = {qh.x, qh.y};
    float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const int lo = (int)((lw[e >> 3] >> (4 * (e & 7))) & 15u);
      const int hi = (int)((hw[e >> 4] >> (2 * (e & 15))) & 3u);
      const float qv = (float)((lo | (hi << 4)) - 32);
      if (e < 16) s0 = fmaf(qv, xf[e], s0);
      else s1 = fmaf(qv, xf[e], s1);
    }
    return fmaf(d * (float)sc0, s0, (d * (float)sc1) * s1);
  }
};

template <>
struct ChunkDot<F_NVFP4> {
  // w = e2m1 * s_b (* s_T in the epilogue)
  __device__ static float run(const uint8_t* rec, const uint8_t*, int row, int w, const float* xf,
                              float) {
    (void)row;
    const uint4 c = lds128(rec + nv_q_off(w));
    const float sb0 = e4m3f(rec[2 * w]), sb1 = e4m3f(rec[2 * w + 1]);
    const uint32_t cw[4] = {c.x, c.y, c.z, c.w};
    float s0 = 0.0f, s1 = 0.0f;
#pragma unroll
    for (int e = 0; e < 32; ++e) {
      const float v = e2m1f((cw[e >> 3] >> (4 * (e & 7))) & 15u);
      if (e < 16) s0 = fmaf(v, xf[e], s0);
      else s1 = fmaf(v, xf[e], s1);
    }
    return fmaf(sb0, s0, sb1 * s1);
  }
};

template <>
struct ChunkDot<F_FP8> {
  // w = e4m3 (* s_row in the epilogue)
  __device__ static float run(const uint8_t* rec, const uint8_t*, int row, int w, const float* xf,
                              float) {
    const uint4 c0 = lds128(rec + fp8_v_off(2 * w, row & 7));
    const uint4 c1 = lds128(rec + fp8_v_off(2 * w + 1, row & 7));
    const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    float s = 0.0f;
#pragma unroll
    for (int e = 0; e < 32; ++e) s = fmaf(e4m3f((cw[e >> 2] >> (8 * (e & 3))) & 0xFFu), xf[e], s);
    return s;
  }
};

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
struct KParams {
  StreamArgs a;
  int stages;
  int stage_bytes;
  int x_off;         // offset of the x slices inside a stage
  int b_off;         // offset of plane B (Q6_K d) inside a stage
  int red_off;       // offset of the reduction buffer
  int stage_base;    // offset of stage 0
  int mt;            // partial stride (rows of x per partial record)
  unsigned* flags;   // [num_ctas]
  float* partials;   // [num_ctas][128][mt]
};

template <int FMT, int MT>
__global__ void __launch_bounds__(kThreads, 1) stream_kernel(const KParams kp) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const StreamArgs& a = kp.a;
  const Layout& L = a.L;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  uint64_t* red_full = empty + kMaxStages;
  uint64_t* red_free = red_full + 1;
  volatile int* misc = reinterpret_cast<volatile int*>(smem + 8 * (2 * kMaxStages + 2));
  Seg* segs = reinterpret_cast<Seg*>(smem + 512);
  float* red = reinterpret_cast<float*>(smem + kp.red_off);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;

  // ---- set-up: header check, segment table, barriers -----------------------
  if (tid == 0) {
    const PackedHeader* h = reinterpret_cast<const PackedHeader*>(a.packed);
    int bad = !(h->magic == kMagic && h->version == kVersion && h->fmt == (uint32_t)L.fmt &&
                h->N == L.N && h->K == L.K && h->E == L.E && h->expert_bytes == L.expert_bytes);
    if (bad) atomicOr(a.status, kStatHeader);
    misc[0] = bad;   // abort flag
    for (int i = 0; i < kp.stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    mbar_init(red_full, kConsumerWarps);
    mbar_init(red_free, kConsumerWarps);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (warp == 0) {
    if (a.ids == nullptr) {
      if (lane == 0) {
        misc[1] = 1;
        segs[0].expert = 0;
        segs[0].R = a.M;
        for (int r = 0; r < 8; ++r) { segs[0].xrow[r] = r; segs[0].yrow[r] = r; }
      }
    } else {
      // Distinct routed experts, ascending. Key = id * 64 + pair index (unique),
      // ranked by counting smaller keys; runs of equal ids become segments whose
      // pairs keep their (token, slot) order.
      const int P = a.M * a.topk;            // <= 64
      int* skeys = reinterpret_cast<int*>(smem + kp.red_off);      // scratch before first use
      int* sorted = skeys + 64;
      bool bad = false;
      for (int p = lane; p < P; p += 32) {
        const int id = a.ids[p];
        bad |= (id < 0 || (int64_t)id >= L.E);
        skeys[p] = (id << 6) | p;
      }
      if (__any_sync(0xffffffffu, bad)) {
        if (lane == 0) { atomicOr(a.status, kStatRange); misc[0] = 1; misc[1] = 0; }
      } else {
        __syncwarp();
        for (int p = lane; p < P; p += 32) {
          const int key = skeys[p];
          int rank = 0;
          for (int q = 0; q < P; ++q) rank += (skeys[q] < key);
          sorted[rank] = key;
        }
        __syncwarp();
        // first-of-run flags over the 64 sorted positions
        const int k0 = lane < P ? sorted[lane] : 0x7fffffff;
        const int k1 = lane + 32 < P ? sorted[lane + 32] : 0x7fffffff;
        const int pk0 = lane >= 1 && lane - 1 < P ? sorted[lane - 1] : -1;
        const int pk1 = lane + 31 < P ? sorted[lane + 31] : -1;
        const bool f0 = lane < P && (lane == 0 || (pk0 >> 6) != (k0 >> 6));
        const bool f1 = lane + 32 < P && ((pk1 >> 6) != (k1 >> 6));
        const unsigned long long fm = (unsigned long long)__ballot_sync(0xffffffffu, f0) |
                                      ((unsigned long long)__ballot_sync(0xffffffffu, f1) << 32);
        // a segment holds at most MT rows of x (ids repeated within a token can
        // exceed that): refuse such routing instead of overflowing
        bool over = false;
        for (int h = 0; h < 2; ++h) {
          const int i = lane + 32 * h;
          if (i >= P) continue;
          const unsigned long long upto = fm & ((i == 63) ? ~0ull : ((2ull << i) - 1));
          over |= (i - (63 - __clzll((long long)upto))) >= MT;
        }
        if (__any_sync(0xffffffffu, over)) {
          if (lane == 0) { atomicOr(a.status, kStatRange); misc[0] = 1; misc[1] = 0; }
        } else {
          for (int h = 0; h < 2; ++h) {
            const int i = lane + 32 * h;
            if (i >= P) continue;
            const int key = h ? k1 : k0;
            const unsigned long long upto = fm & ((i == 63) ? ~0ull : ((2ull << i) - 1));
            const int start = 63 - __clzll((long long)upto);
            const int seg = __popcll(upto) - 1;
            const unsigned long long above = (start == 63) ? 0ull : (fm >> (start + 1)) << (start + 1);
            const int next = above ? __ffsll((long long)above) - 1 : P;
            const int pair = key & 63, slot = i - start;
            Seg& sg = segs[seg];
            if (i == start) { sg.expert = key >> 6; sg.R = next - start; }
            sg.xrow[slot] = a.x_per_pair ? pair : pair / a.topk;
            sg.yrow[slot] = pair;
          }
          if (lane == 0) misc[1] = __popcll(fm);
        }
      }
    }
  }
  __syncthreads();
  if (misc[0]) return;

  const int64_t nseg = misc[1];
  const int64_t G = L.k_groups;
  const int64_t tiles = nseg * L.row_tiles;
  const int64_t S = tiles * G;
  const int64_t P = gridDim.x;
  const int64_t c = blockIdx.x;
  const int64_t s0 = (c * S) / P, s1 = ((c + 1) * S) / P;
  if (s0 >= s1) return;

  if (warp == 0) {
    // ---------------------------- producer --------------------------------
    if (lane != 0) return;
    int64_t it = 0;
    for (int64_t s = s0; s < s1; ++s, ++it) {
      const int stage = (int)(it % kp.stages);
      if (it >= kp.stages) {
        const uint32_t par = (uint32_t)(((it / kp.stages) - 1) & 1);
        if (!mbar_wait(&empty[stage], par, a.status)) { misc[0] = 1; break; }
      }
      if (misc[0]) break;
      const int64_t T = s / G, g = s % G;
      const Seg& sg = segs[T / L.row_tiles];
      const int64_t t = T % L.row_tiles;
      uint8_t* st = smem + kp.stage_base + (int64_t)stage * kp.stage_bytes;
      const uint8_t* plane = a.packed + kHeaderBytes + sg.expert * L.expert_bytes + g * L.group_bytes;
      const uint32_t abytes = (uint32_t)(kSlabRows * L.rec);
      const uint32_t bbytes = (FMT == F_Q6_K) ? (uint32_t)(kSlabRows * 2) : 0u;
      const int64_t kv = (L.K - g * kSlabK) < kSlabK ? (L.K - g * kSlabK) : kSlabK;
      const uint32_t xbytes = (uint32_t)(kv * 2);
      const int R = sg.R < MT ? sg.R : MT;
      mbar_expect_tx(&full[stage], abytes + bbytes + xbytes * (uint32_t)R);
      bulk_g2s(st, plane + t * kSlabRows * L.rec, abytes, &full[stage]);
      if (FMT == F_Q6_K) bulk_g2s(st + kp.b_off, plane + L.plane_a + t * kSlabRows * 2, bbytes, &full[stage]);
      for (int r = 0; r < R; ++r)
        bulk_g2s(st + kp.x_off + r * (kSlabK * 2), a.x + (int64_t)sg.xrow[r] * L.K + g * kSlabK, xbytes,
                 &full[stage]);
    }
    // drain: copies issued into stages the consumers may not have waited for
    if (misc[0]) {
      const int64_t issued = it;
      for (int64_t j = (issued > kp.stages ? issued - kp.stages : 0); j < issued; ++j)
        (void)mbar_wait(&full[j % kp.stages], (uint32_t)((j / kp.stages) & 1), a.status);
    }
    return;
  }

  // ------------------------------ consumers ---------------------------------
  const int w = warp - 1;               // chunk index of this warp
  const int ctid = tid - 32;            // 0..255
  float acc[4][MT];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int r = 0; r < MT; ++r) acc[i][r] = 0.0f;
  int64_t it = 0;
  int flushes = 0;
  for (int64_t s = s0; s < s1; ++s, ++it) {
    if (misc[0]) break;
    const int stage = (int)(it % kp.stages);
    const int64_t T = s / G, g = s % G;
    const Seg& sg = segs[T / L.row_tiles];
    if (!mbar_wait(&full[stage], (uint32_t)((it / kp.stages) & 1), a.status)) { misc[0] = 1; break; }
    const uint8_t* st = smem + kp.stage_base + (int64_t)stage * kp.stage_bytes;
    const int64_t k0 = g * kSlabK + (int64_t)w * kChunk;
    if (k0 < L.K) {
      for (int r = 0; r < sg.R && r < MT; ++r) {
        float xf[32];
        const uint8_t* xs = st + kp.x_off + r * (kSlabK * 2) + w * 64;
        float xsum = 0.0f;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const uint4 v = lds128(xs + 16 * h);
          const uint32_t vw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            xf[8 * h + 2 * u] = bf2f(vw[u]);
            xf[8 * h + 2 * u + 1] = bf2f(vw[u] >> 16);
          }
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) xsum += xf[e];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int row = lane + 32 * i;
          const float v = ChunkDot<FMT>::run(st + row * L.rec, st + kp.b_off, row, w, xf, xsum);
#pragma unroll
          for (int rr = 0; rr < MT; ++rr)
            if (rr == r) acc[i][rr] += v;
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[stage]);

    const bool tile_end = (s + 1 == s1) || ((s + 1) / G != T);
    if (!tile_end) continue;

    // ---- flush tile T ------------------------------------------------------
    const int64_t head = T * G, tail = (T + 1) * G;
    const bool full_cover = (s0 <= head) && (s1 >= tail);
    const bool reducer = (s0 <= head);
    const int R = sg.R < MT ? sg.R : MT;
    if (flushes > 0) {
      if (!mbar_wait(red_free, (uint32_t)((flushes - 1) & 1), a.status)) { misc[0] = 1; break; }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int r = 0; r < MT; ++r) red[(w * kSlabRows + lane + 32 * i) * MT + r] = acc[i][r];
    __syncwarp();
    if (lane == 0) mbar_arrive(red_full);
    if (!mbar_wait(red_full, (uint32_t)(flushes & 1), a.status)) { misc[0] = 1; break; }

    const int64_t t = T % L.row_tiles;
    const uint8_t* extras = a.packed + kHeaderBytes + sg.expert * L.expert_bytes + L.k_groups * L.group_bytes;
    // pairs handled by this thread: p = ctid + 256 j, p < 128 * R
    float vals[(kSlabRows * MT + 255) / 256];
    int np = 0;
    for (int p = ctid; p < kSlabRows * R; p += 256, ++np) {
      const int row = p / R, r = p % R;
      float v = 0.0f;
#pragma unroll
      for (int ww = 0; ww < kConsumerWarps; ++ww) v += red[(ww * kSlabRows + row) * MT + r];
      vals[np] = v;
    }
    bool ok = true;
    if (!full_cover && !reducer) {
      // publish this CTA's partial sums of its first tile
      float* part = kp.partials + c * (kSlabRows * kp.mt);
      np = 0;
      for (int p = ctid; p < kSlabRows * R; p += 256, ++np) {
        const int row = p / R, r = p % R;
        part[row * kp.mt + r] = vals[np];
      }
      __threadfence();
    } else if (!full_cover && reducer) {
      // add the peers' partial sums in CTA order
      for (int64_t cp = c + 1; cp < P; ++cp) {
        const int64_t ps0 = (cp * S) / P, ps1 = ((cp + 1) * S) / P;
        if (ps0 >= tail) break;
        if (ps0 >= ps1) continue;           // an empty range publishes nothing
        const unsigned* flag = kp.flags + cp;
        if (ld_acquire(flag) == 0u) {
          const unsigned long long t0 = globaltimer();
          while (ld_acquire(flag) == 0u) {
            if (globaltimer() - t0 > kTimeoutNs) { atomicOr(a.status, kStatTimeout); ok = false; break; }
          }
        }
        if (!ok) break;
        const float* part = kp.partials + cp * (kSlabRows * kp.mt);
        np = 0;
        for (int p = ctid; p < kSlabRows * R; p += 256, ++np) {
          const int row = p / R, r = p % R;
          vals[np] += __ldcg(part + row * kp.mt + r);
        }
      }
    }
    if (ok && (full_cover || reducer)) {
      np = 0;
      for (int p = ctid; p < kSlabRows * R; p += 256, ++np) {
        const int row = p / R, r = p % R;
        const int64_t n = t * kSlabRows + row;
        if (n >= L.N) continue;
        float v = vals[np];
        if (FMT == F_NVFP4) v *= *reinterpret_cast<const float*>(extras);
        if (FMT == F_FP8) v *= reinterpret_cast<const float*>(extras)[n];
        a.y[(int64_t)sg.yrow[r] * L.N + n] = v;
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(red_free);
    if (!ok) { misc[0] = 1; break; }
    if (!full_cover) {
      if (!reducer) {
        if (ctid == 0) {
          if (!mbar_wait(red_free, (uint32_t)(flushes & 1), a.status)) misc[0] = 1;
          else st_release(kp.flags + c, 1u);
        }
      } else if (ctid == 0) {
        // every consumer thread has read the peers' flags and sums: reset the flags
        if (!mbar_wait(red_free, (uint32_t)(flushes & 1), a.status)) misc[0] = 1;
        else {
          for (int64_t cp = c + 1; cp < P; ++cp) {
            const int64_t ps0 = (cp * S) / P, ps1 = ((cp + 1) * S) / P;
            if (ps0 >= tail) break;
            if (ps0 < ps1) kp.flags[cp] = 0u;
          }
        }
      }
    }
    ++flushes;
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int r = 0; r < MT; ++r) acc[i][r] = 0.0f;
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
WsPlan ws_plan_stream(int M, int64_t tiles_max, int num_ctas) {
  (void)tiles_max;
  WsPlan p;
  const int mt = (M <= 1) ? 1 : 8;
  p.counters_off = 256;
  p.counters_bytes = align_up((int64_t)num_ctas * 4, 256);
  p.partials_off = p.counters_off + p.counters_bytes;
  p.partials_bytes = align_up((int64_t)num_ctas * kSlabRows * mt * 4, 256);
  p.total = p.partials_off + p.partials_bytes;
  return p;
}

int num_sms_current_device() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

template <int FMT, int MT>
static cudaError_t launch_t(const StreamArgs& a, cudaStream_t s) {
  int dev = 0, smem_max = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (err != cudaSuccess) return err;
  KParams kp;
  kp.a = a;
  kp.mt = MT;
  kp.red_off = 512 + kMaxSeg * (int)sizeof(Seg);
  const int red_bytes = kConsumerWarps * kSlabRows * MT * 4;
  kp.stage_base = (int)align_up(kp.red_off + red_bytes, 1024);
  const int abytes = kSlabRows * a.L.rec;
  kp.b_off = (int)align_up(abytes, 128);
  const int bbytes = (FMT == F_Q6_K) ? kSlabRows * 2 : 0;
  kp.x_off = (int)align_up(kp.b_off + bbytes, 128);
  kp.stage_bytes = (int)align_up(kp.x_off + MT * kSlabK * 2, 1024);
  kp.stages = (smem_max - kp.stage_base) / kp.stage_bytes;
  if (kp.stages > kMaxStages) kp.stages = kMaxStages;
  if (kp.stages < 2) return cudaErrorInvalidConfiguration;
  const WsPlan plan = ws_plan_stream(MT, 0, a.num_ctas);
  kp.flags = reinterpret_cast<unsigned*>(a.ws + plan.counters_off);
  kp.partials = reinterpret_cast<float*>(a.ws + plan.partials_off);
  const int smem = kp.stage_base + kp.stages * kp.stage_bytes;
  err = cudaFuncSetAttribute(stream_kernel<FMT, MT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.num_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;   // peers wait on each other's flags
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, stream_kernel<FMT, MT>, kp);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

template <int FMT>
static cudaError_t launch_fmt(const StreamArgs& a, cudaStream_t s, int* variant) {
  const bool grouped = a.ids != nullptr;
  *variant = grouped ? 3 : (a.M <= 1 ? 1 : 2);
  if (a.M <= 1) return launch_t<FMT, 1>(a, s);   // grouped at M = 1: one x row per expert
  return launch_t<FMT, 8>(a, s);
}

cudaError_t launch_stream(const StreamArgs& a, cudaStream_t s, int* variant) {
  switch (a.L.fmt) {
    case F_Q8_0: return launch_fmt<F_Q8_0>(a, s, variant);
    case F_Q4_K: return launch_fmt<F_Q4_K>(a, s, variant);
    case F_Q6_K: return launch_fmt<F_Q6_K>(a, s, variant);
    case F_NVFP4: return launch_fmt<F_NVFP4>(a, s, variant);
    case F_FP8: return launch_fmt<F_FP8>(a, s, variant);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qmv
