// qmv_stream.cu -- the decode GEMV: y[M,N] = x[M,K] . W[N,K]^T with W packed
// (one matrix), and its grouped per-expert form over a stacked tower.
//
// Batch-1 decode is bound by weight delivery: the bytes read divided by the
// bandwidth set the ceiling ("Qwen3.8-27B on one Tenstorrent P150", section
// "Measuring the ceiling": removing arithmetic changed nothing, removing weight
// reads halved latency). So the kernel is built around streaming the packed
// weights from HBM exactly once per call for all M rows of x:
//
//  * persistent grid of one or two CTAs per SM (chosen per call by the entry
//    point); the work is the list of slabs (segment, 128-row tile, 256-value
//    k-group) in tile-major order, cut into equal contiguous ranges, one per CTA
//    (split-K at slab granularity);
//  * warp 0 is a producer: one elected lane streams each slab (and the matching
//    256-value slice of every x row routed to it) into a ring of shared-memory
//    stages with cp.async.bulk, completion tracked by mbarriers; no multicast;
//  * the other eight warps are consumers: warp w decodes rows 16w .. 16w+15 of a
//    slab on mma.sync (see qmv_slab.cuh), the decode in registers and the inner
//    product factored per block: y += scale * sum(q * x) (- min * sum x);
//  * a CTA takes half an SM: with a grid of one CTA per SM the next call's CTAs
//    are resident beside the running ones and copy their first weight slabs
//    meanwhile; with two per SM the call's own warps hide each other's latency;
//  * a row tile split between CTAs is finished by the CTA that holds its first
//    k-groups: the others publish their partial sums in the workspace, each word
//    non-zero so that it is its own completion flag (no fence, no flag word), and
//    the finishing CTA adds them in CTA order -- deterministic, no float atomics --
//    and clears them for the next call.
//
// Grouped form: the distinct routed experts are found on the device (sorted,
// each expert once, "A 320B MoE on a free Kaggle TPU", "The decode kernel's
// cost is not 'distinct experts'"); each becomes a segment whose slabs are
// streamed once and dotted with every x row routed to it.
//
// Every wait (mbarrier, peer partial sum) is bounded in time; on expiry the CTA latches
// QMV_ETIMEOUT in the device status word and stops.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include "qmv_internal.h"
#include "qmv_slab.cuh"

namespace qmv {

constexpr int kConsumerWarps = 8;       // consumer warps (16 rows of a slab each)
constexpr int kThreads = 32 * (1 + kConsumerWarps);
// CTAs resident per SM: a CTA takes half of the SM (shared memory and registers),
// so that the next call's CTA is resident beside the running one and runs its
// prologue and first weight copies during the running call's compute.
template <int MT> constexpr int ctas_per_sm() { return 2; }
constexpr int kMaxStages = 16;
// bytes of plane B per 128-row tile (Q6_K d, NVFP4 block scales, IQ4_XS scale fields
// and codebook)
template <int FMT> constexpr int plane_b_tile() {
  return FMT == F_Q6_K ? kSlabRows * 2 : FMT == F_NVFP4 ? kSlabRows * 16 : FMT == F_IQ4_XS ? kIq4TileB
       : FMT == F_IQ3_S ? kSlabRows * 14 : FMT == F_IQ2_S ? kSlabRows * 18 : 0;
}
// the grid formats' f16 grid, copied into shared memory once per CTA
template <int FMT> constexpr int grid_smem_bytes() { return FMT == F_IQ3_S ? 512 * 4 * 2 : FMT == F_IQ2_S ? 1024 * 8 * 2 : 0; }
// the mbarrier of that copy (a spare slot after the stage barriers)
constexpr int kGridBarOff = 256;
constexpr int kMaxSeg = 64;
// the reducer's gather list (built by the producer warp): kMaxGather entries in the
// misc area of shared memory, then the mbarrier that publishes them
// (after misc[0..11], the control words of the misc area at byte 272)
constexpr int kGatherOff = 320;
constexpr int kMaxGather = 36;
constexpr int kGbarOff = 472;
static_assert(kGatherOff + 4 * kMaxGather <= kGbarOff && kGbarOff + 8 <= 512, "misc area");
constexpr unsigned long long kTimeoutNs = 1000000000ull;   // 1 s
constexpr uint32_t kSuspendNs = 2000;    // a waiting thread sleeps up to this long per try (wakes on completion)

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
__device__ __forceinline__ void mbar_inval(uint64_t* b) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(b)) : "memory");
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
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(b)), "r"(parity), "r"(kSuspendNs)
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
// 16-byte global -> shared copy; completion is tracked per thread (cp_async_arrive_noinc)
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
// the barrier counts one arrival of this thread once all its earlier cp.async have landed
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* b) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(b)) : "memory");
}
__device__ __forceinline__ uint32_t ld_relaxed(const unsigned* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_relaxed(unsigned* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
// A piece as stored in the workspace: never zero, so that each word is its own
// completion flag. +0.0 is stored as the NaN pattern 0x7FFFFFFF (no finite sum
// produces it) and decoded back; every other value is stored as it is.
constexpr uint32_t kZeroCode = 0x7FFFFFFFu;
__device__ __forceinline__ uint32_t encode_piece(float v) {
  const uint32_t u = __float_as_uint(v);
  return u == 0u ? kZeroCode : u;
}
__device__ __forceinline__ float decode_piece(uint32_t u) { return u == kZeroCode ? 0.0f : __uint_as_float(u); }
__device__ __forceinline__ uint4 lds128(const void* p) {
  return *reinterpret_cast<const uint4*>(p);
}

// ---------------------------------------------------------------------------
// the kernel
// ---------------------------------------------------------------------------
struct KParams {
  StreamArgs a;
  int stages;
  int stage_bytes;
  int x_off;         // offset of the x slices inside a stage
  int b_off;         // offset of plane B (Q6_K d) inside a stage
  int tbl_off;       // offset of the per-warp scale tables
  int grid_off;      // offset of the grid formats' f16 grid
  int stage_base;    // offset of stage 0
  int mt;            // partial stride (token columns per partial record)
  int cells;         // dense: the number of cells V (> 0); grouped: 0 (cells of gp slabs per unit)
  int cpc;           // dense: cells per CTA (the plans use 1; the kernel also takes 2)
  int gp;            // grouped: slabs (k-groups) per cell: 1, 2 or 4
  int maxslots;      // published pieces a CTA may hold (slots per CTA in the workspace)
  int fault;         // test hook: 1 = peers publish nothing (reducers' bounded waits run
                     // out); 2 = reducers abandon their gathers at once (pieces left behind)
  unsigned long long peer_wait_ns;   // bound of a reducer's wait for a peer's piece
  float* partials;   // [num_ctas][maxslots][128][mt]
};

// The cell partition of one call's slab sequence (S slabs in units of UL slabs; see
// the kernel). Dense calls: kp.cells = V cells of floor(i S / V) slabs, kp.cpc per
// CTA. Grouped calls: each unit is cut into CU = ceil(UL / gp) cells of gp slabs, and
// CTA c holds cells [floor(c C / P), floor((c+1) C / P)) of the C cells. 32-bit
// arithmetic: i * Sr < V * V and c * Cr < P * P.
struct CellMap {
  bool grouped;
  int V, cpc, Sq, Sr;        // dense
  int CU, UL, gp, P, Cq, Cr; // grouped
  __device__ __forceinline__ int cell_start(int i) const {
    if (grouped) {
      const int k = (i % CU) * gp;
      return (i / CU) * UL + (k < UL ? k : UL);
    }
    return i * Sq + (i * Sr) / V;
  }
  __device__ __forceinline__ int first_cell(int c) const {
    if (grouped) return c * Cq + (c * Cr) / P;
    const int k = c * cpc;
    return k < V ? k : V;
  }
  __device__ __forceinline__ int cta_start(int c) const { return cell_start(first_cell(c)); }
  // the cell of slab p (grouped)
  __device__ __forceinline__ int cell_of(int p) const { return (p / UL) * CU + (p % UL) / gp; }
  // dense: the start of a two-cell CTA's second cell (else the range end)
  __device__ __forceinline__ int cta_mid(int c) const {
    if (grouped || cpc != 2) return cta_start(c + 1);
    const int k = 2 * c + 1;
    return cell_start(k < V ? k : V);
  }
};
__device__ __forceinline__ CellMap cell_map(int cells, int cpc, int gp, int S, int UL, int P) {
  CellMap m;
  m.grouped = cells <= 0;
  m.V = cells > 0 ? cells : 1;
  m.cpc = cells > 0 ? cpc : 1;
  m.Sq = S / m.V;
  m.Sr = S % m.V;
  m.UL = UL;
  m.gp = gp > 0 ? gp : 1;
  m.CU = (UL + m.gp - 1) / m.gp;
  m.P = P;
  const int C = (S / UL) * m.CU;
  m.Cq = C / P;
  m.Cr = C % P;
  return m;
}

// The next piece of unit [head, tail) from slab *p on, held by CTA *cp or a later one
// (*cp is advanced to it): returns the piece's workspace word index (a multiple of
// 128) with its pass in bit 0, and moves *p to the piece's end.
__device__ __forceinline__ int next_piece(const CellMap cm, int head, int tail, int G, int UG, int maxslots,
                                       int pstride, int* p, int* cp) {
  const int q = *p;
  int c = *cp;
  while (cm.cta_start(c + 1) <= q) ++c;               // the CTA holding slab q
  const int ps = (UG == 2 && q - head >= G) ? 1 : 0;
  int pe, slot;
  if (!cm.grouped) {
    const int m = cm.cta_mid(c);
    const int kc = (q >= m) ? 1 : 0;                  // its first or second cell
    pe = kc ? cm.cta_start(c + 1) : m;
    slot = kc * UG + ps;
  } else {
    const int ci = cm.cell_of(q);
    pe = cm.cell_start(ci + 1);
    slot = (ci - cm.first_cell(c)) * UG + ps;
  }
  if (pe > tail) pe = tail;
  if (UG == 2 && ps == 0 && head + G < pe) pe = head + G;
  *p = pe;
  *cp = c;
  return (c * maxslots + slot) * pstride + ps;
}

// ---------------------------------------------------------------------------
// Cold paths, out of line: their code stays away from the decode loop, whose
// instruction footprint must stay small (one copy each; their calls are rare).
// ---------------------------------------------------------------------------
// Set-up (one thread): the CTA's slab range in the cells of the call, into
// misc[6] = start, misc[7] = end, misc[8] = the start of a two-cell CTA's second cell
// (dense calls; else the end).
__device__ __noinline__ void cta_range(volatile int* misc, int cells, int cpc, int gp, int S, int UL, int P,
                                       int c) {
  const CellMap cm = cell_map(cells, cpc, gp, S, UL, P);
  misc[6] = cm.cta_start(c);
  misc[7] = cm.cta_start(c + 1);
  misc[8] = cm.cta_mid(c);
}

// The producer's gather list, built by the whole producer warp: the pieces of the
// CTA's last unit that later CTAs hold, when this CTA holds the unit's first slab, in
// slab order. Lane l takes the l-th cell after the CTA's range (a piece, or two when
// the cell holds both passes of a fused unit); a warp prefix sum places the entries.
// At most kMaxGather entries in glist, their count in misc[2]; when more pieces
// follow, misc[5] = 1 and misc[3], misc[4] = where they start (slab, a CTA at or
// before its holder).
__device__ __noinline__ void build_gather_list(volatile int* misc, volatile int* glist, int cells, int cpc, int gp,
                                               int S, int UL, int G, int UG, int P, int c, int maxslots,
                                               int pstride, int lane) {
  const int s0 = misc[6], s1 = misc[7];
  const int head = ((s1 - 1) / UL) * UL, tail = head + UL;
  int n = 0, more = 0, rest = tail;
  if (head >= s0 && tail > s1) {
    const CellMap cm = cell_map(cells, cpc, gp, S, UL, P);
    const int ncells = cm.grouped ? (S / UL) * cm.CU : cm.V;
    const int base = cm.first_cell(c + 1);
    for (int round = 0;; ++round) {
      const int i = base + 32 * round + lane;
      int cnt = 0, e0 = -1, e1 = -1, cs = tail;
      if (i < ncells) cs = cm.cell_start(i);
      if (cs < tail) {
        int ce = cm.cell_start(i + 1);
        if (ce > tail) ce = tail;
        // the CTA holding cell i
        int cp;
        if (!cm.grouped) {
          cp = i / cm.cpc;
        } else {
          cp = (int)(((int64_t)i * P) / ((int64_t)(S / UL) * cm.CU));
          while (cp + 1 <= P && cm.first_cell(cp + 1) <= i) ++cp;
          while (cp > 0 && cm.first_cell(cp) > i) --cp;
        }
        const int ord = i - cm.first_cell(cp);
        const int ps0 = (UG == 2 && cs - head >= G) ? 1 : 0;
        e0 = (cp * maxslots + ord * UG + ps0) * pstride + ps0;
        cnt = 1;
        if (UG == 2 && ps0 == 0 && head + G < ce) {       // the cell also holds up slabs
          e1 = (cp * maxslots + ord * UG + 1) * pstride + 1;
          cnt = 2;
        }
      }
      // exclusive prefix of cnt over the lanes
      int pre = cnt;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, pre, d);
        if (lane >= d) pre += v;
      }
      const int total = __shfl_sync(0xffffffffu, pre, 31);
      pre -= cnt;
      if (n + total > kMaxGather) {                    // the rest: computed by the reducer
        more = 1;
        rest = __shfl_sync(0xffffffffu, cs, 0);        // the first cell of this round
        break;
      }
      if (cnt > 0) glist[n + pre] = e0;
      if (cnt > 1) glist[n + pre + 1] = e1;
      n += total;
      const bool done = __any_sync(0xffffffffu, i >= ncells || cs >= tail);
      if (done) break;
    }
    if (lane == 0 && more) {
      misc[3] = rest;
      misc[4] = c + 1;
    }
  }
  if (lane == 0) {
    misc[2] = n;
    misc[5] = more;
  }
  __syncwarp();
}

// The reducer's gather past the end of the producer's list (rare: a unit cut into
// more pieces than the list holds): the remaining pieces of unit [head, tail), computed
// here in slab order, KB at a time so that their load latencies overlap, added into
// uacc[pass][e] (e: this thread's outputs, rows rA/rB x tokens 2tq, 2tq+1; at M = 1
// e = 0, 2 only). Each word is cleared after it is read. Returns false when a bounded
// wait ran out (the status is latched).
struct GatherArgs {
  volatile int* misc;
  const volatile int* glist;
  unsigned* parts;
  unsigned* status;
  unsigned long long wait_ns;
  int cells, cpc, gp, S, UL, G, P, maxslots, pstride, mt, R, tq, rA, rB, head, tail;
};
template <int MT, bool SW>
__device__ __noinline__ bool gather_unit(const GatherArgs ga, float* uacc /* [UG][4] */) {
  constexpr int UG = SW ? 2 : 1;
  constexpr int KB = (MT == 1 ? 8 : 4) / (SW ? 2 : 1);
  constexpr int NE = MT == 1 ? 2 : 4;                  // outputs e of this thread (M = 1: e = 0, 2)
  // (called only when the producer's list did not hold every piece: the list has
  // been gathered inline; this continues from where it stopped)
  const int n = 0;
  const bool more = true;
  int i = 0, p = ga.misc[3], cp = ga.misc[4];
  for (;;) {
    int pc[KB];
#pragma unroll
    for (int k = 0; k < KB; ++k) {
      pc[k] = -1;
      if (i < n) {
        pc[k] = ga.glist[i++];
      } else if (more && p < ga.tail) {
        pc[k] = next_piece(cell_map(ga.cells, ga.cpc, ga.gp, ga.S, ga.UL, ga.P), ga.head, ga.tail, ga.G, UG,
                           ga.maxslots, ga.pstride, &p, &cp);
      }
    }
    if (pc[0] < 0) return true;
    uint32_t u[KB][NE];
#pragma unroll
    for (int k = 0; k < KB; ++k) {
#pragma unroll
      for (int j = 0; j < NE; ++j) {
        const int e = MT == 1 ? 2 * j : j;
        const int tok = 2 * ga.tq + (e & 1), row = (e < 2) ? ga.rA : ga.rB;
        u[k][j] = 0u;
        if (pc[k] >= 0 && tok < ga.R) u[k][j] = ld_relaxed(ga.parts + (pc[k] & ~1) + row * ga.mt + tok);
      }
    }
#pragma unroll
    for (int k = 0; k < KB; ++k) {
#pragma unroll
      for (int j = 0; j < NE; ++j) {
        const int e = MT == 1 ? 2 * j : j;
        const int tok = 2 * ga.tq + (e & 1), row = (e < 2) ? ga.rA : ga.rB;
        if (pc[k] < 0 || tok >= ga.R) continue;
        unsigned* wp = ga.parts + (pc[k] & ~1) + row * ga.mt + tok;
        uint32_t v = u[k][j];
        if (v == 0u) {
          const unsigned long long t0 = globaltimer();
          while ((v = ld_relaxed(wp)) == 0u) {
            if (globaltimer() - t0 > ga.wait_ns) break;
          }
          if (v == 0u) {
            atomicOr(ga.status, kStatTimeout);
            ga.misc[0] = 1;
            return false;
          }
        }
        st_relaxed(wp, 0u);
        float* dst = uacc + ((SW && (pc[k] & 1)) ? 4 * (UG - 1) : 0) + e;
        *dst = __fadd_rn(*dst, decode_piece(v));
      }
    }
  }
}

// SW: fused gate|up with the SwiGLU epilogue. The tower holds 2E experts: the E
// gate matrices, then the E up matrices (E = 1 for the dense call). Each segment is
// one (routed) expert e; a row tile's gate k-groups (expert e) and then the same
// rows' up k-groups (expert E + e) form one unit over the same x rows, so a thread
// ends a unit holding g and u of its outputs and writes silu(g) * u.
//
// The slab sequence: segment-major, then row tile, then (SW) pass gate/up, then
// k-group. A cursor walks it.
// position in the slab sequence (segment, row tile, SW pass, k-group)
template <bool SW>
struct Cursor {
  int g, pass, t, seg;
  __device__ __forceinline__ void init(int s, int G, int RT) {
    g = s % G;
    int u = s / G;
    pass = 0;
    if constexpr (SW) { pass = u & 1; u >>= 1; }
    t = u % RT;
    seg = u / RT;
  }
  __device__ __forceinline__ void next(int G, int RT) {
    if (++g < G) return;
    g = 0;
    if constexpr (SW) {
      if (++pass < 2) return;
      pass = 0;
    }
    if (++t == RT) { t = 0; ++seg; }
  }
};

// What the producer waits for before it copies the activations: the previous kernel
// in the stream (griddepcontrol.wait), and in the second phase of the MLP layer kernel
// also every CTA's first phase (a generation counter in global memory; counter ==
// nullptr: none). The wait is bounded and latches QMV_ETIMEOUT.
struct DepWait {
  const unsigned* counter;
  unsigned target;
};
__device__ __forceinline__ bool dep_wait(const DepWait& d, unsigned* status) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (d.counter == nullptr) return true;
  const unsigned long long t0 = globaltimer();
  for (;;) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(d.counter) : "memory");
    if ((int)(v - d.target) >= 0) break;
    if (globaltimer() - t0 > kTimeoutNs) {
      atomicOr(status, kStatTimeout);
      return false;
    }
    __nanosleep(100);
  }
  // the activations were written by plain stores of other CTAs: order them before
  // this thread's bulk copies (the async proxy)
  asm volatile("fence.proxy.async.global;" ::: "memory");
  return true;
}

// One streaming GEMV pass (the whole kernel for qmv_gemv and its relatives; each of
// the two phases of the MLP layer kernel). YB: the epilogue writes bf16 outputs.
template <int FMT, int MT, bool SW, bool GR, bool YB>
__device__ __forceinline__ void stream_body(const KParams& kp, uint8_t* smem, const DepWait dep) {
  const StreamArgs& a = kp.a;
  const Layout& L = a.L;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + kMaxStages;
  volatile int* misc = reinterpret_cast<volatile int*>(smem + 8 * (2 * kMaxStages + 2));
  Seg* segs = reinterpret_cast<Seg*>(smem + 512);
  float2* tbls = reinterpret_cast<float2*>(smem + kp.tbl_off);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;

  // Everything that could depend on the previous kernel (the activations, the
  // workspace, the outputs) is touched only after griddepcontrol.wait (a no-op when
  // launched without the attribute).

  // ---- set-up: header check, segment table, barriers -----------------------
  if (tid == 0) {
    const PackedHeader* h = reinterpret_cast<const PackedHeader*>(a.packed);
    int bad = !(h->magic == kMagic && h->version == kVersion && h->fmt == (uint32_t)L.fmt &&
                h->N == L.N && h->K == L.K && h->E == L.E && h->expert_bytes == L.expert_bytes);
    if (bad) atomicOr(a.status, kStatHeader);
    misc[0] = bad;   // abort flag
    for (int i = 0; i < kp.stages; ++i) {
      mbar_init(&full[i], MT == 1 ? 1 : 1 + 32);   // M > 1: + one cp.async arrival per producer lane
      mbar_init(&empty[i], kConsumerWarps);
    }
    mbar_init(reinterpret_cast<uint64_t*>(smem + kGbarOff), 1);
    mbar_init(reinterpret_cast<uint64_t*>(smem + kGridBarOff), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  if (MT == 1 && warp >= 1) {
    // the zero pad after x row 0 of every stage (the unit-column B operand of the
    // sub-blocks a thread does not own is read from it; copies never write it)
    for (int i = tid - 32; i < kp.stages * (kXZeroBytes / 4); i += (int)blockDim.x - 32) {
      uint8_t* st = smem + kp.stage_base + (i / (kXZeroBytes / 4)) * kp.stage_bytes;
      *reinterpret_cast<uint32_t*>(st + kp.x_off + kXZero + 4 * (i % (kXZeroBytes / 4))) = 0u;
    }
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
      int* skeys = reinterpret_cast<int*>(smem + kp.tbl_off);      // scratch before first use
      asm volatile("griddepcontrol.wait;" ::: "memory");          // ids come from earlier work
      int* sorted = skeys + 64;
      bool bad = false;
      for (int p = lane; p < P; p += 32) {
        const int id = a.ids[p];
        bad |= (id < 0 || (int64_t)id >= (SW ? L.E / 2 : L.E));   // SW: ids index the gate half
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
  if (tid == 0 && !misc[0]) {
    // the CTA's slab range in the cells of this call (CellMap), in misc[6..8]; 32-bit
    // slab counts (the host refuses larger problems)
    cta_range(misc, kp.cells, kp.cpc, kp.gp, misc[1] * (int)L.row_tiles * (int)L.k_groups * (SW ? 2 : 1),
              (int)L.k_groups * (SW ? 2 : 1), (int)gridDim.x, (int)blockIdx.x);
  }
  __syncthreads();
  if (misc[0]) return;

  const int nseg = misc[1];
  // slab counts fit in 32 bits (the host refuses larger problems)
  const int G = (int)L.k_groups;
  const int RT = (int)L.row_tiles;
  const int S = nseg * RT * G * (SW ? 2 : 1);
  const int Eh = SW ? (int)(L.E / 2) : 0;        // SW: the up matrix of expert e is expert Eh + e
  const int P = (int)gridDim.x;
  const int c = (int)blockIdx.x;
  // Cells: the fixed partition of the slab sequence that the accumulation order
  // follows (pieces never cross a cell boundary). Dense calls: V = kp.cells cells,
  // cell i = slabs [floor(i S / V), floor((i+1) S / V)), kp.cpc consecutive cells per
  // CTA; V depends on the matrix and the SM count only, never on M, so every M sums
  // in the same order. Grouped calls: each unit is cut into cells of gp slabs (gp a
  // function of K only), and CTA c holds a contiguous range of whole cells. In 32-bit
  // arithmetic (i * Sr < V * V).
  constexpr bool dense_cells = !GR;       // GR: a grouped call (its own instances)
  const int s0 = misc[6], s1 = misc[7];
  if (s0 >= s1) return;
  // the last k-group is narrower than 256 only for formats with 16/32-value blocks
  constexpr bool kMayBeRagged = (FMT == F_Q8_0 || FMT == F_NVFP4 || FMT == F_FP8);
  const int kv_last = (int)(L.K - (int64_t)(G - 1) * kSlabK);

  // M = 1: one lane of the producer warp streams the slabs of [s0, s1) into the stages
  auto produce1 = [&]() {
    Cursor<SW> cur;
    cur.init(s0, G, RT);
    int stage = 0;
    uint32_t rphase = 0;          // parity of the current round over the stage ring
    int it = 0;
    const uint32_t abytes = (uint32_t)(kSlabRows * L.rec);
    const uint32_t bbytes = (uint32_t)plane_b_tile<FMT>();
    // The first round of stages: weights first (independent of earlier kernels),
    // then wait for the previous grid, then the activations of those stages.
    const int first = (s1 - s0) < kp.stages ? (s1 - s0) : kp.stages;
    // grouped: the weights of every stage are fetched only now (they follow from the
    // ids), and all CTAs start at once; the first stage goes alone, so that it lands
    // first and the consumers start while the others are in flight
    const int first_w = (GR && first > 1) ? 1 : first;
    {
      Cursor<SW> c2 = cur;
      for (int i = 0; i < first_w; ++i) {
        const Seg& sg = segs[c2.seg];
        uint8_t* st = smem + kp.stage_base + i * kp.stage_bytes;
        const uint8_t* plane =
            a.packed + L.base + (sg.expert + c2.pass * Eh) * L.expert_bytes + c2.g * L.group_bytes;
        const int kv = (kMayBeRagged && c2.g == G - 1) ? kv_last : kSlabK;
        const int R = sg.R < MT ? sg.R : MT;
        mbar_expect_tx(&full[i], abytes + bbytes + (uint32_t)(kv * 2) * (uint32_t)R);
        bulk_g2s(st, plane + (int64_t)c2.t * kSlabRows * L.rec, abytes, &full[i]);
        if (bbytes) bulk_g2s(st + kp.b_off, plane + L.plane_a + (int64_t)c2.t * bbytes, bbytes, &full[i]);
        c2.next(G, RT);
      }
    }
    if (!dep_wait(dep, a.status)) misc[0] = 1;
    for (int s = s0; s < s1; ++s, ++it) {
      if (it >= kp.stages) {      // round r >= 1 waits for the consumers' release of round r-1
        if (!mbar_wait(&empty[stage], rphase ^ 1u, a.status)) { misc[0] = 1; break; }
      }
      if (misc[0]) break;
      const Seg& sg = segs[cur.seg];
      uint8_t* st = smem + kp.stage_base + stage * kp.stage_bytes;
      const uint8_t* plane =
          a.packed + L.base + (sg.expert + cur.pass * Eh) * L.expert_bytes + cur.g * L.group_bytes;
      const int kv = (kMayBeRagged && cur.g == G - 1) ? kv_last : kSlabK;
      const uint32_t xbytes = (uint32_t)(kv * 2);
      const int R = sg.R < MT ? sg.R : MT;
      if (it >= first_w) {
        mbar_expect_tx(&full[stage], abytes + bbytes + xbytes * (uint32_t)R);
        bulk_g2s(st, plane + (int64_t)cur.t * kSlabRows * L.rec, abytes, &full[stage]);
        if (bbytes) bulk_g2s(st + kp.b_off, plane + L.plane_a + (int64_t)cur.t * bbytes, bbytes, &full[stage]);
      }
      for (int r = 0; r < R; ++r)
        bulk_g2s(st + kp.x_off + r * kXStride, a.x + (int64_t)sg.xrow[r] * L.K + (int64_t)cur.g * kSlabK, xbytes,
                 &full[stage]);
      if (GR && it == 0 && first > 1 && !mbar_wait(&full[0], 0u, a.status)) misc[0] = 1;
      if (++stage == kp.stages) { stage = 0; rphase ^= 1u; }
      cur.next(G, RT);
    }
    // drain: copies issued into stages the consumers may not have waited for
    if (misc[0]) {
      const int issued = it;
      for (int j = (issued > kp.stages ? issued - kp.stages : 0); j < issued; ++j)
        (void)mbar_wait(&full[j % kp.stages], (uint32_t)((j / kp.stages) & 1), a.status);
    }
  };

  // M > 1: the producer warp streams the slabs of [s0, s1) into the stages. One lane
  // moves the weights with bulk copies; the 32 lanes copy the slices of the x rows
  // with 16-byte cp.async, each lane's copies tracked by the stage's full barrier
  // (cp.async.mbarrier.arrive.noinc: 32 more arrivals), so R x rows cost no more
  // than one bulk copy.
  // lanes taking part: M = 1 -> lane 0 only (the others leave), M > 1 -> all 32
  constexpr unsigned kPMask = (MT == 1) ? 1u : 0xffffffffu;
  auto produce8 = [&]() {
    Cursor<SW> cur;
    cur.init(s0, G, RT);
    int stage = 0;
    uint32_t rphase = 0;          // parity of the current round over the stage ring
    int it = 0;
    const uint32_t abytes = (uint32_t)(kSlabRows * L.rec);
    const uint32_t bbytes = (uint32_t)plane_b_tile<FMT>();
    // The first round of stages: weights first (independent of earlier kernels),
    // then wait for the previous grid, then the activations of those stages.
    const int first = (s1 - s0) < kp.stages ? (s1 - s0) : kp.stages;
    if (lane == 0) {
      Cursor<SW> c2 = cur;
      for (int i = 0; i < first; ++i) {
        const Seg& sg = segs[c2.seg];
        uint8_t* st = smem + kp.stage_base + i * kp.stage_bytes;
        const uint8_t* plane =
            a.packed + L.base + (sg.expert + c2.pass * Eh) * L.expert_bytes + c2.g * L.group_bytes;
        const int kv = (kMayBeRagged && c2.g == G - 1) ? kv_last : kSlabK;
        const int R = sg.R < MT ? sg.R : MT;
        const uint32_t xtx = (MT == 1) ? (uint32_t)(kv * 2) * (uint32_t)R : 0u;
        mbar_expect_tx(&full[i], abytes + bbytes + xtx);
        bulk_g2s(st, plane + (int64_t)c2.t * kSlabRows * L.rec, abytes, &full[i]);
        if (bbytes) bulk_g2s(st + kp.b_off, plane + L.plane_a + (int64_t)c2.t * bbytes, bbytes, &full[i]);
        c2.next(G, RT);
      }
    }
    {
      bool ok = true;
      if (lane == 0) ok = dep_wait(dep, a.status);
      else asm volatile("griddepcontrol.wait;" ::: "memory");
      ok = __shfl_sync(kPMask, ok, 0);
      if (!ok && lane == 0) misc[0] = 1;
      __syncwarp(kPMask);
    }
    for (int s = s0; s < s1; ++s, ++it) {
      if (it >= kp.stages) {      // round r >= 1 waits for the consumers' release of round r-1
        bool ok = true;
        if (lane == 0) ok = mbar_wait(&empty[stage], rphase ^ 1u, a.status);
        ok = __shfl_sync(kPMask, ok, 0);
        if (!ok) { if (lane == 0) misc[0] = 1; break; }
      }
      if (__shfl_sync(kPMask, misc[0], 0)) break;
      const Seg& sg = segs[cur.seg];
      uint8_t* st = smem + kp.stage_base + stage * kp.stage_bytes;
      const uint8_t* plane =
          a.packed + L.base + (sg.expert + cur.pass * Eh) * L.expert_bytes + cur.g * L.group_bytes;
      const int kv = (kMayBeRagged && cur.g == G - 1) ? kv_last : kSlabK;
      const uint32_t xbytes = (uint32_t)(kv * 2);
      const int R = sg.R < MT ? sg.R : MT;
      if (lane == 0 && it >= first) {
        mbar_expect_tx(&full[stage], abytes + bbytes + (MT == 1 ? xbytes * (uint32_t)R : 0u));
        bulk_g2s(st, plane + (int64_t)cur.t * kSlabRows * L.rec, abytes, &full[stage]);
        if (bbytes) bulk_g2s(st + kp.b_off, plane + L.plane_a + (int64_t)cur.t * bbytes, bbytes, &full[stage]);
      }
      if (MT == 1) {
        if (lane == 0)
          for (int r = 0; r < R; ++r)
            bulk_g2s(st + kp.x_off + r * kXStride, a.x + (int64_t)sg.xrow[r] * L.K + (int64_t)cur.g * kSlabK,
                     xbytes, &full[stage]);
      } else {
        const int chunks = (int)(xbytes / 16);       // 16-byte pieces of one row's slice
        for (int r = 0; r < R; ++r) {
          const uint8_t* src =
              reinterpret_cast<const uint8_t*>(a.x + (int64_t)sg.xrow[r] * L.K + (int64_t)cur.g * kSlabK);
          uint8_t* dst = st + kp.x_off + r * kXStride;
          for (int c16 = lane; c16 < chunks; c16 += 32) cp_async16(dst + 16 * c16, src + 16 * c16);
        }
        cp_async_arrive_noinc(&full[stage]);
      }
      if (++stage == kp.stages) { stage = 0; rphase ^= 1u; }
      cur.next(G, RT);
    }
    // drain: copies issued into stages the consumers may not have waited for. At
    // M > 1 the first-round stages not reached above still expect the lanes'
    // arrivals: the lanes arrive on them without copies, so they complete.
    if (__shfl_sync(kPMask, misc[0], 0)) {
      const int issued = it > first ? it : first;
      if (MT > 1)
        for (int j = it; j < first; ++j) mbar_arrive(&full[j]);
      __syncwarp(kPMask);
      if (lane == 0)
        for (int j = (issued > kp.stages ? issued - kp.stages : 0); j < issued; ++j)
          (void)mbar_wait(&full[j % kp.stages], (uint32_t)((j / kp.stages) & 1), a.status);
    }
    if (MT > 1) asm volatile("cp.async.wait_all;" ::: "memory");
  };

  if (warp == 0) {
    // ---------------------------- producer --------------------------------
    // the grid formats: the f16 grid (one table for the call) lands once, before the
    // first slab is decoded; the producer waits for it before it leaves
    const bool grid_copy = is_grid_fmt(FMT) && !misc[0];
    if (grid_copy && lane == 0) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");   // after the set-up's plain stores
      uint64_t* gb = reinterpret_cast<uint64_t*>(smem + kGridBarOff);
      mbar_expect_tx(gb, (uint32_t)grid_smem_bytes<FMT>());
      bulk_g2s(smem + kp.grid_off, a.packed + kHeaderBytes, (uint32_t)grid_smem_bytes<FMT>(), gb);
    }
    if constexpr (MT == 1) {
      if (lane == 0) produce1();
    } else {
      produce8();
    }
    if (grid_copy && lane == 0) (void)mbar_wait(reinterpret_cast<uint64_t*>(smem + kGridBarOff), 0u, a.status);
    // the gather list of the CTA's last unit: built once here, where the warp has time,
    // instead of by every consumer warp at the end
    __syncwarp();
    build_gather_list(misc, reinterpret_cast<volatile int*>(smem + kGatherOff), kp.cells, kp.cpc, kp.gp, S,
                      G * (SW ? 2 : 1), G, SW ? 2 : 1, P, c, kp.maxslots, kSlabRows * kp.mt, lane);
    if (lane == 0) mbar_arrive(reinterpret_cast<uint64_t*>(smem + kGbarOff));   // release: the list is visible
    __syncwarp();
    return;
  }
  // ------------------------------ consumers ---------------------------------
  // After an abort (a wait that timed out, here or in another warp) a warp still
  // walks its slab sequence but skips the waits, the arithmetic and the stores.
  //
  // The accumulation order (the same for every M): a unit is a row tile of one
  // segment (SW: its gate k-groups, then its up k-groups); a piece is a maximal run
  // of a unit's slabs inside one cell and one pass. Per output, a piece's value is
  // (A_0 + A_1) + (A_2 + A_3) of its slabs (qmv_slab.cuh), and a unit's value (per
  // pass) is the fp32 sum of its pieces in k order, starting from zero. The CTA
  // holding a unit's first slab (its reducer) adds its own pieces as it goes and then
  // the pieces that later CTAs published, in order; every other CTA publishes each
  // piece of the unit in the workspace slot (CTA, piece ordinal).
  const int w = warp - 1;               // this warp owns rows 16w .. 16w+15 of a slab
  constexpr bool kConvX = (MT > 1) && (FMT == F_NVFP4 || FMT == F_FP8 || FMT >= F_IQ4_XS);
  const int g = lane >> 2, tq = lane & 3;
  float2* tbl = tbls + w * (16 * kTblStride);
  const int rA = 16 * w + g, rB = rA + 8;
  constexpr int UG = SW ? 2 : 1;          // passes per unit (gate, up)
  const int UL = UG * G;                  // slabs per unit
  const int pstride = kSlabRows * kp.mt;  // words of one published piece
  unsigned* const parts = reinterpret_cast<unsigned*>(kp.partials);
  float pa1[2];                           // M = 1: this thread's A_t of rows rA, rB
  float pa8[4][4];                        // M > 1: A_0 .. A_3 of the thread's four outputs
  float uacc[UG][4];                      // the unit's value per pass (reducer)
  int T = s0 / UL;                        // current unit
  int tt = T % RT, seg = T / RT;
  int stage = 0;
  uint32_t fphase = 0;                   // parity of the full barrier for this stage round
  bool aborted = false;
  int cell_ord = 0;                      // grouped: ordinal of the current cell in the range
  if constexpr (is_grid_fmt(FMT)) {
    // the grid formats decode from the f16 grid in shared memory (passed to the
    // decoders in the place of the scale tables, which they do not use)
    tbl = reinterpret_cast<float2*>(smem + kp.grid_off);
    if (!misc[0] && !mbar_wait(reinterpret_cast<uint64_t*>(smem + kGridBarOff), 0u, a.status)) {
      misc[0] = 1;
      aborted = true;
    }
  }
  for (int s = s0; s < s1;) {
    const Seg& sg = segs[seg];
    const int R = sg.R < MT ? sg.R : MT;
    const bool has_x = g < R;
    const int head = T * UL, tail = head + UL;
    const int send = tail < s1 ? tail : s1;
    const bool reducer = (s0 <= head);
#pragma unroll
    for (int pp = 0; pp < UG; ++pp)
#pragma unroll
      for (int e = 0; e < 4; ++e) uacc[pp][e] = 0.f;
    while (s < send) {
      // ---- one piece [s, pe): inside one cell and one pass of unit T ----
      aborted = aborted || misc[0];
      int pe = send;
      int ce = 0;                                   // grouped: the end of s's cell
      if constexpr (!dense_cells) {
        const int gsh = kp.gp >> 1;
        ce = head + ((((s - head) >> gsh) + 1) << gsh);
        if (ce > tail) ce = tail;
        if (ce < pe) pe = ce;
      } else {
        const int sm = misc[8];
        if (s < sm && sm < pe) pe = sm;
      }
      if (SW && s - head < G && head + G < pe) pe = head + G;
      if constexpr (MT == 1) {
        pa1[0] = pa1[1] = 0.f;
      } else {
#pragma unroll
        for (int t = 0; t < 4; ++t)
#pragma unroll
          for (int e = 0; e < 4; ++e) pa8[t][e] = 0.f;
      }
      for (; s < pe; ++s) {
        bool have = false;
        if (!aborted) {
          if (!mbar_wait(&full[stage], fphase, a.status)) {
            misc[0] = 1;
            aborted = true;
          } else {
            have = true;
          }
        }
        if constexpr (kConvX) {
          // the f16-operand formats at M > 1: the eight consumer warps turn the stage's x
          // rows from bf16 into f16 in place, warp w row w, 16 bytes per lane (zeros past
          // a ragged K), once for all warps; every warp meets the barrier once per slab,
          // whether it waited for the slab or not
          if (have && w < R) {
            uint4* xv = reinterpret_cast<uint4*>(smem + kp.stage_base + stage * kp.stage_bytes + kp.x_off +
                                                 w * kXStride + 16 * lane);
            const int gk = (s - head) % G;
            uint4 v = *xv;
            if (kMayBeRagged && gk == G - 1 && 8 * lane >= kv_last) {
              v = make_uint4(0u, 0u, 0u, 0u);
            } else {
              v.x = bf16x2_to_f16x2(v.x);
              v.y = bf16x2_to_f16x2(v.y);
              v.z = bf16x2_to_f16x2(v.z);
              v.w = bf16x2_to_f16x2(v.w);
            }
            *xv = v;
          }
          asm volatile("bar.sync 1, 256;" ::: "memory");
        }
        if (have) {
          const uint8_t* st = smem + kp.stage_base + stage * kp.stage_bytes;
          const uint8_t* xrow0 = st + kp.x_off;
          // a last k-group narrower than 256: its padded blocks are zero and the x
          // beyond K is never copied, so the stale tail of each x row is zeroed (by
          // one thread of each warp, before that warp reads it; the converted formats
          // zeroed it above)
          if (!kConvX && kMayBeRagged && (s - head) % G == G - 1 && kv_last < kSlabK) {
            if (has_x && tq == 0) {
              uint8_t* xw = const_cast<uint8_t*>(xrow0) + g * kXStride;
              for (int o = kv_last * 2; o < kSlabK * 2; o += 4) *reinterpret_cast<uint32_t*>(xw + o) = 0u;
            }
            __syncwarp();
          }
          if constexpr (MT == 1) {
            Slab<FMT, 1>::run(st, st + kp.b_off, xrow0, R, w, lane, tbl, pa1);
          } else {
            Slab<FMT, MT>::run(st, st + kp.b_off, xrow0 + (has_x ? g : 0) * kXStride, R, w, lane, tbl, pa8);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[stage]);
        }
        if (++stage == kp.stages) { stage = 0; fphase ^= 1u; }
      }
      // ---- the piece's value: (A_0 + A_1) + (A_2 + A_3) per output ----
      const int pass = (SW && pe - 1 - head >= G) ? 1 : 0;   // the piece's pass (from its last slab)
      float pv[4];
      if constexpr (MT == 1) {
        // unit columns: quad position tq holds A_tq of rows rA, rB (token 0)
        float vA = pa1[0], vB = pa1[1];
        vA = __fadd_rn(vA, __shfl_xor_sync(0xffffffffu, vA, 1));
        vB = __fadd_rn(vB, __shfl_xor_sync(0xffffffffu, vB, 1));
        vA = __fadd_rn(vA, __shfl_xor_sync(0xffffffffu, vA, 2));
        vB = __fadd_rn(vB, __shfl_xor_sync(0xffffffffu, vB, 2));
        pv[0] = vA; pv[1] = 0.f; pv[2] = vB; pv[3] = 0.f;
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) pv[e] = quad_join(pa8[0][e], pa8[1][e], pa8[2][e], pa8[3][e]);
      }
      if (reducer) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (MT == 1 && (e & 1)) continue;            // M = 1: token 0 only
          if (SW && pass) uacc[UG - 1][e] = __fadd_rn(uacc[UG - 1][e], pv[e]);
          else uacc[0][e] = __fadd_rn(uacc[0][e], pv[e]);
        }
      } else if (!aborted && kp.fault != 1) {
        // peer: publish the piece. Each stored word is its own completion flag: it is
        // never zero (+0.0 is stored as a NaN pattern that no sum produces here, and
        // decoded back to +0.0), and the reducer waits for each word to become
        // non-zero -- no fence, no flag.
        asm volatile("griddepcontrol.wait;" ::: "memory");   // the workspace after earlier kernels
        // dense: the piece is in the CTA's second cell iff its last slab is (pieces do
        // not cross cells); grouped: one slot per (cell, pass) of the CTA's range
        const int slot = dense_cells ? ((pe - 1 >= misc[8] ? 1 : 0) * UG + pass) : (cell_ord * UG + pass);
        unsigned* part = parts + ((int64_t)c * kp.maxslots + slot) * pstride;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (MT == 1 && (e & 1)) continue;
          const int tok = 2 * tq + (e & 1), row = (e < 2) ? rA : rB;
          if (tok < R) st_relaxed(part + row * kp.mt + tok, encode_piece(pv[e]));
        }
      }
      if constexpr (!dense_cells) {
        if (pe == ce) ++cell_ord;
      }
    }

    // ---- end of unit T in this CTA: this thread owns rows rA, rB and tokens 2tq, 2tq+1 ----
    asm volatile("griddepcontrol.wait;" ::: "memory");   // workspace and y after earlier kernels
    if (reducer && !aborted && tail > s1) {
      if (!mbar_wait(reinterpret_cast<uint64_t*>(smem + kGbarOff), 0u, a.status)) { misc[0] = 1; aborted = true; }
      if (kp.fault == 2) { atomicOr(a.status, kStatTimeout); misc[0] = 1; aborted = true; }
      // the pieces of unit T that later CTAs published, in slab order, from the list
      // the producer warp built, KB at a time so that their load latencies overlap; each
      // word is cleared after it is read (the workspace is all zero again when the
      // call ends)
      constexpr int KB = SW ? 2 : 4;
      constexpr int NE = MT == 1 ? 2 : 4;          // outputs e of this thread (M = 1: e = 0, 2)
      const volatile int* glist = reinterpret_cast<const volatile int*>(smem + kGatherOff);
      const int n = misc[2];
      for (int i0 = 0; i0 < n && !aborted; i0 += KB) {
        uint32_t u[KB][NE];
        int pc[KB];
#pragma unroll
        for (int k = 0; k < KB; ++k) {
          pc[k] = (i0 + k < n) ? glist[i0 + k] : -1;
#pragma unroll
          for (int j = 0; j < NE; ++j) {
            const int e = MT == 1 ? 2 * j : j;
            const int tok = 2 * tq + (e & 1), row = (e < 2) ? rA : rB;
            u[k][j] = 0u;
            if (pc[k] >= 0 && tok < R) u[k][j] = ld_relaxed(parts + (pc[k] & ~1) + row * kp.mt + tok);
          }
        }
#pragma unroll
        for (int k = 0; k < KB; ++k) {
#pragma unroll
          for (int j = 0; j < NE; ++j) {
            const int e = MT == 1 ? 2 * j : j;
            const int tok = 2 * tq + (e & 1), row = (e < 2) ? rA : rB;
            if (pc[k] < 0 || tok >= R || aborted) continue;
            unsigned* wp = parts + (pc[k] & ~1) + row * kp.mt + tok;
            uint32_t v = u[k][j];
            if (v == 0u) {
              const unsigned long long t0 = globaltimer();
              while ((v = ld_relaxed(wp)) == 0u) {
                if (globaltimer() - t0 > kp.peer_wait_ns) break;
              }
              if (v == 0u) { atomicOr(a.status, kStatTimeout); misc[0] = 1; aborted = true; continue; }
            }
            st_relaxed(wp, 0u);
            const float f = decode_piece(v);
            if (SW && (pc[k] & 1)) uacc[UG - 1][e] = __fadd_rn(uacc[UG - 1][e], f);
            else uacc[0][e] = __fadd_rn(uacc[0][e], f);
          }
        }
      }
      if (!aborted && misc[5]) {
        GatherArgs ga;
        ga.misc = misc;
        ga.glist = reinterpret_cast<const volatile int*>(smem + kGatherOff);
        ga.parts = parts;
        ga.status = a.status;
        ga.wait_ns = kp.peer_wait_ns;
        ga.cells = kp.cells; ga.cpc = kp.cpc; ga.gp = kp.gp; ga.S = S; ga.UL = UL; ga.G = G; ga.P = P;
        ga.maxslots = kp.maxslots; ga.pstride = pstride; ga.mt = kp.mt; ga.R = R; ga.tq = tq;
        ga.rA = rA; ga.rB = rB; ga.head = head; ga.tail = tail;
        if (!gather_unit<MT, SW>(ga, &uacc[0][0])) aborted = true;
      }
    }
    if (reducer && !aborted) {
      const uint8_t* extras = a.packed + L.base + sg.expert * L.expert_bytes + L.k_groups * L.group_bytes;
      const uint8_t* extras_u = extras + (int64_t)Eh * L.expert_bytes;     // SW: the up expert's
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int tok = 2 * tq + (e & 1), row = (e < 2) ? rA : rB;
        const int64_t n = (int64_t)tt * kSlabRows + row;
        if ((MT == 1 && (e & 1)) || tok >= R || n >= L.N) continue;
        float v = uacc[0][e];
        if (FMT == F_NVFP4) v *= *reinterpret_cast<const float*>(extras);
        if (FMT == F_FP8) v *= reinterpret_cast<const float*>(extras)[n];
        if (SW) {
          float uv = uacc[UG - 1][e];
          if (FMT == F_NVFP4) uv *= *reinterpret_cast<const float*>(extras_u);
          if (FMT == F_FP8) uv *= reinterpret_cast<const float*>(extras_u)[n];
          v = (v / (1.0f + expf(-v))) * uv;               // silu(g) * u
        }
        if constexpr (YB)
          reinterpret_cast<__nv_bfloat16*>(a.y)[(int64_t)sg.yrow[tok] * L.N + n] = __float2bfloat16_rn(v);
        else
          a.y[(int64_t)sg.yrow[tok] * L.N + n] = v;
      }
    }
    ++T;
    if (++tt == RT) { tt = 0; ++seg; }
  }
}

// The decode GEMV kernel: one pass. Programmatic dependent launch: the next kernel
// in the stream may start its own prologue and weight prefetch as SMs free up.
template <int FMT, int MT, bool SW, bool GR>
__global__ void __launch_bounds__(kThreads, ctas_per_sm<MT>()) stream_kernel(const KParams kp) {
  extern __shared__ __align__(1024) uint8_t smem[];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  stream_body<FMT, MT, SW, GR, false>(kp, smem, DepWait{nullptr, 0u});
}

// The MLP layer in one launch: phase 1 is the fused gate|up pass with the SwiGLU
// epilogue, writing h as bf16 into the workspace; phase 2 is the down projection over
// h. Between them every CTA arrives on a generation counter (its h rows are stored);
// each CTA's producer issues its first phase-2 weight copies at once and waits on the
// counter only before it copies h. All CTAs of the grid are resident together (at
// most ctas_per_sm() per SM, as for the GEMV), so the wait ends.
template <int FMT, int MT>
__global__ void __launch_bounds__(kThreads, ctas_per_sm<MT>())
    layer_kernel(const KParams kp1, const KParams kp2, unsigned* counter) {
  extern __shared__ __align__(1024) uint8_t smem[];
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  stream_body<FMT, MT, true, false, true>(kp1, smem, DepWait{nullptr, 0u});
  __syncthreads();
  unsigned target = 0u;
  if (threadIdx.x == 0) {
    // this CTA's h stores (every warp passed the barrier above) before its arrival
    asm volatile("fence.proxy.async.global;" ::: "memory");
    __threadfence();
    const unsigned old = atomicAdd(counter, 1u);
    target = (old / gridDim.x + 1u) * gridDim.x;
    // phase 1's barriers are idle: invalidate them for phase 2's set-up
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    for (int i = 0; i < kp1.stages; ++i) {
      mbar_inval(&full[i]);
      mbar_inval(&full[kMaxStages + i]);
    }
    mbar_inval(reinterpret_cast<uint64_t*>(smem + kGbarOff));
    mbar_inval(reinterpret_cast<uint64_t*>(smem + kGridBarOff));
  }
  __syncthreads();
  stream_body<FMT, MT, false, false, false>(kp2, smem, DepWait{counter, target});
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
static int64_t piece_bytes(int M) { return (int64_t)kSlabRows * (M <= 1 ? 1 : 8) * 4; }

StreamPlan plan_stream_dense(int64_t slabs, int M, int passes, int sms) {
  StreamPlan p;
  // Long calls (8 slabs or more per cell at two cells per SM): one cell per CTA, two
  // CTAs per SM, whose warps hide each other's latency. Shorter calls: one cell per
  // SM and one CTA per SM, so that the next call's CTAs are resident beside this
  // call's and copy their first slabs meanwhile, and a unit spans fewer cells (fewer
  // pieces to gather). The cells, and so the order of the sums, depend on the matrix
  // and the SM count only, never on M.
  const bool long_call = slabs >= 16 * (int64_t)sms;
  const int64_t vmax = long_call ? 2 * (int64_t)sms : (int64_t)sms;
  const int64_t v = slabs < vmax ? slabs : vmax;
  p.cells = (int)(v > 0 ? v : 1);
  p.cpc = 1;
  p.gp = 1;
  p.grid = (p.cells + p.cpc - 1) / p.cpc;
  p.maxslots = p.cpc * passes;          // a CTA publishes pieces of its first unit only
  p.ws_bytes = align_up((int64_t)p.grid * p.maxslots * piece_bytes(M), 256);
  return p;
}

StreamPlan plan_stream_grouped(int64_t slabs_max, int M, int passes, int64_t k_groups, int sms) {
  (void)M;
  StreamPlan p;
  const int64_t unit = passes * k_groups;
  p.cells = 0;
  p.cpc = 1;
  // cells of gp k-groups within a unit (a function of K alone, so the order of the
  // sums is the same for every M and routing): a reducer gathers a quarter of the
  // pieces it would with one cell per slab; CTA ranges are whole cells
  p.gp = (k_groups % 4 == 0) ? 4 : (k_groups % 2 == 0 ? 2 : 1);
  const int64_t cells_max = (slabs_max + p.gp - 1) / p.gp;
  const int64_t n = 2 * (int64_t)sms;
  p.grid = (int)(cells_max < n ? (cells_max > 0 ? cells_max : 1) : n);
  {   // as few CTAs as give the same cells per CTA at most
    const int64_t per = (cells_max + p.grid - 1) / p.grid;
    p.grid = (int)((cells_max + per - 1) / per);
  }
  // a CTA publishes the slabs of its first unit but the unit's first one; the slot of
  // a slab is (its ordinal in the CTA's range) x passes + its pass
  const int64_t per_cta = (slabs_max + p.grid - 1) / p.grid;
  const int64_t ms = (unit - 1 < per_cta ? unit - 1 : per_cta) * passes;
  p.maxslots = (int)(ms > 0 ? ms : 1);
  p.ws_bytes = align_up((int64_t)p.grid * p.maxslots * piece_bytes(M), 256);
  return p;
}

static int g_fault = 0;
static unsigned long long g_peer_wait_ns = kTimeoutNs;

void set_split_fault(int mode, unsigned long long peer_wait_ns) {
  g_fault = (mode == 1 || mode == 2) ? mode : 0;
  g_peer_wait_ns = (g_fault == 1 && peer_wait_ns > 0) ? peer_wait_ns : kTimeoutNs;
}

int num_sms_current_device() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// The kernel parameters of one pass (shared-memory layout, stage count, the plan's
// cells), validated; *smem = the dynamic shared memory the pass needs.
template <int FMT, int MT, bool SW>
static cudaError_t prep_kp(const StreamArgs& a, KParams& kp, int* smem_out, int* dev_out) {
  int dev = 0, smem_max = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  err = cudaDeviceGetAttribute(&smem_max, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
  if (err != cudaSuccess) return err;
  int smem_sm = 0;
  err = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev);
  if (err != cudaSuccess) return err;
  int sm_count = 0;
  err = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  if (a.num_ctas < 1 || a.num_ctas > ctas_per_sm<MT>() * sm_count) return cudaErrorInvalidConfiguration;
  // per CTA: its share of the SM less the 1 KB the hardware reserves per CTA
  const int smem_cta = smem_sm / ctas_per_sm<MT>() - 1024;
  if (smem_cta < smem_max) smem_max = smem_cta;
  kp.a = a;
  kp.mt = MT;
  kp.tbl_off = 512 + kMaxSeg * (int)sizeof(Seg);
  // the per-warp scale tables serve the token-column (M > 1) decoders only
  const int tbl_bytes = (MT > 1) ? kConsumerWarps * 16 * kTblStride * (int)sizeof(float2) : 0;
  // the grid lies past the segment sort's scratch (512 B at tbl_off, written before
  // the grid copy lands), whether or not scale tables follow
  kp.grid_off = (int)align_up(kp.tbl_off + (tbl_bytes > 512 ? tbl_bytes : 512), 128);
  kp.stage_base = (int)align_up(kp.grid_off + grid_smem_bytes<FMT>(), 1024);
  const int abytes = kSlabRows * a.L.rec;
  kp.b_off = (int)align_up(abytes, 128);
  const int bbytes = plane_b_tile<FMT>();
  kp.x_off = (int)align_up(kp.b_off + bbytes, 128);
  kp.stage_bytes = (int)align_up(kp.x_off + MT * kXStride, 1024);
  kp.stages = (smem_max - kp.stage_base) / kp.stage_bytes;
  if (kp.stages > kMaxStages) kp.stages = kMaxStages;
  if (kp.stages < 2) return cudaErrorInvalidConfiguration;
  const int64_t pairs = (int64_t)a.M * a.topk;
  const int64_t e_ids = SW ? a.L.E / 2 : a.L.E;      // experts the ids may name
  const int64_t segs_max = a.ids ? (pairs < e_ids ? pairs : e_ids) : 1;
  if (!slab_count_ok(a.L, segs_max * (SW ? 2 : 1))) return cudaErrorInvalidValue;
  kp.cells = a.cells;
  kp.cpc = a.cpc;
  kp.gp = a.gp;
  kp.maxslots = a.maxslots;
  kp.fault = g_fault;
  kp.peer_wait_ns = g_peer_wait_ns;
  if (a.cells > 0 && (a.cpc < 1 || a.cpc > 2 || (int64_t)a.num_ctas * a.cpc < a.cells)) return cudaErrorInvalidValue;
  if (a.maxslots < 1 || (int64_t)a.num_ctas * a.maxslots * kSlabRows * MT * 4 > a.ws_bytes)
    return cudaErrorInvalidValue;
  kp.partials = reinterpret_cast<float*>(a.ws);
  *smem_out = kp.stage_base + kp.stages * kp.stage_bytes;
  *dev_out = dev;
  return cudaSuccess;
}

template <int FMT, int MT, bool SW>
static cudaError_t launch_t(const StreamArgs& a, cudaStream_t s) {
  KParams kp;
  int smem = 0, dev = 0;
  cudaError_t err = prep_kp<FMT, MT, SW>(a, kp, &smem, &dev);
  if (err != cudaSuccess) return err;
  // grouped calls have instances of their own (cells, and at M = 1 the producer's
  // first-stage start)
  const bool gr = a.ids != nullptr;
  void (*kern)(const KParams) = gr ? stream_kernel<FMT, MT, SW, true> : stream_kernel<FMT, MT, SW, false>;
  if (gr != (a.cells <= 0)) return cudaErrorInvalidValue;
  // opt in to the large dynamic shared memory once per device and instance (not per
  // launch, so that stream capture records launches only)
  static int opted[2][64] = {{0}};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (opted[gr][dev] < smem) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    opted[gr][dev] = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a.num_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  // The grid has at most ctas_per_sm() CTAs per SM (checked above) and that many
  // fit on an SM, so every CTA of the grid is resident at once as soon as the
  // previous kernel's CTAs have left (none of which waits on this grid): a
  // reducer's bounded wait on its peers' partial sums ends. With one CTA per SM the
  // next call's CTAs take the free slots early; programmatic stream serialization
  // lets their prologue overlap this grid (see griddepcontrol in the kernel).
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, kern, kp);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

template <int FMT, int MT>
static cudaError_t launch_layer_t(const StreamArgs& a1, const StreamArgs& a2, unsigned* counter, cudaStream_t s) {
  KParams kp1, kp2;
  int smem1 = 0, smem2 = 0, dev = 0;
  cudaError_t err = prep_kp<FMT, MT, true>(a1, kp1, &smem1, &dev);
  if (err != cudaSuccess) return err;
  err = prep_kp<FMT, MT, false>(a2, kp2, &smem2, &dev);
  if (err != cudaSuccess) return err;
  if (a1.num_ctas != a2.num_ctas || a1.ids || a2.ids || a1.cells <= 0 || a2.cells <= 0) return cudaErrorInvalidValue;
  const int smem = smem1 > smem2 ? smem1 : smem2;
  void (*kern)(const KParams, const KParams, unsigned*) = layer_kernel<FMT, MT>;
  static int opted[64] = {0};
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (opted[dev] < smem) {
    err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (err != cudaSuccess) return err;
    opted[dev] = smem;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)a1.num_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = s;
  // at most ctas_per_sm() CTAs per SM (checked in prep_kp), so the whole grid is
  // resident at once once the kernels before it have left: the wait between the
  // phases ends
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  err = cudaLaunchKernelEx(&cfg, kern, kp1, kp2, counter);
  if (err != cudaSuccess) return err;
  return cudaGetLastError();
}

template <int FMT>
static cudaError_t launch_layer_fmt(const StreamArgs& a1, const StreamArgs& a2, unsigned* counter, cudaStream_t s) {
  if (a1.M <= 1) return launch_layer_t<FMT, 1>(a1, a2, counter, s);
  return launch_layer_t<FMT, 8>(a1, a2, counter, s);
}

cudaError_t launch_layer(const StreamArgs& a1, const StreamArgs& a2, unsigned* counter, cudaStream_t s) {
  switch (a1.L.fmt) {
    case F_Q8_0: return launch_layer_fmt<F_Q8_0>(a1, a2, counter, s);
    case F_Q4_K: return launch_layer_fmt<F_Q4_K>(a1, a2, counter, s);
    case F_Q5_K: return launch_layer_fmt<F_Q5_K>(a1, a2, counter, s);
    case F_Q6_K: return launch_layer_fmt<F_Q6_K>(a1, a2, counter, s);
    case F_NVFP4: return launch_layer_fmt<F_NVFP4>(a1, a2, counter, s);
    case F_FP8: return launch_layer_fmt<F_FP8>(a1, a2, counter, s);
    case F_IQ4_XS: return launch_layer_fmt<F_IQ4_XS>(a1, a2, counter, s);
    case F_IQ3_S: return launch_layer_fmt<F_IQ3_S>(a1, a2, counter, s);
    case F_IQ2_S: return launch_layer_fmt<F_IQ2_S>(a1, a2, counter, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int FMT>
static cudaError_t launch_fmt(const StreamArgs& a, cudaStream_t s, int* variant) {
  const bool grouped = a.ids != nullptr;
  *variant = grouped ? 3 : (a.M <= 1 ? 1 : 2);
  if (a.swiglu) {
    *variant = grouped ? 10 : 9;
    if (a.M <= 1) return launch_t<FMT, 1, true>(a, s);
    return launch_t<FMT, 8, true>(a, s);
  }
  if (a.M <= 1) return launch_t<FMT, 1, false>(a, s);   // grouped at M = 1: one x row per expert
  return launch_t<FMT, 8, false>(a, s);
}

cudaError_t launch_stream(const StreamArgs& a, cudaStream_t s, int* variant) {
  switch (a.L.fmt) {
    case F_Q8_0: return launch_fmt<F_Q8_0>(a, s, variant);
    case F_Q4_K: return launch_fmt<F_Q4_K>(a, s, variant);
    case F_Q5_K: return launch_fmt<F_Q5_K>(a, s, variant);
    case F_Q6_K: return launch_fmt<F_Q6_K>(a, s, variant);
    case F_NVFP4: return launch_fmt<F_NVFP4>(a, s, variant);
    case F_FP8: return launch_fmt<F_FP8>(a, s, variant);
    case F_IQ4_XS: return launch_fmt<F_IQ4_XS>(a, s, variant);
    case F_IQ3_S: return launch_fmt<F_IQ3_S>(a, s, variant);
    case F_IQ2_S: return launch_fmt<F_IQ2_S>(a, s, variant);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qmv
