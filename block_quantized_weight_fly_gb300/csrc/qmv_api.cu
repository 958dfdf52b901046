// qmv_api.cu -- the extern "C" entry points of libqmv (declared in include/qmv.h):
// host-side argument validation, the per-device status word, and dispatch to the
// kernels. Nothing here allocates memory, synchronizes a stream or reads device
// data, except qmv_device_status(), which is a diagnostics hook and says so.
#include <atomic>
#include <cstdint>
#include <cuda_runtime.h>
#include "qmv.h"
#include "qmv_internal.h"

namespace {

using namespace qmv;

__device__ unsigned g_status;               // per-device latched status bits

constexpr int kMaxDevices = 64;
// device addresses of the status word, looked up once per device; host threads that
// race on the first look-up store the same value (the address of the symbol in the
// device's current context: after cudaDeviceReset the library must be reloaded)
std::atomic<unsigned*> g_status_ptr[kMaxDevices];
thread_local int g_last_route = 0;

unsigned* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  unsigned* cached = g_status_ptr[dev].load(std::memory_order_acquire);
  if (cached == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status) != cudaSuccess) return nullptr;
    cached = static_cast<unsigned*>(p);
    g_status_ptr[dev].store(cached, std::memory_order_release);
  }
  return cached;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

qmv_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QMV_OK : QMV_ECUDA; }

bool valid_fmt(int f) { return f >= QMV_Q8_0 && f <= QMV_IQ2_S; }

void apply_plan(StreamArgs* a, const StreamPlan& p) {
  a->num_ctas = p.grid;
  a->cells = p.cells;
  a->cpc = p.cpc;
  a->gp = p.gp;
  a->maxslots = p.maxslots;
}

// The MLP layer entry's workspace: the two passes' published pieces (sized for the
// layer's grid, the larger of the two plans'), h as bf16 [M][N_ff], and the counter the
// CTAs arrive on between the passes.
struct LayerPlan {
  StreamPlan p1, p2;
  int grid;
  int64_t off2, off_h, off_cnt, total;
};
bool layer_plan(int fmt, int M, int64_t N_ff, int64_t K_h, int sms, Layout* L1, Layout* L2, LayerPlan* lp) {
  if (!make_layout(fmt, N_ff, K_h, 2, L1) || !make_layout(fmt, K_h, N_ff, 1, L2)) return false;
  if (!slab_count_ok(*L1, 2) || !slab_count_ok(*L2, 1)) return false;
  lp->p1 = plan_stream_dense(2 * L1->row_tiles * L1->k_groups, M, 2, sms);
  lp->p2 = plan_stream_dense(L2->row_tiles * L2->k_groups, M, 1, sms);
  lp->grid = lp->p1.grid > lp->p2.grid ? lp->p1.grid : lp->p2.grid;
  const int64_t pb = 128 * (M <= 1 ? 1 : 8) * 4;
  const int64_t w1 = align_up((int64_t)lp->grid * lp->p1.maxslots * pb, 256);
  const int64_t w2 = align_up((int64_t)lp->grid * lp->p2.maxslots * pb, 256);
  lp->off2 = w1;
  lp->off_h = w1 + w2;
  lp->off_cnt = lp->off_h + align_up((int64_t)M * N_ff * 2, 256);
  lp->total = lp->off_cnt + 256;
  return true;
}

}  // namespace

extern "C" {

size_t qmv_canon_size(qmv_fmt fmt, int64_t N, int64_t K, int64_t E) {
  if (!valid_fmt(fmt) || N <= 0 || K <= 0 || E <= 0) return 0;
  const int64_t bv = (fmt == QMV_Q8_0) ? 32 : (fmt == QMV_NVFP4) ? 16 : (fmt == QMV_FP8_ROW) ? 1 : 256;
  if (K % bv) return 0;
  // the grid formats' stream starts with the tower's grid (one table for all experts)
  const int64_t grid = is_grid_fmt((int)fmt) ? (int64_t)grid_entries((int)fmt) * grid_width((int)fmt) : 0;
  return (size_t)(grid + E * canon_matrix_bytes((int)fmt, N, K));
}

size_t qmv_pack_size(qmv_fmt fmt, int64_t N, int64_t K, int64_t E) {
  Layout L;
  if (!make_layout((int)fmt, N, K, E, &L)) return 0;
  return (size_t)L.total;
}

qmv_status qmv_pack(qmv_fmt fmt, const void* canon, int64_t N, int64_t K, int64_t E, void* dst,
                    cudaStream_t stream) {
  if (!valid_fmt(fmt) || !canon || !dst || N <= 0 || K <= 0 || E <= 0) return QMV_EINVAL;
  Layout L;
  if (!make_layout((int)fmt, N, K, E, &L)) return QMV_EUNSUPPORTED;
  if (!aligned(dst, 256)) return QMV_EALIGN;
  qmv_status st = from_cuda(launch_pack(L, static_cast<const uint8_t*>(canon), static_cast<uint8_t*>(dst), stream));
  if (st == QMV_OK) g_last_route = (int)fmt * 100 + 6;
  return st;
}

qmv_status qmv_quantize(qmv_fmt fmt, const float* W, int64_t rows, int64_t K, float tensor_scale,
                        void* canon, cudaStream_t stream) {
  if (!valid_fmt(fmt) || !W || !canon || rows <= 0 || K <= 0) return QMV_EINVAL;
  if (qmv_canon_size(fmt, rows, K, 1) == 0) return QMV_EUNSUPPORTED;
  if (fmt >= QMV_IQ4_XS) return QMV_EUNSUPPORTED;     // needs a codebook (an input, not a rounding)
  if (fmt == QMV_NVFP4 && !(tensor_scale >= 0.0f)) return QMV_EINVAL;
  if (!aligned(W, 4)) return QMV_EALIGN;
  qmv_status st = from_cuda(launch_quantize((int)fmt, W, rows, K, tensor_scale, static_cast<uint8_t*>(canon), stream));
  if (st == QMV_OK) g_last_route = (int)fmt * 100 + 7;
  return st;
}

qmv_status qmv_quantize_codebook(qmv_fmt fmt, const float* W, int64_t rows, int64_t K, const void* codebook,
                                 void* canon, cudaStream_t stream) {
  if (fmt != QMV_IQ4_XS && fmt != QMV_IQ3_S && fmt != QMV_IQ2_S) return valid_fmt(fmt) ? QMV_EUNSUPPORTED : QMV_EINVAL;
  if (!W || !codebook || !canon || rows <= 0 || K <= 0) return QMV_EINVAL;
  if (qmv_canon_size(fmt, rows, K, 1) == 0) return QMV_EUNSUPPORTED;
  if (!aligned(W, 4)) return QMV_EALIGN;
  qmv_status st = from_cuda(launch_quantize_codebook((int)fmt, W, rows, K, static_cast<const uint8_t*>(codebook),
                                                     static_cast<uint8_t*>(canon), stream));
  if (st == QMV_OK) g_last_route = (int)fmt * 100 + 7;
  return st;
}

qmv_status qmv_dequant(qmv_fmt fmt, const void* packed, int64_t N, int64_t K, int64_t E, int64_t row0,
                       int64_t rows, float* W_out, cudaStream_t stream) {
  if (!valid_fmt(fmt) || !packed || !W_out || N <= 0 || K <= 0 || E <= 0) return QMV_EINVAL;
  if (row0 < 0 || rows < 0 || row0 + rows > N * E) return QMV_EINVAL;
  Layout L;
  if (!make_layout((int)fmt, N, K, E, &L)) return QMV_EUNSUPPORTED;
  if (!aligned(packed, 256) || !aligned(W_out, 4)) return QMV_EALIGN;
  unsigned* status = status_ptr();
  if (!status) return QMV_ECUDA;
  qmv_status st = from_cuda(launch_dequant(L, static_cast<const uint8_t*>(packed), row0, rows, W_out, status, stream));
  if (st == QMV_OK) g_last_route = (int)fmt * 100 + 5;
  return st;
}

size_t qmv_workspace_size(int entry, qmv_fmt fmt, int M, int64_t N, int64_t K, int64_t E, int topk) {
  if (!valid_fmt(fmt) || M <= 0 || N <= 0 || K <= 0) return 0;
  if (entry == QMV_ENTRY_INT8DOT) {          // independent of the device
    Layout L;
    if ((fmt != QMV_Q8_0 && fmt != QMV_Q4_K) || M > QMV_MAX_M || !make_layout((int)fmt, N, K, 1, &L)) return 0;
    return (size_t)int8dot_workspace_bytes(M, K);
  }
  const int sms = num_sms_current_device();
  if (sms <= 0) return 0;
  if (entry == QMV_ENTRY_GEMV || entry == QMV_ENTRY_SWIGLU) {
    const int passes = entry == QMV_ENTRY_SWIGLU ? 2 : 1;
    Layout L;
    if (M > QMV_MAX_M || !make_layout((int)fmt, N, K, passes, &L)) return 0;
    return (size_t)plan_stream_dense(passes * L.row_tiles * L.k_groups, M, passes, sms).ws_bytes;
  }
  if (entry == QMV_ENTRY_GROUPED || entry == QMV_ENTRY_GROUPED_SWIGLU) {
    const int passes = entry == QMV_ENTRY_GROUPED_SWIGLU ? 2 : 1;
    Layout L;
    if (M > QMV_MAX_M || topk < 1 || E < 1 || !make_layout((int)fmt, N, K, passes * E, &L)) return 0;
    const int64_t experts = (int64_t)M * topk < E ? (int64_t)M * topk : E;
    return (size_t)plan_stream_grouped(passes * experts * L.row_tiles * L.k_groups, M, passes, L.k_groups, sms)
        .ws_bytes;
  }
  if (entry == QMV_ENTRY_MLP_LAYER) {
    Layout L1, L2;
    LayerPlan lp;
    if (M > QMV_MAX_M || !layer_plan((int)fmt, M, N, K, sms, &L1, &L2, &lp)) return 0;
    return (size_t)lp.total;
  }
  if (entry == QMV_ENTRY_KQUANT) {
    if ((fmt != QMV_Q4_K && fmt != QMV_Q5_K && fmt != QMV_Q6_K) || K % 256) return 0;
    return (size_t)kq_workspace_bytes(align_up(M, 128), K, sms);
  }
  if (entry == QMV_ENTRY_W4A4) {
    // the activation's NVFP4 tiles (per 256-value k-group, m_pad rows x (128 B codes +
    // 16 B scales)), then the split-K partial sums
    if (fmt != QMV_NVFP4 || K % 256) return 0;
    const int64_t m_pad = align_up(M, 128);
    return (size_t)(align_up((K / 256) * m_pad * 144, 256) + w4a4_partials_bytes(sms));
  }
  return 0;
}

qmv_status qmv_gemv(qmv_fmt fmt, const void* packed_W, const uint16_t* x, float* y, int M, int64_t N,
                    int64_t K, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!valid_fmt(fmt) || !packed_W || !x || !y || !ws) return QMV_EINVAL;
  if (M < 1 || M > QMV_MAX_M || N <= 0 || K <= 0) return QMV_EINVAL;
  Layout L;
  if (!make_layout((int)fmt, N, K, 1, &L) || !slab_count_ok(L, 1)) return QMV_EUNSUPPORTED;
  if (!aligned(packed_W, 256) || !aligned(ws, 256) || !aligned(x, 16) || !aligned(y, 4)) return QMV_EALIGN;
  const int sms = num_sms_current_device();
  if (sms <= 0) return QMV_ECUDA;
  const StreamPlan plan = plan_stream_dense(L.row_tiles * L.k_groups, M, 1, sms);
  if (ws_bytes < (size_t)plan.ws_bytes) return QMV_EWORKSPACE;
  unsigned* status = status_ptr();
  if (!status) return QMV_ECUDA;
  StreamArgs a;
  a.L = L;
  a.packed = static_cast<const uint8_t*>(packed_W);
  a.x = x; a.y = y; a.ids = nullptr;
  a.M = M; a.topk = 1; a.x_per_pair = 0; a.swiglu = 0;
  a.ws = static_cast<uint8_t*>(ws); a.ws_bytes = (int64_t)ws_bytes;
  a.status = status;
  apply_plan(&a, plan);
  int variant = 0;
  qmv_status st = from_cuda(launch_stream(a, stream, &variant));
  if (st == QMV_OK) g_last_route = (int)fmt * 100 + variant;
  return st;
}

qmv_status qmv_grouped(qmv_fmt fmt, const void* tower, const int32_t* expert_ids, const uint16_t* x,
                       int x_per_pair, float* y, int M, int topk, int64_t N, int64_t K, int64_t E,
                       void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!valid_fmt(fmt) || !tower || !expert_ids || !x || !y || !ws) return QMV_EINVAL;
  if (M < 1 || M > QMV_MAX_M || topk < 1 || topk > 8 || N <= 0 || K <= 0 || E <= 0) return QMV_EINVAL;
  if (x_per_pair != 0 && x_per_pair != 1) return QMV_EINVAL;
  if (E > (int64_t)1 << 24) return QMV_EUNSUPPORTED;   // ids are packed with a 6-bit pair index
  Layout L;
  if (!make_layout((int)fmt, N, K, E, &L)) return QMV_EUNSUPPORTED;
  if (!slab_count_ok(L, (int64_t)M * topk < E ? (int64_t)M * topk : E)) return QMV_EUNSUPPORTED;
  if (!aligned(tower, 256) || !aligned(ws, 256) || !aligned(x, 16) || !aligned(y, 4) ||
      !aligned(expert_ids, 4))
    return QMV_EALIGN;
  const int sms = num_sms_current_device();
  if (sms <= 0) return QMV_ECUDA;
  // the distinct experts are found on the device: size the grid for the most
  // there can be (CTAs beyond the slab count get empty ranges)
  const int64_t experts = (int64_t)M * topk < E ? (int64_t)M * topk : E;
  const StreamPlan plan = plan_stream_grouped(experts * L.row_tiles * L.k_groups, M, 1, L.k_groups, sms);
  if (ws_bytes < (size_t)plan.ws_bytes) return QMV_EWORKSPACE;
  unsigned* status = status_ptr();
  if (!status) return QMV_ECUDA;
  StreamArgs a;
  a.L = L;
  a.packed = static_cast<const uint8_t*>(tower);
  a.x = x; a.y = y; a.ids = expert_ids;
  a.M = M; a.topk = topk; a.x_per_pair = x_per_pair; a.swiglu = 0;
  a.ws = static_cast<uint8_t*>(ws); a.ws_bytes = (int64_t)ws_bytes;
  a.status = status;
  apply_plan(&a, plan);
  int variant = 0;
  qmv_status st = from_cuda(launch_stream(a, stream, &variant));
  if (st == QMV_OK) g_last_route = (int)fmt * 100 + variant;
  return st;
}

qmv_status qmv_gemv_swiglu(qmv_fmt fmt, const void* tower, const uint16_t* x, float* h, int M, int64_t N,
                           int64_t K, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!valid_fmt(fmt) || !tower || !x || !h || !ws) return QMV_EINVAL;
  if (M < 1 || M > QMV_MAX_M || N <= 0 || K <= 0) return QMV_EINVAL;
  Layout L;
  if (!make_layout((int)fmt, N, K, 2, &L) || !slab_count_ok(L, 2)) return QMV_EUNSUPPORTED;
  if (!aligned(tower, 256) || !aligned(ws, 256) || !aligned(x, 16) || !aligned(h, 4)) return QMV_EALIGN;
  const int sms = num_sms_current_device();
  if (sms <= 0) return QMV_ECUDA;
  const StreamPlan plan = plan_stream_dense(2 * L.row_tiles * L.k_groups, M, 2, sms);
  if (ws_bytes < (size_t)plan.ws_bytes) return QMV_EWORKSPACE;
  unsigned* status = status_ptr();
  if (!status) return QMV_ECUDA;
  StreamArgs a;
  a.L = L;
  a.packed = static_cast<const uint8_t*>(tower);
  a.x = x; a.y = h; a.ids = nullptr;
  a.M = M; a.topk = 1; a.x_per_pair = 0; a.swiglu = 1;
  a.ws = static_cast<uint8_t*>(ws); a.ws_bytes = (int64_t)ws_bytes;
  a.status = status;
  apply_plan(&a, plan);
  int variant = 0;
  qmv_status st = from_cuda(launch_stream(a, stream, &variant));
  if (st == QMV_OK) g_last_route = (int)fmt * 100 + variant;
  return st;
}

qmv_status qmv_mlp_layer(qmv_fmt fmt, const void* gateup, const void* down, const uint16_t* x, float* y, int M,
                         int64_t N_ff, int64_t K_h, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!valid_fmt(fmt) || !gateup || !down || !x || !y || !ws) return QMV_EINVAL;
  if (M < 1 || M > QMV_MAX_M || N_ff <= 0 || K_h <= 0) return QMV_EINVAL;
  if (!aligned(gateup, 256) || !aligned(down, 256) || !aligned(ws, 256) || !aligned(x, 16) || !aligned(y, 4))
    return QMV_EALIGN;
  const int sms = num_sms_current_device();
  if (sms <= 0) return QMV_ECUDA;
  Layout L1, L2;
  LayerPlan lp;
  if (!layer_plan((int)fmt, M, N_ff, K_h, sms, &L1, &L2, &lp)) return QMV_EUNSUPPORTED;
  if (ws_bytes < (size_t)lp.total) return QMV_EWORKSPACE;
  unsigned* status = status_ptr();
  if (!status) return QMV_ECUDA;
  uint8_t* w = static_cast<uint8_t*>(ws);
  StreamArgs a1, a2;
  a1.L = L1;
  a1.packed = static_cast<const uint8_t*>(gateup);
  a1.x = x;
  a1.y = reinterpret_cast<float*>(w + lp.off_h);          // h, written as bf16
  a1.ids = nullptr;
  a1.M = M; a1.topk = 1; a1.x_per_pair = 0; a1.swiglu = 1;
  a1.ws = w; a1.ws_bytes = lp.off2;
  a1.status = status;
  apply_plan(&a1, lp.p1);
  a1.num_ctas = lp.grid;
  a2.L = L2;
  a2.packed = static_cast<const uint8_t*>(down);
  a2.x = reinterpret_cast<const uint16_t*>(w + lp.off_h);
  a2.y = y;
  a2.ids = nullptr;
  a2.M = M; a2.topk = 1; a2.x_per_pair = 0; a2.swiglu = 0;
  a2.ws = w + lp.off2; a2.ws_bytes = lp.off_h - lp.off2;
  a2.status = status;
  apply_plan(&a2, lp.p2);
  a2.num_ctas = lp.grid;
  qmv_status st = from_cuda(launch_layer(a1, a2, reinterpret_cast<unsigned*>(w + lp.off_cnt), stream));
  if (st == QMV_OK) g_last_route = (int)fmt * 100 + 12;
  return st;
}

qmv_status qmv_grouped_swiglu(qmv_fmt fmt, const void* tower, const int32_t* expert_ids, const uint16_t* x,
                              float* h, int M, int topk, int64_t N, int64_t K, int64_t E, void* ws,
                              size_t ws_bytes, cudaStream_t stream) {
  if (!valid_fmt(fmt) || !tower || !expert_ids || !x || !h || !ws) return QMV_EINVAL;
  if (M < 1 || M > QMV_MAX_M || topk < 1 || topk > 8 || N <= 0 || K <= 0 || E <= 0) return QMV_EINVAL;
  if (E > (int64_t)1 << 23) return QMV_EUNSUPPORTED;   // ids are packed with a 6-bit pair index
  Layout L;
  if (!make_layout((int)fmt, N, K, 2 * E, &L)) return QMV_EUNSUPPORTED;
  const int64_t experts = (int64_t)M * topk < E ? (int64_t)M * topk : E;
  if (!slab_count_ok(L, 2 * experts)) return QMV_EUNSUPPORTED;
  if (!aligned(tower, 256) || !aligned(ws, 256) || !aligned(x, 16) || !aligned(h, 4) ||
      !aligned(expert_ids, 4))
    return QMV_EALIGN;
  const int sms = num_sms_current_device();
  if (sms <= 0) return QMV_ECUDA;
  const StreamPlan plan = plan_stream_grouped(2 * experts * L.row_tiles * L.k_groups, M, 2, L.k_groups, sms);
  if (ws_bytes < (size_t)plan.ws_bytes) return QMV_EWORKSPACE;
  unsigned* status = status_ptr();
  if (!status) return QMV_ECUDA;
  StreamArgs a;
  a.L = L;
  a.packed = static_cast<const uint8_t*>(tower);
  a.x = x; a.y = h; a.ids = expert_ids;
  a.M = M; a.topk = topk; a.x_per_pair = 0; a.swiglu = 1;
  a.ws = static_cast<uint8_t*>(ws); a.ws_bytes = (int64_t)ws_bytes;
  a.status = status;
  apply_plan(&a, plan);
  int variant = 0;
  qmv_status st = from_cuda(launch_stream(a, stream, &variant));
  if (st == QMV_OK) g_last_route = (int)fmt * 100 + variant;
  return st;
}

qmv_status qmv_gemm_kquant(qmv_fmt fmt, const void* packed_W, const uint16_t* x, float* y, int M, int64_t N,
                           int64_t K, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!valid_fmt(fmt) || !packed_W || !x || !y || !ws || M < 1 || N <= 0 || K <= 0) return QMV_EINVAL;
  if (fmt != QMV_Q4_K && fmt != QMV_Q5_K && fmt != QMV_Q6_K) return QMV_EUNSUPPORTED;
  Layout L;
  if (!make_layout((int)fmt, N, K, 1, &L)) return QMV_EUNSUPPORTED;
  if (!aligned(packed_W, 256) || !aligned(ws, 256) || !aligned(x, 16) || !aligned(y, 4)) return QMV_EALIGN;
  const int sms = num_sms_current_device();
  if (sms <= 0) return QMV_ECUDA;
  const int64_t m_pad = align_up(M, 128);
  if (L.row_tiles * (m_pad / 128) * L.k_groups * (int64_t)sms >= ((int64_t)1 << 31)) return QMV_EUNSUPPORTED;
  if (ws_bytes < (size_t)kq_workspace_bytes(m_pad, K, sms)) return QMV_EWORKSPACE;
  unsigned* status = status_ptr();
  if (!status) return QMV_ECUDA;
  qmv_status st = from_cuda(launch_kq(L, static_cast<const uint8_t*>(packed_W), x, y, M,
                                      static_cast<uint8_t*>(ws), status, stream));
  if (st == QMV_OK) g_last_route = (int)fmt * 100 + 11;
  return st;
}

qmv_status qmv_quant_act_nvfp4(const uint16_t* x, float x_scale, uint8_t* codes, uint8_t* scales, int M,
                               int64_t K, cudaStream_t stream) {
  if (!x || !codes || !scales || M < 1 || K <= 0 || !(x_scale >= 0.0f)) return QMV_EINVAL;
  if (K % 16) return QMV_EUNSUPPORTED;
  if (!aligned(x, 16) || !aligned(codes, 8)) return QMV_EALIGN;
  qmv_status st = from_cuda(launch_quant_act(x, x_scale, codes, scales, M, K, stream));
  if (st == QMV_OK) g_last_route = QMV_NVFP4 * 100 + 8;
  return st;
}

qmv_status qmv_gemm_nvfp4_w4a4(const void* packed_W, const uint16_t* x, float x_scale, float* y, int M,
                               int64_t N, int64_t K, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!packed_W || !x || !y || !ws || M < 1 || N <= 0 || K <= 0 || !(x_scale >= 0.0f)) return QMV_EINVAL;
  if (K % 256) return QMV_EUNSUPPORTED;
  Layout L;
  if (!make_layout(QMV_NVFP4, N, K, 1, &L)) return QMV_EUNSUPPORTED;
  if (!aligned(packed_W, 256) || !aligned(ws, 256) || !aligned(x, 16) || !aligned(y, 16)) return QMV_EALIGN;
  const int64_t m_pad = align_up(M, 128);
  const int sms = num_sms_current_device();
  if (sms <= 0) return QMV_ECUDA;
  if (m_pad / 128 > sms) return QMV_EUNSUPPORTED;       // one CTA group per 128 tokens
  const int64_t planes_bytes = align_up((K / 256) * m_pad * 144, 256);
  if (ws_bytes < (size_t)(planes_bytes + w4a4_partials_bytes(sms))) return QMV_EWORKSPACE;
  unsigned* status = status_ptr();
  if (!status) return QMV_ECUDA;
  uint8_t* planes = static_cast<uint8_t*>(ws);
  uint8_t* partials = planes + planes_bytes;
  qmv_status st = from_cuda(launch_quant_act_tiled(x, x_scale, planes, M, m_pad, K, stream));
  if (st != QMV_OK) return st;
  st = from_cuda(launch_w4a4(L, static_cast<const uint8_t*>(packed_W), planes, partials, x_scale, y, M, m_pad,
                             status, stream));
  if (st == QMV_OK) g_last_route = QMV_NVFP4 * 100 + 4;
  return st;
}

qmv_status qmv_gemv_int8dot(qmv_fmt fmt, const void* packed_W, const uint16_t* x, float* y, int M, int64_t N,
                            int64_t K, void* ws, size_t ws_bytes, cudaStream_t stream) {
  if (!valid_fmt(fmt) || !packed_W || !x || !y || !ws) return QMV_EINVAL;
  if (M < 1 || M > QMV_MAX_M || N <= 0 || K <= 0) return QMV_EINVAL;
  if (fmt != QMV_Q8_0 && fmt != QMV_Q4_K) return QMV_EUNSUPPORTED;
  Layout L;
  if (!make_layout((int)fmt, N, K, 1, &L)) return QMV_EUNSUPPORTED;
  if ((N + 7) / 8 >= ((int64_t)1 << 31)) return QMV_EUNSUPPORTED;
  if (!aligned(packed_W, 256) || !aligned(ws, 256) || !aligned(x, 16) || !aligned(y, 4)) return QMV_EALIGN;
  if (ws_bytes < (size_t)int8dot_workspace_bytes(M, K)) return QMV_EWORKSPACE;
  unsigned* status = status_ptr();
  if (!status) return QMV_ECUDA;
  qmv_status st = from_cuda(launch_int8dot(L, static_cast<const uint8_t*>(packed_W), x, y, M,
                                           static_cast<uint8_t*>(ws), status, stream));
  if (st == QMV_OK) g_last_route = (int)fmt * 100 + 13;
  return st;
}

const char* qmv_status_str(qmv_status s) {
  switch (s) {
    case QMV_OK: return "ok";
    case QMV_EINVAL: return "invalid argument";
    case QMV_EALIGN: return "misaligned pointer";
    case QMV_EUNSUPPORTED: return "unsupported shape or format";
    case QMV_ECUDA: return "CUDA error";
    case QMV_EHEADER: return "packed header does not match the arguments";
    case QMV_ETIMEOUT: return "a bounded device wait timed out";
    case QMV_ERANGE: return "expert id out of range";
    case QMV_EWORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

int qmv_last_route(void) { return g_last_route; }

void qmv_debug_split_k_fault(int mode, uint64_t wait_limit_ns) {
  set_split_fault(mode, (unsigned long long)wait_limit_ns);
}

qmv_status qmv_device_status(int reset) {
  unsigned* p = status_ptr();
  if (!p) return QMV_ECUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return QMV_ECUDA;
  unsigned v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(v)) != cudaSuccess) return QMV_ECUDA;
  if (reset) {
    unsigned z = 0;
    if (cudaMemcpyToSymbol(g_status, &z, sizeof(z)) != cudaSuccess) return QMV_ECUDA;
  }
  if (v & kStatHeader) return QMV_EHEADER;
  if (v & kStatTimeout) return QMV_ETIMEOUT;
  if (v & kStatRange) return QMV_ERANGE;
  return QMV_OK;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// qmv_gemv_noalloc: qmv_gemv with its split-K scratch in the library's own
// device image instead of a caller workspace.
// ---------------------------------------------------------------------------

// The one scratch array all qmv_gemv_noalloc calls on a device share (the partial
// sums of the split-K reduction). 1 MiB covers the need of qmv_gemv up to 256 SMs
// at M = 2..8 (and more SMs at M = 1).
static __device__ __align__(256) unsigned char g_gemv_scratch[QMV_STATIC_SCRATCH_BYTES];

namespace {

std::atomic<uint8_t*> g_scratch_ptr[kMaxDevices];     // as g_status_ptr

// Set-up, once per device, with that device current: the device address of the
// scratch array. The first qmv_gemv_noalloc call on each device runs it.
qmv_status scratch_ptr(uint8_t** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return QMV_ECUDA;
  uint8_t* ptr = g_scratch_ptr[dev].load(std::memory_order_acquire);
  if (ptr == nullptr) {
    if (cudaGetSymbolAddress((void**)&ptr, g_gemv_scratch) != cudaSuccess) return QMV_ECUDA;
    g_scratch_ptr[dev].store(ptr, std::memory_order_release);
  }
  *out = ptr;
  return QMV_OK;
}

}  // namespace

extern "C" qmv_status qmv_gemv_noalloc(qmv_fmt fmt, const void* packed_W, const uint16_t* x, float* y,
                                       int M, int64_t N, int64_t K, cudaStream_t stream) {
  if (!valid_fmt(fmt) || !packed_W || !x || !y) return QMV_EINVAL;
  if (M < 1 || M > QMV_MAX_M || N <= 0 || K <= 0) return QMV_EINVAL;
  Layout L;
  if (!make_layout((int)fmt, N, K, 1, &L) || !slab_count_ok(L, 1)) return QMV_EUNSUPPORTED;
  if (!aligned(packed_W, 256) || !aligned(x, 16) || !aligned(y, 4)) return QMV_EALIGN;
  const int sms = num_sms_current_device();
  if (sms <= 0) return QMV_ECUDA;
  // the plan of qmv_gemv: the same cells, and so the same order of the sums, whose
  // results this entry reproduces bit for bit
  const StreamPlan plan = plan_stream_dense(L.row_tiles * L.k_groups, M, 1, sms);
  if ((size_t)plan.ws_bytes > (size_t)QMV_STATIC_SCRATCH_BYTES) return QMV_EWORKSPACE;
  uint8_t* scratch = nullptr;
  qmv_status st = scratch_ptr(&scratch);
  if (st != QMV_OK) return st;
  unsigned* status = status_ptr();
  if (!status) return QMV_ECUDA;
  // The array keeps whatever the previous call left; the partial-sum words must
  // start at zero (a successful call leaves them zero, a failed one may not).
  st = from_cuda(cudaMemsetAsync(scratch, 0, (size_t)plan.ws_bytes, stream));
  if (st != QMV_OK) return st;
  StreamArgs a;
  a.L = L;
  a.packed = static_cast<const uint8_t*>(packed_W);
  a.x = x; a.y = y; a.ids = nullptr;
  a.M = M; a.topk = 1; a.x_per_pair = 0; a.swiglu = 0;
  a.ws = scratch; a.ws_bytes = (int64_t)QMV_STATIC_SCRATCH_BYTES;
  a.status = status;
  apply_plan(&a, plan);
  int variant = 0;
  st = from_cuda(launch_stream(a, stream, &variant));
  if (st == QMV_OK) g_last_route = (int)fmt * 100 + variant;
  return st;
}
