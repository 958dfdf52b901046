// qmv_internal.h -- host-side launchers shared between the library's translation units.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>
#include "qmv_layout.cuh"

namespace qmv {

// device status bits (latched with atomicOr into the per-device status word)
constexpr unsigned kStatHeader = 1u;
constexpr unsigned kStatTimeout = 2u;
constexpr unsigned kStatRange = 4u;

// Arguments of the streaming GEMV kernel (dense and grouped forms).
struct StreamArgs {
  Layout L;
  const uint8_t* packed;     // packed buffer (header at offset 0)
  const uint16_t* x;         // bf16 activations
  float* y;                  // fp32 outputs
  const int32_t* ids;        // grouped: expert ids [M][topk]; dense: nullptr
  int M;                     // tokens (rows of x for dense)
  int topk;                  // grouped: slots per token; dense: 1
  int x_per_pair;            // grouped: 1 if x has one row per (token, slot)
  int swiglu;                // 1: fused gate|up over a 2-expert tower, y = silu(gate.x) * (up.x)
  uint8_t* ws;               // workspace: per-CTA partial sums (zero between calls)
  int64_t ws_bytes;
  unsigned* status;          // per-device status word
  int num_ctas;              // persistent grid size
  int cells;                 // dense: cells of the accumulation order (> 0); grouped: 0
  int cpc;                   // dense: cells per CTA (1 or 2)
  int gp;                    // grouped: slabs per cell
  int maxslots;              // workspace slots (published pieces) per CTA
};

// Grid, accumulation cells and workspace of one stream-kernel call (host side),
// shared by the entry points and the workspace size query.
//  - dense: V cells, a function of the matrix and the SM count only, so that every M
//    (and the no-workspace entry) adds in the same order: V = min(2 x SMs, slabs) for
//    long calls (16 slabs per SM or more; two CTAs per SM), else min(SMs, slabs) (one
//    CTA per SM, so the next call's CTAs fit beside it); one cell per CTA;
//  - grouped: each unit cut into cells of gp k-groups (4, 2 or 1: a function of K
//    only), whatever the routing; CTAs take whole cells, at most two CTAs per SM.
// passes: 1, or 2 for the fused gate|up (gate and up sums).
struct StreamPlan {
  int grid, cells, cpc, gp, maxslots;
  int64_t ws_bytes;          // split-K workspace (published pieces), 256-byte multiple
};
StreamPlan plan_stream_dense(int64_t slabs, int M, int passes, int sms);
StreamPlan plan_stream_grouped(int64_t slabs_max, int M, int passes, int64_t k_groups, int sms);
// Test hook of the reduction (see qmv_debug_split_k_fault in qmv.h): mode 1, peers
// publish nothing and reducers wait peer_wait_ns, then latch QMV_ETIMEOUT; mode 2,
// reducers latch QMV_ETIMEOUT at once and leave the peers' pieces in the workspace;
// mode 0 restores normal operation.
void set_split_fault(int mode, unsigned long long peer_wait_ns);

int num_sms_current_device();

// The streaming kernel numbers its slabs (segment, row tile, k-group) with 32-bit
// integers: segments x row tiles x k-groups must stay below 2^31.
inline bool slab_count_ok(const Layout& L, int64_t segments) {
  return segments * L.row_tiles * L.k_groups < ((int64_t)1 << 31);
}

cudaError_t launch_pack(const Layout& L, const uint8_t* canon, uint8_t* dst, cudaStream_t s);
cudaError_t launch_dequant(const Layout& L, const uint8_t* packed, int64_t row0, int64_t rows,
                           float* out, unsigned* status, cudaStream_t s);
cudaError_t launch_quantize(int fmt, const float* W, int64_t rows, int64_t K, float ts,
                            uint8_t* canon, cudaStream_t s);
// the codebook formats: IQ4_XS's 16 int8 entries (passed to the kernel by value),
// or the grid of IQ3_S / IQ2_S (host bytes, copied to the front of canon first)
struct Codebook16 { int8_t v[16]; };
cudaError_t launch_quantize_codebook(int fmt, const float* W, int64_t rows, int64_t K, const uint8_t* codebook,
                                     uint8_t* canon, cudaStream_t s);
cudaError_t launch_quant_act(const uint16_t* x, float xs, uint8_t* codes, uint8_t* scales, int M,
                             int64_t K, cudaStream_t s);
// NVFP4 activation quantizer into the W4A4 GEMM's tiled activation planes
cudaError_t launch_quant_act_tiled(const uint16_t* x, float xs, uint8_t* planes, int M, int64_t m_pad, int64_t K,
                                   cudaStream_t s);
// W4A4 block-scaled GEMM (tcgen05): y[M][N] = x_scale * s_T * (x codes . W codes) with
// the activation planes written by launch_quant_act_tiled
cudaError_t launch_w4a4(const Layout& L, const uint8_t* packed, const uint8_t* act_planes, uint8_t* partials,
                        float x_scale, float* y, int M, int64_t m_pad, unsigned* status, cudaStream_t s);
// bytes of the W4A4 split-K region (partial-sum slots, then flags) for a device of `sms` SMs
int64_t w4a4_partials_bytes(int sms);
// K-quant (Q4_K) prefill GEMM (tcgen05, f16 operands): the x pre-pass, then the GEMM.
// ws: [x tiles: m_pad*K*2][sum tiles: m_tiles*(K/256)*4096][partial tiles: sms*64 KB][flags]
cudaError_t launch_kq(const Layout& L, const uint8_t* packed, const uint16_t* x, float* y, int M, uint8_t* ws,
                      unsigned* status, cudaStream_t s);
int64_t kq_workspace_bytes(int64_t m_pad, int64_t K, int sms);
// int8-dot GEMV (Q8_0, Q4_K; M <= 8): x quantized to int8 per 32 values into ws, then
// one warp per weight row with dp4a. ws: [codes: M*K, 256-aligned][scales: M*(K/32)*4]
cudaError_t launch_int8dot(const Layout& L, const uint8_t* packed, const uint16_t* x, float* y, int M, uint8_t* ws,
                           unsigned* status, cudaStream_t s);
int64_t int8dot_workspace_bytes(int M, int64_t K);
// returns the route variant launched (1 = M=1, 2 = M>1, 3 = grouped, 9 = fused gate|up SwiGLU)
cudaError_t launch_stream(const StreamArgs& a, cudaStream_t s, int* variant);
// The MLP layer in one launch (layer_kernel): a1 = the fused gate|up pass (its y = h,
// written as bf16), a2 = the down pass over h; both with the same num_ctas. counter:
// a workspace word the CTAs count their arrivals on between the phases.
cudaError_t launch_layer(const StreamArgs& a1, const StreamArgs& a2, unsigned* counter, cudaStream_t s);

}  // namespace qmv
