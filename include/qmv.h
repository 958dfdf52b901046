/*
 * qmv.h -- C ABI of libqmv: decode-time matmul y[M,N] = x[M,K] . W[N,K]^T with W
 * kept in a packed block-quantized format and decoded on the fly inside the
 * kernel, on one NVIDIA GB300 (sm_103a).
 *
 * The operation is the keep-quant matmul seam Y = X . W^T with a quantized W,
 * over one matrix (E = 1) or a stacked expert tower weight[E*N, K]
 * ("feat(BACKEND-TENSTORRENT-KEEPQUANT): the 27B arm — on-core decode residency,
 * TT grouped keep-quant GEMM, e2e gate", scope item 2 and the "Re-anchor" comment).
 * Formats: GGUF-style Q8_0 / Q4_K / Q6_K keep-quant blocks (same issue, artifact
 * table and "Budget on the 32 GB P150"), Q5_K (the 5-bit member named with them in
 * scope item 1 and owed by the grouped kernel in the "Re-anchor" comment), and NVFP4
 * E2M1 codes with E4M3 block scales plus row-scaled FP8 ("I Built a Custom
 * Blackwell Kernel for Qwen3.8-27B", "What the custom path actually does").
 *
 * Conventions for every entry point:
 *  - Ownership: the caller allocates and owns every buffer. The library never
 *    allocates or frees memory, never synchronizes a stream, and never reads
 *    device data on the host. All work is enqueued on `stream`.
 *  - Pointers marked "device" must be device memory of the current device.
 *    packed buffers and workspaces must be 256-byte aligned; x and y 16-byte
 *    aligned.
 *  - Errors: arguments are validated on the host before anything is launched;
 *    a failed check returns its status and launches nothing. A launch failure
 *    returns QMV_ECUDA. Faults detected on the device (a packed header that does
 *    not match the arguments, an expert id out of range, a pipeline wait that
 *    timed out) are latched in a per-device status word that
 *    qmv_device_status() reads; the kernel then skips its work.
 *  - Numerics: weights are decoded exactly (see qmv_dequant); products with the
 *    bf16 activations are exact in fp32 and accumulate in fp32. NVFP4 and FP8_ROW
 *    take x as f16 (exact for 2^-14 <= |x| <= 65504); the Q4_K decoders scale
 *    x by 2^63 or 2^67 (exact for |x| < 2^61, products normal for
 *    |x| >= 2^-60), the Q6_K decoders by 2^63 .. 2^71 (exact for |x| < 2^56);
 *    the other K-quant paths take bf16 x as it is.
 *
 * Canonical byte layouts (the input of qmv_pack and output of qmv_quantize):
 *   Q8_0  34 B per 32 values : fp16 d | 32 x int8 q;           w = d * q
 *   Q4_K 144 B per 256 values: fp16 d | fp16 dmin | 12 B scales | 128 B nibbles
 *         scales: 96-bit little-endian bitstream of sixteen 6-bit fields, fields
 *         0..7 = sc_j, 8..15 = m_j for the eight 32-value sub-blocks; nibble byte b
 *         holds element 2b (low) and 2b+1 (high);   w = (d * sc_j) * q - dmin * m_j
 *   Q5_K 176 B per 256 values: fp16 d | fp16 dmin | 12 B scales | 32 B qh | 128 B nibbles
 *         header and nibbles exactly as Q4_K (low 4 bits of q); qh bit e (byte e/8,
 *         bit e%8) = bit 4 of element e; q = 0..31; w = (d * sc_j) * q - dmin * m_j
 *         (the pages print no byte layout for Q5_K: this is the Q4_K reading plus
 *         one bit plane)
 *   Q6_K 210 B per 256 values: 128 B ql | 64 B qh | 16 x int8 sc | fp16 d
 *         q = ql nibble | (qh 2 bits << 4); ql byte b holds elements 2b, 2b+1;
 *         qh byte b holds elements 4b..4b+3 at bits 0,2,4,6; w = (d * sc_j) * (q - 32)
 *   NVFP4 per matrix: E2M1 codes [N][K/2] (element 2i = low nibble of byte i) |
 *         E4M3 scales [N][K/16] | fp32 tensor scale s_T; w = (e2m1 * e4m3) * s_T
 *   FP8_ROW per matrix: E4M3 codes [N][K] | fp32 row scales [N];  w = e4m3 * s_n
 *   A tower of E experts is E such matrices back to back.
 */
#ifndef QMV_H
#define QMV_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QMV_Q8_0 = 1,
    QMV_Q4_K = 2,
    QMV_Q6_K = 3,
    QMV_NVFP4 = 4,
    QMV_FP8_ROW = 5,
    QMV_Q5_K = 6,
    QMV_IQ4_XS = 7,        /* codebook format: 136 B / 256 values, a per-matrix 16-entry
                              int8 codebook at the end of each matrix's canonical stream
                              ("A 320B MoE on a free Kaggle TPU", "What '3-bit' costs,
                              measured") */
    QMV_IQ3_S = 8,         /* grid formats (same article and section; "The kernel, and
                              why 64 tok/s is not a bandwidth number"): 110 / 82 B per 256
                              values; groups of 4 / 8 weights are entries of the format's */
    QMV_IQ2_S = 9          /* grid (512 x 4 / 1024 x 8 uint8 magnitudes, at the front of a
                              tower's canonical stream) with one sign bit per weight */
} qmv_fmt;

typedef enum {
    QMV_OK = 0,
    QMV_EINVAL = 1,        /* bad argument (null pointer, size, M out of range, ...) */
    QMV_EALIGN = 2,        /* a pointer is not aligned as required */
    QMV_EUNSUPPORTED = 3,  /* valid request this build does not serve (K not a multiple of
                              the lane granule, format not allowed on this entry point) */
    QMV_ECUDA = 4,         /* a CUDA runtime call or kernel launch failed */
    QMV_EHEADER = 5,       /* device status: packed header does not match the arguments */
    QMV_ETIMEOUT = 6,      /* device status: a bounded pipeline wait ran out */
    QMV_ERANGE = 7,        /* device status: an expert id was outside [0, E), or one expert
                              got more than 8 rows of x (ids repeated within a token) */
    QMV_EWORKSPACE = 8     /* workspace too small for this call */
} qmv_status;

/* Entry ids for qmv_workspace_size. */
enum {
  QMV_ENTRY_GEMV = 1,
  QMV_ENTRY_GROUPED = 2,
  QMV_ENTRY_W4A4 = 3,
  QMV_ENTRY_SWIGLU = 4,
  QMV_ENTRY_GROUPED_SWIGLU = 5,
  QMV_ENTRY_KQUANT = 6,
  QMV_ENTRY_MLP_LAYER = 7,
  QMV_ENTRY_INT8DOT = 8
};

/* Largest decode batch served by qmv_gemv / qmv_grouped (M rows of x). */
#define QMV_MAX_M 8

/* Bytes of the canonical stream of an E-expert tower of [N, K] matrices (IQ3_S and
 * IQ2_S: the grid once, then the blocks of all E*N rows).
 * Returns 0 for an unknown format or a K that is not a multiple of the block. */
size_t qmv_canon_size(qmv_fmt fmt, int64_t N, int64_t K, int64_t E);

/* Bytes of the device ("packed") layout, header included. The packed layout
 * regroups each matrix into slabs of 128 rows x 256 values whose fields sit in
 * 16-byte planes, so one bulk copy moves a slab and every lane's 128-bit load
 * is aligned; rows are padded to a multiple of 128 with zero blocks. The slab
 * bytes are the canonical bytes, only reordered (the per-value cost is
 * unchanged). K must be a multiple of 32 (Q8_0, NVFP4, FP8_ROW) or 256 (Q4_K,
 * Q5_K, Q6_K and the codebook formats). Returns 0 if unsupported. IQ4_XS repeats its
 * 16-byte codebook after the scale fields of every 128-row tile of every k-group
 * (16 B per slab, so that each slab copy brings it along); IQ3_S and IQ2_S store
 * their grid once, as f16 values, after the header (4 / 16 KiB). */
size_t qmv_pack_size(qmv_fmt fmt, int64_t N, int64_t K, int64_t E);

/* Repack canonical bytes into the device layout. Defined by: the stacked keep-quant
 * tower loader whose packed residency the grouped kernel consumes, loaded once
 * ("feat(BACKEND-TENSTORRENT-KEEPQUANT): the 27B arm — on-core decode residency, TT
 * grouped keep-quant GEMM, e2e gate", Scope item 2: load-phase streaming, experts
 * packed and fully resident), laid out as dense planes with the row on the lane axis
 * ("A 320B MoE on a free Kaggle TPU", "The 110 GB claim, checked against the tensor
 * index"). canon: device, qmv_canon_size bytes (the canonical stream of a whole
 * tower; NVFP4 carries its per-matrix tensor scale inside it, FP8_ROW its row
 * scales, IQ4_XS its codebook). dst: device, qmv_pack_size bytes, 256-B aligned; fully overwritten
 * (header, slabs, padding). One-time load-phase work, not part of the per-token
 * path. */
qmv_status qmv_pack(qmv_fmt fmt, const void* canon, int64_t N, int64_t K, int64_t E,
                    void* dst, cudaStream_t stream);

/* Encode fp32 W[rows, K] (device, row-major) into canonical bytes (device,
 * qmv_canon_size(fmt, rows, K, 1) bytes) with the round-to-nearest quantizers
 * used for synthetic data. Defined by: quantizing on the host side of the load path,
 * one tensor at a time, from the original weights ("Qwen3.8-27B on one Tenstorrent
 * P150", "2. Building the 27B quant"); plain rounding, not the error-compensated
 * variant of its section 8. tensor_scale is the NVFP4 per-tensor scale s_T (a given
 * constant); ignored for other formats. IQ4_XS returns QMV_EUNSUPPORTED: its
 * encoding needs a codebook, which is an input of the format, not a rounding rule.
 * Not on the per-token path. */
qmv_status qmv_quantize(qmv_fmt fmt, const float* W, int64_t rows, int64_t K,
                        float tensor_scale, void* canon, cudaStream_t stream);

/* The encoder of the codebook formats: as qmv_quantize, with the format's table (a
 * host pointer, read during the call) in place of a rounding constant ("A 320B MoE
 * on a free Kaggle TPU", "What '3-bit' costs, measured": a weight is an entry of
 * the format's codebook). IQ4_XS: the matrix's 16 int8 values; per 32-value
 * sub-block the scale that maps its element of largest magnitude onto the entry of
 * largest magnitude, 6 bits under an fp16 d; each element takes the nearest entry;
 * canon = the blocks, then the codebook. IQ3_S / IQ2_S: the grid, 512 x 4 / 1024 x 8
 * uint8 magnitudes; per 32 / 16 values an odd 4-bit scale (2 sc + 1) under fp16 d
 * sized by the grid's largest magnitude; per group the signs of its weights and
 * the nearest entry in squared error; canon = the grid, then the blocks (encode a
 * whole tower as one [E*N, K] matrix). canon: device, qmv_canon_size(fmt, rows, K, 1)
 * bytes. Other formats: QMV_EUNSUPPORTED. Not on the per-token path. */
qmv_status qmv_quantize_codebook(qmv_fmt fmt, const float* W, int64_t rows, int64_t K,
                                 const void* codebook, void* canon, cudaStream_t stream);

/* BlockToFloat on the device layout: W_out[r][k] (fp32, device) for rows
 * row0 .. row0+rows-1 of the stacked tower (row = e*N + n). Defined by: the CPU
 * BlockToFloat that the on-core word-shadow decode is held bit-exact against
 * ("feat(BACKEND-TENSTORRENT-KEEPQUANT) ...", the W4 residency paragraph). Bit-exact
 * with the canonical decode formulas above, in that op order. Used to check the
 * layout. N, E and row0 are this library's additions (a window of a tower). */
qmv_status qmv_dequant(qmv_fmt fmt, const void* packed, int64_t N, int64_t K, int64_t E,
                       int64_t row0, int64_t rows, float* W_out, cudaStream_t stream);

/* Workspace bytes needed by an entry point for these sizes (host-only query; it
 * reads the SM count of the current device). This library's own call (the pages
 * stage nothing per call: "feat(BACKEND-TENSTORRENT-KEEPQUANT) ...", Scope item 1,
 * capture-safety -- every buffer is sized and allocated before capture, and replay
 * allocates nothing); E and topk size the grouped entries. The workspace must be zero-filled
 * once before its first use. It holds the partial sums of row tiles split
 * between CTAs (a zero word means "not yet written"); a call that returns
 * without a device status error leaves the whole workspace zero again, so the
 * same workspace serves the next call as is. After a device status error,
 * zero-fill it again. Calls sharing one workspace must not overlap. */
size_t qmv_workspace_size(int entry, qmv_fmt fmt, int M, int64_t N, int64_t K, int64_t E,
                          int topk);

/* Decode GEMV, M = 1..8: y[m][n] = sum_k W[n][k] * x[m][k]. Defined by: the dense
 * keep-quant matmul Y = X . W^T whose kernel decodes the packed weight words per call
 * ("feat(BACKEND-TENSTORRENT-KEEPQUANT) ...", Scope item 1, MatmulBTQuantKernel; the
 * "Re-anchor" comment: E = 1 covers dense), the M = 2..8 rows being the verify block
 * of speculative decoding ("Qwen3.8-27B on one Tenstorrent P150", "5. DFlash2 on
 * Blackhole"). Every row of an M-row call equals the one-row call on that row bit
 * for bit: the order of the fp32 sums depends on (N, K) and the SM count only.
 * packed_W: device layout of one [N, K] matrix (E = 1). x: device bf16 [M][K]
 * (raw bits, row-major). y: device fp32 [M][N], fully overwritten. ws: device,
 * qmv_workspace_size(QMV_ENTRY_GEMV, ...) bytes. The weights are streamed from
 * HBM once per call for all M rows. */
qmv_status qmv_gemv(qmv_fmt fmt, const void* packed_W, const uint16_t* x, float* y, int M,
                    int64_t N, int64_t K, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Bytes of the device scratch array built into the library for qmv_gemv_noalloc. */
#define QMV_STATIC_SCRATCH_BYTES (4u << 20)

/* qmv_gemv without a workspace argument; it allocates nothing. The pages have no
 * counterpart: it is a library convenience. It serves callers that cannot hand
 * over device memory per call -- an engine whose allocator has already reserved
 * the device for its own pool, or a plugin interface that passes only input and
 * output pointers -- and that must not call cudaMalloc/cudaFree on the decode
 * path, since those can fail under a full pool or synchronize the device.
 * The split-K partial sums live instead in one fixed array of
 * QMV_STATIC_SCRATCH_BYTES in the library's device image.
 * Set-up: the first call on each device (with that device current) looks up the
 * array's device address; make that first call before any stream capture.
 * Every call on a device shares the one array, which keeps what the last call
 * left: each call first clears the words it uses on `stream` (cudaMemsetAsync, no
 * allocation). Calls that overlap in time (on other streams or host threads)
 * race on the array; the caller must serialize them.
 * It runs qmv_gemv's grid and adds up in the same cells and order, so its results
 * equal qmv_gemv's bit for bit. Its partial sums take one 128 x c x 4-byte record
 * per cell of the slab sequence (at most 2 cells per SM; c = 1 at M = 1, else 8;
 * rounded up to 256): at most 8 KiB per SM, 1,245,184 bytes on a 152-SM GB300.
 * Returns QMV_EWORKSPACE
 * when that exceeds QMV_STATIC_SCRATCH_BYTES (M = 2..8 on a device of more than 512
 * SMs). Otherwise arguments, results and errors as qmv_gemv. */
qmv_status qmv_gemv_noalloc(qmv_fmt fmt, const void* packed_W, const uint16_t* x, float* y,
                            int M, int64_t N, int64_t K, cudaStream_t stream);

/* Grouped per-expert GEMV over a stacked tower of E experts.
 * expert_ids: device int32 [M][topk] (ids within a token distinct; never read
 * on the host). x: device bf16, [M][K] if x_per_pair == 0 (every slot of a
 * token uses its row) or [M*topk][K] if x_per_pair == 1 (one row per (token,
 * slot)). y: device fp32 [M][topk][N], fully overwritten:
 *   y[t][j][:] = W_{expert_ids[t][j]} . x_row(t, j).
 * Each distinct routed expert's rows are streamed once per call, for every row
 * of x routed to it ("A 320B MoE on a free Kaggle TPU", "The decode kernel's
 * cost is not 'distinct experts'"). M = 1..8, topk = 1..8. */
qmv_status qmv_grouped(qmv_fmt fmt, const void* tower, const int32_t* expert_ids,
                       const uint16_t* x, int x_per_pair, float* y, int M, int topk,
                       int64_t N, int64_t K, int64_t E, void* ws, size_t ws_bytes,
                       cudaStream_t stream);

/* Fused gate|up decode GEMV with the SwiGLU epilogue, M = 1..8:
 *   h[m][n] = silu(g) * u,  g = sum_k Wg[n][k] x[m][k],  u = sum_k Wu[n][k] x[m][k],
 *   silu(g) = g / (1 + exp(-g)),
 * one pass over the two matrices that share x: the MLP's gate/up projection read as
 * one, with the SwiGLU fused behind it ("Qwen3.8-27B on one Tenstorrent P150",
 * "4. Measuring the ceiling, and lots of dead ends"). tower: the device layout of a 2-expert tower,
 * gate = expert 0, up = expert 1 (qmv_pack with E = 2). x: device bf16 [M][K].
 * h: device fp32 [M][N], fully overwritten. ws: device,
 * qmv_workspace_size(QMV_ENTRY_SWIGLU, ...) bytes, zero-filled once (as for
 * qmv_gemv). Each gate and up row is streamed from HBM once per call. */
qmv_status qmv_gemv_swiglu(qmv_fmt fmt, const void* tower, const uint16_t* x, float* h, int M,
                           int64_t N, int64_t K, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Grouped fused gate|up with the SwiGLU epilogue: the routed experts' first MLP
 * projection in one call, M = 1..8, topk = 1..8:
 *   h[t][j][n] = silu(g) * u,  g = W_{e} . x[t],  u = W_{E+e} . x[t],  e = expert_ids[t][j],
 * the union of qmv_grouped (each distinct routed expert streamed once per call)
 * and qmv_gemv_swiglu (gate and up read in one pass, SwiGLU in the epilogue).
 * tower: the device layout of a 2E-expert tower (qmv_pack with 2E experts): the E
 * gate matrices first (expert e), then the E up matrices (expert E + e).
 * expert_ids: device int32 [M][topk] in 0..E-1, distinct within a token (an id
 * outside that range latches QMV_ERANGE in the device status and writes nothing). x: device bf16
 * [M][K]. h: device fp32 [M][topk][N], fully overwritten. ws: device,
 * qmv_workspace_size(QMV_ENTRY_GROUPED_SWIGLU, ...) bytes, zero-filled once (as
 * for qmv_gemv). E <= 2^23. */
/* The dense MLP layer in one launch: h = silu(x W_gate^T) * (x W_up^T) (as
 * qmv_gemv_swiglu), rounded to bf16, then y = h W_down^T (as qmv_gemv over the bf16
 * h). Defined by the matmul seam applied twice around the SwiGLU ("Qwen3.8-27B on one
 * Tenstorrent P150", "4. Measuring the ceiling, and lots of dead ends": the fused
 * gate/up and down of the decode MLP) and the joined gate|up projection ("I Built a
 * Custom Blackwell Kernel for Qwen3.8-27B", "What the custom path actually does").
 * One kernel: its CTAs run the gate|up pass, store their rows of h in the workspace
 * and arrive on a counter there; each CTA copies its first down-projection weights
 * at once and waits (bounded: QMV_ETIMEOUT) for every CTA's arrival before it reads
 * h. The results equal qmv_gemv_swiglu, a bf16 round-to-nearest-even of h, then
 * qmv_gemv, bit for bit (the same cells in both passes). gateup: the packed tower of
 * 2 matrices [N_ff, K_h] (gate, then up; as qmv_gemv_swiglu). down: the packed
 * [K_h, N_ff] matrix. Both of format fmt. x: device bf16 [M][K_h], 16-byte aligned.
 * y: device fp32 [M][K_h], fully overwritten. M = 1..8. ws: device,
 * qmv_workspace_size(QMV_ENTRY_MLP_LAYER, fmt, M, N_ff, K_h, 1, 1) bytes, 256-byte
 * aligned, zero-filled once: the two passes' partial sums (zero again after every
 * successful call), h, and the arrival counter (which counts on across calls; zero-
 * fill the workspace again after a status error). Calls sharing a workspace must
 * not overlap. */
qmv_status qmv_mlp_layer(qmv_fmt fmt, const void* gateup, const void* down, const uint16_t* x, float* y,
                         int M, int64_t N_ff, int64_t K_h, void* ws, size_t ws_bytes, cudaStream_t stream);

qmv_status qmv_grouped_swiglu(qmv_fmt fmt, const void* tower, const int32_t* expert_ids,
                              const uint16_t* x, float* h, int M, int topk, int64_t N, int64_t K,
                              int64_t E, void* ws, size_t ws_bytes, cudaStream_t stream);

/* NVFP4 activation quantizer (W4A4 prefill: "I Built a Custom Blackwell Kernel for
 * Qwen3.8-27B", "What the custom path actually does", quantising the activation into
 * Blackwell's FP4 format with a static input scale): per 16-value block of bf16 x[M][K],
 * s_b = e4m3_rne_sat(amax_b / (6 x_scale)); codes = e2m1_rne_sat(x / (s_b x_scale)),
 * zero when s_b is zero. x_scale: the static per-site activation scale.
 * codes: device [M][K/2] (element 2i in the low nibble); scales: device [M][K/16]. */
qmv_status qmv_quant_act_nvfp4(const uint16_t* x, float x_scale, uint8_t* codes,
                               uint8_t* scales, int M, int64_t K, cudaStream_t stream);

/* NVFP4 W4A4 prefill GEMM: the activation is quantized to NVFP4 (as
 * qmv_quant_act_nvfp4) into ws, then a tcgen05 block-scaled MMA computes
 * y[m][n] = x_scale * s_T * sum_b s_b(x) s_b(W) sum_i e2m1(x) e2m1(W)
 * in fp32 ("I Built a Custom Blackwell Kernel", "What the custom path actually
 * does": W4A4 tensor-core kernels after quantising the activation).
 * The MMA is tcgen05.mma kind::mxf4nvf4.block_scale (E2M1 x E2M1, UE4M3 scale per
 * 16 values, fp32 accumulator in tensor memory), reading the packed weight tiles
 * as they are. packed_W: device layout of one NVFP4 [N, K] matrix; K a multiple
 * of 256. M: 1 .. 128 x (number of SMs), meant for prefill (M >= 128); larger M
 * returns QMV_EUNSUPPORTED (split the tokens into calls). ws: device,
 * qmv_workspace_size(QMV_ENTRY_W4A4, QMV_NVFP4, M, N, K, 1, 1) bytes: the
 * activation's NVFP4 tiles (rewritten by every call), then one slot of split-K
 * partial sums and one publication flag per SM. As for qmv_gemv, zero-fill the
 * workspace once; a call that returns without a device status error leaves every
 * flag zero again. Calls sharing a workspace must not overlap.
 * y: device fp32 [M][N], 16-byte aligned, fully overwritten. */
qmv_status qmv_gemm_nvfp4_w4a4(const void* packed_W, const uint16_t* x, float x_scale,
                               float* y, int M, int64_t N, int64_t K, void* ws,
                               size_t ws_bytes, cudaStream_t stream);

/* K-quant prefill GEMM on the 5th-generation tensor cores, for M in the hundreds to
 * thousands of tokens: y[m][n] = sum_k x[m][k] BlockToFloat(W)[n][k], each weight
 * superblock streamed from HBM once per call rather than once per 8 tokens (the
 * re-streaming prefill bug: "Qwen3.8-27B on one Tenstorrent P150", "3. Porting the 9B
 * stack to 27B geometry", its prefill fixes). fmt: QMV_Q4_K, QMV_Q5_K or QMV_Q6_K (others
 * return QMV_EUNSUPPORTED). Per superblock,
 * tcgen05.mma kind::f16 forms sum_k (sc_j q) x and sum_j m_j xsum_j in fp32 tensor memory
 * (sc_j q <= 1953 and m_j exact in f16; x in f16, exact for |x| in [2^-14, 65504]; xsum_j = the
 * fp32 sum of x over the 32-value sub-block, as two f16 terms, so |xsum_j| < 65504),
 * and y gathers d 2^14 and dmin times them in fp32. Q6_K: sc_u (q - 32) can need 12
 * significant bits, so the int8 scale is split, sc_u = 16 sh_u + sl_u, and each K step
 * takes two MMAs, (q - 32) 16 sh_u and (q - 32) sl_u (both exact in f16); y gathers d
 * times the sum. packed_W: the device layout of one
 * Q4_K, Q5_K or Q6_K [N, K] matrix (qmv_pack); K a multiple of 256; any N and M >= 1. x: device bf16
 * [M][K], 16-byte aligned. y: device fp32 [M][N], fully overwritten. ws: device,
 * qmv_workspace_size(QMV_ENTRY_KQUANT, fmt, M, N, K, 1, 1) bytes: x's f16 tiles and
 * sub-block sums (rewritten by every call), one 64 KB slot of split-K partial sums and
 * one publication flag per SM. Zero-fill the workspace once; a call that returns without
 * a device status error leaves every flag zero again. Calls sharing a workspace must not
 * overlap. Launches two kernels (the x pre-pass, then the GEMM). */
qmv_status qmv_gemm_kquant(qmv_fmt fmt, const void* packed_W, const uint16_t* x, float* y, int M,
                           int64_t N, int64_t K, void* ws, size_t ws_bytes, cudaStream_t stream);

/* The int8-dot decode GEMV (the lever the keep-quant issue books as the repayment of
 * its slow decode: "feat(BACKEND-TENSTORRENT-KEEPQUANT) ...", "Scope", its "Out of
 * scope" line and the accepted-cost note). x is quantized to int8 per 32-value block,
 * d = amax / 127 (fp32, round to nearest) and q = clamp(rint(x / d), -127, 127), all
 * zero when d = 0; then y[m][n] = sum over blocks of the weight block's scale(s) times d
 * times the int32 dot of the weight codes with q (Q4_K: d sc_j dx sum(q x_q) -
 * dmin m_j dx sum(x_q)), the products in int32 (dp4a), the rest in fp32. The result
 * is the GEMV of the quantized x, not of x: it differs from qmv_gemv by x's int8
 * rounding (up to d/2 per value). fmt: QMV_Q8_0 or QMV_Q4_K (others return
 * QMV_EUNSUPPORTED). packed_W: the device layout of one [N, K] matrix (qmv_pack).
 * x: device bf16 [M][K], 16-byte aligned, M = 1 .. QMV_MAX_M. y: device fp32 [M][N],
 * fully overwritten. ws: device, qmv_workspace_size(QMV_ENTRY_INT8DOT, fmt, M, N, K,
 * 1, 1) bytes, 256-byte aligned: x's int8 codes [M][K], then the block scales
 * [M][K/32] (fp32), both rewritten by every call, so no zero-fill is needed; calls
 * sharing a workspace must not overlap. Launches two kernels (the quantizer, then the
 * GEMV, chained by programmatic dependent launch); a header that disagrees with the
 * arguments latches QMV_EHEADER in the device status and leaves y unwritten. */
qmv_status qmv_gemv_int8dot(qmv_fmt fmt, const void* packed_W, const uint16_t* x, float* y, int M,
                            int64_t N, int64_t K, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Human-readable name of a status. */
const char* qmv_status_str(qmv_status s);

/* Route id of the kernel the last successful call on this host thread launched:
 * format * 100 + variant (1 = M=1 streaming CUDA-core GEMV, 2 = M>1 streaming
 * mma.sync GEMV, 3 = grouped, 4 = W4A4 tcgen05, 5 = dequant, 6 = pack,
 * 7 = quantize, 8 = activation quantizer, 9 = fused gate|up SwiGLU, 11 = K-quant
 * prefill, 12 = MLP layer, 13 = int8-dot GEMV). Test hook. */
int qmv_last_route(void);

/* Test hook for the split-K reduction of qmv_gemv, qmv_grouped and their SwiGLU and
 * no-workspace forms; it changes the launches made after it, from any host thread
 * (a process-wide setting, not thread-safe; for tests only).
 *   mode 1: peers publish no partial sums, so every reducer that needs one waits
 *           wait_limit_ns (0: one second), then latches QMV_ETIMEOUT in the device
 *           status word, skips its outputs and exits;
 *   mode 2: reducers latch QMV_ETIMEOUT and exit without reading their peers'
 *           partial sums, which stay in the workspace (or the built-in scratch);
 *   mode 0: normal operation.
 * No other wait is affected; nothing faults and the context stays usable. After such
 * a call, zero-fill the workspace and clear the status, as after any device status
 * error (qmv_gemv_noalloc clears its scratch itself). */
void qmv_debug_split_k_fault(int mode, uint64_t wait_limit_ns);

/* Read (and, if reset != 0, clear) the device status word of the current
 * device. Synchronizes the device. Returns QMV_OK or the first latched device
 * status (QMV_EHEADER, QMV_ETIMEOUT, QMV_ERANGE). Test and diagnostics hook. */
qmv_status qmv_device_status(int reset);

#ifdef __cplusplus
}
#endif
#endif
