/* ggufdq.h -- C ABI of the GB300 GGUF block-dequant GEMV / MoE library.
 *
 * The library computes matrix-vector products over GGUF block-quantized weights that stay
 * in their raw GGUF block layout in device memory and are decoded inside the product, plus
 * the mixture-of-experts step built on them.  The operations follow the engine pages of the
 * diskformer npm package:
 *   - qwen3_moe_ssd.js (diskformer 0.0.1 -> 0.3.0): header comment (Q8_0 blocks kept
 *     bit-exact, dot products equal llama.cpp's up to summation order); WGSL kernels
 *     matmulQ8, matmulF32, topk, expertQ8, siluMulMoe, moeAccum.
 *   - qwen35_moe_ssd.js (diskformer 0.5.4 -> 0.6.6): BATCH_KERNELS matmulQ8T (token-major
 *     batches, one weight read serves several tokens), topkB, expertQ8B, siluMul2B.
 *   - gemma4_moe_ssd.js (diskformer 0.5.4 -> 0.6.6): Q4_0 layout (Q4DOT comment), Q6_K
 *     layout (Q6P comment), matmulQ4, matmulQ6K.
 *   - ternary_bonsai_2_dflash.js (diskformer 0.5.4 -> 0.6.6): the K-quant block layouts
 *     ("Layouts follow ggml-quants.c"), dequantQ4K / dequantQ6K, WG_GEMM_Q4K / WG_GEMM_Q6K.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The library never
 *     allocates device memory, never synchronises the stream and keeps no host state; all
 *     work is enqueued on `stream` (NULL = the legacy default stream).
 *   - Weights `w` are raw GGUF blocks, row-major: row m of an [M][N] tensor is N / QK
 *     consecutive blocks.  Block layouts (QK elements, bytes):
 *       QG_TYPE_Q8_0  (32, 34):  f16 d, int8 q[32];            w = d * q
 *       QG_TYPE_Q4_0  (32, 18):  f16 d, u8 qs[16];  byte j holds element j (low nibble)
 *                                and j + 16 (high nibble);      w = (nibble - 8) * d
 *       QG_TYPE_Q4_K (256, 144): f16 d, f16 dmin, u8 scales[12] (8 packed 6-bit scales and
 *                                mins), u8 qs[128];             w = d*sc*q - dmin*m
 *       QG_TYPE_Q6_K (256, 210): u8 ql[128], u8 qh[64], int8 scales[16], f16 d;
 *                                                               w = d * scale * (q - 32)
 *   - Activations and outputs are f32, token-major: x[t][k] at x + t*N + k, y[t][m] at
 *     y + t*M + m.  Accumulation is f32; results equal the exact products up to f32
 *     summation order.
 *   - Alignment: `w`, every f32 tensor and every expert base must be 16-byte aligned;
 *     expert strides must be multiples of 16 bytes.
 *   - Errors: argument checks run on the host before anything is enqueued and return a
 *     non-zero qg_status with nothing launched.  QG_ECUDA reports a launch failure
 *     (cudaGetLastError).  Kernels never trap: a device-side check that fails (an expert
 *     id out of range, a bounded wait that expired) sets a device status word that
 *     qg_device_status() reads, and the affected outputs are undefined.
 *   - Outputs never alias inputs, except x_inout in moe_combine / moe_layer.
 */
#ifndef GGUFDQ_H
#define GGUFDQ_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QG_API __attribute__((visibility("default")))
#else
#define QG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; the header does not need the CUDA headers. */
typedef struct CUstream_st *qg_stream_t;

/* ggml type ids of the supported block formats */
enum {
  QG_TYPE_Q4_0 = 2,
  QG_TYPE_Q8_0 = 8,
  QG_TYPE_Q4_K = 12,
  QG_TYPE_Q6_K = 14
};

typedef enum qg_status {
  QG_OK = 0,
  QG_EINVAL_SHAPE = 1,  /* a size is out of range or not a multiple of the block size */
  QG_EINVAL_PTR = 2,    /* a required pointer is NULL */
  QG_EALIGN = 3,        /* a pointer or stride is not 16-byte aligned */
  QG_EUNSUPPORTED = 4,  /* block type not supported by this call */
  QG_ECUDA = 5,         /* a CUDA call or kernel launch failed */
  QG_EDEVICE_ID = 6,    /* device status bit: an expert id or slot was out of range */
  QG_ETIMEOUT = 7,      /* device status bit: a bounded wait inside a kernel expired */
  QG_EWORKSPACE = 8     /* workspace pointer NULL or smaller than the size query says */
} qg_status;

/* Library ABI version (incremented on incompatible changes). */
QG_API int qg_version(void);

/* Short description of a status code; never NULL. */
QG_API const char *qg_strerror(int status);

/* Elements and bytes per block of `type`; returns QG_EUNSUPPORTED for other types. */
QG_API qg_status qg_block_shape(int type, int *qk, int *block_bytes);

/* Device status word of the current device: a bitwise OR of (1 << QG_EDEVICE_ID) and
 * (1 << QG_ETIMEOUT) for every kernel that detected such a condition since the last clear.
 * Synchronises the device.  When `clear` is non-zero the word is reset to 0. */
QG_API qg_status qg_device_status(uint32_t *status_out, int clear);

/* Static weights, a setting of one stream (off by default).  Every launch of this library
 * waits for the preceding kernel in its stream (programmatic dependent launch) before it
 * touches memory.  A caller whose weight buffers are immutable model parameters - written
 * once, before any GEMV that reads them, and never by a kernel enqueued ahead of a GEMV in
 * the same stream - may call qg_set_static_weights(stream, 1): the dense GEMVs (qgemv_*,
 * qgemv_t, qgemv_multi) and the one-token MoE layer enqueued on that stream then start
 * streaming their first weight tiles while the preceding kernel drains, and only the
 * activations and outputs wait for it.  Leave it off when a kernel in the stream may write
 * the weights (quantise-in-place, a loader that copies through a kernel): the GEMV could read
 * stale bytes.  Host-to-device copies are ordered either way.
 *   - The setting belongs to the (device, stream handle) pair that is current at the call,
 *     and other streams and other users of the library in the process are not affected.
 *     Clear it before destroying the stream: a new stream may reuse the handle.
 *   - It takes effect for launches enqueued (or captured) after the call.
 *   - Returns the previous setting of that stream (0 or 1), or -1 when 256 streams already
 *     hold the setting. */
QG_API int qg_set_static_weights(qg_stream_t stream, int enable);

/* ---- dense quantized GEMV, one token ----------------------------------------------------
 * y[m] = sum_k W[m][k] * x[k] for m < M  (matmulQ8 / matmulQ4 / matmulQ6K on the pages, and
 * the Q4_K row dot of WG_GEMM_Q4K).  w: M*N/QK raw blocks; x: f32[N]; y: f32[M].
 * N must be a positive multiple of QK (32 for Q8_0 / Q4_0, 256 for Q4_K / Q6_K), M >= 0
 * (M == 0 enqueues nothing), M, N <= 2^31 - 1. */
QG_API qg_status qgemv_q8_0(const void *w, const float *x, float *y, int64_t M, int64_t N, qg_stream_t stream);
QG_API qg_status qgemv_q4_0(const void *w, const float *x, float *y, int64_t M, int64_t N, qg_stream_t stream);
QG_API qg_status qgemv_q4_k(const void *w, const float *x, float *y, int64_t M, int64_t N, qg_stream_t stream);
QG_API qg_status qgemv_q6_k(const void *w, const float *x, float *y, int64_t M, int64_t N, qg_stream_t stream);

/* ---- dense quantized GEMV over T token columns, one weight pass ---------------------------
 * Y[t][m] = sum_k W[m][k] * X[t][k] for t < T, m < M  (matmulQ8T in qwen35_moe_ssd.js: every
 * weight byte read serves all T tokens).  x: f32[T][N]; y: f32[T][M]; 1 <= T <= 16.
 * Same shape rules as above. */
QG_API qg_status qgemv_t(int type, const void *w, const float *x, float *y, int64_t M, int64_t N, int T,
                  qg_stream_t stream);

/* ---- several matrices over the same activations, one launch ------------------------------
 * Y_j[t][m] = sum_k W_j[m][k] * X[t][k] for j < n (n <= 4), every W_j of the same type and row
 * length N, X shared.  The decode steps whose projections read one normalised input (q, k and
 * v of attention; gate and up of the FFN) stream all their rows in a single pass of the
 * kernel instead of one launch each.  w, y and M are HOST arrays of n entries (device pointers
 * to raw blocks and f32 [T][M_j] outputs, row counts); a matrix with M_j == 0 is skipped.
 * Same shape and alignment rules as qgemv_t. */
QG_API qg_status qgemv_multi(int type, int n, const void *const *w, float *const *y, const int64_t *M, int64_t N,
                      const float *x, int T, qg_stream_t stream);

/* ---- prefill dequant-GEMM, T >= 17 token rows --------------------------------------------
 * Y[t][m] = sum_k W[m][k] * X[t][k] with W decoded to bf16 and X rounded to bf16 for the
 * tensor cores, f32 accumulation (the tiled matmulQ8T generalised to a prefill chunk).
 * Workspace: at least qgemm_workspace_size(type, M, N, T) bytes of device memory, 16-byte
 * aligned, used for the bf16 copy of X; may be NULL when the size is 0.  T >= 1 is
 * accepted (T <= 16 is routed to qgemv_t, which is exact in f32). */
QG_API size_t qgemm_workspace_size(int type, int64_t M, int64_t N, int64_t T);
QG_API qg_status qgemm(int type, const void *w, const float *x, float *y, int64_t M, int64_t N, int64_t T,
                void *workspace, size_t workspace_bytes, qg_stream_t stream);

/* ---- MoE step ----------------------------------------------------------------------------
 * Shapes: T tokens, hidden size H, expert FFN size F, E router experts, k picks per token.
 * Limits: 1 <= k <= 32, k <= E <= 256 (the pages' topk limits), H and F multiples of the
 * block QK, H % 4 == 0.
 * Expert weights: expert e lives in pool slot s = slots[e] (slots == NULL: s = e); its gate
 * rows (F x H), up rows (F x H) and down rows (H x F) are raw blocks at
 * w_gate + s*expert_stride, w_up + s*expert_stride, w_down + s*expert_stride.  This covers
 * the pages' per-expert record (gate || up || down contiguous, expertQ8 with
 * rowsPerExpert) and GGUF's separate ffn_{gate,up,down}_exps tensors.  0 <= s < n_slots.
 * ids / weights: int32 [T][k] expert ids in pick order and f32 [T][k] combine weights.
 * Pairs z = t*k + j index the per-pick buffers (act is f32 [T*k][F]).
 *
 * Workspace: moe_workspace_size(T, k, E, H, F) bytes of device memory, 16-byte aligned,
 * zero-filled by the caller once before its first use.  Its first 260 KB are a fixed header
 * whose words keep their meaning from call to call: the one-token layer's grid-barrier
 * counter and call counter (64-bit words that every moe_layer call at T = 1 advances), its
 * logits tagged with the call, and the router's per-tile tickets (every call leaves them at
 * zero again).  Their offsets do not depend on the
 * call's shape, so one workspace sized for the largest shape it will serve (the largest T, k,
 * E, H, F) may serve any call whose moe_workspace_size is not larger.  The rest holds scratch
 * that each call rewrites: the router logits, the per-pick down rows and, for more than 16
 * tokens, the grouped bf16 rows.  A NULL, misaligned or too small workspace returns
 * QG_EWORKSPACE (QG_EALIGN when misaligned) with nothing launched.  Calls that share a
 * workspace must not run concurrently. */
QG_API size_t moe_workspace_size(int T, int k, int E, int H, int F);

/* Router (matmulF32 + topk / topkB): logits l[t][e] = sum_h wr[e][h] * xn[t][h] (f32
 * weights), softmax over the E logits, k greedy picks of the largest (ties to the lowest
 * expert id), weights p_j / sum of the picked p (norm_topk_prob).  Picks are taken on the
 * logits, which gives the same order as taking them on the softmax probabilities.
 * xn: f32 [T][H]; wr: f32 [E][H]; ids: int32 [T][k]; weights: f32 [T][k];
 * logits_out: optional f32 [T][E] copy of the logits (NULL to skip). */
QG_API qg_status moe_route_topk(const float *xn, const float *wr, int T, int H, int E, int k, int32_t *ids,
                         float *weights, float *logits_out, void *workspace, size_t workspace_bytes,
                         qg_stream_t stream);

/* The router of moe_route_topk for callers that cannot hand the library a workspace: for
 * instance a host engine whose device memory is entirely reserved by its own allocator before
 * it calls in, or a binding that exposes only input and output tensors.  The library keeps a
 * fixed 68 KB scratch area in device memory (1024 ticket words, then 16384 logits) and
 * allocates nothing (no cudaMalloc, no allocating library call).
 *   - Limits: T * E <= 16384 and T <= 16384 (at most 1024 tiles of 16 tokens); larger shapes
 *     return QG_EWORKSPACE.  Every other argument check is moe_route_topk's, and all of them
 *     run before anything is enqueued.
 *   - The scratch address is looked up once per device, on the first call with that device
 *     current; make that first call before any stream capture.
 *   - Each call clears the tickets of its shape on `stream` (one memset) before the router
 *     runs; with logits_out == NULL the logits live in the scratch area.
 *   - One scratch area per device: calls that overlap (other streams, other host threads)
 *     race on it and must be serialised by the caller.
 * Results are the same as moe_route_topk's.  The engine pages have no counterpart: their
 * router buffers are allocated by the engine. */
QG_API qg_status moe_route_topk_noalloc(const float *xn, const float *wr, int T, int H, int E, int k, int32_t *ids,
                                 float *weights, float *logits_out, qg_stream_t stream);

/* Gate/up expert rows with SwiGLU (expertQ8 with a shared input, then siluMulMoe): for each
 * pair z = t*k + j with expert e = ids[z]:  g = Wg[s] . xn[t],  u = Wu[s] . xn[t]  (F rows
 * each),  act[z][i] = g_i / (1 + exp(-g_i)) * u_i.  Experts are grouped so that each picked
 * expert's rows are read once for all its tokens.  An id outside [0, E) or a slot outside
 * [0, n_slots) sets QG_EDEVICE_ID in the device status and that pair's act row is zero. */
QG_API qg_status moe_expert_swiglu(int type, const void *w_gate, const void *w_up, int64_t expert_stride,
                            const int32_t *slots, int n_slots, int E, const int32_t *ids, const float *xn,
                            int T, int k, int H, int F, float *act, void *workspace, size_t workspace_bytes,
                            qg_stream_t stream);

/* Down expert rows and the weighted combine (expertQ8 with a per-pick input, then
 * moeAccum):  x_inout[t][h] = (add_residual ? x_inout[t][h] : 0)
 *                              + sum_j weights[t][j] * (Wd[s_j] . act[t*k + j])[h].
 * The expert sum is formed first and the residual added last, as the pages order it. */
QG_API qg_status moe_combine(int type, const void *w_down, int64_t expert_stride, const int32_t *slots, int n_slots,
                      int E, const int32_t *ids, const float *weights, const float *act, int T, int k, int H,
                      int F, float *x_inout, int add_residual, void *workspace, size_t workspace_bytes,
                      qg_stream_t stream);

/* The whole MoE step: moe_route_topk, moe_expert_swiglu, moe_combine (add_residual = 1).
 * xn: router / expert input [T][H]; x_inout: residual stream [T][H], updated in place;
 * ids, weights, act: caller buffers that receive the intermediates. */
QG_API qg_status moe_layer(int type, const float *xn, const float *wr, const void *w_gate, const void *w_up,
                    const void *w_down, int64_t expert_stride, const int32_t *slots, int n_slots, int T, int H,
                    int F, int E, int k, int32_t *ids, float *weights, float *act, float *x_inout,
                    void *workspace, size_t workspace_bytes, qg_stream_t stream);

/* ---- the steps on either side of a GEMV chain ----------------------------------------------
 * Embedding row gather (embedQ8 in qwen3_moe_ssd.js, embedQ6K in gemma4_moe_ssd.js):
 *   out[i][k] = w(ids[i], k) * scale   for i < n, k < N,
 * w(r, .) the dequantized row r of the [V][N] table in raw blocks of `type` (any of the four),
 * decoded by the GEMV's own decoders; the product is one f32 rounding (scale = 1 is exact;
 * embedQ6K's page multiplies by sqrt(H)).  table: device, 16-byte aligned, V*N/QK blocks;
 * ids: device int32[n]; out: device f32[n][N], 16-byte aligned.  N a positive multiple of QK,
 * 1 <= V, 0 <= n (n == 0 enqueues nothing).  An id outside [0, V) gives a zero row and sets
 * QG_EDEVICE_ID in the device status. */
QG_API qg_status qg_embed_rows(int type, const void *table, int64_t V, int64_t N, const int32_t *ids, int n,
                               float scale, float *out, qg_stream_t stream);

/* RMSNorm (rmsnorm in qwen3_moe_ssd.js, rmsnormB for a token batch; with a factor, rmsnormK
 * of gemma4_moe_ssd.js, the MoE router's input with k = 1/sqrt(H)):
 *   y[t][i] = ((x[t][i] * s_t) * k) * w[i],   s_t = 1 / sqrt(mean_i x[t][i]^2 + eps),
 * sums in f32; k = 1 is plain RMSNorm.  x, y: device f32[T][N]; w: device f32[N]; all 16-byte
 * aligned; y may be x.  N a positive multiple of 4, 0 <= T <= 65535, eps >= 0. */
QG_API qg_status qg_rmsnorm(const float *x, const float *w, int T, int64_t N, float eps, float k, float *y,
                            qg_stream_t stream);

/* argmax per row (argmax in qwen3_moe_ssd.js, argmaxRows in qwen35_dense.js): ids[t] = the
 * lowest index of the largest value of row t of logits[T][n]; NaN is never picked and a row
 * with nothing but NaN gives 0.  logits, ids: device, 4-byte aligned; 0 <= T <= 8191.  Each
 * row is scanned by a cluster of 8 CTAs whose partial picks meet in distributed shared memory. */
QG_API qg_status qg_argmax_rows(const float *logits, int T, int64_t n, int32_t *ids, qg_stream_t stream);

/* Tied head and greedy pick in one call (encodeHead of qwen3_moe_ssd.js: the head GEMV over
 * the vocabulary, then argmax): logits[t][m] = sum_k W[m][k] * x[t][k] as qgemv_t, then
 * ids[t] = argmax_m logits[t][m] as qg_argmax_rows.  logits: device f32[T][M] (caller
 * buffer, written); ids: device int32[T]; 1 <= T <= 16; other rules as qgemv_t.  A caller
 * that wants only the tokens reads back T ids instead of T * M logits. */
QG_API qg_status qg_head_argmax(int type, const void *w, int64_t M, int64_t N, const float *x, int T, float *logits,
                                int32_t *ids, qg_stream_t stream);

/* ---- MoE variants on the same kernels -----------------------------------------------------
 * The Gemma 4 MoE (gemma4_moe_ssd.js: Q4_0 experts, geglu, moeSum's per-expert down scale; its
 * router input is qg_rmsnorm with k = 1/sqrt(H)) and the Qwen3.5/3.6 MoE (qwen35_moe_ssd.js:
 * moeAccumShared, the sigmoid-gated shared expert) differ from the Qwen3 MoE above only in the
 * expert activation and the combine.  A variant is a HOST struct; NULL is the Qwen3 MoE. */
#define QG_ACT_SILU 0      /* act = SiLU(g) * u                         (siluMulMoe) */
#define QG_ACT_GELU_TANH 1 /* act = GELU(g) * u, tanh form, argument clamped to [-10, 10] (geglu) */
typedef struct qg_moe_variant {
  int act;                  /* QG_ACT_SILU or QG_ACT_GELU_TANH */
  const float *down_scale;  /* NULL, or device f32[E]: pick j's down row is scaled by down_scale[id_j] */
  const float *shared_out;  /* NULL, or device f32[T][H] (16-byte aligned): the shared expert's output */
  const float *shared_gate; /* with shared_out: device f32[T], the shared expert's gate logit */
} qg_moe_variant;

/* moe_expert_swiglu with the variant's activation (act[z][i] = SiLU or GELU of gate, times up). */
QG_API qg_status moe_expert_act(int type, const void *w_gate, const void *w_up, int64_t expert_stride,
                                const int32_t *slots, int n_slots, int E, const int32_t *ids, const float *xn, int T,
                                int k, int H, int F, const qg_moe_variant *variant, float *act, void *workspace,
                                size_t workspace_bytes, qg_stream_t stream);

/* moe_combine with the variant's combine (moeSum, then moeAccumShared):
 *   x_inout[t][h] = (add_residual ? x_inout[t][h] : 0)
 *                   + (sum_j (dn_j[h] * down_scale[id_j]) * weights[t][j]  +  shared_out[t][h] * s(shared_gate[t])),
 * dn_j = Wd[s_j] . act[t*k + j], s the logistic function, the expert sum in pick order first,
 * the shared term next, the residual last. */
QG_API qg_status moe_combine_ex(int type, const void *w_down, int64_t expert_stride, const int32_t *slots,
                                int n_slots, int E, const int32_t *ids, const float *weights, const float *act, int T,
                                int k, int H, int F, const qg_moe_variant *variant, float *x_inout, int add_residual,
                                void *workspace, size_t workspace_bytes, qg_stream_t stream);

/* moe_layer with a variant: router with top-k, moe_expert_act, moe_combine_ex (add_residual =
 * 1).  A NULL or default variant is moe_layer itself (one launch at T = 1); other variants run
 * the three steps at every T.  A variant with shared_out and no shared_gate (or the reverse)
 * returns QG_EINVAL_PTR, an unknown act QG_EINVAL_SHAPE, all before anything is enqueued. */
QG_API qg_status moe_layer_ex(int type, const float *xn, const float *wr, const void *w_gate, const void *w_up,
                              const void *w_down, int64_t expert_stride, const int32_t *slots, int n_slots, int T,
                              int H, int F, int E, int k, const qg_moe_variant *variant, int32_t *ids, float *weights,
                              float *act, float *x_inout, void *workspace, size_t workspace_bytes,
                              qg_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GGUFDQ_H */
