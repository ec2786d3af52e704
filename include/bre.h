/*
 * bre.h -- C ABI of libbre: a routed mixture-of-experts FFN layer over
 * block-quantised expert weights, plus the Engram hashed-row gather-decode,
 * for one NVIDIA GB300 (sm_103a).
 *
 * Sources, by page title and section:
 *   [S] Strata-DSV4.1 README -- "DeepSeek-V4.1-Flash" (40 layers x 384 routed
 *       experts, top-6); "Results" (selection-only route bias, mixing weights
 *       stay exact; prefill and decode time split); "Latest (2026-10-14)" (a
 *       verify pass serves the union of the pass's experts once per layer);
 *       V4-Flash "How it works" (finish = shared expert + routed sum);
 *       "Verifying it" (expert tier against a dequantised F32 reference).
 *   [I] strix-llama.cpp issue "Feature Request: support DeepSeek V4.1 Flash
 *       with bounded SSD expert caching" -- "Feature Description" (264-byte
 *       Engram rows: 256 E4M3 values + 8 E8M0 scales; Q2_K / Q8_0 formats);
 *       "DeepSeek V4.1 Engram graph integration" (rows gathered per token);
 *       "Stack progress" (request-union planning; split routing from expert
 *       execution); ROCm cached-expert notes (errors surfaced after
 *       synchronisation with safe in-range indices).
 *   [V] vllm.cpp PR, DeepSeek-V4-Flash-Vision -- device router notes (top-k
 *       on the biased score, weights gathered from the unbiased scores; one
 *       warp per row; refusal by name).
 *
 * Conventions (every entry point):
 *   - All pointers are DEVICE pointers unless marked "host".  The caller owns
 *     and allocates every buffer, workspaces included; the library allocates
 *     nothing and keeps no state beyond a per-device attribute cache.
 *   - Work is enqueued on `stream` and is asynchronous; nothing synchronises.
 *   - Arguments the host can check (null pointers, sizes, alignment, shapes
 *     the kernels do not support) return BRE_ERR_ARG / BRE_ERR_UNSUPPORTED
 *     before any launch.  A failed launch returns BRE_ERR_CUDA.
 *   - Data-dependent faults never trap: kernels clamp to a safe index, write
 *     zeros for the affected values and OR a BRE_DEVERR_* bit into the
 *     caller's int32 `dev_err` word (may be NULL), read after synchronising.
 *   - BF16 values are passed as raw 16-bit patterns (uint16_t storage).
 */
#ifndef BRE_H
#define BRE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *bre_stream_t; /* a cudaStream_t; NULL = legacy default stream */

typedef enum {
  BRE_OK = 0,
  BRE_ERR_ARG = 1,         /* invalid argument (null pointer, bad size or alignment) */
  BRE_ERR_UNSUPPORTED = 2, /* valid but outside what the kernels implement */
  BRE_ERR_CUDA = 3,        /* a CUDA call or launch failed */
  BRE_ERR_WORKSPACE = 4    /* workspace missing or smaller than the *_workspace() size */
} bre_status;

/* bits of the device error word */
#define BRE_DEVERR_EXPERT_ID 1 /* an expert id outside [0, E): pair excluded, its output zero */
#define BRE_DEVERR_ROW_ID 2    /* an Engram row id outside [0, n_rows): row decoded as +0 */
#define BRE_DEVERR_TIMEOUT 4   /* a bounded device wait gave up; outputs of that CTA are invalid */

typedef enum { BRE_FMT_Q2_K = 1, BRE_FMT_Q8_0 = 2, BRE_FMT_Q2_K_R16 = 3 } bre_fmt;

/* One FFN weight set.  gate, up: [n_experts][d_ff][d] and down: [n_experts][d][d_ff]
 * weights, each row stored as consecutive quant blocks along its inner
 * (contraction) axis.  Q2_K block (84 B / 256 weights): uint8 scales[16]
 * (low nibble scale, high nibble min), uint8 qs[64] (code i in bits
 * 2*(i%4) of qs[i/4]), fp16 d, fp16 dmin; w = d*sc*q - dmin*m for weight i
 * in sub-block i/16.  Q8_0 block (34 B / 32 weights): fp16 d, int8 q[32];
 * w = d*q.  Q2_K_R16: the same Q2_K blocks regrouped by bre_repack_q2k_r16
 * into 1344-byte tiles of 16 rows x one block (layout below); the matrix
 * has the same size.  expert_stride_*: bytes from one expert's matrix to the
 * next (ignored when n_experts == 1).  Base pointers and strides must be
 * 16-byte aligned. */
typedef struct {
  const void *gate;
  const void *up;
  const void *down;
  int32_t fmt; /* bre_fmt */
  int32_t n_experts;
  int32_t d;
  int32_t d_ff;
  int64_t expert_stride_gate;
  int64_t expert_stride_up;
  int64_t expert_stride_down;
} bre_ffn_weights;

const char *bre_status_string(bre_status s);

/* Router: score, bias, top-k, renormalised weights ([S] "Results";
 * [V] router notes).  For each token t and expert e:
 *   z = x[t,:] . w_r[:,e]  -- FP32, 32 partial sums (partial j takes fmaf over
 *       rows c = j, j+32, ... in ascending order, from +0), then a butterfly
 *       p_j += p_(j^o) for o = 16, 8, 4, 2, 1; z = p_0
 *   s = 1 / (1 + exp(-z)) in float by a fixed sequence of IEEE operations
 *       (Cody-Waite range reduction, degree-7 Taylor polynomial of exp with fmaf,
 *       exact scaling by 2^n; z < -88 gives s = 0), so it is reproducible bit for bit
 *   key = s + bias[e]  (float)
 * ids[t,:] = the k experts with the largest key, ordered by key descending
 * then id ascending (a NaN key ranks last); w[t,j] = s_j / S with
 * S = (((s_0 + s_1) + s_2) ...) in slot order -- weights use the UNBIASED
 * scores.
 *   x_bf16 [T][d] BF16; w_r [d][E] FP32 row-major; bias [E] FP32 or NULL;
 *   topk_ids [T][k] int32 out; topk_w [T][k] FP32 out.
 *   ws: moe_route_workspace(T, E) bytes of scratch, zero-filled once after
 *   allocation (the call leaves it ready for the next call).
 * Requires 1 <= k <= min(E, 32), E <= 1024, d % 32 == 0. */
size_t moe_route_workspace(int T, int E);
bre_status moe_route(const void *x_bf16, const float *w_r, const float *bias, int T, int d, int E, int k,
                     int32_t *topk_ids, float *topk_w, void *ws, size_t ws_bytes, bre_stream_t stream);

/* moe_route without a workspace argument, for callers that cannot allocate device memory:
 * serving loops that must not call cudaMalloc on the hot path (it may synchronise the whole
 * device), and integrations that are handed only pre-allocated input and output buffers with
 * no allocator to ask for scratch.  The pages have no counterpart: it is an interface
 * convenience of this library.  It computes exactly what moe_route computes.
 *   Scratch: one fixed device array inside the library (256 bytes plus the larger of
 *   4 * BRE_ROUTE_STATIC_MAX_TE and 397,312 bytes, about 388 KB), held by every GPU that
 *   loads the library until the process exits.  T * E above BRE_ROUTE_STATIC_MAX_TE, or a
 *   shape whose moe_route_workspace exceeds the array, returns BRE_ERR_WORKSPACE.  Allocates
 *   nothing: no cudaMalloc, cudaFree or allocating library routine.
 *   The first call on a device looks up the array's device address (and may load the
 *   library's device code); make that first call before any stream capture.
 *   Every call shares the array: calls that overlap on the GPU (different streams or host
 *   threads without ordering) race.  Each call clears the part that must start at zero
 *   with a memset on `stream`. */
#define BRE_ROUTE_STATIC_MAX_TE 32768
bre_status moe_route_static(const void *x_bf16, const float *w_r, const float *bias, int T, int d, int E, int k,
                            int32_t *topk_ids, float *topk_w, bre_stream_t stream);

/* Expert permutation: the union of selected experts, each run once per call
 * ([S] "Latest (2026-10-14)"; [I] "Stack progress", request-union planning).
 * Stable counting sort of pair ids p = t*k + j by expert id:
 *   offsets [E+1]: exclusive prefix sum of per-expert pair counts (valid ids only)
 *   perm [T*k]: perm[offsets[e] + r] = r-th smallest p with ids[p] == e
 *   inv [T*k]: inv[perm[q]] = q
 *   active [E]: ascending experts with at least one pair (rest -1); n_active [1].
 * Pairs with an id outside [0, E) are placed after every group, in p order,
 * and set BRE_DEVERR_EXPERT_ID. */
bre_status moe_permute(const int32_t *topk_ids, int T, int k, int E, int32_t *offsets, int32_t *perm,
                       int32_t *inv, int32_t *active, int32_t *n_active, int32_t *dev_err,
                       bre_stream_t stream);

/* moe_route with the per-row rule of the vllm.cpp PR "DeepSeek-V4-Flash-Vision tower", device
 * router notes (SqrtSoftplusRouteTopk):
 *   score: BRE_SCORE_SIGMOID (the float sigmoid above) or BRE_SCORE_SQRT_SOFTPLUS:
 *     s = sqrt(softplus(z)), softplus(z) = max(z, 0) + log1p(exp(-|z|)), in float with every
 *     step one IEEE operation (exp(-|z|) by the sigmoid's exp, 0 for |z| > 87; log1p(e) =
 *     2 atanh(u), u = e / (2 + e), by the degree-7 series in u^2 with fmaf), so it is
 *     reproducible bit for bit;
 *   row t is a media row when vision_bias and is_media are both given and is_media[t] != 0:
 *     its key is s + vision_bias[e] and it selects the top k; a text row's key is s + bias[e]
 *     (bias NULL: s);
 *   tid2eid [vocab][k] int32 (or NULL): a hash layer -- a TEXT row's ids are
 *     tid2eid[token_ids[t]][0..k) in table order, with no key; media rows select as above;
 *   weights always from the UNBIASED s of the row's ids, S summed in slot order.
 *   Hash rows: token_ids[t] outside [0, vocab) sets BRE_DEVERR_ROW_ID and gives ids -1 and
 *   weights 0; a table id outside [0, E) sets BRE_DEVERR_EXPERT_ID, is written as it is (so
 *   moe_permute places it after every group) and counts s = 0.
 *   vision_bias [E] FP32, is_media [T] uint8, token_ids [T] int32: device pointers.
 *   dev_err may be NULL.  Other arguments, limits and ws as for moe_route; with no option set
 *   (score 0, all pointers NULL) it computes exactly what moe_route computes. */
#define BRE_SCORE_SIGMOID 0
#define BRE_SCORE_SQRT_SOFTPLUS 1
bre_status moe_route_ex(const void *x_bf16, const float *w_r, const float *bias, int T, int d, int E, int k,
                        int score, const float *vision_bias, const uint8_t *is_media, const int32_t *tid2eid,
                        const int32_t *token_ids, int vocab, int32_t *topk_ids, float *topk_w, int32_t *dev_err,
                        void *ws, size_t ws_bytes, bre_stream_t stream);

/* moe_route followed by moe_permute, with the same arguments and outputs as the two calls
 * (ws: moe_route_workspace(T, E) bytes, zero-filled once after allocation).  For batches of
 * at most 32 tokens the router kernel's last CTA (the one that merges every token's
 * candidates) also builds the permutation, so the pair is one launch.  Otherwise the router's
 * launches are followed by the permutation; above 1,024 pairs it runs as three grid-wide
 * launches over chunks of 1,024 pairs that keep their per-chunk key counts in ws (the router's
 * score buffer, no longer needed by then), with the same result as moe_permute.  Router ids
 * are always in [0, E), so dev_err is only touched by the second form. */
bre_status moe_route_permute(const void *x_bf16, const float *w_r, const float *bias, int T, int d, int E, int k,
                             int32_t *topk_ids, float *topk_w, int32_t *offsets, int32_t *perm, int32_t *inv,
                             int32_t *active, int32_t *n_active, int32_t *dev_err, void *ws, size_t ws_bytes,
                             bre_stream_t stream);

/* Regroup Q2_K matrices into the Q2_K_R16 tiles the expert FFN reads (a layout of
 * this library, done once when weights are loaded; the pages' Q2_K block, strix-llama.cpp
 * issue "Feature Description", is unchanged in content).  src: n_matrices matrices of
 * [rows][cols/256] Q2_K blocks, src_stride bytes apart; dst: the same number of bytes per
 * matrix, dst_stride apart, must not overlap src.  Tile (rt, b) of rows 16 rt .. 16 rt + 15 and
 * block b sits at byte (rt * (cols/256) + b) * 1344 of the matrix; inside a tile, for row
 * 8 rr + g (g < 8) and lane L = 4 g + t (t < 4):
 *   [512 rr + 16 L, +16): four words W(p, w) (p, w in {0,1}, at word 2p + w); bits 16h + 2s
 *     of W(p, w) hold code 8w + s (s < 8) of sub-block 4t + 2p + h (h in {0, 1}) of the row;
 *   [1024 + 8 L, +8): two words, the scales then the mins of sub-blocks 4t .. 4t+3 of rows g
 *     and g + 8: the nibble of (row 8 rr + g, sub-block 4t + 2p + h) at bit 16h + 4 (2 rr + p);
 *   [1280 + 8 g + 4 rr, +4): fp16 d then fp16 dmin of row 8 rr + g.
 * Requires rows % 16 == 0, cols % 256 == 0, pointers and strides 16-byte aligned. */
bre_status bre_repack_q2k_r16(const void *src, void *dst, int n_matrices, int rows, int cols, int64_t src_stride,
                              int64_t dst_stride, bre_stream_t stream);

/* Routed expert FFN plus the always-on shared expert ([S] V4-Flash "How it
 * works", finish step; "Verifying it"): for every active expert e and each of
 * its pairs p (token t = p / k):
 *   h = silu(gate_e . x_t) * (up_e . x_t);  y_pairs[inv[p]] = down_e . h
 * and for the shared expert (weight 1) on every token: y_shared[t].  No
 * SwiGLU clamp.  Weights are dequantised exactly; accumulation is FP32.
 *   routed: fmt BRE_FMT_Q2_K_R16 (bre_repack_q2k_r16 of the Q2_K experts), n_experts = E.
 *   shared: fmt BRE_FMT_Q8_0, n_experts = 1, or NULL (then y_shared is not written).
 *   x_bf16 [T][d]; offsets/perm/active/n_active from moe_permute (k pairs per
 *   token); y_pairs [T*k][d] FP32 out, row q = permuted position q (rows of
 *   pairs with an invalid id are not written); y_shared [T][d] FP32 out.
 *   ws: moe_expert_ffn_workspace(T, ...) bytes, zero-filled once after allocation.
 *   Its leading part holds the decode path's (T <= 8) item counters and a
 *   scheduling word, which each such call sets before use; a workspace sized for T serves every call with
 *   T' <= T (same k, d, d_ff, d_ff_shared).  Calls sharing one workspace must be
 *   ordered.  The workspace
 *   must not overlap any buffer of the call enqueued just before this one on the
 *   stream (for T <= 8 its first kernel packs x into the workspace while a
 *   preceding moe_route_permute may still be running; it reads only x_bf16).
 * Shapes: d and d_ff multiples of 256. */
size_t moe_expert_ffn_workspace(int T, int k, int E, int d, int d_ff, int d_ff_shared);
bre_status moe_expert_ffn(const bre_ffn_weights *routed, const bre_ffn_weights *shared, const void *x_bf16,
                          int T, int k, const int32_t *offsets, const int32_t *perm, const int32_t *active,
                          const int32_t *n_active, float *y_pairs, float *y_shared, void *ws, size_t ws_bytes,
                          int32_t *dev_err, bre_stream_t stream);

/* Weighted combine ([S] "How it works", finish: shared expert + routed sum):
 *   acc[t] = y_shared[t] + sum_j topk_w[t,j] * y_pairs[inv[t*k+j]],  out[t] = bf16_rne(acc[t])
 * FP32 accumulation from y_shared (or 0 when NULL), j ascending.  A pair whose
 * position inv >= offsets[E] (invalid id) contributes nothing.
 *   out_bf16 [T][d] out; out_f32 [T][d] out (the value before rounding), or NULL. */
bre_status moe_combine(const float *y_pairs, const float *topk_w, const int32_t *inv, const int32_t *offsets,
                       int E, const float *y_shared, int T, int k, int d, void *out_bf16, float *out_f32,
                       bre_stream_t stream);

/* Residual update of a stack of MoE layers with no attention (verify batch of
 * [S] "Latest (2026-10-14)"):
 *   x_out = bf16_rne(x + bf16(moe) * scale)   (product and sum each rounded)
 *   u_out = bf16_rne(x_out * r),  r = 1 / sqrtf(mean(x_out^2) + eps)
 * where the sum of squares uses the router's 32-partial order.  u_out (the
 * next layer's MoE input) may be NULL.  x, moe, x_out, u_out: [T][d] BF16. */
bre_status moe_residual_norm(const void *x_bf16, const void *moe_bf16, int T, int d, float scale, float eps,
                             void *x_out_bf16, void *u_out_bf16, bre_stream_t stream);

/* Engram gather-decode ([I] "Feature Description"; "DeepSeek V4.1 Engram
 * graph integration").  Row layout: 256 E4M3 (OCP, bias 7, no inf) bytes, then
 * 8 E8M0 scale bytes, one per 32 values.  For each token t, table tau, head h:
 *   v_h[c] = e4m3(row[c]) * 2^(row[256 + c/32] - 127),  row = tables[tau][ids[t,tau,h]]
 *   out[t, tau*256 + c] = bf16_rne(((v_0 + v_1) + v_2) + ...)   (FP32, h ascending)
 * NaN results are written as 0x7FC0; -0 is kept.
 *   tables: HOST array of n_tables device pointers (8-byte aligned);
 *   n_rows: HOST array [n_tables]; row_ids [T][n_tables][H] int64;
 *   out_bf16 [T][n_tables*256].  An id outside [0, n_rows) decodes as +0 and
 *   sets BRE_DEVERR_ROW_ID.  Requires 1 <= n_tables <= 8, 1 <= H <= 64. */
bre_status engram_gather_decode(const uint8_t *const *tables, const int64_t *n_rows, int n_tables,
                                const int64_t *row_ids, int T, int H, void *out_bf16, int32_t *dev_err,
                                bre_stream_t stream);

/* Engram gate and residual injection (strix-llama.cpp issue, "Placement"), for one Engram layer:
 *   rows: the R table rows of token t (row_ids [T][R] int64, device) decoded as
 *     engram_gather_decode does (e4m3 x 2^(e8m0 - 127), BF16) and concatenated -> x_t [R * 256];
 *   kv_t = engram_kv.weight . x_t, FP32 accumulation; w_kv_bf16 [5W][R * 256] BF16 (rows are the
 *     outputs); kv_t = four keys [4][W] then one shared value [W];
 *   for each hyper-connection branch h < 4 of resid_bf16 [T][4][W] (BF16, updated in place):
 *     dot = sum_i r[h,i] q_norm[h,i] k_norm[h,i] key[h,i]
 *           * 1/sqrt(mean(r[h,:]^2) + eps) * 1/sqrt(mean(key[h,:]^2) + eps) * 1/sqrt(W)
 *     gate = sigmoid(copysign(sqrt(max(|dot|, 1e-6)), dot))
 *     r[h,i] = bf16(r[h,i] + gate * bf16(value[i]))        (FP32 arithmetic, one rounding each)
 *   mask [T] uint8 or NULL: tokens with mask[t] != 0 keep their residual byte for byte.
 *   q_norm, k_norm [4][W] FP32.  kv_out [T][5W] FP32 and gate_out [T][4] FP32 are optional
 *   (NULL: not written; masked tokens get gate 0).  A row id outside [0, n_rows) decodes as
 *   zeros and sets BRE_DEVERR_ROW_ID in dev_err (may be NULL).
 *   ws: engram_inject_workspace(T, R, W) bytes, zero-filled once after allocation (each call
 *   leaves its counter at zero).  Requires W % 16 == 0, W <= 8192 and R <= 24 (the tokens' rows
 *   are held in shared memory; batches of 8 tokens run one after the other, each reading w_kv
 *   once). */
size_t engram_inject_workspace(int T, int R, int W);
bre_status engram_inject(const uint8_t *table, int64_t n_rows, const int64_t *row_ids, int R, const void *w_kv_bf16,
                         int W, void *resid_bf16, const float *q_norm, const float *k_norm, const uint8_t *mask, int T,
                         float eps, float *kv_out, float *gate_out, int32_t *dev_err, void *ws, size_t ws_bytes,
                         bre_stream_t stream);

/* Budget, in SM clock cycles, of the bounded waits inside the expert FFN kernels
 * (moe_expert_ffn, both paths) for calls made after this one, from any thread of the process;
 * 0 restores the defaults (about 1 s on the decode path, 2 s on the grouped-GEMM path).  A wait
 * that runs out sets BRE_DEVERR_TIMEOUT in the call's dev_err; the kernel then waits, with the
 * default budget, for the copies and tensor-core operations it has in flight, frees its tensor
 * memory and returns, and that call's outputs are invalid.  The next call on the same workspace
 * needs nothing done to it (the decode path clears its counters at the start of every call).  A small budget exercises that path (the ROCm cached-expert notes of the
 * strix-llama.cpp issue: errors surface after synchronisation rather than as a trap); serving
 * code leaves the default.  Negative: BRE_ERR_ARG. */
bre_status bre_set_ffn_wait_limit(int64_t cycles);

/* Dequantise n_blocks blocks of format fmt to FP32 on the device, with the
 * same decode the FFN kernels use (exact: every product is exact in FP32 and
 * the one rounding is the final subtraction).  out [n_blocks * 256 or * 32]. */
bre_status bre_dequant(int fmt, const void *blocks, int64_t n_blocks, float *out, bre_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* BRE_H */
