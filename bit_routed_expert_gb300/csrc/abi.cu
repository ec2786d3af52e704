// extern "C" entry points of libbre: host-side argument checks, then the launchers.
#include <atomic>

#include <cuda_runtime.h>

#include "bre.h"
#include "kernels.h"

namespace bre {

namespace {
struct DevAttr {
  int sms = 0;
  int smem_optin = 0;
};
DevAttr g_attr[64];

const DevAttr& attr() {
  int dev = 0;
  cudaGetDevice(&dev);
  DevAttr& a = g_attr[dev & 63];
  if (a.sms == 0) {
    cudaDeviceGetAttribute(&a.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaDeviceGetAttribute(&a.sms, cudaDevAttrMultiProcessorCount, dev);
  }
  return a;
}
}  // namespace

std::atomic<long long> g_ffn_wait{0};   // 0: the kernels' default budgets

long long ffn_wait_budget(long long dflt) {
  const long long v = g_ffn_wait.load(std::memory_order_relaxed);
  return v > 0 ? v : dflt;
}

int device_sm_count() { return attr().sms; }
int device_max_smem_optin() { return attr().smem_optin; }

}  // namespace bre

using namespace bre;

static inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
static inline bre_status cuda_status(cudaError_t e) { return e == cudaSuccess ? BRE_OK : BRE_ERR_CUDA; }

extern "C" {

const char* bre_status_string(bre_status s) {
  switch (s) {
    case BRE_OK: return "ok";
    case BRE_ERR_ARG: return "invalid argument";
    case BRE_ERR_UNSUPPORTED: return "unsupported shape or format";
    case BRE_ERR_CUDA: return "CUDA error";
    case BRE_ERR_WORKSPACE: return "workspace too small";
  }
  return "unknown status";
}

size_t moe_route_workspace(int T, int E) { return (T > 0 && E > 0) ? route_ws_bytes(T, E) : 0; }

bre_status moe_route(const void* x_bf16, const float* w_r, const float* bias, int T, int d, int E, int k,
                     int32_t* topk_ids, float* topk_w, void* ws, size_t ws_bytes, bre_stream_t stream) {
  if (!x_bf16 || !w_r || !topk_ids || !topk_w || T <= 0 || d <= 0 || E <= 0 || k <= 0) return BRE_ERR_ARG;
  if (k > E || k > 32 || E > 1024 || d % 32 != 0) return BRE_ERR_UNSUPPORTED;
  if (!aligned(x_bf16, 16) || !aligned(w_r, 16)) return BRE_ERR_ARG;
  if (!ws || ws_bytes < route_ws_bytes(T, E) || !aligned(ws, 256)) return BRE_ERR_WORKSPACE;
  return cuda_status(launch_route(static_cast<const uint16_t*>(x_bf16), w_r, bias, T, d, E, k, topk_ids, topk_w, ws,
                                  reinterpret_cast<cudaStream_t>(stream)));
}

bre_status moe_route_ex(const void* x_bf16, const float* w_r, const float* bias, int T, int d, int E, int k,
                        int score, const float* vision_bias, const uint8_t* is_media, const int32_t* tid2eid,
                        const int32_t* token_ids, int vocab, int32_t* topk_ids, float* topk_w, int32_t* dev_err,
                        void* ws, size_t ws_bytes, bre_stream_t stream) {
  if (!x_bf16 || !w_r || !topk_ids || !topk_w || T <= 0 || d <= 0 || E <= 0 || k <= 0) return BRE_ERR_ARG;
  if (score != BRE_SCORE_SIGMOID && score != BRE_SCORE_SQRT_SOFTPLUS) return BRE_ERR_ARG;
  if (tid2eid && (!token_ids || vocab <= 0)) return BRE_ERR_ARG;
  if (k > E || k > 32 || E > 1024 || d % 32 != 0) return BRE_ERR_UNSUPPORTED;
  if (!aligned(x_bf16, 16) || !aligned(w_r, 16)) return BRE_ERR_ARG;
  if (!ws || ws_bytes < route_ws_bytes(T, E) || !aligned(ws, 256)) return BRE_ERR_WORKSPACE;
  return cuda_status(launch_route_ex(static_cast<const uint16_t*>(x_bf16), w_r, bias, T, d, E, k, score, vision_bias,
                                     is_media, tid2eid, tid2eid ? token_ids : nullptr, tid2eid ? vocab : 0, topk_ids,
                                     topk_w, dev_err, ws, reinterpret_cast<cudaStream_t>(stream)));
}

bre_status moe_route_permute(const void* x_bf16, const float* w_r, const float* bias, int T, int d, int E, int k,
                             int32_t* topk_ids, float* topk_w, int32_t* offsets, int32_t* perm, int32_t* inv,
                             int32_t* active, int32_t* n_active, int32_t* dev_err, void* ws, size_t ws_bytes,
                             bre_stream_t stream) {
  if (!x_bf16 || !w_r || !topk_ids || !topk_w || !offsets || !perm || !inv || !active || !n_active || T <= 0 ||
      d <= 0 || E <= 0 || k <= 0)
    return BRE_ERR_ARG;
  if (k > E || k > 32 || E > 1024 || d % 32 != 0) return BRE_ERR_UNSUPPORTED;
  if (!aligned(x_bf16, 16) || !aligned(w_r, 16)) return BRE_ERR_ARG;
  if (!ws || ws_bytes < route_ws_bytes(T, E) || !aligned(ws, 256)) return BRE_ERR_WORKSPACE;
  return cuda_status(launch_route_permute(static_cast<const uint16_t*>(x_bf16), w_r, bias, T, d, E, k, topk_ids,
                                          topk_w, offsets, perm, inv, active, n_active, dev_err, ws,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

bre_status moe_permute(const int32_t* topk_ids, int T, int k, int E, int32_t* offsets, int32_t* perm, int32_t* inv,
                       int32_t* active, int32_t* n_active, int32_t* dev_err, bre_stream_t stream) {
  if (!topk_ids || !offsets || !perm || !inv || !active || !n_active || T <= 0 || k <= 0 || E <= 0)
    return BRE_ERR_ARG;
  if (E > 1024) return BRE_ERR_UNSUPPORTED;
  return cuda_status(
      launch_permute(topk_ids, T, k, E, offsets, perm, inv, active, n_active, dev_err, reinterpret_cast<cudaStream_t>(stream)));
}

size_t moe_expert_ffn_workspace(int T, int k, int E, int d, int d_ff, int d_ff_shared) {
  if (T <= 0 || k <= 0 || d <= 0 || d_ff <= 0 || d_ff_shared < 0) return 0;
  return ffn_ws_bytes(T, k, E, d, d_ff, d_ff_shared);
}

static bool weights_ok(const bre_ffn_weights* w, int fmt) {
  if (!w->gate || !w->up || !w->down || w->fmt != fmt || w->n_experts <= 0) return false;
  if (!aligned(w->gate, 16) || !aligned(w->up, 16) || !aligned(w->down, 16)) return false;
  if (w->n_experts > 1 && (w->expert_stride_gate % 16 || w->expert_stride_up % 16 || w->expert_stride_down % 16))
    return false;
  return true;
}

bre_status moe_expert_ffn(const bre_ffn_weights* routed, const bre_ffn_weights* shared, const void* x_bf16, int T,
                          int k, const int32_t* offsets, const int32_t* perm, const int32_t* active,
                          const int32_t* n_active, float* y_pairs, float* y_shared, void* ws, size_t ws_bytes,
                          int32_t* dev_err, bre_stream_t stream) {
  if (!routed || !x_bf16 || !offsets || !perm || !active || !n_active || !y_pairs || T <= 0 || k <= 0)
    return BRE_ERR_ARG;
  if (!weights_ok(routed, BRE_FMT_Q2_K_R16)) return BRE_ERR_ARG;
  if (shared && (!weights_ok(shared, BRE_FMT_Q8_0) || shared->n_experts != 1 || !y_shared)) return BRE_ERR_ARG;
  if (!aligned(x_bf16, 16) || !aligned(y_pairs, 16) || (y_shared && !aligned(y_shared, 16))) return BRE_ERR_ARG;
  bre_status st = ffn_check_shapes(routed, shared, T);
  if (st != BRE_OK) return st;
  const int Fs = shared ? shared->d_ff : 0;
  if (!ws || !aligned(ws, 256) || ws_bytes < ffn_ws_bytes(T, k, routed->n_experts, routed->d, routed->d_ff, Fs))
    return BRE_ERR_WORKSPACE;
  FfnArgs a{routed, shared, static_cast<const uint16_t*>(x_bf16), T, k, offsets, perm, active, n_active,
            y_pairs, y_shared, ws, ws_bytes, dev_err};
  return cuda_status(launch_ffn(a, reinterpret_cast<cudaStream_t>(stream)));
}

bre_status moe_combine(const float* y_pairs, const float* topk_w, const int32_t* inv, const int32_t* offsets, int E,
                       const float* y_shared, int T, int k, int d, void* out_bf16, float* out_f32,
                       bre_stream_t stream) {
  if (!y_pairs || !topk_w || !inv || !offsets || !out_bf16 || T <= 0 || k <= 0 || d <= 0 || E <= 0) return BRE_ERR_ARG;
  if (d % 8 != 0) return BRE_ERR_UNSUPPORTED;
  if (!aligned(y_pairs, 16) || !aligned(out_bf16, 16) || (y_shared && !aligned(y_shared, 16)) ||
      (out_f32 && !aligned(out_f32, 16)))
    return BRE_ERR_ARG;
  return cuda_status(launch_combine(y_pairs, topk_w, inv, offsets, E, y_shared, T, k, d,
                                    static_cast<uint16_t*>(out_bf16), out_f32, reinterpret_cast<cudaStream_t>(stream)));
}

bre_status moe_residual_norm(const void* x_bf16, const void* moe_bf16, int T, int d, float scale, float eps,
                             void* x_out_bf16, void* u_out_bf16, bre_stream_t stream) {
  if (!x_bf16 || !moe_bf16 || !x_out_bf16 || T <= 0 || d <= 0) return BRE_ERR_ARG;
  if ((size_t)d * 4 > (size_t)device_max_smem_optin()) return BRE_ERR_UNSUPPORTED;
  return cuda_status(launch_residual_norm(static_cast<const uint16_t*>(x_bf16), static_cast<const uint16_t*>(moe_bf16), T,
                                          d, scale, eps, static_cast<uint16_t*>(x_out_bf16),
                                          static_cast<uint16_t*>(u_out_bf16), reinterpret_cast<cudaStream_t>(stream)));
}

bre_status engram_gather_decode(const uint8_t* const* tables, const int64_t* n_rows, int n_tables,
                                const int64_t* row_ids, int T, int H, void* out_bf16, int32_t* dev_err,
                                bre_stream_t stream) {
  if (!tables || !n_rows || !row_ids || !out_bf16 || T <= 0 || H <= 0 || n_tables <= 0) return BRE_ERR_ARG;
  if (n_tables > 8 || H > 64) return BRE_ERR_UNSUPPORTED;
  if (!aligned(out_bf16, 16) || !aligned(row_ids, 8)) return BRE_ERR_ARG;
  EngramTables tabs{};
  for (int i = 0; i < n_tables; ++i) {
    if (!tables[i] || n_rows[i] < 0 || !aligned(tables[i], 8)) return BRE_ERR_ARG;
    tabs.ptr[i] = tables[i];
    tabs.n_rows[i] = n_rows[i];
  }
  return cuda_status(launch_engram(tabs, n_tables, row_ids, T, H, static_cast<uint16_t*>(out_bf16), dev_err,
                                   reinterpret_cast<cudaStream_t>(stream)));
}

size_t engram_inject_workspace(int T, int R, int W) {
  return (T > 0 && R > 0 && W > 0) ? engram_inject_ws_bytes(T, R, W) : 0;
}

bre_status engram_inject(const uint8_t* table, int64_t n_rows, const int64_t* row_ids, int R, const void* w_kv_bf16,
                         int W, void* resid_bf16, const float* q_norm, const float* k_norm, const uint8_t* mask, int T,
                         float eps, float* kv_out, float* gate_out, int32_t* dev_err, void* ws, size_t ws_bytes,
                         bre_stream_t stream) {
  if (!table || !row_ids || !w_kv_bf16 || !resid_bf16 || !q_norm || !k_norm || T <= 0 || R <= 0 || W <= 0 ||
      n_rows <= 0 || !(eps >= 0.0f))
    return BRE_ERR_ARG;
  if (W % 16 != 0 || W > 8192 || R > 24) return BRE_ERR_UNSUPPORTED;
  if (!aligned(table, 8) || !aligned(row_ids, 8) || !aligned(w_kv_bf16, 16) || !aligned(resid_bf16, 2) ||
      !aligned(q_norm, 4) || !aligned(k_norm, 4) || (kv_out && !aligned(kv_out, 4)) ||
      (gate_out && !aligned(gate_out, 4)))
    return BRE_ERR_ARG;
  if (!ws || ws_bytes < engram_inject_ws_bytes(T, R, W) || !aligned(ws, 256)) return BRE_ERR_WORKSPACE;
  return cuda_status(launch_engram_inject(table, n_rows, row_ids, R, static_cast<const uint16_t*>(w_kv_bf16), W,
                                          static_cast<uint16_t*>(resid_bf16), q_norm, k_norm, mask, T, eps, kv_out,
                                          gate_out, dev_err, ws, reinterpret_cast<cudaStream_t>(stream)));
}

bre_status bre_set_ffn_wait_limit(int64_t cycles) {
  if (cycles < 0) return BRE_ERR_ARG;
  g_ffn_wait.store((long long)cycles, std::memory_order_relaxed);
  return BRE_OK;
}

bre_status bre_repack_q2k_r16(const void* src, void* dst, int n_matrices, int rows, int cols, int64_t src_stride,
                              int64_t dst_stride, bre_stream_t stream) {
  if (!src || !dst || n_matrices <= 0 || rows <= 0 || cols <= 0) return BRE_ERR_ARG;
  if (rows % 16 || cols % 256) return BRE_ERR_UNSUPPORTED;
  const int64_t bytes = (int64_t)rows * (cols / 256) * 84;
  if (n_matrices > 1 && (src_stride < bytes || dst_stride < bytes)) return BRE_ERR_ARG;
  if (!aligned(src, 16) || !aligned(dst, 16) || src_stride % 16 || dst_stride % 16) return BRE_ERR_ARG;
  return cuda_status(launch_repack_q2k_r16(static_cast<const uint8_t*>(src), static_cast<uint8_t*>(dst), n_matrices,
                                           rows, cols, n_matrices > 1 ? src_stride : bytes,
                                           n_matrices > 1 ? dst_stride : bytes, reinterpret_cast<cudaStream_t>(stream)));
}

bre_status bre_dequant(int fmt, const void* blocks, int64_t n_blocks, float* out, bre_stream_t stream) {
  if (!blocks || !out || n_blocks <= 0) return BRE_ERR_ARG;
  if (fmt != BRE_FMT_Q2_K && fmt != BRE_FMT_Q8_0) return BRE_ERR_UNSUPPORTED;
  return cuda_status(launch_dequant(fmt, static_cast<const uint8_t*>(blocks), n_blocks, out,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
