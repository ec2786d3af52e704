// Internal launcher declarations of libbre (host side).
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bre.h"

namespace bre {

struct EngramTables {
  const uint8_t* ptr[8];
  long long n_rows[8];
};

cudaError_t launch_engram(const EngramTables& tabs, int n_tables, const int64_t* ids, int T, int H, uint16_t* out,
                          int32_t* err, cudaStream_t s);
size_t engram_inject_ws_bytes(int T, int R, int W);
cudaError_t launch_engram_inject(const uint8_t* table, long long n_rows, const int64_t* row_ids, int R,
                                 const uint16_t* w_kv, int W, uint16_t* resid, const float* q_norm,
                                 const float* k_norm, const uint8_t* mask, int T, float eps, float* kv_out,
                                 float* gate_out, int32_t* err, void* ws, cudaStream_t s);

// router
size_t route_ws_bytes(int T, int E);
cudaError_t launch_route(const uint16_t* x, const float* w_r, const float* bias, int T, int d, int E, int k,
                         int32_t* ids, float* w, void* ws, cudaStream_t s);
cudaError_t launch_route_ex(const uint16_t* x, const float* w_r, const float* bias, int T, int d, int E, int k,
                            int score, const float* vision_bias, const uint8_t* is_media, const int32_t* tid2eid,
                            const int32_t* token_ids, int vocab, int32_t* ids, float* w, int32_t* err, void* ws,
                            cudaStream_t s);
// scratch (device, >= ceil(T k / 1024) (E + 1) int32) lets more than 1,024 pairs be permuted by
// three grid-wide launches instead of one CTA; without it (or when too small) one CTA does all
cudaError_t launch_permute(const int32_t* ids, int T, int k, int E, int32_t* offsets, int32_t* perm, int32_t* inv,
                           int32_t* active, int32_t* n_active, int32_t* err, cudaStream_t s, void* scratch = nullptr,
                           size_t scratch_bytes = 0);
// route, then permute; for small batches the router kernel's last CTA (the one that merges every
// token) permutes too
cudaError_t launch_route_permute(const uint16_t* x, const float* w_r, const float* bias, int T, int d, int E, int k,
                                 int32_t* ids, float* w, int32_t* offsets, int32_t* perm, int32_t* inv,
                                 int32_t* active, int32_t* n_active, int32_t* err, void* ws, cudaStream_t s);

// expert FFN
struct FfnArgs {
  const bre_ffn_weights* routed;
  const bre_ffn_weights* shared;
  const uint16_t* x;
  int T, k;
  const int32_t* offsets;
  const int32_t* perm;
  const int32_t* active;
  const int32_t* n_active;
  float* y_pairs;
  float* y_shared;
  void* ws;
  size_t ws_bytes;
  int32_t* err;
};
constexpr int DECODE_T_MAX = 8;   // larger batches take the grouped-GEMM path
// Leading bytes of the FFN workspace that hold the decode path's item counters and tail
// position (set by every decode call); both paths place everything else after them.
size_t ffn_reserved_bytes(int k, int d, int F, int Fs);
size_t ffn_ws_bytes(int T, int k, int E, int d, int F, int Fs);
size_t ffn_gemm_ws_bytes(int T, int k, int d, int F, int Fs);
bre_status ffn_check_shapes(const bre_ffn_weights* routed, const bre_ffn_weights* shared, int T);
cudaError_t launch_ffn(const FfnArgs& a, cudaStream_t s);
cudaError_t launch_gemm(const FfnArgs& a, cudaStream_t s);

cudaError_t launch_combine(const float* y_pairs, const float* topk_w, const int32_t* inv, const int32_t* offsets,
                           int E, const float* y_shared, int T, int k, int d, uint16_t* out, float* out_f32,
                           cudaStream_t s);
cudaError_t launch_residual_norm(const uint16_t* x, const uint16_t* moe, int T, int d, float scale, float eps,
                                 uint16_t* x_out, uint16_t* u_out, cudaStream_t s);
cudaError_t launch_dequant(int fmt, const uint8_t* blocks, int64_t n_blocks, float* out, cudaStream_t s);
// Q2_K [n_mat][rows][cols/256 blocks] -> Q2_K_R16 (repack.cu)
cudaError_t launch_repack_q2k_r16(const uint8_t* src, uint8_t* dst, long long n_mat, int rows, int cols,
                                  long long src_stride, long long dst_stride, cudaStream_t s);

// tiled tensor map over global memory: dims innermost first, strides (bytes) of dims 1..rank-1
bool encode_tiled(CUtensorMap* m, CUtensorMapDataType type, int rank, const void* base, const uint64_t* dims,
                  const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swizzle);

// Launch with programmatic dependent launch allowed: the kernel may be scheduled while the
// previous kernel on the stream drains, so every kernel launched this way calls pdl_wait()
// before it reads another kernel's results or writes memory an earlier kernel may still read.
template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Budget (SM clock cycles) of the expert FFN kernels' pipeline waits: the value set by
// bre_set_ffn_wait_limit, or dflt when none is set.  The waits that drain a kernel's own copies
// before it exits always use the default budget.
long long ffn_wait_budget(long long dflt);

// device attributes (cached per device)
int device_sm_count();
int device_max_smem_optin();

}  // namespace bre
