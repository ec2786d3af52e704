// moe_route_static: the router with its scratch in a fixed device array instead of a
// caller-provided workspace, for callers that cannot allocate device memory.
//
// Who needs it: serving loops that may not call cudaMalloc on the hot path because it can
// synchronise the whole device and stall every stream, and host integrations (plugins, runtimes
// that own the allocator) that are handed only pre-allocated input and output buffers and have
// no way to ask for scratch.  This call allocates nothing: it neither calls cudaMalloc/cudaFree
// nor any library routine that allocates.
//
// The scratch is one file-scope device array of ROUTE_STATIC_SCRATCH bytes (about 388 KB),
// loaded with the library and held by every GPU that loads it until the process exits.  All calls share
// it, so calls that overlap on the GPU (other streams, other host threads) race and must be
// ordered by the caller.  The selection tickets at its start must be zero before a call; they are
// cleared with a memset on the caller's stream at every call.
#include <cuda_runtime.h>

#include <mutex>

#include "bre.h"
#include "kernels.h"

namespace {

// tickets, then either the scores of a large batch (T*E floats) or, for a small batch (at most
// 32 tokens), the selection candidates (1024 expert slots x 12 bytes a token) followed by the hash
// rows' table scores (32 floats a token): the largest moe_route_workspace of any shape the call
// accepts (T * E <= BRE_ROUTE_STATIC_MAX_TE, E <= 1024), less its 256-byte ticket area
constexpr size_t ROUTE_STATIC_SCORES = (size_t)BRE_ROUTE_STATIC_MAX_TE * sizeof(float);
constexpr size_t ROUTE_STATIC_CANDIDATES = (size_t)32 * 1024 * 12 + (size_t)32 * 32 * 4;
constexpr size_t ROUTE_STATIC_SCRATCH =
    256 + (ROUTE_STATIC_SCORES > ROUTE_STATIC_CANDIDATES ? ROUTE_STATIC_SCORES : ROUTE_STATIC_CANDIDATES);

static __device__ __align__(256) unsigned char g_route_scratch[ROUTE_STATIC_SCRATCH];

std::mutex g_mu;
void* g_scratch_ptr[64] = {};

// Device address of the scratch array on the current device (looked up once per device;
// in host code the array's name is only a stand-in and must not be passed to a kernel).
cudaError_t scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" bre_status moe_route_static(const void* x_bf16, const float* w_r, const float* bias, int T, int d, int E,
                                       int k, int32_t* topk_ids, float* topk_w, bre_stream_t stream) {
  if (!x_bf16 || !w_r || !topk_ids || !topk_w || T <= 0 || d <= 0 || E <= 0 || k <= 0) return BRE_ERR_ARG;
  if (k > E || k > 32 || E > 1024 || d % 32 != 0) return BRE_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(x_bf16) % 16 || reinterpret_cast<uintptr_t>(w_r) % 16) return BRE_ERR_ARG;
  if ((long long)T * E > BRE_ROUTE_STATIC_MAX_TE) return BRE_ERR_WORKSPACE;   // beyond the fixed scratch
  if (bre::route_ws_bytes(T, E) > ROUTE_STATIC_SCRATCH) return BRE_ERR_WORKSPACE;
  void* scratch = nullptr;
  if (scratch_for_current_device(&scratch) != cudaSuccess) return BRE_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, 256, s) != cudaSuccess) return BRE_ERR_CUDA;   // the ticket
  return bre::launch_route(static_cast<const uint16_t*>(x_bf16), w_r, bias, T, d, E, k, topk_ids, topk_w, scratch, s) ==
                 cudaSuccess
             ? BRE_OK
             : BRE_ERR_CUDA;
}
