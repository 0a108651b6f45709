// moe_route_permute without a caller-provided workspace, for callers that
// cannot allocate device memory (see include/nvfp4moe.h).  The scratch lives
// in a fixed array reserved in every device's memory when the library loads.
#include "../../include/nvfp4moe.h"
#include "internal.h"

#include <cstdio>
#include <mutex>

namespace nvf {
void set_last_error(const char* msg);
nvf_status route_precheck(int32_t T, int32_t E, int32_t k, int32_t shared);
}

namespace {

constexpr size_t kScratchBytes = NVF_ROUTE_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a host-side handle: its
// device address must be looked up per device before it is handed to a kernel.
static __device__ __align__(256) unsigned char g_route_scratch[kScratchBytes];

std::mutex g_mu;
void* g_addr[kMaxDevices] = {};

// Device address of the scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_addr[dev] == nullptr) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" nvf_status moe_route_permute_noalloc(const float* logits, const float* bias, int32_t T, int32_t E,
                                                int32_t k, int32_t renormalize, int32_t shared_expert,
                                                int32_t* topk_ids, float* topk_w, int32_t* expert_offsets,
                                                int32_t* tile_offsets, int32_t* perm_to_src, int32_t* src_to_perm,
                                                int32_t* perm_token, void* stream) {
  // Device and argument checks first, exactly as the workspace entry point makes them.
  nvf_status st = nvf::route_precheck(T, E, k, shared_expert);
  if (st != NVF_OK) return st;
  size_t need = 0;
  st = moe_route_permute_workspace_size(T, E, &need);
  if (st != NVF_OK) return st;
  if (need > kScratchBytes) {
    char msg[256];
    std::snprintf(msg, sizeof(msg),
                  "moe_route_permute_noalloc: T=%d, E=%d needs %zu bytes of scratch, more than the fixed %zu; "
                  "use moe_route_permute with a workspace",
                  T, E, need, kScratchBytes);
    nvf::set_last_error(msg);
    return NVF_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    char msg[256];
    std::snprintf(msg, sizeof(msg), "moe_route_permute_noalloc: device address of the scratch: %s",
                  cudaGetErrorString(e));
    nvf::set_last_error(msg);
    return NVF_ERR_CUDA;
  }
  return moe_route_permute(logits, bias, T, E, k, renormalize, shared_expert, topk_ids, topk_w, expert_offsets,
                           tile_offsets, perm_to_src, src_to_perm, perm_token, scratch, kScratchBytes, stream);
}
