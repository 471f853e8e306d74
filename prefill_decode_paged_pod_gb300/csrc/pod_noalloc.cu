// pod_noalloc.cu — run a POD plan without any device allocation by the caller.
//
// Some callers cannot call cudaMalloc: plugins whose host application owns all
// device memory through its own pool and forbids direct allocation, processes
// that run under a fixed device-memory budget where a late allocation can
// fail, and serving loops that cannot afford the implicit synchronisation of
// cudaMalloc/cudaFree. For them the scratch the POD kernels need (plan
// metadata, split partials, device status word) lives in the fixed array
// below, which every GPU that loads this library holds until the process exits.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "../../include/pod.h"

void pod_set_last_error(const std::string& msg);

#define POD_STATIC_SCRATCH_BYTES (32u << 20)  // 32 MiB

static __device__ __align__(256) unsigned char g_pod_static_scratch[POD_STATIC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the static array on the current device. The host-side
// name of the array is only a stand-in, so the address must be asked for once
// per device, with that device current.
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_pod_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" {

size_t pod_static_scratch_capacity(void) { return (size_t)POD_STATIC_SCRATCH_BYTES; }

pod_status pod_run_static_scratch(pod_handle h, const void* q_p, const void* kv_p,
                                  const void* q_d, const void* kv_d, const float* sinks,
                                  void* out_p, float* lse_p, void* out_d, float* lse_d,
                                  void* stream) {
  if (!h) {
    pod_set_last_error("handle is NULL");
    return POD_ERR_INVALID_ARG;
  }
  const size_t need = pod_workspace_size(h);
  if (need > (size_t)POD_STATIC_SCRATCH_BYTES) {
    pod_set_last_error("plan needs " + std::to_string(need) +
                       " bytes of scratch; the static scratch holds " +
                       std::to_string((size_t)POD_STATIC_SCRATCH_BYTES) +
                       " (use pod_run with a caller-allocated workspace)");
    return POD_ERR_WORKSPACE;
  }
  void* scratch = nullptr;
  cudaError_t e = scratch_address(&scratch);
  if (e != cudaSuccess) {
    pod_set_last_error(std::string("static scratch set-up failed: ") + cudaGetErrorString(e));
    return POD_ERR_CUDA;
  }
  // Upload this plan's metadata (status word zeroed) into the shared array,
  // then run the existing launch path on it.
  pod_status st = pod_bind_workspace(h, scratch, POD_STATIC_SCRATCH_BYTES, stream);
  if (st != POD_OK) return st;
  return pod_run(h, q_p, kv_p, q_d, kv_d, sinks, scratch, out_p, lse_p, out_d, lse_d, stream);
}

}  // extern "C"
