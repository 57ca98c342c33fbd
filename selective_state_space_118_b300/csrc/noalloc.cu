// noalloc.cu -- mamba_scan_fwd_noalloc: the prefill scan for callers that
// cannot call cudaMalloc (a plugin whose host framework owns every byte of
// device memory through its own pool, or a latency-critical path that must not
// take cudaMalloc's implicit synchronisation).  Instead of a caller-provided
// workspace it uses one fixed array that the library itself holds in device
// memory; everything else is mamba_scan_fwd, unchanged.
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "../../include/mamba_ssm.h"

namespace {

constexpr size_t kScratchBytes = MAMBA_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch.  Every GPU that loads the library holds these bytes until the
// process exits.  In host code this name is only a stand-in for the device
// array, never a usable address: the device address is looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and remembered.
mamba_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MAMBA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MAMBA_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return MAMBA_OK;
}

}  // namespace

extern "C" mamba_status mamba_scan_fwd_noalloc(const mamba_scan_args* args, void* stream) {
  if (args == nullptr) return MAMBA_ERR_INVALID_ARG;
  // Too large for the fixed scratch: refuse before anything runs.
  if (mamba_scan_workspace_size(args->batch, args->seqlen, args->d_inner, args->n_chunks) > kScratchBytes)
    return MAMBA_ERR_WORKSPACE;
  void* scratch = nullptr;
  const mamba_status st = scratch_address(&scratch);
  if (st != MAMBA_OK) return st;
  mamba_scan_args a = *args;
  a.workspace = scratch;
  a.workspace_bytes = kScratchBytes;
  return mamba_scan_fwd(&a, stream);
}
