// noalloc.cu -- mamba_scan_fwd_noalloc: the prefill scan for callers that
// cannot call cudaMalloc (a plugin whose host framework owns every byte of
// device memory through its own pool, or a latency-critical path that must not
// take cudaMalloc's implicit synchronisation).  Instead of a caller-provided
// workspace it uses one fixed array that the library itself holds in device
// memory; everything else is mamba_scan_fwd, unchanged.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <mutex>

#include "../../include/mamba_ssm.h"

namespace {

constexpr size_t kScratchBytes = MAMBA_NOALLOC_SCRATCH_BYTES;

// The scratch.  Every GPU that loads the library holds these bytes until the
// process exits.  In host code this name is only a stand-in for the device
// array, never a usable address: the device address is looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// The array's address is a property of the CUDA context the module is loaded
// into, not of the device: a plugin may run its own (non-primary) context,
// and cudaDeviceReset replaces the primary one (the module is loaded again,
// possibly elsewhere).  So the address is remembered per context, keyed by
// the context's unique id (never reused within a process, unlike the handle).
typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

struct DriverFns {
  CtxGetCurrentFn get_current = nullptr;
  CtxGetIdFn get_id = nullptr;
};

const DriverFns& driver_fns() {
  static DriverFns f;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_current = reinterpret_cast<CtxGetCurrentFn>(p);
    p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      f.get_id = reinterpret_cast<CtxGetIdFn>(p);
  });
  return f;
}

struct Entry {
  unsigned long long ctx_id;
  void* addr;
};
constexpr int kCacheEntries = 64;
std::mutex g_mutex;
Entry g_cache[kCacheEntries];
int g_used = 0;

// Unique id of the calling thread's current context (false: none current, or
// the driver does not answer).
bool current_context_id(unsigned long long* id) {
  const DriverFns& f = driver_fns();
  if (!f.get_current || !f.get_id) return false;
  CUcontext ctx = nullptr;
  if (f.get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
  return f.get_id(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch in the current context.  The first call in a
// context looks it up with cudaGetSymbolAddress (which also makes the
// runtime's context current when none was) and remembers it; later calls in
// that context take the remembered address.  Nothing here allocates.
mamba_status scratch_address(void** out) {
  unsigned long long id = 0;
  const bool have_id = current_context_id(&id);
  if (have_id) {
    std::lock_guard<std::mutex> lock(g_mutex);
    for (int i = 0; i < g_used; ++i)
      if (g_cache[i].ctx_id == id) {
        *out = g_cache[i].addr;
        return MAMBA_OK;
      }
  }
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return MAMBA_ERR_CUDA;
  // the lookup may have created the context: take its id now
  if (have_id || current_context_id(&id)) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_used < kCacheEntries) g_cache[g_used++] = Entry{id, p};  // a full table: look up every call
  }
  *out = p;
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
