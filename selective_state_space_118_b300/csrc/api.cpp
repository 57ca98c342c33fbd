// api.cpp -- the C ABI of libmamba_ssm.so (declared in include/mamba_ssm.h):
// argument checks, the chunking plan, tensor-map encoding and kernel launches.
// Never allocates, frees or synchronises (except mamba_last_error).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/mamba_ssm.h"
#include "launch.h"

using mamba::IoType;

namespace {

constexpr int kT = 64;   // tokens per tile (multiple of every chunk)
constexpr int kCT = 16;  // channels per CTA
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) return 148;
  return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t esize(mamba_dtype io) { return io == MAMBA_BF16 ? 2 : 4; }

size_t round256(size_t v) { return (v + 255) & ~size_t(255); }

// The chunking plan: how many chunks of how many tokens.
struct Plan {
  int n_chunks;
  int chunk_len;
};

Plan make_plan(int batch, int seqlen, int d_inner, int n_chunks_req) {
  Plan pl{1, seqlen};
  if (seqlen <= 0) return pl;
  const int tiles = (seqlen + kT - 1) / kT;
  int n = n_chunks_req;
  if (n <= 0) {
    // Enough CTAs for ~4 per SM; each chunk keeps at least 4 tiles.
    const long ctas = (long)batch * (d_inner / kCT);
    const long target = 4L * sm_count();
    n = ctas >= (3 * target) / 4 ? 1 : (int)((target + ctas - 1) / ctas);
    const int max_by_len = tiles / 4 > 0 ? tiles / 4 : 1;
    if (n > max_by_len) n = max_by_len;
  }
  if (n > tiles) n = tiles;
  if (n < 1) n = 1;
  const int tiles_per_chunk = (tiles + n - 1) / n;
  pl.chunk_len = tiles_per_chunk * kT;
  pl.n_chunks = (tiles + tiles_per_chunk - 1) / tiles_per_chunk;
  if (pl.n_chunks == 1) pl.chunk_len = seqlen;
  return pl;
}

struct Workspace {
  size_t bc, carry, hloc, sum_dt, counters, total;
};

// bc: B and C widened to fp32 and interleaved, (B, L, 32); then, in chunked
// mode only, the carries, chunk summaries and arrival counters.
Workspace workspace_layout(int batch, int seqlen, int d_inner, const Plan& pl) {
  Workspace w{0, 0, 0, 0, 0, 0};
  const size_t B = batch, L = seqlen, D = d_inner, n = pl.n_chunks;
  w.bc = 0;
  w.total = round256(B * L * 32 * sizeof(float));
  if (pl.n_chunks <= 1) return w;
  w.carry = w.total;
  w.hloc = round256(w.carry + B * n * D * 16 * sizeof(float));
  w.sum_dt = round256(w.hloc + B * (n - 1) * D * 16 * sizeof(float));
  w.counters = round256(w.sum_dt + B * (n - 1) * D * sizeof(float));
  w.total = round256(w.counters + B * (D / kCT) * sizeof(unsigned));
  return w;
}

// 3-D tiled map over a (B, L, inner) row-major tensor: box (box_inner, 64, 1).
bool encode3d(CUtensorMap* m, const void* base, mamba_dtype io, int inner, int L, int B,
              int box_inner = 16) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const size_t es = esize(io);
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)L, (cuuint64_t)B};
  cuuint64_t strides[2] = {(cuuint64_t)inner * es, (cuuint64_t)inner * es * (cuuint64_t)L};
  cuuint32_t box[3] = {(cuuint32_t)box_inner, (cuuint32_t)kT, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, io == MAMBA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3,
                  const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

mamba_status check_common(int batch, int d_inner, int d_state, int d_conv, mamba_dtype io) {
  if (batch <= 0 || d_inner <= 0) return MAMBA_ERR_INVALID_ARG;
  if (io != MAMBA_F32 && io != MAMBA_BF16) return MAMBA_ERR_UNSUPPORTED;
  if (d_state != MAMBA_D_STATE || d_conv != MAMBA_D_CONV) return MAMBA_ERR_UNSUPPORTED;
  if (d_inner % kCT != 0) return MAMBA_ERR_UNSUPPORTED;
  return MAMBA_OK;
}

}  // namespace

extern "C" {

int mamba_abi_version(void) { return 100; }

const char* mamba_status_string(mamba_status s) {
  switch (s) {
    case MAMBA_OK: return "ok";
    case MAMBA_ERR_INVALID_ARG: return "invalid argument";
    case MAMBA_ERR_UNSUPPORTED: return "unsupported configuration";
    case MAMBA_ERR_CUDA: return "CUDA error";
    case MAMBA_ERR_TIMEOUT: return "device-side wait timed out";
    case MAMBA_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

int mamba_scan_default_chunks(int batch, int seqlen, int d_inner) {
  if (batch <= 0 || seqlen <= 0 || d_inner <= 0 || d_inner % kCT) return 1;
  return make_plan(batch, seqlen, d_inner, 0).n_chunks;
}

size_t mamba_scan_workspace_size(int batch, int seqlen, int d_inner, int n_chunks) {
  if (batch <= 0 || seqlen <= 0 || d_inner <= 0 || d_inner % kCT) return 0;
  return workspace_layout(batch, seqlen, d_inner, make_plan(batch, seqlen, d_inner, n_chunks)).total;
}

mamba_status mamba_scan_fwd(const mamba_scan_args* a, void* stream_v) {
  if (!a) return MAMBA_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_v);
  mamba_status st = check_common(a->batch, a->d_inner, a->d_state, a->d_conv, a->io);
  if (st != MAMBA_OK) return st;
  if (a->seqlen < 0 || a->n_chunks < 0) return MAMBA_ERR_INVALID_ARG;
  if (!a->A_log || !a->Dskip || !a->conv_w) return MAMBA_ERR_INVALID_ARG;
  const void* aligned_ptrs[] = {a->A_log, a->Dskip, a->conv_w, a->conv_b, a->h0, a->conv_state0,
                                a->final_h, a->final_conv_state};
  for (const void* p : aligned_ptrs)
    if (p && !aligned16(p)) return MAMBA_ERR_INVALID_ARG;

  const size_t B = a->batch, D = a->d_inner, es = esize(a->io);
  if (a->seqlen == 0) {
    // Nothing to scan: the final state is the initial one.
    if (a->final_h && a->final_h != a->h0) {
      cudaError_t e = a->h0 ? cudaMemcpyAsync(a->final_h, a->h0, B * D * 16 * sizeof(float),
                                              cudaMemcpyDeviceToDevice, stream)
                            : cudaMemsetAsync(a->final_h, 0, B * D * 16 * sizeof(float), stream);
      if (e != cudaSuccess) return MAMBA_ERR_CUDA;
    }
    if (a->final_conv_state && a->final_conv_state != a->conv_state0) {
      cudaError_t e = a->conv_state0 ? cudaMemcpyAsync(a->final_conv_state, a->conv_state0, B * 3 * D * es,
                                                       cudaMemcpyDeviceToDevice, stream)
                                     : cudaMemsetAsync(a->final_conv_state, 0, B * 3 * D * es, stream);
      if (e != cudaSuccess) return MAMBA_ERR_CUDA;
    }
    return MAMBA_OK;
  }

  const void* io_ptrs[] = {a->x, a->z, a->dt_raw, a->Bm, a->Cm, a->y};
  for (const void* p : io_ptrs)
    if (!p || !aligned16(p)) return MAMBA_ERR_INVALID_ARG;
  if ((long long)a->seqlen * (long long)D > (1LL << 40)) return MAMBA_ERR_UNSUPPORTED;

  const Plan pl = make_plan(a->batch, a->seqlen, a->d_inner, a->n_chunks);
  const Workspace ws = workspace_layout(a->batch, a->seqlen, a->d_inner, pl);

  if (!a->workspace || a->workspace_bytes < ws.total) return MAMBA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0) return MAMBA_ERR_INVALID_ARG;
  char* wsp = static_cast<char*>(a->workspace);
  float* bc = reinterpret_cast<float*>(wsp + ws.bc);

  // x, z, dt_raw, bc, y
  CUtensorMap maps[5];
  const void* bases[5] = {a->x, a->z, a->dt_raw, bc, a->y};
  for (int i = 0; i < 5; ++i) {
    const bool is_bc = i == 3;
    if (!encode3d(&maps[i], bases[i], is_bc ? MAMBA_F32 : a->io, is_bc ? 32 : a->d_inner, a->seqlen,
                  a->batch, is_bc ? 32 : 16))
      return MAMBA_ERR_CUDA;
  }

  mamba::ScanParams p;
  std::memset(&p, 0, sizeof(p));
  p.batch = a->batch;
  p.seqlen = a->seqlen;
  p.d_inner = a->d_inner;
  p.chunk_len = pl.chunk_len;
  p.n_chunks = pl.n_chunks;
  p.A_log = a->A_log;
  p.Dskip = a->Dskip;
  p.conv_w = a->conv_w;
  p.conv_b = a->conv_b;
  p.h0 = a->h0;
  p.conv_state0 = a->conv_state0;
  p.x = a->x;
  p.final_h = a->final_h;
  p.final_conv_state = a->final_conv_state;
  p.flags = a->flags;
  p.timeout_ns = a->wait_timeout_ns ? a->wait_timeout_ns : kDefaultTimeoutNs;
  const IoType io = a->io == MAMBA_BF16 ? IoType::BF16 : IoType::F32;

  if (mamba::launch_bc_widen(io, a->Bm, a->Cm, bc, (long)B * a->seqlen, stream) != cudaSuccess)
    return MAMBA_ERR_CUDA;
  if (pl.n_chunks > 1) {
    p.carry = reinterpret_cast<float*>(wsp + ws.carry);
    p.hloc = reinterpret_cast<float*>(wsp + ws.hloc);
    p.sum_dt = reinterpret_cast<float*>(wsp + ws.sum_dt);
    p.counters = reinterpret_cast<unsigned*>(wsp + ws.counters);
    if (cudaMemsetAsync(p.counters, 0, B * (D / kCT) * sizeof(unsigned), stream) != cudaSuccess)
      return MAMBA_ERR_CUDA;
    const CUtensorMap smaps[3] = {maps[0], maps[2], maps[3]};  // x, dt_raw, bc
    dim3 g1((unsigned)(D / kCT), (unsigned)B, (unsigned)(pl.n_chunks - 1));
    if (mamba::launch_summary(io, smaps, p, g1, stream) != cudaSuccess) return MAMBA_ERR_CUDA;
  }
  dim3 g2((unsigned)(D / kCT), (unsigned)B, (unsigned)pl.n_chunks);
  if (mamba::launch_scan(io, maps, p, g2, stream) != cudaSuccess) return MAMBA_ERR_CUDA;
  return MAMBA_OK;
}

mamba_status mamba_step(const mamba_step_args* a, void* stream_v) {
  if (!a) return MAMBA_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_v);
  mamba_status st = check_common(a->batch, a->d_inner, a->d_state, a->d_conv, a->io);
  if (st != MAMBA_OK) return st;
  const void* req[] = {a->h, a->conv_state, a->x_t, a->z_t, a->dt_raw_t, a->B_t, a->C_t,
                       a->A_log, a->Dskip, a->conv_w, a->y_t};
  for (const void* p : req)
    if (!p) return MAMBA_ERR_INVALID_ARG;
  const void* al[] = {a->h, a->A_log, a->conv_w, a->conv_b};
  for (const void* p : al)
    if (p && !aligned16(p)) return MAMBA_ERR_INVALID_ARG;
  mamba::StepParams p;
  p.batch = a->batch;
  p.d_inner = a->d_inner;
  p.h = a->h;
  p.conv_state = a->conv_state;
  p.x_t = a->x_t;
  p.z_t = a->z_t;
  p.dt_raw_t = a->dt_raw_t;
  p.B_t = a->B_t;
  p.C_t = a->C_t;
  p.A_log = a->A_log;
  p.Dskip = a->Dskip;
  p.conv_w = a->conv_w;
  p.conv_b = a->conv_b;
  p.y_t = a->y_t;
  const IoType io = a->io == MAMBA_BF16 ? IoType::BF16 : IoType::F32;
  if (mamba::launch_step(io, p, stream) != cudaSuccess) return MAMBA_ERR_CUDA;
  return MAMBA_OK;
}

mamba_status mamba_last_error(void* stream_v) {
  unsigned code = 0;
  if (mamba::take_device_error(&code, reinterpret_cast<cudaStream_t>(stream_v)) != cudaSuccess)
    return MAMBA_ERR_CUDA;
  return static_cast<mamba_status>(code);
}

}  // extern "C"
