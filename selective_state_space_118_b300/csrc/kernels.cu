// kernels.cu -- the one translation unit holding the device code (prefill,
// chunk carries, decode step and the sticky error word) and its launchers.
#include <cuda_bf16.h>

#include "gemm_tc.cuh"
#include "launch.h"
#include "scan_bwd.cuh"
#include "scan_complex.cuh"
#include "scan_fwd.cuh"
#include "ssd.cuh"
#include "step.cuh"

namespace mamba {

size_t scan_smem_bytes(IoType io) {
  return (io == IoType::BF16 ? sizeof(MainSmem<__nv_bfloat16>) : sizeof(MainSmem<float>)) + 128;
}

template <typename IO, bool kY>
static cudaError_t launch_scan_y(const CUtensorMap* m, const ScanParams& p, dim3 grid, cudaStream_t s) {
  const size_t smem = sizeof(MainSmem<IO>) + 128;
  cudaError_t e = cudaFuncSetAttribute(scan_fwd_kernel<IO, kY>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  scan_fwd_kernel<IO, kY><<<grid, kLanes, smem, s>>>(m[0], m[1], m[2], m[3], p);
  return cudaGetLastError();
}

// y null: the states-only pass (for the backward's checkpoints)
template <typename IO>
static cudaError_t launch_scan_t(const CUtensorMap* m, const ScanParams& p, dim3 grid, cudaStream_t s) {
  return p.y != nullptr ? launch_scan_y<IO, true>(m, p, grid, s) : launch_scan_y<IO, false>(m, p, grid, s);
}

// Launch configuration of a programmatic dependent: the kernel may start
// while the one before it in the stream drains, and waits for it
// (griddepcontrol.wait) before reading anything.
static void set_pdl(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&attr)[1]) {
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
}

template <typename IO, bool kY>
static cudaError_t launch_fused_y(const CUtensorMap* m, const ScanParams& p, unsigned ctas, cudaStream_t s) {
  const size_t smem = fused_smem_bytes<IO>() + 128;
  cudaError_t e = cudaFuncSetAttribute(scan_fused_kernel<IO, kY>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas);
  cfg.blockDim = dim3(kLanes);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  set_pdl(cfg, attr);
  return cudaLaunchKernelEx(&cfg, scan_fused_kernel<IO, kY>, m[0], m[1], m[2], m[3], p);
}

template <typename IO>
static cudaError_t launch_fused_t(const CUtensorMap* m, const ScanParams& p, unsigned ctas, cudaStream_t s) {
  return p.y != nullptr ? launch_fused_y<IO, true>(m, p, ctas, s) : launch_fused_y<IO, false>(m, p, ctas, s);
}

cudaError_t launch_scan_fused(IoType io, const CUtensorMap maps[4], const ScanParams& p, unsigned ctas,
                              cudaStream_t stream) {
  return io == IoType::BF16 ? launch_fused_t<__nv_bfloat16>(maps, p, ctas, stream)
                            : launch_fused_t<float>(maps, p, ctas, stream);
}

template <typename IO>
static cudaError_t launch_widen_t(const void* Bm, const void* Cm, float* bc, long rows, int ld, unsigned* counters,
                                  int n_counters, bool pdl, bool mode_pairs, cudaStream_t s) {
  const long n = rows * 8;
  long blocks = (n + 255) / 256;
  if (blocks > 148L * 16) blocks = 148L * 16;
  if (blocks < 1) blocks = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(256);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  if (pdl) set_pdl(cfg, attr);
  if (mode_pairs)
    return cudaLaunchKernelEx(&cfg, bc_widen_kernel<IO, true>, static_cast<const IO*>(Bm),
                              static_cast<const IO*>(Cm), bc, rows, ld, counters, n_counters);
  return cudaLaunchKernelEx(&cfg, bc_widen_kernel<IO, false>, static_cast<const IO*>(Bm), static_cast<const IO*>(Cm),
                            bc, rows, ld, counters, n_counters);
}

cudaError_t launch_bc_widen(IoType io, const void* Bm, const void* Cm, float* bc, long rows, int ld,
                            cudaStream_t stream, unsigned* counters, int n_counters, bool pdl, bool mode_pairs) {
  return io == IoType::BF16
             ? launch_widen_t<__nv_bfloat16>(Bm, Cm, bc, rows, ld, counters, n_counters, pdl, mode_pairs, stream)
             : launch_widen_t<float>(Bm, Cm, bc, rows, ld, counters, n_counters, pdl, mode_pairs, stream);
}

cudaError_t launch_scan(IoType io, const CUtensorMap maps[4], const ScanParams& p, dim3 grid,
                        cudaStream_t stream) {
  return io == IoType::BF16 ? launch_scan_t<__nv_bfloat16>(maps, p, grid, stream)
                            : launch_scan_t<float>(maps, p, grid, stream);
}

// ---------------------------------------------------------------- tensor-core GEMM
cudaError_t launch_gemm_tc(const CUtensorMap& a, const CUtensorMap& w, const CUtensorMap& c, const GemmParams& p,
                           cudaStream_t s) {
  const size_t smem = sizeof(GemmSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  // clusters of two CTAs, one 256-row tile each at a time
  const long tiles = ((p.M + 2 * kGemmBM - 1) / (2 * kGemmBM)) * (long)((p.N + p.bn - 1) / p.bn);
  const long clusters = tiles < sms / 2 ? tiles : sms / 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(2 * clusters));
  cfg.blockDim = dim3(kGemmThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel, a, w, c, p);
}

// ---------------------------------------------------------------- complex scan
template <typename IO, bool kTrap, bool kSummary>
static cudaError_t launch_complex_pass(const CUtensorMap* m, const ComplexParams& p, dim3 grid, cudaStream_t s) {
  const size_t smem = sizeof(MainSmem<IO>) + 128;
  cudaError_t e = cudaFuncSetAttribute(complex_scan_kernel<IO, kTrap, kSummary>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  complex_scan_kernel<IO, kTrap, kSummary><<<grid, kLanes, smem, s>>>(m[0], m[1], m[2], m[3], p);
  return cudaGetLastError();
}

template <typename IO, bool kTrap>
static cudaError_t launch_complex_t(const CUtensorMap* m, const ComplexParams& p, cudaStream_t s) {
  if (p.n_chunks > 1 && (p.flags & kFlagExactCarry) == 0) {  // carry walks and main pass, one launch
    const size_t smem = fused_smem_bytes<IO>() + 128;
    cudaError_t e = cudaFuncSetAttribute(complex_fused_kernel<IO, kTrap>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const unsigned ctas = (unsigned)((2 * p.n_chunks - 1) * p.n_groups * p.batch);
    complex_fused_kernel<IO, kTrap><<<ctas, kLanes, smem, s>>>(m[0], m[1], m[2], m[3], p);
    return cudaGetLastError();
  }
  if (p.n_chunks > 1) {
    cudaError_t e =
        launch_complex_pass<IO, kTrap, true>(m, p, dim3((unsigned)p.n_groups, (unsigned)p.batch, (unsigned)(p.n_chunks - 1)), s);
    if (e != cudaSuccess) return e;
    const long n = (long)p.batch * p.d_inner;
    complex_fold_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(p);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  return launch_complex_pass<IO, kTrap, false>(m, p, dim3((unsigned)p.n_groups, (unsigned)p.batch, (unsigned)p.n_chunks), s);
}

cudaError_t launch_complex(IoType io, bool trapezoidal, const CUtensorMap maps[4], const ComplexParams& p,
                           cudaStream_t stream) {
  if (io == IoType::BF16)
    return trapezoidal ? launch_complex_t<__nv_bfloat16, true>(maps, p, stream)
                       : launch_complex_t<__nv_bfloat16, false>(maps, p, stream);
  return trapezoidal ? launch_complex_t<float, true>(maps, p, stream) : launch_complex_t<float, false>(maps, p, stream);
}

// Launched with programmatic stream serialization: the kernel may be
// scheduled while the previous kernel in the stream finishes, and waits for
// it (griddepcontrol.wait) before touching memory.
cudaError_t launch_step(IoType io, const StepParams& p, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((p.d_inner + kStepChannels - 1) / kStepChannels),
                     (unsigned)p.batch);
  cfg.blockDim = dim3(kStepThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (io == IoType::BF16) return cudaLaunchKernelEx(&cfg, step_kernel<__nv_bfloat16>, p);
  return cudaLaunchKernelEx(&cfg, step_kernel<float>, p);
}

void scan_occupancy(IoType io, int* main_per_sm, int* summary_per_sm) {
  int a = 0, b = 0;
  if (io == IoType::BF16) {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, scan_fwd_kernel<__nv_bfloat16, true>, kLanes,
                                                      sizeof(MainSmem<__nv_bfloat16>) + 128) != cudaSuccess) a = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, scan_fused_kernel<__nv_bfloat16, true>, kLanes,
                                                      fused_smem_bytes<__nv_bfloat16>() + 128) != cudaSuccess) b = 0;
  } else {
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&a, scan_fwd_kernel<float, true>, kLanes,
                                                      sizeof(MainSmem<float>) + 128) != cudaSuccess) a = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, scan_fused_kernel<float, true>, kLanes,
                                                      fused_smem_bytes<float>() + 128) != cudaSuccess) b = 0;
  }
  *main_per_sm = a;
  *summary_per_sm = b;
}

template <typename IO>
static cudaError_t launch_bwd_t(const CUtensorMap* m, const BwdParams& p, dim3 grid, cudaStream_t s) {
  const size_t smem = sizeof(BwdSmem<IO>) + 128;
  cudaError_t e = cudaFuncSetAttribute(scan_bwd_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  scan_bwd_kernel<IO><<<grid, kLanes, smem, s>>>(m[0], m[1], m[2], m[3], m[4], p);
  return cudaGetLastError();
}

template <typename IO>
static cudaError_t launch_carries_t(const CUtensorMap* m, const ScanParams& fp, const BwdParams& bp,
                                   unsigned n_fwd, unsigned n_adj, cudaStream_t s) {
  const size_t smem = sizeof(CarriesSmem<IO>) + 128;
  cudaError_t e =
      cudaFuncSetAttribute(scan_carries_kernel<IO>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  scan_carries_kernel<IO><<<n_fwd + n_adj, kLanes, smem, s>>>(m[0], m[1], m[2], m[3], m[4], fp, bp, n_fwd);
  return cudaGetLastError();
}

static unsigned grid_for(long n, int threads) {
  long blocks = (n + threads - 1) / threads;
  if (blocks > 148L * 16) blocks = 148L * 16;
  if (blocks < 1) blocks = 1;
  return (unsigned)blocks;
}

cudaError_t launch_bwd(IoType io, const CUtensorMap maps[5], const BwdParams& p, dim3 grid, cudaStream_t stream) {
  return io == IoType::BF16 ? launch_bwd_t<__nv_bfloat16>(maps, p, grid, stream)
                            : launch_bwd_t<float>(maps, p, grid, stream);
}

cudaError_t launch_carries(IoType io, const CUtensorMap maps[5], const ScanParams& fp, const BwdParams& bp,
                           unsigned n_fwd, unsigned n_adj, cudaStream_t stream) {
  return io == IoType::BF16 ? launch_carries_t<__nv_bfloat16>(maps, fp, bp, n_fwd, n_adj, stream)
                            : launch_carries_t<float>(maps, fp, bp, n_fwd, n_adj, stream);
}

cudaError_t launch_bwd_finish(IoType io, const BwdParams& p, float* dB, float* dC, float* dA_log, float* dD,
                              float* dconv_w, float* dconv_b, cudaStream_t stream) {
  if (p.n_chunks > 1) {
    const long n = (long)p.batch * (p.n_chunks - 1) * p.d_inner;
    if (io == IoType::BF16)
      bwd_edges_kernel<__nv_bfloat16><<<grid_for(n, 256), 256, 0, stream>>>(p);
    else
      bwd_edges_kernel<float><<<grid_for(n, 256), 256, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const long rows = (long)p.batch * p.seqlen;
  bwd_reduce_bc_kernel<<<grid_for(rows * 8, 256), 256, 0, stream>>>(p.part_bc, p.n_groups, rows, dB, dC);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  bwd_reduce_param_kernel<<<grid_for((long)p.d_inner * 22, 256), 256, 0, stream>>>(
      p.part_param, p.batch * p.n_chunks, p.d_inner, dA_log, dD, dconv_w, dconv_b);
  return cudaGetLastError();
}

cudaError_t launch_io_to_f32(IoType io, const void* src, float* dst, long n, cudaStream_t stream) {
  if (io == IoType::BF16)
    io_to_f32_kernel<__nv_bfloat16><<<grid_for(n, 256), 256, 0, stream>>>(
        static_cast<const __nv_bfloat16*>(src), dst, n);
  else
    io_to_f32_kernel<float><<<grid_for(n, 256), 256, 0, stream>>>(static_cast<const float*>(src), dst, n);
  return cudaGetLastError();
}

// u = silu(conv(x)) for the layer's x_proj (B, L, D), the conv's inputs
// before t = 0 zero.  A thread owns one 16-byte vector of channels (8 in
// bf16) over a run of kConvRun tokens of one batch row: its conv taps stay in
// registers and the window of the last three inputs slides along, so every x
// is read once (plus three before the run) and every u written once, with
// 16-byte accesses (a warp covers 512 contiguous bytes of a row).  The
// arithmetic is the scan's own (conv4, silu), so u equals the scan's internal
// u before its rounding to the I/O dtype.
constexpr int kConvRun = 32;

template <typename IO>
__global__ void __launch_bounds__(128) conv_silu_kernel(const IO* __restrict__ x, const float* __restrict__ conv_w,
                                                        const float* __restrict__ conv_b, IO* __restrict__ u,
                                                        int L, int D) {
  constexpr int kV = 16 / sizeof(IO);  // channels per 16-byte vector
  const int c0 = (blockIdx.x * blockDim.x + threadIdx.x) * kV;
  if (c0 >= D) return;
  const int b = blockIdx.z;
  const int t0 = blockIdx.y * kConvRun;
  const int t1 = min(t0 + kConvRun, L);
  float4 w[kV];
  float bias[kV];
#pragma unroll
  for (int v = 0; v < kV; ++v) {
    w[v] = __ldg(reinterpret_cast<const float4*>(conv_w + (size_t)(c0 + v) * 4));
    bias[v] = conv_b ? __ldg(conv_b + c0 + v) : 0.0f;
  }
  const IO* xr = x + (size_t)b * L * D + c0;
  IO* ur = u + (size_t)b * L * D + c0;
  float m3[kV], m2[kV], m1[kV];
  {
    IO in[3][kV];
#pragma unroll
    for (int k = 0; k < 3; ++k) {
      const int t = t0 - 3 + k;
      if (t >= 0) {
        *reinterpret_cast<uint4*>(&in[k][0]) = __ldg(reinterpret_cast<const uint4*>(xr + (size_t)t * D));
      } else {
#pragma unroll
        for (int v = 0; v < kV; ++v) in[k][v] = from_f32<IO>(0.0f);
      }
    }
#pragma unroll
    for (int v = 0; v < kV; ++v) {
      m3[v] = to_f32(in[0][v]);
      m2[v] = to_f32(in[1][v]);
      m1[v] = to_f32(in[2][v]);
    }
  }
  for (int t = t0; t < t1; ++t) {
    IO in[kV], out[kV];
    *reinterpret_cast<uint4*>(in) = __ldg(reinterpret_cast<const uint4*>(xr + (size_t)t * D));
#pragma unroll
    for (int v = 0; v < kV; ++v) {
      const float x0 = to_f32(in[v]);
      out[v] = from_f32<IO>(silu(conv4(w[v], bias[v], m3[v], m2[v], m1[v], x0)));
      m3[v] = m2[v];
      m2[v] = m1[v];
      m1[v] = x0;
    }
    *reinterpret_cast<uint4*>(ur + (size_t)t * D) = *reinterpret_cast<const uint4*>(out);
  }
}

cudaError_t launch_conv_silu(IoType io, const void* x, const float* conv_w, const float* conv_b, void* u, int B,
                             int L, int D, cudaStream_t stream) {
  const int kV = io == IoType::BF16 ? 8 : 4;
  const dim3 grid((unsigned)((D / kV + 127) / 128), (unsigned)((L + kConvRun - 1) / kConvRun), (unsigned)B);
  if (io == IoType::BF16)
    conv_silu_kernel<__nv_bfloat16><<<grid, 128, 0, stream>>>(static_cast<const __nv_bfloat16*>(x), conv_w, conv_b,
                                                              static_cast<__nv_bfloat16*>(u), L, D);
  else
    conv_silu_kernel<float><<<grid, 128, 0, stream>>>(static_cast<const float*>(x), conv_w, conv_b,
                                                      static_cast<float*>(u), L, D);
  return cudaGetLastError();
}

cudaError_t launch_ssd(const CUtensorMap maps[5], const SsdParams& p, cudaStream_t stream) {
  const long tiles = (long)p.heads * p.n_chunks * p.batch;  // persistent kernels walk the tiles
  if (tiles >= (1L << 31)) return cudaErrorInvalidValue;
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t st_smem = sizeof(StSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(ssd_states_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)st_smem);
  if (e != cudaSuccess) return e;
  // the three launches are programmatic dependents, each of the kernel before
  // it (whose results it waits for before touching memory)
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  set_pdl(cfg, attr);
  cfg.stream = stream;
  cfg.gridDim = dim3((unsigned)(tiles < 2L * sms ? tiles : 2L * sms));
  cfg.blockDim = dim3(kStThreads);
  cfg.dynamicSmemBytes = st_smem;
  e = cudaLaunchKernelEx(&cfg, ssd_states_kernel, maps[0], maps[2], p);
  if (e != cudaSuccess) return e;
  const size_t pass_smem = sizeof(PassSmem) + 128;
  e = cudaFuncSetAttribute(ssd_pass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pass_smem);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(2u, (unsigned)p.heads, (unsigned)p.batch);
  cfg.blockDim = dim3(kPassThreads);
  cfg.dynamicSmemBytes = pass_smem;
  e = cudaLaunchKernelEx(&cfg, ssd_pass_kernel, p);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(SsdOutSmem) + 1024;
  e = cudaFuncSetAttribute(ssd_output_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3((unsigned)(tiles < sms ? tiles : sms));
  cfg.blockDim = dim3(kSsdOutThreads);
  cfg.dynamicSmemBytes = smem;
  return cudaLaunchKernelEx(&cfg, ssd_output_kernel, maps[0], maps[1], maps[2], maps[3], maps[4], p);
}

cudaError_t take_device_error(unsigned* code, cudaStream_t stream) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  e = cudaMemcpyFromSymbol(code, g_mamba_error, sizeof(unsigned));
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  return cudaMemcpyToSymbol(g_mamba_error, &zero, sizeof(unsigned));
}

}  // namespace mamba
