// launch.h -- host-side launchers of the kernels (defined in kernels.cu),
// called by the C ABI in api.cpp.  Internal; not part of the public header.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "params.h"

namespace mamba {

enum class IoType { F32, BF16 };

// Dynamic shared memory of the prefill kernels for an I/O type.
size_t scan_smem_bytes(IoType io);

// B, C rows (16 values each, `ld` elements apart) in the I/O dtype -> bc
// (rows, 32) fp32; also zeroes n_counters words at `counters` (when given).
// pdl: launched as a programmatic dependent of the kernel before it.
// mode_pairs: the complex scan's layout (quads across two modes).
cudaError_t launch_bc_widen(IoType io, const void* Bm, const void* Cm, float* bc, long rows, int ld,
                            cudaStream_t stream, unsigned* counters = nullptr, int n_counters = 0,
                            bool pdl = false, bool mode_pairs = false);
// u = silu(conv(x)), (B, L, D) in the I/O dtype, zero conv inputs before t = 0.
cudaError_t launch_conv_silu(IoType io, const void* x, const float* conv_w, const float* conv_b, void* u, int B,
                             int L, int D, cudaStream_t stream);
// maps: x, z, dt_raw, bc (3-D tiled tensor maps).
// The chunked mode's carry pass and main pass as one launch of `ctas`
// one-warp CTAs (the carry tasks first, by ticket; maps: x, z, dt_raw, bc),
// a programmatic dependent of the B/C widening that zeroed its counters.
cudaError_t launch_scan_fused(IoType io, const CUtensorMap maps[4], const ScanParams& p, unsigned ctas,
                              cudaStream_t stream);
cudaError_t launch_scan(IoType io, const CUtensorMap maps[4], const ScanParams& p, dim3 grid,
                        cudaStream_t stream);
// maps: x, dt_raw, and the B half of bc.
cudaError_t launch_step(IoType io, const StepParams& p, cudaStream_t stream);
// The complex-valued scan: in chunked mode the summaries, the fold and the
// main pass; otherwise the main pass.  maps: x, z, dt_raw, bc.
cudaError_t launch_complex(IoType io, bool trapezoidal, const CUtensorMap maps[4], const ComplexParams& p,
                           cudaStream_t stream);

// Backward.  maps: x, z, dt_raw, dy, bc.  launch_carries runs the forward's
// chunk carries (n_fwd warps) and the adjoint carries (n_adj warps) in one
// launch; launch_bwd_finish runs the edge dx fix-up (chunked mode) and the
// fixed-order sums of the dB | dC and parameter partials.
cudaError_t launch_bwd(IoType io, const CUtensorMap maps[5], const BwdParams& p, dim3 grid, cudaStream_t stream);
cudaError_t launch_carries(IoType io, const CUtensorMap maps[5], const ScanParams& fp, const BwdParams& bp,
                           unsigned n_fwd, unsigned n_adj, cudaStream_t stream);
cudaError_t launch_bwd_finish(IoType io, const BwdParams& p, float* dB, float* dC, float* dA_log, float* dD,
                              float* dconv_w, float* dconv_b, cudaStream_t stream);
// Mamba-2's chunked scan: chunk end states, state passing, output.  maps
// (4-D, for the output kernel): x, z, B, C, y.
cudaError_t launch_ssd(const CUtensorMap maps[5], const SsdParams& p, cudaStream_t stream);
cudaError_t launch_io_to_f32(IoType io, const void* src, float* dst, long n, cudaStream_t stream);

// Resident CTAs per SM of the main-pass kernel and of the fused carry and
// main-pass kernel (0 when no device answers); both need less dynamic shared
// memory than the default limit.
void scan_occupancy(IoType io, int* main_per_sm, int* summary_per_sm);

// C = A W^T [+ bias] on the tensor cores (gemm_tc.cuh).  a: A (K x M, box
// 64 x 128), w: W (K x N, box 64 x bn/2), both bf16 with the 128-byte swizzle;
// c: C (N x M, box 32 x 32, 64-byte swizzle) for the stores.
cudaError_t launch_gemm_tc(const CUtensorMap& a, const CUtensorMap& w, const CUtensorMap& c, const GemmParams& p,
                           cudaStream_t s);

// Reads and clears the sticky device error word of the current device
// (synchronises the stream first).
cudaError_t take_device_error(unsigned* code, cudaStream_t stream);

}  // namespace mamba
