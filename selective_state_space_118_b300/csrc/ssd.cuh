// ssd.cuh -- Mamba-2's scan in its chunked matrix form on the tensor cores.
//
// The structure of "Jamba -- SSM-Transformer Hibrido" (ai-engineering.academy),
// section "Mamba-3: a linha de base de SSM puro em 2026", items 1 and 2: the
// state matrix is a scaled identity, discretised with Euler's method.  Heads of
// P = 64 channels share dt and A, so the decay from token s to token t,
// exp(A (cum_t - cum_s)), is one number per (t, s) for the whole head, and
// within a chunk of Q = 64 tokens the scan is a pair of small matrix products:
//   Y_diag = (mask(t >= s) * exp(A (cum_t - cum_s)) * dt_s * (C B^T)) X
//   Y_off  = exp(A cum_t) (C S_in)          (S_in: the state entering the chunk)
//   S_end  = (exp(A (cum_last - cum_s)) dt_s B_s)^T X + exp(A cum_last) S_in
// Three kernels: ssd_states_kernel (each chunk's end state from zero),
// ssd_pass_kernel (the states entering the chunks, serially per head, in
// fp32), ssd_output_kernel (Y_diag + Y_off + D x, gated).  The products use
// warp-level mma (m16n8k16, bf16 operands, fp32 accumulation): with d_state 16
// the path does ~200 tensor FLOPs per element against 6-8 bytes of traffic,
// HBM-bound, so warp-level mma keeps up and lets the first product's
// accumulators feed the second as operands without leaving registers.
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "params.h"
#include "ptx.cuh"
#include "ssm_math.cuh"

namespace mamba {

constexpr int kSsdQ = 64;          // tokens per chunk
constexpr int kSsdP = 64;          // channels per head
constexpr int kSsdN = 16;          // d_state
constexpr int kSsdThreads = 128;   // 4 warps: 16 chunk rows each
constexpr int kXs = kSsdP + 8;     // padded bf16 row of x / state tiles (144 B: ldmatrix rows conflict-free)
constexpr int kBs = kSsdN + 8;     // padded bf16 row of B / C tiles (48 B)

__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2(uint32_t (&r)[2], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x2_trans(uint32_t (&r)[2], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x2.trans.shared.b16 {%0,%1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(addr));
}

// two floats as a bf16 pair (lo in the low half: the smaller column)
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ float2 unpack_bf16(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xffff0000u));
}

// fp32 pair (a, b) as hi + lo bf16 pairs: hi = bf16(v), lo = bf16(v - hi), so
// that hi + lo carries ~16 significant bits into a bf16 tensor-core product.
__device__ __forceinline__ void split_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
  hi = pack_bf16(a, b);
  const float2 h = unpack_bf16(hi);
  lo = pack_bf16(__fsub_rn(a, h.x), __fsub_rn(b, h.y));
}

// A chunk's inputs in shared memory (rows past the sequence's end are zero,
// with dt = 0: no decay and no input there).
struct SsdTile {
  __nv_bfloat16 x[kSsdQ][kXs];
  __nv_bfloat16 B[kSsdQ][kBs];
  __nv_bfloat16 C[kSsdQ][kBs];
  float acum[kSsdQ];  // inclusive cumulative sum of dt * A (base 2) within the chunk
  float dt[kSsdQ];
};

// Offset of value (n, p) of a chunk state in the sliced layout: slice
// q = 2 n + p / 32 of (batch row, head) bh, chunk c.
__device__ __forceinline__ size_t ssd_slice(size_t bh, int n, int p, int c, int n_chunks) {
  return ((bh * 32 + (size_t)(2 * n + p / 32)) * n_chunks + c) * 32 + (p % 32);
}

// Loads x, B (and C and z when given) of chunk c of head h, batch row b into
// shared memory with asynchronous 16-byte copies (zero past the sequence's
// end), and dt with the decay prefix: computed here (from_cum false), or read
// from the states kernel's copy.  `more`, run while the copies fly, lets the
// caller put its own loads in flight too.  Ends with a block barrier.
template <typename More>
__device__ __forceinline__ void ssd_load_tile(const SsdParams& p, SsdTile& s, int b, int h, int c, bool with_c,
                                              bool from_cum, __nv_bfloat16 (*zt)[kXs], More more) {
  const int tid = threadIdx.x;
  const int t0 = c * kSsdQ;
  const int H = p.heads, G = p.groups, L = p.seqlen;
  const int g = h / (H / G);
  const __nv_bfloat16* xb = static_cast<const __nv_bfloat16*>(p.x);
  const __nv_bfloat16* zb = static_cast<const __nv_bfloat16*>(p.z);
  // x (and z): 64 rows of 128 bytes = 8 pieces of 16 bytes each
  for (int i = tid; i < kSsdQ * 8; i += kSsdThreads) {
    const int r = i >> 3, q = i & 7;
    const int t = t0 + r;
    const bool in = t < L;
    const size_t o = (((size_t)b * L + (in ? t : 0)) * H + h) * kSsdP + q * 8;
    cp_async16(smem_u32(&s.x[r][q * 8]), xb + o, in);
    if (zt) cp_async16(smem_u32(&zt[r][q * 8]), zb + o, in);
  }
  // B (and C): 64 rows of 32 bytes = 2 pieces each
  const __nv_bfloat16* Bb = static_cast<const __nv_bfloat16*>(p.Bm);
  const __nv_bfloat16* Cb = static_cast<const __nv_bfloat16*>(p.Cm);
  for (int i = tid; i < kSsdQ * 2; i += kSsdThreads) {
    const int r = i >> 1, q = i & 1;
    const int t = t0 + r;
    const bool in = t < L;
    const size_t o = (((size_t)b * L + (in ? t : 0)) * G + g) * kSsdN + q * 8;
    cp_async16(smem_u32(&s.B[r][q * 8]), Bb + o, in);
    if (with_c) cp_async16(smem_u32(&s.C[r][q * 8]), Cb + o, in);
  }
  more();
  if (from_cum) {  // dt and the decay prefix as the states kernel computed them
    if (tid < kSsdQ) {
      const float2 v = reinterpret_cast<const float2*>(p.cum)[(((size_t)b * H + h) * p.n_chunks + c) * kSsdQ + tid];
      s.acum[tid] = v.x;
      s.dt[tid] = v.y;
    }
    cp_async_wait_all();
    __syncthreads();
    return;
  }
  // dt and dt * A, then the inclusive prefix sum over the 64 tokens: two
  // warps, then warp 1 adds warp 0's total
  if (tid < kSsdQ) {
    const float A2 = a2_from_log(p.A_log[h]);  // A log2(e)
    const int t = t0 + tid;
    float dt = 0.0f;
    if (t < L) dt = softplus(to_f32(static_cast<const __nv_bfloat16*>(p.dt_raw)[((size_t)b * L + t) * H + h]));
    s.dt[tid] = dt;
    float v = __fmul_rn(dt, A2);  // in base 2
    const int lane = tid & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v = __fadd_rn(v, u);
    }
    s.acum[tid] = v;
  }
  cp_async_wait_all();
  __syncthreads();
  if (tid >= 32 && tid < kSsdQ) s.acum[tid] = __fadd_rn(s.acum[tid], s.acum[31]);
  __syncthreads();
}

// ---------------------------------------------------------------- chunk end states
// S_c[n][p] = sum_j 2^(acum_last - acum_j) dt_j B_j[n] x_j[p]: a 16 x 64 product
// over the 64 tokens; warp w computes columns 16w .. 16w + 15.
// grid (H, n_chunks, B), 128 threads.
__global__ void __launch_bounds__(kSsdThreads) ssd_states_kernel(const __grid_constant__ SsdParams p) {
  __shared__ __align__(128) SsdTile s;
  __shared__ float wj[kSsdQ];
  const int h = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
  ssd_load_tile(p, s, b, h, c, false, false, nullptr, [] {});
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float last = s.acum[kSsdQ - 1];
  if (tid < kSsdQ) wj[tid] = __fmul_rn(ex2_approx(__fsub_rn(last, s.acum[tid])), s.dt[tid]);
  const size_t bh = (size_t)b * p.heads + h;
  const size_t chunk = bh * p.n_chunks + c;
  if (tid == 0) p.totals[chunk] = last;
  if (tid < kSsdQ)  // the output kernel's copy of the chunk's dt and decay prefix
    reinterpret_cast<float2*>(p.cum)[chunk * kSsdQ + tid] = make_float2(s.acum[tid], s.dt[tid]);
  __syncthreads();

  const int g = lane >> 2, t = lane & 3;
  float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
  for (int kb = 0; kb < kSsdQ / 16; ++kb) {
    // A = (w o B)^T (16 states x 16 tokens): B^T through a transposing load
    uint32_t a[4];
    {
      const int r = lane & 7, m = lane >> 3;  // matrix m: states (m & 1) * 8, tokens (m >> 1) * 8
      ldsm_x4_trans(a, smem_u32(&s.B[kb * 16 + (m >> 1) * 8 + r][(m & 1) * 8]));
    }
    // w o B in fp32, as two bf16 terms (hi + lo) so that the product keeps ~16 bits
    uint32_t ahi[4], alo[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int k = kb * 16 + (q >> 1) * 8 + 2 * t;  // tokens of this register's pair
      const float2 v = unpack_bf16(a[q]);
      split_bf16(__fmul_rn(v.x, wj[k]), __fmul_rn(v.y, wj[k + 1]), ahi[q], alo[q]);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt) {
      uint32_t bx[2];
      ldsm_x2_trans(bx, smem_u32(&s.x[kb * 16 + (lane & 15)][warp * 16 + nt * 8]));
      mma_16816(acc[nt], ahi, bx[0], bx[1]);
      mma_16816(acc[nt], alo, bx[0], bx[1]);
    }
  }
#pragma unroll
  for (int nt = 0; nt < 2; ++nt) {
    const int col = warp * 16 + nt * 8 + 2 * t;
    *reinterpret_cast<float2*>(p.S_c + ssd_slice(bh, g, col, c, p.n_chunks)) = make_float2(acc[nt][0], acc[nt][1]);
    *reinterpret_cast<float2*>(p.S_c + ssd_slice(bh, g + 8, col, c, p.n_chunks)) =
        make_float2(acc[nt][2], acc[nt][3]);
  }
}

// ---------------------------------------------------------------- state passing
// The state entering chunk c: S_in[0] = h0 (or 0), S_in[c + 1] = 2^(total_c)
// S_in[c] + S_c[c], in fp32.  One thread per state value walks the chunks in
// order; a warp holds one slice (32 values), so each step's loads and stores
// are 128 contiguous bytes, and each thread keeps kPassAhead chunks' loads in
// flight (the chain itself is one fma per chunk).  The chunks' decay factors
// 2^(total) are staged in shared memory, kPassBlock at a time.
// grid (32 / kPassSlices, H, B), 32 * kPassSlices threads.
constexpr int kPassSlices = 4;
constexpr int kPassAhead = 16;
constexpr int kPassBlock = 512;

__global__ void __launch_bounds__(32 * kPassSlices) ssd_pass_kernel(const __grid_constant__ SsdParams p) {
  __shared__ float fac[kPassBlock];
  const int h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31;
  const int q = blockIdx.x * kPassSlices + (tid >> 5);  // this warp's slice
  const size_t bh = (size_t)b * p.heads + h;
  const int nC = p.n_chunks;
  const int n = q / 2, col = 32 * (q % 2) + lane;  // this thread's state value (row n, column col)
  const float* src = p.S_c + (bh * 32 + q) * (size_t)nC * 32 + lane;
  float* dst = p.S_in + (bh * 32 + q) * (size_t)nC * 32 + lane;
  const float* tot = p.totals + bh * nC;
  float S = p.h0 ? p.h0[bh * kSsdN * kSsdP + n * kSsdP + col] : 0.0f;
  float ahead[kPassAhead];
#pragma unroll
  for (int k = 0; k < kPassAhead; ++k) ahead[k] = k < nC ? __ldcs(src + (size_t)k * 32) : 0.0f;
  for (int c0 = 0; c0 < nC; c0 += kPassAhead) {
    if (c0 % kPassBlock == 0) {  // the next block of decay factors
      __syncthreads();
      for (int i = tid; i < kPassBlock && c0 + i < nC; i += 32 * kPassSlices) fac[i] = ex2_approx(__ldg(tot + c0 + i));
      __syncthreads();
    }
#pragma unroll
    for (int k = 0; k < kPassAhead; ++k) {
      const int c = c0 + k;
      if (c < nC) {
        __stcs(dst + (size_t)c * 32, S);
        const float v = ahead[k];
        if (c + kPassAhead < nC) ahead[k] = __ldcs(src + (size_t)(c + kPassAhead) * 32);
        S = __fmaf_rn(fac[c % kPassBlock], S, v);
      }
    }
  }
  if (p.final_state) p.final_state[bh * kSsdN * kSsdP + n * kSsdP + col] = S;
}

// ---------------------------------------------------------------- output
// grid (H, n_chunks, B), 128 threads; warp w produces chunk rows 16w .. 16w + 15.
struct SsdOutSmem {
  SsdTile t;                       // x is overwritten by y at the end (each thread its own values)
  __nv_bfloat16 z[kSsdQ][kXs];
  __nv_bfloat16 s_hi[kSsdN][kXs];  // the entering state split into two bf16 terms
  __nv_bfloat16 s_lo[kSsdN][kXs];
  float fdt[kSsdThreads / 32][kSsdQ];  // per warp: 2^(ref - acum_j) dt_j
};

__global__ void __launch_bounds__(kSsdThreads) ssd_output_kernel(const __grid_constant__ SsdParams p) {
  __shared__ __align__(128) SsdOutSmem sm;
  SsdTile& s = sm.t;
  const int h = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t bh = (size_t)b * p.heads + h;
  // tiles by asynchronous copies; meanwhile the entering state (32 slices of
  // 32 values), fp32 -> hi + lo bf16 pairs
  ssd_load_tile(p, s, b, h, c, true, true, p.z ? sm.z : nullptr, [&] {
    float4 v[kSsdN * kSsdP / 4 / kSsdThreads];
#pragma unroll
    for (int k = 0; k < kSsdN * kSsdP / 4 / kSsdThreads; ++k) {
      const int e = 4 * (tid + k * kSsdThreads), q = e / 32, n = q / 2, col = 32 * (q % 2) + e % 32;
      v[k] = __ldcs(reinterpret_cast<const float4*>(p.S_in + ssd_slice(bh, n, col, c, p.n_chunks)));
    }
#pragma unroll
    for (int k = 0; k < kSsdN * kSsdP / 4 / kSsdThreads; ++k) {
      const int e = 4 * (tid + k * kSsdThreads), q = e / 32, n = q / 2, col = 32 * (q % 2) + e % 32;
      uint32_t h01, l01, h23, l23;
      split_bf16(v[k].x, v[k].y, h01, l01);
      split_bf16(v[k].z, v[k].w, h23, l23);
      *reinterpret_cast<uint2*>(&sm.s_hi[n][col]) = make_uint2(h01, h23);
      *reinterpret_cast<uint2*>(&sm.s_lo[n][col]) = make_uint2(l01, l23);
    }
  });

  const int g = lane >> 2, t = lane & 3;
  const int i0 = warp * 16 + g, i1 = i0 + 8;  // this thread's two rows
  // C rows of this warp as the A operand (16 rows x 16 states)
  uint32_t ca[4];
  {
    const int r = lane & 7, m = lane >> 3;  // matrix m: rows (m & 1) * 8, states (m >> 1) * 8
    ldsm_x4(ca, smem_u32(&s.C[warp * 16 + (m & 1) * 8 + r][(m >> 1) * 8]));
  }
  // G = C B^T over the columns j <= this warp's last row, masked and scaled
  // by the decay 2^(acum_i - acum_j) dt_j.  Where the warp's 16 rows span a
  // decay of at most 2^60 (ref: acum at its first row), the factor splits
  // as 2^(acum_i - ref) * 2^(ref - acum_j): one exponential per row and one
  // per column (shared through fdt) instead of one per pair; neither factor
  // overflows, and a product that underflows is one far below fp32's
  // precision of the sum.  Otherwise each pair takes its own exponential.
  const float ref = s.acum[warp * 16];
  const bool split = __fsub_rn(ref, s.acum[warp * 16 + 15]) <= 60.0f;  // the same for the whole warp
  if (split) {
    for (int j = lane; j < warp * 16 + 16; j += 32)
      sm.fdt[warp][j] = __fmul_rn(ex2_approx(__fsub_rn(ref, s.acum[j])), s.dt[j]);
    __syncwarp();
  }
  const float a0 = s.acum[i0], a1 = s.acum[i1];
  const float r0 = ex2_approx(__fsub_rn(a0, ref)), r1 = ex2_approx(__fsub_rn(a1, ref));
  float G[8][4];
#pragma unroll
  for (int jt = 0; jt < 8; ++jt) {
    G[jt][0] = G[jt][1] = G[jt][2] = G[jt][3] = 0.0f;
    if (jt <= 2 * warp + 1) {
      uint32_t bb[2];
      ldsm_x2(bb, smem_u32(&s.B[jt * 8 + (lane & 7)][(lane >> 3 & 1) * 8]));
      mma_16816(G[jt], ca, bb[0], bb[1]);
      const int j0 = jt * 8 + 2 * t;
      if (split) {
        const float2 f = *reinterpret_cast<const float2*>(&sm.fdt[warp][j0]);
        G[jt][0] = j0 <= i0 ? __fmul_rn(__fmul_rn(G[jt][0], r0), f.x) : 0.0f;
        G[jt][1] = j0 + 1 <= i0 ? __fmul_rn(__fmul_rn(G[jt][1], r0), f.y) : 0.0f;
        G[jt][2] = j0 <= i1 ? __fmul_rn(__fmul_rn(G[jt][2], r1), f.x) : 0.0f;
        G[jt][3] = j0 + 1 <= i1 ? __fmul_rn(__fmul_rn(G[jt][3], r1), f.y) : 0.0f;
      } else {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int j = j0 + e;
          const float aj = s.acum[j], dtj = s.dt[j];
          G[jt][e] = j <= i0 ? __fmul_rn(G[jt][e], __fmul_rn(ex2_approx(__fsub_rn(a0, aj)), dtj)) : 0.0f;
          G[jt][2 + e] = j <= i1 ? __fmul_rn(G[jt][2 + e], __fmul_rn(ex2_approx(__fsub_rn(a1, aj)), dtj)) : 0.0f;
        }
      }
    }
  }
  // Y = G X (k blocks up to the diagonal) and C S_in (hi and lo parts)
  float Y[8][4], Yo[8][4];
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) Y[nt][0] = Y[nt][1] = Y[nt][2] = Y[nt][3] = Yo[nt][0] = Yo[nt][1] = Yo[nt][2] =
      Yo[nt][3] = 0.0f;
#pragma unroll
  for (int kb = 0; kb < kSsdQ / 16; ++kb) {
    if (kb <= warp) {
      // the accumulators of G, as A operands (hi + lo bf16 terms)
      uint32_t ah[4], al[4];
      split_bf16(G[2 * kb][0], G[2 * kb][1], ah[0], al[0]);
      split_bf16(G[2 * kb][2], G[2 * kb][3], ah[1], al[1]);
      split_bf16(G[2 * kb + 1][0], G[2 * kb + 1][1], ah[2], al[2]);
      split_bf16(G[2 * kb + 1][2], G[2 * kb + 1][3], ah[3], al[3]);
#pragma unroll
      for (int np = 0; np < 4; ++np) {  // two 8-column tiles per transposing load
        uint32_t bx[4];
        ldsm_x4_trans(bx, smem_u32(&s.x[kb * 16 + (lane & 15)][np * 16 + (lane >> 4) * 8]));
        mma_16816(Y[2 * np], ah, bx[0], bx[1]);
        mma_16816(Y[2 * np + 1], ah, bx[2], bx[3]);
        mma_16816(Y[2 * np], al, bx[0], bx[1]);
        mma_16816(Y[2 * np + 1], al, bx[2], bx[3]);
      }
    }
  }
#pragma unroll
  for (int np = 0; np < 4; ++np) {
    uint32_t bh_[4], bl_[4];
    ldsm_x4_trans(bh_, smem_u32(&sm.s_hi[lane & 15][np * 16 + (lane >> 4) * 8]));
    ldsm_x4_trans(bl_, smem_u32(&sm.s_lo[lane & 15][np * 16 + (lane >> 4) * 8]));
    mma_16816(Yo[2 * np], ca, bh_[0], bh_[1]);
    mma_16816(Yo[2 * np + 1], ca, bh_[2], bh_[3]);
    mma_16816(Yo[2 * np], ca, bl_[0], bl_[1]);
    mma_16816(Yo[2 * np + 1], ca, bl_[2], bl_[3]);
  }
  // y = (Y + 2^(acum_i) Yo + D x) silu(z), written over this thread's own x
  // values once every warp is done reading x
  __syncthreads();
  const float e0 = ex2_approx(s.acum[i0]), e1 = ex2_approx(s.acum[i1]);
  const float Dh = p.Dskip[h];
  const bool gate = p.z != nullptr;
#pragma unroll
  for (int nt = 0; nt < 8; ++nt) {
    const int col = nt * 8 + 2 * t;
    uint32_t* w0 = reinterpret_cast<uint32_t*>(&s.x[i0][col]);
    uint32_t* w1 = reinterpret_cast<uint32_t*>(&s.x[i1][col]);
    const float2 x0 = unpack_bf16(*w0), x1 = unpack_bf16(*w1);
    float y00 = __fmaf_rn(Dh, x0.x, __fmaf_rn(e0, Yo[nt][0], Y[nt][0]));
    float y01 = __fmaf_rn(Dh, x0.y, __fmaf_rn(e0, Yo[nt][1], Y[nt][1]));
    float y10 = __fmaf_rn(Dh, x1.x, __fmaf_rn(e1, Yo[nt][2], Y[nt][2]));
    float y11 = __fmaf_rn(Dh, x1.y, __fmaf_rn(e1, Yo[nt][3], Y[nt][3]));
    if (gate) {
      const float2 z0 = unpack_bf16(*reinterpret_cast<const uint32_t*>(&sm.z[i0][col]));
      const float2 z1 = unpack_bf16(*reinterpret_cast<const uint32_t*>(&sm.z[i1][col]));
      y00 = __fmul_rn(y00, silu(z0.x));
      y01 = __fmul_rn(y01, silu(z0.y));
      y10 = __fmul_rn(y10, silu(z1.x));
      y11 = __fmul_rn(y11, silu(z1.y));
    }
    *w0 = pack_bf16(y00, y01);
    *w1 = pack_bf16(y10, y11);
  }
  __syncthreads();
  // store: 8 channels (16 bytes) per access
  const int H = p.heads, L = p.seqlen;
  for (int i = tid; i < kSsdQ * 8; i += kSsdThreads) {
    const int r = i >> 3, q = i & 7;
    const int tt = c * kSsdQ + r;
    if (tt < L)
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.y) + (((size_t)b * L + tt) * H + h) * kSsdP + q * 8) =
          *reinterpret_cast<const uint4*>(&s.x[r][q * 8]);
  }
}

}  // namespace mamba
