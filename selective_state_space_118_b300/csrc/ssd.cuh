// ssd.cuh -- Mamba-2's scan in its chunked matrix form on the tensor cores.
//
// The structure of "Jamba -- SSM-Transformer Hibrido" (ai-engineering.academy),
// section "Mamba-3: a linha de base de SSM puro em 2026", items 1 and 2: the
// state matrix is a scaled identity, discretised with Euler's method.  Heads of
// P = 64 channels share dt and A, so the decay from token s to token t,
// exp(A (cum_t - cum_s)), is one number per (t, s) for the whole head, and
// within a chunk of Q = 128 tokens the scan is a few small matrix products:
//   Y_diag = (mask(t >= s) * exp(A (cum_t - cum_s)) * dt_s * (C B^T)) X
//   Y_off  = exp(A cum_t) (C S_in)          (S_in: the state entering the chunk)
//   S_end  = (exp(A (cum_last - cum_s)) dt_s B_s)^T X + exp(A cum_last) S_in
// Three kernels: ssd_states_kernel (each chunk's end state from zero, a
// 16 x 64 product: warp-level mma m16n8k16, 16 rows being below the
// 5th-generation MMA's smallest M), ssd_pass_kernel (the states entering the
// chunks, serially per head, in fp32) and ssd_output_kernel (Y_diag + Y_off +
// D x, gated) on tcgen05: its three products are 128-row MMAs with the
// accumulators in tensor memory and the tiles brought in by TMA.  fp32
// quantities entering a product (the decay-weighted B rows and C B^T
// entries, the entering state) go in as two bf16 terms (hi + lo, ~16
// significant bits).
#pragma once
#include <cuda_bf16.h>

#include <cstdint>

#include "params.h"
#include "ptx.cuh"
#include "scan_fwd.cuh"
#include "ssm_math.cuh"

namespace mamba {

constexpr int kSsdQ = 128;         // tokens per chunk
constexpr int kSsdP = 64;          // channels per head
constexpr int kSsdN = 16;          // d_state
constexpr int kSsdThreads = 128;   // 4 warps
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
  // dt and dt * A, then the inclusive prefix sum over the chunk's tokens:
  // per warp, then each warp adds the totals of the warps before it
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
  const int w = tid >> 5;
  float off = 0.0f;  // the earlier warps' totals, read before any is updated
  if (tid < kSsdQ)
    for (int k = 0; k < w; ++k) off = __fadd_rn(off, s.acum[32 * k + 31]);
  __syncthreads();
  if (tid < kSsdQ && w > 0) s.acum[tid] = __fadd_rn(s.acum[tid], off);
  __syncthreads();
}

// ---------------------------------------------------------------- chunk end states
// S_c[n][p] = sum_j 2^(acum_last - acum_j) dt_j B_j[n] x_j[p]: a 16 x 64 product
// over the chunk's tokens; warp w computes columns 16w .. 16w + 15.
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
// One CTA (8 warps) per (head, chunk, batch row): thread t serves chunk row
// i = t % 128 (TMEM lane i) and half t / 128 of that row's columns.  Tiles by TMA: x and z (128 tokens x 64 channels, 128-byte
// swizzle: the K = token dimension's rows of 128 bytes, an MN-major operand),
// B and C (128 tokens x 16 states, 32-byte swizzle, K-major).  Three MMA
// groups, issued by one thread, accumulators in tensor memory:
//   G  = C B^T              128 x 128, K = 16          (TMEM columns 0..127)
//   Yo = C (S_hi + S_lo)    128 x 64,  K = 16 twice    (columns 128..191)
//   Y  = (G_hi + G_lo) X    128 x 64,  K = 128 twice   (columns 192..255)
// Between them each thread reads its row of G, masks it to s <= t, scales it
// by the decay 2^(acum_i - acum_j) dt_j and writes it, as hi + lo bf16 terms,
// into shared memory in the K-major 128-byte-swizzled layout of an A
// operand.  The epilogue: y = Y + 2^(acum_i) Yo + D x, times silu(z), written
// over the thread's row of the x tile and stored by TMA.
constexpr int kSsdTmemCols = 256;
constexpr int kSsdOutThreads = 256;

struct SsdTcSmem {
  __nv_bfloat16 x[kSsdQ * kSsdP];        // 16 KB, then y
  __nv_bfloat16 z[kSsdQ * kSsdP];        // 16 KB
  __nv_bfloat16 ghi[2][kSsdQ * 64];      // G's columns 0..63 and 64..127: rows of 128 bytes
  __nv_bfloat16 glo[2][kSsdQ * 64];
  __nv_bfloat16 shi[kSsdN * kSsdP];      // S_in: rows n of 64 channels (128 bytes)
  __nv_bfloat16 slo[kSsdN * kSsdP];
  __nv_bfloat16 c[kSsdQ * kSsdN];        // rows of 32 bytes
  __nv_bfloat16 b[kSsdQ * kSsdN];
  float acum[kSsdQ];
  float dt[kSsdQ];
  float fdt[kSsdQ];                      // 2^(ref - acum_j) dt_j
  uint64_t bar_tile, bar_mma1, bar_mma2;
  uint32_t tmem_base;
};

// 16-byte piece `piece` of row `row` in a 128-byte-swizzled tile of 128-byte rows.
__device__ __forceinline__ uint32_t sw128(uint32_t base, int row, int piece) {
  return base + row * 128 + ((piece ^ (row & 7)) << 4);
}

__global__ void __launch_bounds__(kSsdOutThreads, 2)
    ssd_output_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_z,
                      const __grid_constant__ CUtensorMap tm_b, const __grid_constant__ CUtensorMap tm_c,
                      const __grid_constant__ CUtensorMap tm_y, const __grid_constant__ SsdParams p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  SsdTcSmem& sm = *reinterpret_cast<SsdTcSmem*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
  const int h = blockIdx.x, c = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5;
  const int H = p.heads, G = p.groups;
  const int g = h / (H / G);
  const int t0 = c * kSsdQ;
  const size_t bh = (size_t)b * H + h;
  const bool gate = p.z != nullptr;

  if (tid == 0) {
    mbar_init(smem_u32(&sm.bar_tile), 1);
    mbar_init(smem_u32(&sm.bar_mma1), 1);
    mbar_init(smem_u32(&sm.bar_mma2), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&sm.tmem_base), kSsdTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = sm.tmem_base;
  if (tid == 0) {
    const uint32_t bar = smem_u32(&sm.bar_tile);
    mbar_arrive_expect_tx(bar, (gate ? 2 : 1) * kSsdQ * kSsdP * 2 + 2 * kSsdQ * kSsdN * 2);
    tma_load_4d(smem_u32(sm.x), &tm_x, 0, h, t0, b, bar);
    if (gate) tma_load_4d(smem_u32(sm.z), &tm_z, 0, h, t0, b, bar);
    tma_load_4d(smem_u32(sm.b), &tm_b, 0, g, t0, b, bar);
    tma_load_4d(smem_u32(sm.c), &tm_c, 0, g, t0, b, bar);
  }
  // while the tiles fly: dt and the decay prefix (the states kernel's), and
  // the entering state as hi + lo bf16 terms in the MN-major layout (row n:
  // 64 channels, 8 channels per 16-byte piece, 128-byte swizzle)
  if (tid < kSsdQ) {
    const float2 v = reinterpret_cast<const float2*>(p.cum)[(bh * p.n_chunks + c) * kSsdQ + tid];
    sm.acum[tid] = v.x;
    sm.dt[tid] = v.y;
    const int n = tid >> 3, piece = tid & 7;  // 16 rows x 8 pieces: one per thread
    const float* src = p.S_in + ssd_slice(bh, n, piece * 8, c, p.n_chunks);
    const float4 a = __ldcs(reinterpret_cast<const float4*>(src));
    const float4 d = __ldcs(reinterpret_cast<const float4*>(src) + 1);
    uint32_t hi[4], lo[4];
    split_bf16(a.x, a.y, hi[0], lo[0]);
    split_bf16(a.z, a.w, hi[1], lo[1]);
    split_bf16(d.x, d.y, hi[2], lo[2]);
    split_bf16(d.z, d.w, hi[3], lo[3]);
    st_shared_v4(sw128(smem_u32(sm.shi), n, piece), hi[0], hi[1], hi[2], hi[3]);
    st_shared_v4(sw128(smem_u32(sm.slo), n, piece), lo[0], lo[1], lo[2], lo[3]);
  }
  fence_proxy_async_smem();
  __syncthreads();
  const float ref = sm.acum[0];
  const bool split = __fsub_rn(ref, sm.acum[kSsdQ - 1]) <= 60.0f;  // the whole chunk's decay span
  if (split && tid < kSsdQ) sm.fdt[tid] = __fmul_rn(ex2_approx(__fsub_rn(ref, sm.acum[tid])), sm.dt[tid]);

  bool ok = true;
  if (tid == 0) {  // G = C B^T and Yo = C S_in
    ok = mbar_wait_bounded(smem_u32(&sm.bar_tile), 0, p.timeout_ns);
    if (ok) {
      tc_fence_after();
      const uint64_t cd = umma_desc(smem_u32(sm.c), 256, 6);
      tc_mma_f16(tmem, cd, umma_desc(smem_u32(sm.b), 256, 6), umma_idesc_bf16(128, 128, false), false);
      const uint32_t io = umma_idesc_bf16(128, 64, true);
      tc_mma_f16(tmem + 128, cd, umma_desc(smem_u32(sm.shi), 1024, 2), io, false);
      tc_mma_f16(tmem + 128, cd, umma_desc(smem_u32(sm.slo), 1024, 2), io, true);
      tc_commit(smem_u32(&sm.bar_mma1));
    }
  }
  ok = __syncthreads_and(ok);
  if (ok) {
    ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&sm.bar_mma1), 0, p.timeout_ns));
    ok = __syncthreads_and(ok);
  }
  const int i = tid & (kSsdQ - 1);  // this thread's row
  const int hf = tid >> 7;           // and half of the row's columns
  const uint32_t lanes = (uint32_t)(32 * (warp & 3)) << 16;
  if (ok) {
    tc_fence_after();
    const float ai = sm.acum[i];
    const float ri = ex2_approx(__fsub_rn(ai, ref));
#pragma unroll 1
    for (int cb = 2 * hf; cb < 2 * hf + 2; ++cb) {  // 32 columns j of G at a time
      uint32_t r[32];
      tmem_ld_32cols(tmem + lanes + 32 * cb, r);
      uint32_t hi[16], lo[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) {
        float v2[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int j = 32 * cb + 2 * e + u;
          float f;
          if (split)
            f = __fmul_rn(ri, sm.fdt[j]);
          else
            f = __fmul_rn(ex2_approx(__fsub_rn(ai, sm.acum[j])), sm.dt[j]);
          v2[u] = j <= i ? __fmul_rn(__uint_as_float(r[2 * e + u]), f) : 0.0f;
        }
        split_bf16(v2[0], v2[1], hi[e], lo[e]);
      }
      // columns 32cb .. 32cb + 31: K block cb / 2, pieces 4 (cb % 2) .. + 3
      const int kb = cb >> 1;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int piece = 4 * (cb & 1) + q;
        st_shared_v4(sw128(smem_u32(sm.ghi[kb]), i, piece), hi[4 * q], hi[4 * q + 1], hi[4 * q + 2], hi[4 * q + 3]);
        st_shared_v4(sw128(smem_u32(sm.glo[kb]), i, piece), lo[4 * q], lo[4 * q + 1], lo[4 * q + 2], lo[4 * q + 3]);
      }
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0 && ok) {  // Y = G X: the hi terms, then the lo terms, 16 tokens of K per MMA
    const uint32_t iy = umma_idesc_bf16(128, 64, true);
    bool acc = false;
#pragma unroll 1
    for (int part = 0; part < 2; ++part) {
      for (int kb = 0; kb < 2; ++kb) {
        const uint32_t gbase = smem_u32(part == 0 ? sm.ghi[kb] : sm.glo[kb]);
#pragma unroll
        for (int ks = 0; ks < 4; ++ks) {
          const uint64_t ad = umma_desc(gbase + 32 * ks, 1024, 2);                         // 16 columns of G
          const uint64_t bd = umma_desc(smem_u32(sm.x) + (kb * 64 + ks * 16) * 128, 1024, 2);  // 16 rows of x
          tc_mma_f16(tmem + 192, ad, bd, iy, acc);
          acc = true;
        }
      }
    }
    tc_commit(smem_u32(&sm.bar_mma2));
  }
  if (ok) {
    ok = __all_sync(0xffffffffu, mbar_wait_bounded(smem_u32(&sm.bar_mma2), 0, p.timeout_ns));
    ok = __syncthreads_and(ok);
  }
  if (ok) {
    tc_fence_after();
    const float ei = ex2_approx(sm.acum[i]);
    const float Dh = p.Dskip[h];
    {
      const int half = hf;  // channels 32 half .. + 31
      uint32_t yv[32], yo[32];
      tmem_ld_32cols(tmem + lanes + 192 + 32 * half, yv);
      tmem_ld_32cols(tmem + lanes + 128 + 32 * half, yo);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int piece = 4 * half + q;
        const uint32_t xa = sw128(smem_u32(sm.x), i, piece);
        uint4 xv = *reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned char*>(sm.x) + (xa - smem_u32(sm.x)));
        uint4 zv = make_uint4(0, 0, 0, 0);
        if (gate)
          zv = *reinterpret_cast<const uint4*>(reinterpret_cast<const unsigned char*>(sm.z) +
                                               (sw128(smem_u32(sm.z), i, piece) - smem_u32(sm.z)));
        const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
        const uint32_t zw[4] = {zv.x, zv.y, zv.z, zv.w};
        uint32_t out[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int k = 8 * q + 2 * e;  // column within the half
          const float2 xx = unpack_bf16(xw[e]);
          float y0 = __fmaf_rn(Dh, xx.x, __fmaf_rn(ei, __uint_as_float(yo[k]), __uint_as_float(yv[k])));
          float y1 = __fmaf_rn(Dh, xx.y, __fmaf_rn(ei, __uint_as_float(yo[k + 1]), __uint_as_float(yv[k + 1])));
          if (gate) {
            const float2 zz = unpack_bf16(zw[e]);
            y0 = __fmul_rn(y0, silu(zz.x));
            y1 = __fmul_rn(y1, silu(zz.y));
          }
          out[e] = pack_bf16(y0, y1);
        }
        st_shared_v4(xa, out[0], out[1], out[2], out[3]);
      }
    }
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    if (ok) {
      tma_store_4d(&tm_y, 0, h, t0, b, smem_u32(sm.x));
      bulk_commit();
      bulk_wait_all();
    } else {
      report_error(4u);  // MAMBA_ERR_TIMEOUT
    }
  }
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kSsdTmemCols);
  }
}

}  // namespace mamba
