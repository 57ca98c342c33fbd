// api.cpp -- the C ABI of libmamba_ssm.so (declared in include/mamba_ssm.h):
// argument checks, the chunking plan, tensor-map encoding and kernel launches.
// Never allocates, frees or synchronises (except mamba_last_error).
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cmath>
#include <cstring>
#include <mutex>

#include "../../include/mamba_ssm.h"
#include "launch.h"

using mamba::IoType;

namespace {

constexpr int kT = mamba::kTileTokens;  // tokens per tile (every chunk and piece is whole tiles)
constexpr int kLanes = 32;  // channels per CTA (one warp)
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

// The chunking plan: n_chunks chunks of chunk_tiles tiles (the last one may
// be shorter), and, in chunked mode, every chunk but the last cut into
// `pieces` summary pieces of piece_tiles tiles (the last piece may be shorter).
struct Plan {
  int n_chunks;
  int chunk_tiles;
  int pieces;
  int piece_tiles;
};

// The machine as the plan sees it: SM count and resident one-warp CTAs per SM
// of the main-pass kernel and of the fused carry-and-main kernel (which runs
// the carry walks), bf16 I/O (from the occupancy calculator; typical B300
// values when no device answers, e.g. in a build without a GPU).
struct Machine {
  int sms;
  int main_per_sm;
  int summary_per_sm;
};

Machine query_machine() {
  Machine m{sm_count(), 16, 16};
  int a = 0, b = 0;
  mamba::scan_occupancy(IoType::BF16, &a, &b);
  if (a > 0) m.main_per_sm = a;
  if (b > 0) m.summary_per_sm = b;
  return m;
}

// The machine of the current device, queried once per device (the plan is
// made on every call; the occupancy queries behind it cost host time).
Machine machine() {
  constexpr int kMaxDev = 64;
  static Machine cache[kMaxDev];
  static bool have[kMaxDev] = {};
  static std::mutex mu;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return query_machine();
  std::lock_guard<std::mutex> lock(mu);
  if (!have[dev]) {
    cache[dev] = query_machine();
    have[dev] = true;
  }
  return cache[dev];
}

// Modelled time of a kernel pass that runs `items` one-warp CTAs of `tiles`
// tiles each at `cost` per tile.  The busiest of the 4 * SM schedulers runs
// ceil(items / (4 SMs)) of them; how fast depends on how many warps share a
// scheduler (a lone warp issues about every other cycle, four or more keep it
// busy), so the rate is the issue efficiency at the resident warp count; each
// CTA pays a fixed set-up of about half a tile.
double pass_time(long items, int tiles, double cost, int sms, int per_sm) {
  const long units = 4L * sms;
  const long resident = items < (long)sms * per_sm ? items : (long)sms * per_sm;
  const double w = (double)resident / units;
  double ipc = 0.25 + 0.2 * w;
  if (ipc > 0.95) ipc = 0.95;
  const long per_unit = (items + units - 1) / units;
  return (double)per_unit * (tiles + 0.5) * cost / ipc;
}

// Carry pieces: 4 tiles (64 tokens).  A boundary's walk stops at a piece
// boundary and drops the state pairs whose decay to the boundary fell below
// the bound at piece boundaries only, so shorter pieces waste less past the
// point where the decay makes earlier tokens negligible; each piece end costs
// a fold of the piece into the accumulated carry.  Measured on the 256k-token
// workload (64 calls of 4,096 tokens): 256-, 64- and 32-token pieces 16.6,
// 16.3 and 16.5 ms per step; the 32k call and the backward alike within 1 %.
constexpr int kPieceTiles = 4;

// Expected tiles walked per chunk boundary when the inputs decay fast (the
// walk stops after the decay reaches 2^-32; ~1,000 tokens for dt ~ 0.02,
// A = -1): used only to size the plan.
constexpr int kCarryTilesEstimate = 64;

// Relative costs of the plan's model: a main-pass tile and a carry-walk tile
// (16 tokens x 32 channels each) and one hop of a carry chain, in units of
// ~1,800 issued warp-instructions.  The model adds the two passes' times;
// they share one launch and overlap in part, and a sweep of the chunk count
// at 4,096 and 32,768 tokens (x 8,192 channels) found the model's choice
// still the fastest.
constexpr double kMainTileCost = 1.0;
constexpr double kCarryTileCost = 0.7;
constexpr double kChainHopCost = 1.5;

// The plan depends only on the sizes (not on the I/O dtype), so that the
// workspace queries, which take no dtype, agree with the call.
Plan make_plan(int batch, int seqlen, int d_inner, int n_chunks_req) {
  const int tiles = (seqlen + kT - 1) / kT;
  Plan pl{1, tiles, 1, tiles};
  if (tiles <= 1 || n_chunks_req == 1) return pl;
  const long groups = (long)batch * ((d_inner + kLanes - 1) / kLanes);
  const Machine mc = machine();
  int lo = 1, hi = tiles < 64 ? tiles : 64;
  if (n_chunks_req > 1) lo = hi = n_chunks_req < tiles ? n_chunks_req : tiles;
  double best = -1.0;
  for (int n = lo; n <= hi; ++n) {
    const int C = (tiles + n - 1) / n;
    const int n_eff = (tiles + C - 1) / C;
    const int P = C < kPieceTiles ? C : kPieceTiles;
    const int m = (C + P - 1) / P;
    // Chunks shorter than the expected walk make every boundary walk its
    // whole chunk and then wait for the previous boundary's carry: the walks
    // run side by side, the folds one after another (a chain of hops of
    // about a tile's time each).  Longer chunks: the walks stop early and the
    // two kinds of warps are costed as passes of their own.
    double t;
    if (n_eff > 1 && C < kCarryTilesEstimate) {
      // Walks over whole chunks: the one launch runs as two phases, all the
      // walks (with chunk 0's main warps beside them), then the later
      // chunks' main warps once their carries are in; each phase lasts a
      // warp's duration (its C tiles, at the issue efficiency of the warps
      // sharing a scheduler) per wave of resident slots, so shorter chunks
      // shorten both phases until a phase spills into a second wave.
      // Measured at 4,096 tokens x 8,192 channels, 8-12 chunks: 17.6, 16.1,
      // 15.5, 16.9, 17.6 ms per 64 calls (this picks 10).
      const long units = 4L * mc.sms;
      const long slots = (long)mc.sms * mc.summary_per_sm;
      const long walks = groups * (n_eff - 1);  // and as many later main warps
      const double waves = (double)((walks + slots - 1) / slots);
      const double w = (double)(walks < slots ? walks : slots) / units;
      const double per_warp = std::ceil(w) / (0.25 + 0.2 * w);
      t = (C + 0.5) * (kCarryTileCost + kMainTileCost) * per_warp * waves + kChainHopCost * (n_eff - 1);
    } else {
      double t_carry = 0.0;
      if (n_eff > 1) t_carry = pass_time(groups * (n_eff - 1), kCarryTilesEstimate, kCarryTileCost, mc.sms,
                                         mc.summary_per_sm);
      t = pass_time(groups * n_eff, C, kMainTileCost, mc.sms, mc.main_per_sm) + t_carry;
    }
    if (best < 0.0 || t < best - 1e-9) {
      best = t;
      pl = Plan{n_eff, C, n_eff > 1 ? m : 1, n_eff > 1 ? P : C};
    }
  }
  return pl;
}

struct Workspace {
  size_t bc, carry, counters, counters_bytes, total;
};

// bc: B and C widened to fp32 in pair quads, (B, L, 32); then, in chunked
// mode only, the carries (B, n_chunks, D, 16) and the counters: a ticket
// counter and (B, groups, n_chunks) ready flags.
Workspace workspace_layout(int batch, int seqlen, int d_inner, const Plan& pl) {
  Workspace w{0, 0, 0, 0, 0};
  const size_t B = batch, L = seqlen, D = d_inner, n = pl.n_chunks;
  const size_t G = (D + kLanes - 1) / kLanes;
  w.bc = 0;
  w.total = round256(B * L * 32 * sizeof(float));
  if (pl.n_chunks <= 1) return w;
  w.carry = w.total;
  w.counters = round256(w.carry + B * n * D * 16 * sizeof(float));
  w.counters_bytes = (1 + B * G * n) * sizeof(unsigned);
  w.total = round256(w.counters + w.counters_bytes);
  return w;
}

// The backward's workspace: the forward's (at offset 0; the checkpointing
// forward pass uses it), then the states entering every tile (B, tiles, D,
// 16), in chunked mode the adjoint carries (B, n_chunks, D, 16) and their
// counters, the per-group dB | dC sums (groups, B * L, 32), the per-chunk
// parameter partials (B * n_chunks, D, 24) and, in chunked mode, the edge
// buffers of the conv (B, n_chunks, 3, D) twice.
struct BwdWorkspace {
  Workspace fwd;
  size_t ckpt, acarry, counters, counters_bytes, part_bc, part_param, edge_dx, edge_dpre, total;
};

BwdWorkspace bwd_workspace_layout(int batch, int seqlen, int d_inner, const Plan& pl) {
  BwdWorkspace w;
  std::memset(&w, 0, sizeof(w));
  w.fwd = workspace_layout(batch, seqlen, d_inner, pl);
  const size_t B = batch, L = seqlen, D = d_inner, n = pl.n_chunks;
  const size_t G = (D + kLanes - 1) / kLanes;
  const size_t tiles = (L + kT - 1) / kT;
  size_t o = w.fwd.total;
  w.ckpt = o;
  o = round256(o + B * tiles * D * 16 * sizeof(float));
  if (n > 1) {
    w.acarry = o;
    o = round256(o + B * n * D * 16 * sizeof(float));
    w.counters = o;
    w.counters_bytes = (1 + B * G * n) * sizeof(unsigned);
    o = round256(o + w.counters_bytes);
  }
  w.part_bc = o;
  o = round256(o + G * B * L * 32 * sizeof(float));
  w.part_param = o;
  o = round256(o + B * n * D * 24 * sizeof(float));
  if (n > 1) {
    w.edge_dx = o;
    o = round256(o + B * n * 3 * D * sizeof(float));
    w.edge_dpre = o;
    o = round256(o + B * n * 3 * D * sizeof(float));
  }
  w.total = o;
  return w;
}

// The layer's workspace: x, z, u (unless the caller takes u), the x_proj
// output (B, L, dt_rank + 32), dt_raw and y, then the scan's workspace, then
// nothing else (the GEMMs need no scratch).
struct LayerWorkspace {
  size_t x, z, u, xdbl, dt_raw, y, scan, total;
  Workspace scan_ws;
};

LayerWorkspace layer_workspace_layout(int batch, int seqlen, int d_inner, int dt_rank, const Plan& pl,
                                      bool need_u) {
  LayerWorkspace w;
  std::memset(&w, 0, sizeof(w));
  const size_t rows = (size_t)batch * seqlen, D = d_inner, R = dt_rank;
  size_t o = 0;
  const size_t act = round256(rows * D * 2);
  w.x = o;
  o += act;
  w.z = o;
  o += act;
  if (need_u) {
    w.u = o;
    o += act;
  }
  w.xdbl = o;
  o += round256(rows * (R + 32) * 2);
  w.dt_raw = o;
  o += act;
  w.y = o;
  o += act;
  w.scan = o;
  w.scan_ws = workspace_layout(batch, seqlen, d_inner, pl);
  o += w.scan_ws.total;
  w.total = o;
  return w;
}

// 3-D tiled map over a (B, L, inner) row-major tensor: box (box_inner, kT, 1).
bool encode3d(CUtensorMap* m, const void* base, mamba_dtype io, int inner, int L, int B, int box_inner) {
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

// 2-D map over a row-major bf16 matrix of `rows` rows of `inner` elements,
// rows `ld` elements apart, read in boxes of 64 elements (128 bytes) x
// box_rows rows with the 128-byte swizzle (the tensor-core GEMM's operands).
bool encode2d_bf16(CUtensorMap* m, const void* base, int inner, long rows, long ld, int box_inner, int box_rows,
                   CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_inner, (cuuint32_t)box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode2d_sw128(CUtensorMap* m, const void* base, int inner, long rows, long ld, int box_rows) {
  return encode2d_bf16(m, base, inner, rows, ld, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

// C = A W^T [+ bias] on the tensor cores (checked arguments: K, lda, ldc
// multiples of 8, 16-byte aligned pointers, M > 0).  The N extent is cut
// evenly into tiles of at most 256 columns, each a multiple of 32; a CTA pair
// loads half of a W tile each (the W box is bn / 2 rows).
mamba_status tc_linear(const void* A, long lda, const void* W, const void* bias, void* C, long ldc, long M, int N,
                       int K, uint64_t timeout_ns, cudaStream_t stream) {
  const int tiles_n = (N + 255) / 256;
  const int bn = ((N + tiles_n - 1) / tiles_n + 31) / 32 * 32;
  CUtensorMap ma, mw, mc;
  if (!encode2d_sw128(&ma, A, K, M, lda, 128) || !encode2d_sw128(&mw, W, K, N, K, bn / 2) ||
      !encode2d_bf16(&mc, C, N, M, ldc, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B))
    return MAMBA_ERR_CUDA;
  mamba::GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.M = M;
  p.N = N;
  p.K = K;
  p.bn = bn;
  p.ldc = (int)ldc;
  p.C = C;
  p.bias = bias;
  p.timeout_ns = timeout_ns;
  return mamba::launch_gemm_tc(ma, mw, mc, p, stream) == cudaSuccess ? MAMBA_OK : MAMBA_ERR_CUDA;
}

// The channel rows of the (B, L, D) tensors are read by bulk tensor copies,
// whose row stride (D elements) must be a multiple of 16 bytes: d_inner a
// multiple of 8 for bf16 and of 4 for fp32.  Groups of channels past D are
// filled with zeros by the copies and masked in every kernel.
int d_inner_multiple(mamba_dtype io) { return io == MAMBA_BF16 ? 8 : 4; }

mamba_status check_common(int batch, int d_inner, int d_state, int d_conv, mamba_dtype io) {
  if (batch <= 0 || d_inner <= 0) return MAMBA_ERR_INVALID_ARG;
  if (io != MAMBA_F32 && io != MAMBA_BF16) return MAMBA_ERR_UNSUPPORTED;
  if (d_state != MAMBA_D_STATE || d_conv != MAMBA_D_CONV) return MAMBA_ERR_UNSUPPORTED;
  if (d_inner % d_inner_multiple(io) != 0) return MAMBA_ERR_UNSUPPORTED;
  return MAMBA_OK;
}

// The forward's parameter block for checked arguments and a workspace of the
// plan's layout.  ckpt (may be null): the state entering every tile is
// stored there.
mamba::ScanParams fwd_params(const mamba_scan_args* a, const Plan& pl, const Workspace& ws, float* ckpt) {
  char* wsp = static_cast<char*>(a->workspace);
  mamba::ScanParams p;
  std::memset(&p, 0, sizeof(p));
  p.batch = a->batch;
  p.seqlen = a->seqlen;
  p.d_inner = a->d_inner;
  p.n_groups = (a->d_inner + kLanes - 1) / kLanes;
  p.chunk_tiles = pl.chunk_tiles;
  p.n_chunks = pl.n_chunks;
  p.piece_tiles = pl.piece_tiles;
  p.pieces = pl.pieces;
  p.A_log = a->A_log;
  p.Dskip = a->Dskip;
  p.conv_w = a->conv_w;
  p.conv_b = a->conv_b;
  p.h0 = a->h0;
  p.conv_state0 = a->conv_state0;
  p.x = a->x;
  p.y = a->y;
  p.final_h = a->final_h;
  p.final_conv_state = a->final_conv_state;
  p.ckpt = ckpt;
  p.seq_tiles = (a->seqlen + kT - 1) / kT;
  p.flags = a->flags;
  p.timeout_ns = a->wait_timeout_ns ? a->wait_timeout_ns : kDefaultTimeoutNs;
  if (pl.n_chunks > 1) {
    p.carry = reinterpret_cast<float*>(wsp + ws.carry);
    p.counters = reinterpret_cast<unsigned*>(wsp + ws.counters);
  }
  return p;
}

// The forward kernels: B/C widening, chunk carries (chunked mode), main pass.
// bc_ld: elements from one token's B (and C) row to the next.
mamba_status launch_forward(const mamba_scan_args* a, const Plan& pl, const Workspace& ws, cudaStream_t stream,
                            int bc_ld = 16) {
  const size_t B = a->batch;
  float* bc = reinterpret_cast<float*>(static_cast<char*>(a->workspace) + ws.bc);

  // x, z, dt_raw, bc (main pass), bc (summary pass)
  CUtensorMap maps[5];
  if (!encode3d(&maps[0], a->x, a->io, a->d_inner, a->seqlen, a->batch, kLanes) ||
      !encode3d(&maps[1], a->z, a->io, a->d_inner, a->seqlen, a->batch, kLanes) ||
      !encode3d(&maps[2], a->dt_raw, a->io, a->d_inner, a->seqlen, a->batch, kLanes) ||
      !encode3d(&maps[3], bc, MAMBA_F32, 32, a->seqlen, a->batch, 32) ||
      !encode3d(&maps[4], bc, MAMBA_F32, 32, a->seqlen, a->batch, 32))
    return MAMBA_ERR_CUDA;

  const mamba::ScanParams p = fwd_params(a, pl, ws, a->tile_states);
  const IoType io = a->io == MAMBA_BF16 ? IoType::BF16 : IoType::F32;

  if (pl.n_chunks > 1) {
    // carries and main pass in one launch, the carry tasks first; the B/C
    // widening before it zeroes its counters, and both launch as programmatic
    // dependents (each waits for the kernel before it, so that a sequence of
    // calls overlaps one launch with the previous one's end)
    const size_t per = (size_t)p.n_groups * B;
    const size_t ctas = (2 * (size_t)pl.n_chunks - 1) * per;
    if (ctas >= (1u << 31)) return MAMBA_ERR_UNSUPPORTED;
    if (mamba::launch_bc_widen(io, a->Bm, a->Cm, bc, (long)B * a->seqlen, bc_ld, stream, p.counters,
                               (int)(ws.counters_bytes / sizeof(unsigned)), true) != cudaSuccess)
      return MAMBA_ERR_CUDA;
    if (mamba::launch_scan_fused(io, maps, p, (unsigned)ctas, stream) != cudaSuccess) return MAMBA_ERR_CUDA;
    return MAMBA_OK;
  }
  if (mamba::launch_bc_widen(io, a->Bm, a->Cm, bc, (long)B * a->seqlen, bc_ld, stream) != cudaSuccess)
    return MAMBA_ERR_CUDA;
  dim3 g2((unsigned)p.n_groups, (unsigned)B, (unsigned)pl.n_chunks);
  if (mamba::launch_scan(io, maps, p, g2, stream) != cudaSuccess) return MAMBA_ERR_CUDA;
  return MAMBA_OK;
}

// The complex scan's plan: chunks of whole tiles, as many as fill the GPU
// with about 16 one-warp CTAs per SM (its chunked mode recomputes every chunk
// but the last once as a summary, so no more chunks than that), at most 64.
Plan complex_plan(int batch, int seqlen, int d_inner, int n_chunks_req) {
  const int tiles = (seqlen + kT - 1) / kT;
  int n = n_chunks_req;
  if (n <= 0) {
    const long groups = (long)batch * ((d_inner + kLanes - 1) / kLanes);
    const long target = 16L * sm_count();
    n = (int)((target + groups - 1) / groups);
    if (n > 64) n = 64;
  }
  if (n > tiles) n = tiles;
  if (n < 1) n = 1;
  const int C = (tiles + n - 1) / n;
  const int P = C < kPieceTiles ? C : kPieceTiles;  // carry pieces of the walked mode
  return Plan{(tiles + C - 1) / C, C, (C + P - 1) / P, P};
}

struct ComplexWorkspace {
  size_t bc, hloc, sdt, carry, counters, counters_bytes, total;
};

ComplexWorkspace complex_workspace_layout(int batch, int seqlen, int d_inner, const Plan& pl) {
  ComplexWorkspace w{0, 0, 0, 0, 0, 0, 0};
  const size_t B = batch, L = seqlen, D = d_inner, n = pl.n_chunks;
  const size_t G = (D + kLanes - 1) / kLanes;
  w.total = round256(B * L * 32 * sizeof(float));
  if (n <= 1) return w;
  // the exact mode's chunk summaries, the entering states, and the walked
  // mode's ticket and flags
  w.hloc = w.total;
  w.sdt = round256(w.hloc + B * n * D * 16 * sizeof(float));
  w.carry = round256(w.sdt + B * n * D * sizeof(float));
  w.counters = round256(w.carry + B * n * D * 16 * sizeof(float));
  w.counters_bytes = (1 + B * G * n) * sizeof(unsigned);
  w.total = round256(w.counters + w.counters_bytes);
  return w;
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
  if (batch <= 0 || seqlen <= 0 || d_inner <= 0 || d_inner % 4) return 1;
  return make_plan(batch, seqlen, d_inner, 0).n_chunks;
}

mamba_status mamba_scan_plan(int batch, int seqlen, int d_inner, int n_chunks, int out[4]) {
  if (!out || batch <= 0 || seqlen <= 0 || d_inner <= 0 || n_chunks < 0) return MAMBA_ERR_INVALID_ARG;
  if (d_inner % 4) return MAMBA_ERR_UNSUPPORTED;
  const Plan pl = make_plan(batch, seqlen, d_inner, n_chunks);
  out[0] = pl.n_chunks;
  out[1] = pl.chunk_tiles * kT;
  out[2] = pl.n_chunks > 1 ? pl.pieces : 0;
  out[3] = pl.n_chunks > 1 ? pl.piece_tiles * kT : 0;
  return MAMBA_OK;
}

size_t mamba_scan_workspace_size(int batch, int seqlen, int d_inner, int n_chunks) {
  if (batch <= 0 || seqlen <= 0 || d_inner <= 0 || d_inner % 4 || n_chunks < 0) return 0;
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
                                a->final_h, a->final_conv_state, a->tile_states};
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
  return launch_forward(a, pl, ws, stream);
}

size_t mamba_scan_bwd_workspace_size(int batch, int seqlen, int d_inner, int n_chunks) {
  if (batch <= 0 || seqlen <= 0 || d_inner <= 0 || d_inner % 4 || n_chunks < 0) return 0;
  return bwd_workspace_layout(batch, seqlen, d_inner, make_plan(batch, seqlen, d_inner, n_chunks)).total;
}

mamba_status mamba_scan_bwd(const mamba_scan_bwd_args* a, void* stream_v) {
  if (!a) return MAMBA_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_v);
  mamba_status st = check_common(a->batch, a->d_inner, a->d_state, a->d_conv, a->io);
  if (st != MAMBA_OK) return st;
  if (a->seqlen < 0 || a->n_chunks < 0) return MAMBA_ERR_INVALID_ARG;
  if (!a->A_log || !a->Dskip || !a->conv_w || !a->dA_log || !a->dDskip || !a->dconv_w)
    return MAMBA_ERR_INVALID_ARG;
  const void* aligned_ptrs[] = {a->A_log, a->Dskip, a->conv_w, a->conv_b, a->h0, a->conv_state0,
                                a->dfinal_h, a->dfinal_conv_state, a->dA_log, a->dDskip, a->dconv_w,
                                a->dconv_b, a->dh0, a->dconv_state0, a->tile_states};
  for (const void* p : aligned_ptrs)
    if (p && !aligned16(p)) return MAMBA_ERR_INVALID_ARG;
  const size_t B = a->batch, D = a->d_inner;
  const IoType io = a->io == MAMBA_BF16 ? IoType::BF16 : IoType::F32;

  if (a->seqlen == 0) {
    // final_h = h0 and final_conv_state = conv_state0; the parameters are unused
    if (cudaMemsetAsync(a->dA_log, 0, D * 16 * sizeof(float), stream) != cudaSuccess ||
        cudaMemsetAsync(a->dDskip, 0, D * sizeof(float), stream) != cudaSuccess ||
        cudaMemsetAsync(a->dconv_w, 0, D * 4 * sizeof(float), stream) != cudaSuccess ||
        (a->dconv_b && cudaMemsetAsync(a->dconv_b, 0, D * sizeof(float), stream) != cudaSuccess))
      return MAMBA_ERR_CUDA;
    if (a->dh0) {
      cudaError_t e = a->dfinal_h ? cudaMemcpyAsync(a->dh0, a->dfinal_h, B * D * 16 * sizeof(float),
                                                    cudaMemcpyDeviceToDevice, stream)
                                  : cudaMemsetAsync(a->dh0, 0, B * D * 16 * sizeof(float), stream);
      if (e != cudaSuccess) return MAMBA_ERR_CUDA;
    }
    if (a->dconv_state0) {
      cudaError_t e = a->dfinal_conv_state
                          ? mamba::launch_io_to_f32(io, a->dfinal_conv_state, a->dconv_state0, (long)(B * 3 * D), stream)
                          : cudaMemsetAsync(a->dconv_state0, 0, B * 3 * D * sizeof(float), stream);
      if (e != cudaSuccess) return MAMBA_ERR_CUDA;
    }
    return MAMBA_OK;
  }

  const void* io_ptrs[] = {a->x, a->z, a->dt_raw, a->Bm, a->Cm, a->dy, a->dx, a->dz, a->ddt_raw, a->dB, a->dC};
  for (const void* p : io_ptrs)
    if (!p || !aligned16(p)) return MAMBA_ERR_INVALID_ARG;
  if ((long long)a->seqlen * (long long)D > (1LL << 40)) return MAMBA_ERR_UNSUPPORTED;

  const Plan pl = make_plan(a->batch, a->seqlen, a->d_inner, a->n_chunks);
  const BwdWorkspace ws = bwd_workspace_layout(a->batch, a->seqlen, a->d_inner, pl);
  if (!a->workspace || a->workspace_bytes < ws.total) return MAMBA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0) return MAMBA_ERR_INVALID_ARG;
  char* wsp = static_cast<char*>(a->workspace);
  // the tile states: the caller's (from its forward call), or recomputed here
  const bool recompute = a->tile_states == nullptr;
  float* ckpt = recompute ? reinterpret_cast<float*>(wsp + ws.ckpt) : const_cast<float*>(a->tile_states);
  const uint64_t timeout = a->wait_timeout_ns ? a->wait_timeout_ns : kDefaultTimeoutNs;

  // The forward pass again, storing the state entering every tile (no y).
  mamba_scan_args fa;
  std::memset(&fa, 0, sizeof(fa));
  fa.batch = a->batch;
  fa.seqlen = a->seqlen;
  fa.d_inner = a->d_inner;
  fa.d_state = a->d_state;
  fa.d_conv = a->d_conv;
  fa.io = a->io;
  fa.x = a->x;
  fa.z = a->z;
  fa.dt_raw = a->dt_raw;
  fa.Bm = a->Bm;
  fa.Cm = a->Cm;
  fa.A_log = a->A_log;
  fa.Dskip = a->Dskip;
  fa.conv_w = a->conv_w;
  fa.conv_b = a->conv_b;
  fa.h0 = a->h0;
  fa.conv_state0 = a->conv_state0;
  fa.workspace = a->workspace;
  fa.workspace_bytes = a->workspace_bytes;
  fa.wait_timeout_ns = timeout;
  fa.flags = a->flags & MAMBA_FLAG_EXACT_CARRY;
  const mamba::ScanParams fp = fwd_params(&fa, pl, ws.fwd, ckpt);

  float* bc = reinterpret_cast<float*>(wsp + ws.fwd.bc);
  CUtensorMap maps[5];  // x, z, dt_raw, dy, bc
  if (!encode3d(&maps[0], a->x, a->io, a->d_inner, a->seqlen, a->batch, kLanes) ||
      !encode3d(&maps[1], a->z, a->io, a->d_inner, a->seqlen, a->batch, kLanes) ||
      !encode3d(&maps[2], a->dt_raw, a->io, a->d_inner, a->seqlen, a->batch, kLanes) ||
      !encode3d(&maps[3], a->dy, a->io, a->d_inner, a->seqlen, a->batch, kLanes) ||
      !encode3d(&maps[4], bc, MAMBA_F32, 32, a->seqlen, a->batch, 32))
    return MAMBA_ERR_CUDA;

  mamba::BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.batch = a->batch;
  p.seqlen = a->seqlen;
  p.d_inner = a->d_inner;
  p.n_groups = (a->d_inner + kLanes - 1) / kLanes;
  p.chunk_tiles = pl.chunk_tiles;
  p.n_chunks = pl.n_chunks;
  p.piece_tiles = pl.piece_tiles;
  p.pieces = pl.pieces;
  p.seq_tiles = (a->seqlen + kT - 1) / kT;
  p.A_log = a->A_log;
  p.Dskip = a->Dskip;
  p.conv_w = a->conv_w;
  p.conv_b = a->conv_b;
  p.conv_state0 = a->conv_state0;
  p.x = a->x;
  p.ckpt = ckpt;
  p.dfinal_h = a->dfinal_h;
  p.dfinal_conv_state = a->dfinal_conv_state;
  p.dx = a->dx;
  p.dz = a->dz;
  p.ddt_raw = a->ddt_raw;
  p.part_bc = reinterpret_cast<float*>(wsp + ws.part_bc);
  p.part_param = reinterpret_cast<float*>(wsp + ws.part_param);
  p.dh0 = a->dh0;
  p.dconv_state0 = a->dconv_state0;
  p.flags = a->flags & MAMBA_FLAG_EXACT_CARRY;
  p.timeout_ns = timeout;

  // 1. B/C rows widened; 2. chunked mode: the forward's chunk carries (when
  // the forward is recomputed) and the adjoint carries, in one launch; 3. the
  // states-only forward pass (when recomputed); 4. the reverse sweep; 5. the
  // edge fix-up and the fixed-order sums
  if (mamba::launch_bc_widen(io, a->Bm, a->Cm, bc, (long)B * a->seqlen, 16, stream) != cudaSuccess)
    return MAMBA_ERR_CUDA;
  if (pl.n_chunks > 1) {
    p.acarry = reinterpret_cast<float*>(wsp + ws.acarry);
    p.counters = reinterpret_cast<unsigned*>(wsp + ws.counters);
    p.edge_dx = reinterpret_cast<float*>(wsp + ws.edge_dx);
    p.edge_dpre = reinterpret_cast<float*>(wsp + ws.edge_dpre);
    if ((recompute && cudaMemsetAsync(fp.counters, 0, ws.fwd.counters_bytes, stream) != cudaSuccess) ||
        cudaMemsetAsync(p.counters, 0, ws.counters_bytes, stream) != cudaSuccess)
      return MAMBA_ERR_CUDA;
    const unsigned n_each = (unsigned)((size_t)(pl.n_chunks - 1) * p.n_groups * B);
    if (mamba::launch_carries(io, maps, fp, p, recompute ? n_each : 0u, n_each, stream) != cudaSuccess)
      return MAMBA_ERR_CUDA;
  }
  dim3 grid((unsigned)p.n_groups, (unsigned)B, (unsigned)pl.n_chunks);
  if (recompute) {
    const CUtensorMap fmaps[4] = {maps[0], maps[1], maps[2], maps[4]};  // x, z (unused), dt_raw, bc
    if (mamba::launch_scan(io, fmaps, fp, grid, stream) != cudaSuccess) return MAMBA_ERR_CUDA;
  }
  if (mamba::launch_bwd(io, maps, p, grid, stream) != cudaSuccess) return MAMBA_ERR_CUDA;
  if (mamba::launch_bwd_finish(io, p, a->dB, a->dC, a->dA_log, a->dDskip, a->dconv_w, a->dconv_b, stream) !=
      cudaSuccess)
    return MAMBA_ERR_CUDA;
  return MAMBA_OK;
}

size_t mamba_layer_workspace_size(int batch, int seqlen, int d_model, int d_inner, int dt_rank, int n_chunks,
                                  int with_u_out) {
  if (batch <= 0 || seqlen <= 0 || d_model <= 0 || d_inner <= 0 || d_inner % 4 || dt_rank <= 0 ||
      n_chunks < 0)
    return 0;
  return layer_workspace_layout(batch, seqlen, d_inner, dt_rank, make_plan(batch, seqlen, d_inner, n_chunks),
                                with_u_out == 0)
      .total;
}

mamba_status mamba_layer_fwd(const mamba_layer_args* a, void* stream_v) {
  if (!a) return MAMBA_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_v);
  mamba_status st = check_common(a->batch, a->d_inner, a->d_state, a->d_conv, a->io);
  if (st != MAMBA_OK) return st;
  if (a->io != MAMBA_BF16) return MAMBA_ERR_UNSUPPORTED;
  if (a->seqlen <= 0 || a->d_model <= 0 || a->dt_rank <= 0 || a->n_chunks < 0) return MAMBA_ERR_INVALID_ARG;
  // 16-byte rows for the tensor-core GEMMs
  if (a->d_model % 8 || a->dt_rank % 8) return MAMBA_ERR_UNSUPPORTED;
  const void* req[] = {a->hidden, a->W_in, a->conv_w, a->W_x, a->W_dt, a->A_log, a->Dskip, a->W_out, a->out};
  for (const void* p : req)
    if (!p || !aligned16(p)) return MAMBA_ERR_INVALID_ARG;
  const void* opt[] = {a->conv_b, a->b_dt, a->u_out, a->final_h, a->final_conv_state};
  for (const void* p : opt)
    if (p && !aligned16(p)) return MAMBA_ERR_INVALID_ARG;
  if ((long long)a->seqlen * (long long)a->d_inner > (1LL << 40)) return MAMBA_ERR_UNSUPPORTED;

  const Plan pl = make_plan(a->batch, a->seqlen, a->d_inner, a->n_chunks);
  const LayerWorkspace ws = layer_workspace_layout(a->batch, a->seqlen, a->d_inner, a->dt_rank, pl, !a->u_out);
  if (!a->workspace || a->workspace_bytes < ws.total) return MAMBA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0) return MAMBA_ERR_INVALID_ARG;
  char* wsp = static_cast<char*>(a->workspace);
  const long M = (long)a->batch * a->seqlen;
  const int H = a->d_model, D = a->d_inner, R = a->dt_rank, XD = a->dt_rank + 32;
  void* x = wsp + ws.x;
  void* z = wsp + ws.z;
  void* u = a->u_out ? a->u_out : static_cast<void*>(wsp + ws.u);
  char* xdbl = wsp + ws.xdbl;
  void* dt_raw = wsp + ws.dt_raw;
  void* y = wsp + ws.y;
  const uint64_t timeout = kDefaultTimeoutNs;
  const char* W_in = static_cast<const char*>(a->W_in);

  // in_proj (two halves: x and z, each contiguous), conv + SiLU, x_proj
  // (dt input | B | C per token), dt_proj with its bias
  if ((st = tc_linear(a->hidden, H, W_in, nullptr, x, D, M, D, H, timeout, stream)) != MAMBA_OK ||
      (st = tc_linear(a->hidden, H, W_in + (size_t)D * H * 2, nullptr, z, D, M, D, H, timeout, stream)) != MAMBA_OK)
    return st;
  if (mamba::launch_conv_silu(IoType::BF16, x, a->conv_w, a->conv_b, u, a->batch, a->seqlen, D, stream) !=
      cudaSuccess)
    return MAMBA_ERR_CUDA;
  if ((st = tc_linear(u, D, a->W_x, nullptr, xdbl, XD, M, XD, D, timeout, stream)) != MAMBA_OK ||
      (st = tc_linear(xdbl, XD, a->W_dt, a->b_dt, dt_raw, D, M, D, R, timeout, stream)) != MAMBA_OK)
    return st;

  // the scan, B and C read in place from the x_proj output
  mamba_scan_args sa;
  std::memset(&sa, 0, sizeof(sa));
  sa.batch = a->batch;
  sa.seqlen = a->seqlen;
  sa.d_inner = D;
  sa.d_state = a->d_state;
  sa.d_conv = a->d_conv;
  sa.io = MAMBA_BF16;
  sa.x = x;
  sa.z = z;
  sa.dt_raw = dt_raw;
  sa.Bm = xdbl + (size_t)R * 2;
  sa.Cm = xdbl + (size_t)(R + 16) * 2;
  sa.A_log = a->A_log;
  sa.Dskip = a->Dskip;
  sa.conv_w = a->conv_w;
  sa.conv_b = a->conv_b;
  sa.y = y;
  sa.final_h = a->final_h;
  sa.final_conv_state = a->final_conv_state;
  sa.workspace = wsp + ws.scan;
  sa.workspace_bytes = ws.scan_ws.total;
  st = launch_forward(&sa, pl, ws.scan_ws, stream, XD);
  if (st != MAMBA_OK) return st;

  // out_proj
  if ((st = tc_linear(y, D, a->W_out, nullptr, a->out, H, M, H, D, timeout, stream)) != MAMBA_OK) return st;
  return MAMBA_OK;
}

constexpr int kSsdChunk = 128;  // tokens per chunk of Mamba-2's scan

size_t mamba2_scan_workspace_size(int batch, int seqlen, int heads) {
  if (batch <= 0 || seqlen <= 0 || heads <= 0) return 0;
  const size_t nC = ((size_t)seqlen + kSsdChunk - 1) / kSsdChunk, BH = (size_t)batch * heads;
  return 2 * round256(BH * nC * 16 * 64 * sizeof(float)) + round256(BH * nC * sizeof(float)) +
         round256(BH * nC * kSsdChunk * 2 * sizeof(float));
}

// 4-D map over a bf16 tensor (B, L, R, inner), rows of `inner` elements, read
// or written in boxes of inner x 1 x `rows` tokens x 1 with the given swizzle.
bool encode4d_tokens(CUtensorMap* m, const void* base, int inner, int R, int L, int B, CUtensorMapSwizzle swizzle,
                     int rows = kSsdChunk) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[4] = {(cuuint64_t)inner, (cuuint64_t)R, (cuuint64_t)L, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)inner * 2, (cuuint64_t)inner * 2 * R, (cuuint64_t)inner * 2 * R * L};
  cuuint32_t box[4] = {(cuuint32_t)inner, 1, (cuuint32_t)rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

mamba_status mamba2_scan_fwd(const mamba2_scan_args* a, void* stream_v) {
  if (!a) return MAMBA_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_v);
  if (a->batch <= 0 || a->heads <= 0 || a->groups <= 0 || a->seqlen < 0) return MAMBA_ERR_INVALID_ARG;
  if (a->io != MAMBA_BF16 || a->head_dim != 64 || a->d_state != MAMBA_D_STATE || a->heads % a->groups)
    return MAMBA_ERR_UNSUPPORTED;
  if (!a->A_log || !a->Dskip) return MAMBA_ERR_INVALID_ARG;
  const void* al[] = {a->A_log, a->Dskip, a->h0, a->final_state, a->z};
  for (const void* p : al)
    if (p && !aligned16(p)) return MAMBA_ERR_INVALID_ARG;
  const size_t BH = (size_t)a->batch * a->heads;
  if (a->seqlen == 0) {
    if (a->final_state && a->final_state != a->h0) {
      cudaError_t e = a->h0 ? cudaMemcpyAsync(a->final_state, a->h0, BH * 16 * 64 * sizeof(float),
                                              cudaMemcpyDeviceToDevice, stream)
                            : cudaMemsetAsync(a->final_state, 0, BH * 16 * 64 * sizeof(float), stream);
      if (e != cudaSuccess) return MAMBA_ERR_CUDA;
    }
    return MAMBA_OK;
  }
  const void* io[] = {a->x, a->dt_raw, a->Bm, a->Cm, a->y};
  for (const void* p : io)
    if (!p || !aligned16(p)) return MAMBA_ERR_INVALID_ARG;
  const size_t need = mamba2_scan_workspace_size(a->batch, a->seqlen, a->heads);
  if (!a->workspace || a->workspace_bytes < need) return MAMBA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0) return MAMBA_ERR_INVALID_ARG;
  const int nC = (a->seqlen + kSsdChunk - 1) / kSsdChunk;
  char* w = static_cast<char*>(a->workspace);
  const size_t st = round256(BH * nC * 16 * 64 * sizeof(float));
  mamba::SsdParams p;
  std::memset(&p, 0, sizeof(p));
  p.batch = a->batch;
  p.seqlen = a->seqlen;
  p.heads = a->heads;
  p.groups = a->groups;
  p.n_chunks = nC;
  p.x = a->x;
  p.z = a->z;
  p.dt_raw = a->dt_raw;
  p.Bm = a->Bm;
  p.Cm = a->Cm;
  p.A_log = a->A_log;
  p.Dskip = a->Dskip;
  p.h0 = a->h0;
  p.y = a->y;
  p.final_state = a->final_state;
  p.S_c = reinterpret_cast<float*>(w);
  p.S_in = reinterpret_cast<float*>(w + st);
  p.totals = reinterpret_cast<float*>(w + 2 * st);
  p.cum = reinterpret_cast<float*>(w + 2 * st + round256(BH * nC * sizeof(float)));
  p.timeout_ns = kDefaultTimeoutNs;
  CUtensorMap maps[5];  // x, z, B, C, y (y stored 32 tokens at a time)
  const int H = a->heads, G = a->groups, L = a->seqlen, Bt = a->batch;
  if (!encode4d_tokens(&maps[0], a->x, 64, H, L, Bt, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode4d_tokens(&maps[1], a->z ? a->z : a->x, 64, H, L, Bt, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !encode4d_tokens(&maps[2], a->Bm, 16, G, L, Bt, CU_TENSOR_MAP_SWIZZLE_32B) ||
      !encode4d_tokens(&maps[3], a->Cm, 16, G, L, Bt, CU_TENSOR_MAP_SWIZZLE_32B) ||
      !encode4d_tokens(&maps[4], a->y, 64, H, L, Bt, CU_TENSOR_MAP_SWIZZLE_128B, 32))
    return MAMBA_ERR_CUDA;
  if (mamba::launch_ssd(maps, p, stream) != cudaSuccess) return MAMBA_ERR_CUDA;
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
  const void* al[] = {a->h, a->A_log, a->conv_w, a->conv_b, a->B_t, a->C_t};
  for (const void* p : al)
    if (p && !aligned16(p)) return MAMBA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(a->h) & 31u) != 0) return MAMBA_ERR_INVALID_ARG;  // 32-byte accesses
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
  p.timeout_ns = kDefaultTimeoutNs;
  p.y_t = a->y_t;
  const IoType io = a->io == MAMBA_BF16 ? IoType::BF16 : IoType::F32;
  if (mamba::launch_step(io, p, stream) != cudaSuccess) return MAMBA_ERR_CUDA;
  return MAMBA_OK;
}

size_t mamba3_scan_workspace_size(int batch, int seqlen, int d_inner, int n_chunks) {
  if (batch <= 0 || seqlen <= 0 || d_inner <= 0 || d_inner % 4 || n_chunks < 0) return 0;
  return complex_workspace_layout(batch, seqlen, d_inner, complex_plan(batch, seqlen, d_inner, n_chunks)).total;
}

mamba_status mamba3_scan_fwd(const mamba3_scan_args* a, void* stream_v) {
  if (!a) return MAMBA_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_v);
  mamba_status st = check_common(a->batch, a->d_inner, a->d_state, a->d_conv, a->io);
  if (st != MAMBA_OK) return st;
  if (a->seqlen < 0 || a->n_chunks < 0) return MAMBA_ERR_INVALID_ARG;
  if (a->discretization != MAMBA3_EULER && a->discretization != MAMBA3_TRAPEZOIDAL) return MAMBA_ERR_UNSUPPORTED;
  if (!a->A_log || !a->theta || !a->Dskip || !a->conv_w) return MAMBA_ERR_INVALID_ARG;
  const void* aligned_ptrs[] = {a->A_log, a->theta, a->Dskip, a->conv_w, a->conv_b, a->h0, a->conv_state0,
                                a->v0, a->final_h, a->final_v, a->final_conv_state};
  for (const void* p : aligned_ptrs)
    if (p && !aligned16(p)) return MAMBA_ERR_INVALID_ARG;
  const size_t B = a->batch, D = a->d_inner, es = esize(a->io);
  if (a->seqlen == 0) {
    // nothing to scan: the final states are the initial ones
    const void* src[] = {a->h0, a->v0, a->conv_state0};
    void* dst[] = {a->final_h, a->final_v, a->final_conv_state};
    const size_t bytes[] = {B * D * 16 * sizeof(float), B * D * 16 * sizeof(float), B * 3 * D * es};
    for (int i = 0; i < 3; ++i) {
      if (!dst[i] || dst[i] == src[i]) continue;
      cudaError_t e = src[i] ? cudaMemcpyAsync(dst[i], src[i], bytes[i], cudaMemcpyDeviceToDevice, stream)
                             : cudaMemsetAsync(dst[i], 0, bytes[i], stream);
      if (e != cudaSuccess) return MAMBA_ERR_CUDA;
    }
    return MAMBA_OK;
  }
  const void* io_ptrs[] = {a->x, a->z, a->dt_raw, a->Bm, a->Cm, a->y};
  for (const void* p : io_ptrs)
    if (!p || !aligned16(p)) return MAMBA_ERR_INVALID_ARG;
  if ((long long)a->seqlen * (long long)D > (1LL << 40)) return MAMBA_ERR_UNSUPPORTED;

  const Plan pl = complex_plan(a->batch, a->seqlen, a->d_inner, a->n_chunks);
  const ComplexWorkspace ws = complex_workspace_layout(a->batch, a->seqlen, a->d_inner, pl);
  if (!a->workspace || a->workspace_bytes < ws.total) return MAMBA_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0) return MAMBA_ERR_INVALID_ARG;
  char* wsp = static_cast<char*>(a->workspace);
  float* bc = reinterpret_cast<float*>(wsp + ws.bc);

  CUtensorMap maps[4];  // x, z, dt_raw, bc
  if (!encode3d(&maps[0], a->x, a->io, a->d_inner, a->seqlen, a->batch, kLanes) ||
      !encode3d(&maps[1], a->z, a->io, a->d_inner, a->seqlen, a->batch, kLanes) ||
      !encode3d(&maps[2], a->dt_raw, a->io, a->d_inner, a->seqlen, a->batch, kLanes) ||
      !encode3d(&maps[3], bc, MAMBA_F32, 32, a->seqlen, a->batch, 32))
    return MAMBA_ERR_CUDA;

  mamba::ComplexParams p;
  std::memset(&p, 0, sizeof(p));
  p.batch = a->batch;
  p.seqlen = a->seqlen;
  p.d_inner = a->d_inner;
  p.n_groups = (a->d_inner + kLanes - 1) / kLanes;
  p.chunk_tiles = pl.chunk_tiles;
  p.n_chunks = pl.n_chunks;
  p.A_log = a->A_log;
  p.theta = a->theta;
  p.Dskip = a->Dskip;
  p.conv_w = a->conv_w;
  p.conv_b = a->conv_b;
  p.h0 = a->h0;
  p.conv_state0 = a->conv_state0;
  p.v0 = a->v0;
  p.x = a->x;
  p.y = a->y;
  p.final_h = a->final_h;
  p.final_v = a->final_v;
  p.final_conv_state = a->final_conv_state;
  p.bc = bc;
  p.timeout_ns = a->wait_timeout_ns ? a->wait_timeout_ns : kDefaultTimeoutNs;
  p.flags = a->flags & MAMBA_FLAG_EXACT_CARRY;
  p.piece_tiles = pl.piece_tiles;
  p.pieces = pl.pieces;
  const bool walked = pl.n_chunks > 1 && p.flags == 0;
  if (pl.n_chunks > 1) {
    p.hloc = reinterpret_cast<float*>(wsp + ws.hloc);
    p.sdt = reinterpret_cast<float*>(wsp + ws.sdt);
    p.carry = reinterpret_cast<float*>(wsp + ws.carry);
    p.counters = reinterpret_cast<unsigned*>(wsp + ws.counters);
    if (walked && (size_t)(2 * pl.n_chunks - 1) * p.n_groups * B >= (1u << 31)) return MAMBA_ERR_UNSUPPORTED;
  }
  const IoType io = a->io == MAMBA_BF16 ? IoType::BF16 : IoType::F32;
  // the widening also zeroes the walked mode's ticket and flags
  if (mamba::launch_bc_widen(io, a->Bm, a->Cm, bc, (long)B * a->seqlen, 16, stream, walked ? p.counters : nullptr,
                             walked ? (int)(ws.counters_bytes / sizeof(unsigned)) : 0, false, true) != cudaSuccess)
    return MAMBA_ERR_CUDA;
  if (mamba::launch_complex(io, a->discretization == MAMBA3_TRAPEZOIDAL, maps, p, stream) != cudaSuccess)
    return MAMBA_ERR_CUDA;
  return MAMBA_OK;
}

mamba_status mamba_linear_fwd(const mamba_linear_args* a, void* stream_v) {
  if (!a) return MAMBA_ERR_INVALID_ARG;
  if (a->M < 0 || a->N <= 0 || a->K <= 0 || a->lda < a->K || a->ldc < a->N) return MAMBA_ERR_INVALID_ARG;
  if (a->M == 0) return MAMBA_OK;  // nothing to compute (an empty A or C may have no address)
  if (!a->A || !a->W || !a->C) return MAMBA_ERR_INVALID_ARG;
  const void* al[] = {a->A, a->W, a->C, a->bias};
  for (const void* p : al)
    if (p && !aligned16(p)) return MAMBA_ERR_INVALID_ARG;
  if (a->K % 8 || a->lda % 8 || a->ldc % 8) return MAMBA_ERR_UNSUPPORTED;
  return tc_linear(a->A, a->lda, a->W, a->bias, a->C, a->ldc, a->M, a->N, a->K,
                   a->wait_timeout_ns ? a->wait_timeout_ns : kDefaultTimeoutNs, reinterpret_cast<cudaStream_t>(stream_v));
}

mamba_status mamba_last_error(void* stream_v) {
  unsigned code = 0;
  if (mamba::take_device_error(&code, reinterpret_cast<cudaStream_t>(stream_v)) != cudaSuccess)
    return MAMBA_ERR_CUDA;
  return static_cast<mamba_status>(code);
}

}  // extern "C"
