// params.h -- kernel parameter blocks (plain structs shared by the launchers
// and the kernels).
#pragma once
#include <cstddef>
#include <cstdint>

namespace mamba {

// Tokens per tile: the unit of the TMA ring and of every chunk and piece.
constexpr int kTileTokens = 16;

// Bits of ScanParams::flags / BwdParams::flags (the public MAMBA_FLAG_*).
constexpr uint32_t kFlagTestStallFirstLoad = 1u;
constexpr uint32_t kFlagExactCarry = 2u;  // chunk-carry walks never drop decayed terms

struct ScanParams {
  int batch, seqlen, d_inner;
  int n_groups;     // ceil(d_inner / 32): one CTA (warp) per group of 32 channels
  int chunk_tiles;  // tiles of kTileTokens tokens per chunk
  int n_chunks;     // chunks of the sequence run in parallel (1: one pass)
  int piece_tiles;  // tiles per carry piece (chunked mode)
  int pieces;       // pieces per chunk = ceil(chunk_tiles / piece_tiles)
  const float* A_log;
  const float* Dskip;
  const float* conv_w;
  const float* conv_b;       // may be null
  const float* h0;           // may be null
  const void* conv_state0;   // may be null
  const void* x;             // plain pointer to x, for the conv inputs before a chunk
  void* y;
  float* final_h;            // may be null
  void* final_conv_state;    // may be null
  float* carry;              // chunked: (B, n_chunks, D, 16) carried-in states (entry 0 unused)
  unsigned* counters;        // chunked: [0] ticket counter, then (B, n_groups, n_chunks) ready
                             // flags; zeroed before every call
  float* ckpt;               // may be null: (B, seq_tiles, D, 16) state entering every tile
  int seq_tiles;             // tiles of the whole sequence (rows of ckpt)
  uint32_t flags;
  uint64_t timeout_ns;
};

// The backward pass (scan_bwd.cuh).  Sizes and plan as in ScanParams; the
// forward states entering every tile come from a checkpointing forward pass.
struct BwdParams {
  int batch, seqlen, d_inner;
  int n_groups, chunk_tiles, n_chunks, piece_tiles, pieces, seq_tiles;
  const float* A_log;
  const float* Dskip;
  const float* conv_w;
  const float* conv_b;              // may be null
  const void* conv_state0;          // may be null
  const void* x;                    // plain pointer to x (conv inputs before a tile)
  const float* ckpt;                // (B, seq_tiles, D, 16)
  const float* dfinal_h;            // (B, D, 16) or null
  const void* dfinal_conv_state;    // (B, 3, D) I/O dtype, or null
  float* acarry;                    // chunked: (B, n_chunks, D, 16) adjoint entering chunk j
                                    // from its right (j < n_chunks - 1)
  unsigned* counters;               // chunked: ticket counter, then (B, n_groups, n_chunks) flags
  void* dx;                         // (B, L, D) I/O dtype
  void* dz;
  void* ddt_raw;
  float* part_bc;                   // (n_groups, B * L, 32): per group sums of dB | dC
  float* part_param;                // (B * n_chunks, D, 24): dA_log(16), dD, dconv_w(4), dconv_b
  float* edge_dx;                   // (B, n_chunks, 3, D): dx of a chunk's last 3 tokens, partial
  float* edge_dpre;                 // (B, n_chunks, 3, D): d(conv output) of its first 3 tokens
  float* dh0;                       // (B, D, 16) or null
  float* dconv_state0;              // (B, 3, D) fp32 or null
  uint32_t flags;                   // kFlagExactCarry or 0
  uint64_t timeout_ns;
};

// Mamba-2's chunked scan (ssd.cuh): heads of 64 channels sharing one scalar
// decay per token, 16 x 64 state per head, chunks of 128 tokens.
struct SsdParams {
  int batch, seqlen, heads, groups, n_chunks;
  const void* x;          // (B, L, H, 64) bf16
  const void* z;          // (B, L, H, 64) bf16 or null
  const void* dt_raw;     // (B, L, H) bf16
  const void* Bm;         // (B, L, G, 16) bf16
  const void* Cm;
  const float* A_log;     // (H)
  const float* Dskip;     // (H)
  const float* h0;        // (B, H, 16, 64) or null
  void* y;                // (B, L, H, 64) bf16
  float* final_state;     // (B, H, 16, 64) or null
  // chunk states, (B, H, n_chunks, 16, 64): one chunk's 16 x 64 state contiguous
  float* S_c;             // each chunk's end state from zero
  float* S_in;            // the state entering each chunk
  float* totals;          // (B, H, n_chunks): sum of dt * A (base 2) over each chunk
  float* cum;             // (B, H, n_chunks, 128, 2): per token, the prefix sum of dt * A and dt
  uint64_t timeout_ns;
};

// The complex-valued scan (scan_complex.cuh): 8 complex modes per channel,
// states and state inputs as 16 fp32 numbers (re, im pairs) per channel.
struct ComplexParams {
  int batch, seqlen, d_inner;
  int n_groups;     // ceil(d_inner / 32)
  int chunk_tiles;  // tiles of kTileTokens tokens per chunk
  int n_chunks;
  const float* A_log;        // (D, 8)
  const float* theta;        // (D, 8)
  const float* Dskip;
  const float* conv_w;
  const float* conv_b;       // may be null
  const float* h0;           // (B, D, 16) or null
  const void* conv_state0;   // (B, 3, D) or null
  const float* v0;           // (B, D, 16) or null: the state input before the first token
  const void* x;             // plain pointer to x, for the conv inputs before a chunk
  void* y;
  float* final_h;            // may be null
  float* final_v;            // may be null
  void* final_conv_state;    // may be null
  const float* bc;           // widened B/C rows (B, L, 32): per mode (Re B, Im B, Re C, Im C)
  float* hloc;               // exact chunked: (B, n_chunks, D, 16) each chunk's end state from zero
  float* sdt;                // exact chunked: (B, n_chunks, D) each chunk's dt sum
  float* carry;              // chunked: (B, n_chunks, D, 16) the state entering each chunk
  unsigned* counters;        // walked chunked mode: ticket, then per (row, group, chunk) a flag
  int piece_tiles;           // walked chunked mode: tiles per carry piece
  int pieces;                // pieces per chunk
  unsigned flags;            // kFlagExactCarry: the exact three-pass chunked mode
  uint64_t timeout_ns;
};

// The tensor-core GEMM (gemm_tc.cuh): row-major C (M x N, bf16, rows ldc
// elements apart) = A W^T [+ bias]; A and W are read through tensor maps.
struct GemmParams {
  long M;
  int N, K;
  int bn;              // columns of an output tile (a multiple of 32, at most 256)
  int ldc;
  void* C;             // bf16
  const void* bias;    // (N) bf16 or null
  uint64_t timeout_ns;
};

struct StepParams {
  int batch, d_inner;
  float* h;           // (B, D, 16)
  void* conv_state;   // (B, 3, D)
  const void* x_t;    // (B, D)
  const void* z_t;
  const void* dt_raw_t;
  const void* B_t;    // (B, 16)
  const void* C_t;
  const float* A_log;
  const float* Dskip;
  const float* conv_w;
  const float* conv_b;  // may be null
  void* y_t;          // (B, D)
  uint64_t timeout_ns;  // limit of the wait for a block of h
};

}  // namespace mamba
