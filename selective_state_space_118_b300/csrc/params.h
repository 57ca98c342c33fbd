// params.h -- kernel parameter blocks (plain structs shared by the launchers
// and the kernels).
#pragma once
#include <cstddef>
#include <cstdint>

namespace mamba {

struct ScanParams {
  int batch, seqlen, d_inner;
  int chunk_len;  // tokens per chunk, a multiple of kT
  int n_chunks;
  const float* A_log;
  const float* Dskip;
  const float* conv_w;
  const float* conv_b;       // may be null
  const float* h0;           // may be null
  const void* conv_state0;   // may be null
  const void* x;             // plain pointer to x, for the conv halo at chunk starts
  float* final_h;            // may be null
  void* final_conv_state;    // may be null
  float* carry;              // chunked: (B, n_chunks, D, 16) carried-in states
  float* hloc;               // chunked: (B, n_chunks-1, D, 16) chunk end states from zero
  float* sum_dt;             // chunked: (B, n_chunks-1, D)
  unsigned* counters;        // chunked: (B, D/16) arrival counters, zero between calls
  uint32_t flags;
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
};

}  // namespace mamba
