/*
 * mamba_ssm.h -- C ABI of the B300 (sm_103a) Mamba selective-scan library
 * (libmamba_ssm.so).
 *
 * The operation.  A Mamba layer's selective state-space scan, as built in
 * "【大模型】- Jamba 混合 SSM-Transformer" (sxl-space.tk), section
 * "实现 > Mamba 层" (MambaBlock.forward and MambaBlock.ssm), with the
 * read-out y_t = C h_t of the lesson "Jamba -- SSM-Transformer Hibrido"
 * (ai-engineering.academy), section "Um SSM em uma pagina".  For every batch
 * row b and channel c, with A_n = -exp(A_log[c,n]) and t = 0..L-1:
 *
 *   u    = silu(conv_b[c] + sum_{k=0..3} conv_w[c,k] * x[b,t-3+k,c])
 *          (causal depthwise conv, d_conv = 4; inputs before t = 0 come from
 *           conv_state0, or are zero)
 *   dt   = softplus(dt_raw[b,t,c])          (beta 1, threshold 20)
 *   h_n  = exp(dt*A_n) * h_n + dt*B[b,t,n]*u  (n = 0..15; h starts at h0 or 0)
 *   y    = (sum_n C[b,t,n]*h_n + D[c]*u) * silu(z[b,t,c])
 *
 * The scan calls take the results of the projections around the scan
 * (in_proj producing x and z, x_proj producing B, C and the dt input,
 * dt_proj) from the caller; mamba_layer_fwd below runs the projections too.
 *
 * Conventions for every call below.
 *  - All tensor pointers are DEVICE pointers (CUDA global memory), row-major
 *    and contiguous, 16-byte aligned, owned by the caller.  The library never
 *    allocates, frees or keeps them.
 *  - `io` tensors (activations) are fp32 or bf16 as chosen by `io`;
 *    parameters and the SSM state h are always fp32.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and never synchronise.  Argument errors are reported
 *    before anything is launched; a launch failure returns MAMBA_ERR_CUDA.
 *  - d_state must be 16 and d_conv 4 (the layer's defaults); d_inner must be
 *    a multiple of 8 for bf16 I/O and of 4 for fp32 (the channel rows are
 *    read by bulk tensor copies, whose row stride must be a multiple of 16
 *    bytes).  The size and plan queries, which take no dtype, accept any
 *    multiple of 4.
 *  - A device-side wait that gives up (it cannot, in a healthy run) sets a
 *    sticky error word that mamba_last_error() reports.
 */
#ifndef MAMBA_SSM_H
#define MAMBA_SSM_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MAMBA_OK = 0,
    MAMBA_ERR_INVALID_ARG = 1,   /* null required pointer, bad size, misalignment */
    MAMBA_ERR_UNSUPPORTED = 2,   /* d_state != 16, d_conv != 4, d_inner not a multiple of 8 (bf16) or 4 (fp32), dtype */
    MAMBA_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed */
    MAMBA_ERR_TIMEOUT = 4,       /* a device-side wait gave up (sticky, see below) */
    MAMBA_ERR_WORKSPACE = 5      /* workspace missing or smaller than required */
} mamba_status;

typedef enum { MAMBA_F32 = 0, MAMBA_BF16 = 1 } mamba_dtype;

#define MAMBA_D_STATE 16
#define MAMBA_D_CONV 4

/* Test switch for mamba_scan_args.flags: the kernel skips issuing its first
 * input copy and so waits on a barrier that never completes; the wait gives
 * up after wait_timeout_ns and the call reports MAMBA_ERR_TIMEOUT through
 * mamba_last_error().  Never set in normal use. */
#define MAMBA_FLAG_TEST_STALL_FIRST_LOAD 0x1u

/* Flag for mamba_scan_args.flags and mamba_scan_bwd_args.flags: exact chunk
 * carries.  In chunked mode (n_chunks > 1) the carry entering a chunk is
 * normally gathered by walking the previous chunk backwards until every
 * state has decayed below 2^-32 on its way to the boundary; what lies
 * further back is then dropped.  The dropped part is at most 2^-32 times the
 * size of the state where the walk stopped, far below fp32 rounding for
 * states of comparable size along the sequence; it can only show when a
 * state >= ~1e5 times larger than the state at the boundary was hidden from
 * y (zero C, D and gate) while it decayed.  With this flag every walk covers
 * its whole chunk and folds in the carry before it: the result then equals
 * the sequential recurrence up to rounding for any inputs, at the cost of a
 * carry pass as long as the main pass.  No effect with n_chunks = 1. */
#define MAMBA_FLAG_EXACT_CARRY 0x2u

/*
 * Prefill: the scan over a whole sequence (MambaBlock.forward minus the
 * projections).
 *
 *   x, z, dt_raw      (B, L, D) io        inputs (read once)
 *   Bm, Cm            (B, L, 16) io       per-token B and C rows
 *   A_log             (D, 16) fp32        A = -exp(A_log)
 *   Dskip             (D) fp32            D, the skip weight
 *   conv_w            (D, 4) fp32         conv taps; conv_w[c,3] multiplies x_t
 *   conv_b            (D) fp32 or NULL    conv bias (NULL: zero)
 *   h0                (B, D, 16) fp32 or NULL     initial state (NULL: zero)
 *   conv_state0       (B, 3, D) io or NULL        the 3 inputs before t = 0,
 *                                                 oldest first (NULL: zero)
 *   y                 (B, L, D) io        output (written once)
 *   final_h           (B, D, 16) fp32 or NULL     state after the last token;
 *                                                 may alias h0
 *   final_conv_state  (B, 3, D) io or NULL        last 3 inputs; may alias
 *                                                 conv_state0
 *   workspace         device scratch of at least mamba_scan_workspace_size()
 *                     bytes, 256-byte aligned (B and C widened to fp32,
 *                     B*L*128 bytes, plus the chunk carries in chunked mode);
 *                     its contents need not be initialised and are not kept
 *   n_chunks          0: the library picks; 1: one sequential pass over L;
 *                     k > 1: L is cut into k chunks (a multiple of 16 tokens
 *                     each, the last one shorter) that run in parallel, each
 *                     chunk's carried-in state being the decayed end states of
 *                     the chunks before it, computed by a first pass over the
 *                     earlier chunks cut into pieces (two passes; results
 *                     agree with the sequential pass to rounding)
 *   flags             0, MAMBA_FLAG_EXACT_CARRY, or MAMBA_FLAG_TEST_* (tests
 *                     only)
 *   wait_timeout_ns   limit of every device-side wait (0: 1 second)
 *   tile_states       NULL, or (B, ceil(L/16), D, 16) fp32: the state entering
 *                     every 16-token tile is stored there (B*L*D*4 bytes,
 *                     rounded up to whole tiles), for mamba_scan_bwd
 *
 * seqlen may be 0 (then only final_h/final_conv_state are written: copies of
 * h0/conv_state0, or zeros).  batch and d_inner must be > 0.
 */
typedef struct mamba_scan_args {
    int batch, seqlen, d_inner, d_state, d_conv;
    mamba_dtype io;
    const void *x, *z, *dt_raw;
    const void *Bm, *Cm;
    const float *A_log, *Dskip, *conv_w, *conv_b;
    const float *h0;
    const void *conv_state0;
    void *y;
    float *final_h;
    void *final_conv_state;
    void *workspace;
    size_t workspace_bytes;
    int n_chunks;
    uint32_t flags;
    uint64_t wait_timeout_ns;
    float *tile_states;   /* NULL, or (B, ceil(L / 16), D, 16) fp32 output: the
                             state entering every 16-token tile, for a later
                             mamba_scan_bwd of the same inputs */
} mamba_scan_args;

/* Bytes of workspace mamba_scan_fwd needs for these sizes and n_chunks
 * (0 = the library's choice); 0 only for invalid sizes or seqlen 0. */
size_t mamba_scan_workspace_size(int batch, int seqlen, int d_inner, int n_chunks);

/* The number of chunks mamba_scan_fwd uses when n_chunks = 0. */
int mamba_scan_default_chunks(int batch, int seqlen, int d_inner);

/* The work plan mamba_scan_fwd follows for these sizes and n_chunks:
 * out[0] = chunks, out[1] = tokens per chunk (the last chunk may be shorter),
 * out[2] = summary pieces per chunk and out[3] = tokens per piece (both 0 for
 * one pass).  MAMBA_ERR_INVALID_ARG / _UNSUPPORTED as for the scan. */
mamba_status mamba_scan_plan(int batch, int seqlen, int d_inner, int n_chunks, int out[4]);

mamba_status mamba_scan_fwd(const mamba_scan_args *args, void *stream);

/*
 * Prefill without any allocation.  The pages have no counterpart of this
 * call: it exists for callers that cannot call cudaMalloc -- for instance a
 * plugin whose host framework owns all device memory through its own pool
 * and forbids allocations from outside it, or a latency-critical path where
 * cudaMalloc's implicit synchronisation is not acceptable.  It runs exactly
 * mamba_scan_fwd, with `workspace` and `workspace_bytes` ignored: the scratch
 * is a fixed array of MAMBA_NOALLOC_SCRATCH_BYTES (32 MiB) that the library
 * holds in every GPU that loads it, until the process exits.
 *
 *  - Calls whose mamba_scan_workspace_size() exceeds that size are rejected
 *    with MAMBA_ERR_WORKSPACE before anything runs (one sequential pass fits
 *    up to batch * seqlen = 262,144 tokens).
 *  - The array's device address belongs to the CUDA context the library's
 *    kernels are loaded into.  The first call in a context (the first on a
 *    device; again after cudaDeviceReset, or from a thread with another
 *    context of its own current) looks it up and remembers it for that
 *    context; make that first call before any stream capture.
 *  - All calls share the one array: calls that may overlap on the GPU (two
 *    streams, or two threads) race and corrupt each other's results; order
 *    them on one stream.  The array keeps the last call's contents; every
 *    call writes or clears everything it reads before reading it (the
 *    chunk counters are cleared at the start of each call).
 */
#define MAMBA_NOALLOC_SCRATCH_BYTES (32u << 20)

mamba_status mamba_scan_fwd_noalloc(const mamba_scan_args *args, void *stream);

/*
 * Backward of the prefill: the gradients of a scalar loss l with respect to
 * every input of mamba_scan_fwd, given dy = dl/dy and optionally
 * dl/dfinal_h and dl/dfinal_conv_state -- the chain rule through the
 * recurrence stated at the top of this file (for training the layer of
 * "实现 > Mamba 层"; the pages train it end to end but print no backward, so
 * this is the plain reverse-mode derivative of that forward).  Unless
 * tile_states is given, the forward pass is recomputed inside the call (it
 * stores the state entering every 16-token tile in the workspace), so
 * nothing from an earlier forward call is needed.
 *
 *   x, z, dt_raw, Bm, Cm, A_log, Dskip, conv_w, conv_b, h0, conv_state0
 *                     the forward's inputs, as for mamba_scan_fwd
 *   dy                (B, L, D) io        dl/dy
 *   dfinal_h          (B, D, 16) fp32 or NULL     dl/dfinal_h (NULL: zero)
 *   dfinal_conv_state (B, 3, D) io or NULL        dl/dfinal_conv_state
 *   dx, dz, ddt_raw   (B, L, D) io        outputs: dl/dx, dl/dz, dl/ddt_raw
 *   dB, dC            (B, L, 16) fp32     outputs: dl/dBm, dl/dCm (sums over
 *                                         the D channels, kept in fp32)
 *   dA_log            (D, 16) fp32        output
 *   dDskip            (D) fp32            output
 *   dconv_w           (D, 4) fp32         output
 *   dconv_b           (D) fp32 or NULL    output (NULL: not written; the
 *                                         bias may still be given)
 *   dh0               (B, D, 16) fp32 or NULL     output: dl/dh0 (the
 *                                         gradient at h0, or at zero)
 *   dconv_state0      (B, 3, D) fp32 or NULL      output: dl/dconv_state0
 *   workspace         at least mamba_scan_bwd_workspace_size() bytes,
 *                     256-byte aligned, contents need not be initialised:
 *                     the forward's workspace, the tile states (B*L*D*4
 *                     bytes, rounded up to whole tiles), the per-32-channel
 *                     sums of dB and dC (B*L*D*4 bytes) and smaller buffers
 *   n_chunks          as for mamba_scan_fwd (the same plan is used); in
 *                     chunked mode the adjoint entering each chunk from the
 *                     right is computed first, the way the forward computes
 *                     its carries, with time reversed
 *   flags             0 or MAMBA_FLAG_EXACT_CARRY (both the forward's carries
 *                     and the adjoint carries then walk whole chunks)
 *   wait_timeout_ns   limit of every device-side wait (0: 1 second)
 *   tile_states       NULL: the forward is recomputed inside the call, storing
 *                     the tile states in the workspace.  Or the tile_states
 *                     output of a mamba_scan_fwd of the same inputs: the
 *                     recomputation is skipped.  When that call had the same
 *                     n_chunks, the gradients are the same bits as with NULL
 *                     (the states are computed the same way in both passes);
 *                     with another n_chunks they differ by rounding only
 *
 * Every output is overwritten.  Results are deterministic (fixed summation
 * orders, no atomics).  seqlen may be 0: then dh0 = dfinal_h,
 * dconv_state0 = dfinal_conv_state (or zeros) and the parameter gradients
 * are zero.
 */
typedef struct mamba_scan_bwd_args {
    int batch, seqlen, d_inner, d_state, d_conv;
    mamba_dtype io;
    const void *x, *z, *dt_raw;
    const void *Bm, *Cm;
    const float *A_log, *Dskip, *conv_w, *conv_b;
    const float *h0;
    const void *conv_state0;
    const void *dy;
    const float *dfinal_h;
    const void *dfinal_conv_state;
    void *dx, *dz, *ddt_raw;
    float *dB, *dC;
    float *dA_log, *dDskip, *dconv_w, *dconv_b;
    float *dh0;
    float *dconv_state0;
    void *workspace;
    size_t workspace_bytes;
    int n_chunks;
    uint32_t flags;
    uint64_t wait_timeout_ns;
    const float *tile_states;  /* NULL, or the tile states a mamba_scan_fwd of the
                                  same inputs wrote: the forward is then not
                                  recomputed */
} mamba_scan_bwd_args;

/* Bytes of workspace mamba_scan_bwd needs (0 only for invalid sizes or
 * seqlen 0). */
size_t mamba_scan_bwd_workspace_size(int batch, int seqlen, int d_inner, int n_chunks);

mamba_status mamba_scan_bwd(const mamba_scan_bwd_args *args, void *stream);

/*
 * The whole Mamba layer of "实现 › Mamba 层" (MambaBlock.forward): the
 * projections around the scan as bf16 tensor-core GEMMs, then the scan.
 * For hidden (B, L, d_model):
 *
 *   x | z   = hidden W_in^T            (in_proj: W_in (2D, d_model); rows
 *                                        0..D-1 give x, D..2D-1 give z)
 *   u       = silu(conv(x))            (causal depthwise conv as for the scan;
 *                                        zero inputs before t = 0)
 *   dt_in | B | C = u W_x^T            (x_proj: W_x (dt_rank + 32, D); per
 *                                        token dt_rank values, then B's 16,
 *                                        then C's 16)
 *   dt_raw  = dt_in W_dt^T + b_dt      (dt_proj: W_dt (D, dt_rank))
 *   y       = the scan (mamba_scan_fwd) of x, z, dt_raw, B, C
 *   out     = y W_out^T                (out_proj: W_out (d_model, D))
 *
 * Every stored intermediate (x, z, u, the x_proj output, dt_raw, y) and out
 * is bf16; the GEMMs accumulate in fp32 on the tensor cores (the
 * tcgen05 GEMM of mamba_linear_fwd), the scan as for mamba_scan_fwd.  The pages'
 * x_proj yields no C; here it yields dt input, B and C, as in the layer the
 * pages describe in prose.
 *
 *   io                MAMBA_BF16 only
 *   hidden            (B, L, d_model) bf16
 *   W_in, W_x, W_dt, W_out   bf16, the nn.Linear weight layouts above
 *   b_dt              (D) bf16 or NULL (the dt_proj bias)
 *   conv_w, conv_b, A_log, Dskip   fp32, as for the scan
 *   out               (B, L, d_model) bf16 output
 *   u_out             (B, L, D) bf16 or NULL: u, for a caller that needs it
 *                     (e.g. to keep for the backward of x_proj)
 *   final_h, final_conv_state   as for the scan (may be NULL)
 *   workspace         at least mamba_layer_workspace_size() bytes, 256-byte
 *                     aligned: the intermediates and the scan's workspace
 *   n_chunks          the scan's, as for mamba_scan_fwd
 *
 * d_model, dt_rank and d_inner must be multiples of 8.
 */
typedef struct mamba_layer_args {
    int batch, seqlen, d_model, d_inner, dt_rank, d_state, d_conv;
    mamba_dtype io;
    const void *hidden;
    const void *W_in;
    const float *conv_w, *conv_b;
    const void *W_x, *W_dt, *b_dt;
    const float *A_log, *Dskip;
    const void *W_out;
    void *out;
    void *u_out;
    float *final_h;
    void *final_conv_state;
    void *workspace;
    size_t workspace_bytes;
    int n_chunks;
} mamba_layer_args;

/* Bytes of workspace mamba_layer_fwd needs (with_u_out: whether u_out will
 * be given; without it u lives in the workspace). */
size_t mamba_layer_workspace_size(int batch, int seqlen, int d_model, int d_inner, int dt_rank, int n_chunks,
                                  int with_u_out);

mamba_status mamba_layer_fwd(const mamba_layer_args *args, void *stream);

/*
 * Mamba-2's scan ("Jamba -- SSM-Transformer Hibrido", section "Mamba-3: a
 * linha de base de SSM puro em 2026", items 1-2: the state matrix a scaled
 * identity, Euler discretisation), in its chunked matrix form on the tensor
 * cores.  Channels come in heads of head_dim = 64 that share dt and A; each
 * head keeps a 16 x 64 state S.  For batch row b, head h (group g = h /
 * (heads / groups) of the B and C rows), t = 0..L-1:
 *
 *   dt      = softplus(dt_raw[b,t,h])
 *   S[n][p] = exp(dt * A_h) S[n][p] + dt B[b,t,g,n] x[b,t,h,p],  A_h = -exp(A_log[h])
 *   y[p]    = (sum_n C[b,t,g,n] S[n][p] + D_h x[b,t,h,p]) * silu(z[b,t,h,p])
 *
 * (the gate only when z is given; S starts at h0, or zero).
 *
 *   x, z, y           (B, L, heads, 64) bf16      (z may be NULL)
 *   dt_raw            (B, L, heads) bf16
 *   Bm, Cm            (B, L, groups, 16) bf16
 *   A_log, Dskip      (heads) fp32
 *   h0, final_state   (B, heads, 16, 64) fp32 or NULL
 *   workspace         mamba2_scan_workspace_size() bytes, 256-byte aligned:
 *                     per (batch row, head, chunk of 128 tokens) the chunk's
 *                     end state and entering state (16 x 64 fp32 each), its
 *                     decay sum, and per token its dt and decay prefix
 *
 * bf16 I/O only; head_dim 64 and d_state 16 only; heads % groups == 0.
 * seqlen may be 0 (then final_state = h0, or zeros).
 */
typedef struct mamba2_scan_args {
    int batch, seqlen, heads, head_dim, groups, d_state;
    mamba_dtype io;
    const void *x, *z, *dt_raw, *Bm, *Cm;
    const float *A_log, *Dskip, *h0;
    void *y;
    float *final_state;
    void *workspace;
    size_t workspace_bytes;
} mamba2_scan_args;

size_t mamba2_scan_workspace_size(int batch, int seqlen, int heads);

mamba_status mamba2_scan_fwd(const mamba2_scan_args *args, void *stream);

/*
 * The complex-valued scan: Mamba-3's state update, from the lesson
 * "Jamba -- SSM-Transformer Hibrido", section "Mamba-3: a linha de base de
 * SSM puro em 2026", item 2 (a complex-valued state, equal to a
 * data-dependent rotary embedding of the state) and item 1 (the
 * exponential-trapezoidal discretization).  The pages print no formula;
 * this library reads them as the Mamba layer of mamba_scan_fwd with its
 * diagonal state made complex.  Per channel c, M = 8 complex modes
 * (d_state = 16 real numbers, the real scan's state size):
 *
 *   u        = silu(conv(x)),  dt = softplus(dt_raw)      (as mamba_scan_fwd)
 *   lambda_n = -exp(A_log[c,n]) + i theta[c,n]
 *   alpha_n  = exp(dt lambda_n)       (decay, and a turn by the angle dt theta_n)
 *   v_n      = (Bm[b,t,2n] + i Bm[b,t,2n+1]) u                (state input)
 *   EULER:        h_n = alpha_n h_n + dt v_n
 *   TRAPEZOIDAL:  h_n = alpha_n (h_n + dt/2 vprev_n) + dt/2 v_n,  vprev = v
 *   y        = (Re(sum_n (Cm[b,t,2n] + i Cm[b,t,2n+1]) h_n) + D[c] u) silu(z)
 *
 * The trapezoidal rule weights the state inputs at both ends of the step
 * (the earlier one carried through the step's decay and turn); it reduces
 * to Euler's rule when the earlier end's weight is moved to the later end.
 *
 *   x, z, dt_raw      (B, L, D) io
 *   Bm, Cm            (B, L, 16) io       8 complex numbers as (re, im) pairs
 *   A_log, theta      (D, 8) fp32
 *   Dskip, conv_w, conv_b, conv_state0, final_conv_state, y   as for
 *                     mamba_scan_fwd
 *   h0, final_h       (B, D, 16) fp32 or NULL     complex state, (re, im)
 *                                                 pairs; final_h may alias h0
 *   v0, final_v       (B, D, 16) fp32 or NULL     the state input v of the
 *                     token before the first one (trapezoidal; NULL: zero)
 *                     and of the last token, so that a sequence split into
 *                     calls carrying (final_h, final_conv_state, final_v)
 *                     into (h0, conv_state0, v0) equals one call; final_v
 *                     may alias v0
 *   workspace         at least mamba3_scan_workspace_size() bytes, 256-byte
 *                     aligned, contents need not be initialised
 *   n_chunks          0: the library picks; 1: one sequential pass; k > 1:
 *                     k chunks in parallel.  The state entering each chunk
 *                     comes, as in mamba_scan_fwd, from a carry walk over
 *                     the chunk before it in 64-token pieces that stops once
 *                     every mode has decayed below 2^-32 from the piece's
 *                     start to the chunk boundary (the terms before it, of
 *                     weight below 2^-32 of their own size, are dropped), in
 *                     one launch with the main pass.  With
 *                     MAMBA_FLAG_EXACT_CARRY nothing is dropped: every chunk
 *                     but the last is first run from a zero state and those
 *                     end states are folded in chunk order (three launches)
 *   discretization    MAMBA3_EULER or MAMBA3_TRAPEZOIDAL
 *   wait_timeout_ns   limit of every device-side wait (0: 1 second)
 *   flags             0 or MAMBA_FLAG_EXACT_CARRY
 *
 * d_state must be 16, d_conv 4, d_inner as for mamba_scan_fwd.  seqlen may be 0
 * (the final states are then copies of the initial ones, or zeros).
 * Precision: a token whose dt keeps every turn dt theta_n of its channel
 * within [-pi, pi] (dt <= pi / max_n |theta_n|) takes the angle as the fp32
 * product dt theta_n (one rounding); any other has its turn reduced to
 * [-pi, pi] exactly (its whole revolutions removed with the product's
 * rounding error kept).  Either way the angle carries dt's own fp32
 * rounding (a few 1e-8 of dt): a mode turning by thousands of radians per
 * token loses the fp32 accuracy of its angle.
 */
#define MAMBA3_EULER 0
#define MAMBA3_TRAPEZOIDAL 1

typedef struct mamba3_scan_args {
    int batch, seqlen, d_inner, d_state, d_conv;
    mamba_dtype io;
    const void *x, *z, *dt_raw;
    const void *Bm, *Cm;
    const float *A_log, *theta, *Dskip, *conv_w, *conv_b;
    const float *h0;
    const void *conv_state0;
    const float *v0;
    void *y;
    float *final_h;
    void *final_conv_state;
    float *final_v;
    void *workspace;
    size_t workspace_bytes;
    int n_chunks;
    int discretization;
    uint64_t wait_timeout_ns;
    unsigned flags;
} mamba3_scan_args;

/* Bytes of workspace mamba3_scan_fwd needs (0 only for invalid sizes or
 * seqlen 0). */
size_t mamba3_scan_workspace_size(int batch, int seqlen, int d_inner, int n_chunks);

mamba_status mamba3_scan_fwd(const mamba3_scan_args *args, void *stream);

/*
 * A linear map on the tensor cores, for the projections around the scan
 * (in_proj, x_proj, dt_proj, out_proj of "【大模型】- Jamba 混合
 * SSM-Transformer", section "实现 > Mamba 层", each an nn.Linear):
 *
 *   C = A W^T (+ bias)      row-major; fp32 accumulation, bf16 result
 *
 *   M, N, K           C is M x N; A is M x K; W is N x K (the nn.Linear weight
 *                     layout, rows K elements apart); M may be 0
 *   A, lda            bf16, rows lda >= K elements apart
 *   W                 bf16
 *   bias              (N) bf16 or NULL
 *   C, ldc            bf16 output, rows ldc >= N elements apart
 *   wait_timeout_ns   limit of every device-side wait (0: 1 second)
 *
 * K must be a multiple of 64 and lda, ldc multiples of 8
 * (MAMBA_ERR_UNSUPPORTED otherwise); pointers 16-byte aligned.  The
 * product runs in hand-written tcgen05 code: 128 x 256 output tiles, the
 * accumulator in tensor memory, operands brought into shared memory by TMA.
 */
typedef struct mamba_linear_args {
    long M;
    int N, K;
    const void *A;
    int lda;
    const void *W;
    const void *bias;
    void *C;
    int ldc;
    uint64_t wait_timeout_ns;
} mamba_linear_args;

mamba_status mamba_linear_fwd(const mamba_linear_args *args, void *stream);

/*
 * Decode: one token through the layer, state updated in place -- the
 * constant-memory recurrence of "Um SSM em uma pagina" (y_t needs only
 * h_{t-1} and x_t).  Bit for bit the same arithmetic as one token of
 * mamba_scan_fwd with n_chunks = 1.
 *
 *   h                 (B, D, 16) fp32     in/out, in place; 32-byte aligned
 *                                         (it is read and written in
 *                                         32-byte pieces)
 *   conv_state        (B, 3, D) io        in/out, in place (shifts by one)
 *   x_t, z_t, dt_raw_t  (B, D) io
 *   B_t, C_t          (B, 16) io          (16-byte aligned, like h)
 *   A_log, Dskip, conv_w, conv_b   as for the scan
 *   y_t               (B, D) io           output
 *
 * h moves in blocks of 64 channels of one row (4 KB) by bulk copies into
 * and out of shared memory; the one device-side wait (for a block to land)
 * gives up after 1 second and reports MAMBA_ERR_TIMEOUT through
 * mamba_last_error, leaving that block's h and y unwritten.
 */
typedef struct mamba_step_args {
    int batch, d_inner, d_state, d_conv;
    mamba_dtype io;
    float *h;
    void *conv_state;
    const void *x_t, *z_t, *dt_raw_t;
    const void *B_t, *C_t;
    const float *A_log, *Dskip, *conv_w, *conv_b;
    void *y_t;
} mamba_step_args;

mamba_status mamba_step(const mamba_step_args *args, void *stream);

/* Synchronises `stream`, then reads and clears the sticky device error word
 * of the current device: MAMBA_OK, or MAMBA_ERR_TIMEOUT if a device-side
 * wait gave up since the last call. */
mamba_status mamba_last_error(void *stream);

/* A static, human-readable name of a status code. */
const char *mamba_status_string(mamba_status s);

/* Library ABI version (major * 100 + minor). */
int mamba_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MAMBA_SSM_H */
