/*
 * m3scan_backward.h -- backward pass of the Mamba-3 scan (libm3scan.so).
 *
 * Part of the same library and C ABI as m3scan.h (status codes, m3_dims,
 * conventions: device pointers, caller-owned buffers, work enqueued on
 * `stream`, no traps).
 */
#ifndef M3SCAN_BACKWARD_H
#define M3SCAN_BACKWARD_H

#include "m3scan.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Backward pass for training: gradients of a loss L with respect to every
 * input of a prefill, given dL/dy (and optionally dL/dh_final).  The pages
 * train their models but describe no backward kernel; this is the exact
 * adjoint of the recurrence above, in f32.  Two kernels compute it:
 *   - chunked (algo M3_ALGO_CHUNKED, and AUTO where the shape has it: P = 64,
 *     N = 64 or 128, R = 1, 2 or 4, chunk 0 or 64 / R): every chunk of every
 *     (sequence, head) unit in parallel.  A first pass sums each chunk's
 *     contribution to the state and to the state's adjoint, a second chains
 *     them across chunks (one thread per state element), a third computes
 *     every gradient of each chunk's tokens from the state at the chunk's
 *     start and the adjoint at its end.  Scratch: about 4 * units * (L/Q + 1)
 *     * N * P * 4 bytes (more than 16 GiB: M3_ERR_UNSUPPORTED).
 *     Deterministic (no float atomics).
 *   - token-serial (algo M3_ALGO_RECURRENT, and AUTO otherwise): walks the
 *     tokens of each unit in order, any shape with R <= 8; a reference
 *     kernel for modest sizes.  Scratch: units * L * (N/2) * P * 8 bytes
 *     (more than 4 GiB: M3_ERR_UNSUPPORTED).
 * Fixed-length batches only (no cu_seqlens).  The inputs are the forward's,
 * in its layouts and in_dtype; every gradient is f32 in its input's layout
 * (dB and dC in the grouped layout, summed over the heads of a group; dA
 * and dD summed over the batch and the tokens).  With `prologue` flags (as
 * in m3_prefill_args: softplus(dt + dt_bias) and the RMS norm of the rows
 * of B, C and the carried B) the inputs are the raw values the prologue
 * reads and the gradients are with respect to them; ddt_bias, if given,
 * receives the gradient of dt_bias.  Scratch is stream-ordered device memory,
 * freed on the stream.  The library writes every output itself.
 * Errors: M3_ERR_INVALID_ARG (null required pointer, seqlen < 1, bad dims,
 * ngroups, algo or prologue bits), M3_ERR_UNSUPPORTED (CHUNKED on a shape
 * without it, scratch over the limit), M3_ERR_ALLOC, M3_ERR_CUDA.
 */
typedef struct m3_backward_args {
  m3_dims dims;
  int64_t seqlen;
  const void* x;         /* the forward's inputs, as in m3_prefill_args      */
  const void* B;
  const void* C;
  const void* dt;
  const void* lam;       /* NULL: lam = 1   */
  const void* theta;     /* NULL: theta = 0 */
  const float* A;
  const float* D;
  const float* h0;       /* [batch][H][N/2][P][2] f32 initial state, or NULL (zero) */
  const void* prev_B;    /* [batch][H][R][N] in_dtype carry, or NULL (none)        */
  const void* prev_x;    /* [batch][H][R][P] in_dtype carry, or NULL               */
  const float* dy;       /* [batch][L][H][R][P] f32: dL/dy                          */
  const float* dh_final; /* [batch][H][N/2][P][2] f32: dL/dh_final, or NULL (zero) */
  float* dx;             /* outputs, f32, in the inputs' layouts                    */
  float* dB;
  float* dC;
  float* ddt;
  float* dlam;           /* or NULL */
  float* dtheta;         /* or NULL */
  float* dA;             /* [H] */
  float* dD;             /* [H] */
  float* dh0;            /* or NULL */
  float* dprev_B;        /* or NULL */
  float* dprev_x;        /* or NULL */
  int32_t ngroups;       /* as in m3_prefill_args */
  int32_t algo;          /* m3_algo: AUTO (0), RECURRENT (token-serial) or CHUNKED */
  int32_t chunk;         /* tokens per chunk of the chunked kernel: 0 or 64 / R */
  int32_t prologue;      /* m3_prologue flags, as in m3_prefill_args; 0 = none */
  const float* dt_bias;  /* [H] f32 (M3_PRO_DT_SOFTPLUS) or NULL                     */
  float* ddt_bias;       /* [H] f32 output: dL/d dt_bias (M3_PRO_DT_SOFTPLUS), or NULL */
} m3_backward_args;

M3_API m3_status m3_scan_prefill_backward(const m3_backward_args* args, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* M3SCAN_BACKWARD_H */
