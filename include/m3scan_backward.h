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
 * adjoint of the recurrence above, walked token by token per (sequence,
 * head) unit in f32 (a reference kernel for modest sizes, not a fast one).
 * Fixed-length batches only (no cu_seqlens).  The inputs are the forward's,
 * in its layouts and in_dtype; every gradient is f32 in its input's layout
 * (dB and dC in the grouped layout, summed over the heads of a group; dA
 * and dD summed over the batch and the tokens).  The library zeroes the
 * accumulated outputs itself.  Scratch: units * L * (N/2) * P * 8 bytes of
 * stream-ordered device memory for the forward history, freed on the
 * stream; more than 4 GiB returns M3_ERR_UNSUPPORTED.
 * Errors: M3_ERR_INVALID_ARG (null required pointer, seqlen < 1, bad dims
 * or ngroups), M3_ERR_UNSUPPORTED, M3_ERR_ALLOC, M3_ERR_CUDA.
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
} m3_backward_args;

M3_API m3_status m3_scan_prefill_backward(const m3_backward_args* args, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* M3SCAN_BACKWARD_H */
