/*
 * m3scan.h -- C ABI of the Mamba-3 SSM state scan library (libm3scan.so).
 *
 * The scan is the hot path of a Mamba-3 mixer layer ("Together AI announces
 * Mamba-3", architecture sections 1-3): an exponential-trapezoid
 * (second-order) discretisation, a complex-valued state applied as a
 * block-diagonal 2x2 rotation (the "RoPE trick"), and SISO or rank-R MIMO
 * input/output.  Per (sequence, head) unit, with N/2 complex state pairs k
 * and head dimension P:
 *
 *   a_t[k]    = exp(dt_t * (A + i*theta_t[k]))
 *   u_t[k][p] = sum_r (B_t[r][2k] + i*B_t[r][2k+1]) * x_t[r][p]
 *   h_t[k][p] = a_t[k]*h_{t-1}[k][p] + (1-lam_t)*dt_t*a_t[k]*u_{t-1}[k][p]
 *               + lam_t*dt_t*u_t[k][p]
 *   y_t[r][p] = sum_k Re(conj(C_t[r][2k] + i*C_t[r][2k+1]) * h_t[k][p]) + D*x_t[r][p]
 *
 * u_{-1} comes from the state's carry (the previous token's B and x), zero
 * for a fresh state.  After a call the state holds h of the last token and
 * the carry holds that token's (B, x), so calls chain exactly: a prefill of
 * L tokens equals a prefill of L1 tokens followed by L - L1 tokens or by
 * single-token decode steps.
 *
 * Conventions for every entry point:
 *   - Tensors are device pointers, dense, row-major, last index innermost.
 *     The caller owns every input and output buffer; the library owns only
 *     the m3_state objects it allocates.
 *   - Work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns before it completes.  Nothing synchronises.
 *   - Every call returns an m3_status.  No exception crosses the ABI and no
 *     kernel traps.  A kernel that gives up a bounded wait records
 *     M3_ERR_TIMEOUT in a device status word that m3_device_status() reads.
 *   - x, B, C, theta, y and the state must be 16-byte aligned.
 *   - Mamba-2 mode ("Together AI announces Mamba-3", section 1 table: the
 *     first-order exponential-Euler rule of Mamba-2; section 2 table: a
 *     real-valued state): `theta` may be NULL, meaning theta = 0 (every
 *     pair is two independent real states, so N real states in all), and
 *     `lam` may be NULL, meaning lam = 1 (h_t = a_t h_{t-1} + dt_t u_t: no
 *     previous-token term).  With both NULL the scan is the first-order real
 *     SSM of Mamba-2 with N states, on the same layouts.
 *   - Floating point: inputs are f32 or bf16 (in_dtype); dt, lam and theta
 *     share that type; A, D, dt_bias and the state are f32; y is f32 or, on
 *     request, bf16 (y_dtype); all arithmetic is f32 (tensor-core products
 *     take f16 hi/lo operand pairs with f32 accumulation).
 */
#ifndef M3SCAN_H
#define M3SCAN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Symbols of the shared library (built with hidden default visibility). */
#if defined(__GNUC__)
#define M3_API __attribute__((visibility("default")))
#else
#define M3_API
#endif

typedef enum m3_status {
  M3_OK = 0,
  M3_ERR_INVALID_ARG = 1, /* null or misaligned pointer, bad size, dims that do not match  */
  M3_ERR_UNSUPPORTED = 2, /* a valid request this build has no kernel for (shape, dtype)    */
  M3_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed                   */
  M3_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up (read by m3_device_status) */
  M3_ERR_ALLOC = 5,       /* device memory allocation failed                               */
  M3_ERR_SCRATCH = 6      /* m3_scan_prefill_noalloc: the request needs more than its fixed scratch */
} m3_status;

typedef enum m3_dtype { M3_F32 = 0, M3_BF16 = 1 } m3_dtype;

/* Which prefill kernel runs. */
typedef enum m3_algo {
  M3_ALGO_AUTO = 0,      /* chunked tensor-core path when the shape has one, else recurrent */
  M3_ALGO_RECURRENT = 1, /* token-by-token f32 recurrence on CUDA cores (any shape)          */
  M3_ALGO_CHUNKED = 2    /* chunked tcgen05/TMEM path (bf16 inputs, supported shapes only)   */
} m3_algo;

/*
 * Fused prologue: the step of a Mamba-3 mixer just before the scan, done by
 * the scan kernels while they load their inputs.  The B/C normalisation is
 * the pages' BC/QK norm ("Mamba-3: an inference-first LLM", section
 * "Implementation and kernel optimisation"; "Together AI announces Mamba-3",
 * Mamba-2 vs Mamba-3 table, normalisation row: QKNorm replaces RMSNorm).
 * The pages do not say how dt is produced; softplus of a biased projection
 * keeps it positive and is the plainest choice.  Flags of the `prologue`
 * argument field; 0 = the inputs are used as given.
 *   M3_PRO_DT_SOFTPLUS: dt holds the pre-activation; the scan uses
 *       softplus(dt + dt_bias[h]) = log(1 + exp(dt + dt_bias[h])).
 *   M3_PRO_BC_NORM: every row of B and of C (one token, group and rank: N
 *       values) is divided by its root mean square, v / sqrt(mean(v^2) +
 *       1e-6), before use; so is the carried previous-token B.  There is no
 *       gain vector (a per-column gain folds into the B and C projection).
 * The carry in m3_state keeps the raw B and x of the last token.
 */
typedef enum m3_prologue {
  M3_PRO_DT_SOFTPLUS = 1,
  M3_PRO_BC_NORM = 2
} m3_prologue;

/* Problem sizes. */
typedef struct m3_dims {
  int32_t batch;    /* sequences (state slots)                                   */
  int32_t nheads;   /* H                                                          */
  int32_t headdim;  /* P (even)                                                   */
  int32_t dstate;   /* N (even): N/2 complex pairs                                */
  int32_t rank;     /* R: 1 = SISO, R > 1 = MIMO                                  */
  int32_t in_dtype; /* m3_dtype of x, B, C, dt, lam, theta and of the carry       */
} m3_dims;

/* Opaque recurrent state: h, the previous-token carry, and its dims. */
typedef struct m3_state m3_state;

/* Raw device pointers of a state (for initialisation, inspection, tests). */
typedef struct m3_state_ptrs {
  m3_dims dims;
  float* h;     /* [batch][H][N/2][P][2] f32, (re, im) innermost     */
  void* prev_B; /* [batch][H][R][N] in_dtype: the last token's B      */
  void* prev_x; /* [batch][H][R][P] in_dtype: the last token's x      */
} m3_state_ptrs;

/* Prefill over a whole sequence batch (or a packed variable-length batch). */
typedef struct m3_prefill_args {
  m3_dims dims;   /* dims.batch rows; 1 when cu_seqlens is given                      */
  int64_t seqlen; /* L: tokens per row (total packed tokens with cu_seqlens)           */
  int32_t chunk;  /* tokens per chunk for M3_ALGO_CHUNKED; 0 = the kernel's default    */
  int32_t algo;   /* m3_algo                                                            */
  const void* x;     /* [batch][L][H][R][P]   in_dtype */
  const void* B;     /* [batch][L][G][R][N]   in_dtype; G = ngroups (H by default) */
  const void* C;     /* [batch][L][G][R][N]   in_dtype */
  const void* dt;    /* [batch][L][H]         in_dtype, > 0 (the pre-activation under
                                                 M3_PRO_DT_SOFTPLUS: any value) */
  const void* lam;   /* [batch][L][H]         in_dtype, in [0, 1]; NULL: lam = 1 */
  const void* theta; /* [batch][L][H][N/2]    in_dtype; NULL: theta = 0        */
  const float* A;    /* [H] f32, < 0 */
  const float* D;    /* [H] f32 */
  const int32_t* cu_seqlens; /* device [nseq+1], nondecreasing, cu[0] = 0, cu[nseq] = L; or NULL */
  int32_t nseq;              /* sequences in the packed batch (ignored without cu_seqlens) */
  void* y;                   /* [batch][L][H][R][P] output, f32 or bf16 (y_dtype) */
  int32_t ngroups; /* G: B and C shared by groups of H/G consecutive heads, laid out
                      [batch][L][G][R][N] (head h uses group h / (H / G)); must divide H;
                      0 (or H) = one B and C per head, [batch][L][H][R][N].  The pages
                      give B and C per head; groups are an addressing variant only (the
                      recurrence of each head is unchanged) */
  int32_t y_dtype; /* m3_dtype of y: M3_F32 (0, the default) or M3_BF16, the f32 result
                      rounded to nearest even (half the output bytes).  Not on the pages,
                      which fix no output type */
  int32_t prologue;      /* m3_prologue flags; 0 = none */
  const float* dt_bias;  /* [H] f32 added to dt before softplus (M3_PRO_DT_SOFTPLUS); NULL = 0 */
} m3_prefill_args;

/* One decode step: a single new token per sequence. */
typedef struct m3_decode_args {
  m3_dims dims;
  const void* x;     /* [batch][H][R][P] in_dtype */
  const void* B;     /* [batch][G][R][N] in_dtype; G = ngroups (H by default) */
  const void* C;     /* [batch][G][R][N] in_dtype */
  const void* dt;    /* [batch][H]       in_dtype */
  const void* lam;   /* [batch][H]       in_dtype; NULL: lam = 1   */
  const void* theta; /* [batch][H][N/2]  in_dtype; NULL: theta = 0 */
  const float* A;    /* [H] f32 */
  const float* D;    /* [H] f32 */
  void* y;           /* [batch][H][R][P] output, f32 or bf16 (y_dtype) */
  int32_t ngroups;   /* as in m3_prefill_args: B and C [batch][G][R][N]; 0 = per head */
  int32_t y_dtype;   /* as in m3_prefill_args: M3_F32 (0) or M3_BF16 */
  int32_t prologue;      /* as in m3_prefill_args */
  const float* dt_bias;  /* [H] f32 or NULL */
} m3_decode_args;

/*
 * Allocate a state for `dims` and zero it on `stream` (h = 0, no carry).
 * *out receives the handle.  The buffers are stream-ordered allocations on
 * `stream` (from the device's default memory pool): work on other streams
 * that uses the state must be ordered after the allocation (an event), and
 * `stream` must outlive the state.  Errors: M3_ERR_INVALID_ARG (bad dims or
 * null out), M3_ERR_ALLOC, M3_ERR_CUDA.
 */
M3_API m3_status m3_state_alloc(const m3_dims* dims, m3_state** out, void* stream);

/*
 * Free a state.  The buffers are returned in stream order on the stream
 * given to m3_state_alloc; nothing waits for the device.  Work on other
 * streams that still uses the state must be ordered before the free on
 * that stream by the caller.  NULL is accepted.
 */
M3_API m3_status m3_state_free(m3_state* st);

/* Fill *out with the state's dims and device pointers. */
M3_API m3_status m3_state_view(const m3_state* st, m3_state_ptrs* out);

/*
 * Prefill: run the scan over every token of args->x etc. and write y.
 * With st == NULL every sequence starts from h = 0 without a carry and no
 * state is kept.  With a state, each sequence starts from its slot's h and
 * carry and the slot receives the final h and the last token's (B, x);
 * st's dims must equal args->dims, except that with cu_seqlens st's batch
 * is nseq.  With cu_seqlens (batch must be 1), each packed sequence
 * [cu[s], cu[s+1]) is its own unit: h and the carry restart at every
 * boundary (from the state slot s when st is given).
 * Errors: M3_ERR_INVALID_ARG (also: ngroups < 0 or not dividing H, an
 * unknown y_dtype, unknown prologue bits), M3_ERR_UNSUPPORTED (algo CHUNKED
 * on a shape or dtype without a chunked kernel, or with theta NULL and
 * M3_PRO_BC_NORM), M3_ERR_CUDA.
 */
M3_API m3_status m3_scan_prefill(const m3_prefill_args* args, m3_state* st, void* stream);

/*
 * The same prefill without any device-memory allocation in the call.  The
 * pages describe no such entry point: it exists for callers that must not
 * allocate while they run -- for example a serving engine that reserves all
 * device memory up front, or code whose device memory is planned in
 * advance.  m3_scan_prefill takes a few MB of stream-ordered pool memory for
 * the handover slots of its balanced schedule (used when a call has more
 * (sequence, head) units than the GPU has SMs); this entry point uses a
 * fixed buffer of M3_NOALLOC_SCRATCH_BYTES that is part of the library's
 * module memory instead, and calls no allocating routine.
 *   - The buffer is module memory: CUDA creates it on a device when it
 *     loads the library's device code there.  Under CUDA's default lazy
 *     module loading that is the first use of the library on the device,
 *     not the moment the library is loaded into the process.  The first
 *     call of this entry point on each device (whatever its arguments)
 *     looks the buffer's address up with that device current, which loads
 *     the module and creates the buffer, and can fail with M3_ERR_CUDA.  A
 *     caller that reserves all free device memory up front makes that
 *     first call before reserving, and before any stream capture.
 *   - A request that needs more scratch than the buffer holds returns
 *     M3_ERR_SCRATCH and enqueues nothing (strict on purpose: the buffer's
 *     size is this entry point's stated maximum; m3_scan_prefill serves
 *     such requests).  The need is about 33 KB per SM at N = 128, P = 64
 *     (the buffer covers up to 240 SMs there).
 *   - The buffer is shared by every call on a device: calls that overlap in
 *     time (different streams without ordering between them, or different
 *     host threads) race on it.  Order such calls.
 * Arguments, results and the other errors are those of m3_scan_prefill.
 */
#define M3_NOALLOC_SCRATCH_BYTES (8u << 20)
M3_API m3_status m3_scan_prefill_noalloc(const m3_prefill_args* args, m3_state* st, void* stream);

/*
 * Decode step: advance every sequence of st by one token, write y, and
 * replace the carry with this token's (B, x).  args->dims must equal st's.
 * Errors: M3_ERR_INVALID_ARG (as for the prefill), M3_ERR_UNSUPPORTED,
 * M3_ERR_CUDA.
 */
M3_API m3_status m3_decode_step(const m3_decode_args* args, m3_state* st, void* stream);

/*
 * Synchronise `stream`, read and clear the library's device status word.
 * Returns M3_OK, or M3_ERR_TIMEOUT if a kernel gave up a bounded wait since
 * the last check, or M3_ERR_CUDA if the synchronisation itself failed.
 */
M3_API m3_status m3_device_status(void* stream);

/* Static, human-readable name of a status code. */
M3_API const char* m3_status_string(m3_status s);

#ifdef __cplusplus
}
#endif

#endif /* M3SCAN_H */
