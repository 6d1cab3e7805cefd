/*
 * CPU oracle of the Mamba-3 SSM state scan.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package's smoke check and
 * the benchmark's CPU-baseline leg load this code.  It shares nothing with
 * the GPU library: no header, helper, table or constant.
 *
 * What it computes: the plain token-by-token recurrence, in complex double,
 * one (sequence, head) unit at a time.  The method is described in words on
 * "Together AI announces Mamba-3" (architecture section 1, exponential-
 * trapezoid discretisation, a second-order rule that accounts for both the
 * input and the state change; section 2, a complex-valued state with N/2
 * complex entries applied as a block-diagonal 2x2 rotation, the "RoPE
 * trick"; section 3, SISO and rank-R MIMO).  The pages print no equation;
 * the recurrence written out here is the statement of the problem this
 * library implements:
 *
 *   a_t[k] = exp(dt_t * (A + i*theta_t[k]))          per complex pair k
 *   b_t[k] = (1 - lam_t) * dt_t * a_t[k]
 *   g_t    = lam_t * dt_t
 *   u_t[k][p] = sum_r Bhat_t[r][k] * x_t[r][p],   Bhat[r][k] = B[r][2k] + i*B[r][2k+1]
 *   h_t[k][p] = a_t[k]*h_{t-1}[k][p] + b_t[k]*u_{t-1}[k][p] + g_t*u_t[k][p]
 *   y_t[r][p] = sum_k Re(conj(Chat_t[r][k]) * h_t[k][p]) + D * x_t[r][p]
 *
 * Readings where the statement is silent (each one listed in the design
 * notes): complex pairs are the interleaved components (2k, 2k+1); C^H is
 * the conjugate transpose; A and D are one scalar per head; u_{-1} is built
 * from the carried previous-token (B, x), zero unless the caller passes
 * one; the final state is h_{L-1} itself; the carry returned is the last
 * token's (B, x); MIMO's skip term is D times each rank's x.
 *
 * Inputs are read as the values stored (f32, bf16 bit patterns, or f64)
 * widened exactly to double.
 */
#include <complex.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define M3O_F32 0
#define M3O_BF16 1
#define M3O_F64 2

/* One unit: where its tokens live in each input tensor and in y. */
typedef struct {
  int64_t ntok;   /* tokens to walk                                          */
  int64_t x0, xs; /* element offset of token 0's x[r=0][p=0]; token stride   */
  int64_t b0, bs; /* the same for B and C (they share a layout)              */
  int64_t s0, ss; /* the same for dt and lam                                 */
  int64_t q0, qs; /* the same for theta                                      */
  int64_t y0, ys; /* the same for y (double output)                          */
  int64_t head;   /* selects A and D                                         */
} m3o_unit;

static double rd(const void* base, int64_t i, int dtype) {
  if (dtype == M3O_F64) return ((const double*)base)[i];
  if (dtype == M3O_F32) return (double)((const float*)base)[i];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 16;
  float f;
  memcpy(&f, &bits, 4);
  return (double)f;
}

/* u[k][p] = sum_r Bhat[r][k] * x[r][p] for one token. */
static void outer(int R, int P, int N, const void* B, int64_t b_off, const void* x, int64_t x_off,
                  int dtype, double complex* u) {
  int K = N / 2;
  for (int k = 0; k < K; ++k)
    for (int p = 0; p < P; ++p) {
      double complex acc = 0.0;
      for (int r = 0; r < R; ++r) {
        double complex bh = rd(B, b_off + (int64_t)r * N + 2 * k, dtype) +
                            I * rd(B, b_off + (int64_t)r * N + 2 * k + 1, dtype);
        acc += bh * rd(x, x_off + (int64_t)r * P + p, dtype);
      }
      u[(int64_t)k * P + p] = acc;
    }
}

static void scan_unit(const m3o_unit* un, int R, int P, int N, int dtype, const void* x,
                      const void* B, const void* C, const void* dt, const void* lam,
                      const void* theta, const double* A, const double* D, double* h,
                      double* prevB, double* prevx, double* y) {
  const int K = N / 2;
  const double Ah = A[un->head], Dh = D[un->head];
  double complex* hs = malloc(sizeof(double complex) * K * P);
  double complex* u = malloc(sizeof(double complex) * K * P);
  double complex* uprev = malloc(sizeof(double complex) * K * P);
  double complex* alpha = malloc(sizeof(double complex) * K);

  for (int64_t i = 0; i < (int64_t)K * P; ++i) hs[i] = h[2 * i] + I * h[2 * i + 1];
  /* u_{-1} from the carried previous token (zero arrays when there is none) */
  outer(R, P, N, prevB, 0, prevx, 0, M3O_F64, uprev);

  for (int64_t t = 0; t < un->ntok; ++t) {
    const int64_t xo = un->x0 + t * un->xs, bo = un->b0 + t * un->bs;
    const int64_t so = un->s0 + t * un->ss, qo = un->q0 + t * un->qs;
    const double dtt = rd(dt, so, dtype), lmt = rd(lam, so, dtype);
    for (int k = 0; k < K; ++k) alpha[k] = cexp(dtt * (Ah + I * rd(theta, qo + k, dtype)));
    const double g = lmt * dtt;
    const double bscale = (1.0 - lmt) * dtt;

    outer(R, P, N, B, bo, x, xo, dtype, u);
    for (int k = 0; k < K; ++k)
      for (int p = 0; p < P; ++p) {
        int64_t i = (int64_t)k * P + p;
        hs[i] = alpha[k] * hs[i] + bscale * alpha[k] * uprev[i] + g * u[i];
      }
    for (int r = 0; r < R; ++r)
      for (int p = 0; p < P; ++p) {
        double acc = 0.0;
        for (int k = 0; k < K; ++k) {
          double complex ch = rd(C, bo + (int64_t)r * N + 2 * k, dtype) +
                              I * rd(C, bo + (int64_t)r * N + 2 * k + 1, dtype);
          acc += creal(conj(ch) * hs[(int64_t)k * P + p]);
        }
        y[un->y0 + t * un->ys + (int64_t)r * P + p] = acc + Dh * rd(x, xo + (int64_t)r * P + p, dtype);
      }
    double complex* sw = uprev;
    uprev = u;
    u = sw;
  }

  for (int64_t i = 0; i < (int64_t)K * P; ++i) {
    h[2 * i] = creal(hs[i]);
    h[2 * i + 1] = cimag(hs[i]);
  }
  if (un->ntok > 0) { /* the carry becomes the last token's (B, x) */
    const int64_t t = un->ntok - 1;
    for (int64_t i = 0; i < (int64_t)R * N; ++i) prevB[i] = rd(B, un->b0 + t * un->bs + i, dtype);
    for (int64_t i = 0; i < (int64_t)R * P; ++i) prevx[i] = rd(x, un->x0 + t * un->xs + i, dtype);
  }
  free(hs);
  free(u);
  free(uprev);
  free(alpha);
}

/*
 * Walk nunits independent units.  h [nunits][N/2][P][2], prevB [nunits][R][N]
 * and prevx [nunits][R][P] hold each unit's initial state and carry on
 * entry and its final state and carry on return.  y receives every token's
 * output at the offsets the unit table gives.  Units run on nthreads
 * threads; each unit's token loop is sequential.
 */
int m3_oracle_run(const m3o_unit* units, int64_t nunits, int R, int P, int N, int dtype,
                  const void* x, const void* B, const void* C, const void* dt, const void* lam,
                  const void* theta, const double* A, const double* D, double* h, double* prevB,
                  double* prevx, double* y, int nthreads) {
  if (N <= 0 || (N & 1) || R <= 0 || P <= 0 || nunits < 0) return -1;
  if (dtype != M3O_F32 && dtype != M3O_BF16 && dtype != M3O_F64) return -1;
  if (nthreads < 1) nthreads = 1;
  const int64_t hsz = (int64_t)N * P; /* N/2 pairs x P x (re, im) */
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
  for (int64_t i = 0; i < nunits; ++i)
    scan_unit(&units[i], R, P, N, dtype, x, B, C, dt, lam, theta, A, D, h + i * hsz,
              prevB + i * (int64_t)R * N, prevx + i * (int64_t)R * P, y);
  return 0;
}
