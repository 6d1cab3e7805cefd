// Token-by-token prefill on CUDA cores, all in f32.
//
// This is the plain recurrence of the statement (exponential-trapezoid
// update of a complex state, "Together AI announces Mamba-3", sections 1-3)
// walked sequentially per (sequence, head) unit.  It serves f32 inputs,
// where tensor-core operands would lose the precision the caller asked
// for, and any shape the chunked tensor-core kernel does not cover.
//
// Layout: one CTA per unit, P x KS threads.  Thread (p, ks) keeps
// h[k][p] for its slice of KPT pairs in registers for the whole sequence,
// so the time loop needs no state traffic at all; the KS threads of one p
// are adjacent lanes and reduce the output over pairs with shuffles.
// Tokens are staged TB at a time in shared memory (B, C, x as f32 and the
// per-pair factor a = exp(dt(A + i*theta)) computed once per token and pair),
// with the previous block's last token kept as row 0 for the trapezoid term.
#pragma once

#include "common.cuh"

namespace m3 {

struct RecurrentParams {
  const void* x;
  const void* B;
  const void* C;
  const void* dt;
  const void* lam;
  const void* theta;
  const float* A;
  const float* D;
  const int32_t* cu_seqlens;  // NULL: fixed length L per batch row
  void* y;        // f32, or bf16 when ybf
  int ybf;
  float* h;       // state slots or NULL
  void* prev_B;   // carry slots or NULL
  void* prev_x;
  int64_t L;      // tokens per row (total with cu_seqlens)
  int H, P, N, K, R;
  int G;          // B and C groups (head h uses group h / (H / G))
  int KS;         // threads per p (power of two <= 32)
  int TB;         // tokens staged per block
  int pro;        // m3_prologue flags
  const float* dt_bias;
};

// BC norm in shared memory: rows [0, nrows) of n values each, scaled in place
// by 1 / sqrt(mean(v^2) + eps), a warp per row.  Callers synchronise around it.
__device__ __forceinline__ void normalize_rows_smem(float* base, int nrows, int n) {
  const int lane = threadIdx.x % 32;
  for (int row = threadIdx.x / 32; row < nrows; row += blockDim.x / 32) {
    float* v = base + (size_t)row * n;
    const float sc = warp_rms_scale(v, n, lane);
    for (int i = lane; i < n; i += 32) v[i] *= sc;
  }
}

// R is the rank when known at compile time; R == 0 reads it from p.R (<= 8).
template <typename T, int KPT, int R_>
__global__ void recurrent_prefill_kernel(const RecurrentParams p) {
  extern __shared__ float smem[];
  constexpr int RMAX = R_ > 0 ? R_ : 8;
  const int R = R_ > 0 ? R_ : p.R;
  const int H = p.H, P = p.P, N = p.N, K = p.K, KS = p.KS, TB = p.TB;
  const int RN = R * N, RP = R * P;
  float* Bs = smem;                                    // [TB+1][R][N], row 0 = previous token
  float* Cs = Bs + (TB + 1) * RN;                      // [TB][R][N]
  float* xs = Cs + TB * RN;                            // [TB+1][R][P], row 0 = previous token
  float2* al = reinterpret_cast<float2*>(xs + (TB + 1) * RP);  // [TB][K]
  float* sc = reinterpret_cast<float*>(al + TB * K);   // [TB][2]: gamma, beta'

  const int unit = blockIdx.x;
  const int seq = unit / H, head = unit % H;
  int64_t tok0, ntok;
  if (p.cu_seqlens) {
    tok0 = p.cu_seqlens[seq];
    ntok = p.cu_seqlens[seq + 1] - tok0;
  } else {
    tok0 = (int64_t)seq * p.L;
    ntok = p.L;
  }
  const int tid = threadIdx.x;
  const int pi = tid / KS, ks = tid % KS;
  const bool active = pi < P;
  const float A = p.A[head], D = p.D[head];

  // initial state and carry
  float hr[KPT], hi[KPT];
#pragma unroll
  for (int j = 0; j < KPT; ++j) {
    const int k = ks * KPT + j;
    hr[j] = 0.f;
    hi[j] = 0.f;
    if (p.h && active && k < K) {
      const float2 v = reinterpret_cast<const float2*>(p.h)[((int64_t)unit * K + k) * P + pi];
      hr[j] = v.x;
      hi[j] = v.y;
    }
  }
  for (int i = tid; i < RN; i += blockDim.x)
    Bs[i] = p.prev_B ? ldf(static_cast<const T*>(p.prev_B), (int64_t)unit * RN + i) : 0.f;
  for (int i = tid; i < RP; i += blockDim.x)
    xs[i] = p.prev_x ? ldf(static_cast<const T*>(p.prev_x), (int64_t)unit * RP + i) : 0.f;
  const bool norm = (p.pro & M3_PRO_BC_NORM) != 0;
  if (norm) {  // the carried B, as every staged B row below
    __syncthreads();
    normalize_rows_smem(Bs, R, N);
  }

  const T* xg = static_cast<const T*>(p.x);
  const T* Bg = static_cast<const T*>(p.B);
  const T* Cg = static_cast<const T*>(p.C);
  const T* dtg = static_cast<const T*>(p.dt);
  const T* lmg = static_cast<const T*>(p.lam);
  const T* thg = static_cast<const T*>(p.theta);

  for (int64_t t0 = 0; t0 < ntok; t0 += TB) {
    const int nb = (ntok - t0 < TB) ? (int)(ntok - t0) : TB;
    __syncthreads();  // previous block fully consumed (row 0 already moved)
    for (int i = tid; i < nb * RN; i += blockDim.x) {
      const int tb = i / RN, e = i % RN;
      const int64_t g = ((tok0 + t0 + tb) * p.G + head / (H / p.G)) * RN + e;
      Bs[(tb + 1) * RN + e] = ldf(Bg, g);
      Cs[tb * RN + e] = ldf(Cg, g);
    }
    for (int i = tid; i < nb * RP; i += blockDim.x) {
      const int tb = i / RP, e = i % RP;
      xs[(tb + 1) * RP + e] = ldf(xg, ((tok0 + t0 + tb) * H + head) * RP + e);
    }
    for (int i = tid; i < nb * K; i += blockDim.x) {
      const int tb = i / K, k = i % K;
      const int64_t ts = (tok0 + t0 + tb) * H + head;
      const float dt = scan_dt(ldf(dtg, ts), p.pro, p.dt_bias, head);
      float s = 0.f, c = 1.f;  // theta = 0 when theta is not given
      if (thg) sincosf(dt * ldf(thg, ts * K + k), &s, &c);
      const float dec = expf(dt * A);
      al[tb * K + k] = make_float2(dec * c, dec * s);
      if (k == 0) {
        const float lm = lmg ? ldf(lmg, ts) : 1.f;  // lam = 1 when lam is not given
        sc[2 * tb] = lm * dt;
        sc[2 * tb + 1] = (1.f - lm) * dt;
      }
    }
    __syncthreads();
    if (norm) {  // rows 1..nb of Bs (row 0 is the previous token, already normalised) and rows 0..nb-1 of Cs
      normalize_rows_smem(Bs + RN, nb * R, N);
      normalize_rows_smem(Cs, nb * R, N);
      __syncthreads();
    }

    for (int tb = 0; tb < nb; ++tb) {
      const float gam = sc[2 * tb], bet = sc[2 * tb + 1];
      const float* Bc = Bs + (tb + 1) * RN;
      const float* Bp = Bs + tb * RN;
      const float* xc = xs + (tb + 1) * RP;
      const float* xp = xs + tb * RP;
      const float* Cc = Cs + tb * RN;
      float xcv[RMAX], xpv[RMAX], yacc[RMAX];
#pragma unroll
      for (int r = 0; r < RMAX; ++r) {
        xcv[r] = (active && r < R) ? xc[r * P + pi] : 0.f;
        xpv[r] = (active && r < R) ? xp[r * P + pi] : 0.f;
        yacc[r] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < KPT; ++j) {
        const int k = ks * KPT + j;
        if (k < K) {
          float ur = 0.f, ui = 0.f, vr = 0.f, vi = 0.f;
#pragma unroll
          for (int r = 0; r < RMAX; ++r) {
            if (r >= R) break;
            ur = fmaf(Bp[r * N + 2 * k], xpv[r], ur);
            ui = fmaf(Bp[r * N + 2 * k + 1], xpv[r], ui);
            vr = fmaf(Bc[r * N + 2 * k], xcv[r], vr);
            vi = fmaf(Bc[r * N + 2 * k + 1], xcv[r], vi);
          }
          const float2 a = al[tb * K + k];
          const float gr = fmaf(bet, ur, hr[j]), gi = fmaf(bet, ui, hi[j]);
          hr[j] = fmaf(a.x, gr, fmaf(-a.y, gi, gam * vr));
          hi[j] = fmaf(a.x, gi, fmaf(a.y, gr, gam * vi));
#pragma unroll
          for (int r = 0; r < RMAX; ++r)
            if (r < R) yacc[r] = fmaf(Cc[r * N + 2 * k], hr[j], fmaf(Cc[r * N + 2 * k + 1], hi[j], yacc[r]));
        }
      }
#pragma unroll
      for (int r = 0; r < RMAX; ++r)
        for (int o = KS / 2; o > 0; o >>= 1) yacc[r] += __shfl_xor_sync(0xffffffffu, yacc[r], o, KS);
      if (active && ks == 0) {
        const int64_t yo = ((tok0 + t0 + tb) * H + head) * RP;
#pragma unroll
        for (int r = 0; r < RMAX; ++r)
          if (r < R) st_y(p.y, yo + r * P + pi, fmaf(D, xcv[r], yacc[r]), p.ybf);
      }
    }
    __syncthreads();
    // the block's last token becomes the previous token of the next block
    for (int i = tid; i < RN; i += blockDim.x) Bs[i] = Bs[nb * RN + i];
    for (int i = tid; i < RP; i += blockDim.x) xs[i] = xs[nb * RP + i];
  }

  // final state and carry
  if (p.h) {
#pragma unroll
    for (int j = 0; j < KPT; ++j) {
      const int k = ks * KPT + j;
      if (active && k < K)
        reinterpret_cast<float2*>(p.h)[((int64_t)unit * K + k) * P + pi] = make_float2(hr[j], hi[j]);
    }
  }
  if (ntok > 0 && p.prev_B) {
    const int64_t last = (tok0 + ntok - 1) * H + head;
    const int64_t lastg = (tok0 + ntok - 1) * p.G + head / (H / p.G);
    T* pB = static_cast<T*>(p.prev_B) + (int64_t)unit * RN;
    T* px = static_cast<T*>(p.prev_x) + (int64_t)unit * RP;
    for (int i = tid; i < RN; i += blockDim.x) pB[i] = Bg[lastg * RN + i];
    for (int i = tid; i < RP; i += blockDim.x) px[i] = xg[last * RP + i];
  }
}

}  // namespace m3
