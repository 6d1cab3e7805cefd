// Backward pass of the scan (token-serial reference kernel, f32).
//
// The pages train their models but give no backward kernel ("Together AI
// announces Mamba-3", sections 1-3 describe the forward recurrence).  This
// kernel is the exact adjoint of that recurrence, walked token by token per
// (sequence, head) unit:
//   forward:  s_t = h_{t-1} + beta'_t u_{t-1},  h_t = a_t s_t + gamma_t u_t
//   backward: G_h(t) = sum_r dy_t[r] Chat_t[r] + G_s(t+1),  G_s(t) = conj(a_t) G_h(t)
//             G_z(t)[k] = conj(a_t[k]) sum_p G_h(t) conj(s_t)   (exponent of a_t)
//             G_u(t) = gamma_t G_h(t) + beta'_{t+1} G_s(t+1)
// with complex gradients kept as dL/dRe + i dL/dIm.  It is a correct,
// simple kernel for training-parity use at modest sizes, not a fast one.
//
// Layout: one CTA per unit; thread i owns state elements e = i, i + NT, ...
// of the K x P grid (e = k * P + p).  A forward phase writes every h_t to a
// scratch history; the reverse phase keeps G_s in a second scratch array.
// Per-token sums over p or k go through shared-memory atomics, the shared
// B / C rows of a group and the per-head dA, dD through global atomics (the
// outputs are zeroed by the host first).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

// A translation unit of its own (backward.cu): its helpers live in their own
// namespace and it defines no library-wide device state.
namespace m3bwd {

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T>
__device__ __forceinline__ float ldf(const T* q, int64_t i) {
  return to_f(q[i]);
}

struct BackwardParams {
  const void* x;
  const void* B;
  const void* C;
  const void* dt;
  const void* lam;    // NULL: lam = 1
  const void* theta;  // NULL: theta = 0
  const float* A;
  const float* D;
  const float* h0;      // [units][K][P][2] or NULL
  const void* prev_B;   // [units][R][N] or NULL
  const void* prev_x;   // [units][R][P] or NULL
  const float* dy;      // [b][L][H][R][P]
  const float* dh_final;  // [units][K][P][2] or NULL
  float* dx;      // [b][L][H][R][P]
  float* dB;      // [b][L][G][R][N] (accumulated)
  float* dC;      // [b][L][G][R][N] (accumulated)
  float* ddt;     // [b][L][H]
  float* dlam;    // [b][L][H] or NULL
  float* dtheta;  // [b][L][H][K] or NULL
  float* dA;      // [H] (accumulated)
  float* dD;      // [H] (accumulated)
  float* dh0;     // [units][K][P][2] or NULL
  float* dprev_B; // [units][R][N] or NULL
  float* dprev_x; // [units][R][P] or NULL
  float2* hist;   // scratch [units][L][K][P]
  float2* gs;     // scratch [units][K][P]
  int64_t L;
  int H, P, N, K, R, G;
};

__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
  return make_float2(a.x * b.x - a.y * b.y, a.x * b.y + a.y * b.x);
}
__device__ __forceinline__ float2 cmul_conj(float2 a, float2 b) {  // a * conj(b)
  return make_float2(a.x * b.x + a.y * b.y, a.y * b.x - a.x * b.y);
}
__device__ __forceinline__ float2 conj_mul(float2 a, float2 b) {  // conj(a) * b
  return make_float2(a.x * b.x + a.y * b.y, a.x * b.y - a.y * b.x);
}

template <typename T>
__global__ void __launch_bounds__(256) backward_kernel(const BackwardParams p) {
  extern __shared__ float bsm[];
  const int R = p.R, P = p.P, K = p.K, N = p.N, H = p.H;
  const int RP = R * P, RK = R * K, KP = K * P;
  float* sx = bsm;                                         // [2][R][P] x of this token and the previous
  float* sdy = sx + 2 * RP;                                // [R][P]
  float* sdx = sdy + RP;                                   // [R][P]
  float2* sB = reinterpret_cast<float2*>(sdx + RP);        // [2][R][K] Bhat of this token and the previous
  float2* sC = sB + 2 * RK;                                // [R][K]
  float2* sa = sC + RK;                                    // [K]
  float2* sGa = sa + K;                                    // [K]
  float2* sdB = sGa + K;                                   // [R][K]
  float2* sdC = sdB + RK;                                  // [R][K]
  float* ssc = reinterpret_cast<float*>(sdC + RK);         // scalars

  const int unit = blockIdx.x;
  const int b = unit / H, head = unit % H;
  const int grp = head / (H / p.G);
  const int tid = threadIdx.x, NT = blockDim.x;
  const float A = p.A[head], Dh = p.D[head];
  const T* xg = static_cast<const T*>(p.x);
  const T* Bg = static_cast<const T*>(p.B);
  const T* Cg = static_cast<const T*>(p.C);
  const T* dtg = static_cast<const T*>(p.dt);
  const T* lmg = static_cast<const T*>(p.lam);
  const T* thg = static_cast<const T*>(p.theta);
  float2* hist = p.hist + (int64_t)unit * p.L * KP;
  float2* gs = p.gs + (int64_t)unit * KP;
  const int64_t tok0 = (int64_t)b * p.L;

  auto dt_at = [&](int64_t t) { return ldf(dtg, (tok0 + t) * H + head); };
  auto lam_at = [&](int64_t t) { return lmg ? ldf(lmg, (tok0 + t) * H + head) : 1.f; };
  // stage x and Bhat of token t (t < 0: the carry) into buffer slot `sl`
  auto stage_xb = [&](int64_t t, int sl) {
    for (int i = tid; i < RP; i += NT) {
      float v = 0.f;
      if (t >= 0) v = ldf(xg, ((tok0 + t) * H + head) * RP + i);
      else if (p.prev_x) v = ldf(static_cast<const T*>(p.prev_x), (int64_t)unit * RP + i);
      sx[sl * RP + i] = v;
    }
    for (int i = tid; i < RK; i += NT) {
      const int r = i / K, k = i % K;
      float2 v = make_float2(0.f, 0.f);
      if (t >= 0) {
        const int64_t o = (((tok0 + t) * p.G + grp) * R + r) * N + 2 * k;
        v = make_float2(ldf(Bg, o), ldf(Bg, o + 1));
      } else if (p.prev_B) {
        const int64_t o = ((int64_t)unit * R + r) * N + 2 * k;
        v = make_float2(ldf(static_cast<const T*>(p.prev_B), o), ldf(static_cast<const T*>(p.prev_B), o + 1));
      }
      sB[sl * RK + i] = v;
    }
  };
  auto stage_a = [&](int64_t t, float dt) {
    const float dec = expf(dt * A);
    for (int k = tid; k < K; k += NT) {
      float s = 0.f, c = 1.f;
      if (thg) sincosf(dt * ldf(thg, ((tok0 + t) * H + head) * K + k), &s, &c);
      sa[k] = make_float2(dec * c, dec * s);
    }
  };
  auto u_of = [&](int sl, int k, int pp) {  // sum_r Bhat[r][k] x[r][p] from slot sl
    float2 u = make_float2(0.f, 0.f);
    for (int r = 0; r < R; ++r) {
      const float2 bv = sB[sl * RK + r * K + k];
      const float xv = sx[sl * RP + r * P + pp];
      u.x = fmaf(bv.x, xv, u.x);
      u.y = fmaf(bv.y, xv, u.y);
    }
    return u;
  };
  auto h0_at = [&](int e) {
    return p.h0 ? make_float2(p.h0[((int64_t)unit * KP + e) * 2], p.h0[((int64_t)unit * KP + e) * 2 + 1])
                : make_float2(0.f, 0.f);
  };

  // ---- forward phase: h_t for every token into the history
  stage_xb(-1, 1);
  for (int64_t t = 0; t < p.L; ++t) {
    const int cur = (int)(t & 1), prv = cur ^ 1;
    const float dt = dt_at(t), lm = lam_at(t);
    stage_xb(t, cur);
    stage_a(t, dt);
    __syncthreads();
    const float bet = (1.f - lm) * dt, gam = lm * dt;
    for (int e = tid; e < KP; e += NT) {
      const int k = e / P, pp = e % P;
      const float2 hp = t ? hist[(t - 1) * KP + e] : h0_at(e);
      const float2 up = u_of(prv, k, pp), ut = u_of(cur, k, pp);
      const float2 s = make_float2(fmaf(bet, up.x, hp.x), fmaf(bet, up.y, hp.y));
      const float2 as = cmul(sa[k], s);
      hist[t * KP + e] = make_float2(fmaf(gam, ut.x, as.x), fmaf(gam, ut.y, as.y));
    }
    __syncthreads();
  }

  // ---- reverse phase
  float dA_part = 0.f, dD_part = 0.f;
  for (int64_t t = p.L - 1; t >= 0; --t) {
    const int cur = (int)(t & 1), prv = cur ^ 1;
    const float dt = dt_at(t), lm = lam_at(t);
    const float bet = (1.f - lm) * dt, gam = lm * dt;
    const float bet_next = (t + 1 < p.L) ? (1.f - lam_at(t + 1)) * dt_at(t + 1) : 0.f;
    stage_xb(t, cur);
    stage_xb(t - 1, prv);
    stage_a(t, dt);
    for (int i = tid; i < RP; i += NT) {
      sdy[i] = p.dy[((tok0 + t) * H + head) * RP + i];
      sdx[i] = 0.f;
    }
    for (int i = tid; i < RK; i += NT) {
      const int r = i / K, k = i % K;
      const int64_t o = (((tok0 + t) * p.G + grp) * R + r) * N + 2 * k;
      sC[i] = make_float2(ldf(Cg, o), ldf(Cg, o + 1));
      sdB[i] = make_float2(0.f, 0.f);
      sdC[i] = make_float2(0.f, 0.f);
    }
    for (int k = tid; k < K; k += NT) sGa[k] = make_float2(0.f, 0.f);
    if (tid < 4) ssc[tid] = 0.f;  // dgamma, dbeta', sum over k for ddt
    __syncthreads();
    float dgam_part = 0.f, dbet_part = 0.f;
    for (int e = tid; e < KP; e += NT) {
      const int k = e / P, pp = e % P;
      const float2 ht = hist[t * KP + e];
      const float2 hp = t ? hist[(t - 1) * KP + e] : h0_at(e);
      const float2 up = u_of(prv, k, pp), ut = u_of(cur, k, pp);
      const float2 s = make_float2(fmaf(bet, up.x, hp.x), fmaf(bet, up.y, hp.y));
      float2 gnext = make_float2(0.f, 0.f);
      if (t + 1 < p.L) {
        gnext = gs[e];
      } else if (p.dh_final) {
        gnext = make_float2(p.dh_final[((int64_t)unit * KP + e) * 2], p.dh_final[((int64_t)unit * KP + e) * 2 + 1]);
      }
      float2 gh = gnext;
      for (int r = 0; r < R; ++r) {
        const float d = sdy[r * P + pp];
        const float2 c = sC[r * K + k];
        gh.x = fmaf(d, c.x, gh.x);
        gh.y = fmaf(d, c.y, gh.y);
      }
      const float2 gsv = conj_mul(sa[k], gh);
      const float2 ga = cmul_conj(gh, s);
      atomicAdd(&sGa[k].x, ga.x);
      atomicAdd(&sGa[k].y, ga.y);
      dgam_part += cmul_conj(gh, ut).x;
      dbet_part += cmul_conj(gsv, up).x;
      const float2 gu = make_float2(gam * gh.x + bet_next * gnext.x, gam * gh.y + bet_next * gnext.y);
      for (int r = 0; r < R; ++r) {
        const float xv = sx[cur * RP + r * P + pp];
        atomicAdd(&sdB[r * K + k].x, gu.x * xv);
        atomicAdd(&sdB[r * K + k].y, gu.y * xv);
        atomicAdd(&sdx[r * P + pp], cmul_conj(gu, sB[cur * RK + r * K + k]).x);
        const float d = sdy[r * P + pp];
        atomicAdd(&sdC[r * K + k].x, d * ht.x);
        atomicAdd(&sdC[r * K + k].y, d * ht.y);
      }
      gs[e] = gsv;
    }
    atomicAdd(&ssc[0], dgam_part);
    atomicAdd(&ssc[1], dbet_part);
    __syncthreads();
    // per-token results
    for (int k = tid; k < K; k += NT) {
      const float2 gz = conj_mul(sa[k], sGa[k]);
      const float th = thg ? ldf(thg, ((tok0 + t) * H + head) * K + k) : 0.f;
      if (p.dtheta) p.dtheta[((tok0 + t) * H + head) * K + k] = dt * gz.y;
      atomicAdd(&ssc[2], gz.x * A + gz.y * th);
      dA_part += dt * gz.x;
    }
    for (int i = tid; i < RP; i += NT) {
      const float xv = sx[cur * RP + i];
      p.dx[((tok0 + t) * H + head) * RP + i] = fmaf(Dh, sdy[i], sdx[i]);
      dD_part += sdy[i] * xv;
    }
    for (int i = tid; i < RK; i += NT) {
      const int r = i / K, k = i % K;
      const int64_t o = (((tok0 + t) * p.G + grp) * R + r) * N + 2 * k;
      atomicAdd(&p.dB[o], sdB[i].x);
      atomicAdd(&p.dB[o + 1], sdB[i].y);
      atomicAdd(&p.dC[o], sdC[i].x);
      atomicAdd(&p.dC[o + 1], sdC[i].y);
    }
    __syncthreads();
    if (tid == 0) {
      const int64_t o = (tok0 + t) * H + head;
      p.ddt[o] = ssc[2] + (1.f - lm) * ssc[1] + lm * ssc[0];
      if (p.dlam) p.dlam[o] = dt * (ssc[0] - ssc[1]);
    }
    __syncthreads();  // before the next token overwrites the staged rows and sums
  }

  // ---- the initial state and the carry: G_s(0), u_{-1} = sum_r Bprev_r xprev_r
  const float bet0 = (1.f - lam_at(0)) * dt_at(0);
  stage_xb(-1, 1);
  for (int i = tid; i < RP; i += NT) sdx[i] = 0.f;
  for (int i = tid; i < RK; i += NT) sdB[i] = make_float2(0.f, 0.f);
  __syncthreads();
  for (int e = tid; e < KP; e += NT) {
    const int k = e / P, pp = e % P;
    const float2 g0 = gs[e];
    if (p.dh0) {
      p.dh0[((int64_t)unit * KP + e) * 2] = g0.x;
      p.dh0[((int64_t)unit * KP + e) * 2 + 1] = g0.y;
    }
    const float2 gu = make_float2(bet0 * g0.x, bet0 * g0.y);
    for (int r = 0; r < R; ++r) {
      const float xv = sx[RP + r * P + pp];
      atomicAdd(&sdB[r * K + k].x, gu.x * xv);
      atomicAdd(&sdB[r * K + k].y, gu.y * xv);
      atomicAdd(&sdx[r * P + pp], cmul_conj(gu, sB[RK + r * K + k]).x);
    }
  }
  __syncthreads();
  if (p.dprev_x)
    for (int i = tid; i < RP; i += NT) p.dprev_x[(int64_t)unit * RP + i] = sdx[i];
  if (p.dprev_B)
    for (int i = tid; i < RK; i += NT) {
      const int r = i / K, k = i % K;
      p.dprev_B[((int64_t)unit * R + r) * N + 2 * k] = sdB[i].x;
      p.dprev_B[((int64_t)unit * R + r) * N + 2 * k + 1] = sdB[i].y;
    }
  // per-head sums over the batch
  atomicAdd(&p.dA[head], dA_part);
  atomicAdd(&p.dD[head], dD_part);
}

}  // namespace m3bwd
