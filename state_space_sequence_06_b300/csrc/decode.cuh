// Single-token decode step: one read-modify-write pass over the f32 state.
//
// "Together AI announces Mamba-3", section 3 (MIMO): decode is bound by
// memory traffic (about 2.5 ops/byte for the SISO update), and a rank-R
// update raises the arithmetic per byte without adding traffic.  This
// kernel therefore moves the state exactly once per step -- one 16-byte
// load and one 16-byte store per two complex entries -- and folds
// everything else into that pass: the decay and rotation a = exp(dt(A +
// i*theta)), the trapezoid term built from the carried previous token, the
// rank-R input u = sum_r Bhat_r x_r^T, the output contraction over the
// pairs, and the carry update.
//
// Layout: one CTA per (sequence, head) unit.  Thread (pp, kg) owns the two
// complex entries h[k][2pp], h[k][2pp+1] (one float4) for k = kg, kg+KG, ...
// so a warp reads 32 consecutive float4 (512 contiguous bytes) per load.
// The per-unit operands (B, C, x and the carry, a few hundred bytes) are
// staged in shared memory; partial outputs are reduced over the KG thread
// groups through shared memory.
#pragma once

#include "common.cuh"

namespace m3 {

struct DecodeParams {
  const void* x;
  const void* B;
  const void* C;
  const void* dt;
  const void* lam;
  const void* theta;
  const float* A;
  const float* D;
  float* y;
  float* h;
  void* prev_B;
  void* prev_x;
  int H, P, N, R;
  int K;   // N / 2
  int PP;  // P / 2
  int KG;  // k groups (blockDim.x / PP)
};

// R is the rank when known at compile time; R == 0 reads it from p.R (<= 8).
template <typename T, int ITEMS, int R_>
__global__ void __launch_bounds__(256) decode_step_kernel(const DecodeParams p) {
  extern __shared__ float smem[];
  constexpr int RMAX = R_ > 0 ? R_ : 8;
  const int R = R_ > 0 ? R_ : p.R;
  const int K = p.K, N = p.N, P = p.P, PP = p.PP, KG = p.KG;
  float2* alpha = reinterpret_cast<float2*>(smem);  // [K]
  float* Bc = smem + 2 * K;                         // [R][N] this token's B
  float* Bp = Bc + R * N;                           // [R][N] previous token's B
  float* Cc = Bp + R * N;                           // [R][N]
  float* xc = Cc + R * N;                           // [R][P]
  float* xp = xc + R * P;                           // [R][P]
  float* red = xp + R * P;                          // [KG][R][P]

  const int unit = blockIdx.x;
  const int head = unit % p.H;
  const int tid = threadIdx.x;
  const int pp = tid % PP, kg = tid / PP;

  // 1. issue the state loads first: they are the traffic that matters.
  float4* hs = reinterpret_cast<float4*>(p.h) + (int64_t)unit * K * PP;
  float4 hv[ITEMS];
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const int k = kg + i * KG;
    if (k < K) hv[i] = ld_stream(hs + (int64_t)k * PP + pp);
  }

  // 2. stage the per-unit operands as f32.
  const T* xg = static_cast<const T*>(p.x) + (int64_t)unit * R * P;
  const T* Bg = static_cast<const T*>(p.B) + (int64_t)unit * R * N;
  const T* Cg = static_cast<const T*>(p.C) + (int64_t)unit * R * N;
  T* pBg = static_cast<T*>(p.prev_B) + (int64_t)unit * R * N;
  T* pxg = static_cast<T*>(p.prev_x) + (int64_t)unit * R * P;
  const float dt = ldf(static_cast<const T*>(p.dt), unit);
  const float lam = ldf(static_cast<const T*>(p.lam), unit);
  const float A = p.A[head], D = p.D[head];
  for (int i = tid; i < R * N; i += blockDim.x) {
    Bc[i] = to_f(Bg[i]);
    Bp[i] = to_f(pBg[i]);
    Cc[i] = to_f(Cg[i]);
  }
  for (int i = tid; i < R * P; i += blockDim.x) {
    xc[i] = to_f(xg[i]);
    xp[i] = to_f(pxg[i]);
  }
  const float decay = expf(dt * A);
  const T* thg = static_cast<const T*>(p.theta) + (int64_t)unit * K;
  for (int k = tid; k < K; k += blockDim.x) {
    float s, c;
    sincosf(dt * to_f(thg[k]), &s, &c);
    alpha[k] = make_float2(decay * c, decay * s);
  }
  __syncthreads();

  // 3. the carry becomes this token's (B, x); the old one is in smem now.
  for (int i = tid; i < R * N; i += blockDim.x) pBg[i] = Bg[i];
  for (int i = tid; i < R * P; i += blockDim.x) pxg[i] = xg[i];

  // 4. update the owned entries and accumulate partial outputs.
  const float gam = lam * dt, bet = (1.f - lam) * dt;
  float ypart[2 * RMAX];  // [R][2]
#pragma unroll
  for (int i = 0; i < 2 * RMAX; ++i) ypart[i] = 0.f;
  const int p0 = 2 * pp;
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const int k = kg + i * KG;
    if (k < K) {
      float ur0 = 0.f, ui0 = 0.f, ur1 = 0.f, ui1 = 0.f;  // u_prev at p0, p0+1
      float vr0 = 0.f, vi0 = 0.f, vr1 = 0.f, vi1 = 0.f;  // u_t at p0, p0+1
#pragma unroll
      for (int r = 0; r < RMAX; ++r) {
        if (r >= R) break;
        const float bpr = Bp[r * N + 2 * k], bpi = Bp[r * N + 2 * k + 1];
        const float bcr = Bc[r * N + 2 * k], bci = Bc[r * N + 2 * k + 1];
        const float xp0 = xp[r * P + p0], xp1 = xp[r * P + p0 + 1];
        const float xc0 = xc[r * P + p0], xc1 = xc[r * P + p0 + 1];
        ur0 = fmaf(bpr, xp0, ur0); ui0 = fmaf(bpi, xp0, ui0);
        ur1 = fmaf(bpr, xp1, ur1); ui1 = fmaf(bpi, xp1, ui1);
        vr0 = fmaf(bcr, xc0, vr0); vi0 = fmaf(bci, xc0, vi0);
        vr1 = fmaf(bcr, xc1, vr1); vi1 = fmaf(bci, xc1, vi1);
      }
      const float2 a = alpha[k];
      // g = h + bet * u_prev ; h' = a * g + gam * u_t
      const float g0r = fmaf(bet, ur0, hv[i].x), g0i = fmaf(bet, ui0, hv[i].y);
      const float g1r = fmaf(bet, ur1, hv[i].z), g1i = fmaf(bet, ui1, hv[i].w);
      float4 o;
      o.x = fmaf(a.x, g0r, fmaf(-a.y, g0i, gam * vr0));
      o.y = fmaf(a.x, g0i, fmaf(a.y, g0r, gam * vi0));
      o.z = fmaf(a.x, g1r, fmaf(-a.y, g1i, gam * vr1));
      o.w = fmaf(a.x, g1i, fmaf(a.y, g1r, gam * vi1));
      st_stream(hs + (int64_t)k * PP + pp, o);
#pragma unroll
      for (int r = 0; r < RMAX; ++r) {
        if (r >= R) break;
        const float cr = Cc[r * N + 2 * k], ci = Cc[r * N + 2 * k + 1];
        ypart[2 * r] = fmaf(cr, o.x, fmaf(ci, o.y, ypart[2 * r]));
        ypart[2 * r + 1] = fmaf(cr, o.z, fmaf(ci, o.w, ypart[2 * r + 1]));
      }
    }
  }

  // 5. reduce the partial outputs over the KG groups.
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    if (r >= R) break;
    red[(kg * R + r) * P + p0] = ypart[2 * r];
    red[(kg * R + r) * P + p0 + 1] = ypart[2 * r + 1];
  }
  __syncthreads();
  float* yg = p.y + (int64_t)unit * R * P;
  for (int i = tid; i < R * P; i += blockDim.x) {
    float s = 0.f;
    for (int g = 0; g < KG; ++g) s += red[g * R * P + i];
    yg[i] = fmaf(D, xc[i], s);
  }
}

}  // namespace m3
