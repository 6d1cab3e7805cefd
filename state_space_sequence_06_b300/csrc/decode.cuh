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
#include "umma.cuh"

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
  void* y;   // f32, or bf16 when ybf
  int ybf;
  float* h;
  void* prev_B;
  void* prev_x;
  int H, P, N, R;
  int G;   // B and C groups (head h uses group h / (H / G))
  int K;   // N / 2
  int PP;  // P / 2
  int KG;  // k groups (blockDim.x / PP)
  int bulk;  // 1: every per-unit input row is a multiple of 16 bytes, so they arrive by bulk copy too
  int pro;   // m3_prologue flags
  const float* dt_bias;
};

// R is the rank when known at compile time; R == 0 reads it from p.R (<= 8).
// YB: y is written in bf16 (else f32); a template flag, so that the f32
// kernel is compiled exactly as without the option.
//
// The unit's state (K*P complex f32, 16-32 KB) moves HBM -> shared memory
// with one bulk asynchronous copy (completing on an mbarrier) issued before
// anything else, is updated in place, and goes back with one bulk copy: the
// bytes in flight per SM are set by shared memory (several CTAs of 16-32 KB
// each), not by registers.  Shared memory also holds, per pair k, a packed
// record of float2 entries {a_k, Bprev_r[k], B_r[k], C_r[k] for r < R} (KW
// float4 per pair) read with 128-bit broadcast loads (every lane of a warp
// works on the same k); each thread keeps the x values of its two p columns
// in registers.
// (rank 4 runs 128-thread CTAs: nine of them resident per SM, their
// registers and shared memory sized for it)
template <typename T, int ITEMS, int R_, bool YB>
__global__ void __launch_bounds__(R_ == 4 ? 128 : 256, R_ == 4 ? 9 : 0) decode_step_kernel(const DecodeParams p) {
  using namespace umma;
  extern __shared__ float4 smem4[];
  __shared__ __align__(8) uint64_t bar;
  constexpr int RMAX = R_ > 0 ? R_ : 8;
  constexpr int KW = (3 * RMAX + 2) / 2;  // float4 per pair record
  const int R = R_ > 0 ? R_ : p.R;
  const int K = p.K, N = p.N, P = p.P, PP = p.PP, KG = p.KG;
  float4* hsm = smem4;                                          // [K][PP]: the state, (re, im) x 2 per float4
  float* xs = reinterpret_cast<float*>(hsm + (size_t)K * PP);   // [2][R][P]: this token's x, previous x
  float4* kd = reinterpret_cast<float4*>(xs + 2 * RMAX * P);   // [K][KW] (16-byte aligned: RMAX * P is even)
  // raw per-unit inputs, when they arrive by bulk copy: B, C, prev B [R][N], x, prev x [R][P], theta [K]
  T* rawB = reinterpret_cast<T*>(kd + (size_t)K * KW);
  // the partial outputs [KG][R][P]: after the raw inputs for rank 1; for
  // higher ranks (larger records and outputs) in the records' and raw
  // inputs' room, once the update is done with them
  constexpr bool kRedOverRecords = R_ != 1;
  const T* raw_end = rawB + (p.bulk ? 3 * R * N + 2 * R * P + K : 0);
  float* red = kRedOverRecords ? reinterpret_cast<float*>(kd)
                               : reinterpret_cast<float*>((reinterpret_cast<uintptr_t>(raw_end) + 15) & ~uintptr_t(15));
  T* rawC = rawB + R * N;
  T* rawPB = rawC + R * N;
  T* rawX = rawPB + R * N;
  T* rawPX = rawX + R * P;
  T* rawTh = rawPX + R * P;

  const int unit = blockIdx.x;
  const int head = unit % p.H;
  const int tid = threadIdx.x;
  const int pp = tid % PP, kg = tid / PP;
  float4* hg = reinterpret_cast<float4*>(p.h) + (int64_t)unit * K * PP;
  const uint32_t state_bytes = (uint32_t)K * PP * 16;

  const T* xg = static_cast<const T*>(p.x) + (int64_t)unit * R * P;
  const int64_t brow = (int64_t)(unit / p.H) * p.G + head / (p.H / p.G);  // this unit's B / C row
  const T* Bg = static_cast<const T*>(p.B) + brow * R * N;
  const T* Cg = static_cast<const T*>(p.C) + brow * R * N;
  T* pBg = static_cast<T*>(p.prev_B) + (int64_t)unit * R * N;
  T* pxg = static_cast<T*>(p.prev_x) + (int64_t)unit * R * P;
  const T* thg = p.theta ? static_cast<const T*>(p.theta) + (int64_t)unit * K : nullptr;
  const uint32_t rn_bytes = (uint32_t)(R * N * sizeof(T)), rp_bytes = (uint32_t)(R * P * sizeof(T));
  const uint32_t th_bytes = p.theta ? (uint32_t)(K * sizeof(T)) : 0u;  // no theta: theta = 0

  // 1. start the copies first: the state is the traffic that matters, the
  //    per-unit inputs ride on the same barrier when their rows allow it.
  if (tid == 0) {
    mbar_init(saddr(&bar), 1);
    mbar_init_fence();
    const uint32_t tx = state_bytes + (p.bulk ? 3 * rn_bytes + 2 * rp_bytes + th_bytes : 0u);
    mbar_arrive_expect_tx(saddr(&bar), tx);
    bulk_g2s(saddr(hsm), hg, state_bytes, saddr(&bar));
    if (p.bulk) {
      bulk_g2s(saddr(rawB), Bg, rn_bytes, saddr(&bar));
      bulk_g2s(saddr(rawC), Cg, rn_bytes, saddr(&bar));
      bulk_g2s(saddr(rawPB), pBg, rn_bytes, saddr(&bar));
      bulk_g2s(saddr(rawX), xg, rp_bytes, saddr(&bar));
      bulk_g2s(saddr(rawPX), pxg, rp_bytes, saddr(&bar));
      if (th_bytes) bulk_g2s(saddr(rawTh), thg, th_bytes, saddr(&bar));
    }
  }
  const float dt = scan_dt(ldf(static_cast<const T*>(p.dt), unit), p.pro, p.dt_bias, head);
  const float lam = p.lam ? ldf(static_cast<const T*>(p.lam), unit) : 1.f;  // no lam: lam = 1
  const float A = p.A[head], D = p.D[head];
  const float decay = expf(dt * A);
  __syncthreads();  // the mbarrier initialisation is visible
  // 2. wait for the copies (bounded), then stage the per-unit operands as f32 pair records.
  bool landed = mbar_try_wait(saddr(&bar), 0);
  for (uint32_t i = 0; !landed && i < (1u << 24); ++i) landed = mbar_try_wait(saddr(&bar), 0);
  if (!__syncthreads_and(landed)) {
    if (tid == 0) atomicExch(&g_status, (int)M3_ERR_TIMEOUT);
    return;
  }
  const T* sB = p.bulk ? rawB : Bg;
  const T* sC = p.bulk ? rawC : Cg;
  const T* sPB = p.bulk ? rawPB : pBg;
  const T* sX = p.bulk ? rawX : xg;
  const T* sPX = p.bulk ? rawPX : pxg;
  const T* sTh = p.bulk ? rawTh : thg;
  // BC norm: one scale per row (B_r, C_r, carried B_r), a warp per row
  __shared__ float s_scale[3 * RMAX];
  const bool norm = (p.pro & M3_PRO_BC_NORM) != 0;
  if (norm) {
    for (int row = tid / 32; row < 3 * R; row += blockDim.x / 32) {
      const T* src = row < R ? sB + row * N : (row < 2 * R ? sC + (row - R) * N : sPB + (row - 2 * R) * N);
      const float sc = warp_rms_scale(src, N, tid % 32);
      if (tid % 32 == 0) s_scale[row] = sc;
    }
    __syncthreads();
  }
  float2* kd2 = reinterpret_cast<float2*>(kd);
  for (int i = tid; i < K * R; i += blockDim.x) {
    const int k = i / R, r = i % R;
    const float fb = norm ? s_scale[r] : 1.f, fc = norm ? s_scale[R + r] : 1.f, fp = norm ? s_scale[2 * R + r] : 1.f;
    float2* rec = kd2 + (size_t)k * 2 * KW;
    rec[1 + r] = make_float2(fp * to_f(sPB[r * N + 2 * k]), fp * to_f(sPB[r * N + 2 * k + 1]));
    rec[1 + R + r] = make_float2(fb * to_f(sB[r * N + 2 * k]), fb * to_f(sB[r * N + 2 * k + 1]));
    rec[1 + 2 * R + r] = make_float2(fc * to_f(sC[r * N + 2 * k]), fc * to_f(sC[r * N + 2 * k + 1]));
  }
  for (int i = tid; i < R * P; i += blockDim.x) {
    xs[i] = to_f(sX[i]);
    xs[R * P + i] = to_f(sPX[i]);
  }
  for (int k = tid; k < K; k += blockDim.x) {
    float sn, cs;
    if (p.theta) {
      sincosf(dt * to_f(sTh[k]), &sn, &cs);
    } else {
      sn = 0.f;
      cs = 1.f;
    }
    kd2[(size_t)k * 2 * KW] = make_float2(decay * cs, decay * sn);
  }
  __syncthreads();  // records staged; the old carry is no longer needed

  // 3. the carry becomes this token's (B, x)
  if (p.bulk) {
    if (tid == 0) {  // straight from the staged copies
      bulk_s2g(pBg, saddr(rawB), rn_bytes);
      bulk_s2g(pxg, saddr(rawX), rp_bytes);
      bulk_commit();
    }
  } else {
    for (int i = tid; i < R * N; i += blockDim.x) pBg[i] = Bg[i];
    for (int i = tid; i < R * P; i += blockDim.x) pxg[i] = xg[i];
  }

  // 4. update the owned entries in place and accumulate partial outputs.
  const float gam = lam * dt, bet = (1.f - lam) * dt;
  const int p0 = 2 * pp;
  float xc0[RMAX], xc1[RMAX], xp0[RMAX], xp1[RMAX];
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    const bool on = r < R;
    xc0[r] = on ? xs[r * P + p0] : 0.f;
    xc1[r] = on ? xs[r * P + p0 + 1] : 0.f;
    xp0[r] = on ? xs[R * P + r * P + p0] : 0.f;
    xp1[r] = on ? xs[R * P + r * P + p0 + 1] : 0.f;
  }
  float ypart[2 * RMAX];
#pragma unroll
  for (int i = 0; i < 2 * RMAX; ++i) ypart[i] = 0.f;
#pragma unroll(R_ == 1 ? ITEMS : 1)
  for (int i = 0; i < ITEMS; ++i) {
    const int k = kg + i * KG;
    if (k < K) {
      const float2* rec = kd2 + (size_t)k * 2 * KW;  // broadcast reads: every lane works on this k
      float ur0 = 0.f, ui0 = 0.f, ur1 = 0.f, ui1 = 0.f;  // u_prev at p0, p0+1
      float vr0 = 0.f, vi0 = 0.f, vr1 = 0.f, vi1 = 0.f;  // u_t at p0, p0+1
#pragma unroll
      for (int r = 0; r < RMAX; ++r) {
        if (r >= R) break;
        const float2 bp = rec[1 + r], bc = rec[1 + R + r];
        ur0 = fmaf(bp.x, xp0[r], ur0); ui0 = fmaf(bp.y, xp0[r], ui0);
        ur1 = fmaf(bp.x, xp1[r], ur1); ui1 = fmaf(bp.y, xp1[r], ui1);
        vr0 = fmaf(bc.x, xc0[r], vr0); vi0 = fmaf(bc.y, xc0[r], vi0);
        vr1 = fmaf(bc.x, xc1[r], vr1); vi1 = fmaf(bc.y, xc1[r], vi1);
      }
      const float2 a = rec[0];
      const float4 hv = hsm[(size_t)k * PP + pp];
      // g = h + bet * u_prev ; h' = a * g + gam * u_t
      const float g0r = fmaf(bet, ur0, hv.x), g0i = fmaf(bet, ui0, hv.y);
      const float g1r = fmaf(bet, ur1, hv.z), g1i = fmaf(bet, ui1, hv.w);
      float4 o;
      o.x = fmaf(a.x, g0r, fmaf(-a.y, g0i, gam * vr0));
      o.y = fmaf(a.x, g0i, fmaf(a.y, g0r, gam * vi0));
      o.z = fmaf(a.x, g1r, fmaf(-a.y, g1i, gam * vr1));
      o.w = fmaf(a.x, g1i, fmaf(a.y, g1r, gam * vi1));
      hsm[(size_t)k * PP + pp] = o;
#pragma unroll
      for (int r = 0; r < RMAX; ++r) {
        if (r >= R) break;
        const float2 cc = rec[1 + 2 * R + r];
        ypart[2 * r] = fmaf(cc.x, o.x, fmaf(cc.y, o.y, ypart[2 * r]));
        ypart[2 * r + 1] = fmaf(cc.x, o.z, fmaf(cc.y, o.w, ypart[2 * r + 1]));
      }
    }
  }

  // 5. write the state back (one bulk copy) and reduce the partial outputs
  //    (over the records and raw inputs: every thread is past the update,
  //    and the carry's copy has read its rows)
  if (kRedOverRecords) {
    if (tid == 0 && p.bulk) bulk_wait_read_all();
    __syncthreads();
  }
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    if (r >= R) break;
    *reinterpret_cast<float2*>(&red[(kg * R + r) * P + p0]) = make_float2(ypart[2 * r], ypart[2 * r + 1]);
  }
  fence_async_smem();
  __syncthreads();
  if (tid == 0) {
    bulk_s2g(hg, saddr(hsm), state_bytes);
    bulk_commit();
  }
  const int64_t y0 = (int64_t)unit * R * P;
  auto y_at = [&](int i) {
    float sum = 0.f;
    for (int g = 0; g < KG; ++g) sum += red[g * R * P + i];
    return fmaf(D, xs[i], sum);
  };
  for (int i = tid; i < R * P; i += blockDim.x) st_y(p.y, y0 + i, y_at(i), YB);
  if (tid == 0) bulk_wait_read_all();  // shared memory must outlive the copy's reads
}

}  // namespace m3
