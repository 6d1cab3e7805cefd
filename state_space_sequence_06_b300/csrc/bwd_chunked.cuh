// Backward pass of the scan, chunked: every chunk of every (sequence,
// head) unit in parallel, f32 arithmetic.
//
// The pages train their models but give no backward kernel ("Together AI
// announces Mamba-3", sections 1-3 give the forward recurrence).  This is
// the exact adjoint of that recurrence, reorganised by chunks of Q tokens
// the way the forward's chunked form is (the Mamba-2 state-space/attention
// duality of the same page's history table).  Inside a chunk, with the
// chunk-local log-decay Lam_t = sum_{s<=t} dt_s A and angle phi_t[k] =
// sum_{s<=t} dt_s theta_s[k] (both from the chunk start), the rotated
// operands Bt = Bhat e^{-i phi}, Ct = Chat e^{-i phi} and the weights
// wp_j = gamma_j + beta'_{j+1}:
//
//   y_t   = sum_{j<=t} Re(Ct_t^H Bt_j) e^{Lam_t - Lam_j} w_tj x_j        (intra)
//         + e^{Lam_t} Re(Ct_t^H H_s) + D x_t                           (inter)
//   H_e   = e^{i phi_end} (e^{Lam_end} H_s + sum_j f_j Bt_j x_j^T),  f_j = e^{Lam_end - Lam_j} wp_j
//
// where H_s is the true state at the chunk start (with the first token's
// previous-token term folded in) and H_e the same at its end.  So a chunk
// needs only H_s and the adjoint dH_e of H_e; everything else is local.
// Three phases:
//   1. chunk_sums (per chunk): Z = e^{i phi_end} sum_j f_j Bt_j x_j^T,
//      U = sum_t e^{Lam_t} Ct_t dy_t^T and alpha = e^{Lam_end + i phi_end}.
//   2. chunk_scan (per unit and state element): H_s(c+1) = alpha_c H_s(c) +
//      Z_c forwards, dH_e(c-1) = conj(alpha_c) dH_e(c) + U_c backwards.
//   3. chunk_grads (per chunk): the chunk's contractions transposed (all
//      gradients of its tokens), its share of dA and dD, and the gradient
//      of the weight wp of its last token (which reaches the next chunk's
//      first token through beta').
// Then unit_final adds that weight term and the carry's terms to the first
// tokens, and head_sums reduces dA and dD (and dt_bias) per head in a fixed
// order: no float atomics, the result is deterministic.
//
// Complex gradients are G_z = dL/dRe z + i dL/dIm z.  In shared memory the
// complex N/2 x P quantities are realified N x P matrices (row 2k the real
// parts of pair k, row 2k+1 the imaginary parts), and B, C rows keep the
// interleaved (re, im) layout of the inputs, so every complex contraction
// is a plain real one.  Each product is a block-wide SIMT matrix product
// out of shared memory (256 threads as 16 x 16, a TM x TN register tile per
// thread, odd row strides so that no two lanes of a warp hit one bank).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <type_traits>

#include "umma.cuh"

namespace m3bwd {

struct ChunkBwdParams {
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
  float* dx;
  float* dB;      // [b][L][GB][R][N]: GB = G (written directly) or H (per head, reduced over groups later)
  float* dC;
  float* ddt;     // [b][L][H]
  float* dlam;    // [b][L][H] or NULL
  float* dtheta;  // [b][L][H][K] or NULL
  float* dh0;     // [units][K][P][2] or NULL
  float* dprev_B; // [units][R][N] or NULL
  float* dprev_x; // [units][R][P] or NULL
  // scratch
  float2* Zs;      // [units][nch][K][P]
  float2* Us;      // [units][nch][K][P]
  float2* Hs;      // [units][nch + 1][K][P]: state at each chunk start, then h_final
  float2* dHe;     // [units][nch][K][P]: adjoint of the state at each chunk end
  float2* dHs0;    // [units][K][P]: adjoint of the state at the unit start
  float2* alpha;   // [units][nch][K]
  float* dwp_last; // [units][nch]
  float* dA_part;  // [units][nch]
  float* dD_part;  // [units][nch]
  int64_t L;
  int nch;
  int H, G, GB;  // heads, B/C groups of the inputs, rows of the dB/dC written here
  int* status;   // the library's device status word (a bounded wait that gives up writes M3_ERR_TIMEOUT)
};

template <typename T>
__device__ __forceinline__ float ldv(const void* p, int64_t i) {
  return to_f(static_cast<const T*>(p)[i]);
}

// Elements i and i + 1 (i even) in one read-only load.
template <typename T>
__device__ __forceinline__ float2 ld_pair(const void* p, int64_t i);
template <>
__device__ __forceinline__ float2 ld_pair<float>(const void* p, int64_t i) {
  return __ldg(reinterpret_cast<const float2*>(static_cast<const float*>(p) + i));
}
template <>
__device__ __forceinline__ float2 ld_pair<__nv_bfloat16>(const void* p, int64_t i) {
  const unsigned w = __ldg(reinterpret_cast<const unsigned*>(static_cast<const __nv_bfloat16*>(p) + i));
  return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Loads of the per-chunk loaders go out U iterations at a time (all loads of
// a batch before its shared-memory stores), so that several are in flight
// per thread: one CTA per SM holds few warps to hide their latency.
constexpr int kLoadBatch = 4;

// Block-wide C (+)= A * B over shared memory, the block's threads as (ty,
// tx) in TY x 16: the thread owns rows ty + TY i (i < TM) and columns
// tx + 16 j (j < TN).  a(m, k) and b(k, n) read the operands.
template <int TM, int TN, int TY = 16, class FA, class FB>
__device__ __forceinline__ void block_mm(float (&acc)[TM][TN], int K, FA a, FB b) {
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll 2
  for (int k = 0; k < K; ++k) {
    float av[TM], bv[TN];
#pragma unroll
    for (int i = 0; i < TM; ++i) av[i] = a(ty + TY * i, k);
#pragma unroll
    for (int j = 0; j < TN; ++j) bv[j] = b(k, tx + 16 * j);
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
  }
}

// The same product when both operands run along k in memory: a(m, k) =
// A[m SA + k], b(k, j) = B[j SB + k], with SA, SB and K multiples of 4 and
// 16-byte aligned rows.  Four k per 16-byte load of each operand, the
// products accumulated in the same order as block_mm.
template <int TM, int TN, int TY = 16>
__device__ __forceinline__ void block_mm_k4(float (&acc)[TM][TN], int K, const float* A, int SA, const float* B,
                                            int SB) {
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll 2
  for (int k = 0; k < K; k += 4) {
    float4 av[TM], bv[TN];
#pragma unroll
    for (int i = 0; i < TM; ++i) av[i] = *reinterpret_cast<const float4*>(A + (ty + TY * i) * SA + k);
#pragma unroll
    for (int j = 0; j < TN; ++j) bv[j] = *reinterpret_cast<const float4*>(B + (tx + 16 * j) * SB + k);
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TN; ++j) {
        acc[i][j] = fmaf(av[i].x, bv[j].x, acc[i][j]);
        acc[i][j] = fmaf(av[i].y, bv[j].y, acc[i][j]);
        acc[i][j] = fmaf(av[i].z, bv[j].z, acc[i][j]);
        acc[i][j] = fmaf(av[i].w, bv[j].w, acc[i][j]);
      }
  }
}

// Only the first operand along k in memory (a(m, k) = A[m SA + k], SA and
// K multiples of 4, 16-byte aligned rows): four k per load of A, B read as
// block_mm does; the same order of accumulation.
template <int TM, int TN, int TY, class FB>
__device__ __forceinline__ void block_mm_ak4(float (&acc)[TM][TN], int K, const float* A, int SA, FB b) {
  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
#pragma unroll 1
  for (int k = 0; k < K; k += 4) {
    float4 av[TM];
#pragma unroll
    for (int i = 0; i < TM; ++i) av[i] = *reinterpret_cast<const float4*>(A + (ty + TY * i) * SA + k);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float bv[TN];
#pragma unroll
      for (int j = 0; j < TN; ++j) bv[j] = b(k + u, tx + 16 * j);
#pragma unroll
      for (int i = 0; i < TM; ++i) {
        const float a = u == 0 ? av[i].x : u == 1 ? av[i].y : u == 2 ? av[i].z : av[i].w;
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(a, bv[j], acc[i][j]);
      }
    }
  }
}

template <int TM, int TN>
__device__ __forceinline__ void zero_acc(float (&acc)[TM][TN]) {
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TN; ++j) acc[i][j] = 0.f;
}

// Sum over the 16 lanes of a half warp (the threads of one tile row ty).
__device__ __forceinline__ float half_warp_sum(float v) {
#pragma unroll
  for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Shapes: P = 64, N in {64, 128}, Q * R = 64 rows per chunk.
template <int N_, int R_>
struct BwdCfg {
  static constexpr int N = N_, R = R_, P = 64, MR = 64, Q = MR / R, K = N / 2;
  // row strides: NS and PS are multiples of 4 (16-byte row starts for the
  // four-wide loads of block_mm_k4) that are not multiples of 8 floats, so
  // the eight lanes of a 16-byte access phase, on eight consecutive rows,
  // hit eight different 16-byte bank groups; MS is odd (scalar accesses down
  // a column meet no bank twice)
  static constexpr int NS = N + 4, PS = P + 4, MS = MR + 1;
  static constexpr int NT = 256;   // chunk sums (two CTAs per SM)
  static constexpr int NTG = 512;  // chunk gradients (one CTA per SM: more warps to hide latency)
  static constexpr int TYG = NTG / 16, TQG = MR / TYG;  // its thread rows, and rows per thread
};

// Per-chunk scalars, shared by the two per-chunk kernels.
template <int Q>
struct ChunkScalars {
  float dt[Q + 1], lam[Q + 1];  // token Q: the next chunk's first (beta' of wp_{Q-1}), 0 past the end
  float Lam[Q], eL[Q], wp[Q], f[Q], gam[Q];
};

// Load dt, lam of the chunk's tokens (and the next token), the local scan
// Lam, the weights; phi[t][k] the local angle scan (theta NULL: 0).
template <typename T, int Q, int K, int NT>
__device__ __forceinline__ void chunk_prologue(const ChunkBwdParams& p, int64_t tok0, int head, int n, float A,
                                               ChunkScalars<Q>& s, float* phi, float* sred) {
  const int tid = threadIdx.x;
  if (tid <= Q) {
    float d = 0.f, l = 1.f;
    const int64_t t = tok0 + tid;
    // token Q is the next chunk's first: only its beta' = (1 - lam) dt is used (0 past the end)
    const bool in = tid < n || (tid == n && (int64_t)(tok0 - (tok0 / p.L) * p.L) + n < p.L);
    if (in) {
      d = ldv<T>(p.dt, t * p.H + head);
      l = p.lam ? ldv<T>(p.lam, t * p.H + head) : 1.f;
    }
    s.dt[tid] = d;
    s.lam[tid] = l;
  }
  __syncthreads();
  // inclusive scan of dt * A over the chunk (whole warps take part: tokens
  // past Q add zero)
  constexpr int QW = (Q + 31) / 32 * 32;
  if (tid < QW) {
    float v = tid < n ? s.dt[tid] * A : 0.f;
    const int lane = tid & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float u = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v += u;
    }
    if (lane == 31) sred[tid >> 5] = v;
    if (tid < Q) s.Lam[tid] = v;
  }
  // theta of the chunk's tokens, staged for the angle scan
  for (int i0 = tid; i0 < Q * K / 2; i0 += NT * kLoadBatch) {
    float2 v[kLoadBatch];
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
      const int i = i0 + u * NT, t = (2 * i) / K;
      v[u] = (i < Q * K / 2 && t < n && p.theta)
                 ? ld_pair<T>(p.theta, (tok0 + t) * p.H * K + (int64_t)head * K + (2 * i) % K)
                 : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
      const int i = i0 + u * NT;
      if (i < Q * K / 2) {
        phi[2 * i] = v[u].x;
        phi[2 * i + 1] = v[u].y;
      }
    }
  }
  __syncthreads();
  if (tid < Q) {
    float v = s.Lam[tid];
    for (int w = 0; w < (tid >> 5); ++w) v += sred[w];
    s.Lam[tid] = v;
  }
  __syncthreads();
  if (tid < Q) {
    const float lam_end = s.Lam[n - 1];
    const bool on = tid < n;
    const float gam = on ? s.lam[tid] * s.dt[tid] : 0.f;
    const float wp = on ? gam + (1.f - s.lam[tid + 1]) * s.dt[tid + 1] : 0.f;
    s.gam[tid] = gam;
    s.wp[tid] = wp;
    s.f[tid] = on ? expf(lam_end - s.Lam[tid]) * wp : 0.f;
    s.eL[tid] = on ? expf(s.Lam[tid]) : 0.f;
  }
  // angle scan in place: thread k walks the chunk's tokens
  for (int k = tid; k < K; k += NT) {
    float ph = 0.f;
    for (int t = 0; t < Q; ++t) {
      ph = fmaf(s.dt[t], phi[t * K + k], ph);
      phi[t * K + k] = ph;
    }
  }
  __syncthreads();
}

// sin and cos of an angle of at most a few tens of radians: one reduction
// by 2 pi (rounded quotient), then the special-function unit on [-pi, pi].
__device__ __forceinline__ void sincos_angle(float x, float* s, float* c) {
  const float q = rintf(x * 0.15915494309189535f);
  __sincosf(fmaf(-q, 6.283185307179586f, x), s, c);
}

// Rows of the chunk's B and C rotated by e^{-i phi_t} into Bt, Ct [MR][NS]
// (zero rows past the chunk's end); one sine and cosine per (token, pair).
template <typename T, int R, int N, int K, int MR, int NS, int NT>
__device__ __forceinline__ void load_rotated(const void* Bsrc, const void* Csrc, int64_t tok0, int G, int grp, int n,
                                             const float* phi, float* Bt, float* Ct) {
  for (int i0 = threadIdx.x; i0 < MR * K; i0 += NT * kLoadBatch) {
    float2 bv[kLoadBatch], cv[kLoadBatch];
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
      const int i = i0 + u * NT, m = i / K, k = i % K, t = m / R, r = m % R;
      bv[u] = cv[u] = make_float2(0.f, 0.f);
      if (i < MR * K && t < n) {
        const int64_t o = (((tok0 + t) * G + grp) * R + r) * N + 2 * k;
        bv[u] = ld_pair<T>(Bsrc, o);
        cv[u] = ld_pair<T>(Csrc, o);
      }
    }
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
      const int i = i0 + u * NT, m = i / K, k = i % K, t = m / R;
      if (i >= MR * K) break;
      float sn = 0.f, cs = 1.f;
      if (t < n) sincos_angle(phi[t * K + k], &sn, &cs);
      const float2 b = bv[u], c = cv[u];
      Bt[m * NS + 2 * k] = b.x * cs + b.y * sn;  // e^{-i phi} (b.x + i b.y)
      Bt[m * NS + 2 * k + 1] = b.y * cs - b.x * sn;
      Ct[m * NS + 2 * k] = c.x * cs + c.y * sn;
      Ct[m * NS + 2 * k + 1] = c.y * cs - c.x * sn;
    }
  }
}

// Rows of x (type T) or dy (f32) of the chunk into dst[MR][PS], scaled by
// scale[t] (NULL: 1), zero past the chunk's end.
template <typename T, int R, int P, int MR, int PS, int NT>
__device__ __forceinline__ void load_rows(const T* src, int64_t tok0, int H, int head, int n, const float* scale,
                                          float* dst) {
  for (int i0 = threadIdx.x; i0 < MR * P / 2; i0 += NT * kLoadBatch) {
    float2 v[kLoadBatch];
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
      const int i = i0 + u * NT, m = (2 * i) / P, q = (2 * i) % P, t = m / R;
      v[u] = (i < MR * P / 2 && t < n) ? ld_pair<T>(src, ((tok0 + t) * H + head) * (R * P) + (m % R) * P + q)
                                       : make_float2(0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
      const int i = i0 + u * NT, m = (2 * i) / P, q = (2 * i) % P, t = m / R;
      if (i >= MR * P / 2) break;
      const float sc = (scale && t < n) ? scale[t] : 1.f;
      dst[m * PS + q] = v[u].x * sc;
      dst[m * PS + q + 1] = v[u].y * sc;
    }
  }
}

// ------------------------------------------------------------------ phase 1

template <typename T, int N_, int R_>
__global__ void __launch_bounds__(256) chunk_sums_kernel(const ChunkBwdParams p) {
  using Cfg = BwdCfg<N_, R_>;
  constexpr int N = Cfg::N, R = Cfg::R, P = Cfg::P, MR = Cfg::MR, Q = Cfg::Q, K = Cfg::K;
  constexpr int NS = Cfg::NS, PS = Cfg::PS, NT = Cfg::NT;
  extern __shared__ float sm[];
  float* Bt = sm;                // [MR][NS]
  float* Ct = Bt + MR * NS;      // [MR][NS]
  float* Xf = Ct + MR * NS;      // [MR][PS]: f_t x_t
  float* Ye = Xf + MR * PS;      // [MR][PS]: e^{Lam_t} dy_t
  float* phi = Ye;               // [Q][K] angles, until dy is loaded (Q K <= MR PS)
  static_assert(Q * K <= MR * PS, "angles fit in the dy tile");
  __shared__ ChunkScalars<Q> s;
  __shared__ float sred[32];
  __shared__ float sPhiEnd[K];

  const int c = blockIdx.x % p.nch, unit = blockIdx.x / p.nch;  // chunk c of unit `unit`
  const int b = unit / p.H, head = unit % p.H, grp = head / (p.H / p.G);
  const int64_t tok0 = (int64_t)b * p.L + (int64_t)c * Q;
  const int n = (int)((p.L - (int64_t)c * Q) < Q ? (p.L - (int64_t)c * Q) : Q);
  const float A = p.A[head];
  chunk_prologue<T, Q, K, NT>(p, tok0, head, n, A, s, phi, sred);
  load_rotated<T, R, N, K, MR, NS, NT>(p.B, p.C, tok0, p.G, grp, n, phi, Bt, Ct);
  load_rows<T, R, P, MR, PS, NT>(static_cast<const T*>(p.x), tok0, p.H, head, n, s.f, Xf);
  for (int k = threadIdx.x; k < K; k += NT) sPhiEnd[k] = phi[(n - 1) * K + k];
  __syncthreads();  // the angles are read: dy goes over them
  load_rows<float, R, P, MR, PS, NT>(p.dy, tok0, p.H, head, n, s.eL, Ye);
  __syncthreads();

  const int ty = threadIdx.x >> 4, tx = threadIdx.x & 15;
  constexpr int TM = N / 16, TN = P / 16;
  const int64_t base = ((int64_t)unit * p.nch + c) * K * P;
  {  // Z = e^{i phi_end} (Bt^T (f x)): rows n of the realified N x P result
    float acc[TM][TN];
    zero_acc(acc);
    block_mm<TM, TN>(acc, MR, [&](int m, int k) { return Bt[k * NS + m]; },
                     [&](int k, int q) { return Xf[k * PS + q]; });
    // rows 2k (re) and 2k + 1 (im) of a pair sit in lanes 16 apart
#pragma unroll
    for (int i = 0; i < TM; ++i) {
      const int row = ty + 16 * i, k = row >> 1;
      float sn, cs;
      sincos_angle(sPhiEnd[k], &sn, &cs);
#pragma unroll
      for (int j = 0; j < TN; ++j) {
        const float mine = acc[i][j], other = __shfl_xor_sync(0xffffffffu, mine, 16);
        const float v = (row & 1) ? fmaf(other, sn, mine * cs) : fmaf(mine, cs, -other * sn);
        reinterpret_cast<float*>(p.Zs + base)[(k * P + tx + 16 * j) * 2 + (row & 1)] = v;
      }
    }
  }
  {  // U = Ct^T (e^{Lam} dy)
    float acc[TM][TN];
    zero_acc(acc);
    block_mm<TM, TN>(acc, MR, [&](int m, int k) { return Ct[k * NS + m]; },
                     [&](int k, int q) { return Ye[k * PS + q]; });
#pragma unroll
    for (int i = 0; i < TM; ++i) {
      const int row = ty + 16 * i, k = row >> 1;
#pragma unroll
      for (int j = 0; j < TN; ++j)
        reinterpret_cast<float*>(p.Us + base)[(k * P + tx + 16 * j) * 2 + (row & 1)] = acc[i][j];
    }
  }
  if (threadIdx.x < K) {
    const int k = threadIdx.x;
    float sn, cs;
    sincosf(sPhiEnd[k], &sn, &cs);
    const float e = expf(s.Lam[n - 1]);
    p.alpha[(int64_t)unit * p.nch * K + (int64_t)c * K + k] = make_float2(e * cs, e * sn);
  }
}

// Phase 1 on the tensor cores: the same two products per chunk, Z = Bt^T
// (f x) and U = Ct^T (e^{Lam} dy) (N x P each, K = MR rows), as tcgen05
// MMAs from 128-byte-swizzled f16 tiles into TMEM.  Every operand is an
// f16 hi + lo pair (hi·hi + hi·lo + lo·hi, about 21 bits, as in the
// forward kernel); the rotated rows are the MN-major A operand (M = N state
// rows), x and dy the MN-major B operand (N = P).  Tiles: the rotated B
// and C rows [N/64 blocks][MR rows][128 B], hi and lo apart; x and dy rows
// [MR rows][128 B]; the local angles share the dy tiles until dy is
// loaded.  One thread issues the MMAs; every thread waits (bounded) on
// their commit, then warp w reads accumulator rows of TMEM lane quarter
// w % 4, Z for w < 4 and U for w >= 4.
__device__ __forceinline__ void half2_hilo(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 f = __half22float2(h);
  const __half2 l = __floats2half2_rn(a - f.x, b - f.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

template <int N, int MR>
struct SumsTcLayout {
  static constexpr int P = 64;
  static constexpr int BT = N * MR * 2;  // one f16 tile of rotated rows
  static constexpr int XT = MR * P * 2;  // one f16 tile of x or dy rows
  static constexpr int OFF_BHI = 0, OFF_BLO = BT, OFF_CHI = 2 * BT, OFF_CLO = 3 * BT;
  static constexpr int OFF_XHI = 4 * BT, OFF_XLO = OFF_XHI + XT, OFF_YHI = OFF_XLO + XT, OFF_YLO = OFF_YHI + XT;
  static constexpr int SMEM = OFF_YLO + XT + 1024;  // + alignment of the tiles to 1024 B
  static constexpr int TCOLS = 2 * P;               // Z, then U
};

constexpr uint32_t kSumsMaxPolls = 1u << 26;  // far beyond the few microseconds the products take

template <typename T, int N_, int R_>
__global__ void __launch_bounds__(256, 2) chunk_sums_tc_kernel(const ChunkBwdParams p) {
  using namespace m3::umma;
  using Cfg = BwdCfg<N_, R_>;
  using Lay = SumsTcLayout<N_, Cfg::MR>;
  constexpr int N = Cfg::N, R = Cfg::R, P = Cfg::P, MR = Cfg::MR, Q = Cfg::Q, K = Cfg::K, NT = Cfg::NT;
  static_assert(NT == 256, "eight warps: four lane quarters for each of Z and U");
  static_assert(Q * K * 4 <= 2 * Lay::XT, "the angles fit in the dy tiles");
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = smraw + ((1024u - (saddr(smraw) & 1023u)) & 1023u);
  float* phi = reinterpret_cast<float*>(sm + Lay::OFF_YHI);  // [Q][K] angles, until dy is loaded
  __shared__ ChunkScalars<Q> s;
  __shared__ float sred[32];
  __shared__ float sPhiEnd[K];
  __shared__ __align__(8) uint64_t bar_mma;
  __shared__ uint32_t tmem_s;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x % p.nch, unit = blockIdx.x / p.nch;
  const int b = unit / p.H, head = unit % p.H, grp = head / (p.H / p.G);
  const int64_t tok0 = (int64_t)b * p.L + (int64_t)c * Q;
  const int n = (int)((p.L - (int64_t)c * Q) < Q ? (p.L - (int64_t)c * Q) : Q);
  const float A = p.A[head];
  if (tid == 0) {
    mbar_init(saddr(&bar_mma), 1);
    mbar_init_fence();
  }
  if (warp == 0) {
    tmem_alloc(saddr(&tmem_s), Lay::TCOLS);
    tmem_relinquish();
  }
  chunk_prologue<T, Q, K, NT>(p, tok0, head, n, A, s, phi, sred);  // (ends with a barrier)

  // rotated B and C rows e^{-i phi_t} (b.x + i b.y) as f16 hi / lo pairs; zero past the chunk's end
  for (int i0 = tid; i0 < MR * K; i0 += NT * kLoadBatch) {
    float2 bv[kLoadBatch], cv[kLoadBatch];
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
      const int i = i0 + u * NT, m = i / K, k = i % K, t = m / R, r = m % R;
      bv[u] = cv[u] = make_float2(0.f, 0.f);
      if (i < MR * K && t < n) {
        const int64_t o = (((tok0 + t) * p.G + grp) * R + r) * N + 2 * k;
        bv[u] = ld_pair<T>(p.B, o);
        cv[u] = ld_pair<T>(p.C, o);
      }
    }
#pragma unroll
    for (int u = 0; u < kLoadBatch; ++u) {
      const int i = i0 + u * NT, m = i / K, k = i % K, t = m / R;
      if (i >= MR * K) break;
      float sn = 0.f, cs = 1.f;
      if (t < n) sincos_angle(phi[t * K + k], &sn, &cs);
      const uint32_t o = ((2 * k) / 64) * (MR * 128) + sw128_offset(m, (2 * k) % 64);
      uint32_t hi, lo;
      half2_hilo(bv[u].x * cs + bv[u].y * sn, bv[u].y * cs - bv[u].x * sn, hi, lo);
      *reinterpret_cast<uint32_t*>(sm + Lay::OFF_BHI + o) = hi;
      *reinterpret_cast<uint32_t*>(sm + Lay::OFF_BLO + o) = lo;
      half2_hilo(cv[u].x * cs + cv[u].y * sn, cv[u].y * cs - cv[u].x * sn, hi, lo);
      *reinterpret_cast<uint32_t*>(sm + Lay::OFF_CHI + o) = hi;
      *reinterpret_cast<uint32_t*>(sm + Lay::OFF_CLO + o) = lo;
    }
  }
  // rows of x (scaled by f_t) or dy (scaled by e^{Lam_t}) as f16 hi / lo pairs
  auto rows = [&](const auto* src, const float* scale, int off_hi, int off_lo) {
    using S = typename std::remove_cv<typename std::remove_pointer<decltype(src)>::type>::type;
    for (int i0 = tid; i0 < MR * P / 2; i0 += NT * kLoadBatch) {
      float2 v[kLoadBatch];
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) {
        const int i = i0 + u * NT, m = (2 * i) / P, q = (2 * i) % P, t = m / R;
        v[u] = (i < MR * P / 2 && t < n) ? ld_pair<S>(src, ((tok0 + t) * p.H + head) * (R * P) + (m % R) * P + q)
                                         : make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) {
        const int i = i0 + u * NT, m = (2 * i) / P, q = (2 * i) % P, t = m / R;
        if (i >= MR * P / 2) break;
        const float sc = t < n ? scale[t] : 0.f;
        uint32_t hi, lo;
        half2_hilo(v[u].x * sc, v[u].y * sc, hi, lo);
        const uint32_t o = sw128_offset(m, q);
        *reinterpret_cast<uint32_t*>(sm + off_hi + o) = hi;
        *reinterpret_cast<uint32_t*>(sm + off_lo + o) = lo;
      }
    }
  };
  rows(static_cast<const T*>(p.x), s.f, Lay::OFF_XHI, Lay::OFF_XLO);
  for (int k = tid; k < K; k += NT) sPhiEnd[k] = phi[(n - 1) * K + k];
  __syncthreads();  // the angles are read: dy goes over them
  rows(p.dy, s.eL, Lay::OFF_YHI, Lay::OFF_YLO);
  fence_async_smem();  // the tiles, written by these threads, are read by the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_s;
  if (tid == 0) {
    constexpr uint32_t idesc = idesc_f16_f32(N, P, 1, 1);
    auto mn = [&](int off, int ks) { return smem_desc(saddr(sm + off) + ks * 2048, MR * 128, 1024, kSwizzle128B); };
#pragma unroll 1
    for (int ks = 0; ks < MR / 16; ++ks) {
      mma_f16(tmem, mn(Lay::OFF_BHI, ks), mn(Lay::OFF_XHI, ks), idesc, ks > 0);
      mma_f16(tmem, mn(Lay::OFF_BHI, ks), mn(Lay::OFF_XLO, ks), idesc, 1);
      mma_f16(tmem, mn(Lay::OFF_BLO, ks), mn(Lay::OFF_XHI, ks), idesc, 1);
      mma_f16(tmem + P, mn(Lay::OFF_CHI, ks), mn(Lay::OFF_YHI, ks), idesc, ks > 0);
      mma_f16(tmem + P, mn(Lay::OFF_CHI, ks), mn(Lay::OFF_YLO, ks), idesc, 1);
      mma_f16(tmem + P, mn(Lay::OFF_CLO, ks), mn(Lay::OFF_YHI, ks), idesc, 1);
    }
    mma_commit(saddr(&bar_mma));
  }
  const bool done = mbar_wait(saddr(&bar_mma), 0, kSumsMaxPolls);
  tc_fence_after();
  if (__syncthreads_and(done)) {
    // warp w: TMEM lane quarter w % 4 (accumulator rows), Z (w < 4) or U
    const int qtr = warp & 3, which = warp >> 2;
    const int row = N == 128 ? 32 * qtr + lane : (lane < 16 ? 16 * qtr + lane : -1);
    const bool re = (lane & 1) == 0;  // rows 2k (re) and 2k + 1 (im) sit in adjacent lanes
    float sn = 0.f, cs = 1.f;
    if (which == 0 && row >= 0) sincos_angle(sPhiEnd[row >> 1], &sn, &cs);
    float2* dst = (which == 0 ? p.Zs : p.Us) + ((int64_t)unit * p.nch + c) * K * P + (row >> 1) * P;
    // two halves of 32 columns: (re, im) of the first 16 from the re lane
    // and of the last 16 from the im lane, each a 128-byte run of [K][P][2]
#pragma unroll 1
    for (int h0 = 0; h0 < P; h0 += 32) {
      float v[32];
#pragma unroll
      for (int cb = 0; cb < 32; cb += 16) {
        float w[16];
        tmem_ld16(tmem + ((uint32_t)(32 * qtr) << 16) + which * P + h0 + cb, w);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[cb + i] = w[i];
      }
      tmem_ld_wait();
      if (which == 0) {  // Z = e^{i phi_end} (Bt^T (f x))
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float other = __shfl_xor_sync(0xffffffffu, v[i], 1);
          v[i] = re ? fmaf(v[i], cs, -other * sn) : fmaf(other, sn, v[i] * cs);
        }
      }
      float2 out[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float other = __shfl_xor_sync(0xffffffffu, re ? v[16 + i] : v[i], 1);
        out[i] = re ? make_float2(v[i], other) : make_float2(other, v[16 + i]);
      }
      if (row >= 0) {
        float2* d = dst + h0 + (re ? 0 : 16);
#pragma unroll
        for (int i = 0; i < 16; i += 2)
          *reinterpret_cast<float4*>(d + i) = make_float4(out[i].x, out[i].y, out[i + 1].x, out[i + 1].y);
      }
    }
  } else {
    // the products did not complete in time: record it, and give them a
    // second bounded wait before the tensor memory goes away
    if (tid == 0) {
      atomicExch(p.status, 4 /* M3_ERR_TIMEOUT */);
      mbar_wait(saddr(&bar_mma), 0, kSumsMaxPolls);
    }
  }
  if (tid < K) {
    const int k = tid;
    float sn, cs;
    sincosf(sPhiEnd[k], &sn, &cs);
    const float e = expf(s.Lam[n - 1]);
    p.alpha[(int64_t)unit * p.nch * K + (int64_t)c * K + k] = make_float2(e * cs, e * sn);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, Lay::TCOLS);
}

// ------------------------------------------------------------------ phase 2

// One thread per complex state element (k, p) of a unit: the forward chain
// of chunk-start states and the backward chain of chunk-end adjoints.
template <typename T>
__global__ void __launch_bounds__(256) chunk_scan_kernel(const ChunkBwdParams p, int R, int N, int P) {
  const int K = N / 2, KP = K * P;
  const int bpu = (KP + blockDim.x - 1) / blockDim.x;  // blocks per unit
  const int unit = blockIdx.x / bpu;
  const int e = (blockIdx.x % bpu) * blockDim.x + threadIdx.x;
  if (e >= KP) return;
  const int k = e / P, q = e % P;
  const int b = unit / p.H, head = unit % p.H;
  const int64_t t0 = (int64_t)b * p.L * p.H + head;  // token 0's (row * H + head)
  // G'_{-1} = h0 + beta'_0 u_{-1}, u_{-1} = sum_r Bhat_prev[r][k] x_prev[r][p]
  float2 h = make_float2(0.f, 0.f);
  if (p.h0) h = reinterpret_cast<const float2*>(p.h0)[(int64_t)unit * KP + e];
  if (p.prev_B && p.prev_x) {
    const float dt0 = ldv<T>(p.dt, t0), lm0 = p.lam ? ldv<T>(p.lam, t0) : 1.f;
    const float bet0 = (1.f - lm0) * dt0;
    for (int r = 0; r < R; ++r) {
      const int64_t ob = ((int64_t)unit * R + r) * N + 2 * k;
      const float xv = bet0 * ldv<T>(p.prev_x, ((int64_t)unit * R + r) * P + q);
      h.x = fmaf(ldv<T>(p.prev_B, ob), xv, h.x);
      h.y = fmaf(ldv<T>(p.prev_B, ob + 1), xv, h.y);
    }
  }
  const float2* __restrict__ al = p.alpha + (int64_t)unit * p.nch * K + k;
  const float2* __restrict__ Z = p.Zs + (int64_t)unit * p.nch * KP + e;
  const float2* __restrict__ U = p.Us + (int64_t)unit * p.nch * KP + e;
  float2* __restrict__ Hs = p.Hs + (int64_t)unit * (p.nch + 1) * KP + e;
  float2* __restrict__ dHe = p.dHe + (int64_t)unit * p.nch * KP + e;
  constexpr int B4 = 4;  // chunks whose inputs are loaded ahead of the serial chain
  for (int c0 = 0; c0 < p.nch; c0 += B4) {
    float2 a[B4], z[B4];
#pragma unroll
    for (int i = 0; i < B4; ++i)
      if (c0 + i < p.nch) {
        a[i] = al[(int64_t)(c0 + i) * K];
        z[i] = Z[(int64_t)(c0 + i) * KP];
      }
#pragma unroll
    for (int i = 0; i < B4; ++i)
      if (c0 + i < p.nch) {
        Hs[(int64_t)(c0 + i) * KP] = h;
        h = make_float2(a[i].x * h.x - a[i].y * h.y + z[i].x, a[i].x * h.y + a[i].y * h.x + z[i].y);
      }
  }
  Hs[(int64_t)p.nch * KP] = h;  // h_final
  float2 g = make_float2(0.f, 0.f);
  if (p.dh_final) g = reinterpret_cast<const float2*>(p.dh_final)[(int64_t)unit * KP + e];
  for (int c1 = p.nch - 1; c1 >= 0; c1 -= B4) {
    float2 a[B4], u[B4];
#pragma unroll
    for (int i = 0; i < B4; ++i)
      if (c1 - i >= 0) {
        a[i] = al[(int64_t)(c1 - i) * K];
        u[i] = U[(int64_t)(c1 - i) * KP];
      }
#pragma unroll
    for (int i = 0; i < B4; ++i)
      if (c1 - i >= 0) {
        dHe[(int64_t)(c1 - i) * KP] = g;
        // dH_s = conj(alpha) dH_e + U
        g = make_float2(a[i].x * g.x + a[i].y * g.y + u[i].x, a[i].x * g.y - a[i].y * g.x + u[i].y);
      }
  }
  p.dHs0[(int64_t)unit * KP + e] = g;
  if (p.dh0) reinterpret_cast<float2*>(p.dh0)[(int64_t)unit * KP + e] = g;
}

// ------------------------------------------------------------------ phase 3

template <typename T, int N_, int R_>
__global__ void __launch_bounds__(BwdCfg<N_, R_>::NTG, 1) chunk_grads_kernel(const ChunkBwdParams p) {
  using Cfg = BwdCfg<N_, R_>;
  constexpr int N = Cfg::N, R = Cfg::R, P = Cfg::P, MR = Cfg::MR, Q = Cfg::Q, K = Cfg::K;
  constexpr int NS = Cfg::NS, PS = Cfg::PS, MS = Cfg::MS, NT = Cfg::NTG, TY = Cfg::TYG;
  extern __shared__ float sm[];
  float* Bt = sm;               // [MR][NS] rotated B rows
  float* Ct = Bt + MR * NS;     // [MR][NS] rotated C rows
  float* X = Ct + MR * NS;      // [MR][PS]
  float* dY = X + MR * PS;      // [MR][PS]
  float* Gs = dY + MR * PS;     // [N][PS] realified state at the chunk start
  float* dG = Gs + N * PS;      // [N][PS] realified adjoint of the chunk-end state, local frame
  float* T1 = dG + N * PS;      // [MR][MS] dM * S, then dS = dM * EW
  float* T2 = T1 + MR * MS;     // [MR][MS] dEW sums, then M = S * EW, then dPhi [MR][K]
  float* phi = T2 + MR * MS;    // [Q][K] local angles; later theta * rcPhi
  __shared__ ChunkScalars<Q> s;
  __shared__ float sred[32];
  __shared__ float sDLam[Q], sDwp[Q], sDgam[Q], sRow[MR], sRow2[MR];
  __shared__ float sDPhiEnd[K], sPhiEndPart[K][2];
  __shared__ float sWarp[NT / 32];
  // MIMO: dEW summed over rank pairs, and its products with EW and E
  constexpr int QS = (R > 1) ? Q * (Q + 1) : 1;
  __shared__ float sEWa[QS], sEWb[QS];

  const int c = blockIdx.x % p.nch, unit = blockIdx.x / p.nch;
  const int b = unit / p.H, head = unit % p.H, grp = head / (p.H / p.G);
  const int tid = threadIdx.x, ty = tid >> 4, tx = tid & 15, lane = tid & 31, warp = tid >> 5;
  const int64_t tok0 = (int64_t)b * p.L + (int64_t)c * Q;
  const int n = (int)((p.L - (int64_t)c * Q) < Q ? (p.L - (int64_t)c * Q) : Q);
  const float A = p.A[head], Dh = p.D[head];
  const int KP = K * P;

  chunk_prologue<T, Q, K, NT>(p, tok0, head, n, A, s, phi, sred);
  load_rotated<T, R, N, K, MR, NS, NT>(p.B, p.C, tok0, p.G, grp, n, phi, Bt, Ct);
  load_rows<T, R, P, MR, PS, NT>(static_cast<const T*>(p.x), tok0, p.H, head, n, nullptr, X);
  load_rows<float, R, P, MR, PS, NT>(p.dy, tok0, p.H, head, n, nullptr, dY);
  {
    // H_s, and dG = e^{-i phi_end} dH_e; dPhi_end[k] = -sum_p Im(conj(dH_e) H_e)
    const float2* hs = p.Hs + ((int64_t)unit * (p.nch + 1) + c) * KP;
    const float2* he = hs + KP;
    const float2* dhe = p.dHe + ((int64_t)unit * p.nch + c) * KP;
    static_assert((K * P) % (NT * kLoadBatch) == 0, "whole batches of state elements");
    for (int e0 = tid; e0 < KP; e0 += NT * kLoadBatch) {
      float2 hb[kLoadBatch], gb[kLoadBatch], nb[kLoadBatch];
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) {
        hb[u] = __ldg(hs + e0 + u * NT);
        gb[u] = __ldg(dhe + e0 + u * NT);
        nb[u] = __ldg(he + e0 + u * NT);
      }
#pragma unroll
      for (int u = 0; u < kLoadBatch; ++u) {
        const int e = e0 + u * NT;
        const int k = e / P, q = e % P;
        const float2 h = hb[u], g = gb[u], hn = nb[u];
        Gs[(2 * k) * PS + q] = h.x;
        Gs[(2 * k + 1) * PS + q] = h.y;
        float sn, cs;
        sincos_angle(phi[(n - 1) * K + k], &sn, &cs);
        dG[(2 * k) * PS + q] = g.x * cs + g.y * sn;  // e^{-i phi_end} g
        dG[(2 * k + 1) * PS + q] = g.y * cs - g.x * sn;
        // (P = 64: the two warps of one k reduce separately)
        float v = -(g.x * hn.y - g.y * hn.x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == 0) sPhiEndPart[k][(q >> 5) & 1] = v;
      }
    }
  }
  if (tid < Q) {
    sDLam[tid] = 0.f;
    sDwp[tid] = 0.f;
    sDgam[tid] = 0.f;
  }
  __syncthreads();
  if (tid < K) sDPhiEnd[tid] = sPhiEndPart[tid][0] + sPhiEndPart[tid][1];

  // EW_tj = e^{Lam_t - Lam_j} w_tj on the lower triangle (w_tj = wp_j, w_tt = gamma_t)
  auto ew_of = [&](int t, int j, float& E) {
    if (t < j || t >= n || j >= n) {
      E = 0.f;
      return 0.f;
    }
    if (t == j) {
      E = 1.f;
      return s.gam[t];
    }
    E = expf(s.Lam[t] - s.Lam[j]);
    return E * s.wp[j];
  };

  // ---- P1: S = Ct Bt^T and dM = dY X^T (MR x MR), their products with EW
  constexpr int TQ = Cfg::TQG, TC = MR / 16;  // rows and columns of an MR x MR tile per thread
  float accS[TQ][TC], accM[TQ][TC];
  zero_acc(accS);
  zero_acc(accM);
  block_mm_k4<TQ, TC, TY>(accS, N, Ct, NS, Bt, NS);
  block_mm_k4<TQ, TC, TY>(accM, P, dY, PS, X, PS);
#pragma unroll
  for (int i = 0; i < TQ; ++i)
#pragma unroll
    for (int j = 0; j < TC; ++j) T1[(ty + TY * i) * MS + tx + 16 * j] = accM[i][j] * accS[i][j];
  __syncthreads();
  // dEW_tj = sum over rank pairs of dM * S; a_tj = dEW EW, b_tj = dEW E (t > j)
  float* ewa = (R == 1) ? T2 : sEWa;
  float* ewb = (R == 1) ? T1 : sEWb;
  constexpr int ES = (R == 1) ? MS : Q + 1;
  for (int i = tid; i < Q * Q; i += NT) {
    const int t = i / Q, j = i % Q;
    float d = 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r)
#pragma unroll
      for (int r2 = 0; r2 < R; ++r2) d += T1[(t * R + r) * MS + j * R + r2];
    float E;
    const float ew = ew_of(t, j, E);
    if (t == j) sDgam[t] = d;
    ewa[t * ES + j] = d * ew;
    ewb[t * ES + j] = t > j ? d * E : 0.f;
  }
  __syncthreads();
  if (tid < Q) {  // row sums: + into dLam_t
    float a = 0.f;
    for (int j = 0; j < Q; ++j) a += ewa[tid * ES + j];
    sRow[tid] = a;
  } else if (tid >= 64 && tid < 64 + Q) {  // column sums: - into dLam_j, + into dwp_j
    const int j = tid - 64;
    float a = 0.f, w = 0.f;
    for (int t = 0; t < Q; ++t) {
      a += ewa[t * ES + j];
      w += ewb[t * ES + j];
    }
    sRow2[j] = a;
    sDwp[j] = w;
  }
  __syncthreads();
  if (tid < Q) sDLam[tid] = sRow[tid] - sRow2[tid];
  // M = S EW into T2, dS = dM EW into T1
#pragma unroll
  for (int i = 0; i < TQ; ++i)
#pragma unroll
    for (int j = 0; j < TC; ++j) {
      const int m = ty + TY * i, m2 = tx + 16 * j;
      float E;
      const float ew = ew_of(m / R, m2 / R, E);
      T2[m * MS + m2] = accS[i][j] * ew;
      T1[m * MS + m2] = accM[i][j] * ew;
    }
  __syncthreads();

  // ---- P2: the inter-chunk output's decay term, dLam_t += e^{Lam_t} sum dy (Ct^H Gs);
  //      and dLam_end += e^{Lam_end} Re sum conj(dG) Gs
  {
    constexpr int TP = P / 16;
    float acc[TQ][TP];
    zero_acc(acc);
    block_mm_ak4<TQ, TP, TY>(acc, N, Ct, NS, [&](int k, int q) { return Gs[k * PS + q]; });
#pragma unroll
    for (int i = 0; i < TQ; ++i) {
      const int m = ty + TY * i;
      float v = 0.f;
#pragma unroll
      for (int j = 0; j < TP; ++j) v = fmaf(dY[m * PS + tx + 16 * j], acc[i][j], v);
      v = half_warp_sum(v);
      if (tx == 0) sRow[m] = v;
    }
    float v = 0.f;
    for (int e = tid; e < N * P; e += NT) v = fmaf(dG[(e / P) * PS + e % P], Gs[(e / P) * PS + e % P], v);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) sWarp[warp] = v;
  }
  __syncthreads();
  if (tid < Q) {
    float v = 0.f;
#pragma unroll
    for (int r = 0; r < R; ++r) v += sRow[tid * R + r];
    sDLam[tid] += s.eL[tid] * v;
  }
  if (tid == 0) {
    float v = 0.f;
    for (int w = 0; w < NT / 32; ++w) v += sWarp[w];
    sred[0] = v * expf(s.Lam[n - 1]);  // added to dLam_end below
  }
  __syncthreads();

  // ---- P5: dX = M^T dY + f_j Bt dG + D dy
  {
    constexpr int TP = P / 16;
    float acc[TQ][TP], acc2[TQ][TP];
    zero_acc(acc);
    zero_acc(acc2);
    block_mm<TQ, TP, TY>(acc, MR, [&](int m, int k) { return T2[k * MS + m]; }, [&](int k, int q) { return dY[k * PS + q]; });
    block_mm_ak4<TQ, TP, TY>(acc2, N, Bt, NS, [&](int k, int q) { return dG[k * PS + q]; });
    float dd = 0.f;
#pragma unroll
    for (int i = 0; i < TQ; ++i) {
      const int m = ty + TY * i, t = m / R;
      if (t < n) {
        float* dst = p.dx + ((tok0 + t) * p.H + head) * (R * P) + (m % R) * P;
#pragma unroll
        for (int j = 0; j < TP; ++j) {
          const int q = tx + 16 * j;
          const float dyv = dY[m * PS + q];
          dst[q] = fmaf(Dh, dyv, fmaf(s.f[t], acc2[i][j], acc[i][j]));
          dd = fmaf(dyv, X[m * PS + q], dd);
        }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) dd += __shfl_xor_sync(0xffffffffu, dd, o);
    if (lane == 0) sWarp[warp] = dd;
  }
  __syncthreads();  // T2 (M) no longer read: it becomes dPhi [MR][K]
  if (tid == 0) {
    float dd = 0.f;
    for (int w = 0; w < NT / 32; ++w) dd += sWarp[w];
    p.dD_part[(int64_t)unit * p.nch + c] = dd;
  }
  float* dPhi = T2;

  // writes dB or dC rows (true frame: e^{i phi} times the rotated-frame
  // gradient) and the rows' share of dPhi, from a 4 x (N/16) tile whose
  // columns tx + 16 j pair up in lanes tx, tx ^ 1
  constexpr int TN = N / 16;
  auto emit = [&](float (&acc)[TQ][TN], const float* rot, float* dst_base, bool first) {
#pragma unroll
    for (int i = 0; i < TQ; ++i) {
      const int m = ty + TY * i, t = m / R;
#pragma unroll
      for (int j = 0; j < TN; ++j) {
        const int col = tx + 16 * j, k = col >> 1;
        const float mine = acc[i][j], other = __shfl_xor_sync(0xffffffffu, mine, 1);
        const float dre = (tx & 1) ? other : mine, dim = (tx & 1) ? mine : other;
        if (!(tx & 1)) {  // Im(conj(d) v) for the pair, v the rotated operand
          const float ph = dre * rot[m * NS + 2 * k + 1] - dim * rot[m * NS + 2 * k];
          dPhi[m * K + k] = first ? ph : dPhi[m * K + k] + ph;
        }
        if (t < n) {
          float sn, cs;
          sincos_angle(phi[t * K + k], &sn, &cs);
          const float v = (tx & 1) ? fmaf(dre, sn, dim * cs) : fmaf(dre, cs, -dim * sn);
          dst_base[((tok0 + t) * p.GB + (p.GB == p.H ? head : grp)) * (R * N) + (m % R) * N + col] = v;
        }
      }
    }
  };

  // ---- P4: dCt = dS Bt + e^{Lam_t} dY Gs^T
  {
    float acc[TQ][TN], acc2[TQ][TN];
    zero_acc(acc);
    zero_acc(acc2);
    block_mm<TQ, TN, TY>(acc, MR, [&](int m, int k) { return T1[m * MS + k]; }, [&](int k, int q) { return Bt[k * NS + q]; });
    block_mm_k4<TQ, TN, TY>(acc2, P, dY, PS, Gs, PS);
#pragma unroll
    for (int i = 0; i < TQ; ++i) {
      const float el = s.eL[(ty + TY * i) / R];
#pragma unroll
      for (int j = 0; j < TN; ++j) acc[i][j] = fmaf(el, acc2[i][j], acc[i][j]);
    }
    emit(acc, Ct, p.dC, true);
  }
  // ---- P6: dBt = dS^T Ct + f_j W, W = X dG^T; q_j = sum_n Bt W
  {
    float acc[TQ][TN], accw[TQ][TN];
    zero_acc(acc);
    zero_acc(accw);
    block_mm<TQ, TN, TY>(acc, MR, [&](int m, int k) { return T1[k * MS + m]; }, [&](int k, int q) { return Ct[k * NS + q]; });
    block_mm_k4<TQ, TN, TY>(accw, P, X, PS, dG, PS);
#pragma unroll
    for (int i = 0; i < TQ; ++i) {
      const int m = ty + TY * i;
      const float fv = s.f[m / R];
      float qv = 0.f;
#pragma unroll
      for (int j = 0; j < TN; ++j) {
        qv = fmaf(Bt[m * NS + tx + 16 * j], accw[i][j], qv);
        acc[i][j] = fmaf(fv, accw[i][j], acc[i][j]);
      }
      qv = half_warp_sum(qv);
      if (tx == 0) sRow[m] = qv;
    }
    emit(acc, Bt, p.dB, false);
  }
  __syncthreads();

  // ---- P7: the per-token scalars
  if (tid == 0) {
    // q_j: dwp_j += e^{Lam_end - Lam_j} q_j, dLam_end += sum f q, dLam_j -= f_j q_j
    const float lam_end = s.Lam[n - 1];
    float fq = 0.f;
    for (int t = 0; t < n; ++t) {
      float qv = 0.f;
      for (int r = 0; r < R; ++r) qv += sRow[t * R + r];
      sDwp[t] += expf(lam_end - s.Lam[t]) * qv;
      sDLam[t] -= s.f[t] * qv;
      fq += s.f[t] * qv;
    }
    sDLam[n - 1] += fq + sred[0];
    // Lam_t = sum_{s<=t} dt_s A: reverse cumulative sum
    float rc = 0.f, da = 0.f;
    for (int t = n - 1; t >= 0; --t) {
      rc += sDLam[t];
      sRow2[t] = A * rc;  // ddt share
      da = fmaf(s.dt[t], rc, da);
    }
    p.dA_part[(int64_t)unit * p.nch + c] = da;
    // wp_j = gamma_j + beta'_{j+1}: the last token's weight reaches the next chunk's first token
    p.dwp_last[(int64_t)unit * p.nch + c] = sDwp[n - 1];
  }
  // dPhi: reverse cumulative sum over the chunk's tokens (from the end's
  // rotation) -> dtheta = dt rcPhi, ddt += sum_k theta rcPhi
  for (int k = tid; k < K; k += NT) {
    float rc = sDPhiEnd[k];
    for (int t = n - 1; t >= 0; --t) {
      for (int r = 0; r < R; ++r) rc += dPhi[(t * R + r) * K + k];
      const float th = p.theta ? ldv<T>(p.theta, ((tok0 + t) * p.H + head) * K + k) : 0.f;
      if (p.dtheta) p.dtheta[((tok0 + t) * p.H + head) * K + k] = s.dt[t] * rc;
      phi[t * K + k] = th * rc;
    }
  }
  __syncthreads();
  if (tid < n) {
    const int t = tid;
    float v = sRow2[t];
    for (int k = 0; k < K; ++k) v += phi[t * K + k];
    // gamma_t = lam dt, beta'_t = (1 - lam) dt; beta'_t's gradient is dwp_{t-1}
    // (the chunk's first token gets the previous chunk's share afterwards)
    const float dgam = sDgam[t] + sDwp[t];
    const float dbet = t > 0 ? sDwp[t - 1] : 0.f;
    const float lm = s.lam[t], d = s.dt[t];
    const int64_t o = (tok0 + t) * p.H + head;
    p.ddt[o] = v + lm * dgam + (1.f - lm) * dbet;
    if (p.dlam) p.dlam[o] = d * (dgam - dbet);
  }
}

// ------------------------------------------------------------------ finishing passes

// Per unit: the weight term that crosses into each chunk's first token, and
// the carry: beta'_0 u_{-1} with u_{-1} = sum_r Bhat_prev[r] x_prev[r]^T.
template <typename T>
__global__ void __launch_bounds__(256) unit_final_kernel(const ChunkBwdParams p, int R, int N, int P, int Q) {
  __shared__ float sred[8];
  const int K = N / 2, KP = K * P;
  const int unit = blockIdx.x, b = unit / p.H, head = unit % p.H;
  const int tid = threadIdx.x;
  const int64_t tok0 = (int64_t)b * p.L;
  for (int c = 1 + tid; c < p.nch; c += blockDim.x) {
    const int64_t o = (tok0 + (int64_t)c * Q) * p.H + head;
    const float dbet = p.dwp_last[(int64_t)unit * p.nch + c - 1];
    const float lm = p.lam ? ldv<T>(p.lam, o) : 1.f, d = ldv<T>(p.dt, o);
    p.ddt[o] += (1.f - lm) * dbet;
    if (p.dlam) p.dlam[o] -= d * dbet;
  }
  // a NULL half of the carry reads as zeros
  auto pB = [&](int64_t i) { return p.prev_B ? ldv<T>(p.prev_B, i) : 0.f; };
  auto px = [&](int64_t i) { return p.prev_x ? ldv<T>(p.prev_x, i) : 0.f; };
  const int64_t o0 = tok0 * p.H + head;
  const float lm0 = p.lam ? ldv<T>(p.lam, o0) : 1.f, dt0 = ldv<T>(p.dt, o0);
  const float bet0 = (1.f - lm0) * dt0;
  const float2* g = p.dHs0 + (int64_t)unit * KP;
  if (p.prev_B && p.prev_x) {
    // dbeta'_0 = Re sum conj(dH_s0) u_{-1}
    float v = 0.f;
    for (int e = tid; e < KP; e += blockDim.x) {
      const int k = e / P, q = e % P;
      float ur = 0.f, ui = 0.f;
      for (int r = 0; r < R; ++r) {
        const float xv = px(((int64_t)unit * R + r) * P + q);
        ur = fmaf(pB(((int64_t)unit * R + r) * N + 2 * k), xv, ur);
        ui = fmaf(pB(((int64_t)unit * R + r) * N + 2 * k + 1), xv, ui);
      }
      v = fmaf(g[e].x, ur, fmaf(g[e].y, ui, v));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if ((tid & 31) == 0) sred[tid >> 5] = v;
    __syncthreads();
    if (tid == 0) {
      float d = 0.f;
      for (int w = 0; w < (int)(blockDim.x / 32); ++w) d += sred[w];
      p.ddt[o0] += (1.f - lm0) * d;
      if (p.dlam) p.dlam[o0] -= dt0 * d;
    }
  }
  // du = beta'_0 dH_s0: dprev_B[r][k] = sum_p du x_prev[r][p], dprev_x[r][p] = Re sum_k du conj(Bhat_prev[r][k])
  if (p.dprev_B)
    for (int i = tid; i < R * K; i += blockDim.x) {
      const int r = i / K, k = i % K;
      float sr = 0.f, si = 0.f;
      for (int q = 0; q < P; ++q) {
        const float xv = px(((int64_t)unit * R + r) * P + q);
        sr = fmaf(g[k * P + q].x, xv, sr);
        si = fmaf(g[k * P + q].y, xv, si);
      }
      p.dprev_B[((int64_t)unit * R + r) * N + 2 * k] = bet0 * sr;
      p.dprev_B[((int64_t)unit * R + r) * N + 2 * k + 1] = bet0 * si;
    }
  if (p.dprev_x)
    for (int i = tid; i < R * P; i += blockDim.x) {
      const int r = i / P, q = i % P;
      float sr = 0.f;
      for (int k = 0; k < K; ++k) {
        const int64_t ob = ((int64_t)unit * R + r) * N + 2 * k;
        sr = fmaf(g[k * P + q].x, pB(ob), fmaf(g[k * P + q].y, pB(ob + 1), sr));
      }
      p.dprev_x[((int64_t)unit * R + r) * P + q] = bet0 * sr;
    }
}

// dA and dD per head: the per-chunk partial sums over the batch, in order.
__global__ void __launch_bounds__(256) head_sums_kernel(const float* dA_part, const float* dD_part, int batch, int H,
                                                        int nch, float* dA, float* dD) {
  __shared__ float sa[256], sd[256];
  const int head = blockIdx.x, tid = threadIdx.x;
  float a = 0.f, d = 0.f;
  for (int i = tid; i < batch * nch; i += blockDim.x) {
    const int b = i / nch, c = i % nch;
    const int64_t o = ((int64_t)b * H + head) * nch + c;
    a += dA_part[o];
    d += dD_part[o];
  }
  sa[tid] = a;
  sd[tid] = d;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (tid < w) {
      sa[tid] += sa[tid + w];
      sd[tid] += sd[tid + w];
    }
    __syncthreads();
  }
  if (tid == 0) {
    dA[head] = sa[0];
    dD[head] = sd[0];
  }
}

// dB / dC of grouped inputs: per-head rows [b][L][H][R*N] summed over the
// heads of each group into [b][L][G][R*N], in head order.
__global__ void __launch_bounds__(256) group_sum_kernel(const float* per_head, float* out, int64_t rows_bl, int H,
                                                        int G, int RN) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t total = rows_bl * G * RN;
  if (i >= total) return;
  const int e = (int)(i % RN);
  const int64_t bg = i / RN;
  const int g = (int)(bg % G);
  const int64_t bl = bg / G;
  const int hpg = H / G;
  float v = 0.f;
  for (int h = g * hpg; h < (g + 1) * hpg; ++h) v += per_head[(bl * H + h) * RN + e];
  out[i] = v;
}

}  // namespace m3bwd
