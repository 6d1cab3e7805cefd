// Chunked prefill on the tensor cores: tcgen05 MMAs with TMEM accumulators,
// inputs staged by TMA.
//
// The recurrence ("Together AI announces Mamba-3", sections 1-3: an
// exponential-trapezoid update of a complex state applied as a rotation,
// SISO or rank-R MIMO) is evaluated chunk by chunk.  The Mamba-2
// state-space/attention duality (same page, history table) turns each
// chunk into dense products.  Inside a chunk of Q tokens, with chunk-local
// cumulative log-decay Lam_i = sum_{s<=i} dt_s A and angle phi_i[k] =
// sum_{s<=i} dt_s theta_s[k], and psi_i = phi_end - phi_i:
//
//   Bt_j = Bhat_j e^{i psi_j},  Ct_t = Chat_t e^{i psi_t}     (rotations, f16)
//   S    = Re(Ct Bt^H)    = realified Ct . Bt^T                (MMA 1)
//   S'   = S * e^{Lam_t - Lam_j} * w_tj  for j <= t, else 0
//          w_tt = lam_t dt_t,  w_tj = lam_j dt_j + (1 - lam_{j+1}) dt_{j+1}
//   Y    = S' X                                                (MMA 2)
//        + e^{Lam_t} Re(Ct^H R),  R = e^{i phi_end} h'_prev     (MMA 3)
//        + D x
//   h'   = e^{Lam_end} R + Bt^T (W X),  W_j = e^{Lam_end - Lam_j} w'_j  (MMA 4)
//
// where w'_j = lam_j dt_j + (1 - lam_{j+1}) dt_{j+1}, the next token's
// trapezoid coefficient included (zero past the end of the sequence), so
// the state carried between chunks already holds the next token's
// previous-token term.  Every rotation angle is chunk-local (the state
// absorbs e^{i phi_end} once per chunk) and every decay is the exponential
// of a difference, so nothing overflows or loses its phase in f32 at any
// sequence length.
//
// One CTA walks the chunks of one (sequence, head) unit and keeps the f32
// state in TMEM for the whole sequence: the state never travels through
// HBM between chunks.  Operands are f16 (bf16 inputs convert exactly; f16's
// 11-bit significand keeps the products within the error budget, bf16's
// 8 bits do not), accumulation is f32.
#pragma once

#include <cuda.h>  // CUtensorMap and its enums (types only: the driver entry point is looked up at run time)

#include "common.cuh"
#include "umma.cuh"

namespace m3 {

struct ChunkParams {
  const __nv_bfloat16* x;
  const __nv_bfloat16* B;
  const __nv_bfloat16* dt;
  const __nv_bfloat16* lam;
  const float* A;
  const float* D;
  const int32_t* cu_seqlens;  // NULL: fixed length L per batch row
  float* y;
  float* h;                 // state slots or NULL
  __nv_bfloat16* prev_B;    // carry slots or NULL
  __nv_bfloat16* prev_x;
  int64_t L;
  int H;
};

__host__ __device__ constexpr int align_up(int v, int a) { return (v + a - 1) / a * a; }
__host__ __device__ constexpr int pow2_at_least(int v) {
  return v <= 32 ? 32 : v <= 64 ? 64 : v <= 128 ? 128 : v <= 256 ? 256 : 512;
}

template <int N_, int R_, int Q_>
struct ChunkCfg {
  static constexpr int N = N_, R = R_, Q = Q_, P = 64;
  static constexpr int K2 = N / 2;  // complex pairs
  static constexpr int MR = Q * R;  // rows of S and Y: (token, rank)
  static constexpr int NT = 128;    // threads: one warpgroup
  static_assert(MR == 64 || MR == 128, "Q*R must be 64 or 128");
  static_assert(N == 64 || N == 128, "N must be 64 or 128");
  static_assert(NT % K2 == 0 && Q % (NT / K2) == 0, "angle-scan split");
  // raw TMA stage: x [Q][R*P], B and C [Q][R*N], theta [Q][K2] (bf16)
  static constexpr int XR = Q * R * P * 2, BR = Q * R * N * 2, TR = Q * K2 * 2;
  static constexpr int OFF_XR = 0;
  static constexpr int OFF_BR = align_up(OFF_XR + XR, 1024);
  static constexpr int OFF_CR = align_up(OFF_BR + BR, 1024);
  static constexpr int OFF_TR = align_up(OFF_CR + BR, 1024);
  static constexpr int STAGE = align_up(OFF_TR + TR, 1024);
  static constexpr uint32_t STAGE_TX = XR + 2 * BR + TR;
  // f16 operand tiles, 128B-swizzled, 64-column blocks of [rows x 128 B]
  static constexpr int CT_BYTES = MR * N * 2;   // Ct, Bt: [MR rows][N], K-major for MMA 1
  static constexpr int XT_BYTES = MR * P * 2;   // Xt, WXt: [MR rows][P], MN-major B operands
  static constexpr int ST_BYTES = MR * MR * 2;  // S': [MR rows][MR], K-major A operand
  static constexpr int RT_BYTES = N * P * 2;    // R: [N rows][P], MN-major B operand
  static constexpr int OFF_CT = 2 * STAGE;
  static constexpr int OFF_BT = OFF_CT + CT_BYTES;
  static constexpr int OFF_XT = OFF_BT + CT_BYTES;
  static constexpr int OFF_WXT = OFF_XT + XT_BYTES;
  static constexpr int OFF_ST = OFF_WXT + XT_BYTES;
  static constexpr int OFF_RT = OFF_ST + ST_BYTES;
  static constexpr int SMEM = OFF_RT + RT_BYTES + 1024;  // + alignment slack
  static_assert(SMEM + 4096 <= 232448, "shared memory of one CTA");
  // TMEM columns (f32): S [MR x MR], Y [MR x P], Yi [MR x P], state [N x P]
  static constexpr int COL_S = 0, COL_Y = MR, COL_YI = MR + P, COL_G = MR + 2 * P;
  static constexpr int TMEM_COLS = pow2_at_least(MR + 3 * P);
};

// TMEM lane holding row `row` of an M-row accumulator (M = 64 uses lanes
// 0-15 of each 32-lane quarter; M = 128 uses lane = row).
__device__ __forceinline__ int acc_row_of(int M, int warp, int lane) {
  return M == 128 ? 32 * warp + lane : (lane < 16 ? 16 * warp + lane : -1);
}

__device__ __forceinline__ uint32_t pack_half2(float a, float b) {
  __half2 h = __floats2half2_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float2 bf2_to_f2(uint32_t v) {
  return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
}

constexpr uint32_t kMaxPolls = 1u << 22;

template <int N, int R, int Q>
__global__ void __launch_bounds__(128, 1)
    chunked_prefill_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_B,
                           const __grid_constant__ CUtensorMap tm_C, const __grid_constant__ CUtensorMap tm_th,
                           const ChunkParams p) {
  using Cfg = ChunkCfg<N, R, Q>;
  constexpr int P = Cfg::P, K2 = Cfg::K2, MR = Cfg::MR, NT = Cfg::NT;
  constexpr int G = NT / K2, TPG = Q / G;  // angle scan: G token groups of TPG tokens
  using namespace umma;

  extern __shared__ uint8_t smem_raw[];
  __shared__ __align__(8) uint64_t full_bar[2];
  __shared__ __align__(8) uint64_t mma_bar;
  __shared__ uint32_t tmem_base_s;
  __shared__ float sDt[Q + 1], sBet[Q + 1], sLam[Q], sGam[Q], sWp[Q], sDw[Q], sELam[Q];
  __shared__ float sWarpTot[4];
  __shared__ float sPsum[G][K2];
  __shared__ float2 sEcs[K2];

  uint8_t* sm = smem_raw + ((1024u - (saddr(smem_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  const int unit = blockIdx.x;
  const int H = p.H;
  const int seq = unit / H, head = unit % H;
  int64_t tok0, ntok;
  if (p.cu_seqlens) {
    tok0 = p.cu_seqlens[seq];
    ntok = (int64_t)p.cu_seqlens[seq + 1] - tok0;
  } else {
    tok0 = (int64_t)seq * p.L;
    ntok = p.L;
  }
  if (ntok <= 0) return;  // nothing to do; the state slot keeps its contents
  const int nchunks = (int)((ntok + Q - 1) / Q);
  const float A = p.A[head], Dh = p.D[head];

  uint8_t* Ct = sm + Cfg::OFF_CT;
  uint8_t* Bt = sm + Cfg::OFF_BT;
  uint8_t* Xt = sm + Cfg::OFF_XT;
  uint8_t* WXt = sm + Cfg::OFF_WXT;
  uint8_t* St = sm + Cfg::OFF_ST;
  uint8_t* Rt = sm + Cfg::OFF_RT;

  if (tid == 0) {
    mbar_init(saddr(&full_bar[0]), 1);
    mbar_init(saddr(&full_bar[1]), 1);
    mbar_init(saddr(&mma_bar), 1);
    mbar_init_fence();
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_B);
    tma_prefetch_desc(&tm_C);
    tma_prefetch_desc(&tm_th);
  }
  if (warp == 0) {
    tmem_alloc(saddr(&tmem_base_s), Cfg::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base_s;
  const uint32_t lane_base = (uint32_t)(32 * warp) << 16;

  auto issue_tma = [&](int c) {
    uint8_t* st = sm + (c & 1) * Cfg::STAGE;
    const uint32_t bar = saddr(&full_bar[c & 1]);
    const int t = (int)(tok0 + (int64_t)c * Q);
    mbar_arrive_expect_tx(bar, Cfg::STAGE_TX);
    tma_load_3d(saddr(st + Cfg::OFF_XR), &tm_x, bar, 0, head, t);
    tma_load_3d(saddr(st + Cfg::OFF_BR), &tm_B, bar, 0, head, t);
    tma_load_3d(saddr(st + Cfg::OFF_CR), &tm_C, bar, 0, head, t);
    tma_load_3d(saddr(st + Cfg::OFF_TR), &tm_th, bar, 0, head, t);
  };
  // TMA loads issued into / consumed from each stage (thread 0's count):
  // use u of stage s completes phase u, so its wait parity is u & 1
  int issued[2] = {0, 0}, consumed[2] = {0, 0};
  if (tid == 0) {
    issue_tma(0);
    issued[0] = 1;
    if (nchunks > 1) {
      issue_tma(1);
      issued[1] = 1;
    }
  }

  // ---- initial state: h'_{-1} = h0 + beta'_0 * sum_r Bprev_r xprev_r^T  (realified rows n)
  const int g_row = acc_row_of(N, warp, lane);  // state row owned by this thread (-1: none)
  {
    const float dt0 = __bfloat162float(p.dt[tok0 * H + head]);
    const float lm0 = __bfloat162float(p.lam[tok0 * H + head]);
    const float bet0 = (1.f - lm0) * dt0;
    for (int cb = 0; cb < P; cb += 16) {
      float v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) v[i] = 0.f;
      if (g_row >= 0 && p.h) {
        const int k = g_row >> 1, ri = g_row & 1;
        const float* hs = p.h + ((int64_t)unit * K2 + k) * P * 2;
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = hs[(cb + i) * 2 + ri];
        if (p.prev_B) {
          for (int r = 0; r < R; ++r) {
            const float b = __bfloat162float(p.prev_B[((int64_t)unit * R + r) * N + g_row]);
            const __nv_bfloat16* xp = p.prev_x + ((int64_t)unit * R + r) * P + cb;
#pragma unroll
            for (int i = 0; i < 16; ++i) v[i] = fmaf(bet0 * b, __bfloat162float(xp[i]), v[i]);
          }
        }
      }
      tmem_st16(tmem + lane_base + Cfg::COL_G + cb, v);
    }
    tmem_st_wait();
  }

  bool ok = true;
  uint32_t mma_phase = 0;
  for (int c = 0; c < nchunks && ok; ++c) {
    const int s = c & 1;
    uint8_t* st = sm + s * Cfg::STAGE;
    const int64_t ct0 = tok0 + (int64_t)c * Q;  // first token of the chunk
    const int nvalid = (ntok - (int64_t)c * Q < Q) ? (int)(ntok - (int64_t)c * Q) : Q;

    // ---- per-token scalars: dt, lam (zero past the sequence end), and the next chunk's first token
    if (tid <= Q) {
      const bool valid = tid < nvalid || (tid == Q && (int64_t)c * Q + Q < ntok);
      float d = 0.f, l = 0.f;
      if (valid) {
        d = __bfloat162float(p.dt[(ct0 + tid) * H + head]);
        l = __bfloat162float(p.lam[(ct0 + tid) * H + head]);
      }
      sDt[tid] = d;
      sBet[tid] = (1.f - l) * d;
      if (tid < Q) sGam[tid] = l * d;
    }
    __syncthreads();
    if (tid < Q) {  // inclusive scan of dt*A over the chunk (whole warps)
      float v = sDt[tid] * A;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      if (lane == 31) sWarpTot[warp] = v;
      sLam[tid] = v;
    }
    __syncthreads();
    if (tid < Q) {
      float off = 0.f;
      for (int w = 0; w < warp; ++w) off += sWarpTot[w];
      sLam[tid] += off;
    }
    __syncthreads();
    const float lam_end = sLam[Q - 1];
    if (tid < Q) {
      const float wp = sGam[tid] + sBet[tid + 1];
      sWp[tid] = wp;
      sDw[tid] = __expf(lam_end - sLam[tid]) * wp;
      sELam[tid] = __expf(sLam[tid]);
    }

    // ---- wait for this chunk's inputs
    {
      const bool got = mbar_wait(saddr(&full_bar[s]), (uint32_t)((c >> 1) & 1), kMaxPolls);
      if (!__syncthreads_and(got)) {
        ok = false;
        break;
      }
      if (tid == 0) consumed[s] += 1;
    }
    const __nv_bfloat16* xr = reinterpret_cast<const __nv_bfloat16*>(st + Cfg::OFF_XR);
    const uint32_t* Br = reinterpret_cast<const uint32_t*>(st + Cfg::OFF_BR);
    const uint32_t* Cr = reinterpret_cast<const uint32_t*>(st + Cfg::OFF_CR);
    const __nv_bfloat16* thr = reinterpret_cast<const __nv_bfloat16*>(st + Cfg::OFF_TR);

    // ---- angle scan and rotation of B and C into the f16 operand tiles
    {
      const int k = tid % K2, g = tid / K2;
      float part = 0.f;
      for (int ii = 0; ii < TPG; ++ii) {
        const int i = g * TPG + ii;
        part = fmaf(sDt[i], __bfloat162float(thr[i * K2 + k]), part);
      }
      sPsum[g][k] = part;
      __syncthreads();
      float off = 0.f, tot = 0.f;
#pragma unroll
      for (int gg = 0; gg < G; ++gg) {
        const float v = sPsum[gg][k];
        off += (gg < g) ? v : 0.f;
        tot += v;
      }
      if (g == 0) {
        float sn, cs;
        sincosf(tot, &sn, &cs);
        sEcs[k] = make_float2(cs, sn);
      }
      float phi = off;
      const int blk = (2 * k) / 64, col = (2 * k) % 64;
      for (int ii = 0; ii < TPG; ++ii) {
        const int i = g * TPG + ii;
        phi = fmaf(sDt[i], __bfloat162float(thr[i * K2 + k]), phi);
        float sn, cs;
        sincosf(tot - phi, &sn, &cs);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          const int row = i * R + r;
          const float2 b = bf2_to_f2(Br[row * K2 + k]);
          const float2 cc = bf2_to_f2(Cr[row * K2 + k]);
          const uint32_t off_b = blk * (MR * 128) + sw128_offset(row, col);
          *reinterpret_cast<uint32_t*>(Bt + off_b) = pack_half2(cs * b.x - sn * b.y, sn * b.x + cs * b.y);
          *reinterpret_cast<uint32_t*>(Ct + off_b) = pack_half2(cs * cc.x - sn * cc.y, sn * cc.x + cs * cc.y);
        }
      }
    }
    // ---- X and W X (f16, MN-major [rows j][p])
    for (int idx = tid; idx < MR * (P / 8); idx += NT) {
      const int row = idx / (P / 8), c8 = idx % (P / 8);
      const uint4 raw = *reinterpret_cast<const uint4*>(xr + row * P + c8 * 8);
      const float w = sDw[row / R];
      const uint32_t rw[4] = {raw.x, raw.y, raw.z, raw.w};
      uint32_t hx[4], hw[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 f = bf2_to_f2(rw[q]);
        hx[q] = pack_half2(f.x, f.y);
        hw[q] = pack_half2(w * f.x, w * f.y);
      }
      const uint32_t o = sw128_offset(row, c8 * 8);
      *reinterpret_cast<uint4*>(Xt + o) = make_uint4(hx[0], hx[1], hx[2], hx[3]);
      *reinterpret_cast<uint4*>(WXt + o) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    }
    fence_async_smem();
    __syncthreads();
    // the raw stage is consumed: prefetch chunk c + 2 into it
    if (tid == 0 && c + 2 < nchunks) {
      issue_tma(c + 2);
      issued[s] += 1;
    }

    // ---- MMA 1: S = Ct Bt^T  (M = MR, N = MR, K = N)
    if (tid == 0) {
      tc_fence_after();
      constexpr uint32_t idesc = idesc_f16_f32(MR, MR, 0, 0);
#pragma unroll
      for (int ks = 0; ks < N / 16; ++ks) {
        const uint32_t koff = (ks / 4) * (MR * 128) + (ks % 4) * 32;
        mma_f16(tmem + Cfg::COL_S, smem_desc(saddr(Ct) + koff, 16, 1024, kSwizzle128B),
                smem_desc(saddr(Bt) + koff, 16, 1024, kSwizzle128B), idesc, ks > 0);
      }
      mma_commit(saddr(&mma_bar));
    }
    {
      const bool got = mbar_wait(saddr(&mma_bar), mma_phase, kMaxPolls);
      mma_phase ^= 1;
      if (!__syncthreads_and(got)) {
        ok = false;
        break;
      }
    }
    tc_fence_after();

    // ---- S -> S' (causal mask, decay, trapezoid weights), f16, K-major [rows t][cols j]
    {
      const int t = acc_row_of(MR, warp, lane);
      const int it = t >= 0 ? t / R : 0;
      const float lam_t = sLam[it], gam_t = sGam[it];
      for (int cb = 0; cb < MR; cb += 16) {
        float v[16];
        tmem_ld16(tmem + lane_base + Cfg::COL_S + cb, v);
        tmem_ld_wait();
        if (t >= 0) {
          uint32_t hv[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            float e[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int j = cb + 2 * q + u, jt = j / R;
              const float w = (jt == it) ? gam_t : sWp[jt];
              e[u] = (jt <= it) ? v[2 * q + u] * __expf(lam_t - sLam[jt]) * w : 0.f;
            }
            hv[q] = pack_half2(e[0], e[1]);
          }
#pragma unroll
          for (int hlf = 0; hlf < 2; ++hlf) {
            const int j = cb + 8 * hlf;
            const uint32_t o = (j / 64) * (MR * 128) + sw128_offset(t, j % 64);
            *reinterpret_cast<uint4*>(St + o) = make_uint4(hv[4 * hlf], hv[4 * hlf + 1], hv[4 * hlf + 2], hv[4 * hlf + 3]);
          }
        }
      }
    }

    // ---- state step: R = e^{i phi_end} h' (f16 operand), TMEM state <- e^{Lam_end} R
    {
      const float elam_end = __expf(lam_end);
      const int n = g_row;
      const float2 ecs = sEcs[n >= 0 ? (n >> 1) : 0];
      const bool re = (n & 1) == 0;
      for (int cb = 0; cb < P; cb += 16) {
        float v[16];
        tmem_ld16(tmem + lane_base + Cfg::COL_G + cb, v);
        tmem_ld_wait();
        float r[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const float other = __shfl_xor_sync(0xffffffffu, v[i], 1);
          r[i] = re ? (ecs.x * v[i] - ecs.y * other) : (ecs.y * other + ecs.x * v[i]);
        }
        if (n >= 0) {
#pragma unroll
          for (int hlf = 0; hlf < 2; ++hlf) {
            const int pc = cb + 8 * hlf;
            const uint32_t o = sw128_offset(n, pc);
            *reinterpret_cast<uint4*>(Rt + o) =
                make_uint4(pack_half2(r[8 * hlf], r[8 * hlf + 1]), pack_half2(r[8 * hlf + 2], r[8 * hlf + 3]),
                           pack_half2(r[8 * hlf + 4], r[8 * hlf + 5]), pack_half2(r[8 * hlf + 6], r[8 * hlf + 7]));
          }
        }
#pragma unroll
        for (int i = 0; i < 16; ++i) r[i] *= elam_end;
        tmem_st16(tmem + lane_base + Cfg::COL_G + cb, r);
      }
      tmem_st_wait();
    }
    fence_async_smem();
    tc_fence_before();
    __syncthreads();

    // ---- MMA 2 (Y = S' X), MMA 3 (Yi = Ct R), MMA 4 (state += Bt^T W X)
    if (tid == 0) {
      tc_fence_after();
      {
        constexpr uint32_t idesc = idesc_f16_f32(MR, P, 0, 1);
#pragma unroll
        for (int ks = 0; ks < MR / 16; ++ks) {
          const uint32_t aoff = (ks / 4) * (MR * 128) + (ks % 4) * 32;
          mma_f16(tmem + Cfg::COL_Y, smem_desc(saddr(St) + aoff, 16, 1024, kSwizzle128B),
                  smem_desc(saddr(Xt) + ks * 2048, MR * 128, 1024, kSwizzle128B), idesc, ks > 0);
        }
      }
      {
        constexpr uint32_t idesc = idesc_f16_f32(MR, P, 0, 1);
#pragma unroll
        for (int ks = 0; ks < N / 16; ++ks) {
          const uint32_t aoff = (ks / 4) * (MR * 128) + (ks % 4) * 32;
          mma_f16(tmem + Cfg::COL_YI, smem_desc(saddr(Ct) + aoff, 16, 1024, kSwizzle128B),
                  smem_desc(saddr(Rt) + ks * 2048, N * 128, 1024, kSwizzle128B), idesc, ks > 0);
        }
      }
      {
        constexpr uint32_t idesc = idesc_f16_f32(N, P, 1, 1);
#pragma unroll
        for (int ks = 0; ks < MR / 16; ++ks) {
          mma_f16(tmem + Cfg::COL_G, smem_desc(saddr(Bt) + ks * 2048, MR * 128, 1024, kSwizzle128B),
                  smem_desc(saddr(WXt) + ks * 2048, MR * 128, 1024, kSwizzle128B), idesc, 1);
        }
      }
      mma_commit(saddr(&mma_bar));
    }
    {
      const bool got = mbar_wait(saddr(&mma_bar), mma_phase, kMaxPolls);
      mma_phase ^= 1;
      if (!__syncthreads_and(got)) {
        ok = false;
        break;
      }
    }
    tc_fence_after();

    // ---- output: y = Y + e^{Lam_t} Yi + D x
    {
      const int t = acc_row_of(MR, warp, lane);
      const int it = t >= 0 ? t / R : 0, rk = t >= 0 ? t % R : 0;
      const bool valid = t >= 0 && it < nvalid;
      const float el = sELam[it];
      float* yrow = p.y + ((ct0 + it) * H + head) * (R * P) + rk * P;
      for (int cb = 0; cb < P; cb += 16) {
        float a[16], b[16];
        tmem_ld16(tmem + lane_base + Cfg::COL_Y + cb, a);
        tmem_ld16(tmem + lane_base + Cfg::COL_YI + cb, b);
        tmem_ld_wait();
        if (valid) {
          float o[16];
#pragma unroll
          for (int hlf = 0; hlf < 2; ++hlf) {
            const uint4 xv = *reinterpret_cast<const uint4*>(Xt + sw128_offset(t, cb + 8 * hlf));
            const uint32_t xs[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&xs[q]));
              const int i0 = 8 * hlf + 2 * q;
              o[i0] = fmaf(Dh, f.x, fmaf(el, b[i0], a[i0]));
              o[i0 + 1] = fmaf(Dh, f.y, fmaf(el, b[i0 + 1], a[i0 + 1]));
            }
          }
#pragma unroll
          for (int q = 0; q < 4; ++q)
            *reinterpret_cast<float4*>(yrow + cb + 4 * q) = make_float4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        }
      }
    }
    tc_fence_before();
    __syncthreads();
  }

  if (ok) {
    tc_fence_after();
    // ---- final state (h of the last token) and carry (the last token's B and x)
    if (p.h) {
      const int n = g_row;
      for (int cb = 0; cb < P; cb += 16) {
        float v[16];
        tmem_ld16(tmem + lane_base + Cfg::COL_G + cb, v);
        tmem_ld_wait();
        if (n >= 0) {
          float* hs = p.h + ((int64_t)unit * K2 + (n >> 1)) * P * 2 + (n & 1);
#pragma unroll
          for (int i = 0; i < 16; ++i) hs[(cb + i) * 2] = v[i];
        }
      }
    }
    if (p.prev_B) {
      const int64_t last = (tok0 + ntok - 1) * H + head;
      for (int i = tid; i < R * N; i += NT) p.prev_B[(int64_t)unit * R * N + i] = p.B[last * R * N + i];
      for (int i = tid; i < R * P; i += NT) p.prev_x[(int64_t)unit * R * P + i] = p.x[last * R * P + i];
    }
  } else {
    if (tid == 0) {
      atomicExch(&g_status, (int)M3_ERR_TIMEOUT);
      // let loads still in flight land before the shared memory goes away
      for (int s2 = 0; s2 < 2; ++s2)
        if (issued[s2] > consumed[s2]) mbar_wait(saddr(&full_bar[s2]), (uint32_t)((issued[s2] - 1) & 1), kMaxPolls);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, Cfg::TMEM_COLS);
}

// ------------------------------------------------------------------ host side

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline PFN_encodeTiled get_encode_tiled() {
  static PFN_encodeTiled fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_encodeTiled>(ptr);
  }
  return fn;
}

// 3-D bf16 tensor [T][H][inner] (inner contiguous), box [Q][1][inner].
inline bool make_map_3d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t H, uint64_t T, uint32_t Q) {
  PFN_encodeTiled enc = get_encode_tiled();
  if (!enc) return false;
  cuuint64_t dims[3] = {inner, H, T};
  cuuint64_t strides[2] = {inner * 2, inner * H * 2};
  cuuint32_t box[3] = {(cuuint32_t)inner, 1, Q};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int N, int R, int Q>
m3_status chunked_launch(const m3_prefill_args* a, float* h, void* prev_B, void* prev_x, int nseq, cudaStream_t s) {
  using Cfg = ChunkCfg<N, R, Q>;
  const int H = a->dims.nheads;
  const uint64_t T = (uint64_t)a->seqlen * (a->cu_seqlens ? 1 : a->dims.batch);
  CUtensorMap mx, mB, mC, mth;
  if (!make_map_3d(&mx, a->x, (uint64_t)R * 64, H, T, Q) || !make_map_3d(&mB, a->B, (uint64_t)R * N, H, T, Q) ||
      !make_map_3d(&mC, a->C, (uint64_t)R * N, H, T, Q) || !make_map_3d(&mth, a->theta, N / 2, H, T, Q))
    return M3_ERR_CUDA;
  ChunkParams p{};
  p.x = static_cast<const __nv_bfloat16*>(a->x);
  p.B = static_cast<const __nv_bfloat16*>(a->B);
  p.dt = static_cast<const __nv_bfloat16*>(a->dt);
  p.lam = static_cast<const __nv_bfloat16*>(a->lam);
  p.A = a->A;
  p.D = a->D;
  p.cu_seqlens = a->cu_seqlens;
  p.y = a->y;
  p.h = h;
  p.prev_B = static_cast<__nv_bfloat16*>(prev_B);
  p.prev_x = static_cast<__nv_bfloat16*>(prev_x);
  p.L = a->seqlen;
  p.H = H;
  auto kern = chunked_prefill_kernel<N, R, Q>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::SMEM) != cudaSuccess)
    return M3_ERR_CUDA;
  const int units = nseq * H;
  kern<<<units, Cfg::NT, Cfg::SMEM, s>>>(mx, mB, mC, mth, p);
  return cudaGetLastError() == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

// Shapes with a chunked kernel: bf16 inputs, P = 64, and (N, R, chunk) in
// {(128, 1, 64), (64, 1, 64), (64, 4, 32), (64, 2, 32), (128, 2, 32)}.
inline m3_status chunked_prefill(const m3_prefill_args* a, float* h, void* prev_B, void* prev_x, int nseq,
                                 cudaStream_t s) {
  const m3_dims& d = a->dims;
  if (d.in_dtype != M3_BF16 || d.headdim != 64) return M3_ERR_UNSUPPORTED;
  const int R = d.rank, N = d.dstate;
  const int Q = a->chunk > 0 ? a->chunk : (R == 1 ? 64 : 32);
#define M3_CH(NN, RR, QQ) \
  if (N == NN && R == RR && Q == QQ) return chunked_launch<NN, RR, QQ>(a, h, prev_B, prev_x, nseq, s);
  M3_CH(128, 1, 64)
  M3_CH(64, 1, 64)
  M3_CH(64, 4, 32)
  M3_CH(64, 2, 32)
  M3_CH(128, 2, 32)
#undef M3_CH
  return M3_ERR_UNSUPPORTED;
}

}  // namespace m3
