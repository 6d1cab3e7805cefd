// C-ABI entry point of the backward pass (declared in m3scan_backward.h):
// argument checks, scratch, the fused prologue's passes and the launches of
// the chunked or the token-serial adjoint kernels.
#include <cuda_runtime.h>

#include "backward.cuh"
#include "bwd_chunked.cuh"
#include "m3scan_backward.h"

namespace m3 {
int* device_status_word();  // (m3scan.cu)
}

namespace m3bwd {

// ------------------------------------------------------------------ prologue passes

constexpr float kBcNormEps = 1e-6f;

__device__ __forceinline__ float softplus_f(float z) { return fmaxf(z, 0.f) + log1pf(expf(-fabsf(z))); }
__device__ __forceinline__ float sigmoid_f(float z) { return 0.5f * (1.f + tanhf(0.5f * z)); }

template <typename T>
__global__ void to_f32_kernel(const T* src, float* dst, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = to_f(src[i]);
}

// dt as the scan sees it: softplus(dt + dt_bias[h]) (heads innermost) or the raw value
template <typename T>
__global__ void dt_prologue_kernel(const T* dt, const float* bias, int H, int softplus, float* dst, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) {
    const float z = to_f(dt[i]);
    dst[i] = softplus ? softplus_f(z + (bias ? bias[i % H] : 0.f)) : z;
  }
}

// rows of N values divided by their RMS (norm) or copied; one warp per row
template <typename T>
__global__ void rows_prologue_kernel(const T* src, float* dst, int64_t rows, int N, int norm) {
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const T* v = src + row * N;
  float sc = 1.f;
  if (norm) {
    float ss = 0.f;
    for (int i = lane; i < N; i += 32) ss = fmaf(to_f(v[i]), to_f(v[i]), ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    sc = rsqrtf(ss / (float)N + kBcNormEps);
  }
  for (int i = lane; i < N; i += 32) dst[row * N + i] = sc * to_f(v[i]);
}

// ddt of the raw pre-activation: ddt * sigmoid(dt + dt_bias[h]), in place
template <typename T>
__global__ void dt_grad_kernel(const T* dt, const float* bias, int H, float* ddt, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    ddt[i] *= sigmoid_f(to_f(dt[i]) + (bias ? bias[i % H] : 0.f));
}

// gradient through n = v / sqrt(mean(v^2) + eps), in place on g (one warp
// per row): dv = s (dn - n mean(dn * n))
template <typename T>
__global__ void rows_norm_grad_kernel(const T* src, float* g, int64_t rows, int N) {
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) / 32;
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const T* v = src + row * N;
  float* d = g + row * N;
  float ss = 0.f;
  for (int i = lane; i < N; i += 32) ss = fmaf(to_f(v[i]), to_f(v[i]), ss);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float sc = rsqrtf(ss / (float)N + kBcNormEps);
  float dn = 0.f;
  for (int i = lane; i < N; i += 32) dn = fmaf(d[i], sc * to_f(v[i]), dn);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) dn += __shfl_xor_sync(0xffffffffu, dn, o);
  const float mean = dn / (float)N;
  for (int i = lane; i < N; i += 32) d[i] = sc * (d[i] - sc * to_f(v[i]) * mean);
}

// dL/d dt_bias[h] = sum over rows of the (raw) ddt; one CTA per head, in order
__global__ void __launch_bounds__(256) bias_grad_kernel(const float* ddt, int64_t rows, int H, float* out) {
  __shared__ float sa[256];
  const int head = blockIdx.x, tid = threadIdx.x;
  float a = 0.f;
  for (int64_t r = tid; r < rows; r += blockDim.x) a += ddt[r * H + head];
  sa[tid] = a;
  __syncthreads();
  for (int w = blockDim.x / 2; w > 0; w >>= 1) {
    if (tid < w) sa[tid] += sa[tid + w];
    __syncthreads();
  }
  if (tid == 0) out[head] = sa[0];
}

}  // namespace m3bwd

namespace {

using namespace m3bwd;

bool bwd_dims_ok(const m3_dims* d) {
  return d && d->batch > 0 && d->nheads > 0 && d->headdim > 0 && d->dstate > 0 && d->dstate % 2 == 0 &&
         d->rank > 0 && d->rank <= 8 && (d->in_dtype == M3_F32 || d->in_dtype == M3_BF16);
}

unsigned grid_for(int64_t n, int threads = 256) {
  const int64_t b = (n + threads - 1) / threads;
  return (unsigned)(b < 148 * 32 ? (b > 0 ? b : 1) : 148 * 32);
}

// the token-serial kernel (any shape)
m3_status serial_backward(const m3_backward_args* a, const void* const in[8], bool f32, int G, cudaStream_t s) {
  const int H = a->dims.nheads;
  const int P = a->dims.headdim, N = a->dims.dstate, K = N / 2, R = a->dims.rank;
  const size_t units = (size_t)a->dims.batch * H;
  const size_t KP = (size_t)K * P;
  const size_t hist_bytes = units * (size_t)a->seqlen * KP * sizeof(float2);
  const size_t gs_bytes = units * KP * sizeof(float2);
  if (hist_bytes + gs_bytes > (size_t(4) << 30)) return M3_ERR_UNSUPPORTED;
  // x, x_prev, dy, dx rows; Bhat, Bhat_prev, Chat, dB, dC rows; a and the sums over p per pair; scalars
  const size_t smem = sizeof(float) * 4 * R * P + sizeof(float2) * (5 * (size_t)R * K + 2 * (size_t)K) + 16;
  if (smem > 200 * 1024) return M3_ERR_UNSUPPORTED;
  auto kern = f32 ? m3bwd::backward_kernel<float> : m3bwd::backward_kernel<__nv_bfloat16>;
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return M3_ERR_CUDA;
  const size_t bc_bytes = (size_t)a->dims.batch * a->seqlen * G * R * N * sizeof(float);
  void* buf = nullptr;
  if (cudaMallocAsync(&buf, hist_bytes + gs_bytes, s) != cudaSuccess) {
    cudaGetLastError();
    return M3_ERR_ALLOC;
  }
  m3bwd::BackwardParams p{};
  p.x = in[0]; p.B = in[1]; p.C = in[2]; p.dt = in[3]; p.lam = in[4]; p.theta = in[5];
  p.A = a->A; p.D = a->D; p.h0 = a->h0; p.prev_B = in[6]; p.prev_x = a->prev_x;
  if (in[7]) p.prev_x = in[7];
  p.dy = a->dy; p.dh_final = a->dh_final;
  p.dx = a->dx; p.dB = a->dB; p.dC = a->dC; p.ddt = a->ddt; p.dlam = a->dlam; p.dtheta = a->dtheta;
  p.dA = a->dA; p.dD = a->dD; p.dh0 = a->dh0; p.dprev_B = a->dprev_B; p.dprev_x = a->dprev_x;
  p.hist = static_cast<float2*>(buf);
  p.gs = reinterpret_cast<float2*>(static_cast<unsigned char*>(buf) + hist_bytes);
  p.L = a->seqlen;
  p.H = H; p.P = P; p.N = N; p.K = K; p.R = R; p.G = G;
  cudaError_t e = cudaMemsetAsync(a->dB, 0, bc_bytes, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(a->dC, 0, bc_bytes, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(a->dA, 0, H * sizeof(float), s);
  if (e == cudaSuccess) e = cudaMemsetAsync(a->dD, 0, H * sizeof(float), s);
  if (e == cudaSuccess) {
    kern<<<(unsigned)units, 256, smem, s>>>(p);
    e = cudaGetLastError();
  }
  const cudaError_t ef = cudaFreeAsync(buf, s);
  return (e == cudaSuccess && ef == cudaSuccess) ? M3_OK : M3_ERR_CUDA;
}

// the chunked kernels for one shape
template <typename T, int NN, int RR>
m3_status chunked_go(const m3_backward_args* a, const void* const in[8], int G, cudaStream_t s) {
  using Cfg = BwdCfg<NN, RR>;
  constexpr int MR = Cfg::MR, NS = Cfg::NS, PS = Cfg::PS, MS = Cfg::MS, Q = Cfg::Q, K = Cfg::K, P = Cfg::P;
  const int H = a->dims.nheads;
  const int64_t L = a->seqlen;
  const int nch = (int)((L + Q - 1) / Q);
  const size_t units = (size_t)a->dims.batch * H;
  const size_t KP = (size_t)K * P;
  const size_t blk = units * nch * KP * sizeof(float2);
  const bool grouped = G != H;
  const size_t bc_head = grouped ? (size_t)a->dims.batch * L * H * RR * NN * sizeof(float) : 0;
  size_t off[12];
  size_t tot = 0;
  auto take = [&](int i, size_t bytes) {
    off[i] = tot;
    tot += (bytes + 255) / 256 * 256;
  };
  take(0, blk);                                   // Zs
  take(1, blk);                                   // Us
  take(2, units * (nch + 1) * KP * sizeof(float2));  // Hs
  take(3, blk);                                   // dHe
  take(4, units * KP * sizeof(float2));           // dHs0
  take(5, units * nch * K * sizeof(float2));      // alpha
  take(6, units * nch * sizeof(float));           // dwp_last
  take(7, units * nch * sizeof(float));           // dA_part
  take(8, units * nch * sizeof(float));           // dD_part
  take(9, bc_head);                               // per-head dB
  take(10, bc_head);                              // per-head dC
  if (tot > (size_t(16) << 30)) return M3_ERR_UNSUPPORTED;
  // chunk sums on the tensor cores; with rank 4 (16-token chunks, four
  // times as many) the f32 kernel, whose fixed cost per chunk is lower
  // (TMEM allocation, the MMA round trip), measured faster
  constexpr bool kSumsTc = RR < 4;
  const size_t smem1 = kSumsTc ? (size_t)SumsTcLayout<NN, MR>::SMEM
                               : sizeof(float) * (2 * MR * NS + 2 * MR * PS);  // (the angles share the dy tile)
  const size_t smem3 = sizeof(float) * (2 * MR * NS + 2 * MR * PS + 2 * NN * PS + 2 * MR * MS + Q * K);
  auto k1 = kSumsTc ? chunk_sums_tc_kernel<T, NN, RR> : chunk_sums_kernel<T, NN, RR>;
  auto k3 = chunk_grads_kernel<T, NN, RR>;
  if (cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1) != cudaSuccess ||
      cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem3) != cudaSuccess)
    return M3_ERR_CUDA;
  void* buf = nullptr;
  if (cudaMallocAsync(&buf, tot, s) != cudaSuccess) {
    cudaGetLastError();
    return M3_ERR_ALLOC;
  }
  auto at = [&](int i) { return static_cast<void*>(static_cast<unsigned char*>(buf) + off[i]); };
  ChunkBwdParams p{};
  p.x = in[0]; p.B = in[1]; p.C = in[2]; p.dt = in[3]; p.lam = in[4]; p.theta = in[5];
  p.A = a->A; p.D = a->D; p.h0 = a->h0; p.prev_B = in[6]; p.prev_x = in[7] ? in[7] : a->prev_x;
  p.dy = a->dy; p.dh_final = a->dh_final;
  p.dx = a->dx;
  p.dB = grouped ? static_cast<float*>(at(9)) : a->dB;
  p.dC = grouped ? static_cast<float*>(at(10)) : a->dC;
  p.ddt = a->ddt; p.dlam = a->dlam; p.dtheta = a->dtheta;
  p.dh0 = a->dh0; p.dprev_B = a->dprev_B; p.dprev_x = a->dprev_x;
  p.Zs = static_cast<float2*>(at(0));
  p.Us = static_cast<float2*>(at(1));
  p.Hs = static_cast<float2*>(at(2));
  p.dHe = static_cast<float2*>(at(3));
  p.dHs0 = static_cast<float2*>(at(4));
  p.alpha = static_cast<float2*>(at(5));
  p.dwp_last = static_cast<float*>(at(6));
  p.dA_part = static_cast<float*>(at(7));
  p.dD_part = static_cast<float*>(at(8));
  p.L = L; p.nch = nch; p.H = H; p.G = G; p.GB = H;
  p.status = m3::device_status_word();
  if (!p.status) {
    cudaFreeAsync(buf, s);
    return M3_ERR_CUDA;
  }
  const unsigned chunks = (unsigned)(units * nch);
  k1<<<chunks, Cfg::NT, smem1, s>>>(p);
  const unsigned bpu = (unsigned)((KP + 255) / 256);
  chunk_scan_kernel<T><<<(unsigned)(units * bpu), 256, 0, s>>>(p, RR, NN, P);
  k3<<<chunks, Cfg::NTG, smem3, s>>>(p);
  unit_final_kernel<T><<<(unsigned)units, 256, 0, s>>>(p, RR, NN, P, Q);
  head_sums_kernel<<<H, 256, 0, s>>>(p.dA_part, p.dD_part, a->dims.batch, H, nch, a->dA, a->dD);
  if (grouped) {
    const int64_t rows_bl = (int64_t)a->dims.batch * L;
    const int64_t n = rows_bl * G * RR * NN;
    group_sum_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(p.dB, a->dB, rows_bl, H, G, RR * NN);
    group_sum_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(p.dC, a->dC, rows_bl, H, G, RR * NN);
  }
  cudaError_t e = cudaGetLastError();
  const cudaError_t ef = cudaFreeAsync(buf, s);
  return (e == cudaSuccess && ef == cudaSuccess) ? M3_OK : M3_ERR_CUDA;
}

template <typename T>
m3_status chunked_backward(const m3_backward_args* a, const void* const in[8], int G, cudaStream_t s) {
  const int N = a->dims.dstate, R = a->dims.rank;
#define M3_BW(NN, RR) \
  if (N == NN && R == RR) return chunked_go<T, NN, RR>(a, in, G, s);
  M3_BW(128, 1)
  M3_BW(64, 1)
  M3_BW(64, 4)
  M3_BW(64, 2)
  M3_BW(128, 2)
#undef M3_BW
  return M3_ERR_UNSUPPORTED;
}

bool chunked_shape(const m3_backward_args* a) {
  const int N = a->dims.dstate, R = a->dims.rank;
  const bool nr = (R == 1 && (N == 64 || N == 128)) || (R == 2 && (N == 64 || N == 128)) || (R == 4 && N == 64);
  return a->dims.headdim == 64 && nr && (a->chunk == 0 || a->chunk == 64 / R);
}

}  // namespace

extern "C" {

M3_API m3_status m3_scan_prefill_backward(const m3_backward_args* a, void* stream) {
  if (!a || !bwd_dims_ok(&a->dims) || a->seqlen < 1) return M3_ERR_INVALID_ARG;
  if (!a->x || !a->B || !a->C || !a->dt || !a->A || !a->D || !a->dy || !a->dx || !a->dB || !a->dC ||
      !a->ddt || !a->dA || !a->dD)
    return M3_ERR_INVALID_ARG;
  const int H = a->dims.nheads;
  if (a->ngroups < 0 || (a->ngroups > 0 && H % a->ngroups != 0)) return M3_ERR_INVALID_ARG;
  if (a->algo < M3_ALGO_AUTO || a->algo > M3_ALGO_CHUNKED || a->chunk < 0) return M3_ERR_INVALID_ARG;
  if (a->prologue & ~(M3_PRO_DT_SOFTPLUS | M3_PRO_BC_NORM)) return M3_ERR_INVALID_ARG;
  const int G = a->ngroups > 0 ? a->ngroups : H;
  const bool chunked = a->algo != M3_ALGO_RECURRENT && chunked_shape(a);
  if (a->algo == M3_ALGO_CHUNKED && !chunked) return M3_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf16 = a->dims.in_dtype == M3_BF16;
  const int P = a->dims.headdim, N = a->dims.dstate, R = a->dims.rank;
  const int64_t L = a->seqlen, tok = (int64_t)a->dims.batch * L, units = (int64_t)a->dims.batch * H;
  const void* in[8] = {a->x, a->B, a->C, a->dt, a->lam, a->theta, a->prev_B, nullptr};

  // The fused prologue: the kernels run on f32 copies of the inputs as the
  // scan sees them (softplus of dt, normalised B / C / carried B rows), and
  // the gradients are chained back to the raw inputs afterwards.
  void* pbuf = nullptr;
  if (a->prologue) {
    const int64_t nx = tok * H * R * P, nbc = tok * G * R * N, ns = tok * H, nth = tok * H * (N / 2);
    const int64_t npb = units * R * N, npx = units * R * P;
    const int64_t nf = nx + 2 * nbc + 2 * ns + nth + npb + npx;
    if (cudaMallocAsync(&pbuf, (size_t)nf * sizeof(float), s) != cudaSuccess) {
      cudaGetLastError();
      return M3_ERR_ALLOC;
    }
    float* f = static_cast<float*>(pbuf);
    float *fx = f, *fB = fx + nx, *fC = fB + nbc, *fdt = fC + nbc, *flam = fdt + ns, *fth = flam + ns;
    float *fpB = fth + nth, *fpx = fpB + npb;
    const int norm = (a->prologue & M3_PRO_BC_NORM) != 0, sp = (a->prologue & M3_PRO_DT_SOFTPLUS) != 0;
    auto go = [&](auto tag) {
      using T = decltype(tag);
      to_f32_kernel<T><<<grid_for(nx), 256, 0, s>>>(static_cast<const T*>(a->x), fx, nx);
      rows_prologue_kernel<T><<<grid_for(nbc / N * 32), 256, 0, s>>>(static_cast<const T*>(a->B), fB, nbc / N, N, norm);
      rows_prologue_kernel<T><<<grid_for(nbc / N * 32), 256, 0, s>>>(static_cast<const T*>(a->C), fC, nbc / N, N, norm);
      dt_prologue_kernel<T><<<grid_for(ns), 256, 0, s>>>(static_cast<const T*>(a->dt), a->dt_bias, H, sp, fdt, ns);
      if (a->lam) to_f32_kernel<T><<<grid_for(ns), 256, 0, s>>>(static_cast<const T*>(a->lam), flam, ns);
      if (a->theta) to_f32_kernel<T><<<grid_for(nth), 256, 0, s>>>(static_cast<const T*>(a->theta), fth, nth);
      if (a->prev_B)
        rows_prologue_kernel<T><<<grid_for(npb / N * 32), 256, 0, s>>>(static_cast<const T*>(a->prev_B), fpB,
                                                                        npb / N, N, norm);
      if (a->prev_x) to_f32_kernel<T><<<grid_for(npx), 256, 0, s>>>(static_cast<const T*>(a->prev_x), fpx, npx);
    };
    if (bf16)
      go(__nv_bfloat16{});
    else
      go(float{});
    in[0] = fx; in[1] = fB; in[2] = fC; in[3] = fdt;
    in[4] = a->lam ? flam : nullptr;
    in[5] = a->theta ? fth : nullptr;
    in[6] = a->prev_B ? fpB : nullptr;
    in[7] = a->prev_x ? fpx : nullptr;
  }
  const bool f32_in = a->prologue != 0 || !bf16;
  m3_status rc;
  if (chunked)
    rc = f32_in ? chunked_backward<float>(a, in, G, s) : chunked_backward<__nv_bfloat16>(a, in, G, s);
  else
    rc = serial_backward(a, in, f32_in, G, s);
  if (rc == M3_OK && a->prologue) {
    // chain back to the raw inputs
    auto go = [&](auto tag) {
      using T = decltype(tag);
      const int64_t ns = tok * H, nbc_rows = tok * G * R;
      if (a->prologue & M3_PRO_DT_SOFTPLUS) {
        dt_grad_kernel<T><<<grid_for(ns), 256, 0, s>>>(static_cast<const T*>(a->dt), a->dt_bias, H, a->ddt, ns);
        if (a->ddt_bias) bias_grad_kernel<<<H, 256, 0, s>>>(a->ddt, tok, H, a->ddt_bias);
      }
      if (a->prologue & M3_PRO_BC_NORM) {
        rows_norm_grad_kernel<T><<<grid_for(nbc_rows * 32), 256, 0, s>>>(static_cast<const T*>(a->B), a->dB, nbc_rows, N);
        rows_norm_grad_kernel<T><<<grid_for(nbc_rows * 32), 256, 0, s>>>(static_cast<const T*>(a->C), a->dC, nbc_rows, N);
        if (a->prev_B && a->dprev_B)
          rows_norm_grad_kernel<T><<<grid_for(units * R * 32), 256, 0, s>>>(static_cast<const T*>(a->prev_B),
                                                                            a->dprev_B, units * R, N);
      }
    };
    if (bf16)
      go(__nv_bfloat16{});
    else
      go(float{});
    if (cudaGetLastError() != cudaSuccess) rc = M3_ERR_CUDA;
  }
  if (!(a->prologue & M3_PRO_DT_SOFTPLUS) && a->ddt_bias && rc == M3_OK) {
    if (cudaMemsetAsync(a->ddt_bias, 0, H * sizeof(float), s) != cudaSuccess) rc = M3_ERR_CUDA;
  }
  if (pbuf && cudaFreeAsync(pbuf, s) != cudaSuccess) rc = M3_ERR_CUDA;
  return rc;
}

}  // extern "C"
