// C-ABI entry point of the backward pass (declared in m3scan_backward.h):
// argument checks, the scratch for the forward history, the zeroing of the
// accumulated outputs and the launch of the token-serial adjoint kernel.
#include <cuda_runtime.h>

#include "backward.cuh"
#include "m3scan_backward.h"

namespace {

bool bwd_dims_ok(const m3_dims* d) {
  return d && d->batch > 0 && d->nheads > 0 && d->headdim > 0 && d->dstate > 0 && d->dstate % 2 == 0 &&
         d->rank > 0 && d->rank <= 8 && (d->in_dtype == M3_F32 || d->in_dtype == M3_BF16);
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
  const int G = a->ngroups > 0 ? a->ngroups : H;
  const int P = a->dims.headdim, N = a->dims.dstate, K = N / 2, R = a->dims.rank;
  const size_t units = (size_t)a->dims.batch * H;
  const size_t KP = (size_t)K * P;
  const size_t hist_bytes = units * (size_t)a->seqlen * KP * sizeof(float2);
  const size_t gs_bytes = units * KP * sizeof(float2);
  if (hist_bytes + gs_bytes > (size_t(4) << 30)) return M3_ERR_UNSUPPORTED;
  // x, x_prev, dy, dx rows; Bhat, Bhat_prev, Chat, dB, dC rows; a and the sums over p per pair; scalars
  const size_t smem = sizeof(float) * 4 * R * P + sizeof(float2) * (5 * (size_t)R * K + 2 * (size_t)K) + 16;
  if (smem > 200 * 1024) return M3_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool bf16 = a->dims.in_dtype == M3_BF16;
  auto kern = bf16 ? m3bwd::backward_kernel<__nv_bfloat16> : m3bwd::backward_kernel<float>;
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
  p.x = a->x; p.B = a->B; p.C = a->C; p.dt = a->dt; p.lam = a->lam; p.theta = a->theta;
  p.A = a->A; p.D = a->D; p.h0 = a->h0; p.prev_B = a->prev_B; p.prev_x = a->prev_x;
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

}  // extern "C"
