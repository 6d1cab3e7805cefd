// Shared device helpers of the m3scan kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "m3scan.h"
#include "m3scan_testing.h"

namespace m3 {

// Library-wide device status word: kernels that give up a bounded wait store
// an m3_status here; m3_device_status() reads and clears it.  (The library is
// one translation unit, m3scan.cu, so this is its only definition.)
__device__ int g_status = 0;

__device__ __forceinline__ float to_f(float v) { return v; }
__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T>
__device__ __forceinline__ float ldf(const T* p, int64_t i) {
  return to_f(p[i]);
}

// Streaming 16-byte state accesses: the state is touched once per step.
__device__ __forceinline__ float4 ld_stream(const float4* p) { return __ldcs(p); }
__device__ __forceinline__ void st_stream(float4* p, float4 v) { __stcs(p, v); }

// Fused prologue: softplus(z) = log(1 + e^z), written as max(z, 0) +
// log1p(e^-|z|) (no overflow, no cancellation), and the epsilon of the RMS
// norm of B and C rows.
__device__ __forceinline__ float softplus_f(float z) { return fmaxf(z, 0.f) + log1pf(expf(-fabsf(z))); }
constexpr float kBcNormEps = 1e-6f;

// dt of head `head` as the scan uses it: the raw value, or softplus(raw +
// bias[head]) under M3_PRO_DT_SOFTPLUS.
__device__ __forceinline__ float scan_dt(float raw, int pro, const float* bias, int head) {
  return (pro & M3_PRO_DT_SOFTPLUS) ? softplus_f(raw + (bias ? bias[head] : 0.f)) : raw;
}

// 1 / sqrt(mean(v^2) + eps) of n values (one warp; every lane gets it).
template <typename T>
__device__ __forceinline__ float warp_rms_scale(const T* v, int n, int lane) {
  float ss = 0.f;
  for (int i = lane; i < n; i += 32) {
    const float f = to_f(v[i]);
    ss = fmaf(f, f, ss);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  return rsqrtf(ss / (float)n + kBcNormEps);
}

// A compile-time flag passed as a value (to generic lambdas).
template <bool B>
struct BoolTag {
  static constexpr bool value = B;
};

// Output element i of y: f32, or bf16 rounded to nearest even when `ybf`
// (the f32 value of the f32 path, rounded once).
__device__ __forceinline__ void st_y(void* y, int64_t i, float v, bool ybf) {
  if (ybf)
    static_cast<__nv_bfloat16*>(y)[i] = __float2bfloat16_rn(v);
  else
    static_cast<float*>(y)[i] = v;
}
// Elements i, i + 1 (i even) as one 8- or 4-byte store.
__device__ __forceinline__ void st_y2(void* y, int64_t i, float v0, float v1, bool ybf) {
  if (ybf)
    *reinterpret_cast<__nv_bfloat162*>(static_cast<__nv_bfloat16*>(y) + i) = __floats2bfloat162_rn(v0, v1);
  else
    *reinterpret_cast<float2*>(static_cast<float*>(y) + i) = make_float2(v0, v1);
}

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Host-side test hooks (include/m3scan_testing.h): a planted fault and a
// shorter wait limit for the next prefill launches, and what the last
// prefill launched.  Atomics, so that concurrent calls never race on them.
struct TestHooks {
  std::atomic<int> fault{0};
  std::atomic<unsigned long long> wait_ns{0};
  std::atomic<int> last_kernel{0}, last_grid{0};
  std::atomic<long long> last_scratch{0};
};
inline TestHooks& test_hooks() {
  static TestHooks h;
  return h;
}
inline void record_launch(int kernel, int grid, long long scratch) {
  TestHooks& t = test_hooks();
  t.last_kernel.store(kernel);
  t.last_grid.store(grid);
  t.last_scratch.store(scratch);
}

}  // namespace m3
