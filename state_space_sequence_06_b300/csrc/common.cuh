// Shared device helpers of the m3scan kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "m3scan.h"

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

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

}  // namespace m3
