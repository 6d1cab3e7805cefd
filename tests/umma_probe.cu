// GPU check of the tcgen05 operand layouts and TMEM accumulator layouts
// that the chunked prefill kernel relies on.  The host lays the operand
// tiles out byte by byte (so a layout hypothesis is a host-side choice),
// the kernel copies them to shared memory, issues the MMAs with the given
// descriptor fields, and dumps all 128 TMEM lanes of the accumulator.
#include <cuda_runtime.h>
#include <stdint.h>

#include "../state_space_sequence_06_b300/csrc/umma.cuh"

using namespace m3::umma;

struct ProbeArgs {
  const uint8_t* a_img;
  const uint8_t* b_img;
  float* out;   // [128][ncols]
  int* err;
  int a_bytes, b_bytes;
  uint32_t a_lbo, a_sbo, b_lbo, b_sbo;
  uint32_t a_kstep, b_kstep;  // bytes per K=16 step
  int nk;
  uint32_t idesc;
  int ncols;  // accumulator columns to dump (multiple of 16, <= 256)
  float* out2;  // optional: the same columns read with the 16x256b shape,
                // [warp][ncols / 16][thread][8] (lanes 32*warp .. 32*warp + 15)
};

constexpr int kTileBytes = 65536;

__global__ void __launch_bounds__(128) umma_probe_kernel(const ProbeArgs p) {
  extern __shared__ uint8_t sm_raw[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base;
  uint8_t* base = sm_raw + ((1024u - (saddr(sm_raw) & 1023u)) & 1023u);
  uint8_t* A = base;
  uint8_t* B = base + kTileBytes;
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  for (int i = tid * 16; i < p.a_bytes; i += blockDim.x * 16)
    *reinterpret_cast<uint4*>(A + i) = *reinterpret_cast<const uint4*>(p.a_img + i);
  for (int i = tid * 16; i < p.b_bytes; i += blockDim.x * 16)
    *reinterpret_cast<uint4*>(B + i) = *reinterpret_cast<const uint4*>(p.b_img + i);
  fence_async_smem();
  if (tid == 0) {
    mbar_init(saddr(&bar), 1);
    mbar_init_fence();
  }
  if (warp == 0) {
    tmem_alloc(saddr(&tmem_base), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  if (tid == 0) {
    for (int k = 0; k < p.nk; ++k) {
      uint64_t da = smem_desc(saddr(A) + k * p.a_kstep, p.a_lbo, p.a_sbo, kSwizzle128B);
      uint64_t db = smem_desc(saddr(B) + k * p.b_kstep, p.b_lbo, p.b_sbo, kSwizzle128B);
      mma_f16(tmem, da, db, p.idesc, k > 0 ? 1u : 0u);
    }
    mma_commit(saddr(&bar));
  }
  __syncwarp();
  if (!mbar_wait(saddr(&bar), 0, 1u << 20)) {
    if (lane == 0) atomicExch(p.err, 1);
  }
  tc_fence_after();
  for (int c = 0; c < p.ncols; c += 16) {
    float v[16];
    tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + c, v);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) p.out[(32 * warp + lane) * p.ncols + c + i] = v[i];
  }
  if (p.out2) {
    for (int c = 0; c < p.ncols; c += 16) {
      float v[8];
      tmem_ld16x256b_x2(tmem + ((uint32_t)(32 * warp) << 16) + c, v);
      tmem_ld_wait();
#pragma unroll
      for (int i = 0; i < 8; ++i) p.out2[((warp * (p.ncols / 16) + c / 16) * 32 + lane) * 8 + i] = v[i];
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

extern "C" int umma_probe_run(const ProbeArgs* p) {
  const int smem = 2 * kTileBytes + 1024;
  if (cudaFuncSetAttribute(umma_probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return -1;
  umma_probe_kernel<<<1, 128, smem>>>(*p);
  if (cudaGetLastError() != cudaSuccess) return -2;
  if (cudaDeviceSynchronize() != cudaSuccess) return -3;
  return 0;
}

// A operand in TMEM: every TMEM lane's 32 words of A columns come from the
// host (so the lane layout is a host-side hypothesis), B is a K-major
// 128B-swizzled tile; D is dumped like above.
struct ProbeTaArgs {
  const uint32_t* a_words;  // [128 lanes][32 words]
  const uint8_t* b_img;     // 64 KB
  float* out;               // [128][ncols]
  int* err;
  uint32_t b_lbo, b_sbo, b_kstep;
  int nk;
  uint32_t idesc;
  int ncols;
  int a_col;    // first TMEM column of A (after the accumulator's)
  int a_kstep;  // TMEM columns per K = 16 step
};

__global__ void __launch_bounds__(128) umma_probe_ta_kernel(const ProbeTaArgs p) {
  extern __shared__ uint8_t sm_raw[];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_base;
  uint8_t* B = sm_raw + ((1024u - (saddr(sm_raw) & 1023u)) & 1023u);
  const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;
  for (int i = tid * 16; i < kTileBytes; i += blockDim.x * 16)
    *reinterpret_cast<uint4*>(B + i) = *reinterpret_cast<const uint4*>(p.b_img + i);
  fence_async_smem();
  if (tid == 0) {
    mbar_init(saddr(&bar), 1);
    mbar_init_fence();
  }
  if (warp == 0) {
    tmem_alloc(saddr(&tmem_base), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  for (int c = 0; c < 32; c += 16) {
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(p.a_words[(32 * warp + lane) * 32 + c + i]);
    tmem_st16(tmem + ((uint32_t)(32 * warp) << 16) + p.a_col + c, v);
  }
  tmem_st_wait();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (tid == 0) {
    for (int k = 0; k < p.nk; ++k) {
      uint64_t db = smem_desc(saddr(B) + k * p.b_kstep, p.b_lbo, p.b_sbo, kSwizzle128B);
      mma_f16_ta(tmem, tmem + p.a_col + k * p.a_kstep, db, p.idesc, k > 0 ? 1u : 0u);
    }
    mma_commit(saddr(&bar));
  }
  __syncwarp();
  if (!mbar_wait(saddr(&bar), 0, 1u << 20)) {
    if (lane == 0) atomicExch(p.err, 1);
  }
  tc_fence_after();
  for (int c = 0; c < p.ncols; c += 16) {
    float v[16];
    tmem_ld16(tmem + ((uint32_t)(32 * warp) << 16) + c, v);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 16; ++i) p.out[(32 * warp + lane) * p.ncols + c + i] = v[i];
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 256);
}

extern "C" int umma_probe_ta_run(const ProbeTaArgs* p) {
  const int smem = kTileBytes + 1024;
  if (p->ncols > 128 || p->a_col < p->ncols || p->a_col + p->nk * p->a_kstep > 256) return -4;
  if (cudaFuncSetAttribute(umma_probe_ta_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return -1;
  umma_probe_ta_kernel<<<1, 128, smem>>>(*p);
  if (cudaGetLastError() != cudaSuccess) return -2;
  if (cudaDeviceSynchronize() != cudaSuccess) return -3;
  return 0;
}
