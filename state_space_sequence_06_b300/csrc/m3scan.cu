// C-ABI implementation of libm3scan: argument checks, state objects and
// kernel dispatch.  The entry points are declared and documented in
// include/m3scan.h.
#include <cuda_runtime.h>

#include <new>

#include "common.cuh"
#include "chunked.cuh"
#include "decode.cuh"
#include "recurrent.cuh"

struct m3_state {
  m3_dims dims;
  float* h;
  void* prev_B;
  void* prev_x;
  cudaStream_t stream;  // the allocation stream: the buffers are stream-ordered on it
};

namespace {

using m3::ceil_div;

size_t dtype_size(int dt) { return dt == M3_BF16 ? 2 : 4; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool dims_ok(const m3_dims* d) {
  return d && d->batch > 0 && d->nheads > 0 && d->headdim > 0 && d->dstate > 0 && d->rank > 0 &&
         (d->dstate % 2) == 0 && (d->headdim % 2) == 0 &&
         (d->in_dtype == M3_F32 || d->in_dtype == M3_BF16) && d->headdim <= 1024 &&
         d->dstate <= 4096 && d->rank <= 64;
}

bool same_dims(const m3_dims& a, const m3_dims& b) {
  return a.batch == b.batch && a.nheads == b.nheads && a.headdim == b.headdim &&
         a.dstate == b.dstate && a.rank == b.rank && a.in_dtype == b.in_dtype;
}

m3_status launch_status() {
  return cudaGetLastError() == cudaSuccess ? M3_OK : M3_ERR_CUDA;
}

// ---------------------------------------------------------------- decode

template <typename T, int ITEMS, bool YB>
m3_status decode_rank(const m3::DecodeParams& p, int threads, size_t smem, int units,
                      cudaStream_t s) {
  switch (p.R) {
#define M3_DEC(RR)                                                                             \
  case RR:                                                                                     \
    if (smem > 48 * 1024 && cudaFuncSetAttribute(m3::decode_step_kernel<T, ITEMS, RR, YB>,      \
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,   \
                                                 (int)smem) != cudaSuccess)                     \
      return M3_ERR_CUDA;                                                                      \
    m3::decode_step_kernel<T, ITEMS, RR, YB><<<units, threads, smem, s>>>(p);                  \
    return launch_status();
    M3_DEC(1) M3_DEC(4)
#undef M3_DEC
    default:
      if (p.R > 8) return M3_ERR_UNSUPPORTED;
      if (smem > 48 * 1024 && cudaFuncSetAttribute(m3::decode_step_kernel<T, ITEMS, 0, YB>,
                                                   cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                   (int)smem) != cudaSuccess)
        return M3_ERR_CUDA;
      m3::decode_step_kernel<T, ITEMS, 0, YB><<<units, threads, smem, s>>>(p);
      return launch_status();
  }
}

template <typename T, bool YB>
m3_status decode_items(const m3::DecodeParams& p, int items, int threads, size_t smem, int units,
                       cudaStream_t s) {
  if (items <= 1) return decode_rank<T, 1, YB>(p, threads, smem, units, s);
  if (items <= 2) return decode_rank<T, 2, YB>(p, threads, smem, units, s);
  if (items <= 4) return decode_rank<T, 4, YB>(p, threads, smem, units, s);
  if (items <= 8) return decode_rank<T, 8, YB>(p, threads, smem, units, s);
  if (items <= 16) return decode_rank<T, 16, YB>(p, threads, smem, units, s);
  return M3_ERR_UNSUPPORTED;
}

template <typename T>
m3_status decode_launch(m3::DecodeParams p, int units, cudaStream_t s) {
  p.K = p.N / 2;
  p.PP = p.P / 2;
  if (p.PP > 256) return M3_ERR_UNSUPPORTED;
  // rank > 1 keeps more per-thread registers (x columns and outputs per
  // rank), and a 16 KB state (N 64) leaves room for more CTAs than
  // 256-thread ones' registers allow: smaller CTAs keep more of them
  // resident per SM
  int kg = (p.R == 1 && p.N > 64 ? 256 : 128) / p.PP;
  if (kg < 1) kg = 1;
  while (ceil_div(p.K, kg) > 16 && p.PP * kg * 2 <= 256) kg *= 2;
  if (kg > p.K) kg = p.K;
  p.KG = kg;
  const int threads = p.PP * kg;
  int items = ceil_div(p.K, kg);
  // the state (K*P complex f32), pair records (KW float4 each, sized for the
  // compile-time rank bound), x and previous x, partial outputs
  const int rmax = p.R == 1 ? 1 : (p.R == 4 ? 4 : 8);
  const size_t kw = (3 * rmax + 2) / 2;
  const size_t esz = sizeof(T);
  const size_t raw = esz * (3 * (size_t)p.R * p.N + 2 * (size_t)p.R * p.P + p.K);
  auto al16 = [](const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
  p.bulk = ((p.R * p.N * esz) % 16 == 0 && (p.R * p.P * esz) % 16 == 0 && (p.K * esz) % 16 == 0 &&
            al16(p.x) && al16(p.B) && al16(p.C) && al16(p.theta) && al16(p.prev_B) && al16(p.prev_x))
               ? 1
               : 0;
  // (layout: state, x rows, the records and raw inputs, then the partial
  // outputs -- which, above rank 1, reuse the records' and raw inputs' room)
  const size_t tail = sizeof(float4) * p.K * kw + (p.bulk ? raw : 0);
  const size_t red = sizeof(float) * (size_t)kg * p.R * p.P;
  const size_t smem = sizeof(float4) * p.K * p.PP + sizeof(float) * 2 * rmax * p.P +
                      (p.R == 1 ? tail + 16 + red : (tail > red ? tail : red));
  if (smem > 200 * 1024) return M3_ERR_UNSUPPORTED;
  return p.ybf ? decode_items<T, true>(p, items, threads, smem, units, s)
               : decode_items<T, false>(p, items, threads, smem, units, s);
}

// ---------------------------------------------------------------- recurrent prefill

template <typename T, int KPT, int RR>
m3_status recurrent_go(const m3::RecurrentParams& p, int units, int threads, size_t smem,
                       cudaStream_t s) {
  if (smem > 48 * 1024 &&
      cudaFuncSetAttribute(m3::recurrent_prefill_kernel<T, KPT, RR>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return M3_ERR_CUDA;
  m3::recurrent_prefill_kernel<T, KPT, RR><<<units, threads, smem, s>>>(p);
  return launch_status();
}

template <typename T, int KPT>
m3_status recurrent_rank(const m3::RecurrentParams& p, int R, int units, int threads, size_t smem,
                         cudaStream_t s) {
  if (R == 1) return recurrent_go<T, KPT, 1>(p, units, threads, smem, s);
  if (R <= 8) return recurrent_go<T, KPT, 0>(p, units, threads, smem, s);
  return M3_ERR_UNSUPPORTED;
}

template <typename T>
m3_status recurrent_launch(m3::RecurrentParams p, int R, int units, cudaStream_t s) {
  p.K = p.N / 2;
  // pairs per thread: 8, with up to 32 threads per p; larger N uses 16 or 32
  int kpt = 8;
  while (ceil_div(p.K, kpt) > 32) kpt *= 2;
  if (kpt > 32) return M3_ERR_UNSUPPORTED;
  int ks = 1;
  while (ks < ceil_div(p.K, kpt)) ks *= 2;
  p.KS = ks;
  const int threads = ceil_div(p.P * ks, 32) * 32;
  if (threads > 1024) return M3_ERR_UNSUPPORTED;
  const int RN = R * p.N, RP = R * p.P;
  auto smem_for = [&](int tb) {
    return sizeof(float) * ((size_t)(tb + 1) * RN + (size_t)tb * RN + (size_t)(tb + 1) * RP +
                            (size_t)tb * 2 * p.K + 2 * (size_t)tb);
  };
  int tb = 32;
  while (tb > 1 && smem_for(tb) > 96 * 1024) tb /= 2;
  p.TB = tb;
  const size_t smem = smem_for(tb);
  if (smem > 200 * 1024) return M3_ERR_UNSUPPORTED;
  switch (kpt) {
    case 8: return recurrent_rank<T, 8>(p, R, units, threads, smem, s);
    case 16: return recurrent_rank<T, 16>(p, R, units, threads, smem, s);
    default: return recurrent_rank<T, 32>(p, R, units, threads, smem, s);
  }
}

}  // namespace

extern "C" {

const char* m3_status_string(m3_status s) {
  switch (s) {
    case M3_OK: return "ok";
    case M3_ERR_INVALID_ARG: return "invalid argument";
    case M3_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case M3_ERR_CUDA: return "CUDA error";
    case M3_ERR_TIMEOUT: return "device wait timed out";
    case M3_ERR_ALLOC: return "device allocation failed";
    case M3_ERR_SCRATCH:
      return "the request needs more scratch than the fixed buffer of m3_scan_prefill_noalloc holds";
  }
  return "unknown status";
}

m3_status m3_state_alloc(const m3_dims* dims, m3_state** out, void* stream) {
  if (!out || !dims_ok(dims)) return M3_ERR_INVALID_ARG;
  *out = nullptr;
  const size_t units = (size_t)dims->batch * dims->nheads;
  const size_t hb = units * dims->dstate * dims->headdim * sizeof(float);
  const size_t bb = units * dims->rank * dims->dstate * dtype_size(dims->in_dtype);
  const size_t xb = units * dims->rank * dims->headdim * dtype_size(dims->in_dtype);
  m3_state* st = new (std::nothrow) m3_state();
  if (!st) return M3_ERR_ALLOC;
  st->dims = *dims;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  st->stream = s;
  // stream-ordered buffers: m3_state_free returns them on the same stream
  // without waiting for the device
  auto release = [&]() {
    if (st->h) cudaFreeAsync(st->h, s);
    if (st->prev_B) cudaFreeAsync(st->prev_B, s);
    if (st->prev_x) cudaFreeAsync(st->prev_x, s);
    delete st;
  };
  if (cudaMallocAsync(reinterpret_cast<void**>(&st->h), hb, s) != cudaSuccess ||
      cudaMallocAsync(&st->prev_B, bb, s) != cudaSuccess || cudaMallocAsync(&st->prev_x, xb, s) != cudaSuccess) {
    cudaGetLastError();
    release();
    return M3_ERR_ALLOC;
  }
  if (cudaMemsetAsync(st->h, 0, hb, s) != cudaSuccess ||
      cudaMemsetAsync(st->prev_B, 0, bb, s) != cudaSuccess ||
      cudaMemsetAsync(st->prev_x, 0, xb, s) != cudaSuccess) {
    release();
    return M3_ERR_CUDA;
  }
  *out = st;
  return M3_OK;
}

m3_status m3_state_free(m3_state* st) {
  if (!st) return M3_OK;
  m3_status rc = M3_OK;
  if (cudaFreeAsync(st->h, st->stream) != cudaSuccess) rc = M3_ERR_CUDA;
  if (cudaFreeAsync(st->prev_B, st->stream) != cudaSuccess) rc = M3_ERR_CUDA;
  if (cudaFreeAsync(st->prev_x, st->stream) != cudaSuccess) rc = M3_ERR_CUDA;
  delete st;
  return rc;
}

m3_status m3_state_view(const m3_state* st, m3_state_ptrs* out) {
  if (!st || !out) return M3_ERR_INVALID_ARG;
  out->dims = st->dims;
  out->h = st->h;
  out->prev_B = st->prev_B;
  out->prev_x = st->prev_x;
  return M3_OK;
}

m3_status m3_decode_step(const m3_decode_args* a, m3_state* st, void* stream) {
  if (!a || !st || !dims_ok(&a->dims) || !same_dims(a->dims, st->dims)) return M3_ERR_INVALID_ARG;
  // lam and theta may be NULL (lam = 1, theta = 0: the Mamba-2 special case)
  if (!a->x || !a->B || !a->C || !a->dt || !a->A || !a->D || !a->y) return M3_ERR_INVALID_ARG;
  if (a->ngroups < 0 || (a->ngroups > 0 && a->dims.nheads % a->ngroups != 0)) return M3_ERR_INVALID_ARG;
  if (a->y_dtype != M3_F32 && a->y_dtype != M3_BF16) return M3_ERR_INVALID_ARG;
  if (a->prologue & ~(M3_PRO_DT_SOFTPLUS | M3_PRO_BC_NORM)) return M3_ERR_INVALID_ARG;
  if (!aligned16(a->x) || !aligned16(a->B) || !aligned16(a->C) || !aligned16(a->theta) ||
      !aligned16(a->y))
    return M3_ERR_INVALID_ARG;
  m3::DecodeParams p{};
  p.x = a->x; p.B = a->B; p.C = a->C; p.dt = a->dt; p.lam = a->lam; p.theta = a->theta;
  p.A = a->A; p.D = a->D; p.y = a->y; p.ybf = a->y_dtype == M3_BF16;
  p.pro = a->prologue; p.dt_bias = a->dt_bias;
  p.h = st->h; p.prev_B = st->prev_B; p.prev_x = st->prev_x;
  p.H = a->dims.nheads; p.P = a->dims.headdim; p.N = a->dims.dstate; p.R = a->dims.rank;
  p.G = a->ngroups > 0 ? a->ngroups : a->dims.nheads;
  const int units = a->dims.batch * a->dims.nheads;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return a->dims.in_dtype == M3_BF16 ? decode_launch<__nv_bfloat16>(p, units, s)
                                     : decode_launch<float>(p, units, s);
}

}  // extern "C"

namespace {

// The prefill of both entry points; `fixed` (fixed_bytes long) replaces the
// pool memory of the balanced schedule's handover slots when given.
m3_status prefill_impl(const m3_prefill_args* a, m3_state* st, void* stream, void* fixed, size_t fixed_bytes) {
  if (!a || !dims_ok(&a->dims) || a->seqlen < 0) return M3_ERR_INVALID_ARG;
  // lam and theta may be NULL (lam = 1, theta = 0: the Mamba-2 special case)
  if (!a->x || !a->B || !a->C || !a->dt || !a->A || !a->D || !a->y) return M3_ERR_INVALID_ARG;
  if (a->ngroups < 0 || (a->ngroups > 0 && a->dims.nheads % a->ngroups != 0)) return M3_ERR_INVALID_ARG;
  if (a->y_dtype != M3_F32 && a->y_dtype != M3_BF16) return M3_ERR_INVALID_ARG;
  if (a->prologue & ~(M3_PRO_DT_SOFTPLUS | M3_PRO_BC_NORM)) return M3_ERR_INVALID_ARG;
  if (!aligned16(a->x) || !aligned16(a->B) || !aligned16(a->C) || !aligned16(a->theta) ||
      !aligned16(a->y))
    return M3_ERR_INVALID_ARG;
  if (a->algo < M3_ALGO_AUTO || a->algo > M3_ALGO_CHUNKED) return M3_ERR_INVALID_ARG;
  const bool varlen = a->cu_seqlens != nullptr;
  if (varlen && (a->dims.batch != 1 || a->nseq <= 0)) return M3_ERR_INVALID_ARG;
  const int nseq = varlen ? a->nseq : a->dims.batch;
  if (st) {
    m3_dims want = a->dims;
    want.batch = nseq;
    if (!same_dims(want, st->dims)) return M3_ERR_INVALID_ARG;
  }
  if (a->seqlen == 0) return M3_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int units = nseq * a->dims.nheads;
  const bool bf16 = a->dims.in_dtype == M3_BF16;

  if (a->algo != M3_ALGO_RECURRENT) {
    m3_status rc = m3::chunked_prefill(a, st ? st->h : nullptr, st ? st->prev_B : nullptr,
                                       st ? st->prev_x : nullptr, nseq, s, fixed, fixed_bytes);
    if (rc != M3_ERR_UNSUPPORTED || a->algo == M3_ALGO_CHUNKED) return rc;
  }
  m3::RecurrentParams p{};
  p.x = a->x; p.B = a->B; p.C = a->C; p.dt = a->dt; p.lam = a->lam; p.theta = a->theta;
  p.A = a->A; p.D = a->D; p.cu_seqlens = a->cu_seqlens; p.y = a->y; p.ybf = a->y_dtype == M3_BF16;
  p.pro = a->prologue; p.dt_bias = a->dt_bias;
  p.h = st ? st->h : nullptr;
  p.prev_B = st ? st->prev_B : nullptr;
  p.prev_x = st ? st->prev_x : nullptr;
  p.L = a->seqlen;
  p.H = a->dims.nheads; p.P = a->dims.headdim; p.N = a->dims.dstate; p.R = a->dims.rank;
  p.G = a->ngroups > 0 ? a->ngroups : a->dims.nheads;
  m3::record_launch(M3_TEST_KERNEL_RECURRENT, units, 0);
  return bf16 ? recurrent_launch<__nv_bfloat16>(p, a->dims.rank, units, s)
              : recurrent_launch<float>(p, a->dims.rank, units, s);
}

// The fixed scratch of m3_scan_prefill_noalloc: module memory of the
// library.  CUDA creates it on a device when it loads the library's device
// code there -- under the default lazy module loading, at the first use of
// the module on that device (the address lookup of the entry point's first
// call does it); no call allocates it.
static __device__ __align__(256) unsigned char g_noalloc_scratch[M3_NOALLOC_SCRATCH_BYTES];

}  // namespace

extern "C" {

m3_status m3_scan_prefill(const m3_prefill_args* a, m3_state* st, void* stream) {
  return prefill_impl(a, st, stream, nullptr, 0);
}

m3_status m3_scan_prefill_noalloc(const m3_prefill_args* a, m3_state* st, void* stream) {
  // The scratch's address on the current device, looked up once per device
  // (atomics: calls from several host threads see either null or the one
  // address).  The cache assumes that the device's primary context lives as
  // long as the library: after a device reset the address is stale.
  static std::atomic<void*> addr[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return M3_ERR_CUDA;
  void* base = addr[dev].load(std::memory_order_acquire);
  if (!base) {
    if (cudaGetSymbolAddress(&base, g_noalloc_scratch) != cudaSuccess || !base) return M3_ERR_CUDA;
    addr[dev].store(base, std::memory_order_release);
  }
  return prefill_impl(a, st, stream, base, M3_NOALLOC_SCRATCH_BYTES);
}

m3_status m3_test_set_fault(int32_t fault, int64_t wait_limit_ns) {
  if (fault != M3_TEST_FAULT_NONE && fault != M3_TEST_FAULT_SKIP_HANDOVER_RELEASE) return M3_ERR_INVALID_ARG;
  if (wait_limit_ns < 0) return M3_ERR_INVALID_ARG;
  m3::test_hooks().fault.store(fault);
  m3::test_hooks().wait_ns.store((unsigned long long)wait_limit_ns);
  return M3_OK;
}

m3_status m3_test_last_launch(m3_launch_info* out) {
  if (!out) return M3_ERR_INVALID_ARG;
  out->kernel = m3::test_hooks().last_kernel.load();
  out->grid = m3::test_hooks().last_grid.load();
  out->scratch_bytes = m3::test_hooks().last_scratch.load();
  return M3_OK;
}

}  // extern "C"

namespace m3 {
// The device address of the status word, for the backward pass's kernels
// (built in another translation unit): NULL if it cannot be had.
int* device_status_word() {
  void* a = nullptr;
  if (cudaGetSymbolAddress(&a, g_status) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return static_cast<int*>(a);
}
}  // namespace m3

extern "C" {

m3_status m3_device_status(void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return M3_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, m3::g_status, sizeof(int)) != cudaSuccess) return M3_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(m3::g_status, &zero, sizeof(int)) != cudaSuccess) return M3_ERR_CUDA;
    return static_cast<m3_status>(v);
  }
  return M3_OK;
}

}  // extern "C"
