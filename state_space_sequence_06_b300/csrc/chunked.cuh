// Chunked prefill on the tensor cores (tcgen05 / TMEM / TMA).
#pragma once

#include "common.cuh"

namespace m3 {

inline m3_status chunked_prefill(const m3_prefill_args* a, float* h, void* prev_B, void* prev_x,
                                 int nseq, cudaStream_t s) {
  (void)a; (void)h; (void)prev_B; (void)prev_x; (void)nseq; (void)s;
  return M3_ERR_UNSUPPORTED;
}

}  // namespace m3
