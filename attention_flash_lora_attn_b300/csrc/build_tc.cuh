// Tensor-core LR-cache build (tcgen05 / TMEM / TMA).  Placeholder until the
// kernel lands: reports every shape as unsupported so the SIMT kernel runs.
#pragma once
#include "fla_common.cuh"

namespace fla {
inline bool build_tc_supported(const void *, int64_t, const void *, const void *, int64_t, int, int, int) {
  return false;
}
inline const char *build_tc_last_error() { return "tensor-core build kernel not built"; }
inline fla_status build_tc_launch(const void *, int64_t, const void *, void *, int64_t, int64_t, int, int,
                                  cudaStream_t) {
  return FLA_ERR_UNSUPPORTED;
}
}  // namespace fla
