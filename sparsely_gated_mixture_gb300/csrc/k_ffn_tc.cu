// Stage 4 experts on the tensor cores (tcgen05 / TMEM / TMA). Placeholder until
// the grouped GEMM lands: reports no support, so the CUDA-core kernel runs.
#include "moe_internal.cuh"

namespace moe {

bool ffn_tc_supported(const moe_config &) { return false; }

cudaError_t launch_ffn_tc(const moe_config &, int, const void *, const int32_t *, const int32_t *,
                          const float *, const void *, const void *, const void *, const void *,
                          void *, float *, DeviceStatus *, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace moe
