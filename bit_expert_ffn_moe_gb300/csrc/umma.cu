// umma.cu -- tcgen05 block-scaled grouped GEMMs (placeholder until implemented).
#include "common.cuh"
namespace moe {
cudaError_t launch_umma_up(const uint8_t*, const uint8_t*, PlanView, const int32_t*, int, int, int, int, int, int64_t,
                           const moe_expert_weights*, uint8_t*, uint8_t*, int*, cudaStream_t, bool) {
    return cudaErrorNotSupported;
}
cudaError_t launch_umma_down(const uint8_t*, const uint8_t*, PlanView, const int32_t*, int, int, int, int, int, int64_t,
                             const moe_expert_weights*, uint16_t*, int*, cudaStream_t, bool) {
    return cudaErrorNotSupported;
}
}  // namespace moe
