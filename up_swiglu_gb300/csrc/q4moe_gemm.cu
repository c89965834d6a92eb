// q4moe_gemm.cu -- tensor-core grouped GEMM for experts with many rows
// (placeholder until the tcgen05 kernel lands: reports itself unsupported,
// so every expert runs on the matvec).
#include "q4moe_internal.cuh"

namespace q4moe {

bool gemm_supported(int64_t, int64_t, const GateUpArgs &) { return false; }

cudaError_t launch_gemm(const GateUpArgs &, cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace q4moe
