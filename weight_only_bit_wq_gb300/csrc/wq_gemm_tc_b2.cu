// 2-bit instantiations of the tensor-core (tcgen05) GEMM kernel.
#include "wq_gemm_tc.cuh"

namespace wq {

cudaError_t launch_gemm_tc_b2(int group, const CUtensorMap& tmW, const CUtensorMap& tmX,
                              const GemmArgs& a, cudaStream_t s) {
    if (group == 128) return tc::launch_tc<2, 128>(tmW, tmX, a, s);
    if (group == 64) return tc::launch_tc<2, 64>(tmW, tmX, a, s);
    if (group == 32) return tc::launch_tc<2, 32>(tmW, tmX, a, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_step_b2(int group, const StepArgs& sa, bool cooperative, int nc, cudaStream_t s) {
    if (group == 128) return tc::launch_step<2, 128>(sa, cooperative, nc, s);
    if (group == 64) return tc::launch_step<2, 64>(sa, cooperative, nc, s);
    if (group == 32) return tc::launch_step<2, 32>(sa, cooperative, nc, s);
    return cudaErrorInvalidValue;
}

}  // namespace wq
