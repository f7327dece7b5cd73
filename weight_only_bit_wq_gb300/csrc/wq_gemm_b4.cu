// 4-bit instantiations of the weight-only GEMM kernel.
#include "wq_gemm_kernel.cuh"

namespace wq {

cudaError_t launch_gemm_b4(int group, int nt, const CUtensorMap& tmW, const CUtensorMap& tmX,
                           const GemmArgs& a, cudaStream_t s) {
    if (nt == 1) {
        if (group == 128) return launch_one<4, 128, 1>(tmW, tmX, a, s);
        if (group == 64) return launch_one<4, 64, 1>(tmW, tmX, a, s);
        if (group == 32) return launch_one<4, 32, 1>(tmW, tmX, a, s);
    } else {
        if (group == 128) return launch_one<4, 128, 2>(tmW, tmX, a, s);
        if (group == 64) return launch_one<4, 64, 2>(tmW, tmX, a, s);
        if (group == 32) return launch_one<4, 32, 2>(tmW, tmX, a, s);
    }
    return cudaErrorInvalidValue;
}

}  // namespace wq
