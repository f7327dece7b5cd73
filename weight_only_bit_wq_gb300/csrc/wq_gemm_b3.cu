// 3-bit instantiations of the weight-only GEMM kernel.
#include "wq_internal.h"

namespace wq {

cudaError_t launch_gemm_b3(int, int, const CUtensorMap&, const CUtensorMap&, const GemmArgs&,
                           cudaStream_t) {
    return cudaErrorNotSupported;
}

}  // namespace wq
