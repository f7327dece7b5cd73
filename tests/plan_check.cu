// Host-only listing of every tensor-core kernel build's compile-time layout:
// stages, shared memory, tensor-memory plan.  Built and run by
// test_build_plans.py; no device code runs.
#include <cstdio>

#include "wq_gemm_tc.cuh"

using namespace wq::tc;

template <int B, int G, int NC>
void row() {
    using L = Lay<B, G, NC>;
    std::printf("%d %d %d %d %d %d %d %d %d %d\n", B, G, NC, L::kStages, L::kSmemBytes,
                static_cast<int>(L::kZtc), L::kNA, L::kND,
                static_cast<int>(L::kColD + L::kND * L::kR0 * NC), L::kThreads);
}

template <int B, int G>
void both() {
    row<B, G, 16>();
    row<B, G, 32>();
}

int main() {
    both<4, 128>(); both<4, 64>(); both<4, 32>();
    both<3, 128>(); both<3, 64>(); both<3, 32>();
    both<2, 128>(); both<2, 64>(); both<2, 32>();
    return 0;
}
