// Host-side declarations shared by the library's translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace wq {

constexpr int kBN = 128;              // weight rows per tile (TMEM lanes)
constexpr int kWordsPerStage = 32;    // packed words per row per TMA box (128 B)
constexpr int kMaxCols = 16;          // max stacked rows M
constexpr int kMaxSplit = 8;          // max CTAs sharing one tile
constexpr int kCountersPerTile = 16;  // split-K arrival counters per tile (one per consumer warp)
constexpr size_t kWsHeader = 256;     // error word + padding

// Values per packed word.
constexpr int values_per_word(int bits) { return bits == 4 ? 8 : bits == 3 ? 10 : 16; }
// 32-word boxes per row per stage, chosen so that a stage holds whole groups
// and the per-stage tensor-memory tiles fit in 512 columns.
constexpr int tc_boxes(int bits, int group) {
    return bits == 4 ? (group == 32 ? 1 : 2) : bits == 3 ? (group == 128 ? 2 : 1) : 1;
}
constexpr int tc_stage_values(int bits, int group) {
    return tc_boxes(bits, group) * kWordsPerStage * values_per_word(bits);
}

struct GemmArgs {
    const uint16_t* scales;
    const uint8_t* zeros;
    float* y;
    float* partials;  // [2 * P][kMaxCols][kBN]
    int* counters;    // [T][kCountersPerTile]
    int* err;         // kernel error word
    int M, N, K, ng;
    int T, I;         // tiles, k-stages per tile
    long long U;      // T * I work units
    int P;            // CTAs
    int meta_vec;     // scales/zeros 16-byte aligned and K/group a multiple of the groups per stage
    int x3d;          // X map is 3-D [K/64][M][64]: one TMA box per stage (K % 64 == 0)
};

// Static stream-K schedule: CTA b owns units [unit_begin(b), unit_begin(b+1)).
inline long long unit_begin(long long U, int P, int b) { return U * b / P; }

// Grid size from (N, K, bits) and the SM count only (never from M).
int choose_grid(int T, int I, int sm_count);

// Tensor-core (tcgen05) GEMM kernels, one translation unit per bit width.
cudaError_t launch_gemm_tc_b4(int group, const CUtensorMap& tmW, const CUtensorMap& tmX,
                              const GemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm_tc_b3(int group, const CUtensorMap& tmW, const CUtensorMap& tmX,
                              const GemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm_tc_b2(int group, const CUtensorMap& tmW, const CUtensorMap& tmX,
                              const GemmArgs& a, cudaStream_t s);

// Elementwise kernels.
cudaError_t launch_pack(const uint8_t* q, uint32_t* wq, int N, int K, int bits, int W,
                        int sm_count, cudaStream_t s);
cudaError_t launch_unpack(const uint32_t* wq, uint8_t* q, int N, int K, int bits, int W,
                          int sm_count, cudaStream_t s);
cudaError_t launch_dequant(const uint32_t* wq, const uint16_t* scales, const uint8_t* zeros,
                           uint16_t* w, int N, int K, int group, int bits, int W, int sm_count,
                           cudaStream_t s);

}  // namespace wq
