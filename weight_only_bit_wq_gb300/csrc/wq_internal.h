// Host-side declarations shared by the library's translation units.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "wq.h"

namespace wq {

constexpr int kBN = 128;              // weight rows per tile (TMEM lanes)
constexpr int kWordsPerStage = 32;    // packed words per row per TMA box (128 B)
constexpr int kMaxCols = 32;          // max stacked rows M
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
// Rows of X per tile of the kernel build that serves M rows: 16 up to 16,
// else 32 (the 32-row build issues two 16-row MMAs per K step).
constexpr int tc_cols(int M) { return M > 16 ? 32 : 16; }

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
    int pdl;          // launched as a programmatic dependent of the previous kernel on the
                      // stream: X is read, and anything written, once that kernel completed
    int epi;          // WQ_EPI_NONE or WQ_EPI_SWIGLU (y is then bf16 [M][N/2])
    int nc;           // rows of X per tile: tc_cols(M); the X map's box has nc rows
};

// One projection of a fused step, as the step kernel reads it from device
// memory.  Units of all projections form one space: projection p owns global
// units [uoff, uoff + T * I) and global tiles [toff, toff + T).
struct ProjDev {  // aligned like its tensor maps
    CUtensorMap tmW;         // packed words [N][W]
    CUtensorMap tmX;         // X [M][K] (3-D map when x3d)
    const uint16_t* scales;  // [N][ng] bf16
    const uint8_t* zeros;    // [N][ng]
    float* y;                // [M][N]
    long long uoff;          // first global unit
    int M, N, ng, T, I;
    int toff;                // first global tile
    int meta_vec, x3d;
    int after;               // X is read once phase `after` of this launch is complete (-1: at once)
    int phase;               // phase of the launch this projection belongs to
    int epi;                 // WQ_EPI_NONE or WQ_EPI_SWIGLU (y is then bf16 [M][N/2])
    int pad[3];
};

// A phase of a fused step: consecutive projections none of which waits for
// another projection of the phase.  Every CTA takes its stream-K share of
// every phase: units [uoff + U b / P, uoff + U (b + 1) / P).
struct PhaseDev {
    long long uoff;  // first global unit
    long long U;     // units of the phase
    int need;        // finished (tile, lane quarter) pairs of a complete phase: 4 x its tiles
    int pad;
};
static_assert(sizeof(ProjDev) % 64 == 0, "ProjDev keeps 64-byte alignment in arrays");

// Kernel-wide arguments of a fused step launch.
struct StepArgs {
    const ProjDev* proj;    // [nproj]
    const PhaseDev* phase;  // [nphase]
    int nproj, nphase;
    float* partials;      // [2 * P][kMaxCols][kBN]
    int* counters;        // [total tiles][kCountersPerTile]
    int* done;            // [nphase] finished (tile, lane quarter) pairs per phase, zero at launch
    int* err;
    long long U;          // total units
    int P;
    int pdl;              // launched as a programmatic dependent of the previous kernel on the
                          // stream (one phase, nothing waits): X is read, and anything written,
                          // once that kernel completed
    int act;              // with pdl: some projection of the launch asks for the activation
                          // epilogue (otherwise the build without it serves)
    int cluster;          // > 1: one phase, k = cluster CTAs per tile, each one segment
                          // (P = k x tiles): launched in clusters of k, split-K sums through
                          // rank 0's shared memory
};

// SMs a GEMM grid leaves free.  A launch that is a programmatic dependent of
// the one before places its CTAs as that launch's CTAs leave their SMs; with
// one CTA per SM the last of them could start only when the slowest CTA of
// the previous launch had exited, after the dependency resolved, with none
// of its packed words loaded, and so ended every launch of a chain last
// (the same CTA index, launch after launch).  A grid of two CTAs fewer than
// SMs lets every CTA start early (one or four fewer measured slower); the
// single projection and the fused launch take the same grid, so that every
// mode splits a projection alike.
#ifndef WQ_SPARE_SMS
#define WQ_SPARE_SMS 2
#endif
constexpr int kSpareSms = WQ_SPARE_SMS;
inline int gemm_sm_budget(int sms) { return sms > kSpareSms ? sms - kSpareSms : 1; }

// Static stream-K schedule: CTA b owns units [unit_begin(b), unit_begin(b+1)).
inline long long unit_begin(long long U, int P, int b) { return U * b / P; }

// Grid size from (N, K, bits) and the SM count only (never from M).
int choose_grid(int T, int I, int sm_count);

// At most `budget` CTAs for T tiles whose stream-K shares start and end on
// tile boundaries, if such a grid lies within 74 % of the budget: whole tiles
// per CTA (the largest divisor of T), or, with split_tiles, k CTAs per tile
// (k T, the largest such); else the budget.  A share that ends inside a tile
// ends with a split-K fix-up, the slowest part of a launch's tail.
int aligned_grid(int T, int budget, bool split_tiles);

// Tensor-core (tcgen05) GEMM kernels, one translation unit per bit width.
cudaError_t launch_gemm_tc_b4(int group, const CUtensorMap& tmW, const CUtensorMap& tmX,
                              const GemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm_tc_b3(int group, const CUtensorMap& tmW, const CUtensorMap& tmX,
                              const GemmArgs& a, cudaStream_t s);
cudaError_t launch_gemm_tc_b2(int group, const CUtensorMap& tmW, const CUtensorMap& tmX,
                              const GemmArgs& a, cudaStream_t s);
// Fused step: all projections of `sa` (one bit width and group size) in one
// persistent launch; cooperative when any projection waits for another; nc
// rows of X per tile (every projection's X map has boxes of nc rows).
cudaError_t launch_step_b4(int group, const StepArgs& sa, bool cooperative, int nc,
                           cudaStream_t s);
cudaError_t launch_step_b3(int group, const StepArgs& sa, bool cooperative, int nc,
                           cudaStream_t s);
cudaError_t launch_step_b2(int group, const StepArgs& sa, bool cooperative, int nc,
                           cudaStream_t s);

// wq_gemm with the launch mode chosen by the caller: pdl = launch as a
// programmatic dependent of the previous kernel on the stream (only where
// that kernel writes none of wq, scales and zeros).
wq_status_t gemm_run(const uint16_t* x, const uint32_t* wq, const uint16_t* scales,
                     const uint8_t* zeros, void* y, int M, int N, int K, int group, int bits,
                     void* workspace, size_t workspace_bytes, cudaStream_t s, bool pdl,
                     int epi);

// Host helpers shared by the entry points (wq_api.cu).
wq_status_t host_cuda_fail(cudaError_t e);
wq_status_t host_sm_count(int* sms);
wq_status_t host_check_gemm(const uint16_t* x, const uint32_t* wq, const uint16_t* scales,
                            const uint8_t* zeros, const void* y, int M, int N, int K, int group,
                            int bits, int epi);
// Tensor maps of one projection; X boxes of nc rows.
wq_status_t host_encode_proj(const uint16_t* x, const uint32_t* wq, const uint16_t* scales,
                             const uint8_t* zeros, int M, int N, int K, int group, int bits,
                             int nc, CUtensorMap* tmW, CUtensorMap* tmX, int* x3d,
                             int* meta_vec);

// Elementwise kernels.
cudaError_t launch_pack(const uint8_t* q, uint32_t* wq, int N, int K, int bits, int W,
                        int sm_count, cudaStream_t s);
cudaError_t launch_unpack(const uint32_t* wq, uint8_t* q, int N, int K, int bits, int W,
                          int sm_count, cudaStream_t s);
cudaError_t launch_dequant(const uint32_t* wq, const uint16_t* scales, const uint8_t* zeros,
                           uint16_t* w, int N, int K, int group, int bits, int W, int sm_count,
                           cudaStream_t s);

}  // namespace wq
