// Load-time repacking and streaming dequantisation (one thread per packed word).
//
// Layout: code k of a row sits in word k / vpw (vpw = 8, 10, 16 for b = 4, 3,
// 2), slot j = k % vpw, at bits [16 (j % 2) + b (j / 2), +b): even slots fill
// the low half-word and odd slots the high half-word, each half least
// significant first.  Rows hold W words, W a multiple of 4; unused slots, pad
// bits and padding words are zero.  Repacking at load time: Agens Engine page,
// section "功能" (加载时重新打包).
#include <cuda_bf16.h>
#include "wq_internal.h"

namespace wq {
namespace {

__device__ __forceinline__ int vpw_of(int bits) { return bits == 4 ? 8 : bits == 3 ? 10 : 16; }

// First bit of slot j inside its word.
__device__ __forceinline__ int slot_shift(int bits, int j) { return 16 * (j & 1) + bits * (j >> 1); }

__global__ void pack_kernel(const uint8_t* __restrict__ q, uint32_t* __restrict__ wq, int N, int K,
                            int bits, int W) {
    const int vpw = vpw_of(bits);
    const uint32_t mask = (1u << bits) - 1u;
    const long long total = static_cast<long long>(N) * W;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long n = idx / W;
        const int w = static_cast<int>(idx - n * W);
        const int k0 = w * vpw;
        const uint8_t* row = q + n * K;
        uint32_t word = 0;
        for (int j = 0; j < vpw; ++j) {
            const int k = k0 + j;
            if (k < K) word |= (static_cast<uint32_t>(row[k]) & mask) << slot_shift(bits, j);
        }
        wq[idx] = word;
    }
}

__global__ void unpack_kernel(const uint32_t* __restrict__ wq, uint8_t* __restrict__ q, int N,
                              int K, int bits, int W) {
    const int vpw = vpw_of(bits);
    const uint32_t mask = (1u << bits) - 1u;
    const long long total = static_cast<long long>(N) * W;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long n = idx / W;
        const int w = static_cast<int>(idx - n * W);
        const int k0 = w * vpw;
        if (k0 >= K) continue;
        const uint32_t word = wq[idx];
        uint8_t* row = q + n * K;
        for (int j = 0; j < vpw; ++j) {
            const int k = k0 + j;
            if (k < K) row[k] = static_cast<uint8_t>((word >> slot_shift(bits, j)) & mask);
        }
    }
}

// w = RNE_bf16((q - z) * s).  q - z is an integer with |q - z| <= 255 (8
// significant bits for any uint8 zero point, at most 5 for the documented
// range) and s is a bf16 (8 bits), so the fp32 product is exact and the cast
// is the only rounding.
__global__ void dequant_kernel(const uint32_t* __restrict__ wq, const uint16_t* __restrict__ scales,
                               const uint8_t* __restrict__ zeros, uint16_t* __restrict__ w, int N,
                               int K, int group, int bits, int W) {
    const int vpw = vpw_of(bits);
    const uint32_t mask = (1u << bits) - 1u;
    const int ng = K / group;
    const long long total = static_cast<long long>(N) * W;
    for (long long idx = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; idx < total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long n = idx / W;
        const int wi = static_cast<int>(idx - n * W);
        const int k0 = wi * vpw;
        if (k0 >= K) continue;
        const uint32_t word = wq[idx];
        uint16_t* out = w + n * K;
        for (int j = 0; j < vpw; ++j) {
            const int k = k0 + j;
            if (k >= K) break;
            const int gidx = k / group;
            const int code = static_cast<int>((word >> slot_shift(bits, j)) & mask);
            const int zp = zeros[n * ng + gidx];
            const float s = __uint_as_float(static_cast<uint32_t>(scales[n * ng + gidx]) << 16);
            const float v = static_cast<float>(code - zp) * s;
            out[k] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
        }
    }
}

int grid_for(long long total, int sm_count) {
    long long blocks = (total + 255) / 256;
    const long long cap = static_cast<long long>(sm_count) * 8;
    if (blocks > cap) blocks = cap;
    return blocks < 1 ? 1 : static_cast<int>(blocks);
}

}  // namespace

cudaError_t launch_pack(const uint8_t* q, uint32_t* wq, int N, int K, int bits, int W,
                        int sm_count, cudaStream_t s) {
    const long long total = static_cast<long long>(N) * W;
    if (total == 0) return cudaSuccess;
    pack_kernel<<<grid_for(total, sm_count), 256, 0, s>>>(q, wq, N, K, bits, W);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint32_t* wq, uint8_t* q, int N, int K, int bits, int W,
                          int sm_count, cudaStream_t s) {
    const long long total = static_cast<long long>(N) * W;
    if (total == 0 || K == 0) return cudaSuccess;
    unpack_kernel<<<grid_for(total, sm_count), 256, 0, s>>>(wq, q, N, K, bits, W);
    return cudaGetLastError();
}

cudaError_t launch_dequant(const uint32_t* wq, const uint16_t* scales, const uint8_t* zeros,
                           uint16_t* w, int N, int K, int group, int bits, int W, int sm_count,
                           cudaStream_t s) {
    const long long total = static_cast<long long>(N) * W;
    if (total == 0 || K == 0) return cudaSuccess;
    dequant_kernel<<<grid_for(total, sm_count), 256, 0, s>>>(wq, scales, zeros, w, N, K, group,
                                                              bits, W);
    return cudaGetLastError();
}

}  // namespace wq
