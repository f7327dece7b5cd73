// wq_gemm_noalloc: the same GEMM as wq_gemm, for callers that must not
// allocate device memory.  Its split-K scratch (partial sums, per-tile arrival
// counters and the error word) lives in one fixed file-scope device array that
// every GPU loading this library holds until the process exits.
// wq_check_noalloc reads and clears that array's error word.
#include <cuda_runtime.h>

#include <deque>
#include <mutex>

#include "wq.h"
#include "wq_internal.h"

namespace {

// Fixed scratch size.  Enough for the split-K partials of up to 2 x (SM count)
// CTAs (4.98 MB on a 152-SM GB300) plus the arrival counters (64 bytes per
// tile) of about 53,000 128-row tiles, i.e. N up to about 6.8 million rows.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

struct NoAllocDevice {
    bool ready = false;
    unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on that device
    int sm_count = 0;
};

std::mutex g_noalloc_mu;
// a deque keeps entries in place as devices are added (handed-out pointers stay valid)
std::deque<NoAllocDevice> g_noalloc_dev;

// The current device's entry (created empty if new).
NoAllocDevice* noalloc_entry(int* dev_out) {
    int dev = 0;
    if (cudaError_t e = cudaGetDevice(&dev); e != cudaSuccess) {
        wq::host_cuda_fail(e);
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (static_cast<int>(g_noalloc_dev.size()) <= dev) g_noalloc_dev.resize(dev + 1);
    *dev_out = dev;
    return &g_noalloc_dev[dev];
}

// One-time set-up for the current device: look up the array's device address
// (in host code the symbol name is only a host-side stand-in) and zero it.
wq_status_t noalloc_setup(cudaStream_t s, NoAllocDevice** out) {
    int dev = 0;
    NoAllocDevice* d = noalloc_entry(&dev);
    if (!d) return WQ_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!d->ready) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return wq::host_cuda_fail(e);
        if (p == nullptr) return WQ_ERR_CUDA;
        if ((e = cudaDeviceGetAttribute(&d->sm_count, cudaDevAttrMultiProcessorCount, dev)) !=
            cudaSuccess)
            return wq::host_cuda_fail(e);
        if ((e = cudaMemsetAsync(p, 0, kNoAllocScratchBytes, s)) != cudaSuccess)
            return wq::host_cuda_fail(e);
        d->scratch = static_cast<unsigned char*>(p);
        d->ready = true;
    }
    *out = d;
    return WQ_OK;
}

}  // namespace

extern "C" wq_status_t wq_gemm_noalloc(const uint16_t* x, const uint32_t* wq,
                                       const uint16_t* scales, const uint8_t* zeros, float* y,
                                       int M, int N, int K, int group, int bits, void* stream) {
    if (N < 0 || M < 0 || K < 0) return WQ_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    NoAllocDevice* d = nullptr;
    if (wq_status_t st = noalloc_setup(s, &d)) return st;
    // The scratch this problem needs (the workspace layout of wq_gemm: error
    // word, partials, counters) must fit the fixed array.
    const long long tiles = (static_cast<long long>(N) + wq::kBN - 1) / wq::kBN;
    const size_t counter_off =
        wq::kWsHeader + size_t(2) * d->sm_count * wq::kMaxCols * wq::kBN * sizeof(float);
    const size_t counter_bytes = static_cast<size_t>(tiles) * wq::kCountersPerTile * sizeof(int);
    const size_t need = counter_off + counter_bytes;
    if (need > kNoAllocScratchBytes) return WQ_ERR_INVALID_ARG;
    // The array keeps whatever the previous call left: re-zero the arrival
    // counters, which must start at zero.
    if (tiles > 0) {
        cudaError_t e = cudaMemsetAsync(d->scratch + counter_off, 0, counter_bytes, s);
        if (e != cudaSuccess) return wq::host_cuda_fail(e);
    }
    return wq_gemm(x, wq, scales, zeros, y, M, N, K, group, bits, d->scratch,
                   kNoAllocScratchBytes, stream);
}

extern "C" wq_status_t wq_check_noalloc(void* stream) {
    int dev = 0;
    NoAllocDevice* d = noalloc_entry(&dev);
    if (!d) return WQ_ERR_CUDA;
    unsigned char* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_noalloc_mu);
        if (!d->ready) return WQ_OK;  // no call on this device yet
        scratch = d->scratch;
    }
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return wq::host_cuda_fail(e);
    int word = 0;
    if ((e = cudaMemcpy(&word, scratch, sizeof word, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return wq::host_cuda_fail(e);
    if (word == 0) return WQ_OK;
    // A launch that gave up may also have left split-K counters behind: zero
    // the whole array (the next call re-zeroes its counters anyway).
    if ((e = cudaMemsetAsync(scratch, 0, kNoAllocScratchBytes, s)) != cudaSuccess ||
        (e = cudaStreamSynchronize(s)) != cudaSuccess)
        return wq::host_cuda_fail(e);
    return WQ_ERR_TIMEOUT;
}
