// C ABI of libwq: argument checks, device queries, tensor maps, workspace and
// dispatch.  Every check happens on the host before any launch; kernels never
// trap.
#include <cudaTypedefs.h>

#include <cstring>
#include <deque>
#include <mutex>

#include "wq.h"
#include "wq_internal.h"

namespace {

thread_local int g_last_cuda_error = 0;

wq_status_t cuda_fail(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return WQ_ERR_CUDA;
}

struct DeviceInfo {
    bool ready = false;
    int sm_count = 0;
    int major = 0, minor = 0;
    void* lib_ws = nullptr;  // library-owned gemm workspace
    size_t lib_ws_bytes = 0;
};

std::mutex g_mu;
// A deque: growing it for a new device keeps earlier entries in place, so a
// DeviceInfo* handed out for one device stays valid while another thread
// registers a second device.
std::deque<DeviceInfo> g_dev;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

wq_status_t device_info(DeviceInfo** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    std::lock_guard<std::mutex> lock(g_mu);
    if (static_cast<int>(g_dev.size()) <= dev) g_dev.resize(dev + 1);
    DeviceInfo& d = g_dev[dev];
    if (!d.ready) {
        if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
            (e = cudaDeviceGetAttribute(&d.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
            return cuda_fail(e);
        d.ready = true;
    }
    if (!(d.major == 10 && d.minor == 3)) return WQ_ERR_UNSUPPORTED;  // built for sm_103a only
    *out = &d;
    return WQ_OK;
}

wq_status_t get_encoder() {
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_encode) return WQ_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess) return cuda_fail(e);
    if (q != cudaDriverEntryPointSuccess || fn == nullptr) return WQ_ERR_UNSUPPORTED;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return WQ_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool valid_bits(int bits) { return bits == 2 || bits == 3 || bits == 4; }
bool valid_group(int g) { return g == 32 || g == 64 || g == 128; }

// Split-K layout inside a workspace.
struct WsLayout {
    size_t partial_off, counter_off, bytes;
};

WsLayout ws_layout(int T, int sm_count) {
    WsLayout l;
    l.partial_off = wq::kWsHeader;
    const size_t partial_bytes =
        static_cast<size_t>(2) * sm_count * wq::kMaxCols * wq::kBN * sizeof(float);
    l.counter_off = l.partial_off + partial_bytes;
    l.bytes = (l.counter_off + static_cast<size_t>(T) * wq::kCountersPerTile * sizeof(int) + 255) /
              256 * 256;
    return l;
}

cudaStream_t as_stream(void* s) { return reinterpret_cast<cudaStream_t>(s); }

}  // namespace

namespace wq {

int aligned_grid(int T, int budget, bool split_tiles) {
    if (T <= 0 || budget <= 0) return budget;
    const int lo = budget * 74 / 100;
    if (T <= budget) {
        const int k = budget / T;
        return split_tiles && k * T >= lo ? k * T : budget;
    }
    for (int P = budget; P >= lo && P > 0; --P)
        if (T % P == 0) return P;
    return budget;
}

// Measured on 34,816 x 5,120 at 12 rows: 136 CTAs of two whole tiles each run
// in 23.9 us against 25.3 us for 150 CTAs with split tiles (3-bit: 32.2
// against 36.6 us).
int choose_grid(int T, int I, int sm_count) {
    const long long U = static_cast<long long>(T) * I;
    long long P = aligned_grid(T, gemm_sm_budget(sm_count), false);
    if (P > U) P = U;
    const long long cap = static_cast<long long>(T) * kMaxSplit;
    if (P > cap) P = cap;
    return P < 1 ? 1 : static_cast<int>(P);
}

}  // namespace wq

extern "C" {

int wq_abi_version(void) { return 104; }

const char* wq_status_string(wq_status_t s) {
    switch (s) {
        case WQ_OK: return "ok";
        case WQ_ERR_INVALID_ARG: return "invalid argument";
        case WQ_ERR_UNSUPPORTED: return "unsupported device or feature";
        case WQ_ERR_CUDA: return "CUDA runtime error";
        case WQ_ERR_TIMEOUT: return "kernel abandoned a bounded wait";
    }
    return "unknown status";
}

int wq_last_cuda_error(void) { return g_last_cuda_error; }

long wq_packed_words_per_row(int K, int bits) {
    if (!valid_bits(bits) || K < 0) return -1;
    const long vpw = wq::values_per_word(bits);
    const long used = (static_cast<long>(K) + vpw - 1) / vpw;
    return (used + 3) / 4 * 4;
}

}  // extern "C"

// ---------------------------------------------------------------- elementwise
extern "C" {

wq_status_t wq_pack(const uint8_t* q, uint32_t* wq, int N, int K, int bits, void* stream) {
    if (!valid_bits(bits) || N < 0 || K < 0) return WQ_ERR_INVALID_ARG;
    const long W = wq_packed_words_per_row(K, bits);
    if (static_cast<long long>(N) * W == 0) return WQ_OK;
    if (!wq || (!q && K > 0) || !aligned(wq, 4)) return WQ_ERR_INVALID_ARG;
    DeviceInfo* d;
    if (wq_status_t st = device_info(&d)) return st;
    cudaError_t e = wq::launch_pack(q, wq, N, K, bits, static_cast<int>(W), d->sm_count, as_stream(stream));
    return e == cudaSuccess ? WQ_OK : cuda_fail(e);
}

wq_status_t wq_unpack(const uint32_t* wq, uint8_t* q, int N, int K, int bits, void* stream) {
    if (!valid_bits(bits) || N < 0 || K < 0) return WQ_ERR_INVALID_ARG;
    if (static_cast<long long>(N) * K == 0) return WQ_OK;
    if (!wq || !q || !aligned(wq, 4)) return WQ_ERR_INVALID_ARG;
    DeviceInfo* d;
    if (wq_status_t st = device_info(&d)) return st;
    const long W = wq_packed_words_per_row(K, bits);
    cudaError_t e = wq::launch_unpack(wq, q, N, K, bits, static_cast<int>(W), d->sm_count, as_stream(stream));
    return e == cudaSuccess ? WQ_OK : cuda_fail(e);
}

wq_status_t wq_dequant(const uint32_t* wq, const uint16_t* scales, const uint8_t* zeros,
                       uint16_t* w, int N, int K, int group, int bits, void* stream) {
    if (!valid_bits(bits) || !valid_group(group) || N < 0 || K < 0 || K % group != 0)
        return WQ_ERR_INVALID_ARG;
    if (static_cast<long long>(N) * K == 0) return WQ_OK;
    if (!wq || !scales || !zeros || !w || !aligned(wq, 4) || !aligned(scales, 2) || !aligned(w, 2))
        return WQ_ERR_INVALID_ARG;
    DeviceInfo* d;
    if (wq_status_t st = device_info(&d)) return st;
    const long W = wq_packed_words_per_row(K, bits);
    cudaError_t e = wq::launch_dequant(wq, scales, zeros, w, N, K, group, bits, static_cast<int>(W),
                                       d->sm_count, as_stream(stream));
    return e == cudaSuccess ? WQ_OK : cuda_fail(e);
}

// ----------------------------------------------------------------------- gemm
size_t wq_workspace_bytes(int M, int N, int K, int group, int bits) {
    if (!valid_bits(bits) || !valid_group(group) || M < 0 || M > wq::kMaxCols || N < 0 || K < 0 ||
        K % group != 0)
        return 0;
    DeviceInfo* d;
    if (device_info(&d) != WQ_OK) return 0;
    const int T = (N + wq::kBN - 1) / wq::kBN;
    return ws_layout(T, d->sm_count).bytes;
}

size_t wq_workspace_bytes_for(int M, int N, int K, int group, int bits, int sm_count) {
    if (!valid_bits(bits) || !valid_group(group) || M < 0 || M > wq::kMaxCols || N < 0 || K < 0 ||
        K % group != 0 || sm_count <= 0)
        return 0;
    const int T = (N + wq::kBN - 1) / wq::kBN;
    return ws_layout(T, sm_count).bytes;
}

wq_status_t wq_workspace_init(void* workspace, size_t bytes, void* stream) {
    if (!workspace || bytes < wq::kWsHeader) return WQ_ERR_INVALID_ARG;
    cudaError_t e = cudaMemsetAsync(workspace, 0, bytes, as_stream(stream));
    return e == cudaSuccess ? WQ_OK : cuda_fail(e);
}

}  // extern "C"

namespace {

// X as one 3-D box per stage: dims {64 values, M rows, K/64 chunks}, the
// chunk stride 128 bytes, so a box of {64, nc, c} lands in shared memory as c
// consecutive [nc rows][128 bytes] swizzled tiles.  Requires K % 64 == 0 (a
// partial chunk would alias the next row instead of reading zeros).
wq_status_t encode_x3d(const uint16_t* x, int M, int K, int chunks, int nc, CUtensorMap* tmX) {
    const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(M), static_cast<cuuint64_t>(K / 64)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(K) * 2, 128};
    const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(nc), static_cast<cuuint32_t>(chunks)};
    const cuuint32_t es[3] = {1, 1, 1};
    CUresult r = g_encode(tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<uint16_t*>(x), dims,
                          strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? WQ_OK : WQ_ERR_INVALID_ARG;
}

wq_status_t encode_maps(const uint16_t* x, const uint32_t* wq, int M, int N, int K, int W,
                        int nc, CUtensorMap* tmW, CUtensorMap* tmX) {
    if (wq_status_t st = get_encoder()) return st;
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(W), static_cast<cuuint64_t>(N)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(W) * 4};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(wq::kWordsPerStage),
                                   static_cast<cuuint32_t>(wq::kBN)};
        const cuuint32_t es[2] = {1, 1};
        CUresult r = g_encode(tmW, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<uint32_t*>(wq), dims,
                              strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return WQ_ERR_INVALID_ARG;
    }
    {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(K) * 2};
        const cuuint32_t box[2] = {64, static_cast<cuuint32_t>(nc)};
        const cuuint32_t es[2] = {1, 1};
        CUresult r = g_encode(tmX, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims,
                              strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (r != CUDA_SUCCESS) return WQ_ERR_INVALID_ARG;
    }
    return WQ_OK;
}

// Library-owned workspace of the current device, grown (and zeroed) on demand.
wq_status_t library_workspace(DeviceInfo* d, size_t need, void** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (d->lib_ws_bytes < need) {
        cudaError_t e;
        if (d->lib_ws) {
            if ((e = cudaDeviceSynchronize()) != cudaSuccess) return cuda_fail(e);
            cudaFree(d->lib_ws);
            d->lib_ws = nullptr;
            d->lib_ws_bytes = 0;
        }
        const size_t bytes = need < (size_t(4) << 20) ? (size_t(4) << 20) : need;
        if ((e = cudaMalloc(&d->lib_ws, bytes)) != cudaSuccess) return cuda_fail(e);
        if ((e = cudaMemset(d->lib_ws, 0, bytes)) != cudaSuccess) return cuda_fail(e);
        d->lib_ws_bytes = bytes;
    }
    *out = d->lib_ws;
    return WQ_OK;
}

}  // namespace

namespace wq {

wq_status_t host_cuda_fail(cudaError_t e) { return cuda_fail(e); }

wq_status_t host_sm_count(int* sms) {
    DeviceInfo* d;
    if (wq_status_t st = device_info(&d)) return st;
    *sms = d->sm_count;
    return WQ_OK;
}

wq_status_t host_check_gemm(const uint16_t* x, const uint32_t* wq, const uint16_t* scales,
                            const uint8_t* zeros, const void* y, int M, int N, int K, int group,
                            int bits, int epi) {
    if (!valid_bits(bits) || !valid_group(group) || M < 0 || M > kMaxCols || N < 0 || K < 0 ||
        K % group != 0)
        return WQ_ERR_INVALID_ARG;
    if (epi != WQ_EPI_NONE && epi != WQ_EPI_SWIGLU) return WQ_ERR_INVALID_ARG;
    if (epi == WQ_EPI_SWIGLU && N % 2 != 0) return WQ_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return WQ_OK;
    if (!y || !aligned(y, epi == WQ_EPI_SWIGLU ? 2 : 4)) return WQ_ERR_INVALID_ARG;
    if (K == 0) return WQ_OK;
    if (!x || !wq || !scales || !zeros || !aligned(x, 16) || !aligned(wq, 16) || !aligned(scales, 2))
        return WQ_ERR_INVALID_ARG;
    return WQ_OK;
}

wq_status_t host_encode_proj(const uint16_t* x, const uint32_t* wq, const uint16_t* scales,
                             const uint8_t* zeros, int M, int N, int K, int group, int bits,
                             int nc, CUtensorMap* tmW, CUtensorMap* tmX, int* x3d,
                             int* meta_vec) {
    const int W = static_cast<int>(wq_packed_words_per_row(K, bits));
    const int sv = tc_stage_values(bits, group);
    if (wq_status_t st = encode_maps(x, wq, M, N, K, W, nc, tmW, tmX)) return st;
    *x3d = K % 64 == 0 ? 1 : 0;
    if (*x3d)
        if (wq_status_t st = encode_x3d(x, M, K, sv / 64, nc, tmX)) return st;
    const int ng = K / group;
    const int gps = sv / group;
    const bool gps_pow2 = (gps & (gps - 1)) == 0;
    *meta_vec = (gps_pow2 && ng % gps == 0 && aligned(scales, 16) && aligned(zeros, 16)) ? 1 : 0;
    return WQ_OK;
}

}  // namespace wq

namespace wq {

wq_status_t gemm_run(const uint16_t* x, const uint32_t* wq, const uint16_t* scales,
                     const uint8_t* zeros, void* y, int M, int N, int K, int group, int bits,
                     void* workspace, size_t workspace_bytes, cudaStream_t s, bool pdl,
                     int epi) {
    if (wq_status_t st = host_check_gemm(x, wq, scales, zeros, y, M, N, K, group, bits, epi))
        return st;
    if (M == 0 || N == 0) return WQ_OK;

    if (K == 0) {  // empty sum: fp32 zeros, or silu(0) * 0 = +0 in bf16
        const size_t bytes = epi == WQ_EPI_SWIGLU ? static_cast<size_t>(M) * (N / 2) * 2
                                                  : static_cast<size_t>(M) * N * sizeof(float);
        cudaError_t e = cudaMemsetAsync(y, 0, bytes, s);
        return e == cudaSuccess ? WQ_OK : cuda_fail(e);
    }
    DeviceInfo* d;
    if (wq_status_t st = device_info(&d)) return st;

    const int T = (N + wq::kBN - 1) / wq::kBN;
    const int sv = wq::tc_stage_values(bits, group);
    const int I = (K + sv - 1) / sv;
    const WsLayout lay = ws_layout(T, d->sm_count);
    void* ws = workspace;
    if (!ws) {
        if (wq_status_t st = library_workspace(d, lay.bytes, &ws)) return st;
    } else if (workspace_bytes < lay.bytes || !aligned(workspace, 16)) {
        return WQ_ERR_INVALID_ARG;
    }

    CUtensorMap tmW, tmX;
    wq::GemmArgs a;
    a.nc = wq::tc_cols(M);
    if (wq_status_t st = wq::host_encode_proj(x, wq, scales, zeros, M, N, K, group, bits, a.nc,
                                              &tmW, &tmX, &a.x3d, &a.meta_vec))
        return st;
    a.scales = scales;
    a.zeros = zeros;
    a.y = static_cast<float*>(y);
    a.epi = epi;
    uint8_t* wsb = static_cast<uint8_t*>(ws);
    a.err = reinterpret_cast<int*>(wsb);
    a.partials = reinterpret_cast<float*>(wsb + lay.partial_off);
    a.counters = reinterpret_cast<int*>(wsb + lay.counter_off);
    a.M = M;
    a.N = N;
    a.K = K;
    a.ng = K / group;
    a.T = T;
    a.I = I;
    a.U = static_cast<long long>(T) * I;
    a.P = wq::choose_grid(T, I, d->sm_count);
    a.pdl = pdl ? 1 : 0;

    cudaError_t e;
    if (bits == 4)
        e = wq::launch_gemm_tc_b4(group, tmW, tmX, a, s);
    else if (bits == 3)
        e = wq::launch_gemm_tc_b3(group, tmW, tmX, a, s);
    else
        e = wq::launch_gemm_tc_b2(group, tmW, tmX, a, s);
    if (e == cudaErrorNotSupported) return WQ_ERR_UNSUPPORTED;
    return e == cudaSuccess ? WQ_OK : cuda_fail(e);
}

}  // namespace wq

extern "C" {

wq_status_t wq_gemm(const uint16_t* x, const uint32_t* wq, const uint16_t* scales,
                    const uint8_t* zeros, float* y, int M, int N, int K, int group, int bits,
                    void* workspace, size_t workspace_bytes, void* stream) {
    return wq::gemm_run(x, wq, scales, zeros, y, M, N, K, group, bits, workspace, workspace_bytes,
                        as_stream(stream), false, WQ_EPI_NONE);
}

wq_status_t wq_gemm_swiglu(const uint16_t* x, const uint32_t* wq, const uint16_t* scales,
                           const uint8_t* zeros, uint16_t* y, int M, int N, int K, int group,
                           int bits, void* workspace, size_t workspace_bytes, void* stream) {
    return wq::gemm_run(x, wq, scales, zeros, y, M, N, K, group, bits, workspace, workspace_bytes,
                        as_stream(stream), false, WQ_EPI_SWIGLU);
}
wq_status_t wq_check_workspace(void* workspace, void* stream) {
    void* ws = workspace;
    if (!ws) {
        DeviceInfo* d;
        if (wq_status_t st = device_info(&d)) return st;
        ws = d->lib_ws;
        if (!ws) return WQ_OK;
    }
    cudaError_t e = cudaStreamSynchronize(as_stream(stream));
    if (e != cudaSuccess) return cuda_fail(e);
    int word = 0;
    if ((e = cudaMemcpy(&word, ws, sizeof word, cudaMemcpyDeviceToHost)) != cudaSuccess) return cuda_fail(e);
    if (word == 0) return WQ_OK;
    // A launch that gave up may have left split-K counters behind: the
    // library buffer is zeroed whole; a caller's workspace gets its error
    // word cleared and must be zeroed again (wq_workspace_init) before reuse.
    DeviceInfo* d = nullptr;
    if (!workspace && device_info(&d) == WQ_OK && d->lib_ws == ws) {
        if ((e = cudaMemset(ws, 0, d->lib_ws_bytes)) != cudaSuccess) return cuda_fail(e);
    } else {
        const int zero = 0;
        if ((e = cudaMemcpy(ws, &zero, sizeof zero, cudaMemcpyHostToDevice)) != cudaSuccess)
            return cuda_fail(e);
    }
    return WQ_ERR_TIMEOUT;
}

// Host-only view of the single-projection grid rule (used by the CPU tests).
int wq_internal_choose_grid(int T, int I, int sm_count) { return wq::choose_grid(T, I, sm_count); }

// Host-only self check of the stream-K schedule (used by the CPU tests):
// returns 0 when every unit of [0, U) belongs to exactly one CTA and the
// closed-form owner of each unit matches the ranges.
int wq_internal_schedule_check(long long U, int P) {
    if (U <= 0 || P <= 0 || P > U) return 1;
    for (int b = 0; b < P; ++b) {
        const long long lo = wq::unit_begin(U, P, b), hi = wq::unit_begin(U, P, b + 1);
        if (hi <= lo) return 2;
        for (long long u = lo; u < hi; ++u) {
            const long long owner = ((u + 1) * P + U - 1) / U - 1;
            if (owner != b) return 3;
        }
    }
    return wq::unit_begin(U, P, P) == U ? 0 : 4;
}

}  // extern "C"
