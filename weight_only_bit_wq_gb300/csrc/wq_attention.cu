// Decode attention over a paged q8_0 KV pool (OpenJet news page,
// "单张 RTX 3090 跑 4 个编码 agent": attention, each agent reading its own KV
// cache, is what grows with the agents in a decode step; the cache is one
// shared pool of 132K tokens in q8_0, managed in pages, a common system
// prompt stored once).
//
// First CUDA path: flash-decoding on the CUDA cores.  A CTA takes one
// (sequence, key/value head, slice of positions); its four warps walk the
// slice 32 positions at a time, one position per lane for the scores (the
// query vectors of the sequence's rows for the head's query heads sit in
// shared memory), then the values one position at a time across the warp
// (lane l owns dims 4l .. 4l + 3), with an online softmax per query vector.
// The four warps' states merge in shared memory in warp order, the slices'
// states in a second kernel in slice order: every result is deterministic.
//
// Layout: q bf16 [rows][Hq][128]; K and V codes int8 [pages][Hkv][T][128],
// binary16 scales [pages][Hkv][T][4] (q8_0: value = scale * code per block
// of 32 dims); page_table int32 [B][max_pages]; seq_len int32 [B]; row_seq,
// row_pos int32 [rows] (row i attends to positions 0 .. row_pos[i] of
// sequence row_seq[i]); out fp32 [rows][Hq][128].
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "wq.h"
#include "wq_internal.h"

namespace {

constexpr int kD = 128;          // head dimension
constexpr int kQB = 16;          // query vectors per pass
constexpr int kWarps = 4;
constexpr int kThreads = 32 * kWarps;
constexpr int kErrBadTable = 2;  // error word: a page or position outside the pool

__device__ __forceinline__ float half_bits(uint16_t h) { return __half2float(__ushort_as_half(h)); }
__device__ __forceinline__ float bf16_bits(uint16_t b) {
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

struct AttnArgs {
    const uint16_t* q;
    const int8_t* kc;
    const uint16_t* kd;
    const int8_t* vc;
    const uint16_t* vd;
    const int* page_table;
    const int* seq_len;
    const int* row_seq;
    const int* row_pos;
    int rows, B, max_pages, Hq, Hkv, T, pages;
    int splits, chunk;  // slices per sequence, positions per slice (a multiple of 128)
    float* part;        // [rows][Hq][splits][2 + kD]: running max, sum, weighted values
    int* err;
};

// Token t of sequence b: its page (or -1 when the table points outside the pool).
__device__ __forceinline__ long token_row(const AttnArgs& a, int b, int g, int t) {
    const int page = __ldg(a.page_table + static_cast<long>(b) * a.max_pages + t / a.T);
    if (page < 0 || page >= a.pages) return -1;
    return (static_cast<long>(page) * a.Hkv + g) * a.T + t % a.T;
}

__global__ void __launch_bounds__(kThreads) attn_split_kernel(const AttnArgs a) {
    __shared__ float qs[kQB][kD];
    __shared__ int q_row[kQB], q_head[kQB], q_pos[kQB];
    __shared__ float wm[kWarps][kQB], wl[kWarps][kQB];
    __shared__ float wacc[kWarps][kQB][kD];
    const int s = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int group = a.Hq / a.Hkv;
    const int L = __ldg(a.seq_len + b);
    if (L > a.splits * a.chunk || L > a.max_pages * a.T) {
        if (threadIdx.x == 0 && s == 0 && g == 0) atomicExch(a.err, kErrBadTable);
        return;
    }
    const int t0 = s * a.chunk;
    const int t1 = min(L, t0 + a.chunk);
    const float scale = rsqrtf(static_cast<float>(kD));
    // query vectors of this (sequence, key/value head), in row order, kQB at a time
    int next_row = 0;
    for (;;) {
        __syncthreads();
        if (threadIdx.x == 0) {
            int n = 0;
            int i = next_row;
            for (; i < a.rows && n + group <= kQB; ++i) {
                if (__ldg(a.row_seq + i) != b) continue;
                const int pos = __ldg(a.row_pos + i);
                const bool ok = pos >= 0 && pos < L;
                if (!ok) atomicExch(a.err, kErrBadTable);
                for (int hh = 0; hh < group; ++hh) {
                    q_row[n] = i;
                    q_head[n] = g * group + hh;
                    q_pos[n] = ok ? pos : -1;  // a bad row attends to nothing
                    ++n;
                }
            }
            next_row = i;
            for (int j = n; j < kQB; ++j) {
                q_row[j] = -1;
                q_head[j] = 0;
                q_pos[j] = -1;
            }
        }
        __syncthreads();
        // every thread counts this pass's query vectors from the shared list
        int qn = 0;
        for (int j = 0; j < kQB; ++j) qn += q_row[j] >= 0 ? 1 : 0;
        if (qn == 0) break;
        for (int e = threadIdx.x; e < kQB * kD; e += kThreads) {
            const int j = e / kD, d = e % kD;
            qs[j][d] = q_row[j] >= 0
                           ? bf16_bits(__ldg(a.q + (static_cast<long>(q_row[j]) * a.Hq + q_head[j]) * kD + d))
                           : 0.f;
        }
        __syncthreads();
        float m[kQB], l[kQB], acc[kQB][4];
#pragma unroll
        for (int j = 0; j < kQB; ++j) {
            m[j] = -INFINITY;
            l[j] = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
        }
        for (int base = t0 + 32 * warp; base < t1; base += 32 * kWarps) {
            const int t = base + lane;
            float sc[kQB];
#pragma unroll
            for (int j = 0; j < kQB; ++j) sc[j] = 0.f;
            long row = t < t1 ? token_row(a, b, g, t) : -1;
            if (t < t1 && row < 0) atomicExch(a.err, kErrBadTable);
            if (row >= 0) {
                const int4* kr = reinterpret_cast<const int4*>(a.kc + row * kD);
                const uint16_t* ks = a.kd + row * (kD / 32);
#pragma unroll
                for (int c = 0; c < kD / 16; ++c) {
                    const int4 w = __ldg(kr + c);
                    const float dsc = half_bits(__ldg(ks + c / 2));
                    const int8_t* cb = reinterpret_cast<const int8_t*>(&w);
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float kv = dsc * static_cast<float>(cb[e]);
#pragma unroll
                        for (int j = 0; j < kQB; ++j) sc[j] = fmaf(qs[j][16 * c + e], kv, sc[j]);
                    }
                }
            }
            // scores, causal mask, running maxima
#pragma unroll
            for (int j = 0; j < kQB; ++j) {
                sc[j] = (row >= 0 && t <= q_pos[j]) ? sc[j] * scale : -INFINITY;
                float mx = sc[j];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float mn = fmaxf(m[j], mx);
                const float keep = mn == -INFINITY ? 1.f : expf(m[j] - mn);
                const float p = sc[j] == -INFINITY ? 0.f : expf(sc[j] - mn);
                float ps = p;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
                l[j] = l[j] * keep + ps;
#pragma unroll
                for (int e = 0; e < 4; ++e) acc[j][e] *= keep;
                m[j] = mn;
                sc[j] = p;  // from here on: this lane's probability for vector j
            }
            // values: position base + tt across the warp, lane l owning dims 4l .. 4l + 3
            for (int tt = 0; tt < 32; ++tt) {
                const long vrow = __shfl_sync(0xffffffffu, row, tt);
                if (vrow < 0) continue;
                const int code4 = __ldg(reinterpret_cast<const int*>(a.vc + vrow * kD) + lane);
                const float dsc = half_bits(__ldg(a.vd + vrow * (kD / 32) + lane / 8));
                const int8_t* cb = reinterpret_cast<const int8_t*>(&code4);
                float v[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) v[e] = dsc * static_cast<float>(cb[e]);
#pragma unroll
                for (int j = 0; j < kQB; ++j) {
                    const float p = __shfl_sync(0xffffffffu, sc[j], tt);
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[j][e] = fmaf(p, v[e], acc[j][e]);
                }
            }
        }
        // merge the warps in warp order
#pragma unroll
        for (int j = 0; j < kQB; ++j) {
            if (lane == 0) {
                wm[warp][j] = m[j];
                wl[warp][j] = l[j];
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) wacc[warp][j][4 * lane + e] = acc[j][e];
        }
        __syncthreads();
        for (int e = threadIdx.x; e < kQB * kD; e += kThreads) {
            const int j = e / kD, d = e % kD;
            if (q_row[j] < 0) continue;
            float mt = -INFINITY;
            for (int w = 0; w < kWarps; ++w) mt = fmaxf(mt, wm[w][j]);
            float lt = 0.f, at = 0.f;
            for (int w = 0; w < kWarps; ++w) {
                const float f = wm[w][j] == -INFINITY ? 0.f : expf(wm[w][j] - mt);
                lt += f * wl[w][j];
                at += f * wacc[w][j][d];
            }
            float* dst = a.part + ((static_cast<long>(q_row[j]) * a.Hq + q_head[j]) * a.splits + s) * (2 + kD);
            if (d == 0) {
                dst[0] = mt;
                dst[1] = lt;
            }
            dst[2 + d] = at;
        }
    }
}

// out[i][h] = (sum over slices of e^(m_s - m) acc_s) / (sum of e^(m_s - m) l_s), slices in order.
__global__ void __launch_bounds__(kD) attn_combine_kernel(const float* part, int splits, int Hq,
                                                          float* out) {
    const long vec = blockIdx.x;  // row * Hq + head
    const int d = threadIdx.x;
    const float* p = part + vec * splits * (2 + kD);
    float mt = -INFINITY;
    for (int s = 0; s < splits; ++s) mt = fmaxf(mt, p[s * (2 + kD)]);
    float lt = 0.f, at = 0.f;
    for (int s = 0; s < splits; ++s) {
        const float ms = p[s * (2 + kD)];
        const float f = ms == -INFINITY ? 0.f : expf(ms - mt);
        lt += f * p[s * (2 + kD) + 1];
        at += f * p[s * (2 + kD) + 2 + d];
    }
    out[vec * kD + d] = lt > 0.f ? at / lt : 0.f;
}

int splits_for(int max_seq_len, int* chunk) {
    // slices of at least 512 positions, at most 64 per sequence
    int splits = (max_seq_len + 511) / 512;
    if (splits > 64) splits = 64;
    if (splits < 1) splits = 1;
    int c = (max_seq_len + splits - 1) / splits;
    c = (c + 127) / 128 * 128;
    *chunk = c;
    return splits;
}

bool aligned(const void* p, size_t n) { return reinterpret_cast<uintptr_t>(p) % n == 0; }

}  // namespace

extern "C" {

size_t wq_paged_attention_workspace_bytes(int rows, int Hq, int max_seq_len) {
    if (rows < 0 || Hq <= 0 || max_seq_len <= 0) return 0;
    int chunk = 0;
    const int splits = splits_for(max_seq_len, &chunk);
    return wq::kWsHeader + static_cast<size_t>(rows) * Hq * splits * (2 + kD) * sizeof(float);
}

wq_status_t wq_paged_attention(const uint16_t* q, const int8_t* k_codes, const uint16_t* k_scales,
                               const int8_t* v_codes, const uint16_t* v_scales,
                               const int* page_table, int max_pages, const int* seq_len, int B,
                               const int* row_seq, const int* row_pos, int rows, int max_seq_len,
                               int Hq, int Hkv, int D, int T, int pages, float* out,
                               void* workspace, size_t workspace_bytes, void* stream) {
    if (D != kD || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Hq / Hkv > kQB || T <= 0 ||
        pages <= 0 || B <= 0 || max_pages <= 0 || rows < 0 || max_seq_len <= 0 ||
        max_seq_len > max_pages * T)
        return WQ_ERR_INVALID_ARG;
    if (rows == 0) return WQ_OK;
    if (!q || !k_codes || !k_scales || !v_codes || !v_scales || !page_table || !seq_len ||
        !row_seq || !row_pos || !out || !workspace)
        return WQ_ERR_INVALID_ARG;
    if (!aligned(k_codes, 16) || !aligned(v_codes, 16) || !aligned(out, 4) ||
        workspace_bytes < wq_paged_attention_workspace_bytes(rows, Hq, max_seq_len) ||
        !aligned(workspace, 16))
        return WQ_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    AttnArgs a;
    a.q = q;
    a.kc = k_codes;
    a.kd = k_scales;
    a.vc = v_codes;
    a.vd = v_scales;
    a.page_table = page_table;
    a.seq_len = seq_len;
    a.row_seq = row_seq;
    a.row_pos = row_pos;
    a.rows = rows;
    a.B = B;
    a.max_pages = max_pages;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.T = T;
    a.pages = pages;
    a.splits = splits_for(max_seq_len, &a.chunk);
    a.err = static_cast<int*>(workspace);
    a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + wq::kWsHeader);
    // every (row, head, slice) state is written: rows of other sequences are
    // never read, and empty slices write m = -inf, l = 0
    cudaError_t e = cudaMemsetAsync(a.part, 0, static_cast<size_t>(rows) * Hq * a.splits * (2 + kD) * sizeof(float), s);
    if (e != cudaSuccess) return WQ_ERR_CUDA;
    attn_split_kernel<<<dim3(a.splits, Hkv, B), kThreads, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return WQ_ERR_CUDA;
    attn_combine_kernel<<<static_cast<unsigned>(rows * Hq), kD, 0, s>>>(a.part, a.splits, Hq, out);
    return cudaGetLastError() == cudaSuccess ? WQ_OK : WQ_ERR_CUDA;
}

}  // extern "C"
