// Decode attention over a paged q8_0 KV pool (OpenJet news page,
// "单张 RTX 3090 跑 4 个编码 agent": attention, each agent reading its own KV
// cache, is what grows with the agents in a decode step; the cache is one
// shared pool of 132K tokens in q8_0, managed in pages, a common system
// prompt stored once).
//
// Two split kernels with one structure; the entry point runs the tensor-core
// one (described above attn_split_tc_kernel), and the CUDA-core one is kept as
// an independent cross-check.  CUDA-core kernel: flash-decoding.  A CTA takes one
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
#include "wq_ptx.cuh"

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

// ------------------------------------------------------------ tensor-core path
// The same CTA, slice and pass structure on the tensor cores (mma.sync
// m16n8k16, binary16 operands, fp32 accumulators).  Each warp takes 16
// positions at a time:
//   scores  S[16 query vectors][8 positions] per n-tile, k running over head
//           dims.  The query vectors are multiplied by a power of two 2^eq
//           (per pass) that puts the largest in [2^14, 2^15), so every bf16
//           query value is exact in binary16 unless it is 2^-32 times smaller
//           than the largest; the codes are exact in binary16.  Each 32-dim
//           block is summed on its own and multiplied by its position's scale
//           in fp32 (the scale varies along positions, the n side).
//   values  O[16 query vectors][8 dims] per n-tile, k running over the 16
//           positions.  The value scale varies along k, so it goes into A: for
//           the n-tile's 32-dim block, A = p * scale * 2^ev, with 2^ev keeping
//           the chunk's largest scale below 2^15, split into its binary16
//           rounding and the binary16 rounding of the remainder (two MMAs,
//           about 22 significant bits); O carries 2^ev until the end.
// The head dims are assigned to k (and, for the values, to n) in a permuted
// order so that each lane's codes come from one 8-byte (keys) or 4-byte
// (values) shared-memory read: for k-step 2 * blk + hh, lane quad position c holds k =
// 2c, 2c + 1 as dims 32 blk + 8c + 4hh + {0, 1} and k = 2c + 8, 2c + 9 as
// dims 32 blk + 8c + 4hh + {2, 3}, the same for the query vectors (A) and the
// keys (B); value n-tile 4 blk + j holds n = lane group r as dim 32 blk + 4r + j.

constexpr float kInvSqrtD = 0.0883883476483184405f;  // 1 / sqrt(128), correctly rounded

__device__ __forceinline__ void mma_f16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                        uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two codes of `u` (four codes with their sign bits flipped, i.e. code + 128
// as unsigned bytes) as binary16x2, exactly: `sel` moves the two bytes into
// the low mantissa bytes of 1024.0 (0x64 high bytes), giving 1024 + code + 128,
// and subtracting 1152 leaves the code.  sel 0x4140: bytes 0 and 1; 0x4342:
// bytes 2 and 3 (the lower-numbered byte in the low half).
__device__ __forceinline__ uint32_t codes_f16x2(uint32_t u, uint32_t sel) {
    const uint32_t h = __byte_perm(u, 0x64646464u, sel);
    const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h),
                              __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480)));
    return *reinterpret_cast<const uint32_t*>(&r);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    const __half2 r = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&r);
}

// Binary16 rounding of x and of what it leaves: hi + lo carries ~22 bits of x.
__device__ __forceinline__ void split_f16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __half2 h = __floats2half2_rn(x0, x1);
    const float2 hf = __half22float2(h);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = pack_f16x2(x0 - hf.x, x1 - hf.y);
}

// 2^e for -126 <= e <= 127, exactly.
__device__ __forceinline__ float pow2i(int e) { return __uint_as_float(static_cast<uint32_t>(e + 127) << 23); }

// floor(log2 x) for a positive normal x.
__device__ __forceinline__ int ilog2f(float x) {
    return static_cast<int>((__float_as_uint(x) >> 23) & 0xffu) - 127;
}

__device__ __forceinline__ float scale_of(uint2 w, int blk) {
    const uint32_t v = blk < 2 ? w.x : w.y;
    return half_bits(static_cast<uint16_t>((blk & 1) ? (v >> 16) : (v & 0xffffu)));
}

// A warp's copy stage: 16 positions of K codes and of V codes (128-byte rows
// whose 16-byte pieces are stored XOR-swizzled by the row, so that the lanes'
// fragment reads hit distinct banks), then their K and V scale quadruples.
constexpr int kOffK = 0, kOffV = 16 * kD, kOffKS = 32 * kD, kOffVS = 32 * kD + 16 * 8;
constexpr int kStageBytes = 32 * kD + 2 * 16 * 8;
constexpr int kRingBytes = kWarps * 2 * kStageBytes;
constexpr int kWaccBytes = kWarps * kQB * kD * 4;
constexpr int kSbufBytes = kRingBytes > kWaccBytes ? kRingBytes : kWaccBytes;
__device__ __forceinline__ int swz(int piece, int row) { return piece ^ (row & 7); }

__global__ void __launch_bounds__(kThreads) attn_split_tc_kernel(const AttnArgs a) {
    __shared__ float qs[kQB][kD];
    __shared__ int q_row[kQB], q_head[kQB], q_pos[kQB];
    __shared__ float wm[kWarps][kQB], wl[kWarps][kQB];
    __shared__ float wmax[kWarps];
    // each warp's two-stage copy ring during the position loop, then the
    // warps' weighted values for the merge
    __shared__ __align__(16) unsigned char sbuf[kSbufBytes];
    float(*wacc)[kQB][kD] = reinterpret_cast<float(*)[kQB][kD]>(sbuf);
    const int s = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gr = lane >> 2, qc = lane & 3;  // lane group (row / n index) and position in the quad
    const int group = a.Hq / a.Hkv;
    const int L = __ldg(a.seq_len + b);
    if (L > a.splits * a.chunk || L > a.max_pages * a.T) {
        if (threadIdx.x == 0 && s == 0 && h == 0) atomicExch(a.err, kErrBadTable);
        return;
    }
    const int t0 = s * a.chunk;
    const int t1 = min(L, t0 + a.chunk);
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
                    q_head[n] = h * group + hh;
                    q_pos[n] = ok ? pos : -1;
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
        int qn = 0;
        for (int j = 0; j < kQB; ++j) qn += q_row[j] >= 0 ? 1 : 0;
        if (qn == 0) break;
        float qmax = 0.f;
        for (int e = threadIdx.x; e < kQB * kD; e += kThreads) {
            const int j = e / kD, d = e % kD;
            const float v = q_row[j] >= 0
                                ? bf16_bits(__ldg(a.q + (static_cast<long>(q_row[j]) * a.Hq + q_head[j]) * kD + d))
                                : 0.f;
            qs[j][d] = v;
            qmax = fmaxf(qmax, fabsf(v));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, o));
        if (lane == 0) wmax[warp] = qmax;
        __syncthreads();
        qmax = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
        // 2^eq puts the largest query value in [2^14, 2^15); zero or subnormal
        // maxima (nothing to scale) keep eq = 0
        const int eq = qmax >= 1.17549435e-38f ? max(-100, min(100, 14 - ilog2f(qmax))) : 0;
        const float qsc = ldexpf(1.f, eq);
        const float ssc = ldexpf(kInvSqrtD, -eq);  // undoes 2^eq and applies 1 / sqrt(D)
        uint32_t qa[8][4];
#pragma unroll
        for (int blk = 0; blk < 4; ++blk)
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int d0 = 32 * blk + 8 * qc + 4 * hh;
                uint32_t* f = qa[2 * blk + hh];
                f[0] = pack_f16x2(qs[gr][d0] * qsc, qs[gr][d0 + 1] * qsc);
                f[1] = pack_f16x2(qs[gr + 8][d0] * qsc, qs[gr + 8][d0 + 1] * qsc);
                f[2] = pack_f16x2(qs[gr][d0 + 2] * qsc, qs[gr][d0 + 3] * qsc);
                f[3] = pack_f16x2(qs[gr + 8][d0 + 2] * qsc, qs[gr + 8][d0 + 3] * qsc);
            }
        const int qp0 = q_pos[gr], qp1 = q_pos[gr + 8];
        float o[16][4];
#pragma unroll
        for (int n = 0; n < 16; ++n)
#pragma unroll
            for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
        float m0 = -INFINITY, m1 = -INFINITY;  // running maxima of rows gr and gr + 8
        float l0 = 0.f, l1 = 0.f;              // this lane's share of the running sums
        int ev = 64;                           // O holds 2^ev times the weighted values (64: not set yet)
        unsigned char* const ring = sbuf + warp * 2 * kStageBytes;
        // Copies one chunk (positions base .. base + 15) into stage st: pool
        // rows of the positions from lanes 0 .. 15, then four 16-byte pieces of
        // K and of V codes per lane (zero-filled for positions outside the
        // slice or the pool) and one 8-byte scale quadruple.  Returns the
        // chunk's readable positions as a bit mask.
        auto issue = [&](int base, int st) -> unsigned {
            long myrow = -1;
            if (lane < 16 && base + lane < t1) {
                myrow = token_row(a, b, h, base + lane);
                if (myrow < 0) atomicExch(a.err, kErrBadTable);
            }
            const unsigned vmask = __ballot_sync(0xffffffffu, myrow >= 0);
            const uint32_t sb = wq::smem_addr(ring + st * kStageBytes);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int c = lane + 32 * i;  // piece c: position c / 8, bytes 16 (c % 8) ..
                const int r = c >> 3, p = c & 7;
                const long row = __shfl_sync(0xffffffffu, myrow, r);
                const uint32_t off = static_cast<uint32_t>(r * kD + (swz(p, r) << 4));
                const long src = row >= 0 ? row * kD + 16 * p : 0;
                const uint32_t n = row >= 0 ? 16u : 0u;
                wq::cp_async_n<16>(sb + kOffK + off, a.kc + src, n);
                wq::cp_async_n<16>(sb + kOffV + off, a.vc + src, n);
            }
            {
                const int r = lane & 15;
                const long row = __shfl_sync(0xffffffffu, myrow, r);
                const uint16_t* src = (lane < 16 ? a.kd : a.vd) + (row >= 0 ? row * (kD / 32) : 0);
                wq::cp_async_n<8>(sb + (lane < 16 ? kOffKS : kOffVS) + 8 * r, src, row >= 0 ? 8u : 0u);
            }
            wq::cp_async_commit();
            return vmask;
        };
        const int step = 16 * kWarps;
        int base = t0 + 16 * warp;
        unsigned vm_cur = base < t1 ? issue(base, 0) : 0u;
        for (int it = 0; base < t1; ++it, base += step) {
            const int st = it & 1;
            // the next chunk's copies fly while this one is computed
            unsigned vm_next = 0u;
            if (base + step < t1)
                vm_next = issue(base + step, st ^ 1);
            else
                wq::cp_async_commit();  // an empty group keeps the count uniform
            wq::cp_async_wait<1>();
            __syncwarp();
            const unsigned char* sg = ring + st * kStageBytes;
            // this lane's positions (chunk-relative): keys n = gr of both
            // n-tiles; C fragment and value positions 2qc + {0, 1}, 8 + 2qc + {0, 1}
            int pj[4];
            pj[0] = 2 * qc;
            pj[1] = 2 * qc + 1;
            pj[2] = 8 + 2 * qc;
            pj[3] = 9 + 2 * qc;
            bool okj[4];
            uint2 ksc[4], vsc[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                okj[j] = ((vm_cur >> pj[j]) & 1u) != 0;
                ksc[j] = *reinterpret_cast<const uint2*>(sg + kOffKS + 8 * pj[j]);
                vsc[j] = *reinterpret_cast<const uint2*>(sg + kOffVS + 8 * pj[j]);
            }
            // scores: sv[nt][i] = C fragment element i of n-tile nt (rows gr, gr, gr + 8, gr + 8;
            // positions base + 8 nt + 2 qc + {0, 1, 0, 1})
            float sv[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                const int r = 8 * nt + gr;
#pragma unroll
                for (int e = 0; e < 4; ++e) sv[nt][e] = 0.f;
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) {
                    const uint2 kw = *reinterpret_cast<const uint2*>(
                        sg + kOffK + r * kD + (swz(2 * blk + (qc >> 1), r) << 4) + ((qc & 1) << 3));
                    float acc[4] = {0.f, 0.f, 0.f, 0.f};
                    const uint32_t u0 = kw.x ^ 0x80808080u, u1 = kw.y ^ 0x80808080u;
                    mma_f16(acc, qa[2 * blk], codes_f16x2(u0, 0x4140), codes_f16x2(u0, 0x4342));
                    mma_f16(acc, qa[2 * blk + 1], codes_f16x2(u1, 0x4140), codes_f16x2(u1, 0x4342));
                    const float d0 = scale_of(ksc[2 * nt], blk), d1 = scale_of(ksc[2 * nt + 1], blk);
                    sv[nt][0] = fmaf(acc[0], d0, sv[nt][0]);
                    sv[nt][1] = fmaf(acc[1], d1, sv[nt][1]);
                    sv[nt][2] = fmaf(acc[2], d0, sv[nt][2]);
                    sv[nt][3] = fmaf(acc[3], d1, sv[nt][3]);
                }
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = 2 * nt + (e & 1);                  // which of pj[]
                    const int t = base + 8 * nt + 2 * qc + (e & 1);  // its position
                    const int qp = e < 2 ? qp0 : qp1;
                    sv[nt][e] = (okj[j] && t <= qp) ? sv[nt][e] * ssc : -INFINITY;
                }
            }
            // online softmax per row: maxima over the chunk's 16 positions (own
            // four values, then the quad), rescale of the running state
            float mx0 = fmaxf(fmaxf(sv[0][0], sv[0][1]), fmaxf(sv[1][0], sv[1][1]));
            float mx1 = fmaxf(fmaxf(sv[0][2], sv[0][3]), fmaxf(sv[1][2], sv[1][3]));
#pragma unroll
            for (int o2 = 1; o2 <= 2; o2 <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
            }
            const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
            const float k0 = mn0 == -INFINITY ? 1.f : __expf(m0 - mn0);
            const float k1 = mn1 == -INFINITY ? 1.f : __expf(m1 - mn1);
            m0 = mn0;
            m1 = mn1;
            float p[2][4];
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float mr = e < 2 ? mn0 : mn1;
                    p[nt][e] = sv[nt][e] == -INFINITY ? 0.f : __expf(sv[nt][e] - mr);
                }
            l0 = l0 * k0 + (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]);
            l1 = l1 * k1 + (p[0][2] + p[0][3]) + (p[1][2] + p[1][3]);
            // the chunk's largest value scale sets 2^ev (only ever lowered; O follows)
            float dmax = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j)
#pragma unroll
                for (int blk = 0; blk < 4; ++blk) dmax = fmaxf(dmax, fabsf(scale_of(vsc[j], blk)));
#pragma unroll
            for (int o2 = 1; o2 <= 2; o2 <<= 1) dmax = fmaxf(dmax, __shfl_xor_sync(0xffffffffu, dmax, o2));
            // binary16 scales are at least 2^-24 when not zero
            const int ev_c = dmax > 0.f ? 14 - ilog2f(dmax) : 64;
            float r0 = k0, r1 = k1;
            if (ev_c < ev) {
                const float f = pow2i(max(ev_c - ev, -126));
                r0 *= f;
                r1 *= f;
                ev = ev_c;
            }
            // once the running maxima settle, most chunks leave O as it is
            // (multiplying by 1 would change nothing)
            if (__any_sync(0xffffffffu, r0 != 1.f || r1 != 1.f)) {
#pragma unroll
                for (int n = 0; n < 16; ++n) {
                    o[n][0] *= r0;
                    o[n][1] *= r0;
                    o[n][2] *= r1;
                    o[n][3] *= r1;
                }
            }
            const float evs = pow2i(min(ev, 127));
            // values, one 32-dim block at a time
#pragma unroll
            for (int blk = 0; blk < 4; ++blk) {
                float ds[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) ds[j] = scale_of(vsc[j], blk) * evs;
                // A: rows gr / gr + 8, k = 2qc, 2qc + 1 (positions pj[0], pj[1]) and
                // k = 2qc + 8, 2qc + 9 (pj[2], pj[3])
                uint32_t ah[4], al[4];
                split_f16x2(p[0][0] * ds[0], p[0][1] * ds[1], ah[0], al[0]);
                split_f16x2(p[0][2] * ds[0], p[0][3] * ds[1], ah[1], al[1]);
                split_f16x2(p[1][0] * ds[2], p[1][1] * ds[3], ah[2], al[2]);
                split_f16x2(p[1][2] * ds[2], p[1][3] * ds[3], ah[3], al[3]);
                // B: the four positions' codes at dims 32 blk + 4 gr + j, transposed
                // so that each 16-bit half holds two positions at one dim
                uint32_t u[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    u[j] = *reinterpret_cast<const uint32_t*>(
                               sg + kOffV + pj[j] * kD + (swz(2 * blk + (gr >> 2), pj[j]) << 4) +
                               ((gr & 3) << 2)) ^
                           0x80808080u;
                const uint32_t t01a = __byte_perm(u[0], u[1], 0x5140), t01b = __byte_perm(u[0], u[1], 0x7362);
                const uint32_t t23a = __byte_perm(u[2], u[3], 0x5140), t23b = __byte_perm(u[2], u[3], 0x7362);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint32_t lo = j < 2 ? t01a : t01b, hi = j < 2 ? t23a : t23b;
                    const uint32_t sel = (j & 1) ? 0x4342u : 0x4140u;
                    const uint32_t b0 = codes_f16x2(lo, sel), b1 = codes_f16x2(hi, sel);
                    mma_f16(o[4 * blk + j], ah, b0, b1);
                    mma_f16(o[4 * blk + j], al, b0, b1);
                }
            }
            __syncwarp();  // every lane has read stage st before it is refilled
            vm_cur = vm_next;
        }
        wq::cp_async_wait<0>();
        // this warp's state: maxima (uniform in the quad), sums over the quad,
        // O without its 2^ev
#pragma unroll
        for (int o2 = 1; o2 <= 2; o2 <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, o2);
            l1 += __shfl_xor_sync(0xffffffffu, l1, o2);
        }
        if (qc == 0) {
            wm[warp][gr] = m0;
            wm[warp][gr + 8] = m1;
            wl[warp][gr] = l0;
            wl[warp][gr + 8] = l1;
        }
        const float inv = pow2i(-min(ev, 126));
        __syncthreads();  // every warp is out of its copy ring before it becomes wacc
#pragma unroll
        for (int blk = 0; blk < 4; ++blk)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const int d = 32 * blk + 8 * qc + j;
                wacc[warp][gr][d] = o[4 * blk + j][0] * inv;
                wacc[warp][gr][d + 4] = o[4 * blk + j][1] * inv;
                wacc[warp][gr + 8][d] = o[4 * blk + j][2] * inv;
                wacc[warp][gr + 8][d + 4] = o[4 * blk + j][3] * inv;
            }
        __syncthreads();
        // merge the warps in warp order (as the CUDA-core kernel)
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

// Slices per sequence: one wave of CTAs over the grid (slots = SMs x the
// tensor-core kernel's resident CTAs per SM), no slice under 256 positions,
// at most 64; the slice length rounded up to 128 positions (whole iterations
// of the CUDA-core kernel's four warps of 32 positions).
int splits_for(int max_seq_len, int B, int Hkv, int slots, int* chunk) {
    const long long heads = static_cast<long long>(B) * Hkv;
    long long want = slots / (heads > 0 ? heads : 1);
    const long long most = (static_cast<long long>(max_seq_len) + 255) / 256;
    if (want > most) want = most;
    if (want > 64) want = 64;
    if (want < 1) want = 1;
    long long c = (max_seq_len + want - 1) / want;
    c = (c + 127) / 128 * 128;
    *chunk = static_cast<int>(c);
    return static_cast<int>((max_seq_len + c - 1) / c);
}

// CTAs the device holds at once: SMs x resident tensor-core split CTAs per SM.
wq_status_t grid_slots(int* slots) {
    int sms = 0;
    if (wq_status_t st = wq::host_sm_count(&sms)) return st;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attn_split_tc_kernel, kThreads, 0) !=
            cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    *slots = sms * per_sm;
    return WQ_OK;
}

bool aligned(const void* p, size_t n) { return reinterpret_cast<uintptr_t>(p) % n == 0; }

}  // namespace

extern "C" {

size_t wq_paged_attention_workspace_bytes(int rows, int Hq, int Hkv, int B, int max_seq_len) {
    if (rows < 0 || Hq <= 0 || Hkv <= 0 || B <= 0 || max_seq_len <= 0) return 0;
    int slots = 0;
    if (grid_slots(&slots) != WQ_OK) return 0;
    int chunk = 0;
    const int splits = splits_for(max_seq_len, B, Hkv, slots, &chunk);
    return wq::kWsHeader + static_cast<size_t>(rows) * Hq * splits * (2 + kD) * sizeof(float);
}

}  // extern "C"

namespace {

// Checks, workspace layout and the two launches; tensor_cores selects the
// split kernel (the CUDA-core one stays as an independent cross-check).
wq_status_t paged_attention(const uint16_t* q, const int8_t* k_codes, const uint16_t* k_scales,
                            const int8_t* v_codes, const uint16_t* v_scales, const int* page_table,
                            int max_pages, const int* seq_len, int B, const int* row_seq,
                            const int* row_pos, int rows, int max_seq_len, int Hq, int Hkv, int D,
                            int T, int pages, float* out, void* workspace, size_t workspace_bytes,
                            void* stream, bool tensor_cores) {
    if (D != kD || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || Hq / Hkv > kQB || T <= 0 ||
        pages <= 0 || B <= 0 || max_pages <= 0 || rows < 0 || max_seq_len <= 0 ||
        max_seq_len > max_pages * T)
        return WQ_ERR_INVALID_ARG;
    if (rows == 0) return WQ_OK;
    if (!q || !k_codes || !k_scales || !v_codes || !v_scales || !page_table || !seq_len ||
        !row_seq || !row_pos || !out || !workspace)
        return WQ_ERR_INVALID_ARG;
    if (!aligned(k_codes, 16) || !aligned(v_codes, 16) || !aligned(k_scales, 8) ||
        !aligned(v_scales, 8) || !aligned(out, 4) ||
        workspace_bytes < wq_paged_attention_workspace_bytes(rows, Hq, Hkv, B, max_seq_len) ||
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
    int slots = 0;
    if (wq_status_t st = grid_slots(&slots)) return st;
    a.splits = splits_for(max_seq_len, B, Hkv, slots, &a.chunk);
    a.err = static_cast<int*>(workspace);
    a.part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + wq::kWsHeader);
    // every (row, head, slice) state is written: rows of other sequences are
    // never read, and empty slices write m = -inf, l = 0
    cudaError_t e = cudaMemsetAsync(a.part, 0, static_cast<size_t>(rows) * Hq * a.splits * (2 + kD) * sizeof(float), s);
    if (e != cudaSuccess) return WQ_ERR_CUDA;
    if (tensor_cores)
        attn_split_tc_kernel<<<dim3(a.splits, Hkv, B), kThreads, 0, s>>>(a);
    else
        attn_split_kernel<<<dim3(a.splits, Hkv, B), kThreads, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return WQ_ERR_CUDA;
    attn_combine_kernel<<<static_cast<unsigned>(rows * Hq), kD, 0, s>>>(a.part, a.splits, Hq, out);
    return cudaGetLastError() == cudaSuccess ? WQ_OK : WQ_ERR_CUDA;
}

}  // namespace

extern "C" {

wq_status_t wq_paged_attention(const uint16_t* q, const int8_t* k_codes, const uint16_t* k_scales,
                               const int8_t* v_codes, const uint16_t* v_scales,
                               const int* page_table, int max_pages, const int* seq_len, int B,
                               const int* row_seq, const int* row_pos, int rows, int max_seq_len,
                               int Hq, int Hkv, int D, int T, int pages, float* out,
                               void* workspace, size_t workspace_bytes, void* stream) {
    return paged_attention(q, k_codes, k_scales, v_codes, v_scales, page_table, max_pages, seq_len,
                           B, row_seq, row_pos, rows, max_seq_len, Hq, Hkv, D, T, pages, out,
                           workspace, workspace_bytes, stream, true);
}

// The same on the CUDA cores (fp32 FMA throughout): not part of include/wq.h;
// the tests compare the two kernels with each other and with the oracle.
wq_status_t wq_internal_paged_attention_cuda_cores(
    const uint16_t* q, const int8_t* k_codes, const uint16_t* k_scales, const int8_t* v_codes,
    const uint16_t* v_scales, const int* page_table, int max_pages, const int* seq_len, int B,
    const int* row_seq, const int* row_pos, int rows, int max_seq_len, int Hq, int Hkv, int D,
    int T, int pages, float* out, void* workspace, size_t workspace_bytes, void* stream) {
    return paged_attention(q, k_codes, k_scales, v_codes, v_scales, page_table, max_pages, seq_len,
                           B, row_seq, row_pos, rows, max_seq_len, Hq, Hkv, D, T, pages, out,
                           workspace, workspace_bytes, stream, false);
}

}  // extern "C"
