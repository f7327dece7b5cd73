// Weight-only low-bit skinny GEMM for sm_103a:
//     Y[M][N] = X[M][K] . dequant(Wq)[N][K]^T,  M <= 16.
//
// One decode-step projection streams every packed weight once and multiplies
// it, while on chip, against all stacked rows of X on tensor cores (OpenJet
// news page, paragraph "并行解码的原理").  Structure of one launch:
//
// * Persistent grid (<= SM count).  Work units are (128-row tile, k-stage)
//   pairs linearised tile-major; CTA b owns a contiguous, equal share of them
//   (stream-K).  The split depends on (N, K, bits, group, SM count) only.
// * Warp 8 is the producer: one lane issues the TMA loads of each stage — the
//   packed tile [128 rows][32 words] and the matching X slice, 128-byte
//   swizzled — into a ring of shared-memory stages with mbarrier completion,
//   and warms L2 with each tile's scales and zero points.
// * Warps 0..7 are consumers, 16 weight rows each.  Each thread fetches the
//   scales and zero points of its two rows one stage ahead into registers.
//   For every stage the warps first permute the X slice once, cooperatively,
//   into the exact mma.sync B fragments (one 16-byte shared load per thread
//   per two MMAs), then each
//   thread unpacks one packed word of each of its two rows per 32-value step
//   with the bf16 "magic number" trick (the code lands in the mantissa of
//   128.0, so a packed bf16x2 subtract of 128 + z gives q - z exactly), feeds
//   the exact (q - z) as the A operand of mma.sync m16n8k16 (weights are the
//   16-row side, the M <= 16 rows of X the narrow n side), and applies the
//   group's bf16 scale to the group's fp32 partial product.
// * A tile split across CTAs is summed by the last CTA to finish it, reading
//   the other partials in k order from the workspace (no float atomics, no
//   waiting on other CTAs), so every output has a fixed reduction order.
//
// The k order inside one MMA is a permutation chosen so that each thread's
// A registers come straight from its packed word; the B fragments hold X in
// the same permuted order.  Column j of an n8 tile is X row j + 8t, fixed, so a
// row's arithmetic never depends on how many rows are stacked with it.
#pragma once
#include "wq_internal.h"
#include "wq_ptx.cuh"

namespace wq {

constexpr int kSmemBudget = 220 * 1024;  // stages + B-fragment buffers

constexpr int round_up(int v, int a) { return (v + a - 1) / a * a; }
constexpr int clamp_int(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }


template <int BITS, int G, int NT>
struct Layout {
    static constexpr int kStageValues = stage_values(BITS);
    static constexpr int kWBytes = kBN * kWordsPerStage * 4;  // 16 KB of packed words
    static constexpr int kXBoxValues = 64;                    // 128 bytes of bf16 per box row
    static constexpr int kXBoxes = kStageValues / kXBoxValues;
    static constexpr int kXBoxBytes = NT * 8 * 128;
    static constexpr int kXBytes = kXBoxes * kXBoxBytes;
    static constexpr int kGPS = kStageValues / G;             // groups per stage (4-bit, 2-bit)
    static constexpr int kStageBytes = round_up(kWBytes + kXBytes, 1024);
    static constexpr int kSteps = kStageValues / 32;          // 32-value word steps
    static constexpr int kXpBytes = kSteps * NT * 32 * 16;    // B fragments of one stage
    static constexpr int kStages = clamp_int((kSmemBudget - 2 * kXpBytes) / kStageBytes, 2, 8);
    static constexpr int kXpOffset = kStages * kStageBytes;
    static constexpr int kBarOffset = kXpOffset + 2 * kXpBytes;
    static constexpr int kSmemBytes = kBarOffset + 256 + 1024;  // barriers/flags + align slack
};

__device__ __forceinline__ int cta_of_unit(long long U, int P, long long u) {
    return static_cast<int>(((u + 1) * P + U - 1) / U - 1);
}

__device__ __forceinline__ long long d_unit_begin(long long U, int P, int b) {
    return U * b / P;
}

__device__ __forceinline__ void record_error(const GemmArgs& a, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicExch(a.err, 1);
}

// ---------------------------------------------------------------------------
// Scales and zero points of one stage's GPS groups for a thread's two rows,
// held in registers: scales as packed bf16 pairs, zero points as packed bytes.
template <int GPS>
struct GroupRegs {
    static constexpr int kS = (GPS + 1) / 2;
    static constexpr int kZ = (GPS + 3) / 4;
    uint32_t s[2][kS];
    uint32_t z[2][kZ];

    // Groups [g0, g0 + GPS) of rows nA, nB.  `vec`: every row's first group of
    // a stage is GPS-aligned and the arrays are 16-byte aligned, so each row's
    // values are one naturally aligned vector load.
    __device__ __forceinline__ void load(const GemmArgs& a, int nA, int nB, long long g0, bool vec) {
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int n = r ? nB : nA;
#pragma unroll
            for (int j = 0; j < kS; ++j) s[r][j] = 0;
#pragma unroll
            for (int j = 0; j < kZ; ++j) z[r][j] = 0;
            if (n >= a.N) continue;
            const long long base = static_cast<long long>(n) * a.ng + g0;
            if (vec) {
                const uint16_t* sp = a.scales + base;
                const uint8_t* zp = a.zeros + base;
                if (GPS == 1) {
                    s[r][0] = __ldg(sp);
                    z[r][0] = __ldg(zp);
                } else if (GPS == 2) {
                    s[r][0] = __ldg(reinterpret_cast<const uint32_t*>(sp));
                    z[r][0] = __ldg(reinterpret_cast<const uint16_t*>(zp));
                } else if (GPS == 4) {
                    const uint2 v = __ldg(reinterpret_cast<const uint2*>(sp));
                    s[r][0] = v.x; s[r][kS > 1 ? 1 : 0] = v.y;
                    z[r][0] = __ldg(reinterpret_cast<const uint32_t*>(zp));
                } else {
#pragma unroll
                    for (int j = 0; j < kS / 4; ++j) {
                        const uint4 v = __ldg(reinterpret_cast<const uint4*>(sp) + j);
                        s[r][4 * j] = v.x; s[r][4 * j + 1] = v.y;
                        s[r][4 * j + 2] = v.z; s[r][4 * j + 3] = v.w;
                    }
                    if (GPS == 8) {
                        const uint2 v = __ldg(reinterpret_cast<const uint2*>(zp));
                        z[r][0] = v.x; z[r][kZ > 1 ? 1 : 0] = v.y;
                    } else {
#pragma unroll
                        for (int j = 0; j < kZ / 4; ++j) {
                            const uint4 v = __ldg(reinterpret_cast<const uint4*>(zp) + j);
                            z[r][4 * j] = v.x; z[r][4 * j + 1] = v.y;
                            z[r][4 * j + 2] = v.z; z[r][4 * j + 3] = v.w;
                        }
                    }
                }
            } else {
#pragma unroll
                for (int gi = 0; gi < GPS; ++gi) {
                    if (g0 + gi < a.ng) {
                        s[r][gi / 2] |= static_cast<uint32_t>(__ldg(a.scales + base + gi)) << (16 * (gi & 1));
                        z[r][gi / 4] |= static_cast<uint32_t>(__ldg(a.zeros + base + gi)) << (8 * (gi & 3));
                    }
                }
            }
        }
    }

    // fp32 scale and bf16x2 (128 + z, 128 + z) of group gi (compile-time) of row r.
    __device__ __forceinline__ float scale(int r, int gi) const {
        const uint32_t w = s[r][gi / 2];
        return __uint_as_float((gi & 1) ? (w & 0xffff0000u) : (w << 16));
    }
    __device__ __forceinline__ uint32_t zz(int r, int gi) const {
        return __byte_perm(z[r][gi / 4], 0x43u, 0x4040u | (0x0101u * static_cast<uint32_t>(gi & 3)));
    }
};

// ---------------------------------------------------------------------------
// Consumers, once per stage: permute the stage's X slice into mma.sync B
// fragments.  Entry ((ws * NT + t) * 32 + lane) holds, for lane (g, c) and
// n8 tile t, the four B registers of the two MMAs of word step ws:
//   4-bit: x[m][8c'+{0,4}], x[m][8c'+{1,5}], x[m][8c'+{2,6}], x[m][8c'+{3,7}]
//          with c' = 4 ws + c (word c' of the stage) and m = g + 8t;
//   2-bit: the same pattern over x[m][b..b+4) and x[m][b+8..b+12),
//          b = 32 ws + 16 (c >> 1) + 4 (c & 1) (half c & 1 of word 2 ws + (c >> 1)).
template <int BITS, int G, int NT>
__device__ __forceinline__ void build_bfrag(const uint8_t* xraw, uint8_t* xp, int tid) {
    using L = Layout<BITS, G, NT>;
    constexpr int kEntries = L::kSteps * NT * 32;
    static_assert(kEntries % (32 * kConsumerWarps) == 0, "entries split evenly");
#pragma unroll
    for (int e = 0; e < kEntries / (32 * kConsumerWarps); ++e) {
        const int E = tid + e * 32 * kConsumerWarps;
        const int ln = E & 31;
        const int wt = E >> 5;
        const int ws = wt / NT;
        const int t = wt - ws * NT;
        const int g = ln >> 2, c = ln & 3;
        const int m = g + 8 * t;
        const uint8_t* row = xraw + (ws >> 1) * L::kXBoxBytes + m * 128;
        uint32_t u0, u1, u2, u3;
        if (BITS == 4) {
            const int chunk = 4 * (ws & 1) + c;
            const uint4 v = *reinterpret_cast<const uint4*>(row + ((chunk ^ g) << 4));
            u0 = v.x; u1 = v.y; u2 = v.z; u3 = v.w;
        } else {
            const int ch = 4 * (ws & 1) + 2 * (c >> 1);
            const int inner = 8 * (c & 1);
            const uint2 lo = *reinterpret_cast<const uint2*>(row + ((ch ^ g) << 4) + inner);
            const uint2 hi = *reinterpret_cast<const uint2*>(row + (((ch + 1) ^ g) << 4) + inner);
            u0 = lo.x; u1 = lo.y; u2 = hi.x; u3 = hi.y;
        }
        *reinterpret_cast<uint4*>(xp + E * 16) =
            make_uint4(__byte_perm(u0, u2, 0x5410), __byte_perm(u0, u2, 0x7632),
                       __byte_perm(u1, u3, 0x5410), __byte_perm(u1, u3, 0x7632));
    }
}

// bf16x2 (128 + q_lo, 128 + q_hi) from the fields selected by `mask`.
__device__ __forceinline__ uint32_t magic_pair(uint32_t v, uint32_t mask) {
    return lop3_and_or(v, mask, 0x43004300u);
}

// ---------------------------------------------------------------------------
// One stage of one consumer warp, 4-bit or 2-bit codes.
//   wrow : this thread's row A in the stage (row B = +1024 bytes)
//   xp   : this stage's B-fragment buffer
template <int BITS, int G, int NT>
__device__ __forceinline__ void stage_pow2(const uint8_t* wrow, const uint8_t* xp,
                                           const GroupRegs<Layout<BITS, G, NT>::kGPS>& gr, int g,
                                           int c, int lane, float (&acc)[NT][4]) {
    using L = Layout<BITS, G, NT>;
    constexpr int kGW = G / 32;  // word steps per group
    float cg[NT][4];
    float sA = 0.f, sB = 0.f;
    uint32_t zzA = 0, zzB = 0;
#pragma unroll
    for (int ws = 0; ws < L::kSteps; ++ws) {
        if (ws % kGW == 0) {
            sA = gr.scale(0, ws / kGW);
            sB = gr.scale(1, ws / kGW);
            zzA = gr.zz(0, ws / kGW);
            zzB = gr.zz(1, ws / kGW);
        }
        uint32_t aw0[4], aw1[4];
        if (BITS == 4) {
            // thread c: word 4*ws + c of the stage row (16-byte chunk ws)
            const int off = ((ws ^ g) << 4) + 4 * c;
            const uint32_t wa = *reinterpret_cast<const uint32_t*>(wrow + off);
            const uint32_t wb = *reinterpret_cast<const uint32_t*>(wrow + 1024 + off);
            aw0[0] = bf16x2_sub(magic_pair(wa, 0x000f000fu), zzA);
            aw0[1] = bf16x2_sub(magic_pair(wb, 0x000f000fu), zzB);
            aw0[2] = bf16x2_sub(magic_pair(wa >> 4, 0x000f000fu), zzA);
            aw0[3] = bf16x2_sub(magic_pair(wb >> 4, 0x000f000fu), zzB);
            aw1[0] = bf16x2_sub(magic_pair(wa >> 8, 0x000f000fu), zzA);
            aw1[1] = bf16x2_sub(magic_pair(wb >> 8, 0x000f000fu), zzB);
            aw1[2] = bf16x2_sub(magic_pair(wa >> 12, 0x000f000fu), zzA);
            aw1[3] = bf16x2_sub(magic_pair(wb >> 12, 0x000f000fu), zzB);
        } else {
            // thread c: half (c & 1) of word 2*ws + (c >> 1)
            const int off = (((ws >> 1) ^ g) << 4) + 4 * (2 * (ws & 1) + (c >> 1));
            const uint32_t sh = 8u * static_cast<uint32_t>(c & 1);
            const uint32_t wa = *reinterpret_cast<const uint32_t*>(wrow + off) >> sh;
            const uint32_t wb = *reinterpret_cast<const uint32_t*>(wrow + 1024 + off) >> sh;
            aw0[0] = bf16x2_sub(magic_pair(wa, 0x00030003u), zzA);
            aw0[1] = bf16x2_sub(magic_pair(wb, 0x00030003u), zzB);
            aw0[2] = bf16x2_sub(magic_pair(wa >> 2, 0x00030003u), zzA);
            aw0[3] = bf16x2_sub(magic_pair(wb >> 2, 0x00030003u), zzB);
            aw1[0] = bf16x2_sub(magic_pair(wa >> 4, 0x00030003u), zzA);
            aw1[1] = bf16x2_sub(magic_pair(wb >> 4, 0x00030003u), zzB);
            aw1[2] = bf16x2_sub(magic_pair(wa >> 6, 0x00030003u), zzA);
            aw1[3] = bf16x2_sub(magic_pair(wb >> 6, 0x00030003u), zzB);
        }
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            const uint4 b = *reinterpret_cast<const uint4*>(xp + ((ws * NT + t) * 32 + lane) * 16);
            if (ws % kGW == 0) {
                mma_16816_zero_c(cg[t], aw0, b.x, b.y);
            } else {
                mma_16816(cg[t], aw0, b.x, b.y);
            }
            mma_16816(cg[t], aw1, b.z, b.w);
        }
        if (ws % kGW == kGW - 1) {
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                acc[t][0] = fmaf(sA, cg[t][0], acc[t][0]);
                acc[t][1] = fmaf(sA, cg[t][1], acc[t][1]);
                acc[t][2] = fmaf(sB, cg[t][2], acc[t][2]);
                acc[t][3] = fmaf(sB, cg[t][3], acc[t][3]);
            }
        }
    }
}

// Store this thread's outputs (rows nA, nB; columns 2c + 8t and 2c + 1 + 8t).
template <int NT>
__device__ __forceinline__ void store_y(const GemmArgs& a, const float (&v)[NT][4], int nA,
                                        int nB, int c) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int m0 = 2 * c + 8 * t, m1 = m0 + 1;
        if (nA < a.N) {
            if (m0 < a.M) a.y[static_cast<size_t>(m0) * a.N + nA] = v[t][0];
            if (m1 < a.M) a.y[static_cast<size_t>(m1) * a.N + nA] = v[t][1];
        }
        if (nB < a.N) {
            if (m0 < a.M) a.y[static_cast<size_t>(m0) * a.N + nB] = v[t][2];
            if (m1 < a.M) a.y[static_cast<size_t>(m1) * a.N + nB] = v[t][3];
        }
    }
}

// End of a tile segment: store Y, or publish the partial and let the last CTA
// of the tile sum all partials in k order.
template <int NT>
__device__ __forceinline__ void finish_segment(const GemmArgs& a, const float (&acc)[NT][4], int t,
                                               bool whole_tile, long long u_lo, int rowA, int c,
                                               int tid, bool dead, volatile int* abort_flag,
                                               volatile int* last_flag) {
    const int nA = t * kBN + rowA, nB = nA + 8;
    if (whole_tile) {
        if (!dead) store_y<NT>(a, acc, nA, nB, c);
        return;
    }
    const int t_first = static_cast<int>(u_lo / a.I);
    const int role = (t == t_first) ? 0 : 1;
    float* mine = a.partials + static_cast<size_t>(2 * blockIdx.x + role) * (kMaxCols * kBN);
    const int lA = rowA, lB = rowA + 8;
#pragma unroll
    for (int tt = 0; tt < NT; ++tt) {
        const int m0 = 2 * c + 8 * tt, m1 = m0 + 1;
        __stcg(mine + m0 * kBN + lA, acc[tt][0]);
        __stcg(mine + m1 * kBN + lA, acc[tt][1]);
        __stcg(mine + m0 * kBN + lB, acc[tt][2]);
        __stcg(mine + m1 * kBN + lB, acc[tt][3]);
    }
    named_bar_sync(1, 32 * kConsumerWarps);
    const long long tu0 = static_cast<long long>(t) * a.I;
    const int b_first = cta_of_unit(a.U, a.P, tu0);
    const int b_last = cta_of_unit(a.U, a.P, tu0 + a.I - 1);
    if (tid == 0) {
        // a CTA with a failed wait leaves the tile unfinished (the host sees
        // the error word and must re-initialise the workspace)
        if (*abort_flag) {
            *last_flag = 0;
        } else {
            const int prev = atomic_add_acq_rel_gpu(a.counters + t, 1);
            *last_flag = (prev == b_last - b_first) ? 1 : 0;
        }
    }
    named_bar_sync(1, 32 * kConsumerWarps);
    if (*last_flag) {
        float tot[NT][4];
#pragma unroll
        for (int tt = 0; tt < NT; ++tt)
#pragma unroll
            for (int j = 0; j < 4; ++j) tot[tt][j] = 0.f;
        for (int b = b_first; b <= b_last; ++b) {
            if (b == static_cast<int>(blockIdx.x)) {
#pragma unroll
                for (int tt = 0; tt < NT; ++tt)
#pragma unroll
                    for (int j = 0; j < 4; ++j) tot[tt][j] += acc[tt][j];
            } else {
                const int tb = static_cast<int>(d_unit_begin(a.U, a.P, b) / a.I);
                const float* src =
                    a.partials + static_cast<size_t>(2 * b + (t == tb ? 0 : 1)) * (kMaxCols * kBN);
#pragma unroll
                for (int tt = 0; tt < NT; ++tt) {
                    const int m0 = 2 * c + 8 * tt, m1 = m0 + 1;
                    tot[tt][0] += __ldcg(src + m0 * kBN + lA);
                    tot[tt][1] += __ldcg(src + m1 * kBN + lA);
                    tot[tt][2] += __ldcg(src + m0 * kBN + lB);
                    tot[tt][3] += __ldcg(src + m1 * kBN + lB);
                }
            }
        }
        store_y<NT>(a, tot, nA, nB, c);
        if (tid == 0) a.counters[t] = 0;
    }
    named_bar_sync(1, 32 * kConsumerWarps);
}

// ---------------------------------------------------------------------------
template <int BITS, int G, int NT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const GemmArgs a) {
    using L = Layout<BITS, G, NT>;
    using GR = GroupRegs<L::kGPS>;
    constexpr int S = L::kStages;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // Align to 1024 bytes (128-byte swizzle atoms) by offsetting the shared
    // array itself, so the compiler keeps every access in the shared space.
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
    uint64_t* empty = full + S;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(empty + S);
    volatile int* last_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
        }
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    const long long u_lo = d_unit_begin(a.U, a.P, blockIdx.x);
    const long long u_hi = d_unit_begin(a.U, a.P, blockIdx.x + 1);
    const int n_units = static_cast<int>(u_hi - u_lo);

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        prefetch_tensormap(&tmW);
        prefetch_tensormap(&tmX);
        const uint64_t pol_w = policy_evict_first();
        const uint64_t pol_x = policy_evict_last();
        int t = static_cast<int>(u_lo / a.I);
        int i = static_cast<int>(u_lo - static_cast<long long>(t) * a.I);
        uint32_t it = 0;
        bool ok = true;
        for (int k = 0; k < n_units; ++k, ++it) {
            if (k == 0 || i == 0) {
                // warm L2 with the tile's scales and zero points (whole rows, rounded inward)
                const int r0 = t * kBN, r1 = min(a.N, r0 + kBN);
                const uintptr_t sb = reinterpret_cast<uintptr_t>(a.scales + static_cast<size_t>(r0) * a.ng);
                const uintptr_t se = reinterpret_cast<uintptr_t>(a.scales + static_cast<size_t>(r1) * a.ng);
                const uintptr_t zb = reinterpret_cast<uintptr_t>(a.zeros + static_cast<size_t>(r0) * a.ng);
                const uintptr_t ze = reinterpret_cast<uintptr_t>(a.zeros + static_cast<size_t>(r1) * a.ng);
                const uintptr_t sb16 = (sb + 15) & ~uintptr_t(15), se16 = se & ~uintptr_t(15);
                const uintptr_t zb16 = (zb + 15) & ~uintptr_t(15), ze16 = ze & ~uintptr_t(15);
                if (se16 > sb16)
                    prefetch_l2_bulk(reinterpret_cast<const void*>(sb16), static_cast<uint32_t>(se16 - sb16));
                if (ze16 > zb16)
                    prefetch_l2_bulk(reinterpret_cast<const void*>(zb16), static_cast<uint32_t>(ze16 - zb16));
            }
            const int slot = static_cast<int>(it % S);
            const uint32_t ph = (it / S) & 1u;
            if (!mbar_wait(&empty[slot], ph ^ 1u, abort_flag)) {
                record_error(a, abort_flag);
                ok = false;
                break;
            }
            uint8_t* st = smem + slot * L::kStageBytes;
            mbar_arrive_expect_tx(&full[slot], L::kWBytes + L::kXBytes);
            tma_load_2d(st, &tmW, i * kWordsPerStage, t * kBN, &full[slot], pol_w);
#pragma unroll
            for (int b = 0; b < L::kXBoxes; ++b)
                tma_load_2d(st + L::kWBytes + b * L::kXBoxBytes, &tmX,
                            i * L::kStageValues + b * L::kXBoxValues, 0, &full[slot], pol_x);
            if (++i == a.I) {
                i = 0;
                ++t;
            }
        }
        if (!ok) {
            // let copies already in flight land before the CTA's shared memory goes away
            const uint32_t first = it > S ? it - S : 0;
            volatile int never = 0;
            for (uint32_t j = first; j < it; ++j) mbar_wait(&full[j % S], (j / S) & 1u, &never);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int tid = threadIdx.x;  // 0 .. 255
    const int g = lane >> 2;
    const int c = lane & 3;
    const int rowA = warp * 16 + g;  // row within the tile
    const bool vec = a.meta_vec != 0;
    const int t_first = static_cast<int>(u_lo / a.I);
    const int i_first = static_cast<int>(u_lo - static_cast<long long>(t_first) * a.I);
    // After a failed wait a warp stops computing but keeps walking the same
    // sequence of named barriers as its siblings, so none of them can block.
    bool dead = false;
    float acc[NT][4];

    // unit k of this CTA is (t, i); scales / zero points are fetched one unit ahead
    int t = t_first, i = i_first;       // unit being computed
    int pt = t_first, pi = i_first;     // unit whose group values are fetched next
    GR gr0, gr1;
    auto fetch = [&](GR& gr) {
        gr.load(a, pt * kBN + rowA, pt * kBN + rowA + 8, static_cast<long long>(pi) * L::kGPS, vec);
        if (++pi == a.I) {
            pi = 0;
            ++pt;
        }
    };
    auto unit = [&](const GR& gr, int k) {
        if (k == 0 || i == 0) {
#pragma unroll
            for (int tt = 0; tt < NT; ++tt)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[tt][j] = 0.f;
        }
        const uint32_t it = static_cast<uint32_t>(k);
        const int slot = static_cast<int>(it % S);
        const uint32_t ph = (it / S) & 1u;
        if (!dead && !mbar_wait(&full[slot], ph, abort_flag)) {
            record_error(a, abort_flag);
            dead = true;
        }
        const uint8_t* st = smem + slot * L::kStageBytes;
        uint8_t* xp = smem + L::kXpOffset + (it & 1u) * L::kXpBytes;
        if (!dead) build_bfrag<BITS, G, NT>(st + L::kWBytes, xp, tid);
        named_bar_sync(2, 32 * kConsumerWarps);
        if (!dead) stage_pow2<BITS, G, NT>(st + rowA * 128, xp, gr, g, c, lane, acc);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        if (i == a.I - 1 || k == n_units - 1) {
            const bool whole = (i == a.I - 1) && (t != t_first || i_first == 0);
            finish_segment<NT>(a, acc, t, whole, u_lo, rowA, c, tid, dead, abort_flag, last_flag);
        }
        if (++i == a.I) {
            i = 0;
            ++t;
        }
    };

    if (n_units > 0) fetch(gr0);
    if (n_units > 1) fetch(gr1);
    for (int k = 0; k < n_units; k += 2) {
        unit(gr0, k);
        if (k + 2 < n_units) fetch(gr0);
        if (k + 1 < n_units) {
            unit(gr1, k + 1);
            if (k + 3 < n_units) fetch(gr1);
        }
    }
}

template <int BITS, int G, int NT>
cudaError_t launch_one(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmArgs& a,
                       cudaStream_t s) {
    using L = Layout<BITS, G, NT>;
    auto kern = gemm_kernel<BITS, G, NT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<a.P, kThreads, L::kSmemBytes, s>>>(tmW, tmX, a);
    return cudaGetLastError();
}

}  // namespace wq
