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
// * Warp 8 is the producer: one lane issues TMA loads of each stage — the
//   packed tile [128 rows][32 words] plus the matching X slice — into a ring
//   of shared-memory stages (128-byte swizzle), with mbarrier completion.
// * Warps 0..7 are consumers, 16 weight rows each.  Per 32-value word step a
//   thread unpacks one word of each of its two rows with the bf16 "magic
//   number" trick (the code lands in the mantissa of 128.0, so a packed
//   bf16x2 subtract of 128 + z gives q - z exactly), feeds the exact (q - z)
//   as the A operand of mma.sync m16n8k16 (weights are the 16-row side, the
//   M <= 16 rows of X the narrow n side), and applies the group's bf16 scale
//   to the group's fp32 partial product.
// * A tile split across CTAs is summed by the last CTA to finish it, reading
//   the other partials in k order from the workspace (no float atomics, no
//   waiting on other CTAs), so every output has a fixed reduction order.
//
// The k order inside one MMA is a permutation chosen so that each thread's
// A registers come straight from its packed word; the B fragment loads X in
// the same permuted order.  Columns of the n8 tile map to X rows through
// perm(j) = (j >> 1) + 4 * (j & 1), which keeps the swizzled X reads free of
// bank conflicts; the mapping is fixed, so a row's arithmetic never depends on
// how many rows are stacked with it.
#pragma once
#include "wq_internal.h"
#include "wq_ptx.cuh"

namespace wq {

template <int BITS, int NT>
struct Layout {
    static constexpr int kStageValues = stage_values(BITS);
    static constexpr int kXBoxValues = 64;  // 128 bytes of bf16 per X box row
    static constexpr int kXBoxes = kStageValues / kXBoxValues;
    static constexpr int kXBoxBytes = NT * 8 * 128;
    static constexpr int kWBytes = kBN * kWordsPerStage * 4;  // 16 KB
    static constexpr int kStageBytes = kWBytes + kXBoxes * kXBoxBytes;
    static constexpr int kStages0 = (200 * 1024) / kStageBytes;
    static constexpr int kStages = kStages0 > 8 ? 8 : kStages0;
    static constexpr int kBarOffset = kStages * kStageBytes;
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
// Per-group scale / zero point, fetched from global memory three 8-group
// blocks ahead.  Thread c of a quad holds groups 8j + c and 8j + 4 + c of its
// two rows; a group's values are broadcast inside the quad with a shuffle.
struct GroupMeta {
    uint32_t s[3][2];  // bf16 scale of row A (low half) and row B (high half)
    uint32_t z[3][2];  // zero point of row A (byte 0) and row B (byte 1)
    int block;         // block index held in slot 0

    __device__ __forceinline__ void load(int slot, int blk, const GemmArgs& a, int nA, int nB,
                                         int c) {
#pragma unroll
        for (int l = 0; l < 2; ++l) {
            const int gg = blk * 8 + l * 4 + c;
            uint32_t sv = 0, zv = 0;
            if (gg < a.ng) {
                if (nA < a.N) {
                    const size_t o = static_cast<size_t>(nA) * a.ng + gg;
                    sv = __ldg(a.scales + o);
                    zv = __ldg(a.zeros + o);
                }
                if (nB < a.N) {
                    const size_t o = static_cast<size_t>(nB) * a.ng + gg;
                    sv |= static_cast<uint32_t>(__ldg(a.scales + o)) << 16;
                    zv |= static_cast<uint32_t>(__ldg(a.zeros + o)) << 8;
                }
            }
            s[slot][l] = sv;
            z[slot][l] = zv;
        }
    }

    __device__ __forceinline__ void start(int gidx, const GemmArgs& a, int nA, int nB, int c) {
        block = gidx >> 3;
        load(0, block, a, nA, nB, c);
        load(1, block + 1, a, nA, nB, c);
        load(2, block + 2, a, nA, nB, c);
    }

    // Values of group gidx (gidx >= the current block start, non-decreasing).
    __device__ __forceinline__ void get(int gidx, const GemmArgs& a, int nA, int nB, int c,
                                        int lane, float& sA, float& sB, uint32_t& zzA,
                                        uint32_t& zzB) {
        const int blk = gidx >> 3;
        if (blk != block) {  // warp-uniform: advance the ring by one block
#pragma unroll
            for (int l = 0; l < 2; ++l) {
                s[0][l] = s[1][l]; z[0][l] = z[1][l];
                s[1][l] = s[2][l]; z[1][l] = z[2][l];
            }
            block = blk;
            load(2, blk + 2, a, nA, nB, c);
        }
        const int r = gidx & 7;
        const uint32_t sv = (r & 4) ? s[0][1] : s[0][0];
        const uint32_t zv = (r & 4) ? z[0][1] : z[0][0];
        const int src = (lane & ~3) | (r & 3);
        const uint32_t ss = __shfl_sync(0xffffffffu, sv, src);
        const uint32_t zs = __shfl_sync(0xffffffffu, zv, src);
        sA = __uint_as_float(ss << 16);
        sB = __uint_as_float(ss & 0xffff0000u);
        // bf16x2 of (128 + z): low byte z, high byte 0x43, in both halves
        zzA = __byte_perm(zs, 0x43u, 0x4040);
        zzB = __byte_perm(zs, 0x43u, 0x4141);
    }
};

// bf16x2 (128 + q_lo, 128 + q_hi) from the fields selected by `mask`.
__device__ __forceinline__ uint32_t magic_pair(uint32_t v, uint32_t mask) {
    return lop3_and_or(v, mask, 0x43004300u);
}

// ---------------------------------------------------------------------------
// One stage of one consumer warp, 4-bit or 2-bit codes.
//   wrow  : shared address of this thread's row A in the stage (row B = +1024)
//   xrow  : shared address of X row perm(g) + 8t in X box 0, per n8 tile t
template <int BITS, int G, int NT>
__device__ __forceinline__ void stage_pow2(uint32_t wrow, const uint32_t (&xrow)[NT], int g,
                                           int c, int xsw, int gidx0, float (&acc)[NT][4],
                                           GroupMeta& gm, const GemmArgs& a, int nA, int nB,
                                           int lane) {
    using L = Layout<BITS, NT>;
    constexpr int kSteps = L::kStageValues / 32;  // 32-value word steps
    constexpr int kGW = G / 32;                   // word steps per group
    float cg[NT][4];
    float sA = 0.f, sB = 0.f;
    uint32_t zzA = 0, zzB = 0;
#pragma unroll
    for (int ws = 0; ws < kSteps; ++ws) {
        if (ws % kGW == 0) gm.get(gidx0 + ws / kGW, a, nA, nB, c, lane, sA, sB, zzA, zzB);
        uint32_t aw0[4], aw1[4];
        if (BITS == 4) {
            // thread c: word 4*ws + c of the stage row (16-byte chunk ws)
            const uint32_t off = static_cast<uint32_t>(((ws ^ g) << 4) + 4 * c);
            const uint32_t wa = lds32(wrow + off);
            const uint32_t wb = lds32(wrow + 1024 + off);
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
            const uint32_t off = static_cast<uint32_t>((((ws >> 1) ^ g) << 4) +
                                                       4 * (2 * (ws & 1) + (c >> 1)));
            const uint32_t sh = 8u * static_cast<uint32_t>(c & 1);
            const uint32_t wa = lds32(wrow + off) >> sh;
            const uint32_t wb = lds32(wrow + 1024 + off) >> sh;
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
            uint32_t u0, u1, u2, u3;
            const uint32_t xb = xrow[t] + static_cast<uint32_t>((ws >> 1) * L::kXBoxBytes);
            if (BITS == 4) {
                // x[m][32 ws + 8c .. +8): 16-byte chunk 4 (ws & 1) + c of the box row
                const uint4 v = lds128(xb + static_cast<uint32_t>(((4 * (ws & 1) + c) ^ xsw) << 4));
                u0 = v.x; u1 = v.y; u2 = v.z; u3 = v.w;
            } else {
                // x[m][base .. base+4) and x[m][base+8 .. base+12), base = 32 ws + 16 (c>>1) + 4 (c&1)
                const int ch = 4 * (ws & 1) + 2 * (c >> 1);
                const uint32_t inner = 8u * static_cast<uint32_t>(c & 1);
                const uint2 lo = lds64(xb + static_cast<uint32_t>((ch ^ xsw) << 4) + inner);
                const uint2 hi = lds64(xb + static_cast<uint32_t>(((ch + 1) ^ xsw) << 4) + inner);
                u0 = lo.x; u1 = lo.y; u2 = hi.x; u3 = hi.y;
            }
            const uint32_t b00 = __byte_perm(u0, u2, 0x5410), b01 = __byte_perm(u0, u2, 0x7632);
            const uint32_t b10 = __byte_perm(u1, u3, 0x5410), b11 = __byte_perm(u1, u3, 0x7632);
            if (ws % kGW == 0) {
                mma_16816_zero_c(cg[t], aw0, b00, b01);
            } else {
                mma_16816(cg[t], aw0, b00, b01, cg[t]);
            }
            mma_16816(cg[t], aw1, b10, b11, cg[t]);
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

// Store this thread's outputs (rows nA, nB; columns c + 8t and c + 4 + 8t).
template <int NT>
__device__ __forceinline__ void store_y(const GemmArgs& a, const float (&v)[NT][4], int nA,
                                        int nB, int c) {
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int m0 = c + 8 * t, m1 = c + 4 + 8 * t;
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

// ---------------------------------------------------------------------------
template <int BITS, int G, int NT>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                const GemmArgs a) {
    using L = Layout<BITS, NT>;
    constexpr int S = L::kStages;
    constexpr int kGPS = L::kStageValues / G;  // groups per stage
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
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

    if (warp == kConsumerWarps) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        prefetch_tensormap(&tmW);
        prefetch_tensormap(&tmX);
        const uint64_t pol_w = policy_evict_first();
        const uint64_t pol_x = policy_evict_last();
        uint32_t it = 0;
        bool ok = true;
        for (long long u = u_lo; u < u_hi && ok;) {
            const int t = static_cast<int>(u / a.I);
            const int i0 = static_cast<int>(u - static_cast<long long>(t) * a.I);
            const int i1 = static_cast<int>(min(static_cast<long long>(a.I),
                                                u_hi - static_cast<long long>(t) * a.I));
            {   // warm L2 with this tile's scales and zero points (whole rows, rounded inward)
                const int r0 = t * kBN, r1 = min(a.N, r0 + kBN);
                const uintptr_t sb = reinterpret_cast<uintptr_t>(a.scales + static_cast<size_t>(r0) * a.ng);
                const uintptr_t se = reinterpret_cast<uintptr_t>(a.scales + static_cast<size_t>(r1) * a.ng);
                const uintptr_t zb = reinterpret_cast<uintptr_t>(a.zeros + static_cast<size_t>(r0) * a.ng);
                const uintptr_t ze = reinterpret_cast<uintptr_t>(a.zeros + static_cast<size_t>(r1) * a.ng);
                const uintptr_t sb16 = (sb + 15) & ~uintptr_t(15), se16 = se & ~uintptr_t(15);
                const uintptr_t zb16 = (zb + 15) & ~uintptr_t(15), ze16 = ze & ~uintptr_t(15);
                if (se16 > sb16) prefetch_l2_bulk(reinterpret_cast<const void*>(sb16), static_cast<uint32_t>(se16 - sb16));
                if (ze16 > zb16) prefetch_l2_bulk(reinterpret_cast<const void*>(zb16), static_cast<uint32_t>(ze16 - zb16));
            }
            for (int i = i0; i < i1; ++i, ++it) {
                const int slot = static_cast<int>(it % S);
                const uint32_t ph = (it / S) & 1u;
                if (!mbar_wait(&empty[slot], ph ^ 1u, abort_flag)) {
                    record_error(a, abort_flag);
                    ok = false;
                    break;
                }
                uint8_t* st = smem + slot * L::kStageBytes;
                mbar_arrive_expect_tx(&full[slot], L::kStageBytes);
                tma_load_2d(st, &tmW, i * kWordsPerStage, t * kBN, &full[slot], pol_w);
#pragma unroll
                for (int b = 0; b < L::kXBoxes; ++b)
                    tma_load_2d(st + L::kWBytes + b * L::kXBoxBytes, &tmX,
                                i * L::kStageValues + b * L::kXBoxValues, 0, &full[slot], pol_x);
            }
            u = static_cast<long long>(t) * a.I + i1;
        }
        if (!ok) {
            // let copies already in flight land before the CTA's shared memory goes away
            const uint32_t first = it > S ? it - S : 0;
            volatile int never = 0;
            for (uint32_t j = first; j < it; ++j)
                mbar_wait(&full[j % S], (j / S) & 1u, &never);
        }
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int g = lane >> 2;
    const int c = lane & 3;
    const int rowA = warp * 16 + g;                 // row within the tile
    const int xsw = (g >> 1) + 4 * (g & 1);         // perm(g): X row of this lane's column
    const uint32_t smem_base = smem_addr(smem);
    uint32_t it = 0;
    // After a failed wait a warp stops computing but keeps walking the same
    // sequence of named barriers as its siblings, so none of them can block.
    bool dead = false;

    for (long long u = u_lo; u < u_hi;) {
        const int t = static_cast<int>(u / a.I);
        const int i0 = static_cast<int>(u - static_cast<long long>(t) * a.I);
        const int i1 = static_cast<int>(min(static_cast<long long>(a.I),
                                            u_hi - static_cast<long long>(t) * a.I));
        const int nA = t * kBN + rowA;
        const int nB = nA + 8;
        float acc[NT][4];
#pragma unroll
        for (int tt = 0; tt < NT; ++tt)
#pragma unroll
            for (int j = 0; j < 4; ++j) acc[tt][j] = 0.f;
        GroupMeta gm;
        gm.start(i0 * kGPS, a, nA, nB, c);

        for (int i = i0; i < i1; ++i, ++it) {
            const int slot = static_cast<int>(it % S);
            const uint32_t ph = (it / S) & 1u;
            if (dead || !mbar_wait(&full[slot], ph, abort_flag)) {
                if (!dead) record_error(a, abort_flag);
                dead = true;
                continue;
            }
            const uint32_t st = smem_base + static_cast<uint32_t>(slot * L::kStageBytes);
            const uint32_t wrow = st + static_cast<uint32_t>(rowA * 128);
            uint32_t xrow[NT];
#pragma unroll
            for (int tt = 0; tt < NT; ++tt)
                xrow[tt] = st + L::kWBytes + static_cast<uint32_t>((xsw + 8 * tt) * 128);
            stage_pow2<BITS, G, NT>(wrow, xrow, g, c, xsw, i * kGPS, acc, gm, a, nA, nB, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
        }

        if (i0 == 0 && i1 == a.I) {
            if (!dead) store_y<NT>(a, acc, nA, nB, c);
        } else {
            // split tile: publish the partial, the last CTA to arrive sums them in k order
            const int t_first = static_cast<int>(u_lo / a.I);
            const int role = (t == t_first) ? 0 : 1;
            float* mine = a.partials + static_cast<size_t>(2 * blockIdx.x + role) * (kMaxCols * kBN);
            const int lA = rowA, lB = rowA + 8;
#pragma unroll
            for (int tt = 0; tt < NT; ++tt) {
                const int m0 = c + 8 * tt, m1 = c + 4 + 8 * tt;
                __stcg(mine + m0 * kBN + lA, acc[tt][0]);
                __stcg(mine + m1 * kBN + lA, acc[tt][1]);
                __stcg(mine + m0 * kBN + lB, acc[tt][2]);
                __stcg(mine + m1 * kBN + lB, acc[tt][3]);
            }
            __threadfence();
            named_bar_sync(1, 32 * kConsumerWarps);
            const long long tu0 = static_cast<long long>(t) * a.I;
            const int b_first = cta_of_unit(a.U, a.P, tu0);
            const int b_last = cta_of_unit(a.U, a.P, tu0 + a.I - 1);
            if (threadIdx.x == 0) {
                // a CTA with a failed wait leaves the tile unfinished (the host
                // sees the error word and must re-initialise the workspace)
                if (*abort_flag) {
                    *last_flag = 0;
                } else {
                    const int prev = atomicAdd(a.counters + t, 1);
                    *last_flag = (prev == b_last - b_first) ? 1 : 0;
                }
            }
            named_bar_sync(1, 32 * kConsumerWarps);
            if (*last_flag) {
                __threadfence();
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
                        const float* src = a.partials +
                            static_cast<size_t>(2 * b + (t == tb ? 0 : 1)) * (kMaxCols * kBN);
#pragma unroll
                        for (int tt = 0; tt < NT; ++tt) {
                            const int m0 = c + 8 * tt, m1 = c + 4 + 8 * tt;
                            tot[tt][0] += __ldcg(src + m0 * kBN + lA);
                            tot[tt][1] += __ldcg(src + m1 * kBN + lA);
                            tot[tt][2] += __ldcg(src + m0 * kBN + lB);
                            tot[tt][3] += __ldcg(src + m1 * kBN + lB);
                        }
                    }
                }
                store_y<NT>(a, tot, nA, nB, c);
                if (threadIdx.x == 0) a.counters[t] = 0;
            }
            named_bar_sync(1, 32 * kConsumerWarps);
        }
        u = static_cast<long long>(t) * a.I + i1;
    }
}

template <int BITS, int G, int NT>
cudaError_t launch_one(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmArgs& a,
                       cudaStream_t s) {
    using L = Layout<BITS, NT>;
    auto kern = gemm_kernel<BITS, G, NT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         L::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<a.P, kThreads, L::kSmemBytes, s>>>(tmW, tmX, a);
    return cudaGetLastError();
}

}  // namespace wq
