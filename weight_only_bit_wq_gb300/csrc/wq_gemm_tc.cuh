// Weight-only low-bit skinny GEMM on the 5th-generation tensor core (sm_103a):
//     Y[M][N] = X[M][K] . dequant(Wq)[N][K]^T,  M <= 16.
//
// A decode-step projection streams every packed weight once and multiplies it,
// while on chip, against all stacked rows of X on tensor cores (OpenJet news
// page, paragraph "并行解码的原理").  One CTA per SM, persistent, stream-K over
// (128-row tile, k-stage) units exactly as the split depends on (N, K, bits,
// group, SM count) only.  Ten warps:
//
// * warp 8  — TMA producer: per stage one 128-row x 128-byte tile of packed
//   words and the matching X slice (16 rows x stage width, rows >= M read as
//   zero), both 128-byte swizzled, into a ring of shared-memory stages;
// * warp 9  — allocates tensor memory and, from one lane, issues the MMAs:
//   tcgen05.mma kind::f16, M = 128 weight rows, N = 16 rows of X, K = 16,
//   A (the weights) from tensor memory, B (X) straight from the swizzled
//   shared tile through a matrix descriptor, fp32 D in tensor memory;
// * warps 0..7 — one weight row per thread (warp w owns TMEM lanes
//   32 (w % 4) .. +31; warps w and w + 4 split each group's K steps).  Each
//   thread unpacks its row's codes with the bf16 "magic number" trick (code q
//   lands in the mantissa of 128.0, giving 128 + q exactly) and stores them to
//   tensor memory as the A tile in natural k order.  The zero point is applied
//   on the tensor core too: a second MMA per K step multiplies the same X by
//   a constant A tile holding -(128 + z) in every column of the row, so each
//   group's D is sum_k x (q - z) up to fp32 accumulation.  The thread then
//   reads its row of the group's D back with tcgen05.ld and adds scale * D to
//   its fp32 accumulators.
//
// Per group the D accumulation order is fixed (data MMA then zero-point MMA
// per K step, K steps ascending) and the columns of one MMA never interact,
// so a row of X gives bit-identical results alone or stacked.  A tile split
// across CTAs is summed by the last CTA to finish it, in k order.
#pragma once
#include "wq_internal.h"
#include "wq_ptx.cuh"

namespace wq {
namespace tc {

constexpr int kN = 16;          // MMA N: rows of X (M padded to 16)
constexpr uint32_t kTmemCols = 512;
constexpr int kSmemBudgetTc = 210 * 1024;

constexpr int round_up_tc(int v, int a) { return (v + a - 1) / a * a; }
constexpr int clamp_tc(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

template <int BITS, int G>
struct Lay {
    static constexpr int kBoxes = tc_boxes(BITS);               // 32-word boxes per row
    static constexpr int kStageValues = tc_stage_values(BITS);  // 512 (4-bit), 512 (2-bit)
    static constexpr int kBoxBytes = kBN * kWordsPerStage * 4;  // 16 KB: 128 rows x 128 bytes
    static constexpr int kWBytes = kBoxes * kBoxBytes;
    static constexpr int kXBoxValues = 64;                      // 128 bytes of bf16
    static constexpr int kXBoxes = kStageValues / kXBoxValues;
    static constexpr int kXBoxBytes = kN * 128;                 // 16 rows x 128 bytes
    static constexpr int kXBytes = kXBoxes * kXBoxBytes;
    static constexpr int kStageBytes = round_up_tc(kWBytes + kXBytes, 1024);
    static constexpr int kGPS = kStageValues / G;               // groups per stage
    static constexpr int kSteps = G / 16;                       // K16 steps per group
    static constexpr int kACols = kSteps * 8;                   // TMEM columns of one A tile
    // Consumer warps: kSplit per TMEM lane quarter, each taking kStepsW of a
    // group's K steps and kColsW of the accumulator's 16 columns.
    static constexpr int kCW = 8;
    static constexpr int kSplit = kCW / 4;
    static constexpr int kStepsW = kSteps / kSplit;
    static constexpr int kColsW = kN / kSplit;
    static constexpr int kWordsW = BITS == 4 ? 2 * kStepsW : kStepsW;  // packed words per warp per group
    static constexpr int kProducerWarp = kCW;
    static constexpr int kMmaWarp = kCW + 1;
    static constexpr int kThreads = 32 * (kCW + 2);
    static constexpr int kStages = clamp_tc(kSmemBudgetTc / kStageBytes, 2, 8);
    static constexpr int kBarOffset = kStages * kStageBytes;
    static constexpr int kSmemBytes = kBarOffset + 512 + 1024;  // barriers/flags + align slack
    // Consumers work in batches of kR groups (half a stage): unpack and store a
    // batch's A tiles, retire the stores once, then read back the previous
    // batch's accumulators.  2 kR slots: a slot is rewritten two batches after
    // its last use, by which time its accumulator has been read.
    static constexpr int kR = kGPS / 2;
    static constexpr int kNB = 2 * kR;
    // Zero point on the tensor core where tensor memory allows: per group an
    // 8-column tile holding -(128 + z) in every column of the row, and one
    // more MMA per K step; otherwise q - z is formed on the CUDA cores.
    static constexpr bool kZtc = (kNB * (kACols + 8) + 15) / 16 * 16 + kNB * kN <= kTmemCols;
    static constexpr uint32_t kColA = 0;                        // kNB A tiles
    static constexpr uint32_t kColZ = kNB * kACols;             // kNB zero-point tiles
    static constexpr uint32_t kColD = (kColZ + (kZtc ? kNB * 8 : 0) + 15) / 16 * 16;  // accumulators
    static_assert(kColD + kNB * kN <= kTmemCols, "tensor memory budget");
    static_assert(kColD % 16 == 0, "accumulators 16-column aligned");
};

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, bits 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(kN >> 3) << 17) |
                            (uint32_t(128 >> 4) << 24);

// Shared-memory matrix descriptor of a K-major operand stored with the 128-byte
// swizzle in 8-row x 128-byte atoms (the layout the TMA writes): start address
// >> 4 in bits 0-13, leading offset (unused for this layout) 1, stride between
// 8-row atoms 1024 bytes (>> 4) in bits 32-45, version 1 in bits 46-47,
// layout "128-byte swizzle" (2) in bits 61-63.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3fffu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// Scale / zero point of the GPS groups of one stage for one row.
template <int GPS>
struct RowMeta {
    static constexpr int kS = (GPS + 1) / 2;
    static constexpr int kZ = (GPS + 3) / 4;
    uint32_t s[kS];
    uint32_t z[kZ];

    __device__ __forceinline__ void load(const GemmArgs& a, int n, long long g0, bool vec) {
#pragma unroll
        for (int j = 0; j < kS; ++j) s[j] = 0;
#pragma unroll
        for (int j = 0; j < kZ; ++j) z[j] = 0;
        if (n >= a.N) return;
        const long long base = static_cast<long long>(n) * a.ng + g0;
        if (vec) {
            const uint16_t* sp = a.scales + base;
            const uint8_t* zp = a.zeros + base;
            if (GPS == 2) {
                s[0] = __ldg(reinterpret_cast<const uint32_t*>(sp));
                z[0] = __ldg(reinterpret_cast<const uint16_t*>(zp));
            } else if (GPS == 4) {
                const uint2 v = __ldg(reinterpret_cast<const uint2*>(sp));
                s[0] = v.x; s[kS > 1 ? 1 : 0] = v.y;
                z[0] = __ldg(reinterpret_cast<const uint32_t*>(zp));
            } else if (GPS == 8) {
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(sp));
                s[0] = v.x; s[kS > 1 ? 1 : 0] = v.y; s[kS > 2 ? 2 : 0] = v.z; s[kS > 3 ? 3 : 0] = v.w;
                const uint2 w = __ldg(reinterpret_cast<const uint2*>(zp));
                z[0] = w.x; z[kZ > 1 ? 1 : 0] = w.y;
            } else {
#pragma unroll
                for (int j = 0; j < kS / 4; ++j) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4*>(sp) + j);
                    s[4 * j] = v.x; s[4 * j + 1] = v.y; s[4 * j + 2] = v.z; s[4 * j + 3] = v.w;
                }
#pragma unroll
                for (int j = 0; j < kZ / 4; ++j) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4*>(zp) + j);
                    z[4 * j] = v.x; z[4 * j + 1] = v.y; z[4 * j + 2] = v.z; z[4 * j + 3] = v.w;
                }
            }
        } else {
#pragma unroll
            for (int gi = 0; gi < GPS; ++gi) {
                if (g0 + gi < a.ng) {
                    s[gi / 2] |= static_cast<uint32_t>(__ldg(a.scales + base + gi)) << (16 * (gi & 1));
                    z[gi / 4] |= static_cast<uint32_t>(__ldg(a.zeros + base + gi)) << (8 * (gi & 3));
                }
            }
        }
    }

    __device__ __forceinline__ float scale(int gi) const {
        const uint32_t w = s[gi / 2];
        return __uint_as_float((gi & 1) ? (w & 0xffff0000u) : (w << 16));
    }
    // bf16x2 (128 + z, 128 + z): low byte z, high byte 0x43, both halves.
    __device__ __forceinline__ uint32_t zero_point(int gi) const {
        return __byte_perm(z[gi / 4], 0x43u, 0x4040u | (0x0101u * static_cast<uint32_t>(gi & 3)));
    }
    // bf16x2 (-(128 + z), -(128 + z)): high byte 0xC3.
    __device__ __forceinline__ uint32_t neg_zero_point(int gi) const {
        return __byte_perm(z[gi / 4], 0xc3u, 0x4040u | (0x0101u * static_cast<uint32_t>(gi & 3)));
    }
};

// bf16x2 (128 + lo, 128 + hi) from the low nibble (or 2-bit field, per
// `mask`) of bytes `sel`-picked from two words.
__device__ __forceinline__ uint32_t magic_bytes(uint32_t a, uint32_t b, uint32_t sel, uint32_t mask) {
    return lop3_and_or(__byte_perm(a, b, sel), mask, 0x43004300u);
}

// Optional exact bf16x2 subtraction of zz = (128 + z, 128 + z).
template <bool SUB>
__device__ __forceinline__ uint32_t minus_zero(uint32_t v, uint32_t zz) {
    return SUB ? bf16x2_sub(v, zz) : v;
}

// Eight bf16x2 registers (k = 0..15 in natural order) from two 4-bit words:
// q - z if SUB, else 128 + q.
template <bool SUB>
__device__ __forceinline__ void unpack4_k16(uint32_t w0, uint32_t w1, uint32_t zz, uint32_t (&p)[8]) {
    const uint32_t v0 = w0 >> 4, v1 = w1 >> 4;
    p[0] = minus_zero<SUB>(magic_bytes(w0, v0, 0x4400u, 0x000f000fu), zz);
    p[1] = minus_zero<SUB>(magic_bytes(w0, v0, 0x5511u, 0x000f000fu), zz);
    p[2] = minus_zero<SUB>(magic_bytes(w0, v0, 0x6622u, 0x000f000fu), zz);
    p[3] = minus_zero<SUB>(magic_bytes(w0, v0, 0x7733u, 0x000f000fu), zz);
    p[4] = minus_zero<SUB>(magic_bytes(w1, v1, 0x4400u, 0x000f000fu), zz);
    p[5] = minus_zero<SUB>(magic_bytes(w1, v1, 0x5511u, 0x000f000fu), zz);
    p[6] = minus_zero<SUB>(magic_bytes(w1, v1, 0x6622u, 0x000f000fu), zz);
    p[7] = minus_zero<SUB>(magic_bytes(w1, v1, 0x7733u, 0x000f000fu), zz);
}

// Eight bf16x2 registers (k = 0..15 in natural order) from one 2-bit word:
// q - z if SUB, else 128 + q.
template <bool SUB>
__device__ __forceinline__ void unpack2_k16(uint32_t w, uint32_t zz, uint32_t (&p)[8]) {
    const uint32_t u1 = w >> 2, u2 = w >> 4, u3 = w >> 6;
    p[0] = minus_zero<SUB>(magic_bytes(w, u1, 0x4400u, 0x00030003u), zz);
    p[1] = minus_zero<SUB>(magic_bytes(u2, u3, 0x4400u, 0x00030003u), zz);
    p[2] = minus_zero<SUB>(magic_bytes(w, u1, 0x5511u, 0x00030003u), zz);
    p[3] = minus_zero<SUB>(magic_bytes(u2, u3, 0x5511u, 0x00030003u), zz);
    p[4] = minus_zero<SUB>(magic_bytes(w, u1, 0x6622u, 0x00030003u), zz);
    p[5] = minus_zero<SUB>(magic_bytes(u2, u3, 0x6622u, 0x00030003u), zz);
    p[6] = minus_zero<SUB>(magic_bytes(w, u1, 0x7733u, 0x00030003u), zz);
    p[7] = minus_zero<SUB>(magic_bytes(u2, u3, 0x7733u, 0x00030003u), zz);
}

__device__ __forceinline__ void record_error_tc(const GemmArgs& a, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicExch(a.err, 1);
}

// NW consecutive packed words starting at word `wi0` of a 128-byte-swizzled row.
template <int NW>
__device__ __forceinline__ void load_words(const uint8_t* row, int wi0, int r, uint32_t (&w)[NW]) {
    const int sw = r & 7;
    if (NW >= 4) {
#pragma unroll
        for (int j = 0; j < NW / 4; ++j) {
            const int chunk = wi0 / 4 + j;
            const uint4 v = *reinterpret_cast<const uint4*>(row + ((chunk ^ sw) << 4));
            w[4 * j] = v.x; w[4 * j + 1] = v.y; w[4 * j + 2] = v.z; w[4 * j + 3] = v.w;
        }
    } else if (NW == 2) {
        const uint2 v = *reinterpret_cast<const uint2*>(row + (((wi0 / 4) ^ sw) << 4) + (wi0 & 3) * 4);
        w[0] = v.x; w[NW > 1 ? 1 : 0] = v.y;
    } else {
        w[0] = *reinterpret_cast<const uint32_t*>(row + (((wi0 / 4) ^ sw) << 4) + (wi0 & 3) * 4);
    }
}

// Segment end for one thread (row r, columns C h .. C h + C - 1): store Y, or
// publish the partial and let the last CTA of the tile sum all partials in k
// order.  NCT = consumer threads (named barrier 1).
template <int C, int NCT>
__device__ __forceinline__ void finish_tile(const GemmArgs& a, const float (&acc)[C], int t,
                                           bool whole, long long u_lo, int r, int h, int tid,
                                           bool dead, volatile int* abort_flag,
                                           volatile int* last_flag) {
    const int n = t * kBN + r;
    if (whole) {
        if (!dead && n < a.N)
#pragma unroll
            for (int j = 0; j < C; ++j)
                if (C * h + j < a.M) a.y[static_cast<size_t>(C * h + j) * a.N + n] = acc[j];
        return;
    }
    const int t_first = static_cast<int>(u_lo / a.I);
    float* mine = a.partials + static_cast<size_t>(2 * blockIdx.x + (t == t_first ? 0 : 1)) *
                                   (kMaxCols * kBN);
#pragma unroll
    for (int j = 0; j < C; ++j) __stcg(mine + (C * h + j) * kBN + r, acc[j]);
    named_bar_sync(1, NCT);
    const long long tu0 = static_cast<long long>(t) * a.I;
    const int b_first = static_cast<int>(((tu0 + 1) * a.P + a.U - 1) / a.U - 1);
    const int b_last = static_cast<int>(((tu0 + a.I) * a.P + a.U - 1) / a.U - 1);
    if (tid == 0) {
        if (*abort_flag) {
            *last_flag = 0;
        } else {
            const int prev = atomic_add_acq_rel_gpu(a.counters + t, 1);
            *last_flag = (prev == b_last - b_first) ? 1 : 0;
        }
    }
    named_bar_sync(1, NCT);
    if (*last_flag) {
        float tot[C];
#pragma unroll
        for (int j = 0; j < C; ++j) tot[j] = 0.f;
        for (int b = b_first; b <= b_last; ++b) {
            if (b == static_cast<int>(blockIdx.x)) {
#pragma unroll
                for (int j = 0; j < C; ++j) tot[j] += acc[j];
            } else {
                const int tb = static_cast<int>((a.U * b / a.P) / a.I);
                const float* src = a.partials +
                                   static_cast<size_t>(2 * b + (t == tb ? 0 : 1)) * (kMaxCols * kBN);
#pragma unroll
                for (int j = 0; j < C; ++j) tot[j] += __ldcg(src + (C * h + j) * kBN + r);
            }
        }
        if (n < a.N)
#pragma unroll
            for (int j = 0; j < C; ++j)
                if (C * h + j < a.M) a.y[static_cast<size_t>(C * h + j) * a.N + n] = tot[j];
        if (tid == 0) a.counters[t] = 0;
    }
    named_bar_sync(1, NCT);
}

template <int BITS, int G>
__global__ void __launch_bounds__(Lay<BITS, G>::kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const GemmArgs a) {
    using L = Lay<BITS, G>;
    constexpr int S = L::kStages;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::kBarOffset);
    uint64_t* empty = full + S;
    uint64_t* filled = empty + S;        // slot's A tile written (8 consumer warps)
    uint64_t* done = filled + L::kNB;    // slot's MMAs complete (tcgen05.commit)
    uint64_t* drain = done + L::kNB;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* last_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], L::kCW + 1);  // consumers read W, MMAs read X
        }
        for (int i = 0; i < L::kNB; ++i) {
            mbar_init(&filled[i], L::kCW);
            mbar_init(&done[i], 1);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
    }
    if (warp == L::kMmaWarp) {
        tmem_alloc(smem_addr(tmem_slot), kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    const long long u_lo = a.U * blockIdx.x / a.P;
    const long long u_hi = a.U * (blockIdx.x + 1) / a.P;
    const int n_units = static_cast<int>(u_hi - u_lo);
    const int t_first = static_cast<int>(u_lo / a.I);
    const int i_first = static_cast<int>(u_lo - static_cast<long long>(t_first) * a.I);

    if (warp == L::kProducerWarp) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        prefetch_tensormap(&tmW);
        prefetch_tensormap(&tmX);
        const uint64_t pol_w = policy_evict_first();
        const uint64_t pol_x = policy_evict_last();
        int t = t_first, i = i_first;
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
            if (!mbar_wait(&empty[slot], ((it / S) & 1u) ^ 1u, abort_flag)) {
                record_error_tc(a, abort_flag);
                ok = false;
                break;
            }
            uint8_t* st = smem + slot * L::kStageBytes;
            mbar_arrive_expect_tx(&full[slot], L::kWBytes + L::kXBytes);
#pragma unroll
            for (int b = 0; b < L::kBoxes; ++b)
                tma_load_2d(st + b * L::kBoxBytes, &tmW, (i * L::kBoxes + b) * kWordsPerStage, t * kBN,
                            &full[slot], pol_w);
            if (a.x3d) {
                tma_load_3d(st + L::kWBytes, &tmX, 0, 0, i * L::kXBoxes, &full[slot], pol_x);
            } else {
#pragma unroll
                for (int b = 0; b < L::kXBoxes; ++b)
                    tma_load_2d(st + L::kWBytes + b * L::kXBoxBytes, &tmX,
                                i * L::kStageValues + b * L::kXBoxValues, 0, &full[slot], pol_x);
            }
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

    if (warp == L::kMmaWarp) {
        // --------------------------------------------------------- MMA issuer
        // The whole warp walks the schedule (uniform control flow); one
        // elected lane issues the MMAs and commits.
        uint32_t gl = 0;
        bool ok = true;
        for (int k = 0; k < n_units && ok; ++k) {
            const int slot = k % S;
            if (!__all_sync(0xffffffffu, mbar_wait(&full[slot], (static_cast<uint32_t>(k) / S) & 1u,
                                                   abort_flag))) {
                ok = false;
                break;
            }
            const uint64_t desc0 = desc_sw128(smem_addr(smem + slot * L::kStageBytes + L::kWBytes));
#pragma unroll
            for (int gi = 0; gi < L::kGPS; ++gi, ++gl) {
                const uint32_t sb = gl % L::kNB;
                if (!__all_sync(0xffffffffu, mbar_wait(&filled[sb], (gl / L::kNB) & 1u, abort_flag))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (elect_one()) {
                    const uint32_t tA = tmem + L::kColA + sb * L::kACols;
                    const uint32_t tD = tmem + L::kColD + sb * kN;
#pragma unroll
                    for (int s = 0; s < L::kSteps; ++s) {
                        const int v0 = gi * G + 16 * s;  // first value of this K step in the stage
                        const uint64_t bdesc =
                            desc0 + static_cast<uint64_t>(((v0 / 64) * L::kXBoxBytes + (v0 % 64) * 2) >> 4);
                        tc_mma_ts(tD, tA + 8 * s, bdesc, kIdesc, s > 0 ? 1u : 0u);
                        if (L::kZtc) tc_mma_ts(tD, tmem + L::kColZ + sb * 8, bdesc, kIdesc, 1u);
                    }
                    tc_commit(&done[sb]);
                    if (gi == L::kGPS - 1) tc_commit(&empty[slot]);
                }
                __syncwarp();
            }
        }
        if (!ok && lane == 0) record_error_tc(a, abort_flag);
        // every MMA issued above has completed once `drain` flips
        if (elect_one()) tc_commit(drain);
        __syncwarp();
        volatile int never = 0;
        mbar_wait(drain, 0, &never);
        named_bar_sync(3, 32 * (L::kCW + 1));
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
        return;
    }

    // ---------------------------------------------------------------- consumers
    const int tid = threadIdx.x;  // 0 .. 255
    const int q = warp & 3;       // TMEM lane quarter
    const int h = warp >> 2;      // which K steps of each group (and columns of D) this warp takes
    const int r = 32 * q + lane;  // tile row == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(32 * q) << 16;
    const bool vec = a.meta_vec != 0;
    // After a failed wait a warp stops touching tensor memory but keeps
    // arriving on barriers and walking the named barriers of its siblings.
    bool dead = false;
    constexpr int C = L::kColsW;
    float acc[C];
#pragma unroll
    for (int j = 0; j < C; ++j) acc[j] = 0.f;

    using RM = RowMeta<L::kGPS>;
    int t = t_first, i = i_first;    // unit being computed
    int pt = t_first, pi = i_first;  // unit whose group values are fetched next
    uint32_t gl = 0;  // groups whose A tiles were written
    // Scales of the previous stage and that stage's segment bookkeeping: its
    // second batch is read back during the next stage.
    uint32_t sprev[RM::kS];
#pragma unroll
    for (int j = 0; j < RM::kS; ++j) sprev[j] = 0;
    int prev_t = 0;
    bool prev_end = false, prev_whole = false;

    auto fetch = [&](RM& m) {
        m.load(a, pt * kBN + r, static_cast<long long>(pi) * L::kGPS, vec);
        if (++pi == a.I) {
            pi = 0;
            ++pt;
        }
    };
    auto scale_of = [](const uint32_t* s, int gi) {
        const uint32_t w = s[gi / 2];
        return __uint_as_float((gi & 1) ? (w & 0xffff0000u) : (w << 16));
    };
    auto finish = [&](int tt, bool wh) {
        finish_tile<C, 32 * L::kCW>(a, acc, tt, wh, u_lo, r, h, tid, dead, abort_flag, last_flag);
#pragma unroll
        for (int j = 0; j < C; ++j) acc[j] = 0.f;
    };
    // Read back the accumulators of the kR groups [g0, g0 + kR), whose scales
    // are s[first .. first + kR), and add scale * D to acc.
    auto read_batch = [&](uint32_t g0, const uint32_t* s, int first) {
        const uint32_t glast = g0 + L::kR - 1;  // MMAs complete in order
        if (!dead && !mbar_wait(&done[glast % L::kNB], (glast / L::kNB) & 1u, abort_flag)) {
            record_error_tc(a, abort_flag);
            dead = true;
        }
        if (dead) return;
        tc_fence_after();
        uint32_t v[L::kR][C];
#pragma unroll
        for (int j = 0; j < L::kR; ++j)
            tmem_ld_cols<C>(tmem + L::kColD + ((g0 + j) % L::kNB) * kN + C * h + lane_off, v[j]);
        tmem_wait_ld();
#pragma unroll
        for (int j = 0; j < L::kR; ++j) {
            const float sc = scale_of(s, first + j);
#pragma unroll
            for (int jj = 0; jj < C; ++jj) acc[jj] = fmaf(sc, __uint_as_float(v[j][jj]), acc[jj]);
        }
    };
    // Unpack and store the A tiles of groups [gb, gb + kR) of the stage.
    auto write_batch = [&](const RM& m, const uint8_t* row0, int gb) {
        if (!dead) {
#pragma unroll
            for (int j = 0; j < L::kR; ++j) {
                const int gi = gb + j;
                const uint32_t sb = (gl + j) % L::kNB;
                uint32_t w[L::kWordsW];
                const uint32_t zz = m.zero_point(gi);
                const int wi = (BITS == 4 ? gi * (G / 8) : gi * (G / 16)) + h * L::kWordsW;
                load_words<L::kWordsW>(row0 + (wi / kWordsPerStage) * L::kBoxBytes,
                                       wi % kWordsPerStage, r, w);
                const uint32_t tA = tmem + L::kColA + sb * L::kACols + lane_off;
#pragma unroll
                for (int hs = 0; hs < L::kStepsW; ++hs) {
                    uint32_t p[8];
                    if (BITS == 4) {
                        unpack4_k16<!L::kZtc>(w[2 * hs], w[2 * hs + 1], zz, p);
                    } else {
                        unpack2_k16<!L::kZtc>(w[hs], zz, p);
                    }
                    tmem_st8(tA + 8 * (h * L::kStepsW + hs), p);
                }
                if (L::kZtc && h == 0)
                    tmem_st8_same(tmem + L::kColZ + sb * 8 + lane_off, m.neg_zero_point(gi));
            }
            tmem_wait_st();
            tc_fence_before();
        }
        __syncwarp();
        if (lane == 0)
#pragma unroll
            for (int j = 0; j < L::kR; ++j) mbar_arrive(&filled[(gl + j) % L::kNB]);
        gl += L::kR;
    };
    auto unit = [&](const RM& m, int k) {
        const int slot = k % S;
        if (!dead && !mbar_wait(&full[slot], (static_cast<uint32_t>(k) / S) & 1u, abort_flag)) {
            record_error_tc(a, abort_flag);
            dead = true;
        }
        const uint8_t* row0 = smem + slot * L::kStageBytes + r * 128;
        // first batch; then the previous stage's second batch is read back
        write_batch(m, row0, 0);
        if (k > 0) {
            read_batch(gl - 2 * L::kR, sprev, L::kR);
            if (prev_end) finish(prev_t, prev_whole);
        }
        // second batch; the stage's words are then no longer needed
        write_batch(m, row0, L::kR);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
        read_batch(gl - 2 * L::kR, m.s, 0);
#pragma unroll
        for (int j = 0; j < RM::kS; ++j) sprev[j] = m.s[j];
        prev_t = t;
        prev_end = (i == a.I - 1) || (k == n_units - 1);
        prev_whole = (i == a.I - 1) && (t != t_first || i_first == 0);
        if (++i == a.I) {
            i = 0;
            ++t;
        }
    };

    RM m0, m1;
    if (n_units > 0) fetch(m0);
    if (n_units > 1) fetch(m1);
    for (int k = 0; k < n_units; k += 2) {
        unit(m0, k);
        if (k + 2 < n_units) fetch(m0);
        if (k + 1 < n_units) {
            unit(m1, k + 1);
            if (k + 3 < n_units) fetch(m1);
        }
    }
    if (n_units > 0) {
        // the last stage's second batch
        read_batch(gl - L::kR, sprev, L::kR);
        finish(prev_t, prev_whole);
    }
    named_bar_sync(3, 32 * (L::kCW + 1));
}

template <int BITS, int G>
cudaError_t launch_tc(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmArgs& a,
                      cudaStream_t s) {
    using L = Lay<BITS, G>;
    auto kern = gemm_tc_kernel<BITS, G>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
    if (e != cudaSuccess) return e;
    kern<<<a.P, L::kThreads, L::kSmemBytes, s>>>(tmW, tmX, a);
    return cudaGetLastError();
}

}  // namespace tc
}  // namespace wq
