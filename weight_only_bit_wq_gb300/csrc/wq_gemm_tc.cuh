// Weight-only low-bit skinny GEMM on the 5th-generation tensor core (sm_103a):
//     Y[M][N] = X[M][K] . dequant(Wq)[N][K]^T,  M <= 32, 2/3/4-bit codes.
//
// A decode-step projection streams every packed weight once and multiplies it,
// while on chip, against all stacked rows of X on tensor cores (OpenJet news
// page, paragraph "并行解码的原理").  One CTA per SM, persistent, stream-K over
// (128-row tile, k-stage) units; the split depends on (N, K, bits, group, SM
// count) only.  Warp roles (warp-specialised, connected by mbarrier rings):
//
// * TMA producer (one lane): per stage one or two 128-row x 128-byte boxes of
//   packed words and the matching X slice (NC = 16 or 32 rows x stage width,
//   rows >= M read as zero), all 128-byte swizzled, into a ring of
//   shared-memory stages;
// * unpack warps (two per TMEM lane quarter, each taking half of every
//   group's K steps): one weight row per thread.  The "magic number" trick
//   turns codes into bf16 — a code q placed in the mantissa of 128.0 reads as
//   128 + q exactly — and the word layout (even-numbered codes in the low
//   half-word, odd-numbered in the high half-word) makes one shift and one
//   LOP3 produce the bf16 pair of two neighbouring codes.  The pairs go to
//   tensor memory (tcgen05.st) as the MMA's A tile;
// * MMA issuer (one elected lane; the warp also owns the TMEM allocation):
//   tcgen05.mma kind::f16, M = 128 weight rows, N = 16 rows of X, K = 16
//   (two such MMAs, one per 16 rows, when the tile carries 32 rows of X),
//   A from tensor memory, B (X) straight from the swizzled shared tile
//   through a matrix descriptor, fp32 D per group in tensor memory.  The zero
//   point is applied on the tensor core: a second MMA per K step multiplies
//   the same X by a constant A tile holding -(128 + z) in every column of the
//   row (written by the unpack warps), so each group's D is sum_k x (q - z)
//   (where tensor memory is too small for those tiles, q - z is formed on
//   the CUDA cores instead);
// * epilogue warps (one per lane quarter): read each group's D back
//   (tcgen05.ld), add scale * D to the row's NC fp32 sums, and store Y (or
//   the gate/up activation) or publish a split-K partial.
//
// Tensor memory holds rings of A-tile batch slots and accumulator slots, so
// the unpack warps run ahead of the tensor core and never wait for a result.
// Per group the D accumulation order is fixed (data MMA then zero-point MMA
// per K step, K steps ascending) and the columns of one MMA never interact,
// so a row of X gives bit-identical results alone or stacked; a 32-row tile
// issues for rows 16..31 the same N = 16 MMA as for rows 0..15, so rows agree
// between the 16- and the 32-row builds too.  A tile split
// across CTAs is summed by the last CTA to finish it, in k order.
#pragma once
#include <cuda_bf16.h>
#include <type_traits>

#include "wq_internal.h"
#include "wq_ptx.cuh"

namespace wq {
namespace tc {

constexpr int kMmaN = 16;  // N of one MMA: 16 rows of X
constexpr uint32_t kTmemCols = 512;
// Shared memory for the stage ring: 16-row builds keep the stage counts
// measured with this budget; 32-row builds take a little more so that every
// format keeps three stages.
constexpr int smem_budget_tc(int nc) { return (nc == 16 ? 220 : 226) * 1024; }
// Unpack warps per TMEM lane quarter (each takes 1 / kSplitWarps of a
// group's K steps): two per lane quarter measured best; more add per-warp
// overhead without adding ALU throughput.
constexpr int kSplitWarps = 2;
// TMEM columns per tcgen05.st of the unpacked A tile: one K step (8 columns)
// per store lets the stores start while the rest of the group is unpacked.
constexpr int kStoreCols = 8;
constexpr uint32_t kFull = 0xffffffffu;

constexpr int round_up_tc(int v, int a) { return (v + a - 1) / a * a; }
constexpr int clamp_tc(int v, int lo, int hi) { return v < lo ? lo : (v > hi ? hi : v); }

// Tensor-memory plan for batch slots of R groups: returns 100 z + 10 na + nd
// for the first of (zero point on the tensor core z, na A slots, nd
// accumulator slots) that fits, trying z = 1 before z = 0, then two
// accumulator slots before one, then three A slots before two, and a single
// A slot only when nothing else fits; 0 if none fits.  z_only >= 0 fixes z:
// the 32-row build keeps the 16-row build's zero-point method, whose fp32
// rounding differs, so that rows agree bitwise between the two builds.
// z0_first: try the zero point on the CUDA cores (z = 0) first.
constexpr int tmem_plan(int R, int a_cols, int n, int cols, int z_only = -1,
                        bool z0_first = false) {
    if (z0_first && z_only < 0) z_only = 0;
    for (int z = 1; z >= 0; --z) {
        if (z_only >= 0 && z != z_only) continue;
        for (int nd = 2; nd >= 1; --nd)
            for (int na = 3; na >= 2; --na)
                if (round_up_tc(na * R * (a_cols + 8 * z), 16) + nd * R * n <= cols)
                    return 100 * z + 10 * na + nd;
        for (int nd = 2; nd >= 1; --nd)
            if (round_up_tc(R * (a_cols + 8 * z), 16) + nd * R * n <= cols)
                return 100 * z + 10 + nd;
    }
    return 0;
}

// Layout of a build for BITS-bit codes, group size G and NC rows of X per
// tile (16 for M <= 16, 32 for M <= 32).
template <int BITS, int G, int NC = 16>
struct Lay {
    static_assert(NC == 16 || NC == 32, "16 or 32 rows of X");
    static constexpr int kVpw = values_per_word(BITS);
    static constexpr int kPpw = kVpw / 2;                    // bf16 pairs per word
    static constexpr int kBoxes = tc_boxes(BITS, G);         // 32-word boxes per row per stage
    static constexpr int kStageWords = kBoxes * kWordsPerStage;
    static constexpr int kStageValues = kStageWords * kVpw;
    static_assert(kStageValues % G == 0, "whole groups per stage");
    static_assert(kStageValues % 64 == 0, "whole 64-value X boxes per stage");
    static constexpr int kBoxBytes = kBN * kWordsPerStage * 4;  // 16 KB
    static constexpr int kWBytes = kBoxes * kBoxBytes;
    static constexpr int kXBoxValues = 64;                      // 128 bytes of bf16
    static constexpr int kXBoxes = kStageValues / kXBoxValues;
    static constexpr int kXBoxBytes = NC * 128;                 // NC rows x 128 bytes
    static constexpr int kXBytes = kXBoxes * kXBoxBytes;
    static constexpr int kGPS = kStageValues / G;               // groups per stage
    // The stage also carries its rows' zero points, kZRow bytes per row (kGPS
    // rounded up to 4, 8 or 16 bytes for aligned shared loads), staged by the
    // producer warp.
    static constexpr int kZRow = kGPS <= 4 ? 4 : kGPS <= 8 ? 8 : 16;
    static constexpr int kZOff = kWBytes + kXBytes;
    static constexpr int kZStageBytes = kBN * kZRow;
    static constexpr bool kZAsync = kZRow == kGPS && (kZRow == 4 || kZRow == 8 || kZRow == 16);
    static constexpr int kStageBytes = round_up_tc(kWBytes + kXBytes + kZStageBytes, 1024);
    static constexpr int kSteps = G / 16;                       // K16 steps per group
    static constexpr int kACols = kSteps * 8;                   // TMEM columns of one A tile
    // Warp roles: kUW unpack warps (kSplit per TMEM lane quarter, each taking
    // kStepsW of every group's K steps), four epilogue warps (one per lane
    // quarter, all 16 accumulator columns), one TMA producer, one MMA issuer.
    static constexpr int kSplit = (kSteps >= kSplitWarps) ? kSplitWarps : kSteps;
    static constexpr int kUW = 4 * kSplit;
    static constexpr int kEW = 4;
    static constexpr int kProducerWarp = kUW + kEW;
    static constexpr int kMmaWarp = kProducerWarp + 1;
    static constexpr int kThreads = 32 * (kMmaWarp + 1);
    static constexpr int kStepsW = kSteps / kSplit;             // K steps per warp per group
    static constexpr int kPairsW = 8 * kStepsW;                 // bf16 pairs per thread per group
    // A stage's groups go through the tensor core in two batches, [0, kR0)
    // and [kR0, kGPS); a batch slot in tensor memory holds kR0 groups.
    static constexpr int kR0 = (kGPS + 1) / 2;
    static constexpr int kStages = clamp_tc(smem_budget_tc(NC) / kStageBytes, 2, 8);
    static constexpr int kBarOffset = kStages * kStageBytes;
    static constexpr int kSmemBytes = kBarOffset + 512 + 1024;  // barriers/flags + align slack
    // Cluster builds (a tile's k <= kFixMaxK contributors in one cluster): the
    // partials of ranks 1 .. k-1 land in rank 0's shared memory after the
    // barriers, [rank - 1][row][NC] fp32.
    static constexpr int kFixMaxK = 4;
    static constexpr int kFixOff = kBarOffset + 512;
    static constexpr int kFixBytes = (kFixMaxK - 1) * kBN * NC * 4;
    static constexpr int kSmemBytesClu = kSmemBytes + kFixBytes;
    static constexpr bool kCluOk = NC == 16 && kSmemBytesClu <= 232448;
    // Tensor memory: kNA batch slots of A tiles (plus zero-point tiles when
    // the zero point goes on the tensor core) and kND batch slots of fp32
    // accumulators, the largest plan that fits in 512 columns.
    // 2-bit codes in groups of 32 and 64 measured faster with the zero point
    // on the CUDA cores, which leaves tensor memory for more slots (groups of
    // 32: two accumulator slots instead of one, a 2-bit 5120 x 17408 GEMM at
    // 8 rows 22.2 -> 20.2 us; groups of 64: three A slots instead of two,
    // 19.15 -> 19.0 us, and 32.4 -> 31.4 us for 34816 x 5120 at 12 rows).
    // 3-bit groups of 128 (22.5 -> 26.8 us), 3-bit groups of 32 and 4-bit
    // groups of 64 (1.5-2.6 % slower) keep the zero point on the tensor core.
    static constexpr int kPlan16 =
        tmem_plan(kR0, kACols, 16, int(kTmemCols), -1, BITS == 2 && G <= 64);
    static constexpr int kPlan =
        NC == 16 ? kPlan16 : tmem_plan(kR0, kACols, NC, int(kTmemCols), kPlan16 / 100);
    static constexpr bool kZtc = kPlan / 100 != 0;
    static constexpr int kNA = (kPlan / 10) % 10;
    static constexpr int kND = kPlan % 10;
    static constexpr uint32_t kColA = 0;                                        // [kNA][kR0][kACols]
    static constexpr uint32_t kColZ = kNA * kR0 * kACols;                       // [kNA][kR0][8]
    static constexpr uint32_t kColD = round_up_tc(kColZ + (kZtc ? kNA * kR0 * 8 : 0), 16);  // [kND][kR0][NC]
    static_assert(kPlan > 0, "no tensor-memory plan fits");
    static_assert(kColD + kND * kR0 * NC <= kTmemCols, "tensor memory budget");
    static_assert(kPairsW == 8 || kPairsW == 16 || kPairsW == 32, "tcgen05.st width");
    static_assert(kEW <= kCountersPerTile, "one split-K counter per epilogue warp");
    static_assert(kR0 >= 1 && kGPS - kR0 >= 1, "two non-empty batches");
};

// Instruction descriptor, kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, bits 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(kMmaN >> 3) << 17) |
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

// Scales (bf16 pairs) and zero points (byte quads) of the GPS groups of one
// stage for one row.
template <int GPS>
struct RowMeta {
    static constexpr int kS = (GPS + 1) / 2;
    static constexpr int kZ = (GPS + 3) / 4;
    uint32_t s[kS];
    uint32_t z[kZ];

    template <class V>
    __device__ __forceinline__ void load(const V& a, int n, long long g0) {
#pragma unroll
        for (int j = 0; j < kS; ++j) s[j] = 0;
#pragma unroll
        for (int j = 0; j < kZ; ++j) z[j] = 0;
        if (n >= a.N) return;
        const long long base = static_cast<long long>(n) * a.ng + g0;
        if constexpr (GPS == 4 || GPS == 8 || GPS == 16) {
            if (a.meta_vec) {
                const uint16_t* sp = a.scales + base;
                const uint8_t* zp = a.zeros + base;
                if constexpr (GPS == 4) {
                    const uint2 v = __ldg(reinterpret_cast<const uint2*>(sp));
                    s[0] = v.x;
                    s[1] = v.y;
                    z[0] = __ldg(reinterpret_cast<const uint32_t*>(zp));
                } else if constexpr (GPS == 8) {
                    const uint4 v = __ldg(reinterpret_cast<const uint4*>(sp));
                    s[0] = v.x;
                    s[1] = v.y;
                    s[2] = v.z;
                    s[3] = v.w;
                    const uint2 w = __ldg(reinterpret_cast<const uint2*>(zp));
                    z[0] = w.x;
                    z[1] = w.y;
                } else {
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        const uint4 v = __ldg(reinterpret_cast<const uint4*>(sp) + j);
                        s[4 * j] = v.x;
                        s[4 * j + 1] = v.y;
                        s[4 * j + 2] = v.z;
                        s[4 * j + 3] = v.w;
                    }
                    const uint4 w = __ldg(reinterpret_cast<const uint4*>(zp));
                    z[0] = w.x;
                    z[1] = w.y;
                    z[2] = w.z;
                    z[3] = w.w;
                }
                return;
            }
        }
#pragma unroll
        for (int gi = 0; gi < GPS; ++gi) {
            if (g0 + gi < a.ng) {
                s[gi / 2] |= static_cast<uint32_t>(__ldg(a.scales + base + gi)) << (16 * (gi & 1));
                z[gi / 4] |= static_cast<uint32_t>(__ldg(a.zeros + base + gi)) << (8 * (gi & 3));
            }
        }
    }

    // Zero points only (the unpack warps need nothing else).
    template <class V>
    __device__ __forceinline__ void load_z(const V& a, int n, long long g0) {
#pragma unroll
        for (int j = 0; j < kZ; ++j) z[j] = 0;
        if (n >= a.N) return;
        const long long base = static_cast<long long>(n) * a.ng + g0;
        if constexpr (GPS == 4 || GPS == 8 || GPS == 16) {
            if (a.meta_vec) {
                const uint8_t* zp = a.zeros + base;
                if constexpr (GPS == 4) {
                    z[0] = __ldg(reinterpret_cast<const uint32_t*>(zp));
                } else if constexpr (GPS == 8) {
                    const uint2 w = __ldg(reinterpret_cast<const uint2*>(zp));
                    z[0] = w.x;
                    z[1] = w.y;
                } else {
                    const uint4 w = __ldg(reinterpret_cast<const uint4*>(zp));
                    z[0] = w.x;
                    z[1] = w.y;
                    z[2] = w.z;
                    z[3] = w.w;
                }
                return;
            }
        }
#pragma unroll
        for (int gi = 0; gi < GPS; ++gi)
            if (g0 + gi < a.ng)
                z[gi / 4] |= static_cast<uint32_t>(__ldg(a.zeros + base + gi)) << (8 * (gi & 3));
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

// Store NC consecutive 32-bit TMEM columns of the warp's 32 lanes.
template <int NC>
__device__ __forceinline__ void tmem_st_cols(uint32_t taddr, const uint32_t (&v)[NC]);
template <>
__device__ __forceinline__ void tmem_st_cols<8>(uint32_t taddr, const uint32_t (&v)[8]) {
    tmem_st8(taddr, v);
}
template <>
__device__ __forceinline__ void tmem_st_cols<16>(uint32_t taddr, const uint32_t (&v)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16};" ::"r"(taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
template <>
__device__ __forceinline__ void tmem_st_cols<32>(uint32_t taddr, const uint32_t (&v)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(
            taddr),
        "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
        "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]),
        "r"(v[16]), "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]),
        "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]),
        "r"(v[30]), "r"(v[31])
        : "memory");
}

__device__ __forceinline__ void record_error_tc(int* err, volatile int* abort_flag) {
    *abort_flag = 1;
    atomicExch(err, 1);
}

// Warp-uniform bounded wait: true only if every lane saw the phase complete.
__device__ __forceinline__ bool wait_all(uint64_t* bar, uint32_t parity, volatile int* abort_flag) {
    return __all_sync(kFull, mbar_wait(bar, parity, abort_flag));
}

// Which packed words of its row a consumer thread reads for one group: the
// bf16 pairs [p0, p0 + kPairsW) of the stage row (pair p = codes 2p, 2p + 1)
// live in words [p0 / kPpw, (p0 + kPairsW - 1) / kPpw].  They are fetched as
// one 8-byte load when they sit in one aligned word pair, else as whole
// 16-byte chunks.
template <int BITS, int G, int H, int GI>
struct WordPlan {
    using L = Lay<BITS, G>;
    static constexpr int kP0 = GI * (G / 2) + H * L::kPairsW;
    static constexpr int kWLo = kP0 / L::kPpw;
    static constexpr int kWHi = (kP0 + L::kPairsW - 1) / L::kPpw;
    static constexpr bool kPair = (kWLo / 2) == (kWHi / 2);
    static constexpr int kBase = kPair ? (kWLo / 2) * 2 : (kWLo / 4) * 4;  // first word loaded
    static constexpr int kChunks = kPair ? 0 : kWHi / 4 - kWLo / 4 + 1;
    static constexpr int kNW = kPair ? 2 : 4 * kChunks;                     // words loaded
};

// Calls f(std::integral_constant<int, I>) for I = B .. E - 1.
template <int B, int E, class F>
__device__ __forceinline__ void static_for(F&& f) {
    if constexpr (B < E) {
        f(std::integral_constant<int, B>{});
        static_for<B + 1, E>(f);
    }
}

// Unpack group GI's K part H for one row and store it as columns
// [H kPairsW, (H + 1) kPairsW) of the group's A tile, with H known at compile
// time (3-bit words do not line up with K steps, so each part has its own
// word pattern).
//   row_sw: shared address of the row inside the stage, with the row's
//           swizzle pattern (row % 8) << 4 already XOR-ed in;
//   tA:     TMEM address of the group's A tile in the warp's lane quarter.
template <int BITS, int G, int NC, int H, int GI>
__device__ __forceinline__ void write_group(uint32_t row_sw, uint32_t tA,
                                            const RowMeta<Lay<BITS, G>::kGPS>& m) {
    using L = Lay<BITS, G, NC>;
    using P = WordPlan<BITS, G, H, GI>;
    uint32_t w[P::kNW];
    if constexpr (P::kPair) {
        constexpr int c = P::kBase / 4;  // 16-byte chunk of the stage row
        constexpr uint32_t box = static_cast<uint32_t>(c / 8) * L::kBoxBytes;
        const uint2 v = lds64(((row_sw + box) ^ static_cast<uint32_t>((c % 8) << 4)) +
                              static_cast<uint32_t>((P::kBase % 4) * 4));
        w[0] = v.x;
        w[1] = v.y;
    } else {
#pragma unroll
        for (int j = 0; j < P::kChunks; ++j) {
            const int c = P::kBase / 4 + j;
            const uint32_t box = static_cast<uint32_t>(c / 8) * L::kBoxBytes;
            const uint4 v = lds128((row_sw + box) ^ static_cast<uint32_t>((c % 8) << 4));
            w[4 * j] = v.x;
            w[4 * j + 1] = v.y;
            w[4 * j + 2] = v.z;
            w[4 * j + 3] = v.w;
        }
    }
    constexpr uint32_t kMask = ((1u << BITS) - 1u) * 0x00010001u;
    const uint32_t zz = L::kZtc ? 0u : m.zero_point(GI);
    // stores of kStoreCols columns, each issued as soon as its pairs are ready
    constexpr int kStW = L::kPairsW < kStoreCols ? L::kPairsW : kStoreCols;
#pragma unroll
    for (int c = 0; c < L::kPairsW / kStW; ++c) {
        uint32_t p[kStW];
#pragma unroll
        for (int j = 0; j < kStW; ++j) {
            const int pp = P::kP0 + c * kStW + j;  // pair index in the stage row
            const int wi = pp / L::kPpw - P::kBase;
            const int sh = (pp % L::kPpw) * BITS;
            const uint32_t v = sh ? (w[wi] >> sh) : w[wi];
            p[j] = lop3_and_or(v, kMask, 0x43004300u);  // (128 + q_2pp, 128 + q_2pp+1)
            if constexpr (!L::kZtc) p[j] = bf16x2_sub(p[j], zz);
        }
        tmem_st_cols<kStW>(tA + H * L::kPairsW + c * kStW, p);
    }
}

// The same for 2- and 4-bit codes with the K part h known only at run time:
// each part covers a whole number of words, so all parts share one word
// pattern and one copy of the code.
template <int BITS, int G, int NC, int GI>
__device__ __forceinline__ void write_group_rt(uint32_t row_sw, uint32_t tA,
                                               const RowMeta<Lay<BITS, G>::kGPS>& m, int h) {
    using L = Lay<BITS, G, NC>;
    constexpr int kWG = (G / 2) / L::kPpw;     // words per group
    constexpr int kWW = L::kPairsW / L::kPpw;  // words per K part
    static_assert(kWG * L::kPpw == G / 2 && kWW * L::kPpw == L::kPairsW, "whole words per part");
    const int w0 = GI * kWG + h * kWW;         // first word of the part (a multiple of kWW)
    uint32_t w[kWW];
    if constexpr (kWW >= 4) {
#pragma unroll
        for (int j = 0; j < kWW / 4; ++j) {
            const uint32_t c = static_cast<uint32_t>(w0 >> 2) + j;  // 16-byte chunk of the stage row
            const uint4 v = lds128((row_sw + (c >> 3) * L::kBoxBytes) ^ ((c & 7u) << 4));
            w[4 * j] = v.x;
            w[4 * j + 1] = v.y;
            w[4 * j + 2] = v.z;
            w[4 * j + 3] = v.w;
        }
    } else {
        const uint32_t c = static_cast<uint32_t>(w0 >> 2);
        const uint32_t addr = ((row_sw + (c >> 3) * L::kBoxBytes) ^ ((c & 7u) << 4)) +
                              static_cast<uint32_t>(w0 & 3) * 4u;
        if constexpr (kWW == 2) {
            const uint2 v = lds64(addr);
            w[0] = v.x;
            w[kWW > 1 ? 1 : 0] = v.y;
        } else {
            w[0] = lds32(addr);
        }
    }
    constexpr uint32_t kMask = ((1u << BITS) - 1u) * 0x00010001u;
    const uint32_t zz = L::kZtc ? 0u : m.zero_point(GI);
    // stores of kStoreCols columns, each issued as soon as its pairs are ready
    constexpr int kStW = L::kPairsW < kStoreCols ? L::kPairsW : kStoreCols;
#pragma unroll
    for (int c = 0; c < L::kPairsW / kStW; ++c) {
        uint32_t p[kStW];
#pragma unroll
        for (int j = 0; j < kStW; ++j) {
            const int i = c * kStW + j;
            const int sh = (i % L::kPpw) * BITS;
            const uint32_t v = sh ? (w[i / L::kPpw] >> sh) : w[i / L::kPpw];
            p[j] = lop3_and_or(v, kMask, 0x43004300u);  // (128 + q_2i, 128 + q_2i+1)
            if constexpr (!L::kZtc) p[j] = bf16x2_sub(p[j], zz);
        }
        tmem_st_cols<kStW>(tA + h * L::kPairsW + c * kStW, p);
    }
}

// Projection data as the warps see it.
struct ProjView {
    const CUtensorMap* tmW;
    const CUtensorMap* tmX;
    const uint16_t* scales;
    const uint8_t* zeros;
    float* y;
    long long uoff;  // first global unit
    int M, N, ng, T, I, toff, after, phase, epi;
    bool meta_vec, x3d;
};

// Kernel-wide context: one projection from the launch parameters, or a table
// of projections in device memory (fused step).
struct Ctx {
    const ProjDev* proj;    // nullptr: the single projection `one`, one phase
    const PhaseDev* phase;
    int nproj, nphase;
    ProjView one;
    float* partials;
    int* counters;
    int* done;
    int* err;
    long long U;
    int P;
    bool pdl;  // X and every write wait for the previous kernel on the stream

    __device__ __forceinline__ ProjView view(int p) const {
        if (proj == nullptr) return one;
        const ProjDev& d = proj[p];
        ProjView v;
        v.tmW = &d.tmW;
        v.tmX = &d.tmX;
        v.scales = d.scales;
        v.zeros = d.zeros;
        v.y = d.y;
        v.uoff = d.uoff;
        v.M = d.M;
        v.N = d.N;
        v.ng = d.ng;
        v.T = d.T;
        v.I = d.I;
        v.toff = d.toff;
        v.after = d.after;
        v.phase = d.phase;
        v.epi = d.epi;
        v.meta_vec = d.meta_vec != 0;
        v.x3d = d.x3d != 0;
        return v;
    }
    // Projection holding global unit u (binary search over the unit offsets).
    __device__ __forceinline__ int proj_of_unit(long long u) const {
        if (proj == nullptr) return 0;
        int lo = 0, hi = nproj - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (proj[mid].uoff <= u)
                lo = mid;
            else
                hi = mid - 1;
        }
        return lo;
    }
    // Phase s covers global units [phase_uoff(s), phase_uoff(s) + phase_units(s)).
    __device__ __forceinline__ long long phase_uoff(int s) const {
        return phase == nullptr ? 0 : phase[s].uoff;
    }
    __device__ __forceinline__ long long phase_units(int s) const {
        return phase == nullptr ? U : phase[s].U;
    }
    // CTAs sharing phase s: all of them, or one per unit when the phase is
    // smaller than the grid (so that every share is contiguous and non-empty).
    __device__ __forceinline__ int phase_ctas(int s) const {
        const long long Us = phase_units(s);
        return Us < P ? static_cast<int>(Us) : P;
    }
    // floor(n / d) for non-negative n and positive d; 32-bit when it fits
    // (64-bit integer division is a long software sequence).
    __device__ __forceinline__ static long long div_fast(unsigned long long n, unsigned long long d) {
        if (n <= 0xffffffffull && d <= 0xffffffffull)
            return static_cast<long long>(static_cast<uint32_t>(n) / static_cast<uint32_t>(d));
        return static_cast<long long>(n / d);
    }
    // CTA b's share of phase s: [sub_lo(s, b), sub_lo(s, b + 1)); empty for b >= phase_ctas(s).
    __device__ __forceinline__ long long sub_lo(int s, int b) const {
        const int Ps = phase_ctas(s);
        const unsigned long long Us = static_cast<unsigned long long>(phase_units(s));
        return phase_uoff(s) + div_fast(Us * static_cast<unsigned>(b < Ps ? b : Ps),
                                        static_cast<unsigned>(Ps));
    }
    // CTA whose share of phase s holds global unit u: ceil((x + 1) Ps / Us) - 1
    // for the unit's index x within the phase.
    __device__ __forceinline__ int owner(long long u, int s) const {
        const unsigned long long Us = static_cast<unsigned long long>(phase_units(s));
        const unsigned long long x = static_cast<unsigned long long>(u - phase_uoff(s));
        return static_cast<int>(div_fast((x + 1) * static_cast<unsigned>(phase_ctas(s)) + Us - 1, Us)) - 1;
    }
};

// A warp's position in its CTA's units: phase s, projection p, tile t,
// k-stage i, global unit u (the CTA's share of phase s ends at u_end).
struct Cursor {
    int s, p, t, i;
    long long u, u_end;
    ProjView v;
    // first non-empty share at or after phase s0
    __device__ __forceinline__ void seek(const Ctx& c, int s0) {
        for (s = s0; s < c.nphase; ++s) {
            u = c.sub_lo(s, blockIdx.x);
            u_end = c.sub_lo(s, blockIdx.x + 1);
            if (u < u_end) break;
        }
        if (s >= c.nphase) return;
        p = c.proj_of_unit(u);
        v = c.view(p);
        const long long l = u - v.uoff;
        t = static_cast<int>(l / v.I);
        i = static_cast<int>(l - static_cast<long long>(t) * v.I);
    }
    __device__ __forceinline__ void init(const Ctx& c) { seek(c, 0); }
    __device__ __forceinline__ bool last_of_share() const { return u + 1 == u_end; }
    __device__ __forceinline__ void next(const Ctx& c) {
        if (++u == u_end) {
            seek(c, s + 1);
            return;
        }
        if (++i == v.I) {
            i = 0;
            if (++t == v.T) {
                t = 0;
                ++p;
                v = c.view(p);
            }
        }
    }
};

// Epilogue kinds a kernel is built for: fp32 Y only, the fused gate/up
// activation only, or either (chosen per projection at run time).  Single
// GEMMs take the first two; a fused step always takes the third, which
// measured no slower than the Y-only build on steps without an activation.
constexpr int kEpiY = 0, kEpiAct = 1, kEpiAny = 2;

// Final values of tile row n (this lane) for all rows of X: fp32 Y, or, for
// the fused gate/up projection, the activation: rows 2j and 2j + 1 (gate and
// up of feature j) are neighbouring lanes, which store bf16(silu(gate) * up)
// at column j of the bf16 [M][N/2] output.
template <int EPI, int NC>
__device__ __forceinline__ void store_final(const ProjView& v, int n, const float (&val)[NC],
                                            int lane) {
    if (EPI == kEpiY || (EPI == kEpiAny && v.epi == WQ_EPI_NONE)) {
        if (n < v.N)
#pragma unroll
            for (int j = 0; j < NC; ++j)
                if (j < v.M) v.y[static_cast<size_t>(j) * v.N + n] = val[j];
        return;
    }
    if constexpr (EPI != kEpiY) {
        // Lane pair (2i, 2i+1) holds rows 2i (gate) and 2i+1 (up) of activation
        // column i.  Both lanes swap their values and split the batch rows: the
        // even lane takes rows 0, 2, 4, ..., the odd lane rows 1, 3, 5, ...  The
        // fast exponential and division keep this path short; their relative
        // error (a few fp32 ulps) is far below the bf16 rounding step.  Where
        // 1 + exp(-g) exceeds 2^126 (gate below about -87.3) the quotient
        // comes out as zero instead of a value under 1e-36 times abs(up).
        __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(v.y);
        const int nf = v.N >> 1, f = n >> 1;
        const bool odd = (lane & 1) != 0;
        const bool live = n < v.N;
#pragma unroll
        for (int jj = 0; jj < NC / 2; ++jj) {
            const float a = val[2 * jj], b = val[2 * jj + 1];
            const float oa = __shfl_xor_sync(kFull, a, 1), ob = __shfl_xor_sync(kFull, b, 1);
            const float g = odd ? ob : a, u = odd ? b : oa;
            const int j = 2 * jj + (odd ? 1 : 0);
            if (live && j < v.M)
                out[static_cast<size_t>(j) * nf + f] =
                    __float2bfloat16_rn(__fdividef(g, 1.0f + __expf(-g)) * u);
        }
    }
}

// End of a tile segment for one epilogue warp (rows 32 q + lane, all
// accumulator columns): store Y, or publish the partial sums and let the
// warp of the last CTA to finish the tile add all partials in k order.  Each
// (tile, lane quarter) pair has its own arrival counter, so warps never wait
// for one another.  In a fused step the warp that writes the final Y rows
// then counts them done for the projection's phase.
//   likely_last: the segment holds the tile's first units and ends the CTA's
//   share; the tile's other contributors took its later units at the start
//   of their shares, so they have usually all arrived already.  Then the
//   warp checks the counter first and, if they have, sums at once without
//   publishing its own partial (two round trips fewer at the end of a share).
//   PAIR: two contributors' partials in flight at a time in the 16-row sum
//   (measured faster in the single-projection and per-phase builds, slower in
//   the fused build, which sits at the register ceiling).
template <int EPI, int NC, bool PAIR>
__device__ __forceinline__ void finish_rows(const Ctx& c, const ProjView& v,
                                            float (&acc)[NC], int t, bool whole,
                                            bool likely_last, int r, int q, int lane) {
    const int n = t * kBN + r;
    const int gt = v.toff + t;
    // only phases that a later phase of the launch waits for are counted
    auto count_done = [&]() {
        if (c.done != nullptr && v.phase + 1 < c.nphase) {
            __syncwarp();
            if (lane == 0) red_add_release_gpu(c.done + v.phase, 1);
        }
    };
    if (whole) {
        store_final<EPI, NC>(v, n, acc, lane);
        count_done();
        return;
    }
    // Slot 0 holds the partial of the tile a CTA's share of the phase starts in,
    // slot 1 that of the tile it ends in (a share that started before this
    // tile's first unit ends in it).
    const long long tu0 = v.uoff + static_cast<long long>(t) * v.I;
    const int b_first = c.owner(tu0, v.phase);
    const int b_last = c.owner(tu0 + v.I - 1, v.phase);
    const int me = static_cast<int>(blockIdx.x);
    int* ctr = c.counters + static_cast<size_t>(gt) * kCountersPerTile + q;
    // contributors after the first start their share inside this tile (slot 0)
    const int first_role = c.sub_lo(v.phase, b_first) < tu0 ? 1 : 0;
    int last = 0;
    if (likely_last) {
        int cnt = 0;
        if (lane == 0) cnt = ld_acquire_gpu(ctr);
        last = __shfl_sync(kFull, cnt, 0) == b_last - b_first ? 1 : 0;  // all others arrived
    }
    bool published = false;
    if (!last) {
        published = true;
        const int own_role = c.sub_lo(v.phase, blockIdx.x) < tu0 ? 1 : 0;
        float* mine = c.partials + static_cast<size_t>(2 * blockIdx.x + own_role) * (kMaxCols * kBN);
#pragma unroll
        for (int j = 0; j < NC; ++j)
            if (j < v.M) __stcg(mine + j * kBN + r, acc[j]);
        // The warp barrier orders every lane's partial before lane 0's release
        // (acq_rel) increment; the reading warp's lane 0 acquires it and the
        // next warp barrier orders the other lanes' reads after that acquire.
        __syncwarp();
        if (lane == 0) last = (atomic_add_acq_rel_gpu(ctr, 1) == b_last - b_first) ? 1 : 0;
        if (!__shfl_sync(kFull, last, 0)) return;
    }
    __syncwarp();  // the other lanes' reads follow lane 0's acquire
    if constexpr (NC == 16) {
        // all contributors in k order (this warp's own sums in place of its
        // partial), one or (PAIR) two contributors' partials in flight at a time
        float tot[NC];
#pragma unroll
        for (int j = 0; j < NC; ++j) tot[j] = 0.f;
        if constexpr (PAIR) {
            for (int b = b_first; b <= b_last; b += 2) {
                const bool two = b + 1 <= b_last;
                const bool own0 = b == me, own1 = two && b + 1 == me;
                // contributors after the first publish into their slot 0
                const float* s0 = c.partials +
                                  static_cast<size_t>(2 * b + (b == b_first ? first_role : 0)) *
                                      (kMaxCols * kBN) +
                                  r;
                const float* s1 =
                    c.partials + static_cast<size_t>(2 * (b + 1)) * (kMaxCols * kBN) + r;
                float p0[NC], p1[NC];
#pragma unroll
                for (int j = 0; j < NC; ++j) {
                    p0[j] = (!own0 && j < v.M) ? __ldcg(s0 + j * kBN) : 0.f;
                    p1[j] = (two && !own1 && j < v.M) ? __ldcg(s1 + j * kBN) : 0.f;
                }
#pragma unroll
                for (int j = 0; j < NC; ++j) tot[j] += own0 ? acc[j] : p0[j];
                if (two) {
#pragma unroll
                    for (int j = 0; j < NC; ++j) tot[j] += own1 ? acc[j] : p1[j];
                }
            }
        } else {
            for (int b = b_first; b <= b_last; ++b) {
                if (b == me) {
#pragma unroll
                    for (int j = 0; j < NC; ++j) tot[j] += acc[j];
                } else {
                    const float* src = c.partials +
                                       static_cast<size_t>(2 * b + (b == b_first ? first_role : 0)) *
                                           (kMaxCols * kBN) +
                                       r;
                    float part[NC];
#pragma unroll
                    for (int j = 0; j < NC; ++j) part[j] = j < v.M ? __ldcg(src + j * kBN) : 0.f;
#pragma unroll
                    for (int j = 0; j < NC; ++j) tot[j] += part[j];
                }
            }
        }
        store_final<EPI, NC>(v, n, tot, lane);
    } else {
        // 32 rows: the same k-ordered sum in acc's registers, so that all 32
        // rows of a contributor's partial load at once.  A warp that found
        // every other contributor arrived holds the tile's first units and
        // starts the sum with its own acc; a warp that published reads its
        // own partial back with the others'.
        int b = b_first;
        if (published) {
#pragma unroll
            for (int j = 0; j < NC; ++j) acc[j] = 0.f;
        } else {
#pragma unroll
            for (int j = 0; j < NC; ++j) acc[j] = 0.f + acc[j];
            ++b;
        }
        for (; b <= b_last; ++b) {
            const float* src = c.partials +
                               static_cast<size_t>(2 * b + (b == b_first ? first_role : 0)) *
                                   (kMaxCols * kBN) +
                               r;
            float part[NC];
#pragma unroll
            for (int j = 0; j < NC; ++j) part[j] = j < v.M ? __ldcg(src + j * kBN) : 0.f;
#pragma unroll
            for (int j = 0; j < NC; ++j) acc[j] += part[j];
        }
        store_final<EPI, NC>(v, n, acc, lane);
    }
    if (lane == 0) *ctr = 0;
    count_done();
}

// End of a tile segment in a cluster build: the launch gives each tile k
// CTAs, ranks 0 .. k-1 of one cluster in k order, one segment each.  Ranks
// 1 .. k-1 store their sums into rank 0's shared memory with asynchronous
// stores that complete on rank 0's `fix` barrier, and are done; rank 0 waits
// (bounded) for them and adds them to its own in rank order, i.e. in k order.
// No global partials, no counters, no L2 round trips.
//   fix_smem, fix_bar: this CTA's buffer and barrier (rank 0's are the ones used)
template <int EPI, int NC>
__device__ __forceinline__ void finish_rows_cluster(const Ctx& c, const ProjView& v,
                                                    const float (&acc)[NC], int t, bool whole,
                                                    int r, int lane, uint32_t fix_smem,
                                                    uint64_t* fix_bar, uint32_t rank,
                                                    uint32_t k, volatile int* abort_flag) {
    static_assert(NC % 4 == 0, "whole float4 pieces");
    const int n = t * kBN + r;
    if (whole) {
        store_final<EPI, NC>(v, n, acc, lane);
        return;
    }
    if (rank != 0) {
        const uint32_t dst =
            map_to_rank(fix_smem + ((rank - 1) * kBN + static_cast<uint32_t>(r)) * NC * 4u, 0u);
        const uint32_t bar = map_to_rank(smem_addr(fix_bar), 0u);
#pragma unroll
        for (int j = 0; j < NC; j += 4)
            st_async_v4(dst + 4u * j, acc[j], acc[j + 1], acc[j + 2], acc[j + 3], bar);
        return;
    }
    if (!__all_sync(kFull, mbar_wait_cluster(fix_bar, 0u, abort_flag))) {
        if (lane == 0) record_error_tc(c.err, abort_flag);
        return;
    }
    float tot[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) tot[j] = acc[j];
    for (uint32_t b = 1; b < k; ++b) {
        const uint32_t src = fix_smem + ((b - 1) * kBN + static_cast<uint32_t>(r)) * NC * 4u;
#pragma unroll
        for (int j = 0; j < NC; j += 4) {
            const uint4 p = lds128(src + 4u * j);
            tot[j] += __uint_as_float(p.x);
            tot[j + 1] += __uint_as_float(p.y);
            tot[j + 2] += __uint_as_float(p.z);
            tot[j + 3] += __uint_as_float(p.w);
        }
    }
    store_final<EPI, NC>(v, n, tot, lane);
}

// Shared-memory barriers of one CTA.
template <int S, int NA, int ND>
struct Bars {
    uint64_t full[S];    // stage's packed words and zero points landed (TMA bytes + producer lanes)
    uint64_t xfull[S];   // stage's X slice landed (TMA bytes)
    uint64_t empty[S];   // stage consumed: unpack warps + one MMA commit
    uint64_t filled[NA]; // A slot written (unpack warps)
    uint64_t afree[NA];  // A slot's MMAs complete (tcgen05.commit)
    uint64_t dfull[ND];  // accumulator slot's MMAs complete (tcgen05.commit)
    uint64_t dfree[ND];  // accumulator slot read back (epilogue warps)
    uint64_t drain;      // every MMA complete
    uint64_t fix;        // cluster builds: the other contributors' partials landed
    uint32_t tmem_base;
    int abort_flag;
    int n_units;         // units of this CTA (all its phase shares)
};

// Ring position: slot index and phase parity of a barrier ring of N entries.
template <int N>
struct Ring {
    uint32_t slot = 0, phase = 0;
    __device__ __forceinline__ void next() {
        if (++slot == N) {
            slot = 0;
            phase ^= 1u;
        }
    }
};

// Unpack warp: turns the stage's packed words into A tiles, batch by batch.
// HT is the warp's K part when fixed at compile time, -1 when read at run time.
template <int BITS, int G, int NC, int HT, class B>
__device__ __forceinline__ void unpack_warp(const Ctx& c, uint32_t smem_u32, B& bars,
                                            uint32_t tmem, volatile int* abort_flag, int warp,
                                            int lane, int n_units) {
    using L = Lay<BITS, G, NC>;
    using RM = RowMeta<L::kGPS>;
    const int h = HT >= 0 ? HT : (warp >> 2);
    const int q = warp & 3;
    const int r = 32 * q + lane;                                       // tile row == TMEM lane
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);  // lane quarter
    const uint32_t row_off = static_cast<uint32_t>(r * 128) | (static_cast<uint32_t>(lane & 7) << 4);
    bool dead = false;  // after a failed wait: no more shared or tensor memory work

    auto fail = [&]() {
        record_error_tc(c.err, abort_flag);
        dead = true;
    };

    Ring<L::kStages> st;
    Ring<L::kNA> as;
    RM cur;
    for (int k = 0; k < n_units; ++k) {
        if (!dead && !wait_all(&bars.full[st.slot], st.phase, abort_flag)) fail();
        // the unit's zero points, staged with its words
        {
            const uint32_t zs = smem_u32 + st.slot * L::kStageBytes + L::kZOff + r * L::kZRow;
            if constexpr (RM::kZ == 1) {
                cur.z[0] = lds32(zs);
            } else if constexpr (RM::kZ == 2) {
                const uint2 v = lds64(zs);
                cur.z[0] = v.x;
                cur.z[RM::kZ > 1 ? 1 : 0] = v.y;
            } else {
                static_assert(RM::kZ <= 4, "zero points per row");
                const uint4 v = lds128(zs);
                cur.z[0] = v.x;
                if constexpr (RM::kZ > 1) cur.z[1] = v.y;
                if constexpr (RM::kZ > 2) cur.z[2] = v.z;
                if constexpr (RM::kZ > 3) cur.z[3] = v.w;
            }
        }
        // Both A slots of this stage must have left the tensor core: the MMAs
        // complete in order, so waiting for the later slot's previous batch
        // covers the earlier one.  (With a single A slot each batch waits for
        // the one before it instead.)
        if constexpr (L::kNA >= 2) {
            Ring<L::kNA> as1 = as;
            as1.next();
            if (!dead && !wait_all(&bars.afree[as1.slot], as1.phase ^ 1u, abort_flag)) fail();
        }
        const uint32_t row_sw = smem_u32 + st.slot * L::kStageBytes + row_off;
        static_for<0, 2>([&](auto bc) {
            constexpr int BB = decltype(bc)::value;
            constexpr int g_lo = BB == 0 ? 0 : L::kR0;
            constexpr int g_hi = BB == 0 ? L::kR0 : L::kGPS;
            if constexpr (L::kNA == 1)
                if (!dead && !wait_all(&bars.afree[as.slot], as.phase ^ 1u, abort_flag)) fail();
            if (!dead) {
                const uint32_t slot_col = as.slot * (L::kR0 * L::kACols);
                static_for<g_lo, g_hi>([&](auto gc) {
                    constexpr int GI = decltype(gc)::value;
                    const uint32_t tA = tl + L::kColA + slot_col + (GI - g_lo) * L::kACols;
                    if constexpr (HT >= 0)
                        write_group<BITS, G, NC, HT, GI>(row_sw, tA, cur);
                    else
                        write_group_rt<BITS, G, NC, GI>(row_sw, tA, cur, h);
                    // the group's zero-point tile, from one of the lane quarter's warps
                    if constexpr (L::kZtc)
                        if (GI % L::kSplit == h)
                            tmem_st8_same(tl + L::kColZ + (as.slot * L::kR0 + (GI - g_lo)) * 8,
                                          cur.neg_zero_point(GI));
                });
                tmem_wait_st();
                tc_fence_before();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars.filled[as.slot]);
            as.next();
        });
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.empty[st.slot]);  // the stage's words are no longer needed
        st.next();
    }
}

// Epilogue warp (lane quarter q).  Per unit it reads the unit's two batches
// of accumulators back (adding scale * D to the row's NC fp32 sums) and ends
// tile segments.
template <int BITS, int G, int NC, int EPI, bool PAIR, bool CLU, class B>
__device__ __forceinline__ void epilogue_warp(const Ctx& c, B& bars, uint32_t tmem,
                                              volatile int* abort_flag, int q, int lane,
                                              int n_units, uint32_t fix_smem, uint32_t crank,
                                              uint32_t csize) {
    using L = Lay<BITS, G, NC>;
    using RM = RowMeta<L::kGPS>;
    const int r = 32 * q + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * q) << 16);
    bool dead = false;
    float acc[NC];
#pragma unroll
    for (int j = 0; j < NC; ++j) acc[j] = 0.f;
    auto fail = [&]() {
        record_error_tc(c.err, abort_flag);
        dead = true;
    };

    Cursor fc;  // unit whose scales and zero points are fetched next
    fc.init(c);
    Cursor cc = fc;  // unit being read back
    auto fetch = [&](RM& m) {
        m.load(fc.v, fc.t * kBN + r, static_cast<long long>(fc.i) * L::kGPS);
        fc.next(c);
    };
    Ring<L::kND> ds;
    // Accumulators of one batch (scales from m) into acc.
    auto read_d = [&](auto bc, const RM& m) {
        constexpr int BB = decltype(bc)::value;
        constexpr int g_lo = BB == 0 ? 0 : L::kR0;
        constexpr int g_hi = BB == 0 ? L::kR0 : L::kGPS;
        if (!dead && !wait_all(&bars.dfull[ds.slot], ds.phase, abort_flag)) fail();
        if (!dead) {
            tc_fence_after();
            // 32 accumulator columns in flight at most (two groups of 16); a
            // 32-row build reads each group in two halves of 16 columns, which
            // measured faster than one 32-column load (fewer live registers)
            constexpr int kPG = NC == 16 ? 2 : 1;
            static_for<0, (g_hi - g_lo + kPG - 1) / kPG>([&](auto pc) {
                constexpr int G0 = g_lo + kPG * decltype(pc)::value;
                constexpr int NG = (G0 + 1 < g_hi) ? kPG : 1;
                if constexpr (NC == 16) {
                    uint32_t v[NG][NC];
                    static_for<0, NG>([&](auto gc) {
                        constexpr int J = decltype(gc)::value;
                        const uint32_t ta = tl + L::kColD + (ds.slot * L::kR0 + (G0 + J - g_lo)) * NC;
                        tmem_ld16(ta, v[J]);
                    });
                    tmem_wait_ld();
                    static_for<0, NG>([&](auto gc) {
                        constexpr int J = decltype(gc)::value;
                        const float sc = m.scale(G0 + J);
#pragma unroll
                        for (int j = 0; j < NC; ++j) acc[j] = fmaf(sc, __uint_as_float(v[J][j]), acc[j]);
                    });
                } else {
                    const uint32_t ta = tl + L::kColD + (ds.slot * L::kR0 + (G0 - g_lo)) * NC;
                    const float sc = m.scale(G0);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {
                        uint32_t v16[16];
                        tmem_ld16(ta + 16 * hh, v16);
                        tmem_wait_ld();
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            acc[16 * hh + j] = fmaf(sc, __uint_as_float(v16[j]), acc[16 * hh + j]);
                    }
                }
            });
            tc_fence_before();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&bars.dfree[ds.slot]);
        ds.next();
    };

    constexpr std::integral_constant<int, 0> kB0{};
    constexpr std::integral_constant<int, 1> kB1{};
    RM cur, nxt;
    if (n_units > 0) fetch(cur);
    bool seg_from_start = cc.i == 0;  // the open segment began at its tile's first k-stage
    for (int k = 0; k < n_units; ++k) {
        if (k + 1 < n_units) fetch(nxt);
        read_d(kB0, cur);
        read_d(kB1, cur);
        // a tile segment ends with the tile or with the CTA's share of the phase
        const bool tile_end = cc.i == cc.v.I - 1;
        const bool end = tile_end || cc.last_of_share();
        if (end) {
            if (!dead) {
                if constexpr (CLU)
                    finish_rows_cluster<EPI, NC>(c, cc.v, acc, cc.t, seg_from_start && tile_end,
                                                 r, lane, fix_smem, &bars.fix, crank, csize,
                                                 abort_flag);
                else
                    finish_rows<EPI, NC, PAIR>(c, cc.v, acc, cc.t, seg_from_start && tile_end,
                                               seg_from_start && !tile_end, r, q, lane);
            }
#pragma unroll
            for (int j = 0; j < NC; ++j) acc[j] = 0.f;
        }
        cc.next(c);
        if (end) seg_from_start = cc.i == 0;
        cur = nxt;
    }
    tc_fence_before();
}

// Producer's dependency check (fused step): true once phase `upto` of the
// launch is complete (one counter per phase; a phase completes only after
// every earlier one, whose results its X waited for); `verified` caches the
// latest phase known complete.
__device__ __forceinline__ bool deps_ready(const Ctx& c, int upto, int& verified) {
    if (verified >= upto) return true;
    if (ld_acquire_gpu(c.done + upto) < __ldg(&c.phase[upto].need)) return false;
    verified = upto;
    // the TMA reads that follow are async-proxy accesses of data the acquire made visible
    fence_proxy_async();
    return true;
}

// The same, waiting (bounded) until it holds.  Each poll is an L2 round
// trip, so the loop needs no sleep.
__device__ __forceinline__ bool wait_deps(const Ctx& c, int upto, int& verified,
                                          volatile int* abort_flag) {
    if (deps_ready(c, upto, verified)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t n = 1;; ++n) {
        if (deps_ready(c, upto, verified)) return true;
        if (*abort_flag) return false;
        if ((n & 15u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) return false;
    }
}

// HOLD: the build can be launched as a programmatic dependent (single
// projections always; a fused step only in its per-phase launches, a separate
// build because the fused kernel's speed measured sensitive to any code added).
// CLU: a per-phase build launched in clusters of k CTAs per tile, whose
// split-K sums travel through rank 0's shared memory (finish_rows_cluster).
template <int BITS, int G, int NC, bool MULTI, int EPI, bool HOLD = !MULTI, bool CLU = false>
__global__ void __launch_bounds__(Lay<BITS, G, NC>::kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const GemmArgs a, const StepArgs sa) {
    using L = Lay<BITS, G, NC>;
    constexpr int S = L::kStages;
    using BarsT = Bars<S, L::kNA, L::kND>;
    static_assert(sizeof(BarsT) <= 512, "barrier block");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
    const uint32_t smem_u32 = smem_addr(smem);
    BarsT& bars = *reinterpret_cast<BarsT*>(smem + L::kBarOffset);
    volatile int* abort_flag = &bars.abort_flag;

    Ctx c;
    if constexpr (MULTI) {
        c.proj = sa.proj;
        c.phase = sa.phase;
        c.nproj = sa.nproj;
        c.nphase = sa.nphase;
        c.partials = sa.partials;
        c.counters = sa.counters;
        c.done = sa.done;
        c.err = sa.err;
        c.U = sa.U;
        c.P = sa.P;
        c.pdl = sa.pdl != 0;
    } else {
        c.proj = nullptr;
        c.phase = nullptr;
        c.nproj = 1;
        c.nphase = 1;
        c.one.tmW = &tmW;
        c.one.tmX = &tmX;
        c.one.scales = a.scales;
        c.one.zeros = a.zeros;
        c.one.y = a.y;
        c.one.uoff = 0;
        c.one.M = a.M;
        c.one.N = a.N;
        c.one.ng = a.ng;
        c.one.T = a.T;
        c.one.I = a.I;
        c.one.toff = 0;
        c.one.after = -1;
        c.one.phase = 0;
        c.one.epi = a.epi;
        c.one.meta_vec = a.meta_vec != 0;
        c.one.x3d = a.x3d != 0;
        c.partials = a.partials;
        c.counters = a.counters;
        c.done = nullptr;
        c.err = a.err;
        c.U = a.U;
        c.P = a.P;
        c.pdl = a.pdl != 0;
    }

    // warp index through a shuffle so that the compiler treats it as uniform
    const int warp = __shfl_sync(kFull, static_cast<int>(threadIdx.x >> 5), 0);
    const int lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&bars.full[s], 1 + 32);  // TMA (expect_tx) + the producer warp's zero points
            mbar_init(&bars.xfull[s], 1);
            mbar_init(&bars.empty[s], L::kUW + 1);
        }
        for (int s = 0; s < L::kNA; ++s) {
            mbar_init(&bars.filled[s], L::kUW);
            mbar_init(&bars.afree[s], 1);
        }
        for (int s = 0; s < L::kND; ++s) {
            mbar_init(&bars.dfull[s], 1);
            mbar_init(&bars.dfree[s], L::kEW);
        }
        mbar_init(&bars.drain, 1);
        if constexpr (CLU) {
            mbar_init(&bars.fix, 1);
            // rank 0 expects the sums of the other k - 1 ranks
            const uint32_t k = cluster_size();
            if (cluster_rank() == 0 && k > 1)
                mbar_arrive_expect_tx(&bars.fix, (k - 1) * kBN * NC * 4u);
        }
        *abort_flag = 0;
        // a dependent launch may place its CTAs on SMs as this grid's CTAs leave
        griddep_launch_dependents();
        long long n = 0;
        for (int ph = 0; ph < c.nphase; ++ph)
            n += c.sub_lo(ph, blockIdx.x + 1) - c.sub_lo(ph, blockIdx.x);
        bars.n_units = static_cast<int>(n);
        fence_mbar_init();
    }
    if (warp == L::kMmaWarp) {
        tmem_alloc(smem_addr(&bars.tmem_base), kTmemCols);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = bars.tmem_base;
    uint32_t crank = 0, csize = 1;
    if constexpr (CLU) {
        // every CTA's barriers are initialised before any of them stores into another
        cluster_sync();
        crank = cluster_rank();
        csize = cluster_size();
    }

    const int n_units = bars.n_units;
    constexpr uint32_t kTail = 32 * (L::kUW + L::kEW + 1);  // warps that meet before dealloc

    if (warp == L::kProducerWarp) {
        // ------------------------------------------------------------ producer
        // Lane 0 issues the TMA loads (and, in a fused step, holds back the X
        // of a projection whose inputs are not complete yet); every lane then
        // stages the zero points of four of the tile's rows into the stage and
        // arrives on the stage's barrier once they have landed.
        const uint64_t pol_w = policy_evict_first();
        const uint64_t pol_x = policy_evict_last();
        Cursor cu;
        cu.init(c);
        int maps_of = -1;   // projection whose tensor maps were last prefetched
        int verified = -1;  // projections 0..verified of the launch known complete
        constexpr int kQ = 8;
        static_assert(S <= kQ, "pending queue holds a ring's worth of stages");
        uint32_t q_slot[kQ] = {};
        const CUtensorMap* q_map[kQ] = {};
        int q_i[kQ] = {}, q_after[kQ] = {}, q_k[kQ] = {};
        bool q_x3d[kQ] = {};
        int q_head = 0, q_n = 0;
        auto issue_x = [&](uint32_t slot, const CUtensorMap* map, int i, bool x3d) {
            uint8_t* stage = smem + slot * L::kStageBytes;
            uint64_t* xb = &bars.xfull[slot];
            mbar_arrive_expect_tx(xb, L::kXBytes);
            if (x3d) {
                tma_load_3d(stage + L::kWBytes, map, 0, 0, i * L::kXBoxes, xb, pol_x);
            } else {
#pragma unroll
                for (int b = 0; b < L::kXBoxes; ++b)
                    tma_load_2d(stage + L::kWBytes + b * L::kXBoxBytes, map,
                                i * L::kStageValues + b * L::kXBoxValues, 0, xb, pol_x);
            }
        };
        auto pop_x = [&]() {
            if constexpr (MULTI) {
                issue_x(q_slot[q_head], q_map[q_head], q_i[q_head], q_x3d[q_head]);
                q_head = (q_head + 1) % kQ;
                --q_n;
            }
        };
        // A dependent launch streams the packed words and zero points of its
        // first stages at once; their X (and everything after) waits until the
        // previous kernel has completed.  Two stages measured best: a longer
        // hold releases a burst of X loads late.
        constexpr int kHeld = S < 2 ? S : 2;
        const bool hold_x = HOLD && c.pdl;
        const int n_held = hold_x ? (n_units < kHeld ? n_units : kHeld) : 0;
        static_assert(kHeld <= 2, "held stages kept in two named slots");
        const CUtensorMap* h_map0 = nullptr;
        const CUtensorMap* h_map1 = nullptr;
        int h_i0 = 0, h_i1 = 0;
        bool h_x3d0 = false, h_x3d1 = false;
        // X of the first `n` held stages (slots 0 and 1) once the previous
        // kernel has completed
        auto release_held = [&](int n) {
            griddep_wait();
            if (n > 0) issue_x(0u, h_map0, h_i0, h_x3d0);
            if (n > 1) issue_x(1u, h_map1, h_i1, h_x3d1);
        };
        Ring<S> st;
        uint32_t it = 0;
        bool ok = true;
        for (int k = 0; k < n_units; ++k, ++it) {
            if (lane == 0) {
                if (cu.p != maps_of) {
                    prefetch_tensormap(cu.v.tmW);
                    prefetch_tensormap(cu.v.tmX);
                    maps_of = cu.p;
                }
                if (k == 0 || cu.i == 0) {
                    // warm L2 with the tile's scales (the epilogue reads them later)
                    const int r0 = cu.t * kBN, r1 = min(cu.v.N, r0 + kBN);
                    const uintptr_t sb = reinterpret_cast<uintptr_t>(cu.v.scales + static_cast<size_t>(r0) * cu.v.ng);
                    const uintptr_t se = reinterpret_cast<uintptr_t>(cu.v.scales + static_cast<size_t>(r1) * cu.v.ng);
                    const uintptr_t sb16 = (sb + 15) & ~uintptr_t(15), se16 = se & ~uintptr_t(15);
                    if (se16 > sb16)
                        prefetch_l2_bulk(reinterpret_cast<const void*>(sb16), static_cast<uint32_t>(se16 - sb16));
                }
                if constexpr (MULTI) {
                    // a held-back stage occupying the slot needed now cannot drain without its X
                    while (ok && q_n > 0 && q_k[q_head] <= k - S) {
                        if (!wait_deps(c, q_after[q_head], verified, abort_flag)) ok = false;
                        else pop_x();
                    }
                }
                if (ok && !mbar_wait(&bars.empty[st.slot], st.phase ^ 1u, abort_flag)) ok = false;
                if (ok) {
                    uint8_t* stage = smem + st.slot * L::kStageBytes;
                    uint64_t* fb = &bars.full[st.slot];
                    mbar_arrive_expect_tx(fb, L::kWBytes);
#pragma unroll
                    for (int b = 0; b < L::kBoxes; ++b)
                        tma_load_2d(stage + b * L::kBoxBytes, cu.v.tmW,
                                    (cu.i * L::kBoxes + b) * kWordsPerStage, cu.t * kBN, fb, pol_w);
                    if (k < n_held) {
                        if (k == 0) {
                            h_map0 = cu.v.tmX;
                            h_i0 = cu.i;
                            h_x3d0 = cu.v.x3d;
                        } else {
                            h_map1 = cu.v.tmX;
                            h_i1 = cu.i;
                            h_x3d1 = cu.v.x3d;
                        }
                        if (k == n_held - 1) release_held(n_held);
                    } else if (!MULTI || cu.v.after < 0 || (q_n == 0 && deps_ready(c, cu.v.after, verified))) {
                        issue_x(st.slot, cu.v.tmX, cu.i, cu.v.x3d);
                    } else {
                        const int e = (q_head + q_n) % kQ;
                        q_slot[e] = st.slot;
                        q_map[e] = cu.v.tmX;
                        q_i[e] = cu.i;
                        q_x3d[e] = cu.v.x3d;
                        q_after[e] = cu.v.after;
                        q_k[e] = k;
                        ++q_n;
                    }
                    if constexpr (MULTI)
                        while (q_n > 0 && deps_ready(c, q_after[q_head], verified)) pop_x();
                }
            }
            ok = __shfl_sync(kFull, ok ? 1 : 0, 0) != 0;
            if (!ok) {
                if (lane == 0) record_error_tc(c.err, abort_flag);
                break;
            }
            // zero points of rows lane, lane + 32, lane + 64, lane + 96
            {
                const uint32_t zdst = smem_u32 + st.slot * L::kStageBytes + L::kZOff;
                const long long g0 = static_cast<long long>(cu.i) * L::kGPS;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int row = lane + 32 * j;
                    const int n = cu.t * kBN + row;
                    const bool in = n < cu.v.N;
                    const uint32_t dst = zdst + row * L::kZRow;
                    if constexpr (L::kZAsync) {
                        if (cu.v.meta_vec) {
                            const uint8_t* src = cu.v.zeros + (in ? static_cast<size_t>(n) * cu.v.ng + g0 : 0);
                            cp_async_n<L::kZRow>(dst, src, in ? L::kZRow : 0);
                            continue;
                        }
                    }
                    uint32_t zw[L::kZRow / 4];
#pragma unroll
                    for (int w = 0; w < L::kZRow / 4; ++w) zw[w] = 0;
                    if (in) {
                        const uint8_t* src = cu.v.zeros + static_cast<size_t>(n) * cu.v.ng + g0;
                        for (int gi = 0; gi < L::kGPS; ++gi)
                            if (g0 + gi < cu.v.ng)
                                zw[gi / 4] |= static_cast<uint32_t>(__ldg(src + gi)) << (8 * (gi & 3));
                    }
#pragma unroll
                    for (int w = 0; w < L::kZRow / 4; ++w) sts32(dst + 4 * w, zw[w]);
                }
                // one arrival per lane: after its copies land, or (plain stores)
                // a release arrive
                if (L::kZAsync && cu.v.meta_vec)
                    cp_async_arrive(&bars.full[st.slot]);
                else
                    mbar_arrive(&bars.full[st.slot]);
            }
            cu.next(c);
            st.next();
        }
        if (lane == 0) {
            if constexpr (MULTI) {
                while (ok && q_n > 0) {
                    if (!wait_deps(c, q_after[q_head], verified, abort_flag)) {
                        record_error_tc(c.err, abort_flag);
                        ok = false;
                    } else {
                        pop_x();
                    }
                }
                // on failure: issue what was held back (the results are discarded)
                // so that every stage in flight completes before shared memory goes away
                while (q_n > 0) pop_x();
            }
            if (!ok) {
                // stages whose X was still held back get it now (the previous
                // kernel always completes), so that every stage in flight lands
                if (hold_x && static_cast<int>(it) < n_held) release_held(static_cast<int>(it));
                // let copies already in flight land before the CTA's shared memory goes away
                const uint32_t first = it > S ? it - S : 0;
                volatile int never = 0;
                for (uint32_t j = first; j < it; ++j) {
                    mbar_wait(&bars.full[j % S], (j / S) & 1u, &never);
                    mbar_wait(&bars.xfull[j % S], (j / S) & 1u, &never);
                }
            }
        }
        return;
    }

    if (warp == L::kMmaWarp) {
        // --------------------------------------------------------- MMA issuer
        // The whole warp walks the schedule (uniform control flow); one
        // elected lane issues the MMAs and commits.
        bool ok = true;
        Ring<S> st;
        Ring<L::kNA> as;
        Ring<L::kND> ds;
        for (int k = 0; k < n_units && ok; ++k) {
            // the MMAs read only the stage's X (A comes from tensor memory)
            if (!wait_all(&bars.xfull[st.slot], st.phase, abort_flag)) {
                ok = false;
                break;
            }
            const uint64_t desc0 = desc_sw128(smem_u32 + st.slot * L::kStageBytes + L::kWBytes);
            static_for<0, 2>([&](auto bc) {
                constexpr int BB = decltype(bc)::value;
                constexpr int g_lo = BB == 0 ? 0 : L::kR0;
                constexpr int g_hi = BB == 0 ? L::kR0 : L::kGPS;
                if (!ok) return;
                if (!wait_all(&bars.filled[as.slot], as.phase, abort_flag) ||
                    !wait_all(&bars.dfree[ds.slot], ds.phase ^ 1u, abort_flag)) {
                    ok = false;
                    return;
                }
                tc_fence_after();
                if (elect_one()) {
                    static_for<g_lo, g_hi>([&](auto gc) {
                        constexpr int GI = decltype(gc)::value;
                        const uint32_t tA = tmem + L::kColA + (as.slot * L::kR0 + (GI - g_lo)) * L::kACols;
                        const uint32_t tZ = tmem + L::kColZ + (as.slot * L::kR0 + (GI - g_lo)) * 8;
                        const uint32_t tD = tmem + L::kColD + (ds.slot * L::kR0 + (GI - g_lo)) * NC;
#pragma unroll
                        for (int s = 0; s < L::kSteps; ++s) {
                            const int v0 = GI * G + 16 * s;  // first value of this K step in the stage
                            const uint64_t bdesc =
                                desc0 + static_cast<uint64_t>(((v0 / 64) * L::kXBoxBytes + (v0 % 64) * 2) >> 4);
                            // rows 16 h .. 16 h + 15 of X: 16 rows of 128 bytes further
                            // into the box, accumulator columns 16 h ..
#pragma unroll
                            for (int hh = 0; hh < NC / kMmaN; ++hh) {
                                const uint64_t bd = bdesc + static_cast<uint64_t>((hh * kMmaN * 128) >> 4);
                                tc_mma_ts(tD + hh * kMmaN, tA + 8 * s, bd, kIdesc, s > 0 ? 1u : 0u);
                                if constexpr (L::kZtc) tc_mma_ts(tD + hh * kMmaN, tZ, bd, kIdesc, 1u);
                            }
                        }
                    });
                    tc_commit(&bars.afree[as.slot]);
                    tc_commit(&bars.dfull[ds.slot]);
                    if (BB == 1) tc_commit(&bars.empty[st.slot]);
                }
                __syncwarp();
                as.next();
                ds.next();
            });
            st.next();
        }
        if (!ok && lane == 0) record_error_tc(c.err, abort_flag);
        // every MMA issued above has completed once `drain` flips
        if (elect_one()) tc_commit(&bars.drain);
        __syncwarp();
        volatile int never = 0;
        mbar_wait(&bars.drain, 0, &never);
        named_bar_sync(3, kTail);
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
        return;
    }

    if (warp >= L::kUW) {
        // ------------------------------------------------------------ epilogue
        epilogue_warp<BITS, G, NC, EPI, HOLD, CLU>(c, bars, tmem, abort_flag, warp & 3, lane, n_units,
                                                   smem_u32 + L::kFixOff, crank, csize);
    } else if constexpr (BITS == 3) {
        // ------------------------------------------------------------ unpack
        static_for<0, L::kSplit>([&](auto hc) {
            constexpr int H = decltype(hc)::value;
            if ((warp >> 2) == H)
                unpack_warp<BITS, G, NC, H>(c, smem_u32, bars, tmem, abort_flag, warp, lane, n_units);
        });
    } else {
        unpack_warp<BITS, G, NC, -1>(c, smem_u32, bars, tmem, abort_flag, warp, lane, n_units);
    }
    named_bar_sync(3, kTail);
}

template <int BITS, int G, int NC>
cudaError_t launch_tc_nc(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmArgs& a,
                         cudaStream_t s) {
    using L = Lay<BITS, G, NC>;
    auto kern = a.epi == WQ_EPI_SWIGLU ? gemm_tc_kernel<BITS, G, NC, false, kEpiAct>
                                       : gemm_tc_kernel<BITS, G, NC, false, kEpiY>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (!a.pdl) {
        kern<<<a.P, L::kThreads, L::kSmemBytes, s>>>(tmW, tmX, a, StepArgs{});
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(a.P));
    cfg.blockDim = dim3(L::kThreads);
    cfg.dynamicSmemBytes = L::kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tmW, tmX, a, StepArgs{});
}

// Single projection: the 16-row build for M <= 16, the 32-row one above.
template <int BITS, int G>
cudaError_t launch_tc(const CUtensorMap& tmW, const CUtensorMap& tmX, const GemmArgs& a,
                      cudaStream_t s) {
    return a.nc == 32 ? launch_tc_nc<BITS, G, 32>(tmW, tmX, a, s)
                      : launch_tc_nc<BITS, G, 16>(tmW, tmX, a, s);
}

// Fused step launch; cooperative (all CTAs resident at once) when projections
// wait for one another.  A per-phase launch none of whose projections asks
// for the activation takes the build without it (measured 3 % faster on the
// per-phase layer chain; the single fused launch measured faster with it).
// A per-phase launch in clusters of sa.cluster CTAs (one tile per cluster).
template <int BITS, int G>
cudaError_t launch_step_cluster(const StepArgs& sa, cudaStream_t s) {
    using L = Lay<BITS, G, 16>;
    if constexpr (!L::kCluOk) {
        return cudaErrorNotSupported;
    } else {
        if (sa.cluster < 2 || sa.cluster > L::kFixMaxK || sa.P % sa.cluster != 0 || sa.act)
            return cudaErrorInvalidValue;
        auto kern = gemm_tc_kernel<BITS, G, 16, true, kEpiY, true, true>;
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytesClu);
        if (e != cudaSuccess) return e;
        CUtensorMap none{};
        GemmArgs a{};
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(sa.P));
        cfg.blockDim = dim3(L::kThreads);
        cfg.dynamicSmemBytes = L::kSmemBytesClu;
        cfg.stream = s;
        cudaLaunchAttribute attr[2];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(sa.cluster);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        // whether the device can place clusters of this size at all (checked
        // once per size; a launch it cannot place is not issued)
        static int placeable[L::kFixMaxK + 1] = {};  // 0 unknown, 1 yes, 2 no
        int& ok = placeable[sa.cluster];
        if (ok == 0) {
            int n = 0;
            ok = cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n >= 1 ? 1 : 2;
            (void)cudaGetLastError();
        }
        if (ok != 1) return cudaErrorNotSupported;
        cfg.numAttrs = sa.pdl ? 2 : 1;
        return cudaLaunchKernelEx(&cfg, kern, none, none, a, sa);
    }
}

template <int BITS, int G, int NC>
cudaError_t launch_step_nc(const StepArgs& sa, bool cooperative, cudaStream_t s) {
    using L = Lay<BITS, G, NC>;
    if constexpr (NC == 16)
        if (sa.cluster > 1) return launch_step_cluster<BITS, G>(sa, s);
    auto kern = !sa.pdl ? gemm_tc_kernel<BITS, G, NC, true, kEpiAny, false>
                : sa.act ? gemm_tc_kernel<BITS, G, NC, true, kEpiAny, true>
                         : gemm_tc_kernel<BITS, G, NC, true, kEpiY, true>;
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmemBytes);
    if (e != cudaSuccess) return e;
    CUtensorMap none{};
    GemmArgs a{};
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(static_cast<unsigned>(sa.P));
    cfg.blockDim = dim3(L::kThreads);
    cfg.dynamicSmemBytes = L::kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    if (sa.pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
    } else {
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = cooperative ? 1 : 0;
    }
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, none, none, a, sa);
}

template <int BITS, int G>
cudaError_t launch_step(const StepArgs& sa, bool cooperative, int nc, cudaStream_t s) {
    return nc == 32 ? launch_step_nc<BITS, G, 32>(sa, cooperative, s)
                    : launch_step_nc<BITS, G, 16>(sa, cooperative, s);
}

}  // namespace tc
}  // namespace wq
