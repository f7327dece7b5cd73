// Plain, slow, fp64 CPU oracle for the weight-only low-bit skinny GEMM.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the library path links, loads or calls
// this file; it shares no code, header, table or constant with the CUDA
// kernels.  Only the tests, the smoke check and the benchmark's CPU-baseline
// leg use it.
//
// What it computes (every step written out as its definition, no blocking or
// reordering beyond a plain loop):
//
//   Y[m][n] = sum_k X[m][k] * W[n][k],   W[n][k] = (q[n][k] - z[n][k/G]) * s[n][k/G]
//
// * One weight stream multiplied against all stacked rows of X: OpenJet news
//   page ("单张 RTX 3090 跑 4 个编码 agent"), paragraph "并行解码的原理" —
//   every weight is read once per decode step and multiplied, while on chip,
//   against every active row (each agent's next token plus its drafts).
// * Weight-only low-bit codes with a per-group scale, group size 128 along K,
//   16-bit activations: Agens SGLang README, "Quick start" (W4A16, group 128).
// * Bit widths 2, 3 and 4, chosen per layer and repacked at load time: Agens
//   Engine page, section "功能" (混合 2/3/4-bit 权重, 加载时重新打包).
// * The pages never write the dequantisation formula, the bit order inside a
//   word or the zero-point storage.  Readings taken here:
//     - asymmetric affine dequantisation w = (q - z) * s, unsigned q, integer z;
//     - codes are packed along K, vpw consecutive codes per 32-bit word,
//       vpw = 8 (b=4), 10 (b=3), 16 (b=2); words run along K ignoring group
//       boundaries.  Inside a word the even-numbered codes fill the low
//       half-word and the odd-numbered codes the high half-word, each half
//       least significant first: code k sits in word k / vpw, slot
//       j = k % vpw, at bits [16*(j % 2) + b*(j / 2), ... + b).  (Load-time
//       repacking is the pages' own step, so the word layout is the
//       implementation's to choose; this one puts two neighbouring codes at
//       the same place in the two 16-bit halves.)  For b = 3 bits 15 and 31
//       stay zero; unused slots are zero; each row is padded with zero words
//       to a multiple of 4 words (16 bytes);
//     - only the low b bits of each code are stored;
//     - scales are bf16 [N][K/G], zero points uint8 [N][K/G], both row-major;
//     - X is bf16 [M][K] row-major, Y is [M][N] row-major.
//
// Fused gate/up activation (wqo_silu_f64, wqo_swiglu_bf16): the pages run
// Qwen-family models (OpenJet news page, title: Qwen3.8-27B) and fuse a
// layer's gate and up projections into one weight stream, but never write the
// activation.  Reading: the gated SiLU unit of those models,
// out[m][j] = silu(gate) * up with silu(g) = g / (1 + e^-g), the gate and up
// rows of feature j interleaved as rows 2j and 2j + 1 of the fused
// projection, rounded once to bf16 (the next projection's X is bf16).
//
// Precision: q - z is an integer of magnitude < 2^8 and s is a bf16 (8
// significant bits), so W is exact in double; X is bf16, so each product is
// exact and only the K-term sum rounds (in double, k ascending).
// Parity status: pinned (tests/test_oracle.py); no function here is unpinned.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

int values_per_word(int bits) {
    if (bits == 4) return 8;
    if (bits == 3) return 10;
    if (bits == 2) return 16;
    return 0;
}

// First bit of slot j (0 <= j < vpw) inside its word.
int slot_shift(int bits, int j) { return 16 * (j % 2) + bits * (j / 2); }

double bf16_bits_to_double(uint16_t b) {
    uint32_t u = static_cast<uint32_t>(b) << 16;
    float f;
    std::memcpy(&f, &u, sizeof f);
    return static_cast<double>(f);
}

}  // namespace

extern "C" {

// Words per packed row: ceil(K / vpw) rounded up to a multiple of 4.
long wqo_words_per_row(int K, int bits) {
    int vpw = values_per_word(bits);
    if (vpw == 0 || K < 0) return -1;
    long used = (static_cast<long>(K) + vpw - 1) / vpw;
    return (used + 3) / 4 * 4;
}

// Pack codes q[N][K] (uint8) into words wq[N][W], following the layout above.
int wqo_pack(const uint8_t* q, uint32_t* wq, int N, int K, int bits) {
    int vpw = values_per_word(bits);
    if (vpw == 0) return 1;
    long W = wqo_words_per_row(K, bits);
    uint32_t mask = (1u << bits) - 1u;
    for (long n = 0; n < N; ++n) {
        for (long w = 0; w < W; ++w) wq[n * W + w] = 0u;
        for (long k = 0; k < K; ++k) {
            uint32_t code = static_cast<uint32_t>(q[n * K + k]) & mask;
            long word = k / vpw;
            int slot = static_cast<int>(k % vpw);
            wq[n * W + word] |= code << slot_shift(bits, slot);
        }
    }
    return 0;
}

// Inverse of the packing: code k of row n.
int wqo_unpack(const uint32_t* wq, uint8_t* q, int N, int K, int bits) {
    int vpw = values_per_word(bits);
    if (vpw == 0) return 1;
    long W = wqo_words_per_row(K, bits);
    uint32_t mask = (1u << bits) - 1u;
    for (long n = 0; n < N; ++n)
        for (long k = 0; k < K; ++k) {
            uint32_t word = wq[n * W + k / vpw];
            q[n * K + k] = static_cast<uint8_t>((word >> slot_shift(bits, static_cast<int>(k % vpw))) & mask);
        }
    return 0;
}

// Exact dequantised weight W[n][k] = (q - z[n][k/G]) * s[n][k/G] in double.
int wqo_dequant_f64(const uint32_t* wq, const uint16_t* s, const uint8_t* z, double* w,
                    int N, int K, int G, int bits) {
    int vpw = values_per_word(bits);
    if (vpw == 0 || G <= 0 || K % G != 0) return 1;
    long W = wqo_words_per_row(K, bits);
    long ng = K / G;
    uint32_t mask = (1u << bits) - 1u;
    for (long n = 0; n < N; ++n)
        for (long k = 0; k < K; ++k) {
            uint32_t code = (wq[n * W + k / vpw] >> slot_shift(bits, static_cast<int>(k % vpw))) & mask;
            long g = k / G;
            double diff = static_cast<double>(code) - static_cast<double>(z[n * ng + g]);
            w[n * K + k] = diff * bf16_bits_to_double(s[n * ng + g]);
        }
    return 0;
}

// Round a double to the nearest bf16 (8 significant bits), ties to even,
// returning the bf16 bit pattern.  Written from the definition: scale the
// significand to an 8-bit integer range, round half to even, scale back.
// Domain: finite values whose magnitude lies in the normal bf16 range or is 0
// (true for every product (q - z) * s with a normal bf16 scale).
uint16_t wqo_bf16_rne(double v) {
    if (v == 0.0) return std::signbit(v) ? 0x8000u : 0x0000u;
    int e;
    double m = std::frexp(v, &e);          // v = m * 2^e, 0.5 <= |m| < 1
    double r = std::nearbyint(std::ldexp(m, 8));  // 8 significant bits, ties to even
    double rounded = std::ldexp(r, e - 8);  // exact: r has at most 9 bits
    float f = static_cast<float>(rounded);  // exact (fits in a float)
    uint32_t u;
    std::memcpy(&u, &f, sizeof u);
    return static_cast<uint16_t>(u >> 16);  // low 16 bits are zero
}

// SiLU, written from its definition: g * sigmoid(g) = g / (1 + e^-g).
double wqo_silu_f64(double g) { return g / (1.0 + std::exp(-g)); }

// out[m][j] = bf16(silu(y[m][2j]) * y[m][2j + 1]) for y [M][N] in double
// (N even), one rounding of the double product.  Domain of wqo_bf16_rne:
// products that are 0 or in the normal bf16 range.
int wqo_swiglu_bf16(const double* y, int M, int N, uint16_t* out) {
    if (M < 0 || N < 0 || N % 2 != 0) return 1;
    const long nf = N / 2;
    for (long m = 0; m < M; ++m)
        for (long j = 0; j < nf; ++j)
            out[m * nf + j] = wqo_bf16_rne(wqo_silu_f64(y[m * N + 2 * j]) * y[m * N + 2 * j + 1]);
    return 0;
}

// bf16(W) with a single rounding of the exact product.
int wqo_dequant_bf16(const uint32_t* wq, const uint16_t* s, const uint8_t* z, uint16_t* w,
                     int N, int K, int G, int bits) {
    std::vector<double> row(static_cast<size_t>(K));
    long W = wqo_words_per_row(K, bits);
    long ng = (G > 0) ? K / G : 0;
    for (long n = 0; n < N; ++n) {
        int rc = wqo_dequant_f64(wq + n * W, s + n * ng, z + n * ng, row.data(), 1, K, G, bits);
        if (rc) return rc;
        for (long k = 0; k < K; ++k) w[n * K + k] = wqo_bf16_rne(row[k]);
    }
    return 0;
}

// Y[m][n] = sum_k X[m][k] * W[n][k] in double, k ascending.  ``threads`` > 0
// sets the OpenMP thread count (rows of W are split across threads; every
// output is still one sequential sum, so the result does not depend on it).
int wqo_gemm_f64(const uint16_t* x, const uint32_t* wq, const uint16_t* s, const uint8_t* z,
                 double* y, int M, int N, int K, int G, int bits, int threads) {
    int vpw = values_per_word(bits);
    if (vpw == 0 || G <= 0 || K % G != 0 || M < 0 || N < 0) return 1;
    long W = wqo_words_per_row(K, bits);
    long ng = K / G;
    std::vector<double> xd(static_cast<size_t>(M) * K);
    for (long i = 0; i < static_cast<long>(M) * K; ++i) xd[i] = bf16_bits_to_double(x[i]);
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel
#endif
    {
        std::vector<double> wrow(static_cast<size_t>(K));
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
        for (long n = 0; n < N; ++n) {
            wqo_dequant_f64(wq + n * W, s + n * ng, z + n * ng, wrow.data(), 1, K, G, bits);
            for (long m = 0; m < M; ++m) {
                double acc = 0.0;
                const double* xr = xd.data() + m * K;
                for (long k = 0; k < K; ++k) acc += xr[k] * wrow[k];
                y[m * N + n] = acc;
            }
        }
    }
    return 0;
}

// Number of OpenMP threads the oracle would use with ``threads`` (0 = default).
int wqo_max_threads(int threads) {
#ifdef _OPENMP
    return threads > 0 ? threads : omp_get_max_threads();
#else
    (void)threads;
    return 1;
#endif
}

}  // extern "C"
