// Plain, slow, fp64 CPU oracle for decode attention over a paged q8_0 KV pool.
//
// TEST INFRASTRUCTURE ONLY.  Nothing in the library path links, loads or calls
// this file; it shares no code, header, table or constant with the CUDA
// kernels.
//
// The workload (OpenJet news page, "单张 RTX 3090 跑 4 个编码 agent"): what grows
// with the number of agents in a decode step is attention, each agent reading
// its own KV cache (paragraph "并行解码的原理"); the cache is one shared pool of
// 132K tokens stored as q8_0 and managed in pages, so that one agent can hold
// most of it while the others stay short, and a shared system prompt is
// stored once (the paragraphs after it).
//
// The pages give neither the attention shapes nor the page layout.  Readings
// taken here:
//   * q8_0 as the format of that name: blocks of 32 consecutive values along
//     the head dimension, each an IEEE binary16 scale d and 32 signed 8-bit
//     codes c; value = d * c;
//   * grouped-query attention: Hq query heads share Hkv key/value heads, query
//     head h reading key/value head h / (Hq / Hkv); head dimension D, a
//     multiple of 32; score = (q . k) / sqrt(D); softmax over the attended
//     positions; output = the softmax-weighted sum of the values;
//   * the pool holds `pages` pages of T tokens; K and V each as codes
//     int8 [pages][Hkv][T][D] and scales fp16 [pages][Hkv][T][D/32];
//     sequence b's logical page p is physical page page_table[b][p], so its
//     token t lives in page page_table[b][t / T], slot t % T (pages may be
//     shared between sequences: a common prompt stored once);
//   * every query row belongs to a sequence and a position: it attends to
//     positions 0 .. pos of its sequence (the new rows' own keys and values
//     are in the cache; a draft row sees the rows before it, not after);
//   * queries are bf16 [rows][Hq][D]; the output is [rows][Hq][D].
//
// Everything is computed in double: the q8_0 values and the bf16 queries are
// exact in double, each score is a plain dot product in ascending d, the
// softmax subtracts the row maximum before exp, and the weighted sum runs over
// ascending positions.
// Parity status: pinned (tests/test_attn_oracle.py).
#include <cmath>
#include <cstdint>
#include <vector>

namespace {

// IEEE binary16 bit pattern -> value (finite inputs; inf and NaN map to
// themselves in double).
double half_value(uint16_t h) {
    const int sign = (h >> 15) & 1;
    const int e = (h >> 10) & 0x1f;
    const int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = std::ldexp(static_cast<double>(m), -24);  // subnormal: m * 2^-24
    else if (e == 31)
        v = m == 0 ? INFINITY : NAN;
    else
        v = std::ldexp(static_cast<double>(1024 + m), e - 25);  // (1 + m/1024) * 2^(e-15)
    return sign ? -v : v;
}

double bf16_value(uint16_t b) {
    const uint32_t u = static_cast<uint32_t>(b) << 16;
    float f;
    static_assert(sizeof f == sizeof u, "float is 32-bit");
    __builtin_memcpy(&f, &u, sizeof f);
    return static_cast<double>(f);
}

}  // namespace

extern "C" {

double wqo_fp16_value(uint16_t h) { return half_value(h); }

// q8_0 blocks -> values: out[32 * i + j] = d[i] * c[32 * i + j].
int wqo_q8_0_dequant(const int8_t* c, const uint16_t* d, long n_blocks, double* out) {
    if (n_blocks < 0 || (n_blocks > 0 && (!c || !d || !out))) return 1;
    for (long i = 0; i < n_blocks; ++i) {
        const double s = half_value(d[i]);
        for (int j = 0; j < 32; ++j) out[32 * i + j] = s * static_cast<double>(c[32 * i + j]);
    }
    return 0;
}

int wqo_paged_attention_f64(const uint16_t* q, const int8_t* kc, const uint16_t* kd,
                            const int8_t* vc, const uint16_t* vd, const int* page_table,
                            const int* seq_len, const int* row_seq, const int* row_pos, int rows,
                            int B, int max_pages, int Hq, int Hkv, int D, int T, int pages,
                            double* out) {
    if (rows < 0 || B <= 0 || max_pages <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 ||
        D <= 0 || D % 32 != 0 || T <= 0 || pages <= 0)
        return 1;
    if (rows == 0) return 0;
    if (!q || !kc || !kd || !vc || !vd || !page_table || !seq_len || !row_seq || !row_pos || !out)
        return 1;
    for (int b = 0; b < B; ++b) {
        if (seq_len[b] < 0 || seq_len[b] > max_pages * T) return 1;
        for (int p = 0; p * T < seq_len[b]; ++p)
            if (page_table[b * max_pages + p] < 0 || page_table[b * max_pages + p] >= pages) return 1;
    }
    for (int i = 0; i < rows; ++i)
        if (row_seq[i] < 0 || row_seq[i] >= B || row_pos[i] < 0 || row_pos[i] >= seq_len[row_seq[i]])
            return 1;
    const int group = Hq / Hkv;
    const int nb = D / 32;
    const double inv_sqrt_d = 1.0 / std::sqrt(static_cast<double>(D));
    std::vector<double> k(D), v(D), score, acc(D);
    for (int i = 0; i < rows; ++i) {
        const int b = row_seq[i];
        const int n = row_pos[i] + 1;  // attended positions 0 .. row_pos
        score.assign(n, 0.0);
        for (int h = 0; h < Hq; ++h) {
            const int g = h / group;
            const uint16_t* qh = q + (static_cast<long>(i) * Hq + h) * D;
            // scores
            for (int t = 0; t < n; ++t) {
                const long page = page_table[b * max_pages + t / T];
                const long tok = ((page * Hkv + g) * T + t % T);
                wqo_q8_0_dequant(kc + tok * D, kd + tok * nb, nb, k.data());
                double s = 0.0;
                for (int d = 0; d < D; ++d) s += bf16_value(qh[d]) * k[d];
                score[t] = s * inv_sqrt_d;
            }
            // softmax
            double mx = score[0];
            for (int t = 1; t < n; ++t)
                if (score[t] > mx) mx = score[t];
            double den = 0.0;
            for (int t = 0; t < n; ++t) {
                score[t] = std::exp(score[t] - mx);
                den += score[t];
            }
            // weighted values
            for (int d = 0; d < D; ++d) acc[d] = 0.0;
            for (int t = 0; t < n; ++t) {
                const long page = page_table[b * max_pages + t / T];
                const long tok = ((page * Hkv + g) * T + t % T);
                wqo_q8_0_dequant(vc + tok * D, vd + tok * nb, nb, v.data());
                for (int d = 0; d < D; ++d) acc[d] += score[t] * v[d];
            }
            double* o = out + (static_cast<long>(i) * Hq + h) * D;
            for (int d = 0; d < D; ++d) o[d] = acc[d] / den;
        }
    }
    return 0;
}

}  // extern "C"
