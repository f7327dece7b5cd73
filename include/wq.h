/*
 * libwq — weight-only low-bit skinny GEMM for the decode step (sm_103a).
 *
 * The operation (OpenJet news page "单张 RTX 3090 跑 4 个编码 agent", paragraph
 * "并行解码的原理"): in a decode step every packed low-bit weight is streamed
 * from memory once and, while on chip, multiplied against all stacked rows
 * (each active agent's next token plus its draft tokens):
 *
 *     Y[M][N] = X[M][K] . dequant(Wq)[N][K]^T,   M = 1..32
 *     dequant(Wq)[n][k] = (q[n][k] - z[n][k/G]) * s[n][k/G]
 *
 * with 2/3/4-bit codes chosen per layer and repacked at load time (Agens
 * Engine page, section "功能": 混合 2/3/4-bit 权重, 加载时重新打包) and a group
 * size of 128 along K for the 4-bit format (Agens SGLang README, "Quick
 * start": W4A16, group size 128).
 *
 * Data layout (all row-major, all pointers are DEVICE pointers owned by the
 * caller unless stated otherwise):
 *   q       uint8  [N][K]        unpacked codes; only the low `bits` bits are used
 *   wq      uint32 [N][W]        packed codes, W = wq_packed_words_per_row(K, bits):
 *                                code k of a row lives in word k / vpw; with
 *                                j = k % vpw it takes bits [16*(j % 2) +
 *                                bits*(j / 2), ... + bits): even-numbered codes
 *                                fill the low half-word and odd-numbered codes
 *                                the high half-word, each half least significant
 *                                first; vpw = 8 (4-bit), 10 (3-bit, bits 15 and
 *                                31 zero), 16 (2-bit); words run along K across
 *                                group boundaries; unused slots and the padding
 *                                words that round a row up to a multiple of 4
 *                                words (16 bytes) are zero
 *   scales  bf16   [N][K/G]      per-group scale s (bf16 bit patterns, uint16)
 *   zeros   uint8  [N][K/G]      per-group zero point z: in [0, 2^bits - 1] as
 *                                the codes (any z <= 127 works); wq_gemm and the
 *                                step driver form 128 + z as a bf16 bit pattern,
 *                                so z >= 128 gives wrong results there (device
 *                                data: not checked); wq_dequant is exact for
 *                                any uint8
 *   x       bf16   [M][K]        activations (bf16 bit patterns)
 *   y       fp32   [M][N]        output
 *   w       bf16   [N][K]        dequantised weights (wq_dequant output)
 *
 * Arguments: bits in {2, 3, 4}; group in {32, 64, 128}; K % group == 0;
 * 0 <= M <= 32 (up to 16 rows per MMA column block: M <= 16 runs the 16-row
 * kernel build, 17..32 the 32-row build, and a row's result is bitwise the
 * same in both); N, K >= 0.  x and wq must be 16-byte aligned, y 4-byte
 * aligned, scales 2-byte aligned (16-byte aligned scales and zeros take a
 * faster path in wq_gemm).  Streams are passed as `void*` holding a
 * cudaStream_t (NULL = the legacy default stream).  Every call is
 * asynchronous on its stream and returns a status; kernels never trap:
 * invalid arguments are rejected on the host before anything is launched.
 * Calls on distinct streams are thread-safe except where a workspace is
 * shared (see wq_gemm).
 */
#ifndef WQ_H
#define WQ_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    WQ_OK = 0,
    WQ_ERR_INVALID_ARG = 1, /* null pointer, bad size/bits/group, misalignment, small workspace */
    WQ_ERR_UNSUPPORTED = 2, /* device is not sm_103, or a feature the build lacks */
    WQ_ERR_CUDA = 3,        /* a CUDA runtime call failed; see wq_last_cuda_error() */
    WQ_ERR_TIMEOUT = 4      /* a kernel gave up a bounded wait (wq_check_workspace) */
} wq_status_t;

/* ABI version of this header (major * 100 + minor). */
int wq_abi_version(void);

/* Static description of a status code. */
const char* wq_status_string(wq_status_t status);

/* cudaError_t of the last failing CUDA call made by this thread inside libwq. */
int wq_last_cuda_error(void);

/* Words per packed row: ceil(K / vpw) rounded up to a multiple of 4, or -1 for
 * bad arguments.  Layout: see the header comment. */
long wq_packed_words_per_row(int K, int bits);

/*
 * wq_pack — repack unpacked codes q[N][K] into wq[N][W] (load time; Agens
 * Engine page, section "功能": 加载时重新打包).  Bit-exact; the padding words of
 * every row are written as zero.  q and wq must not overlap.
 */
wq_status_t wq_pack(const uint8_t* q, uint32_t* wq, int N, int K, int bits, void* stream);

/* wq_unpack — inverse of wq_pack (a test aid): wq[N][W] -> q[N][K].  No
 * passage of the pages defines it; it exists to check the packed layout. */
wq_status_t wq_unpack(const uint32_t* wq, uint8_t* q, int N, int K, int bits, void* stream);

/*
 * wq_dequant — materialise bf16 weights w[N][K] = RNE_bf16((q - z) * s), the
 * exact product rounded once to nearest even.  Group-wise scale and zero point
 * along K: Agens SGLang README, "Quick start" (W4A16, group size 128).
 * Bit-exact against the plain definition (Agens SGLang README, "Server
 * environment variables": fast paths are bit-exact with the plain path).
 */
wq_status_t wq_dequant(const uint32_t* wq, const uint16_t* scales, const uint8_t* zeros,
                       uint16_t* w, int N, int K, int group, int bits, void* stream);

/*
 * Workspace for wq_gemm on the CURRENT device (its SM count sets the grid):
 * split-K partial sums and per-tile arrival counters (it depends on N and the
 * SM count, never on M; call it with the device that will run the GEMM
 * current).  Returns 0 for bad arguments.  No passage of the pages defines it;
 * it sizes the library's own scratch.
 */
size_t wq_workspace_bytes(int M, int N, int K, int group, int bits);

/*
 * The same for a device with sm_count SMs (sm_count > 0), whether or not it
 * is the current one: a workspace sized for sm_count serves every device
 * with at most that many SMs.  Host arithmetic only (no CUDA call).  Returns
 * 0 for bad arguments.  No passage of the pages defines it.
 */
size_t wq_workspace_bytes_for(int M, int N, int K, int group, int bits, int sm_count);

/* Zero a caller-owned workspace (required once before its first use; every
 * wq_gemm call leaves it zeroed again). */
wq_status_t wq_workspace_init(void* workspace, size_t workspace_bytes, void* stream);

/*
 * wq_gemm — Y[M][N] = X[M][K] . dequant(Wq)[N][K]^T with fp32 accumulation
 * (OpenJet news page, paragraph "并行解码的原理": one pass over the packed
 * weights against all stacked rows, on tensor cores).
 *
 * Numerics: (q - z) enters the tensor-core product exactly; the bf16 scale is
 * applied per group in fp32; Y is fp32.  The reduction order of every output
 * depends only on (N, K, group, bits, SM count), never on M or on the other
 * rows of X, so a row's result is bit-identical whether it is computed alone
 * or stacked with other rows (OpenJet news page, "新提示不会让所有人停摆":
 * results bit-identical to processing alone), and repeated calls are
 * bit-identical.
 *
 * workspace: device buffer of at least wq_workspace_bytes(...) bytes, zeroed
 * once by wq_workspace_init; calls that share one workspace must be ordered
 * (same stream).  workspace == NULL uses a library-owned buffer per device,
 * allocated (and zeroed) on the first call on that device — make that first
 * call outside stream capture; the library buffer must not be used by calls
 * that overlap on the GPU.
 */
wq_status_t wq_gemm(const uint16_t* x, const uint32_t* wq, const uint16_t* scales,
                    const uint8_t* zeros, float* y, int M, int N, int K, int group, int bits,
                    void* workspace, size_t workspace_bytes, void* stream);

/* Epilogues: what a projection writes from its fp32 sums acc[M][N]. */
#define WQ_EPI_NONE 0   /* y: fp32 [M][N] = acc */
#define WQ_EPI_SWIGLU 1 /* y: bf16 [M][N/2], y[m][j] = bf16(silu(acc[m][2j]) * acc[m][2j+1]) */

/*
 * wq_gemm_swiglu — the fused gate/up projection of a gated MLP with its
 * activation applied in the epilogue: y[m][j] = RNE_bf16(silu(g) * u) with
 * g = acc[m][2j], u = acc[m][2j+1], silu(g) = g / (1 + e^-g) in fp32 with the
 * fast exponential and division (a few fp32 ulps, far below the bf16 step; a
 * gate below about -87.3 gives 0 where the exact value is under 1e-36 |u|),
 * acc the wq_gemm sums.  The pages fuse gate and up into one weight stream (OpenJet
 * news page, "并行解码的原理": one pass over every weight per step) for
 * Qwen-family models without naming the activation; SwiGLU is the reading.
 * Layout: N even; weight rows (and their scale and zero-point rows) are
 * interleaved at load time, row 2j = gate row of feature j, row 2j + 1 = up
 * row; y is bf16 [M][N/2] row-major (the down projection's X), 2-byte
 * aligned.  Everything else (x, wq, scales, zeros, workspace, errors) as
 * wq_gemm; the fp32 sums are those of wq_gemm bit for bit, so y equals the
 * activation applied to wq_gemm's output to within one bf16 step.
 */
wq_status_t wq_gemm_swiglu(const uint16_t* x, const uint32_t* wq, const uint16_t* scales,
                           const uint8_t* zeros, uint16_t* y, int M, int N, int K, int group,
                           int bits, void* workspace, size_t workspace_bytes, void* stream);

/*
 * wq_gemm_noalloc — wq_gemm without any device allocation.  The paper has no
 * counterpart: this entry point exists for callers that cannot call cudaMalloc,
 * e.g. code running inside a framework or server that owns all device memory
 * through its own pool, code on a path where an allocation would synchronise
 * the device or break a fixed memory budget, and code that must not fail
 * halfway through a step for lack of memory.  The caller still passes x, wq,
 * scales, zeros and y (same layout and rules as wq_gemm).
 *
 * Scratch: a fixed 8 MiB file-scope device array inside libwq, held by every
 * GPU that loads the library until the process exits.  The first call on a
 * device sets it up (looks up its device address and zeroes it on `stream`);
 * make that first call before any stream capture.  Every call re-zeroes the
 * per-tile counters it needs.  Problems whose scratch (wq_workspace_bytes)
 * would exceed 8 MiB — N beyond about 6.8 million rows on a 152-SM GPU — are
 * rejected with WQ_ERR_INVALID_ARG before anything is launched.  All calls
 * share the one array, so calls that overlap on the GPU (different streams,
 * or different host threads without ordering) race and give wrong results;
 * order them on one stream.  Nothing is allocated or freed.  The kernel's
 * error word (a bounded wait that ran out) sits in the same array: read it
 * with wq_check_noalloc.
 */
wq_status_t wq_gemm_noalloc(const uint16_t* x, const uint32_t* wq, const uint16_t* scales,
                            const uint8_t* zeros, float* y, int M, int N, int K, int group,
                            int bits, void* stream);

/*
 * wq_check_noalloc — the error word of wq_gemm_noalloc's fixed array on the
 * current device, read after synchronising `stream`: WQ_OK, or WQ_ERR_TIMEOUT
 * if a wq_gemm_noalloc kernel abandoned a bounded wait since the last check
 * (its y is then wrong).  Clears the word and, after WQ_ERR_TIMEOUT, zeroes
 * the whole array (no allocation).  WQ_OK before the first call on a device.
 * The paper has no counterpart (see wq_gemm_noalloc).
 */
wq_status_t wq_check_noalloc(void* stream);

/*
 * Read back the kernel error word of a workspace (NULL = the library buffer
 * of the current device) after synchronising `stream`: WQ_OK, or
 * WQ_ERR_TIMEOUT if a kernel abandoned a bounded wait since the last check.
 * Clears the word.  After WQ_ERR_TIMEOUT the library buffer has been zeroed
 * whole; a caller-owned workspace may still hold split-K counters of the
 * abandoned launch and must be zeroed again (wq_workspace_init) before reuse.
 */
wq_status_t wq_check_workspace(void* workspace, void* stream);

/* ---------------------------------------------------------------------------
 * Decode-step driver: a whole layer stack's projections on one stream
 * (OpenJet news page, paragraph "并行解码的原理": every projection of every
 * layer streams its weights once per step, and the whole step runs as one
 * persistent kernel with no per-layer launch).
 * ------------------------------------------------------------------------ */
typedef struct wq_proj_desc {
    const uint16_t* x;       /* [M][K] bf16 */
    const uint32_t* wq;      /* [N][W] */
    const uint16_t* scales;  /* [N][K/G] bf16 */
    const uint8_t* zeros;    /* [N][K/G] */
    void* y;                 /* fp32 [M][N]; bf16 [M][N/2] with WQ_EPI_SWIGLU */
    int M, N, K, group, bits;
    /* Fused mode only: x is produced by projections 0..after of the same
     * call (through whatever the caller computes in between), so it is read
     * only once those have written all of y; -1 = x is ready when the call
     * starts.  Must be smaller than the projection's own index.  Ignored in
     * sequential mode, where stream order already serialises everything. */
    int after;
    /* WQ_EPI_NONE: y is fp32 [M][N]; WQ_EPI_SWIGLU: y is bf16 [M][N/2] as in
     * wq_gemm_swiglu (N even, gate/up rows interleaved). */
    int epilogue;
} wq_proj_desc_t;

/* Step modes.
 * 0 (sequential): one wq_gemm launch per projection, in order.  Each launch
 *   that directly follows another of the step is a programmatic dependent
 *   launch: its CTAs start as the previous kernel's leave and load their
 *   first packed weights, zero points and scales at once, while x and y are
 *   touched only after the previous kernel has completed.  So the packed
 *   weights, scales and zero points of a step must not be written by the
 *   step itself (x may be: it is produced by the previous projection).
 * WQ_STEP_FUSED: one persistent launch per run of consecutive projections
 *   with the same bit width and group size.  The launch streams the units of
 *   all its projections back to back (stream-K across projection
 *   boundaries), so projections overlap unless `after` says otherwise;
 *   packed weights of a waiting projection are still streamed in while it
 *   waits, only its X is held back.  Launches that wait are cooperative
 *   (all CTAs resident).  The split-K order differs from single calls, so
 *   results agree with wq_gemm to rounding, not bit for bit; a row alone is
 *   still bit-identical to the same row stacked. */
#define WQ_STEP_FUSED 1u
/* With WQ_STEP_FUSED: each dependency phase of a run (a projection whose
 * `after` names a projection of the current phase starts a new one) is its own
 * persistent launch over all of that phase's projections, and stream order --
 * every launch after the first a programmatic dependent of the one before --
 * replaces the device-side waits between phases.  Independent projections of a
 * phase still share one launch and one stream-K split.  Each launch takes a
 * grid whose shares fall on tile boundaries where one lies near the SM count,
 * so its split can differ from WQ_STEP_FUSED's: results agree with the fused
 * launch to rounding; a row alone is still bit-identical to the same row
 * stacked, and repeated steps are bit-identical.  A launch with two CTAs per
 * tile runs one thread-block cluster per tile, whose split-K sums meet in
 * shared memory instead of global memory.  Not part of the pages: a launch
 * plan for the same step. */
#define WQ_STEP_PHASES 2u

/* Workspace bytes for a step in the given mode (0 for invalid input).  In
 * fused mode it holds the error word, split-K partials and counters, the
 * per-projection completion counters and the projection table. */
size_t wq_step_workspace_bytes(const wq_proj_desc_t* projs, int count, unsigned flags);

/* Run the step once.  Sequential mode accepts any workspace wq_gemm accepts
 * (NULL = the library buffer); fused mode needs `workspace` of at least
 * wq_step_workspace_bytes(), 16-byte aligned, zeroed once (wq_workspace_init)
 * before its first use.  Every launch leaves the workspace's counters zeroed,
 * so one workspace serves, one step at a time on one stream, every descriptor
 * set it is large enough for. */
wq_status_t wq_step_run(const wq_proj_desc_t* projs, int count, void* workspace,
                        size_t workspace_bytes, void* stream);
wq_status_t wq_step_run_ex(const wq_proj_desc_t* projs, int count, unsigned flags,
                           void* workspace, size_t workspace_bytes, void* stream);

typedef struct wq_step_graph* wq_step_graph_t;

/* Capture the step once into a CUDA graph (no host work per replay).  The
 * descriptors' pointers are baked in: the buffers must stay alive and in
 * place while the graph exists.  `workspace` must be non-NULL.  In fused mode
 * the graph owns a device copy of the projection table (allocated here, freed
 * by wq_step_graph_destroy). */
wq_status_t wq_step_graph_create(const wq_proj_desc_t* projs, int count, void* workspace,
                                 size_t workspace_bytes, void* stream, wq_step_graph_t* out);
wq_status_t wq_step_graph_create_ex(const wq_proj_desc_t* projs, int count, unsigned flags,
                                    void* workspace, size_t workspace_bytes, void* stream,
                                    wq_step_graph_t* out);
wq_status_t wq_step_graph_launch(wq_step_graph_t graph, void* stream);
void wq_step_graph_destroy(wq_step_graph_t graph);

/*
 * wq_paged_attention — decode attention over a paged q8_0 KV pool (OpenJet
 * news page, paragraphs after "并行解码的原理": one shared pool in q8_0,
 * managed in pages; attention, each agent reading its own cache, is what grows
 * with the agents).  Query row i attends to positions 0 .. row_pos[i] of
 * sequence row_seq[i]; query head h reads key/value head h / (Hq / Hkv):
 *   out[i][h] = sum_t softmax_t(q[i][h] . k[t] / sqrt(D)) v[t]
 * with k and v dequantised from q8_0 (blocks of 32 signed 8-bit codes along
 * the head dimension, value = binary16 scale * code).
 *
 * Layout (device pointers): q bf16 [rows][Hq][D]; k_codes, v_codes int8
 * [pages][Hkv][T][D] (16-byte aligned); k_scales, v_scales binary16
 * [pages][Hkv][T][D/32] (8-byte aligned); page_table int32 [B][max_pages] (sequence b's token t
 * in physical page page_table[b][t / T], slot t % T; pages may be shared);
 * seq_len int32 [B]; row_seq, row_pos int32 [rows]; out fp32 [rows][Hq][D].
 * D = 128; Hq a multiple of Hkv with Hq / Hkv <= 16; max_seq_len (host) bounds
 * every seq_len and max_pages * T >= max_seq_len.  workspace: at least
 * wq_paged_attention_workspace_bytes(rows, Hq, Hkv, B, max_seq_len) bytes (the
 * slices per sequence follow the current device's size), 16-byte
 * aligned, its first word zero; a page index outside the pool, a position
 * past its sequence or a sequence longer than max_seq_len sets that word to 2
 * (the affected rows read nothing).  Rows whose row_seq is not in [0, B)
 * produce zeros.  Deterministic: the same inputs give the same bits.
 */
size_t wq_paged_attention_workspace_bytes(int rows, int Hq, int Hkv, int B, int max_seq_len);
wq_status_t wq_paged_attention(const uint16_t* q, const int8_t* k_codes, const uint16_t* k_scales,
                               const int8_t* v_codes, const uint16_t* v_scales,
                               const int* page_table, int max_pages, const int* seq_len, int B,
                               const int* row_seq, const int* row_pos, int rows, int max_seq_len,
                               int Hq, int Hkv, int D, int T, int pages, float* out,
                               void* workspace, size_t workspace_bytes, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* WQ_H */
