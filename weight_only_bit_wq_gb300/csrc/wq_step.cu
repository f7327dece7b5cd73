// Decode-step driver: a layer stack's projections on one stream (OpenJet news
// page, paragraph "并行解码的原理": every projection of every layer streams its
// packed weights once per step; the whole step runs as one persistent kernel
// with no per-layer launch).
//
// Sequential mode launches wq_gemm once per projection.  Fused mode builds a
// table of projections (tensor maps, pointers, unit and tile offsets) and
// launches one persistent kernel per run of consecutive projections with the
// same bit width and group size; the kernel streams the units of the whole
// run, and a projection whose X depends on earlier ones waits for them on
// device-side completion counters while its packed weights are already being
// loaded.  Either sequence can be captured once into a CUDA graph.
#include <cuda_runtime.h>

#include <algorithm>
#include <new>
#include <vector>

#include "wq.h"
#include "wq_internal.h"

namespace {

size_t round256(size_t v) { return (v + 255) / 256 * 256; }

// A run: projections [begin, end) of one bit width and group size, all with
// M, N, K > 0 (other projections run through wq_gemm on their own); nc rows
// of X per tile, enough for the run's largest M.
struct Run {
    int begin, end, bits, group;
    bool fused;
    int nc;
};

std::vector<Run> split_runs(const wq_proj_desc_t* projs, int count) {
    std::vector<Run> runs;
    for (int i = 0; i < count; ++i) {
        const wq_proj_desc_t& p = projs[i];
        const bool fusable = p.M > 0 && p.N > 0 && p.K > 0;
        if (fusable && !runs.empty() && runs.back().fused && runs.back().end == i &&
            runs.back().bits == p.bits && runs.back().group == p.group) {
            runs.back().end = i + 1;
            runs.back().nc = std::max(runs.back().nc, wq::tc_cols(p.M));
        } else {
            runs.push_back({i, i + 1, p.bits, p.group, fusable, wq::tc_cols(p.M)});
        }
    }
    return runs;
}

// Fused-mode workspace layout, shared by every run of a step (runs execute
// one after another in stream order).
struct FusedLayout {
    size_t partial_off, counter_off, done_off, table_off, bytes;
};

int tiles_of(const wq_proj_desc_t& p) { return (p.N + wq::kBN - 1) / wq::kBN; }

// Device tables of a step: one projection slot and one phase slot per
// projection; run r uses the slots starting at its first projection.
size_t table_bytes(int count) {
    return static_cast<size_t>(count) * (sizeof(wq::ProjDev) + sizeof(wq::PhaseDev));
}
struct Tables {
    wq::ProjDev* proj;
    wq::PhaseDev* phase;
};
Tables tables_at(void* base, int count) {
    Tables t;
    t.proj = static_cast<wq::ProjDev*>(base);
    t.phase = reinterpret_cast<wq::PhaseDev*>(t.proj + count);
    return t;
}

// Workspace of a fused step: error word, split-K partials, split-K counters,
// completion counters, projection tables.  The offsets depend on the
// descriptor set (its tile and projection counts), so one set's completion
// counters or tables can sit where another set's split-K counters are; every
// call therefore leaves all of them zeroed (the kernel its split-K counters,
// memsets after the launch the rest), and one workspace serves every set it is
// large enough for.
FusedLayout fused_layout(const wq_proj_desc_t* projs, int count, const std::vector<Run>& runs,
                         int sms) {
    size_t max_tiles = 0, max_count = 0;
    for (const Run& r : runs) {
        if (!r.fused) continue;
        size_t t = 0;
        for (int i = r.begin; i < r.end; ++i) t += static_cast<size_t>(tiles_of(projs[i]));
        max_tiles = std::max(max_tiles, t);
        max_count = std::max(max_count, static_cast<size_t>(r.end - r.begin));
    }
    FusedLayout l;
    l.partial_off = wq::kWsHeader;
    l.counter_off = l.partial_off +
                    round256(size_t(2) * sms * wq::kMaxCols * wq::kBN * sizeof(float));
    l.done_off = l.counter_off + round256(max_tiles * wq::kCountersPerTile * sizeof(int));
    l.table_off = l.done_off + round256(max_count * sizeof(int));
    l.bytes = l.table_off + round256(table_bytes(count));
    return l;
}

wq_status_t check_all(const wq_proj_desc_t* projs, int count) {
    if (count < 0 || (count > 0 && !projs)) return WQ_ERR_INVALID_ARG;
    for (int i = 0; i < count; ++i) {
        const wq_proj_desc_t& p = projs[i];
        if (wq_status_t st = wq::host_check_gemm(p.x, p.wq, p.scales, p.zeros, p.y, p.M, p.N, p.K,
                                                 p.group, p.bits, p.epilogue))
            return st;
        if (p.after >= i || p.after < -1) return WQ_ERR_INVALID_ARG;
    }
    return WQ_OK;
}

// Host-side tables of one run.  The run is cut into phases: a projection
// that waits for a projection of the current phase starts a new phase, and
// every projection of a later phase then waits for all earlier phases (its X
// is held back; its packed weights still stream).  Returns the total units and
// whether anything waits.
wq_status_t build_table(const wq_proj_desc_t* projs, const Run& r, std::vector<wq::ProjDev>& out,
                        std::vector<wq::PhaseDev>& phases, long long* units, bool* waits) {
    out.assign(static_cast<size_t>(r.end - r.begin), wq::ProjDev{});
    phases.clear();
    long long uoff = 0;
    int toff = 0;
    int phase_start = 0;  // first projection (run-relative) of the current phase
    *waits = false;
    const int sv = wq::tc_stage_values(r.bits, r.group);
    for (int i = r.begin; i < r.end; ++i) {
        const wq_proj_desc_t& p = projs[i];
        const int li = i - r.begin;
        wq::ProjDev& d = out[static_cast<size_t>(li)];
        if (wq_status_t st = wq::host_encode_proj(p.x, p.wq, p.scales, p.zeros, p.M, p.N, p.K,
                                                  p.group, p.bits, r.nc, &d.tmW, &d.tmX, &d.x3d,
                                                  &d.meta_vec))
            return st;
        // a producer before this run is complete by stream order
        const int after = p.after >= r.begin ? p.after - r.begin : -1;
        if (li == 0 || after >= phase_start) {
            if (li > 0) *waits = true;
            phase_start = li;
            phases.push_back({uoff, 0, 0, 0});
        }
        d.scales = p.scales;
        d.zeros = p.zeros;
        d.y = static_cast<float*>(p.y);
        d.epi = p.epilogue;
        d.M = p.M;
        d.N = p.N;
        d.ng = p.K / p.group;
        d.T = tiles_of(p);
        d.I = (p.K + sv - 1) / sv;
        d.uoff = uoff;
        d.toff = toff;
        d.phase = static_cast<int>(phases.size()) - 1;
        // a later phase waits for the one before it (which completes only after
        // every earlier one: its X waited for them)
        d.after = phase_start > 0 ? static_cast<int>(phases.size()) - 2 : -1;
        const long long u = static_cast<long long>(d.T) * d.I;
        phases.back().U += u;
        phases.back().need += 4 * d.T;  // 4 lane quarters per tile
        uoff += u;
        toff += d.T;
    }
    *units = uoff;
    return WQ_OK;
}

// Per-phase launches (WQ_STEP_PHASES): phase p of a run becomes a launch of
// its own over the projections [first[p], first[p + 1]) of the run, so its
// table entries are rebased to the phase (units and tiles from 0, phase 0,
// no dependency: stream order replaces the device-side waits) and phase p's
// PhaseDev sits at the slot of its first projection.
void to_phase_tables(std::vector<wq::ProjDev>& host, const std::vector<wq::PhaseDev>& phases,
                     std::vector<wq::PhaseDev>& per_slot, std::vector<int>& first) {
    const int n = static_cast<int>(host.size());
    per_slot.assign(static_cast<size_t>(n), wq::PhaseDev{});
    first.assign(phases.size() + 1, n);
    for (int li = n - 1; li >= 0; --li) first[static_cast<size_t>(host[li].phase)] = li;
    for (size_t p = 0; p < phases.size(); ++p) {
        const int f = first[p];
        per_slot[static_cast<size_t>(f)] = {0, phases[p].U, phases[p].need, 0};
        const int toff0 = host[static_cast<size_t>(f)].toff;
        for (int li = f; li < first[p + 1]; ++li) {
            wq::ProjDev& d = host[static_cast<size_t>(li)];
            d.uoff -= phases[p].uoff;
            d.toff -= toff0;
            d.phase = 0;
            d.after = -1;
        }
    }
}

// Reset the run's completion counters and launch its persistent kernel.
wq_status_t launch_run(const Run& r, Tables tab, int nphase, long long units, bool waits,
                       uint8_t* ws, const FusedLayout& lay, int sms, cudaStream_t s) {
    const int n = r.end - r.begin;
    int* done = reinterpret_cast<int*>(ws + lay.done_off);
    cudaError_t e = cudaMemsetAsync(done, 0, static_cast<size_t>(n) * sizeof(int), s);
    if (e != cudaSuccess) return wq::host_cuda_fail(e);
    wq::StepArgs sa{};
    sa.proj = tab.proj + r.begin;
    sa.phase = tab.phase + r.begin;
    sa.nproj = n;
    sa.nphase = nphase;
    sa.partials = reinterpret_cast<float*>(ws + lay.partial_off);
    sa.counters = reinterpret_cast<int*>(ws + lay.counter_off);
    sa.done = done;
    sa.err = reinterpret_cast<int*>(ws);
    sa.U = units;
    sa.P = static_cast<int>(std::min<long long>(wq::gemm_sm_budget(sms), units));
    sa.pdl = 0;
    if (r.bits == 4)
        e = wq::launch_step_b4(r.group, sa, waits, r.nc, s);
    else if (r.bits == 3)
        e = wq::launch_step_b3(r.group, sa, waits, r.nc, s);
    else
        e = wq::launch_step_b2(r.group, sa, waits, r.nc, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(done, 0, static_cast<size_t>(n) * sizeof(int), s);
    return e == cudaSuccess ? WQ_OK : wq::host_cuda_fail(e);
}

// One launch per phase of a run (tables from to_phase_tables); every launch
// that follows another kernel of the step is a programmatic dependent one.
// Per-phase launches with two CTAs per tile run one cluster per tile
// (split-K sums through shared memory); see phase_grid.
#ifndef WQ_CLUSTER_FIXUP
#define WQ_CLUSTER_FIXUP 1
#endif

// Grid of a per-phase launch over T tiles of I units each (uniform_i: every
// projection of the phase has I units per tile) and U units in all: shares on
// tile boundaries where such a grid lies near the budget, and, where that
// gives each tile two CTAs of one segment each, one cluster (pair) per tile.
// Clusters of three measured slower: a cluster needs all its SMs free in one
// GPC as the previous launch drains, and triples are placed later than
// pairs (8-layer chain: pairs only 0.538 ms, pairs and triples 0.543, triples
// only 0.585, none 0.547).
struct PhaseGrid {
    int P, cluster;
};
PhaseGrid phase_grid(int T, int I, bool uniform_i, long long U, int budget, int nc, bool act) {
    PhaseGrid g{};
    const int Pa = uniform_i ? wq::aligned_grid(T, budget, true) : budget;
    g.P = static_cast<int>(std::min<long long>(Pa, U));
    const int k = T > 0 ? g.P / T : 0;
    if (WQ_CLUSTER_FIXUP && uniform_i && k == 2 && k * T == g.P && I >= k && nc == 16 && !act)
        g.cluster = k;
    return g;
}

wq_status_t launch_phases(const wq_proj_desc_t* projs, const Run& r, Tables tab,
                          const std::vector<wq::PhaseDev>& phases, const std::vector<int>& first,
                          const std::vector<wq::ProjDev>& host, uint8_t* ws,
                          const FusedLayout& lay, int sms, cudaStream_t s, bool& prev_kernel) {
    for (size_t p = 0; p < phases.size(); ++p) {
        bool act = false;
        for (int li = first[p]; li < first[p + 1]; ++li)
            act = act || projs[r.begin + li].epilogue == WQ_EPI_SWIGLU;
        wq::StepArgs sa{};
        sa.proj = tab.proj + r.begin + first[p];
        sa.phase = tab.phase + r.begin + first[p];
        sa.nproj = first[p + 1] - first[p];
        sa.nphase = 1;
        sa.partials = reinterpret_cast<float*>(ws + lay.partial_off);
        sa.counters = reinterpret_cast<int*>(ws + lay.counter_off);
        sa.done = reinterpret_cast<int*>(ws + lay.done_off);
        sa.err = reinterpret_cast<int*>(ws);
        sa.U = phases[p].U;
        // a grid whose shares fall on tile boundaries where the phase's tiles
        // all have the same number of units (measured on the layer chain:
        // q/k/v on 112 CTAs, o and down on 120, gate/up on 136 instead of 150
        // each, 3 % faster)
        int T = 0, I = -1;
        bool uniform_i = true;
        for (int li = first[p]; li < first[p + 1]; ++li) {
            const wq::ProjDev& d = host[static_cast<size_t>(li)];
            T += d.T;
            if (I < 0) I = d.I;
            else if (d.I != I) uniform_i = false;
        }
        const PhaseGrid pg =
            phase_grid(T, I, uniform_i, phases[p].U, wq::gemm_sm_budget(sms), r.nc, act);
        sa.P = pg.P;
        sa.cluster = pg.cluster;
        sa.pdl = prev_kernel ? 1 : 0;
        sa.act = act ? 1 : 0;
        cudaError_t e = cudaSuccess;
        for (int attempt = 0; attempt < 2; ++attempt) {
            if (r.bits == 4)
                e = wq::launch_step_b4(r.group, sa, false, r.nc, s);
            else if (r.bits == 3)
                e = wq::launch_step_b3(r.group, sa, false, r.nc, s);
            else
                e = wq::launch_step_b2(r.group, sa, false, r.nc, s);
            if (e == cudaSuccess || sa.cluster == 0) break;
            // clusters the device cannot place: the same grid without them
            (void)cudaGetLastError();
            sa.cluster = 0;
        }
        if (e != cudaSuccess) return wq::host_cuda_fail(e);
        prev_kernel = true;
    }
    return WQ_OK;
}

wq_status_t run_single(const wq_proj_desc_t& p, void* workspace, size_t workspace_bytes,
                       cudaStream_t s, bool pdl = false) {
    return wq::gemm_run(p.x, p.wq, p.scales, p.zeros, p.y, p.M, p.N, p.K, p.group, p.bits,
                        workspace, workspace_bytes, s, pdl, p.epilogue);
}

bool launches_kernel(const wq_proj_desc_t& p) { return p.M > 0 && p.N > 0 && p.K > 0; }

// Sequential mode: one wq_gemm per projection.  Every GEMM that directly
// follows another is a programmatic dependent launch: its CTAs start as the
// previous kernel's leave and stream their first packed words at once, and
// X is read only after the previous kernel has completed (no GEMM of a step
// writes packed words, scales or zero points).
wq_status_t run_sequential(const wq_proj_desc_t* projs, int count, void* workspace,
                           size_t workspace_bytes, cudaStream_t s) {
    bool prev_gemm = false;
    for (int i = 0; i < count; ++i) {
        if (wq_status_t st = run_single(projs[i], workspace, workspace_bytes, s, prev_gemm)) return st;
        prev_gemm = launches_kernel(projs[i]);
    }
    return WQ_OK;
}

// Upload every run's tables to `base` (table_bytes(count) of device memory),
// synchronously: graphs do this once before capturing.
wq_status_t upload_tables(const wq_proj_desc_t* projs, int count, void* base, bool phased) {
    const Tables tab = tables_at(base, count);
    std::vector<wq::ProjDev> host;
    std::vector<wq::PhaseDev> phases, per_slot;
    std::vector<int> first;
    for (const Run& r : split_runs(projs, count)) {
        if (!r.fused) continue;
        long long units = 0;
        bool waits = false;
        if (wq_status_t st = build_table(projs, r, host, phases, &units, &waits)) return st;
        if (phased) to_phase_tables(host, phases, per_slot, first);
        const std::vector<wq::PhaseDev>& ph = phased ? per_slot : phases;
        cudaError_t e = cudaMemcpy(tab.proj + r.begin, host.data(),
                                   host.size() * sizeof(wq::ProjDev), cudaMemcpyHostToDevice);
        if (e == cudaSuccess)
            e = cudaMemcpy(tab.phase + r.begin, ph.data(), ph.size() * sizeof(wq::PhaseDev),
                           cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return wq::host_cuda_fail(e);
    }
    return WQ_OK;
}

// Fused step.  With `tables` (device, uploaded by upload_tables) the launches
// read those; without, each run's tables are staged into the workspace's
// table area (slots per projection, so no run overwrites another's) first.
// stall_first_phase: test hook only (wq_internal_step_stall_probe): phase 0
// of every run gets a completion threshold no launch reaches, so the
// projections waiting for it run out their bounded waits.
wq_status_t run_fused(const wq_proj_desc_t* projs, int count, void* workspace,
                      size_t workspace_bytes, cudaStream_t s, void* tables, bool phased,
                      bool stall_first_phase = false) {
    int sms = 0;
    if (wq_status_t st = wq::host_sm_count(&sms)) return st;
    const std::vector<Run> runs = split_runs(projs, count);
    const FusedLayout lay = fused_layout(projs, count, runs, sms);
    if (!workspace || workspace_bytes < lay.bytes ||
        reinterpret_cast<uintptr_t>(workspace) % 16 != 0)
        return WQ_ERR_INVALID_ARG;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    const Tables tab = tables_at(tables ? tables : ws + lay.table_off, count);
    std::vector<wq::ProjDev> host;
    std::vector<wq::PhaseDev> phases, per_slot;
    std::vector<int> first;
    bool prev_kernel = false;  // the last operation issued by this call was one of its kernels
    for (const Run& r : runs) {
        if (!r.fused) {
            if (wq_status_t st = run_single(projs[r.begin], workspace, workspace_bytes, s)) return st;
            prev_kernel = launches_kernel(projs[r.begin]);
            continue;
        }
        long long units = 0;
        bool waits = false;
        if (wq_status_t st = build_table(projs, r, host, phases, &units, &waits)) return st;
        if (stall_first_phase && phases.size() > 1) phases[0].need = 0x7fffffff;
        if (phased) to_phase_tables(host, phases, per_slot, first);
        if (!tables) {
            // pageable sources: each copy is staged before the call returns
            const std::vector<wq::PhaseDev>& ph = phased ? per_slot : phases;
            cudaError_t e = cudaMemcpyAsync(tab.proj + r.begin, host.data(),
                                            host.size() * sizeof(wq::ProjDev),
                                            cudaMemcpyHostToDevice, s);
            if (e == cudaSuccess)
                e = cudaMemcpyAsync(tab.phase + r.begin, ph.data(),
                                    ph.size() * sizeof(wq::PhaseDev), cudaMemcpyHostToDevice, s);
            if (e != cudaSuccess) return wq::host_cuda_fail(e);
            prev_kernel = false;
        }
        if (phased) {
            if (wq_status_t st =
                    launch_phases(projs, r, tab, phases, first, host, ws, lay, sms, s, prev_kernel))
                return st;
        } else if (wq_status_t st = launch_run(r, tab, static_cast<int>(phases.size()), units,
                                               waits, ws, lay, sms, s)) {
            return st;
        }
        if (!tables) {
            // staged tables are zeroed again once the launches have read them
            cudaError_t e = cudaMemsetAsync(tab.proj + r.begin, 0,
                                            host.size() * sizeof(wq::ProjDev), s);
            if (e == cudaSuccess)
                e = cudaMemsetAsync(tab.phase + r.begin, 0,
                                    (phased ? per_slot : phases).size() * sizeof(wq::PhaseDev), s);
            if (e != cudaSuccess) return wq::host_cuda_fail(e);
            prev_kernel = false;
        }
        if (phased) continue;
        prev_kernel = false;  // a fused run's launch follows its counters' reset, not a kernel
    }
    return WQ_OK;
}

}  // namespace

struct wq_step_graph {
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    void* tables = nullptr;  // fused mode: device copy of every run's tables
};

extern "C" {

size_t wq_step_workspace_bytes(const wq_proj_desc_t* projs, int count, unsigned flags) {
    if (check_all(projs, count) != WQ_OK) return 0;
    size_t need = wq::kWsHeader;
    for (int i = 0; i < count; ++i) {
        const wq_proj_desc_t& p = projs[i];
        need = std::max(need, wq_workspace_bytes(p.M, p.N, p.K, p.group, p.bits));
    }
    if (flags & WQ_STEP_FUSED) {
        int sms = 0;
        if (wq::host_sm_count(&sms) != WQ_OK) return 0;
        need = std::max(need, fused_layout(projs, count, split_runs(projs, count), sms).bytes);
    }
    return need;
}

wq_status_t wq_step_run_ex(const wq_proj_desc_t* projs, int count, unsigned flags,
                           void* workspace, size_t workspace_bytes, void* stream) {
    if (wq_status_t st = check_all(projs, count)) return st;
    if (flags & ~(WQ_STEP_FUSED | WQ_STEP_PHASES)) return WQ_ERR_INVALID_ARG;
    if ((flags & WQ_STEP_PHASES) && !(flags & WQ_STEP_FUSED)) return WQ_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (flags & WQ_STEP_FUSED)
        return run_fused(projs, count, workspace, workspace_bytes, s, nullptr,
                         (flags & WQ_STEP_PHASES) != 0);
    return run_sequential(projs, count, workspace, workspace_bytes, s);
}

wq_status_t wq_step_run(const wq_proj_desc_t* projs, int count, void* workspace,
                        size_t workspace_bytes, void* stream) {
    return wq_step_run_ex(projs, count, 0u, workspace, workspace_bytes, stream);
}

wq_status_t wq_step_graph_create_ex(const wq_proj_desc_t* projs, int count, unsigned flags,
                                    void* workspace, size_t workspace_bytes, void* stream,
                                    wq_step_graph_t* out) {
    if (!out || !workspace || count <= 0 || !projs) return WQ_ERR_INVALID_ARG;
    *out = nullptr;
    if (wq_status_t st = check_all(projs, count)) return st;
    if (flags & ~(WQ_STEP_FUSED | WQ_STEP_PHASES)) return WQ_ERR_INVALID_ARG;
    if ((flags & WQ_STEP_PHASES) && !(flags & WQ_STEP_FUSED)) return WQ_ERR_INVALID_ARG;
    const bool phased = (flags & WQ_STEP_PHASES) != 0;
    wq_step_graph* g = new (std::nothrow) wq_step_graph;
    if (!g) return WQ_ERR_CUDA;
    wq_status_t st = WQ_OK;
    if (flags & WQ_STEP_FUSED) {
        cudaError_t e = cudaMalloc(&g->tables, table_bytes(count));
        if (e != cudaSuccess) st = wq::host_cuda_fail(e);
        if (st == WQ_OK) st = upload_tables(projs, count, g->tables, phased);
    }
    // Capture needs a non-legacy stream: use the caller's, or a private one.
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaStream_t own = nullptr;
    if (st == WQ_OK && s == nullptr) {
        if (cudaStreamCreateWithFlags(&own, cudaStreamNonBlocking) != cudaSuccess) st = WQ_ERR_CUDA;
        s = own;
    }
    if (st == WQ_OK && cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal) != cudaSuccess)
        st = WQ_ERR_CUDA;
    if (st == WQ_OK) {
        wq_status_t run;
        if (flags & WQ_STEP_FUSED) {
            run = run_fused(projs, count, workspace, workspace_bytes, s, g->tables, phased);
        } else {
            run = run_sequential(projs, count, workspace, workspace_bytes, s);
        }
        cudaError_t e = cudaStreamEndCapture(s, &g->graph);
        if (run != WQ_OK) st = run;
        else if (e != cudaSuccess) st = wq::host_cuda_fail(e);
    }
    if (st == WQ_OK) {
        cudaError_t e = cudaGraphInstantiate(&g->exec, g->graph, 0);
        if (e != cudaSuccess) st = wq::host_cuda_fail(e);
    }
    if (own) cudaStreamDestroy(own);
    if (st != WQ_OK) {
        wq_step_graph_destroy(g);
        return st;
    }
    *out = g;
    return WQ_OK;
}

wq_status_t wq_step_graph_create(const wq_proj_desc_t* projs, int count, void* workspace,
                                 size_t workspace_bytes, void* stream, wq_step_graph_t* out) {
    return wq_step_graph_create_ex(projs, count, 0u, workspace, workspace_bytes, stream, out);
}

wq_status_t wq_step_graph_launch(wq_step_graph_t g, void* stream) {
    if (!g || !g->exec) return WQ_ERR_INVALID_ARG;
    return cudaGraphLaunch(g->exec, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? WQ_OK
               : WQ_ERR_CUDA;
}

void wq_step_graph_destroy(wq_step_graph_t g) {
    if (!g) return;
    if (g->exec) cudaGraphExecDestroy(g->exec);
    if (g->graph) cudaGraphDestroy(g->graph);
    if (g->tables) cudaFree(g->tables);
    delete g;
}

// Test hook for the bounded-wait path (not part of include/wq.h): runs the
// fused step like wq_step_run_ex(WQ_STEP_FUSED) but with phase 0 of every run
// never reported complete, so every projection that waits for it gives up
// after the kernels' wait limit and the workspace's error word reads
// WQ_ERR_TIMEOUT through wq_check_workspace.  Nothing faults or traps: the
// waits end, the CTAs free their tensor memory and exit.
wq_status_t wq_internal_step_stall_probe(const wq_proj_desc_t* projs, int count, void* workspace,
                                         size_t workspace_bytes, void* stream) {
    if (wq_status_t st = check_all(projs, count)) return st;
    return run_fused(projs, count, workspace, workspace_bytes,
                     reinterpret_cast<cudaStream_t>(stream), nullptr, false, true);
}

}  // extern "C"

// Host-only view of the per-phase grid rule (used by the CPU tests).
extern "C" int wq_internal_phase_grid(int T, int I, int uniform_i, long long U, int budget, int nc,
                                      int act, int* P, int* cluster) {
    if (!P || !cluster || T <= 0 || U <= 0 || budget <= 0) return 1;
    const PhaseGrid g = phase_grid(T, I, uniform_i != 0, U, budget, nc, act != 0);
    *P = g.P;
    *cluster = g.cluster;
    return 0;
}
