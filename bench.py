#!/usr/bin/env python
"""Decode-step weight-stream benchmark for libwq.

One "step" is one decode step of a 64-layer projection stack (q, k, v, o,
fused gate/up and down of a 5120-hidden / 17408-FFN decoder, 4-bit codes,
group 128): one fused persistent launch (WQ_STEP_FUSED) honouring the layer
dependency chain, replayed as a CUDA graph, every packed weight streamed from
HBM once (11.08 GB of weights, scales and zero points, far larger than the
129 MB L2, so no flush is needed between steps).

The JSON line reports the effective weight-stream bandwidth (packed weight
bytes / step time) at the headline row count, the M sweep, the same step in
other modes (with the gate/up activation feeding down, without dependencies,
one launch per projection), per-config single-call figures, the dominant
kernel's roofline, an end-to-end figure through the C ABI with host buffers,
and the CPU oracle baseline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs an independent replica of the step on
its own GPU (the path has no exchange step); the value is the bytes all ranks
streamed divided by the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "weight-only 4-bit GEMM weight-stream GB/s (decode step, 64 layers x 6 projections)"
HEADLINE_M = 16
MAX_M = 32  # widest row stack of the sweep
L2_BYTES_FALLBACK = 129 * 2 ** 20


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--m", type=int, default=HEADLINE_M, help="headline stacked-row count")
    ap.add_argument("--no-sweep", action="store_true")
    ap.add_argument("--no-configs", action="store_true")
    ap.add_argument("--no-attention", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0, help="CPU oracle sample budget")
    ap.add_argument("--layers", type=int, default=64)
    ap.add_argument("--profile-config", default=None,
                    help="only run CALLS calls of this config (a seeded GEMM config, \"step\", \"step-phased\" or \"attention\"; for ncu captures)")
    ap.add_argument("--calls", type=int, default=3)
    ap.add_argument("--e2e-chunk-layers", default="taper",
                    help="layers per copy/compute chunk of the end-to-end step: taper, a "
                         "number, or a list adding up to the layer count")
    return ap.parse_args(argv)


# ---------------------------------------------------------------- byte model
def proj_bytes(M, N, K, group, bits):
    """Algorithmic bytes of one call: packed + scales + zeros + X + Y."""
    from weight_only_bit_wq_gb300 import wq_packed_words_per_row

    W = wq_packed_words_per_row(K, bits)
    ng = K // group
    packed = N * W * 4
    return {"packed": packed, "meta": N * ng * 3, "x": M * K * 2, "y": M * N * 4,
            "total": packed + N * ng * 3 + M * K * 2 + M * N * 4}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# ------------------------------------------------------------ distributed
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def dist_init(world, backend):
    import torch.distributed as dist

    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def reduce_max(dist, value: float, device=None) -> float:
    """Maximum of `value` over ranks (identity for one process)."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(dist, value: float, device=None) -> float:
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def whole_job_gbs(dist, bytes_this_rank: float, ms_this_rank: float, device=None):
    """(GB/s, slowest rank's ms, bytes of all ranks): every rank's bytes over the max time."""
    ms_max = reduce_max(dist, ms_this_rank, device)
    total = reduce_sum(dist, float(bytes_this_rank), device)
    return total / (ms_max * 1e-3) / 1e9, ms_max, total


# ----------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi clock / throttle samples every 200 ms while active."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        if self.path and os.path.exists(self.path):
            with open(self.path) as f:
                for line in f:
                    parts = [p.strip() for p in line.split(",")]
                    if len(parts) >= 9:
                        rows.append(parts)
            os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None

        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        mx = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons, "samples": len(rows)}


# ------------------------------------------------------------- our path
# Sources of the dominant GEMM kernel: a recorded DRAM-traffic figure is used
# only while these files are unchanged.
GEMM_SOURCES = ("wq_gemm_tc.cuh", "wq_gemm_tc_b4.cu", "wq_ptx.cuh", "wq_internal.h")


def kernel_source_digest() -> str:
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "weight_only_bit_wq_gb300", "csrc")
    for name in GEMM_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(name.encode() + f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel_key: str):
    """DRAM bytes per launch from a committed ncu summary, if it matches these sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(kernel_key)
    if not e or e.get("source_digest") != kernel_source_digest():
        return None
    return e.get("dram_bytes_per_launch")


def time_launches(launch, stream, steps, warmup, dist):
    """ms per launch: W untimed, then K timed, barrier + synchronize on both sides."""
    import torch

    for _ in range(warmup):
        launch()
    stream.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        launch()
    e1.record(stream)
    e1.synchronize()
    torch.cuda.synchronize()
    barrier(dist)
    return e0.elapsed_time(e1) / steps


class StepStack:
    """Device-resident packed weights of the whole stack plus X/Y per row count."""

    def __init__(self, layers, device):
        import torch

        import synth
        import weight_only_bit_wq_gb300 as wq

        self.wq = wq
        self.device = device
        self.projs = synth.step_projections(MAX_M, layers)
        self.weights = []
        for p in self.projs:
            q, s, z = synth.gen_weights_torch(p, device)
            self.weights.append((wq.wq_pack(q, p.bits), s, z))
            del q
        torch.cuda.synchronize()
        # activations for up to MAX_M rows per projection (row m never depends on M)
        self.xs = [synth.gen_x(p) for p in self.projs]
        self.ws = wq.new_workspace(MAX_M, 34816, 17408, 128, 4, device=device)
        self.after = layer_dependencies(len(self.projs))
        self.ws_fused = None  # sized from the first fused descriptor set (independent of M)

    def fused_workspace(self, cdescs):
        if self.ws_fused is None:
            self.ws_fused = self.wq.new_step_workspace(cdescs, self.wq.WQ_STEP_FUSED,
                                                       device=self.device)
        return self.ws_fused

    def buffers(self, M):
        """Contiguous device X/Y for all projections at row count M, plus descriptors."""
        import numpy as np
        import torch

        xs = [np.ascontiguousarray(x[:M]).reshape(-1) for x in self.xs]
        x_host = torch.from_numpy(np.concatenate(xs).view(np.int16)).pin_memory()
        x_dev = x_host.to(self.device)
        ny = sum(M * p.N for p in self.projs)
        y_dev = torch.empty(ny, dtype=torch.float32, device=self.device)
        descs, xo, yo = [], 0, 0
        for i, (p, (wqw, s, z)) in enumerate(zip(self.projs, self.weights)):
            nx = M * p.K
            descs.append(dict(x=x_dev[xo:xo + nx], wq=wqw, scales=s, zeros=z,
                              y=y_dev[yo:yo + M * p.N], M=M, N=p.N, K=p.K, group=p.group,
                              bits=p.bits, after=self.after[i]))
            xo += nx
            yo += M * p.N
        return x_host, x_dev, y_dev, descs

    def step_bytes(self, M):
        tot = {"packed": 0, "meta": 0, "x": 0, "y": 0, "total": 0}
        for p in self.projs:
            for k, v in proj_bytes(M, p.N, p.K, p.group, p.bits).items():
                tot[k] += v
        return tot


def layer_dependencies(n):
    """`after` of each projection of the step (6 per layer: q, k, v, o, gate/up, down): q, k
    and v read the layer input (the previous layer's down output), o reads attention over q, k,
    v, gate/up reads o (through the residual and norm), down reads gate/up (through the
    activation).  Only the ordering is modelled: the synthetic X buffers are not computed."""
    after = []
    for i in range(n):
        base, j = i - i % 6, i % 6
        after.append(base - 1 if j < 3 else base + j - 1)
    return after


def count_runs(descs):
    """Fused launches per step: runs of consecutive projections of one format."""
    runs, prev = 0, None
    for d in descs:
        key = (d["bits"], d["group"])
        runs += key != prev
        prev = key
    return runs


def count_phases(descs):
    """Launches per step with one launch per dependency phase: a projection that waits for a
    projection of the current phase starts a new phase (the library's rule)."""
    phases, start = 0, 0
    for i, d in enumerate(descs):
        if i == 0 or d.get("after", -1) >= start:
            phases += 1
            start = i
    return phases


def run_sweep_point(stack, M, stream, steps, warmup, dist, clocks=None, e2e=False, mode="fused"):
    """ms per step of the whole stack, as one CUDA graph: fused (one persistent launch per
    step, honouring the layer dependency chain), fused-swiglu (the same, with each gate/up
    projection's epilogue writing silu(gate) * up as the down projection's bf16 X),
    fused-independent (no dependencies) or sequential (one launch per projection)."""
    import torch

    wq = stack.wq
    x_host, x_dev, y_dev, descs = stack.buffers(M)
    if mode == "fused-independent":
        for d in descs:
            d["after"] = -1
    if mode == "fused-swiglu":
        for i, p in enumerate(stack.projs):
            if p.name.endswith("gate_up"):
                act = torch.empty((M, p.N // 2), dtype=torch.bfloat16, device=stack.device)
                descs[i]["y"] = act
                descs[i]["epilogue"] = wq.WQ_EPI_SWIGLU
                assert stack.projs[i + 1].name.endswith("down") and descs[i + 1]["K"] == p.N // 2
                descs[i + 1]["x"] = act
    cd = wq.make_descs(descs)
    stream.wait_stream(torch.cuda.current_stream())
    if mode == "sequential":
        ws, flags, launches = stack.ws, 0, len(descs)
    elif mode == "phased":
        ws, flags, launches = (stack.fused_workspace(cd), wq.WQ_STEP_FUSED | wq.WQ_STEP_PHASES,
                               count_phases(descs))
    else:
        ws, flags, launches = stack.fused_workspace(cd), wq.WQ_STEP_FUSED, count_runs(descs)
    graph = wq.StepGraph(cd, ws, stream=stream, flags=flags)
    if clocks is not None:
        with clocks:
            ms = time_launches(lambda: graph.launch(stream=stream), stream, steps, warmup, dist)
    else:
        ms = time_launches(lambda: graph.launch(stream=stream), stream, steps, warmup, dist)
    out = {"M": M, "ms_per_step": ms, "launches_per_step": launches, "projections": len(descs)}
    if e2e:
        y_host = torch.empty(y_dev.numel(), dtype=torch.float32).pin_memory()

        def e2e_step():
            x_dev.copy_(x_host, non_blocking=True)
            graph.launch(stream=stream)
            y_host.copy_(y_dev, non_blocking=True)

        with torch.cuda.stream(stream):
            ms_e2e = time_launches(e2e_step, stream, max(3, steps // 2), 2, dist)
        out["e2e_ms"] = ms_e2e
        out["h2d_bytes"] = x_host.numel() * 2
        out["d2h_bytes"] = y_host.numel() * 4
    wq.wq_check_workspace(ws, stream=stream)
    graph.close()
    return out


def e2e_chunks(layers, spec):
    """Layers per chunk of the end-to-end step: "taper" (chunks of 8 layers with the first
    and last split into 2 + 6 and 6 + 2, so that only a small first copy in and a small
    last copy out are exposed; measured 4.54 against 4.64 ms for even chunks of 8 on the
    64-layer step), `spec` layers each ("8"), or an explicit list ("2,6,8,...") that must
    add up to the layer count."""
    if spec == "taper":
        if layers >= 16 and (layers - 16) % 8 == 0:
            return [2, 6] + [8] * ((layers - 16) // 8) + [6, 2]
        spec = "8"
    parts = [int(v) for v in str(spec).split(",") if v.strip()]
    if len(parts) == 1:
        n = parts[0]
        return [min(n, layers - i) for i in range(0, layers, n)]
    if sum(parts) != layers or min(parts) < 1:
        raise ValueError(f"chunk list {spec} does not cover {layers} layers")
    return parts


def run_e2e_pipelined(stack, M, stream, steps, warmup, dist, mode, chunk_spec="taper"):
    """ms per step end to end through the C ABI: every step copies all X from pinned host
    memory and reads all Y back, chunk by chunk (e2e_chunks) on two copy streams, so that
    a chunk's copies overlap the step graphs of the other chunks.  Each chunk is its own
    step graph in the headline's mode; stream order carries the layer chain from one chunk
    to the next."""
    import torch

    wq = stack.wq
    x_host, x_dev, y_dev, descs = stack.buffers(M)
    y_host = torch.empty(y_dev.numel(), dtype=torch.float32).pin_memory()
    flags = {"fused": wq.WQ_STEP_FUSED, "phased": wq.WQ_STEP_FUSED | wq.WQ_STEP_PHASES,
             "sequential": 0}[mode]
    sizes = e2e_chunks(len(descs) // 6, chunk_spec)
    stream.wait_stream(torch.cuda.current_stream())
    chunks, xo, yo, c0 = [], 0, 0, 0
    for layers in sizes:
        per = 6 * layers
        sub = [dict(d) for d in descs[c0:c0 + per]]
        for d in sub:  # dependencies on earlier chunks are met by stream order
            d["after"] = d["after"] - c0 if d["after"] >= c0 else -1
        nx = sum(d["M"] * d["K"] for d in sub)
        ny = sum(d["M"] * d["N"] for d in sub)
        cd = wq.make_descs(sub)
        ws = stack.ws if mode == "sequential" else stack.fused_workspace(cd)
        chunks.append((wq.StepGraph(cd, ws, stream=stream, flags=flags), xo, nx, yo, ny, ws))
        xo += nx
        yo += ny
        c0 += per
    h2d, d2h = torch.cuda.Stream(stack.device), torch.cuda.Stream(stack.device)
    ev_x = [torch.cuda.Event() for _ in chunks]
    ev_c = [torch.cuda.Event() for _ in chunks]
    ev_y = [torch.cuda.Event() for _ in chunks]

    def step():
        h2d.wait_stream(stream)  # after the step's start (and the previous step's graphs)
        for i, (_, xo, nx, _, _, _) in enumerate(chunks):
            with torch.cuda.stream(h2d):
                x_dev[xo:xo + nx].copy_(x_host[xo:xo + nx], non_blocking=True)
            ev_x[i].record(h2d)
        for i, (g, _, _, yo, ny, _) in enumerate(chunks):
            stream.wait_event(ev_x[i])
            g.launch(stream=stream)
            ev_c[i].record(stream)
            d2h.wait_event(ev_c[i])
            with torch.cuda.stream(d2h):
                y_host[yo:yo + ny].copy_(y_dev[yo:yo + ny], non_blocking=True)
            ev_y[i].record(d2h)
        stream.wait_event(ev_y[-1])  # the step ends when its last Y is on the host

    ms = time_launches(step, stream, steps, warmup, dist)
    torch.cuda.synchronize()
    for g, *_, ws in chunks:
        wq.wq_check_workspace(ws, stream=stream)
        g.close()
    return {"e2e_ms": ms, "h2d_bytes": x_host.numel() * 2, "d2h_bytes": y_host.numel() * 4,
            "chunks": len(chunks), "chunk_layers": sizes}


def run_dominant(stack, M, stream, steps, warmup, dist):
    """ms per launch of the dominant projection (fused gate/up), 64 launches per graph."""
    import torch

    wq = stack.wq
    _, _, _, descs = stack.buffers(M)
    sel = [dict(d, after=-1) for d, p in zip(descs, stack.projs) if p.name.endswith("gate_up")]
    graph = wq.StepGraph(wq.make_descs(sel), stack.ws, stream=stream)
    stream.wait_stream(torch.cuda.current_stream())
    ms = time_launches(lambda: graph.launch(stream=stream), stream, max(3, steps // 2), 2, dist)
    graph.close()
    d = sel[0]
    return ms / len(sel), proj_bytes(M, d["N"], d["K"], d["group"], d["bits"]), len(sel)


CONFIG_MIN_CALLS = 200  # calls timed per config


def graph_call_times(launch, stream, launches, warmup, calls_per_launch):
    """µs per call of each of `launches` timed graph launches (CUDA events between
    consecutive launches on the launching stream)."""
    import torch

    for _ in range(warmup):
        launch()
    stream.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(launches + 1)]
    ev[0].record(stream)
    for i in range(launches):
        launch()
        ev[i + 1].record(stream)
    ev[-1].synchronize()
    return [ev[i].elapsed_time(ev[i + 1]) * 1e3 / calls_per_launch for i in range(launches)]


def percentiles(samples):
    """Median, 10th and 90th percentile (linear interpolation)."""
    import numpy as np

    a = np.asarray(samples, dtype=np.float64)
    return float(np.median(a)), float(np.percentile(a, 10)), float(np.percentile(a, 90))


def run_configs(device, stream, peak, l2_bytes):
    """Single-call figures for the seeded configs, rotating weight copies past L2."""
    import numpy as np
    import torch

    import synth
    import weight_only_bit_wq_gb300 as wq

    out = {}
    for name, p in synth.CONFIGS.items():
        b = proj_bytes(p.M, p.N, p.K, p.group, p.bits)
        reps = int(min(1024, max(4, -(-4 * l2_bytes // b["total"]))))
        q, s, z = synth.gen_weights_torch(p, device)
        try:
            w0 = wq.wq_pack(q, p.bits)
        finally:
            del q
        x = torch.from_numpy(synth.gen_x(p).view(np.int16)).to(device)
        y = torch.empty((p.M, p.N), dtype=torch.float32, device=device)
        copies = [(w0, s, z)] + [(w0.clone(), s.clone(), z.clone()) for _ in range(reps - 1)]
        ws = wq.new_workspace(p.M, p.N, p.K, p.group, p.bits, device=device)
        try:
            wq.wq_gemm(x, w0, s, z, p.N, p.group, p.bits, out=y, workspace=ws)
        except wq.WQError as e:
            out[name] = {"status": str(e)}
            continue
        descs = wq.make_descs([dict(x=x, wq=c[0], scales=c[1], zeros=c[2], y=y, M=p.M, N=p.N,
                                    K=p.K, group=p.group, bits=p.bits) for c in copies])
        stream.wait_stream(torch.cuda.current_stream())
        g = wq.StepGraph(descs, ws, stream=stream)
        launches = max(5, -(-CONFIG_MIN_CALLS // reps))
        per_call = graph_call_times(lambda: g.launch(stream=stream), stream, launches, 2, reps)
        g.close()
        us, p10, p90 = percentiles(per_call)
        out[name] = {"M": p.M, "N": p.N, "K": p.K, "bits": p.bits, "group": p.group,
                     "us_per_call": round(us, 3), "us_p10": round(p10, 3), "us_p90": round(p90, 3),
                     "weight_gbs": round(b["packed"] / (us * 1e-6) / 1e9, 1),
                     "roofline_frac": round(b["total"] / (us * 1e-6) / 1e9 / peak, 4),
                     "bytes_per_call": b["total"], "rotated_copies": reps,
                     "timed_calls": launches * reps}
        del copies, descs
        torch.cuda.empty_cache()
    return out


# Decode attention over the paged q8_0 pool: four agents, each with 32768
# positions of its own sequence (a 4096-token system prompt stored once and
# shared), three query rows per agent (one token, two drafts), 40 query heads
# over 8 key/value heads of 128 dims, 64-token pages: 118,784 tokens in the pool.
ATTN_CASE = dict(seq_lens=(32768,) * 4, rows_per_seq=3, Hq=40, Hkv=8, D=128, T=64, seed=31,
                 shared_prefix=4096)


def attention_bytes(p):
    """Algorithmic bytes of one call: every sequence reads its positions' K and V
    codes and scales once (the shared prefix once per sequence), plus q and out."""
    kv = sum(p.seq_lens) * p.Hkv * 2 * (p.D + 2 * (p.D // 32))
    rows = len(p.seq_lens) * p.rows_per_seq
    return kv + rows * p.Hq * p.D * (2 + 4)


def run_attention(device, stream, peak, steps, warmup):
    """µs per call of wq_paged_attention (tensor-core kernel) and, for context,
    of the CUDA-core kernel, on the pool above (every call reads more than L2)."""
    import ctypes

    import torch

    import synth
    import weight_only_bit_wq_gb300 as wq

    p = synth.PagedAttention("bench", **ATTN_CASE)
    t = synth.gen_paged_attention_torch(p, device)
    rows, Hq, D = t["q"].shape
    pages, Hkv, T, _ = t["kc"].shape
    B, max_pages = t["page_table"].shape
    msl = max(p.seq_lens)
    out = torch.empty((rows, Hq, D), dtype=torch.float32, device=device)
    n = int(wq._lib().wq_paged_attention_workspace_bytes(rows, Hq, Hkv, B, msl))
    ws = torch.zeros(max(n, 256), dtype=torch.uint8, device=device)
    lib = wq._lib()
    cc = lib.wq_internal_paged_attention_cuda_cores
    cc.argtypes = lib.wq_paged_attention.argtypes
    cc.restype = ctypes.c_int
    ptr = lambda x: ctypes.c_void_p(x.data_ptr())
    args = (ptr(t["q"]), ptr(t["kc"]), ptr(t["kd"]), ptr(t["vc"]), ptr(t["vd"]),
            ptr(t["page_table"]), max_pages, ptr(t["seq_len"]), B, ptr(t["row_seq"]),
            ptr(t["row_pos"]), rows, msl, Hq, Hkv, D, T, pages, ptr(out), ptr(ws), ws.numel(),
            ctypes.c_void_p(stream.cuda_stream))
    stream.wait_stream(torch.cuda.current_stream())
    nbytes = attention_bytes(p)
    res = {"workload": "decode attention over a paged q8_0 pool: 4 sequences x 32768 positions "
                       "(4096-token prefix stored once), 3 query rows each, 40 query / 8 kv heads "
                       "of 128, 64-token pages", "bytes_per_call": nbytes}
    for name, fn in (("tensor_cores", lib.wq_paged_attention), ("cuda_cores", cc)):
        def launch():
            st = fn(*args)
            if st != 0:
                raise RuntimeError(f"{name}: status {st}")
        ms = time_launches(launch, stream, steps, warmup, None)
        us = ms * 1e3
        res[name] = {"us_per_call": round(us, 2),
                     "achieved_gbs": round(nbytes / (us * 1e-6) / 1e9, 1),
                     "frac": round(nbytes / (us * 1e-6) / 1e9 / peak, 4)}
    torch.cuda.synchronize()
    word = int(ws[:4].view(torch.int32).item())
    if word != 0:
        raise RuntimeError(f"attention error word {word}")
    del t, out, ws
    torch.cuda.empty_cache()
    return res


# ------------------------------------------------------------ CPU oracle
def cpu_sample(M, row_budget):
    """A bounded sample of the decode step: the first rows of layer 0's gate/up and down."""
    import numpy as np
    import torch

    import synth

    projs = synth.step_projections(M, 1)
    picks = [(projs[4], row_budget), (projs[5], max(1, row_budget // 4))]
    sample = []
    for p, rows in picks:
        import dataclasses

        ps = dataclasses.replace(p, N=rows)  # rows 0..rows-1 of the same projection
        q, s, z = synth.gen_weights_torch(ps, "cpu", row_chunk=256)
        sample.append((ps, q.numpy(), s.numpy().view(np.uint16), z.numpy(), synth.gen_x(ps)))
    return sample


def time_oracle(sample, seconds, passes=None, threads=0):
    """Time full oracle passes (pack + fp64 GEMM) over the sample on all host cores
    (or on `threads` of them)."""
    import oracle

    packed = sum(ps.N * oracle.words_per_row(ps.K, ps.bits) * 4 for ps, *_ in sample)
    done, t0 = 0, time.perf_counter()
    times = []
    while True:
        t1 = time.perf_counter()
        for ps, q, s, z, x in sample:
            oracle.gemm_f64(x, oracle.pack(q, ps.bits), s, z, ps.K, ps.group, ps.bits, threads)
        times.append(time.perf_counter() - t1)
        done += 1
        if passes is not None and done >= passes:
            break
        if passes is None and time.perf_counter() - t0 >= seconds:
            break
    return packed, times, oracle.max_threads(threads)


def cpu_model():
    """The host CPU's model from /proc/cpuinfo (x86 model name, or Arm implementer and part)."""
    import re

    try:
        with open("/proc/cpuinfo") as f:
            text = f.read()
    except OSError:
        return None
    m = re.search(r"^model name\s*:\s*(.+)$", text, re.M)
    if m:
        return m.group(1).strip()
    imp = re.search(r"^CPU implementer\s*:\s*(\S+)$", text, re.M)
    part = re.search(r"^CPU part\s*:\s*(\S+)$", text, re.M)
    if imp and part:
        return f"Arm implementer {imp.group(1)}, part {part.group(1)}"
    return None


def cpu_baseline(M, seconds):
    import oracle

    sample = cpu_sample(M, 2048)
    cores = oracle.max_threads()
    time_oracle(sample, 0, passes=1, threads=cores)  # warm-up
    packed, times, cores = time_oracle(sample, seconds, threads=cores)
    gbs = packed * len(times) / sum(times) / 1e9
    desc = (f"layer-0 gate/up rows 0..{sample[0][0].N - 1} and down rows 0..{sample[1][0].N - 1} "
            f"at M={M} ({packed / 1e6:.1f} MB packed per pass, {len(times)} passes, "
            f"pack + fp64 GEMM)")
    out = {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
           "sample": desc, "cpu_model": cpu_model()}
    # the same sample on one core, for the scaling of the oracle itself (context only)
    try:
        _, t1, _ = time_oracle(sample, seconds / 4, threads=1)
        out["single_thread_value"] = round(packed * len(t1) / sum(t1) / 1e9, 4)
    except Exception as e:  # context only: never fail the benchmark over it
        out["single_thread_value"] = None
        out["single_thread_error"] = str(e)[:200]
    finally:
        time_oracle(sample, 0, passes=1, threads=cores)  # leave the oracle on all cores
    return out


# ------------------------------------------------------------------- main
WORKLOAD = ("decode-step projection stack: 64 layers x {q 5120->5120, k 5120->1024, v 5120->1024, "
            "o 5120->5120, gate/up 5120->34816, down 17408->5120}, 4-bit codes, group 128, "
            "bf16 activations, fp32 output")
DATA = ("synthetic, seeded SplitMix64: codes U{0..15}, bf16 scales U(0.005,0.02), zero points "
        "U{0..15}, activations bf16 N(0,1)")


HEAD_MODES = ("fused", "phased", "sequential")  # the step modes that honour the layer chain
CHAIN = ("q, k, v after the previous down; o after q, k, v; gate/up after o; down after "
         "gate/up")


def choose_head(ms_by_mode):
    """The headline mode: the fastest of the modes that honour the layer chain
    (a tie keeps the first listed)."""
    best = None
    for m in HEAD_MODES:
        if m in ms_by_mode and (best is None or ms_by_mode[m] < ms_by_mode[best]):
            best = m
    return best


def _config(M, layers, world, mode="fused", launches=1):
    how = {"fused": "one persistent launch per step (WQ_STEP_FUSED) honouring the layer "
                    "dependency chain on device-side counters: " + CHAIN,
           "phased": "one persistent launch per dependency phase (WQ_STEP_FUSED | "
                     "WQ_STEP_PHASES: q, k and v in one launch, then o, gate/up, down), as one "
                     "CUDA graph of programmatic dependent launches (stream order honours the "
                     "layer dependency chain: " + CHAIN + ")",
           "sequential": "one wq_gemm launch per projection on one stream, as one CUDA graph "
                         "(stream order honours the layer dependency chain: " + CHAIN + ")"}[mode]
    return {"workload": WORKLOAD, "M": M, "layers": layers, "launches_per_step": launches,
            "mode": how, "headline": f"the fastest of {', '.join(HEAD_MODES)}: {mode}",
            "l2": "inputs larger than L2 (every step streams all packed weights; no flush)",
            "parallelism": f"{world} independent replicas" if world > 1 else "one GPU"}


def _gpu_id(device):
    import torch

    try:
        return "GPU-" + str(torch.cuda.get_device_properties(device).uuid)
    except Exception:
        return str(device.index or 0)


def main_ours(args):
    import torch

    rank, world, local = dist_env()
    dist = dist_init(world, "nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import __graft_entry__

    if rank == 0:
        __graft_entry__.build()
    barrier(dist)
    if rank != 0:
        __graft_entry__.build()
    peak, peak_kind = load_peaks()
    l2 = getattr(torch.cuda.get_device_properties(device), "L2_cache_size", L2_BYTES_FALLBACK)
    stream = torch.cuda.Stream(device)
    import synth

    stack = StepStack(args.layers, device)
    clocks = ClockSampler(_gpu_id(device)) if rank == 0 else None

    # the headline: the fastest of the modes that honour the layer chain
    heads, head_ms = {}, {}
    for mode in HEAD_MODES:
        heads[mode] = run_sweep_point(stack, args.m, stream, args.steps, args.warmup, dist,
                                      clocks=clocks, e2e=True, mode=mode)
        head_ms[mode] = reduce_max(dist, heads[mode]["ms_per_step"], device)
    head_mode = choose_head(head_ms)
    head = heads[head_mode]
    sb = stack.step_bytes(args.m)
    value, ms_max, packed_all = whole_job_gbs(dist, sb["packed"], head["ms_per_step"], device)
    serial_e2e_max = reduce_max(dist, head["e2e_ms"], device)
    pipe = run_e2e_pipelined(stack, args.m, stream, max(3, args.steps // 2), 2, dist, head_mode,
                             chunk_spec=args.e2e_chunk_layers)
    e2e_max = reduce_max(dist, pipe["e2e_ms"], device)

    sweep = []
    if not args.no_sweep:
        for M in synth.STEP_M_SWEEP:
            r = run_sweep_point(stack, M, stream, max(3, args.steps // 4), 2, dist, mode=head_mode)
            b = stack.step_bytes(M)
            ms = reduce_max(dist, r["ms_per_step"], device)
            sweep.append({"M": M, "ms_per_step": round(ms, 4),
                          "us_per_projection": round(ms * 1e3 / r["projections"], 3),
                          "weight_gbs": round(b["packed"] / (ms * 1e-3) / 1e9, 1),
                          "roofline_frac": round(b["total"] / (ms * 1e-3) / 1e9 / peak, 4)})
    # both chain modes, and the fused step with the activation epilogue or
    # without dependencies
    modes = {m: {"ms_per_step": round(head_ms[m], 4),
                 "launches_per_step": heads[m]["launches_per_step"],
                 "weight_gbs": round(sb["packed"] / (head_ms[m] * 1e-3) / 1e9, 1)}
             for m in HEAD_MODES}
    for mode in ("fused-swiglu", "fused-independent"):
        r = run_sweep_point(stack, args.m, stream, max(3, args.steps // 4), 2, dist, mode=mode)
        ms = reduce_max(dist, r["ms_per_step"], device)
        modes[mode] = {"ms_per_step": round(ms, 4), "launches_per_step": r["launches_per_step"],
                       "weight_gbs": round(sb["packed"] / (ms * 1e-3) / 1e9, 1)}

    # dominant kernel: the fused step kernel (one launch per step), or the
    # single-projection kernel (one launch per projection)
    n_launch = head["launches_per_step"]
    if head_mode == "fused":
        kernel_key = f"gemm_tc_kernel<4,128,fused> step 64 layers M={args.m}"
        timing = "CUDA events around the step graph (one fused launch per step)"
    elif head_mode == "phased":
        kernel_key = f"gemm_tc_kernel<4,128,fused> step 64 layers, one launch per phase, M={args.m}"
        timing = (f"CUDA events around the step graph of {n_launch} launches; per launch: the "
                  f"step's bytes and time over {n_launch}")
    else:
        kernel_key = f"gemm_tc_kernel<4,128> step 64 layers, one launch per projection, M={args.m}"
        timing = (f"CUDA events around the step graph of {n_launch} launches; per launch: the "
                  f"step's bytes and time over {n_launch}")
    achieved = sb["total"] / (ms_max * 1e-3) / 1e9
    # the largest projection alone, one launch per call (context for the fused figure)
    dom_ms, dom_b, dom_n = run_dominant(stack, args.m, stream, args.steps, args.warmup, dist)
    dom_ms = reduce_max(dist, dom_ms, device)
    single = {"kernel": f"gemm_tc_kernel<4,128> N=34816 K=5120 M={args.m}",
              "launch_us": round(dom_ms * 1e3, 3), "bytes_per_launch": dom_b["total"],
              "achieved_gbs": round(dom_b["total"] / (dom_ms * 1e-3) / 1e9, 1),
              "frac": round(dom_b["total"] / (dom_ms * 1e-3) / 1e9 / peak, 4),
              "timing": f"CUDA events around a graph of {dom_n} launches (one per layer)"}

    configs = None
    if rank == 0 and not args.no_configs:
        configs = run_configs(device, stream, peak, l2)
    attention = None
    if rank == 0 and not args.no_attention:
        attention = run_attention(device, stream, peak, max(3, args.steps // 2), 3)
    barrier(dist)
    cpu = cpu_baseline(args.m, args.cpu_seconds) if (rank == 0 and world == 1) else None
    clock_info = clocks.summary() if clocks is not None else None

    if rank == 0:
        line = {
            "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_max, 4),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": DATA, "config": _config(args.m, args.layers, world, head_mode, n_launch),
            "us_per_projection": round(ms_max * 1e3 / head["projections"], 3),
            "step_bytes": sb["total"], "step_packed_bytes": sb["packed"],
            "roofline_frac_step": round(sb["total"] / (ms_max * 1e-3) / 1e9 / peak, 4),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                         "unit": "GB/s", "frac": round(achieved / peak, 4),
                         "traffic": recorded_traffic(kernel_key), "kernel": kernel_key,
                         "bytes_per_launch": round(sb["total"] / n_launch),
                         "launch_us": round(ms_max * 1e3 / n_launch, 3),
                         "timing": timing,
                         "peak_source": f"{peak_kind} hbm_gbs (MEASURED_PEAKS.json)"},
            "step_modes": modes, "single_launch": single, "attention": attention,
            "cpu_baseline": cpu,
            "e2e": {"value": round(packed_all / (e2e_max * 1e-3) / 1e9, 1), "unit": "GB/s",
                    "h2d_bytes_per_step": pipe["h2d_bytes"], "d2h_bytes_per_step": pipe["d2h_bytes"],
                    "ms_per_step": round(e2e_max, 4),
                    "how": (f"every step: all X from pinned host memory to the device and all Y "
                            f"back, in {pipe['chunks']} chunks of {pipe['chunk_layers']} layers on two "
                            f"copy streams overlapping the other chunks' step graphs (the headline's "
                            f"mode, launched through the C ABI); the step ends when its last Y is "
                            f"on the host"),
                    "serial_ms_per_step": round(serial_e2e_max, 4),
                    "serial_how": "all X to the device, then the whole step graph, then all Y back"},
            "gpu_launches": head["launches_per_step"] * args.steps,
            "clocks": clock_info, "sweep": sweep, "configs": configs,
        }
        print(json.dumps(line), flush=True)
    barrier(dist)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main_reference(args):
    rank, world, _ = dist_env()
    if world > 1 and rank != 0:
        return 0
    sys.path.insert(0, ROOT)
    import oracle

    oracle.build()
    M = args.m
    # size the sample so that K + W passes take about a minute in total
    probe = cpu_sample(M, 256)
    _, t_probe, cores = time_oracle(probe, 0, passes=2)
    per_row = min(t_probe) / 256
    target = max(0.2, min(3.0, 60.0 / max(1, args.steps + args.warmup)))
    rows = int(max(64, min(16384, target / max(per_row, 1e-9))))
    sample = cpu_sample(M, rows)
    time_oracle(sample, 0, passes=max(1, args.warmup))
    packed, times, cores = time_oracle(sample, 0, passes=max(1, args.steps))
    ms = 1e3 * sum(times) / len(times)
    value = packed / (ms * 1e-3) / 1e9
    desc = (f"layer-0 gate/up rows 0..{rows - 1} and down rows 0..{max(1, rows // 4) - 1} at M={M} "
            f"({packed / 1e6:.1f} MB packed per step, pack + fp64 GEMM)")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": DATA,
            "config": _config(M, args.layers, world),
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                             "kind": "oracle", "sample": desc},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
            "gpu_launches": 0}
    print(json.dumps(line), flush=True)
    return 0


def main_profile(args):
    """A few plain calls of one seeded config on cuda:0 (small enough for ncu); config "step"
    runs the fused decode step of --layers layers instead."""
    import numpy as np
    import torch

    import __graft_entry__
    import synth
    import weight_only_bit_wq_gb300 as wq

    __graft_entry__.build()
    device = torch.device("cuda", 0)
    if args.profile_config == "attention":
        pa = synth.PagedAttention("bench", **ATTN_CASE)
        t = synth.gen_paged_attention_torch(pa, device)
        for _ in range(args.calls):
            out = wq.wq_paged_attention(t["q"], t["kc"], t["kd"], t["vc"], t["vd"],
                                        t["page_table"], t["seq_len"], t["row_seq"], t["row_pos"],
                                        max(pa.seq_lens))
        torch.cuda.synchronize()
        print(json.dumps({"profile_config": "attention", "calls": args.calls,
                          "bytes_per_call": attention_bytes(pa),
                          "max_abs_out": float(out.abs().max())}))
        return 0
    if args.profile_config in ("step", "step-phased"):
        stack = StepStack(args.layers, device)
        _, _, _, descs = stack.buffers(args.m)
        cd = wq.make_descs(descs)
        ws = stack.fused_workspace(cd)
        flags = wq.WQ_STEP_FUSED | (wq.WQ_STEP_PHASES if args.profile_config == "step-phased" else 0)
        for _ in range(args.calls):
            wq.wq_step_run(cd, ws, flags=flags)
        torch.cuda.synchronize()
        wq.wq_check_workspace(ws)
        b = stack.step_bytes(args.m)
        print(json.dumps({"profile_config": args.profile_config, "layers": args.layers, "M": args.m,
                          "calls": args.calls, "bytes_per_call": b["total"]}))
        return 0
    p = synth.CONFIGS[args.profile_config]
    if args.m != HEADLINE_M:
        p = p.with_m(args.m) if p.x_row_seeds is None or args.m <= len(p.x_row_seeds) else p
    q, s, z = synth.gen_weights_torch(p, device)
    wqw = wq.wq_pack(q, p.bits)
    del q
    x = torch.from_numpy(synth.gen_x(p).view(np.int16)).to(device)
    ws = wq.new_workspace(p.M, p.N, p.K, p.group, p.bits, device=device)
    y = torch.empty((p.M, p.N), dtype=torch.float32, device=device)
    for _ in range(args.calls):
        wq.wq_gemm(x, wqw, s, z, p.N, p.group, p.bits, out=y, workspace=ws)
    torch.cuda.synchronize()
    wq.wq_check_workspace(ws)
    print(json.dumps({"profile_config": p.name, "M": p.M, "N": p.N, "K": p.K, "calls": args.calls}))
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.profile_config:
        return main_profile(args)
    if args.impl == "reference":
        return main_reference(args)
    return main_ours(args)


if __name__ == "__main__":
    sys.exit(main())
