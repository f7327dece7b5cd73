"""Seeded synthetic inputs for the weight-only low-bit skinny GEMM.

This module is shared by the CPU oracle tests and by the GPU path's tests and
benchmark.  It holds NO arithmetic of the method itself (no packing, no
dequantisation, no contraction): it only draws the integer codes q, the
per-group bf16 scales s, the per-group integer zero points z and the bf16
activations x, with the shapes and value distributions of the workloads below.

Generator
---------
One counter-based generator, SplitMix64 (Steele, Lea, Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014): the i-th 64-bit draw of a stream
with key ``key`` is ``mix(key + (i + 1) * 0x9E3779B97F4A7C15)`` with the
SplitMix64 finaliser ``mix``.  Each tensor element owns a fixed counter
(element (n, k) of a row-major [N][K] tensor uses counter ``n*K + k``), so any
subset of rows can be regenerated on its own: the oracle recomputes sampled
rows of a full-size workload without generating the rest.

Value recipes
-------------
* uniform integers on [lo, hi]: ``lo + ((u >> 32) * (hi - lo + 1)) >> 32``
  (multiply-shift, Lemire 2019).
* uniform reals on [a, b): ``u24 = u >> 40`` as float32 times 2**-24, then
  ``a + (b - a) * u24`` in float32, then rounded once to bf16 by torch's
  float32 -> bfloat16 cast (round to nearest even).
* standard normals: Box-Muller (cosine branch) in float64 from two draws
  (counters 2i and 2i+1), rounded to float32, optionally scaled in float32
  (outlier channels), then rounded once to bf16 by torch's cast.

bf16 tensors are returned as their uint16 bit patterns so both sides see the
same bytes.  Integer draws and uniform reals can also be produced on a CUDA
device with torch integer/float32 ops that give the same bits (used to build
multi-gigabyte weight stacks for the benchmark without a host round-trip);
normals are always drawn on the host.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Sequence

import numpy as np

_GAMMA = 0x9E3779B97F4A7C15
_C1 = 0xBF58476D1CE4E5B9
_C2 = 0x94D049BB133111EB
_MASK64 = (1 << 64) - 1

# Stream identifiers: one independent SplitMix64 stream per tensor kind.
STREAMS = {"q": 1, "s": 2, "z": 3, "x": 4, "outlier": 5, "kv_code": 6, "kv_scale": 7,
           "attn_q": 8, "page": 9}


def _mix_int(z: int) -> int:
    z &= _MASK64
    z = ((z ^ (z >> 30)) * _C1) & _MASK64
    z = ((z ^ (z >> 27)) * _C2) & _MASK64
    return z ^ (z >> 31)


def stream_key(seed: int, stream: str, index: int = 0) -> int:
    """64-bit key of stream ``stream`` (and sub-stream ``index``) for ``seed``."""
    raw = (seed * 0x100000001B3 + STREAMS[stream] * 0x10001 + index * 0x9E37) & _MASK64
    return _mix_int(_mix_int(raw) ^ 0xD1B54A32D192ED03)


# ---------------------------------------------------------------- numpy side
def _mix_np(z: np.ndarray) -> np.ndarray:
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_C1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_C2)
    return z ^ (z >> np.uint64(31))


def draws_u64(key: int, counters: np.ndarray) -> np.ndarray:
    """SplitMix64 draws for the given counters (uint64 array, any shape)."""
    c = counters.astype(np.uint64, copy=False)
    with np.errstate(over="ignore"):
        return _mix_np(np.uint64(key) + (c + np.uint64(1)) * np.uint64(_GAMMA))


def _uniform_int(u: np.ndarray, lo: int, hi: int) -> np.ndarray:
    span = np.uint64(hi - lo + 1)
    with np.errstate(over="ignore"):
        return (np.uint64(lo) + (((u >> np.uint64(32)) * span) >> np.uint64(32))).astype(np.int64)


def _uniform_f32(u: np.ndarray, a: float, b: float) -> np.ndarray:
    u24 = (u >> np.uint64(40)).astype(np.float32) * np.float32(2.0 ** -24)
    a32, b32 = np.float32(a), np.float32(b)
    return (a32 + (b32 - a32) * u24).astype(np.float32)


def _normal_f32(key: int, counters: np.ndarray) -> np.ndarray:
    c = counters.astype(np.uint64, copy=False)
    ua = draws_u64(key, c * np.uint64(2))
    ub = draws_u64(key, c * np.uint64(2) + np.uint64(1))
    u1 = ((ua >> np.uint64(11)).astype(np.float64) + 0.5) * 2.0 ** -53
    u2 = (ub >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    return (np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * math.pi * u2)).astype(np.float32)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 with torch's cast (nearest even); return uint16 bits."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


# ------------------------------------------------------------ workload specs
@dataclasses.dataclass(frozen=True)
class Projection:
    """One weight-only quantised projection Y[M,N] = X[M,K] . dequant(Wq)[N,K]^T."""

    name: str
    M: int
    N: int
    K: int
    bits: int
    group: int
    seed: int
    s_range: tuple = (0.005, 0.02)
    z_range: Optional[tuple] = None  # default: [0, 2**bits - 1]
    outlier_frac: float = 0.0  # fraction of K channels scaled by outlier_scale
    outlier_scale: float = 20.0
    x_row_seeds: Optional[tuple] = None  # one seed per x row (default: all rows use ``seed``)
    index: int = 0  # sub-stream index (distinct projections of one model)

    @property
    def ng(self) -> int:
        return self.K // self.group

    @property
    def q_range(self) -> tuple:
        return (0, (1 << self.bits) - 1)

    @property
    def zr(self) -> tuple:
        return self.z_range if self.z_range is not None else (0, (1 << self.bits) - 1)

    def with_m(self, M: int) -> "Projection":
        seeds = self.x_row_seeds[:M] if self.x_row_seeds is not None else None
        return dataclasses.replace(self, M=M, x_row_seeds=seeds)


def _cfg(name, M, K, N, bits, group, seed, **kw) -> Projection:
    return Projection(name=name, M=M, N=N, K=K, bits=bits, group=group, seed=seed, **kw)


# The seeded workloads.  Shapes are those of a 64-layer, 5120-hidden,
# 17408-FFN decoder served to several agents at once (each agent's next token
# plus its draft tokens stacked as rows of X).
CONFIGS: Dict[str, Projection] = {
    # small single-row case
    "C1": _cfg("C1", 1, 1024, 1024, 4, 128, 0),
    # 4 agents x 1 row, attention-output projection; x row r drawn with seed 1 + r
    "C2": _cfg("C2", 4, 5120, 5120, 4, 128, 1, x_row_seeds=(1, 2, 3, 4)),
    # 4 agents x (1 token + 2 drafts) = 12 rows, fused gate/up, 1% outlier channels x20
    "C3": _cfg("C3", 12, 5120, 34816, 4, 128, 5, outlier_frac=0.01),
    # down projection at three bit widths
    "C4a": _cfg("C4a", 8, 17408, 5120, 4, 128, 6, s_range=(0.005, 0.04)),
    "C4b": _cfg("C4b", 8, 17408, 5120, 3, 128, 6, s_range=(0.005, 0.04)),
    "C4c": _cfg("C4c", 8, 17408, 5120, 2, 64, 6, s_range=(0.005, 0.04)),
}

# Decode-step stack: 64 layers x {q, k, v, o, gate/up, down}, 4-bit, group 128.
STEP_LAYERS = 64
STEP_PROJ = (("q", 5120, 5120), ("k", 5120, 1024), ("v", 5120, 1024),
             ("o", 5120, 5120), ("gate_up", 5120, 34816), ("down", 17408, 5120))
STEP_SEED = 7
STEP_M_SWEEP = (1, 2, 4, 8, 12, 16, 24, 32)


def step_projections(M: int, layers: int = STEP_LAYERS) -> List[Projection]:
    out = []
    for l in range(layers):
        for j, (nm, K, N) in enumerate(STEP_PROJ):
            out.append(_cfg(f"L{l}.{nm}", M, K, N, 4, 128, STEP_SEED, index=l * len(STEP_PROJ) + j))
    return out


# ------------------------------------------------------------- generation
def gen_weights(p: Projection, rows: Optional[Sequence[int]] = None) -> Dict[str, np.ndarray]:
    """q [R][K] uint8, s [R][ng] uint16 (bf16 bits), z [R][ng] uint8 for rows ``rows``."""
    rows_a = np.arange(p.N, dtype=np.uint64) if rows is None else np.asarray(rows, dtype=np.uint64)
    K, ng = np.uint64(p.K), np.uint64(p.ng)
    kq = np.arange(p.K, dtype=np.uint64)
    kg = np.arange(p.ng, dtype=np.uint64)
    cq = rows_a[:, None] * K + kq[None, :]
    cg = rows_a[:, None] * ng + kg[None, :]
    q = _uniform_int(draws_u64(stream_key(p.seed, "q", p.index), cq), *p.q_range).astype(np.uint8)
    z = _uniform_int(draws_u64(stream_key(p.seed, "z", p.index), cg), *p.zr).astype(np.uint8)
    s32 = _uniform_f32(draws_u64(stream_key(p.seed, "s", p.index), cg), *p.s_range)
    return {"q": q, "s": f32_to_bf16_bits(s32), "z": z}


def outlier_channels(p: Projection) -> np.ndarray:
    """round(frac*K) distinct K channels, chosen by sorting per-channel draws."""
    n_out = int(round(p.outlier_frac * p.K))
    if n_out == 0:
        return np.zeros(0, dtype=np.int64)
    u = draws_u64(stream_key(p.seed, "outlier", p.index), np.arange(p.K, dtype=np.uint64))
    return np.sort(np.argsort(u, kind="stable")[:n_out]).astype(np.int64)


def gen_x(p: Projection) -> np.ndarray:
    """x [M][K] as uint16 bf16 bits: N(0,1), outlier channels scaled in float32."""
    kk = np.arange(p.K, dtype=np.uint64)
    rows = []
    for m in range(p.M):
        if p.x_row_seeds is not None:
            key, base = stream_key(p.x_row_seeds[m], "x", p.index), np.uint64(0)
        else:
            key, base = stream_key(p.seed, "x", p.index), np.uint64(m) * np.uint64(p.K)
        rows.append(_normal_f32(key, base + kk))
    x32 = np.stack(rows) if rows else np.zeros((0, p.K), dtype=np.float32)
    ch = outlier_channels(p)
    if ch.size:
        x32[:, ch] = x32[:, ch] * np.float32(p.outlier_scale)
    return f32_to_bf16_bits(x32)


# ---------------------------------------------------------- torch (device)
def _t_lshr(z, s: int):
    return (z >> s) & ((1 << (64 - s)) - 1)


def _t_signed(c: int) -> int:
    return c - (1 << 64) if c >= (1 << 63) else c


def _t_mix(z):
    z = (z ^ _t_lshr(z, 30)) * _t_signed(_C1)
    z = (z ^ _t_lshr(z, 27)) * _t_signed(_C2)
    return z ^ _t_lshr(z, 31)


def _t_draws(key: int, counters):
    return _t_mix(counters.add(1).mul_(_t_signed(_GAMMA)).add_(_t_signed(key)))


def gen_weights_torch(p: Projection, device, row_chunk: int = 4096):
    """Same values as ``gen_weights`` built on ``device`` with torch int64/float32 ops.

    Returns uint8 q [N][K], int16 s bits [N][ng] (bf16 pattern), uint8 z [N][ng].
    """
    import torch

    q = torch.empty((p.N, p.K), dtype=torch.uint8, device=device)
    s = torch.empty((p.N, p.ng), dtype=torch.int16, device=device)
    z = torch.empty((p.N, p.ng), dtype=torch.uint8, device=device)
    kq = torch.arange(p.K, dtype=torch.int64, device=device)
    kg = torch.arange(p.ng, dtype=torch.int64, device=device)
    keys = {nm: stream_key(p.seed, nm, p.index) for nm in ("q", "s", "z")}
    a32 = torch.tensor(np.float32(p.s_range[0]), device=device)
    b32 = torch.tensor(np.float32(p.s_range[1]), device=device)

    def uint_range(u, lo, hi):
        return lo + ((_t_lshr(u, 32) * (hi - lo + 1)) >> 32)

    for r0 in range(0, p.N, row_chunk):
        r1 = min(p.N, r0 + row_chunk)
        rr = torch.arange(r0, r1, dtype=torch.int64, device=device)
        uq = _t_draws(keys["q"], rr[:, None] * p.K + kq[None, :])
        q[r0:r1] = uint_range(uq, *p.q_range).to(torch.uint8)
        del uq
        cg = rr[:, None] * p.ng + kg[None, :]
        z[r0:r1] = uint_range(_t_draws(keys["z"], cg), *p.zr).to(torch.uint8)
        u24 = _t_lshr(_t_draws(keys["s"], cg), 40).to(torch.float32) * (2.0 ** -24)
        s32 = a32 + (b32 - a32) * u24
        s[r0:r1] = s32.to(torch.bfloat16).view(torch.int16)
    return q, s, z


# ------------------------------------------------- paged q8_0 attention inputs
@dataclasses.dataclass(frozen=True)
class PagedAttention:
    """A decode step's attention over a shared paged KV pool: sequences of
    ``seq_lens`` tokens (the last ``rows_per_seq`` of each are this step's query
    rows), the first ``shared_prefix`` tokens of every sequence stored once in
    pages all sequences share."""
    name: str
    seq_lens: tuple
    rows_per_seq: int
    Hq: int
    Hkv: int
    D: int
    T: int  # tokens per page
    seed: int
    shared_prefix: int = 0
    spare_pages: int = 3  # pool pages no sequence uses
    scale_range: tuple = (0.002, 0.02)


def gen_paged_attention(p: PagedAttention) -> Dict[str, np.ndarray]:
    """Codes U{-127..127} and fp16 scales U(scale_range) for every page of the
    pool, bf16 N(0,1) queries, and page tables that place each sequence's
    logical pages on distinct physical pages in a seeded shuffled order (the
    shared prefix's pages are the same physical pages in every sequence)."""
    out, shape = _paged_tables(p)
    n_codes = int(np.prod(shape))
    n_scales = n_codes // 32
    for i, kv in enumerate(("k", "v")):
        cu = draws_u64(stream_key(p.seed, "kv_code", i), np.arange(n_codes, dtype=np.uint64))
        out[kv + "c"] = (_uniform_int(cu, 0, 254) - 127).astype(np.int8).reshape(shape)
        su = draws_u64(stream_key(p.seed, "kv_scale", i), np.arange(n_scales, dtype=np.uint64))
        d32 = _uniform_f32(su, *p.scale_range)
        out[kv + "d"] = d32.astype(np.float16).view(np.uint16).reshape(shape[:3] + (p.D // 32,))
    return out


def gen_paged_attention_torch(p: PagedAttention, device, chunk: int = 1 << 22):
    """The values of ``gen_paged_attention``, with the K and V codes and scales
    built on ``device`` by torch int64/float32 ops (the page tables and queries
    are small and come from the host).  Codes are int8 tensors, scales and
    queries int16 tensors holding the binary16 / bf16 bit patterns, the
    tables int32 tensors."""
    import torch

    host, shape = _paged_tables(p)
    out = {"q": torch.from_numpy(host["q"].view(np.int16)).to(device)}
    for k in ("page_table", "seq_len", "row_seq", "row_pos"):
        out[k] = torch.from_numpy(np.ascontiguousarray(host[k], dtype=np.int32)).to(device)
    n_codes = int(np.prod(shape))
    n_scales = n_codes // 32
    a32 = torch.tensor(np.float32(p.scale_range[0]), device=device)
    b32 = torch.tensor(np.float32(p.scale_range[1]), device=device)
    for i, kv in enumerate(("k", "v")):
        codes = torch.empty(n_codes, dtype=torch.int8, device=device)
        key = stream_key(p.seed, "kv_code", i)
        for c0 in range(0, n_codes, chunk):
            c1 = min(n_codes, c0 + chunk)
            u = _t_draws(key, torch.arange(c0, c1, dtype=torch.int64, device=device))
            codes[c0:c1] = ((_t_lshr(u, 32) * 255) >> 32).sub_(127).to(torch.int8)
        out[kv + "c"] = codes.view(shape)
        scales = torch.empty(n_scales, dtype=torch.int16, device=device)
        key = stream_key(p.seed, "kv_scale", i)
        for c0 in range(0, n_scales, chunk):
            c1 = min(n_scales, c0 + chunk)
            u24 = _t_lshr(_t_draws(key, torch.arange(c0, c1, dtype=torch.int64, device=device)),
                          40).to(torch.float32) * (2.0 ** -24)
            scales[c0:c1] = (a32 + (b32 - a32) * u24).to(torch.float16).view(torch.int16)
        out[kv + "d"] = scales.view(shape[:3] + (p.D // 32,))
    return out


def _paged_tables(p: PagedAttention):
    """Page tables, sequence lengths, query rows and bf16 queries of ``p``,
    and the shape [pages][Hkv][T][D] of the pool's code arrays."""
    B = len(p.seq_lens)
    assert p.shared_prefix % p.T == 0 and all(n >= p.shared_prefix for n in p.seq_lens)
    assert all(n >= p.rows_per_seq for n in p.seq_lens)
    n_shared = p.shared_prefix // p.T
    own = [(n - p.shared_prefix + p.T - 1) // p.T for n in p.seq_lens]
    pages = n_shared + sum(own) + p.spare_pages
    order = np.argsort(draws_u64(stream_key(p.seed, "page"), np.arange(pages, dtype=np.uint64)),
                       kind="stable").astype(np.int32)
    max_pages = max(n_shared + o for o in own)
    table = np.zeros((B, max_pages), dtype=np.int32)
    nxt = n_shared
    for b in range(B):
        table[b, :n_shared] = order[:n_shared]
        table[b, n_shared:n_shared + own[b]] = order[nxt:nxt + own[b]]
        nxt += own[b]
    shape = (pages, p.Hkv, p.T, p.D)
    out = {}
    rows = B * p.rows_per_seq
    qn = _normal_f32(stream_key(p.seed, "attn_q"), np.arange(rows * p.Hq * p.D, dtype=np.uint64))
    out["q"] = f32_to_bf16_bits(qn).reshape(rows, p.Hq, p.D)
    out["page_table"] = table
    out["seq_len"] = np.array(p.seq_lens, dtype=np.int32)
    out["row_seq"] = np.repeat(np.arange(B, dtype=np.int32), p.rows_per_seq)
    out["row_pos"] = np.concatenate([np.arange(n - p.rows_per_seq, n, dtype=np.int32)
                                     for n in p.seq_lens])
    return out, shape
