"""ctypes front end of the fp64 CPU oracle (``wq_oracle.cpp``: the GEMM and
its epilogue; ``attn_oracle.cpp``: decode attention over a paged q8_0 KV pool).

TEST INFRASTRUCTURE ONLY: imported by the tests, the smoke check and the
benchmark's CPU-baseline leg, never by the library.  It shares no code with the
CUDA path.  ``build()`` compiles the C++ source with g++ and OpenMP.

All bf16 arrays cross this boundary as uint16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRCS = [os.path.join(_HERE, "wq_oracle.cpp"), os.path.join(_HERE, "attn_oracle.cpp")]
_LIB = os.path.join(_HERE, "liboracle.so")
_lib: Optional[ctypes.CDLL] = None


def build(force: bool = False) -> str:
    """Compile liboracle.so (plain C++17, OpenMP, no FMA contraction)."""
    newest = max(os.path.getmtime(f) for f in _SRCS)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < newest:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
               "-shared", "-fPIC", "-o", tmp, *_SRCS]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i = ctypes.c_int
        lib.wqo_words_per_row.argtypes = [i, i]
        lib.wqo_words_per_row.restype = ctypes.c_long
        lib.wqo_pack.argtypes = [P, P, i, i, i]
        lib.wqo_unpack.argtypes = [P, P, i, i, i]
        lib.wqo_dequant_f64.argtypes = [P, P, P, P, i, i, i, i]
        lib.wqo_dequant_bf16.argtypes = [P, P, P, P, i, i, i, i]
        lib.wqo_bf16_rne.argtypes = [ctypes.c_double]
        lib.wqo_bf16_rne.restype = ctypes.c_uint16
        lib.wqo_gemm_f64.argtypes = [P, P, P, P, P, i, i, i, i, i, i]
        lib.wqo_silu_f64.argtypes = [ctypes.c_double]
        lib.wqo_silu_f64.restype = ctypes.c_double
        lib.wqo_swiglu_bf16.argtypes = [P, i, i, P]
        lib.wqo_max_threads.argtypes = [i]
        lib.wqo_fp16_value.argtypes = [ctypes.c_uint16]
        lib.wqo_fp16_value.restype = ctypes.c_double
        lib.wqo_q8_0_dequant.argtypes = [P, P, ctypes.c_long, P]
        lib.wqo_q8_0_dequant.restype = ctypes.c_int
        lib.wqo_paged_attention_f64.argtypes = [P, P, P, P, P, P, P, P, P] + [i] * 8 + [P]
        lib.wqo_paged_attention_f64.restype = ctypes.c_int
        for fn in (lib.wqo_pack, lib.wqo_unpack, lib.wqo_dequant_f64, lib.wqo_dequant_bf16,
                   lib.wqo_gemm_f64, lib.wqo_max_threads):
            fn.restype = ctypes.c_int
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return ctypes.c_void_p(a.ctypes.data)


def words_per_row(K: int, bits: int) -> int:
    return int(_load().wqo_words_per_row(K, bits))


def pack(q: np.ndarray, bits: int) -> np.ndarray:
    q = np.ascontiguousarray(q, dtype=np.uint8)
    N, K = q.shape
    out = np.zeros((N, words_per_row(K, bits)), dtype=np.uint32)
    if _load().wqo_pack(_ptr(q), _ptr(out), N, K, bits):
        raise ValueError("oracle pack: bad arguments")
    return out


def unpack(wq: np.ndarray, K: int, bits: int) -> np.ndarray:
    wq = np.ascontiguousarray(wq, dtype=np.uint32)
    N = wq.shape[0]
    out = np.zeros((N, K), dtype=np.uint8)
    if _load().wqo_unpack(_ptr(wq), _ptr(out), N, K, bits):
        raise ValueError("oracle unpack: bad arguments")
    return out


def dequant_f64(wq, s, z, K: int, group: int, bits: int) -> np.ndarray:
    wq = np.ascontiguousarray(wq, dtype=np.uint32)
    s = np.ascontiguousarray(s, dtype=np.uint16)
    z = np.ascontiguousarray(z, dtype=np.uint8)
    N = wq.shape[0]
    out = np.zeros((N, K), dtype=np.float64)
    if _load().wqo_dequant_f64(_ptr(wq), _ptr(s), _ptr(z), _ptr(out), N, K, group, bits):
        raise ValueError("oracle dequant: bad arguments")
    return out


def dequant_bf16(wq, s, z, K: int, group: int, bits: int) -> np.ndarray:
    wq = np.ascontiguousarray(wq, dtype=np.uint32)
    s = np.ascontiguousarray(s, dtype=np.uint16)
    z = np.ascontiguousarray(z, dtype=np.uint8)
    N = wq.shape[0]
    out = np.zeros((N, K), dtype=np.uint16)
    if _load().wqo_dequant_bf16(_ptr(wq), _ptr(s), _ptr(z), _ptr(out), N, K, group, bits):
        raise ValueError("oracle dequant: bad arguments")
    return out


def bf16_rne(v: float) -> int:
    return int(_load().wqo_bf16_rne(float(v)))


def gemm_f64(x, wq, s, z, K: int, group: int, bits: int, threads: int = 0) -> np.ndarray:
    """Y[M][N] (float64) for x [M][K] bf16 bits and packed rows wq [N][W]."""
    x = np.ascontiguousarray(x, dtype=np.uint16)
    wq = np.ascontiguousarray(wq, dtype=np.uint32)
    s = np.ascontiguousarray(s, dtype=np.uint16)
    z = np.ascontiguousarray(z, dtype=np.uint8)
    M, N = x.shape[0], wq.shape[0]
    y = np.zeros((M, N), dtype=np.float64)
    if _load().wqo_gemm_f64(_ptr(x), _ptr(wq), _ptr(s), _ptr(z), _ptr(y), M, N, K, group, bits,
                            threads):
        raise ValueError("oracle gemm: bad arguments")
    return y


def silu_f64(g: float) -> float:
    """silu(g) = g / (1 + e^-g) in double."""
    return _load().wqo_silu_f64(float(g))


def swiglu_bf16(y: np.ndarray) -> np.ndarray:
    """bf16 bit patterns [M][N/2] of silu(y[:, 2j]) * y[:, 2j + 1], one rounding."""
    y = np.ascontiguousarray(y, dtype=np.float64)
    M, N = y.shape
    out = np.empty((M, N // 2), dtype=np.uint16)
    rc = _load().wqo_swiglu_bf16(_ptr(y), M, N, _ptr(out))
    if rc:
        raise ValueError("swiglu_bf16: N must be even")
    return out


def max_threads(threads: int = 0) -> int:
    return int(_load().wqo_max_threads(threads))


def step_floor_seconds(weight_bytes: float, bandwidth_bytes_per_s: float) -> float:
    """Closed-form decode-step floor when every weight byte is read once per step.

    OpenJet news page, paragraph "并行解码的原理": the step is bound by reading all
    weights from memory once, so its time is at least bytes / bandwidth.
    """
    return weight_bytes / bandwidth_bytes_per_s


# ------------------------------------------------------ paged decode attention
def fp16_value(h: int) -> float:
    """IEEE binary16 bit pattern -> value."""
    return float(_load().wqo_fp16_value(int(h) & 0xFFFF))


def q8_0_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """q8_0 blocks: codes int8 [..., 32 n], scales fp16 bits uint16 [..., n] ->
    float64 [..., 32 n] with value = scale * code per block of 32."""
    c = np.ascontiguousarray(codes, dtype=np.int8)
    d = np.ascontiguousarray(scales, dtype=np.uint16)
    assert c.size == 32 * d.size
    out = np.empty(c.shape, dtype=np.float64)
    if _load().wqo_q8_0_dequant(_ptr(c), _ptr(d), d.size, _ptr(out)):
        raise ValueError("oracle q8_0_dequant: bad arguments")
    return out


def paged_attention_f64(q: np.ndarray, kc: np.ndarray, kd: np.ndarray, vc: np.ndarray,
                        vd: np.ndarray, page_table: np.ndarray, seq_len: np.ndarray,
                        row_seq: np.ndarray, row_pos: np.ndarray) -> np.ndarray:
    """Decode attention over a paged q8_0 pool.

    q: bf16 bits uint16 [rows][Hq][D]; kc, vc: int8 [pages][Hkv][T][D];
    kd, vd: fp16 bits uint16 [pages][Hkv][T][D/32]; page_table: int32 [B][max_pages];
    seq_len: int32 [B]; row_seq, row_pos: int32 [rows] (row i attends to positions
    0 .. row_pos[i] of sequence row_seq[i]).  Returns float64 [rows][Hq][D]."""
    q = np.ascontiguousarray(q, dtype=np.uint16)
    kc = np.ascontiguousarray(kc, dtype=np.int8)
    vc = np.ascontiguousarray(vc, dtype=np.int8)
    kd = np.ascontiguousarray(kd, dtype=np.uint16)
    vd = np.ascontiguousarray(vd, dtype=np.uint16)
    pt = np.ascontiguousarray(page_table, dtype=np.int32)
    sl = np.ascontiguousarray(seq_len, dtype=np.int32)
    rs = np.ascontiguousarray(row_seq, dtype=np.int32)
    rp = np.ascontiguousarray(row_pos, dtype=np.int32)
    rows, Hq, D = q.shape
    pages, Hkv, T, D2 = kc.shape
    assert D2 == D and vc.shape == kc.shape
    assert kd.shape == (pages, Hkv, T, D // 32) and vd.shape == kd.shape
    B, max_pages = pt.shape
    out = np.zeros((rows, Hq, D), dtype=np.float64)
    if _load().wqo_paged_attention_f64(_ptr(q), _ptr(kc), _ptr(kd), _ptr(vc), _ptr(vd), _ptr(pt),
                                       _ptr(sl), _ptr(rs), _ptr(rp), rows, B, max_pages, Hq, Hkv,
                                       D, T, pages, _ptr(out)):
        raise ValueError("oracle paged_attention_f64: bad arguments")
    return out
