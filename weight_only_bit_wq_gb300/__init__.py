"""Python binding of libwq (ctypes; argument marshalling only).

Every entry point has the name of the C function it calls (include/wq.h) and
passes torch tensors' device pointers plus the current CUDA stream.  All
arithmetic runs in libwq's CUDA kernels; there is no fallback: if libwq.so is
missing or a call fails, an exception is raised.

bf16 tensors may be given as torch.bfloat16 or as their int16/uint16 bit
patterns; packed words are held in torch.int32 tensors (bit patterns of the
uint32 words).
"""
from __future__ import annotations

import ctypes
import os
from typing import List, Optional, Sequence

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libwq.so")

WQ_OK, WQ_ERR_INVALID_ARG, WQ_ERR_UNSUPPORTED, WQ_ERR_CUDA, WQ_ERR_TIMEOUT = range(5)

EXPORTED = ("wq_abi_version", "wq_status_string", "wq_last_cuda_error", "wq_packed_words_per_row",
            "wq_pack", "wq_unpack", "wq_dequant", "wq_workspace_bytes", "wq_workspace_bytes_for", "wq_workspace_init",
            "wq_gemm", "wq_gemm_swiglu", "wq_check_workspace", "wq_gemm_noalloc", "wq_check_noalloc",
            "wq_step_workspace_bytes", "wq_step_run",
            "wq_step_run_ex", "wq_step_graph_create", "wq_step_graph_create_ex",
            "wq_step_graph_launch", "wq_step_graph_destroy", "wq_paged_attention_workspace_bytes",
            "wq_paged_attention")

# Step modes (include/wq.h).
WQ_STEP_FUSED = 1
WQ_STEP_PHASES = 2
# Projection epilogues (include/wq.h).
WQ_EPI_NONE, WQ_EPI_SWIGLU = 0, 1


class WQError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        lib = _lib()
        msg = lib.wq_status_string(status).decode()
        if status == WQ_ERR_CUDA:
            msg += f" (cudaError {lib.wq_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")


class ProjDesc(ctypes.Structure):
    _fields_ = [("x", ctypes.c_void_p), ("wq", ctypes.c_void_p), ("scales", ctypes.c_void_p),
                ("zeros", ctypes.c_void_p), ("y", ctypes.c_void_p), ("M", ctypes.c_int),
                ("N", ctypes.c_int), ("K", ctypes.c_int), ("group", ctypes.c_int),
                ("bits", ctypes.c_int), ("after", ctypes.c_int), ("epilogue", ctypes.c_int)]


_LIB: Optional[ctypes.CDLL] = None


def _lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libwq.so is not built ({LIB_PATH}); run weight_only_bit_wq_gb300.build.build()")
        lib = ctypes.CDLL(LIB_PATH)
        P, I, S = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
        sig = {
            "wq_abi_version": ([], I),
            "wq_status_string": ([I], ctypes.c_char_p),
            "wq_last_cuda_error": ([], I),
            "wq_packed_words_per_row": ([I, I], ctypes.c_long),
            "wq_pack": ([P, P, I, I, I, P], I),
            "wq_unpack": ([P, P, I, I, I, P], I),
            "wq_dequant": ([P, P, P, P, I, I, I, I, P], I),
            "wq_workspace_bytes": ([I, I, I, I, I], S),
            "wq_workspace_bytes_for": ([I, I, I, I, I, I], S),
            "wq_workspace_init": ([P, S, P], I),
            "wq_gemm": ([P, P, P, P, P, I, I, I, I, I, P, S, P], I),
            "wq_gemm_swiglu": ([P, P, P, P, P, I, I, I, I, I, P, S, P], I),
            "wq_check_workspace": ([P, P], I),
            "wq_gemm_noalloc": ([P, P, P, P, P, I, I, I, I, I, P], I),
            "wq_check_noalloc": ([P], I),
            "wq_paged_attention_workspace_bytes": ([I, I, I, I, I], S),
            "wq_paged_attention": ([P, P, P, P, P, P, I, P, I, P, P, I, I, I, I, I, I, I, P, P, S, P], I),
            "wq_step_workspace_bytes": ([P, I, ctypes.c_uint], S),
            "wq_step_run": ([P, I, P, S, P], I),
            "wq_step_run_ex": ([P, I, ctypes.c_uint, P, S, P], I),
            "wq_step_graph_create": ([P, I, P, S, P, P], I),
            "wq_step_graph_create_ex": ([P, I, ctypes.c_uint, P, S, P, P], I),
            "wq_step_graph_launch": ([P, P], I),
            "wq_step_graph_destroy": ([P], None),
            "wq_internal_schedule_check": ([ctypes.c_longlong, I], I),
            "wq_internal_choose_grid": ([I, I, I], I),
            "wq_internal_phase_grid": ([I, I, I, ctypes.c_longlong, I, I, I, P, P], I),
        }
        for name, (args, res) in sig.items():
            fn = getattr(lib, name, None)
            if fn is None:  # an older library: the call fails when it is made
                continue
            fn.argtypes = args
            fn.restype = res
        _LIB = lib
    return _LIB


def _check(status: int, where: str) -> None:
    if status != WQ_OK:
        raise WQError(status, where)


def _stream(stream=None) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t: Optional[torch.Tensor]) -> ctypes.c_void_p:
    if t is None:
        return ctypes.c_void_p(0)
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return ctypes.c_void_p(t.data_ptr())


def abi_version() -> int:
    return int(_lib().wq_abi_version())


def wq_packed_words_per_row(K: int, bits: int) -> int:
    return int(_lib().wq_packed_words_per_row(K, bits))


def wq_pack(q: torch.Tensor, bits: int, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """uint8 codes [N][K] -> packed words [N][W] (int32 bit patterns)."""
    N, K = q.shape
    W = wq_packed_words_per_row(K, bits)
    if out is None:
        out = torch.empty((N, max(W, 0)), dtype=torch.int32, device=q.device)
    _check(_lib().wq_pack(_ptr(q), _ptr(out), N, K, bits, _stream(stream)), "wq_pack")
    return out


def wq_unpack(wq: torch.Tensor, K: int, bits: int, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    N = wq.shape[0]
    if out is None:
        out = torch.empty((N, K), dtype=torch.uint8, device=wq.device)
    _check(_lib().wq_unpack(_ptr(wq), _ptr(out), N, K, bits, _stream(stream)), "wq_unpack")
    return out


def wq_dequant(wq, scales, zeros, K: int, group: int, bits: int, out=None, stream=None) -> torch.Tensor:
    """bf16 weights [N][K] = RNE((q - z) * s)."""
    N = wq.shape[0]
    if out is None:
        out = torch.empty((N, K), dtype=torch.bfloat16, device=wq.device)
    _check(_lib().wq_dequant(_ptr(wq), _ptr(scales), _ptr(zeros), _ptr(out), N, K, group, bits,
                             _stream(stream)), "wq_dequant")
    return out


def wq_workspace_bytes(M: int, N: int, K: int, group: int, bits: int) -> int:
    return int(_lib().wq_workspace_bytes(M, N, K, group, bits))


def wq_workspace_bytes_for(M: int, N: int, K: int, group: int, bits: int, sm_count: int) -> int:
    return int(_lib().wq_workspace_bytes_for(M, N, K, group, bits, sm_count))


def wq_workspace_init(ws: torch.Tensor, stream=None) -> torch.Tensor:
    _check(_lib().wq_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "wq_workspace_init")
    return ws


def new_workspace(M: int, N: int, K: int, group: int, bits: int, device="cuda") -> torch.Tensor:
    """A zeroed workspace for wq_gemm calls of this shape (or smaller)."""
    nbytes = wq_workspace_bytes(M, N, K, group, bits)
    if nbytes == 0:
        raise WQError(WQ_ERR_INVALID_ARG, "wq_workspace_bytes")
    return wq_workspace_init(torch.empty(nbytes, dtype=torch.uint8, device=device))


def wq_gemm(x, wq, scales, zeros, N: int, group: int, bits: int, out=None, workspace=None,
            stream=None) -> torch.Tensor:
    """Y[M][N] (fp32) = X[M][K] . dequant(Wq)[N][K]^T."""
    M, K = x.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib().wq_gemm(_ptr(x), _ptr(wq), _ptr(scales), _ptr(zeros), _ptr(out), M, N, K, group,
                          bits, _ptr(workspace), nbytes, _stream(stream)), "wq_gemm")
    return out


def wq_gemm_swiglu(x, wq, scales, zeros, N: int, group: int, bits: int, out=None, workspace=None,
                   stream=None) -> torch.Tensor:
    """bf16 [M][N/2] = silu(gate) * up of the fused gate/up projection (rows 2j, 2j + 1 of the
    weights are the gate and up rows of feature j)."""
    M, K = x.shape
    if out is None:
        out = torch.empty((M, N // 2), dtype=torch.bfloat16, device=x.device)
    nbytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check(_lib().wq_gemm_swiglu(_ptr(x), _ptr(wq), _ptr(scales), _ptr(zeros), _ptr(out), M, N, K,
                                 group, bits, _ptr(workspace), nbytes, _stream(stream)),
           "wq_gemm_swiglu")
    return out


def wq_paged_attention(q, kc, kd, vc, vd, page_table, seq_len, row_seq, row_pos, max_seq_len: int,
                       out=None, workspace=None, stream=None) -> torch.Tensor:
    """fp32 [rows][Hq][D] decode attention over a paged q8_0 pool (include/wq.h).

    q bf16 [rows][Hq][D]; kc, vc int8 [pages][Hkv][T][D]; kd, vd binary16 bits
    [pages][Hkv][T][D/32]; page_table int32 [B][max_pages]; seq_len int32 [B];
    row_seq, row_pos int32 [rows]; all on the device.  The workspace's first word
    is the kernel's error word (2: a table entry outside the pool)."""
    rows, Hq, D = q.shape
    pages, Hkv, T, _ = kc.shape
    B, max_pages = page_table.shape
    if out is None:
        out = torch.empty((rows, Hq, D), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = int(_lib().wq_paged_attention_workspace_bytes(rows, Hq, Hkv, B, max_seq_len))
        workspace = torch.zeros(max(n, 256), dtype=torch.uint8, device=q.device)
    nbytes = workspace.numel() * workspace.element_size()
    _check(_lib().wq_paged_attention(_ptr(q), _ptr(kc), _ptr(kd), _ptr(vc), _ptr(vd),
                                     _ptr(page_table), max_pages, _ptr(seq_len), B, _ptr(row_seq),
                                     _ptr(row_pos), rows, max_seq_len, Hq, Hkv, D, T, pages,
                                     _ptr(out), _ptr(workspace), nbytes, _stream(stream)),
           "wq_paged_attention")
    return out


def wq_check_workspace(workspace=None, stream=None) -> None:
    _check(_lib().wq_check_workspace(_ptr(workspace), _stream(stream)), "wq_check_workspace")


def wq_gemm_noalloc(x, wq, scales, zeros, N: int, group: int, bits: int, out=None,
                    stream=None) -> torch.Tensor:
    """wq_gemm with its scratch in the library's fixed device array (no device allocation
    inside libwq; `out`, if given, is the caller's fp32 [M][N] buffer)."""
    M, K = x.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=x.device)
    _check(_lib().wq_gemm_noalloc(_ptr(x), _ptr(wq), _ptr(scales), _ptr(zeros), _ptr(out), M, N,
                                  K, group, bits, _stream(stream)), "wq_gemm_noalloc")
    return out


def wq_check_noalloc(stream=None) -> None:
    _check(_lib().wq_check_noalloc(_stream(stream)), "wq_check_noalloc")


def make_descs(projs: Sequence[dict]) -> ctypes.Array:
    """Descriptor array from dicts with keys x, wq, scales, zeros, y, M, N, K, group, bits and
    optionally after (fused mode: x depends on projections 0..after; default -1)."""
    arr = (ProjDesc * len(projs))()
    for i, p in enumerate(projs):
        arr[i] = ProjDesc(p["x"].data_ptr(), p["wq"].data_ptr(), p["scales"].data_ptr(),
                          p["zeros"].data_ptr(), p["y"].data_ptr(), p["M"], p["N"], p["K"],
                          p["group"], p["bits"], p.get("after", -1), p.get("epilogue", WQ_EPI_NONE))
    return arr


def wq_step_workspace_bytes(descs: ctypes.Array, flags: int = 0) -> int:
    return int(_lib().wq_step_workspace_bytes(ctypes.cast(descs, ctypes.c_void_p), len(descs),
                                              flags))


def new_step_workspace(descs: ctypes.Array, flags: int = 0, device=None) -> torch.Tensor:
    """A zeroed workspace for a step of these descriptors in this mode."""
    n = wq_step_workspace_bytes(descs, flags)
    if n == 0:
        raise ValueError("invalid step descriptors")
    ws = torch.zeros(n, dtype=torch.uint8, device=device or "cuda")
    return ws


def wq_step_run(descs: ctypes.Array, workspace: torch.Tensor, stream=None, flags: int = 0) -> None:
    _check(_lib().wq_step_run_ex(ctypes.cast(descs, ctypes.c_void_p), len(descs), flags,
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _stream(stream)),
           "wq_step_run_ex")


class StepGraph:
    """A captured decode step (wq_step_graph_create / _launch / _destroy)."""

    def __init__(self, descs: ctypes.Array, workspace: torch.Tensor, stream=None, flags: int = 0):
        self._descs = descs
        self._ws = workspace
        h = ctypes.c_void_p(0)
        _check(_lib().wq_step_graph_create_ex(ctypes.cast(descs, ctypes.c_void_p), len(descs),
                                              flags, _ptr(workspace),
                                              workspace.numel() * workspace.element_size(),
                                              _stream(stream), ctypes.byref(h)),
               "wq_step_graph_create_ex")
        self._h = h

    def launch(self, stream=None) -> None:
        _check(_lib().wq_step_graph_launch(self._h, _stream(stream)), "wq_step_graph_launch")

    def close(self) -> None:
        if self._h:
            _lib().wq_step_graph_destroy(self._h)
            self._h = ctypes.c_void_p(0)

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
