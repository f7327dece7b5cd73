"""wq_gemm_noalloc: the GEMM for callers that cannot allocate device memory
(a framework or server that owns every byte of GPU memory through its own
pool, or a step that must not allocate part-way through).  It keeps its scratch
in a fixed array inside the library instead of a workspace argument.

This file is collected last on purpose.  Its checks, through the C ABI: two
calls in a row give Y bit for bit equal to wq_gemm's (the same kernel with the
same split; the second call sees whatever the first left in the shared array)
and within the GEMM tolerance of the fp64 oracle; the array's error word reads
back clean (wq_check_noalloc); a 300,160-row problem runs; a problem whose
counters would not fit the fixed array, and bad arguments, are refused before
anything is launched.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from wqtest import ARITH_TOL, REL_TOL, dev, oracle_gemm, rel_err, to_dev_host_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__.build()
    import weight_only_bit_wq_gb300 as wq
    L = ctypes.CDLL(wq.LIB_PATH)
    P, I = ctypes.c_void_p, ctypes.c_int
    L.wq_gemm_noalloc.argtypes = [P, P, P, P, P, I, I, I, I, I, P]
    L.wq_gemm_noalloc.restype = I
    L.wq_check_noalloc.argtypes = [P]
    L.wq_check_noalloc.restype = I
    return L


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _call(lib, d, y, p):
    return lib.wq_gemm_noalloc(ctypes.c_void_p(d["x"].data_ptr()), ctypes.c_void_p(d["wq"].data_ptr()),
                               ctypes.c_void_p(d["s"].data_ptr()), ctypes.c_void_p(d["z"].data_ptr()),
                               ctypes.c_void_p(y.data_ptr()), p.M, p.N, p.K, p.group, p.bits,
                               _stream())


def test_noalloc_matches_wq_gemm_and_oracle_twice(lib):
    import weight_only_bit_wq_gb300 as wq
    # first a shape whose tiles are split across CTAs, then a different one
    cases = [synth.Projection("a", 12, 3000, 5120, 4, 128, 901, outlier_frac=0.01),
             synth.Projection("b", 5, 1030, 2048, 2, 64, 902, s_range=(0.005, 0.04))]
    for p in cases:
        w, x, d = to_dev_host_inputs(p)
        ref = wq.wq_gemm(d["x"], d["wq"], d["s"], d["z"], p.N, p.group, p.bits).cpu().numpy()
        y_ref = oracle_gemm(p, w, x)
        for _ in range(2):
            y = torch.full((p.M, p.N), float("nan"), dtype=torch.float32, device=dev())
            assert _call(lib, d, y, p) == wq.WQ_OK
            got = y.cpu().numpy()
            # same kernel, same split, same reduction order: bit for bit
            assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))
            err = rel_err(got, y_ref)
            assert err <= REL_TOL and err <= ARITH_TOL, err
        assert lib.wq_check_noalloc(_stream()) == wq.WQ_OK


def test_noalloc_tall_problem_runs_oversized_is_refused(lib):
    # The fixed array holds the split-K partials (two slots per CTA) and 64
    # bytes of arrival counters per 128-row tile: a 300,160-row problem fits and
    # matches wq_gemm bit for bit; 2^30 rows (2^23 tiles, 512 MiB of counters)
    # do not and are refused before anything is launched, as are bad arguments.
    import weight_only_bit_wq_gb300 as wq
    p = synth.Projection("tall", 3, 300160, 256, 4, 128, 903)
    q, s, z = synth.gen_weights_torch(p, dev())
    wqw = wq.wq_pack(q, p.bits)
    x = torch.from_numpy(synth.gen_x(p).view(np.int16)).to(dev())
    ref = wq.wq_gemm(x, wqw, s, z, p.N, p.group, p.bits).cpu().numpy()
    y = torch.full((p.M, p.N), float("nan"), dtype=torch.float32, device=dev())
    st = lib.wq_gemm_noalloc(ctypes.c_void_p(x.data_ptr()), ctypes.c_void_p(wqw.data_ptr()),
                             ctypes.c_void_p(s.data_ptr()), ctypes.c_void_p(z.data_ptr()),
                             ctypes.c_void_p(y.data_ptr()), p.M, p.N, p.K, p.group, p.bits,
                             _stream())
    assert st == wq.WQ_OK
    assert np.array_equal(y.cpu().numpy().view(np.uint32), ref.view(np.uint32))
    assert lib.wq_check_noalloc(_stream()) == wq.WQ_OK
    P = ctypes.c_void_p
    # refused on the host: the pointers below are never touched
    assert lib.wq_gemm_noalloc(P(16), P(16), P(16), P(16), P(16), 1, 1 << 30, 128, 128, 4,
                               _stream()) == wq.WQ_ERR_INVALID_ARG
    # M > 32, an odd group size and K not a multiple of the group
    assert lib.wq_gemm_noalloc(P(16), P(16), P(16), P(16), P(16), 33, 128, 128, 128, 4,
                               _stream()) == wq.WQ_ERR_INVALID_ARG
    assert lib.wq_gemm_noalloc(P(16), P(16), P(16), P(16), P(16), 1, 128, 128, 96, 4,
                               _stream()) == wq.WQ_ERR_INVALID_ARG
    assert lib.wq_gemm_noalloc(P(16), P(16), P(16), P(16), P(16), 1, 128, 100, 32, 4,
                               _stream()) == wq.WQ_ERR_INVALID_ARG
