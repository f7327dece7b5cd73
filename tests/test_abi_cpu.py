"""CPU-side checks of the C ABI: the library loads, exports every declared
symbol, and rejects bad arguments on the host before touching a GPU."""
import ctypes
import os
import re

import pytest

import __graft_entry__

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def wq():
    __graft_entry__.build()
    import weight_only_bit_wq_gb300 as m
    return m


def _declared():
    text = open(os.path.join(ROOT, "include", "wq.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(wq_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(wq):
    names = _declared()
    assert "wq_gemm" in names and "wq_pack" in names and "wq_dequant" in names
    lib = ctypes.CDLL(wq.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert set(wq.EXPORTED) <= set(names)


def test_abi_version_and_words(wq):
    assert wq.abi_version() == 104
    assert wq.wq_packed_words_per_row(17408, 3) == 1744
    assert wq.wq_packed_words_per_row(5120, 4) == 640
    assert wq.wq_packed_words_per_row(17408, 2) == 1088
    assert wq.wq_packed_words_per_row(10, 5) == -1


def test_workspace_bytes_for_any_sm_count(wq):
    f = wq.wq_workspace_bytes_for
    n = f(16, 5120, 5120, 128, 4, 152)
    # split-K partial slots (two per CTA, 32 x 128 fp32 each) and 16 arrival
    # counters per 128-row tile, in whole 256-byte blocks
    assert n % 256 == 0
    assert n >= 2 * 152 * 32 * 128 * 4 + 40 * 16 * 4
    assert f(1, 5120, 5120, 128, 4, 152) == n          # never depends on M
    assert f(16, 5120, 17408, 128, 4, 152) == n        # nor on K
    assert f(16, 5120, 5120, 32, 2, 152) == n          # nor on the format
    assert f(16, 5120, 5120, 128, 4, 76) < n < f(16, 5120, 5120, 128, 4, 304)
    assert f(16, 34816, 5120, 128, 4, 152) > n         # more tiles, more counters
    for bad in ((16, 5120, 5120, 128, 4, 0), (16, 5120, 5120, 128, 5, 152),
                (33, 5120, 5120, 128, 4, 152), (16, 5120, 100, 32, 4, 152),
                (16, -1, 5120, 128, 4, 152)):
        assert f(*bad) == 0, bad


def _gemm(lib, M=4, N=8, K=128, group=128, bits=4, x=16, w=16, s=16, z=16, y=16):
    P = ctypes.c_void_p
    return lib.wq_gemm(P(x), P(w), P(s), P(z), P(y), M, N, K, group, bits, P(0), 0, P(0))


def test_gemm_rejects_bad_arguments_on_host(wq):
    lib = wq._lib()
    bad = wq.WQ_ERR_INVALID_ARG
    assert _gemm(lib, bits=5) == bad
    assert _gemm(lib, bits=1) == bad
    assert _gemm(lib, group=96) == bad
    assert _gemm(lib, K=100, group=32) == bad     # K % group != 0
    assert _gemm(lib, M=33) == bad
    assert _gemm(lib, M=-1) == bad
    assert _gemm(lib, N=-3) == bad
    assert _gemm(lib, y=0) == bad                 # null output
    assert _gemm(lib, y=2) == bad                 # misaligned output


def test_empty_problems_are_no_ops(wq):
    lib = wq._lib()
    assert _gemm(lib, M=0, x=0, w=0, s=0, z=0, y=0) == wq.WQ_OK
    assert _gemm(lib, N=0, x=0, w=0, s=0, z=0, y=0) == wq.WQ_OK
    P = ctypes.c_void_p
    assert lib.wq_pack(P(0), P(0), 0, 64, 4, P(0)) == wq.WQ_OK
    assert lib.wq_unpack(P(0), P(0), 5, 0, 4, P(0)) == wq.WQ_OK
    assert lib.wq_dequant(P(0), P(0), P(0), P(0), 0, 128, 128, 4, P(0)) == wq.WQ_OK


def test_elementwise_rejects_bad_arguments(wq):
    lib = wq._lib()
    P = ctypes.c_void_p
    bad = wq.WQ_ERR_INVALID_ARG
    assert lib.wq_pack(P(16), P(16), 4, 64, 5, P(0)) == bad
    assert lib.wq_pack(P(16), P(0), 4, 64, 4, P(0)) == bad
    assert lib.wq_pack(P(16), P(18), 4, 64, 4, P(0)) == bad
    assert lib.wq_dequant(P(16), P(16), P(16), P(16), 4, 100, 32, 4, P(0)) == bad
    assert lib.wq_dequant(P(16), P(0), P(16), P(16), 4, 128, 32, 4, P(0)) == bad
    assert lib.wq_step_run(P(0), 3, P(0), 0, P(0)) == bad
    assert lib.wq_step_graph_create(P(0), 1, P(0), 0, P(0), P(0)) == bad


@pytest.mark.parametrize("U,P", [(1, 1), (7, 7), (10, 4), (5440, 152), (160, 64), (32, 32),
                                 (1000003, 152), (272 * 20, 152), (17, 5)])
def test_stream_k_schedule_partitions_units(wq, U, P):
    assert wq._lib().wq_internal_schedule_check(U, P) == 0


def test_single_projection_grid_rule(wq):
    # at most SMs - 2 CTAs; where the tiles outnumber them and a divisor of the
    # tile count lies within 74 % of that budget, whole tiles per CTA
    g = wq._lib().wq_internal_choose_grid
    assert g(272, 10, 152) == 136      # 34,816 rows: two whole tiles per CTA
    assert g(300, 10, 152) == 150      # 150 divides 300
    assert g(2345, 2, 152) == 150      # no divisor of 2345 in [111, 150]
    assert g(40, 34, 152) == 150       # fewer tiles than CTAs: the budget
    assert g(8, 34, 152) == 64         # at most 8 CTAs per tile
    assert g(3, 1, 152) == 3           # at most one CTA per unit
    assert g(272, 10, 2) == 1


def _phase_grid(wq, T, I, uniform, U, budget=150, nc=16, act=0):
    P, k = ctypes.c_int(0), ctypes.c_int(0)
    assert wq._lib().wq_internal_phase_grid(T, I, uniform, U, budget, nc, act, ctypes.byref(P),
                                            ctypes.byref(k)) == 0
    return P.value, k.value


def test_phase_grid_rule(wq):
    # the decode layer's phases on a 150-CTA budget
    assert _phase_grid(wq, 56, 10, 1, 560) == (112, 2)    # q, k, v: two CTAs per tile, clustered
    assert _phase_grid(wq, 40, 10, 1, 400) == (120, 0)    # o: three per tile, not clustered
    assert _phase_grid(wq, 272, 10, 1, 2720) == (136, 0)  # gate/up: two whole tiles per CTA
    assert _phase_grid(wq, 40, 34, 1, 1360) == (120, 0)   # down
    # no cluster where a rank would get no unit, for the 32-row build, with the
    # activation epilogue, or with unequal tiles (then no alignment either)
    assert _phase_grid(wq, 40, 2, 1, 80) == (80, 2)
    assert _phase_grid(wq, 40, 1, 1, 40) == (40, 0)
    assert _phase_grid(wq, 56, 10, 1, 560, nc=32) == (112, 0)
    assert _phase_grid(wq, 56, 10, 1, 560, act=1) == (112, 0)
    assert _phase_grid(wq, 56, 10, 0, 500) == (150, 0)
    # no k CTAs per tile within 74 % of the budget
    assert _phase_grid(wq, 100, 10, 1, 1000) == (150, 0)
    assert _phase_grid(wq, 8, 34, 1, 272) == (144, 0)     # 18 CTAs per tile: no cluster


def test_gemm_rejects_misaligned_operands(wq):
    # x and wq feed TMA boxes: both 16-byte aligned; bf16 scales 2-byte aligned
    lib = wq._lib()
    bad = wq.WQ_ERR_INVALID_ARG
    assert _gemm(lib, x=8) == bad
    assert _gemm(lib, w=20) == bad
    assert _gemm(lib, s=17) == bad
    assert _gemm(lib, x=0) == bad    # null input with K > 0
    assert _gemm(lib, z=0) == bad


def test_swiglu_needs_gate_up_pairs(wq):
    # rows 2j and 2j + 1 are gate and up of feature j: N must be even
    lib = wq._lib()
    P = ctypes.c_void_p
    odd = lib.wq_gemm_swiglu(P(16), P(16), P(16), P(16), P(16), 4, 9, 128, 128, 4, P(0), 0, P(0))
    assert odd == wq.WQ_ERR_INVALID_ARG
    assert lib.wq_gemm_swiglu(P(16), P(16), P(16), P(16), P(16), 0, 8, 128, 128, 4, P(0), 0,
                              P(0)) == wq.WQ_OK  # empty


def _descs(wq, afters, epilogue=0, N=256):
    arr = (wq.ProjDesc * len(afters))()
    for i, a in enumerate(afters):
        arr[i] = wq.ProjDesc(16, 16, 16, 16, 16, 4, N, 128, 128, 4, a, epilogue)
    return ctypes.cast(arr, ctypes.c_void_p), len(afters)


@pytest.mark.parametrize("afters", [[-1, 1], [0, 2, -1], [-2], [-1, 0, 5]],
                         ids=["self", "forward", "below-minus-one", "past-end"])
def test_step_rejects_bad_dependencies(wq, afters):
    # a projection may only wait for an earlier one (or none: -1)
    lib = wq._lib()
    P = ctypes.c_void_p
    d, n = _descs(wq, afters)
    for flags in (0, wq.WQ_STEP_FUSED):
        assert lib.wq_step_run_ex(d, n, flags, P(16), 1 << 20, P(0)) == wq.WQ_ERR_INVALID_ARG
    g = P(0)
    assert lib.wq_step_graph_create_ex(d, n, 0, P(16), 1 << 20, P(0),
                                       ctypes.byref(g)) == wq.WQ_ERR_INVALID_ARG


def test_step_rejects_bad_flags_and_epilogues(wq):
    lib = wq._lib()
    P = ctypes.c_void_p
    d, n = _descs(wq, [-1, 0])
    assert lib.wq_step_run_ex(d, n, 0x10, P(16), 1 << 20, P(0)) == wq.WQ_ERR_INVALID_ARG
    # per-phase launches only exist as a variant of the fused mode
    assert lib.wq_step_run_ex(d, n, wq.WQ_STEP_PHASES, P(16), 1 << 20, P(0)) == wq.WQ_ERR_INVALID_ARG
    g = P(0)
    assert lib.wq_step_graph_create_ex(d, n, wq.WQ_STEP_PHASES, P(16), 1 << 20, P(0),
                                       ctypes.byref(g)) == wq.WQ_ERR_INVALID_ARG
    d, n = _descs(wq, [-1], epilogue=7)
    assert lib.wq_step_run_ex(d, n, 0, P(16), 1 << 20, P(0)) == wq.WQ_ERR_INVALID_ARG
    d, n = _descs(wq, [-1], epilogue=wq.WQ_EPI_SWIGLU, N=255)  # odd gate/up width
    assert lib.wq_step_run_ex(d, n, 0, P(16), 1 << 20, P(0)) == wq.WQ_ERR_INVALID_ARG
