"""GPU parity of wq_paged_attention against the fp64 oracle: grouped-query
heads, pages shared by a common prefix and placed in shuffled order, draft
rows seeing only earlier positions, long sequences split across CTAs, bitwise
determinism, and a table entry outside the pool reported in the error word.
All calls go through the C ABI."""
import ctypes
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from wqtest import dev

pytestmark = pytest.mark.gpu

TOL = 1e-4  # fp32 accumulation over <= 4096 positions, relative to max|out|


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _to_dev(d):
    t = {}
    for k in ("kc", "vc"):
        t[k] = torch.from_numpy(d[k]).to(dev())
    for k in ("kd", "vd", "q"):
        t[k] = torch.from_numpy(d[k].view(np.int16)).to(dev())
    for k in ("page_table", "seq_len", "row_seq", "row_pos"):
        t[k] = torch.from_numpy(np.ascontiguousarray(d[k], dtype=np.int32)).to(dev())
    return t


def _cuda_cores(wq):
    # the CUDA-core kernel (fp32 FMA), exported for cross-checks only
    fn = wq._lib().wq_internal_paged_attention_cuda_cores
    fn.argtypes = wq._lib().wq_paged_attention.argtypes
    fn.restype = ctypes.c_int
    return fn


def _run(d, max_seq_len=None, workspace=None, cuda_cores=False):
    import weight_only_bit_wq_gb300 as wq
    t = _to_dev(d)
    msl = int(d["seq_len"].max()) if max_seq_len is None else max_seq_len
    if not cuda_cores:
        out = wq.wq_paged_attention(t["q"], t["kc"], t["kd"], t["vc"], t["vd"], t["page_table"],
                                    t["seq_len"], t["row_seq"], t["row_pos"], msl,
                                    workspace=workspace)
    else:
        rows, Hq, D = t["q"].shape
        pages, Hkv, T, _ = t["kc"].shape
        B, max_pages = t["page_table"].shape
        out = torch.empty((rows, Hq, D), dtype=torch.float32, device=dev())
        n = int(wq._lib().wq_paged_attention_workspace_bytes(rows, Hq, Hkv, B, msl))
        ws = torch.zeros(max(n, 256), dtype=torch.uint8, device=dev())
        p = lambda x: ctypes.c_void_p(x.data_ptr())
        st = _cuda_cores(wq)(p(t["q"]), p(t["kc"]), p(t["kd"]), p(t["vc"]), p(t["vd"]),
                             p(t["page_table"]), max_pages, p(t["seq_len"]), B, p(t["row_seq"]),
                             p(t["row_pos"]), rows, msl, Hq, Hkv, D, T, pages, p(out), p(ws),
                             ws.numel(), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert st == 0
    torch.cuda.synchronize()
    return out.cpu().numpy()


def _oracle(d):
    return oracle.paged_attention_f64(d["q"], d["kc"], d["kd"], d["vc"], d["vd"], d["page_table"],
                                      d["seq_len"], d["row_seq"], d["row_pos"])


CASES = [
    synth.PagedAttention("a1", (37, 100, 64), 3, 8, 2, 128, 16, 21, shared_prefix=32),
    synth.PagedAttention("a2", (5, 3, 300, 1024), 3, 40, 8, 128, 64, 22, shared_prefix=0),
    synth.PagedAttention("a3", (2048, 700), 1, 16, 16, 128, 32, 23, shared_prefix=512),
    synth.PagedAttention("a4", (4096, 33, 129, 3000), 3, 10, 2, 128, 64, 24, shared_prefix=0),
    # more query vectors per key/value head than one pass holds: 4 rows x 5
    # heads (passes of 15 and 5), and 7 rows x 16 heads (one row per pass)
    synth.PagedAttention("a5", (300, 77, 1500), 4, 20, 4, 128, 32, 25, shared_prefix=64),
    synth.PagedAttention("a6", (129, 40), 7, 16, 1, 128, 16, 26, shared_prefix=0),
    # 17-token pages (positions straddle pages at every offset), a one-token
    # sequence, and a shared 17-token prefix
    synth.PagedAttention("a7", (50, 1, 17, 260), 1, 6, 3, 128, 17, 27, shared_prefix=0),
    synth.PagedAttention("a8", (34, 51, 90), 2, 6, 3, 128, 17, 28, shared_prefix=17),
]


@pytest.mark.parametrize("cuda_cores", [False, True], ids=["tensor-cores", "cuda-cores"])
@pytest.mark.parametrize("p", CASES, ids=lambda p: p.name)
def test_attention_matches_oracle(p, cuda_cores):
    d = synth.gen_paged_attention(p)
    got = _run(d, cuda_cores=cuda_cores)
    ref = _oracle(d)
    assert np.abs(got - ref).max() <= TOL * np.abs(ref).max()


def _scaled_queries(d, factor):
    # bf16 queries times a power of two (exact)
    q = (d["q"].astype(np.uint32) << 16).view(np.float32) * np.float32(factor)
    return (q.view(np.uint32) >> 16).astype(np.uint16)


@pytest.mark.parametrize("scale_range,q_factor", [((1e-5, 8.0), 1.0), ((0.002, 0.02), 32.0),
                                                  ((1e-4, 1e-3), 2.0 ** -7)],
                         ids=["wide-scales", "peaked", "small"])
def test_attention_extreme_ranges(scale_range, q_factor):
    # value scales over six decades, sharply peaked softmax (large queries),
    # and small queries with small scales: the binary16 operands of the
    # tensor-core kernel keep their bits through the power-of-two scalings
    p = dataclasses.replace(CASES[0], scale_range=scale_range)
    d = dict(synth.gen_paged_attention(p))
    d["q"] = _scaled_queries(d, q_factor)
    ref = _oracle(d)
    for cc in (False, True):
        got = _run(d, cuda_cores=cc)
        assert np.abs(got - ref).max() <= TOL * np.abs(ref).max(), cc


def test_attention_is_deterministic_and_placement_free():
    p = CASES[0]
    d = synth.gen_paged_attention(p)
    a = _run(d)
    b = _run(d)
    assert (a.view(np.uint32) == b.view(np.uint32)).all()
    # the same pages elsewhere in the pool give the same bits
    pages = d["kc"].shape[0]
    perm = np.random.default_rng(9).permutation(pages)
    moved = dict(d)
    for k in ("kc", "kd", "vc", "vd"):
        arr = np.empty_like(d[k])
        arr[perm] = d[k]
        moved[k] = arr
    moved["page_table"] = perm[d["page_table"]].astype(np.int32)
    c = _run(moved)
    assert (a.view(np.uint32) == c.view(np.uint32)).all()


@pytest.mark.parametrize("fault", ["page-outside-pool", "position-past-sequence"])
def test_bad_table_is_reported(fault):
    # the kernels check every table entry and position before reading: the
    # error word says 2 and the affected rows read nothing
    import weight_only_bit_wq_gb300 as wq
    p = CASES[0]
    d = dict(synth.gen_paged_attention(p))
    if fault == "page-outside-pool":
        d["page_table"] = d["page_table"].copy()
        d["page_table"][1, 2] = d["kc"].shape[0] + 5
    else:
        d["row_pos"] = d["row_pos"].copy()
        d["row_pos"][0] = int(d["seq_len"][d["row_seq"][0]]) + 3
    n = int(wq._lib().wq_paged_attention_workspace_bytes(len(d["row_seq"]), p.Hq, p.Hkv,
                                                          len(p.seq_lens), int(d["seq_len"].max())))
    ws = torch.zeros(n, dtype=torch.uint8, device=dev())
    got = _run(d, workspace=ws)
    assert int(ws[:4].view(torch.int32).item()) == 2
    assert np.isfinite(got).all()
    if fault == "position-past-sequence":
        assert (got[0] == 0).all()


# The workload the benchmark times: four agents x 32768 positions of their own
# sequences (a 4096-token prefix stored once and shared), three query rows each,
# 40 query heads over 8 key/value heads, 64-token pages.
BENCH_CASE = synth.PagedAttention("bench", (32768,) * 4, 3, 40, 8, 128, 64, 31,
                                  shared_prefix=4096)


def test_bench_workload_sampled_rows():
    # full size, as timed; the oracle computes sampled rows from a host copy of
    # the device pool (the device generator gives the numpy generator's bits)
    import weight_only_bit_wq_gb300 as wq
    p = BENCH_CASE
    t = synth.gen_paged_attention_torch(p, dev())
    out = wq.wq_paged_attention(t["q"], t["kc"], t["kd"], t["vc"], t["vd"], t["page_table"],
                                t["seq_len"], t["row_seq"], t["row_pos"], max(p.seq_lens))
    torch.cuda.synchronize()
    got = out.cpu().numpy()
    host = {k: v.cpu().numpy() for k, v in t.items()}
    rows = np.array([0, 4, 8, 11])  # first and last rows, each agent once
    ref = oracle.paged_attention_f64(host["q"][rows].view(np.uint16), host["kc"],
                                     host["kd"].view(np.uint16), host["vc"],
                                     host["vd"].view(np.uint16), host["page_table"],
                                     host["seq_len"], host["row_seq"][rows], host["row_pos"][rows])
    assert np.abs(got[rows] - ref).max() <= TOL * np.abs(ref).max()
