"""Wider row stacks, 17 to 32 rows of X (eight agents with their draft rows,
or decode rows with a chunk of prefill): the 32-row build of the kernel
against the oracle, bitwise batch invariance against the 16-row build, the
fused step and the gate/up activation at those widths.  All calls go through
the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synth
from wqtest import (ARITH_TOL, REL_TOL, check_activation, dev, oracle_gemm, rel_err,
                    to_dev_host_inputs)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _wq():
    import weight_only_bit_wq_gb300 as wq
    return wq


FORMATS = [(4, 128), (4, 64), (4, 32), (3, 128), (3, 64), (3, 32), (2, 128), (2, 64), (2, 32)]
SHAPES = [(17, 300, 1280), (24, 130, 1920), (32, 257, 2560), (29, 128, 640)]


@pytest.mark.parametrize("fmt", FORMATS, ids=lambda f: f"b{f[0]}g{f[1]}")
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_wide_gemm_matches_oracle(fmt, M, N, K):
    bits, G = fmt
    p = synth.Projection("w", M, N, K, bits, G, 1300 + M + N + bits, s_range=(0.005, 0.04),
                         outlier_frac=0.01)
    w, x, d = to_dev_host_inputs(p)
    y = _wq().wq_gemm(d["x"], d["wq"], d["s"], d["z"], N, G, bits)
    err = rel_err(y.cpu().numpy(), oracle_gemm(p, w, x))
    assert err <= REL_TOL and err <= ARITH_TOL, err


@pytest.mark.parametrize("fmt", [(4, 128), (3, 128), (2, 32)], ids=lambda f: f"b{f[0]}g{f[1]}")
def test_wide_rows_equal_narrow_calls_bitwise(fmt):
    # rows of a 32-row call equal the same rows from 16-row and 1-row calls,
    # which run the 16-row build
    bits, G = fmt
    M, N, K = 32, 640, 2560
    p = synth.Projection("wb", M, N, K, bits, G, 1400)
    w, x, d = to_dev_host_inputs(p)
    wq = _wq()
    y = wq.wq_gemm(d["x"], d["wq"], d["s"], d["z"], N, G, bits).cpu().numpy().view(np.uint32)
    y16 = wq.wq_gemm(d["x"][:16].contiguous(), d["wq"], d["s"], d["z"], N, G, bits)
    assert (y16.cpu().numpy().view(np.uint32) == y[:16]).all()
    y20 = wq.wq_gemm(d["x"][:20].contiguous(), d["wq"], d["s"], d["z"], N, G, bits)
    assert (y20.cpu().numpy().view(np.uint32) == y[:20]).all()
    for m in (0, 17, 31):
        ym = wq.wq_gemm(d["x"][m:m + 1].contiguous(), d["wq"], d["s"], d["z"], N, G, bits)
        assert (ym.cpu().numpy().view(np.uint32)[0] == y[m]).all(), m


@pytest.mark.parametrize("name,M", [("C3", 24), ("C4a", 32), ("C4b", 20)])
def test_wide_full_size_sampled_rows(name, M):
    import dataclasses
    p = dataclasses.replace(synth.CONFIGS[name], M=M, x_row_seeds=None)
    q, s, z = synth.gen_weights_torch(p, dev())
    wq = _wq()
    wqw = wq.wq_pack(q, p.bits)
    del q
    x = synth.gen_x(p)
    y = wq.wq_gemm(torch.from_numpy(x.view(np.int16)).to(dev()), wqw, s, z, p.N, p.group,
                   p.bits).cpu().numpy()
    rng = np.random.default_rng(5)
    rows = np.unique(np.concatenate([[0, 127, 128, p.N - 1], rng.integers(0, p.N, 64)]))
    ws = synth.gen_weights(p, rows=rows)
    y_ref = oracle.gemm_f64(x, oracle.pack(ws["q"], p.bits), ws["s"], ws["z"], p.K, p.group,
                            p.bits)
    err = rel_err(y[:, rows], y_ref)
    assert err <= REL_TOL and err <= ARITH_TOL, err


def test_wide_swiglu_matches_oracle():
    M, N, K, bits, G = 27, 1280, 2560, 4, 128
    p = synth.Projection("wgu", M, N, K, bits, G, 1500)
    w, x, d = to_dev_host_inputs(p)
    out = _wq().wq_gemm_swiglu(d["x"], d["wq"], d["s"], d["z"], N, G, bits)
    got = out.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    assert got.shape == (M, N // 2)
    check_activation(got, oracle_gemm(p, w, x))


@pytest.mark.parametrize("deps", [False, True], ids=["independent", "layer-chain"])
def test_wide_fused_step_matches_oracle(deps):
    # a miniature decode layer twice at 24 rows, mixed with an 8-row
    # projection that shares the 32-row launch
    wq = _wq()
    shapes = [(640, 640), (640, 128), (640, 128), (640, 640), (640, 1792), (896, 640)]
    projs = []
    for i, (K, N) in enumerate(shapes * 2):
        M = 8 if i == 1 else 24
        p = synth.Projection(f"ws{i}", M, N, K, 4, 128, 1600, index=i)
        w, x, d = to_dev_host_inputs(p)
        d["y"] = torch.empty((M, N), dtype=torch.float32, device=dev())
        projs.append((p, w, x, d))
    after = [-1, -1, -1, 2, 3, 4, 5, 5, 5, 8, 9, 10] if deps else [-1] * 12
    descs = wq.make_descs([dict(x=d["x"], wq=d["wq"], scales=d["s"], zeros=d["z"], y=d["y"],
                                M=p.M, N=p.N, K=p.K, group=p.group, bits=p.bits, after=after[i])
                           for i, (p, w, x, d) in enumerate(projs)])
    ws = wq.new_step_workspace(descs, wq.WQ_STEP_FUSED)
    for _ in range(2):
        for p, w, x, d in projs:
            d["y"].fill_(float("nan"))
        wq.wq_step_run(descs, ws, flags=wq.WQ_STEP_FUSED)
        torch.cuda.synchronize()
        wq.wq_check_workspace(ws)
        for p, w, x, d in projs:
            err = rel_err(d["y"].cpu().numpy(), oracle_gemm(p, w, x))
            assert err <= REL_TOL and err <= ARITH_TOL, (p.name, err)
