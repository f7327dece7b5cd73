"""Decode-step driver: back-to-back projections, direct and graph-captured,
bit-identical to individual wq_gemm calls and within tolerance of the oracle."""
import numpy as np
import pytest
import torch

import synth
from wqtest import ARITH_TOL, REL_TOL, dev, oracle_gemm, rel_err, to_dev_host_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _stack(M):
    # a two-layer miniature of the projection stack, mixed bit widths
    shapes = [(640, 512, 4, 128), (640, 128, 4, 128), (640, 640, 2, 64), (1280, 640, 4, 64),
              (640, 1536, 4, 128), (1536, 640, 2, 32)] * 2
    projs = []
    for i, (K, N, bits, G) in enumerate(shapes):
        p = synth.Projection(f"p{i}", M, N, K, bits, G, 300, index=i)
        w, x, d = to_dev_host_inputs(p)
        d["y"] = torch.empty((M, N), dtype=torch.float32, device=dev())
        projs.append((p, w, x, d))
    return projs


@pytest.mark.parametrize("M", [1, 12])
def test_step_run_and_graph_match_single_calls(M):
    import weight_only_bit_wq_gb300 as wq
    projs = _stack(M)
    ref = []
    for p, w, x, d in projs:
        ref.append(wq.wq_gemm(d["x"], d["wq"], d["s"], d["z"], p.N, p.group, p.bits).cpu().numpy())
    descs = wq.make_descs([dict(x=d["x"], wq=d["wq"], scales=d["s"], zeros=d["z"], y=d["y"], M=p.M,
                                N=p.N, K=p.K, group=p.group, bits=p.bits) for p, w, x, d in projs])
    ws = wq.new_workspace(16, 1536, 1280, 32, 2)
    wq.wq_step_run(descs, ws)
    torch.cuda.synchronize()
    for (p, w, x, d), r in zip(projs, ref):
        assert (d["y"].cpu().numpy().view(np.uint32) == r.view(np.uint32)).all()
        d["y"].fill_(float("nan"))
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    g = wq.StepGraph(descs, ws, stream=stream)
    for _ in range(2):
        g.launch(stream=stream)
    stream.synchronize()
    for (p, w, x, d), r in zip(projs, ref):
        assert (d["y"].cpu().numpy().view(np.uint32) == r.view(np.uint32)).all()
    g.close()
    p, w, x, d = projs[3]
    err = rel_err(d["y"].cpu().numpy(), oracle_gemm(p, w, x))
    assert err <= REL_TOL and err <= ARITH_TOL
    wq.wq_check_workspace(ws)
