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


def _descs(wq, projs, after=None):
    return wq.make_descs([dict(x=d["x"], wq=d["wq"], scales=d["s"], zeros=d["z"], y=d["y"], M=p.M,
                               N=p.N, K=p.K, group=p.group, bits=p.bits,
                               after=-1 if after is None else after[i])
                          for i, (p, w, x, d) in enumerate(projs)])


def _layer_after(n):
    # the dependency chain of a decode layer, repeated: q, k, v read the layer
    # input (the previous down), o waits for q, k, v, gate/up for o, down for gate/up
    after = []
    for i in range(n):
        j = i % 6
        base = i - j
        after.append({0: base - 1, 1: base - 1, 2: base - 1, 3: base + 2, 4: base + 3,
                      5: base + 4}[j] if i >= 1 else -1)
    return [a if a < i else -1 for i, a in enumerate(after)]


def _uniform_stack(M, bits, G, layers=2):
    # a miniature decode layer (q, k, v, o, gate/up, down) in one format, so a
    # fused launch holds whole layers and their dependency chain
    shapes = [(640, 640), (640, 128), (640, 128), (640, 640), (640, 1792), (896, 640)]
    projs = []
    for i, (K, N) in enumerate(shapes * layers):
        p = synth.Projection(f"u{i}", M, N, K, bits, G, 400, index=i)
        w, x, d = to_dev_host_inputs(p)
        d["y"] = torch.empty((M, N), dtype=torch.float32, device=dev())
        projs.append((p, w, x, d))
    return projs


FUSED_FORMATS = [(4, 128), (3, 128), (2, 64), (4, 32), (3, 64), (2, 128)]


@pytest.mark.parametrize("fmt", FUSED_FORMATS, ids=lambda f: f"b{f[0]}g{f[1]}")
@pytest.mark.parametrize("deps", [False, True], ids=["independent", "layer-chain"])
def test_fused_uniform_stack_matches_oracle(fmt, deps):
    import weight_only_bit_wq_gb300 as wq
    projs = _uniform_stack(7, *fmt)
    after = _layer_after(len(projs)) if deps else None
    descs = _descs(wq, projs, after)
    ws = wq.new_step_workspace(descs, wq.WQ_STEP_FUSED)
    refs = [oracle_gemm(p, w, x) for p, w, x, d in projs]
    # one launch for the run, then one launch per phase (each launch with its own
    # grid, so the modes agree to rounding); each mode twice: the repeat checks
    # that counters were left clean and is bitwise equal
    for flags in (wq.WQ_STEP_FUSED, wq.WQ_STEP_FUSED | wq.WQ_STEP_PHASES):
        first = None
        for _ in range(2):
            for p, w, x, d in projs:
                d["y"].fill_(float("nan"))
            wq.wq_step_run(descs, ws, flags=flags)
            torch.cuda.synchronize()
            wq.wq_check_workspace(ws)
            ys = [d["y"].cpu().numpy() for p, w, x, d in projs]
            if first is None:
                first = ys
                for (p, w, x, d), y, r in zip(projs, ys, refs):
                    err = rel_err(y, r)
                    assert err <= REL_TOL and err <= ARITH_TOL, (flags, p.name, err)
            else:
                for (p, w, x, d), y, r in zip(projs, ys, first):
                    assert np.array_equal(y.view(np.uint32), r.view(np.uint32)), (flags, p.name)


def _chain_outputs(wq, projs, M, flags, ws=None):
    descs = wq.make_descs([dict(x=d["x"][:M], wq=d["wq"], scales=d["s"], zeros=d["z"],
                                y=d["y"][:M], M=M, N=p.N, K=p.K, group=p.group, bits=p.bits,
                                after=i - 1) for i, (p, w, x, d) in enumerate(projs)])
    if ws is None:
        ws = wq.new_step_workspace(descs, wq.WQ_STEP_FUSED)
    for p, w, x, d in projs:
        d["y"].fill_(float("nan"))
    wq.wq_step_run(descs, ws, flags=flags)
    torch.cuda.synchronize()
    wq.wq_check_workspace(ws)
    return [d["y"][:M].cpu().numpy() for p, w, x, d in projs], ws


@pytest.mark.parametrize("fmt", [(4, 128), (3, 128), (2, 64), (4, 32)], ids=lambda f: f"b{f[0]}g{f[1]}")
def test_phased_cluster_fixup_matches_oracle(fmt):
    # Per-phase launches whose grid gives each tile two CTAs (here the 56-tile
    # projection on a 150-CTA budget) run as one cluster per tile and add the
    # split-K sums through shared memory (formats whose build has no room for
    # the cluster buffer, and the 40-tile projections with three CTAs per
    # tile, take the global-memory path).
    # A chain of one projection per phase, against the oracle, bitwise across
    # repeats and across row counts.
    import weight_only_bit_wq_gb300 as wq
    bits, G = fmt
    shapes = [(2048, 5120), (5120, 5120), (1536, 7168), (17408, 5120)]  # (K, N)
    M = 5
    projs = []
    for i, (K, N) in enumerate(shapes):
        p = synth.Projection(f"c{i}", M, N, K, bits, G, 500, index=i)
        w, x, d = to_dev_host_inputs(p)
        d["y"] = torch.empty((M, N), dtype=torch.float32, device=dev())
        projs.append((p, w, x, d))
    flags = wq.WQ_STEP_FUSED | wq.WQ_STEP_PHASES
    ys, ws = _chain_outputs(wq, projs, M, flags)
    for (p, w, x, d), y in zip(projs, ys):
        err = rel_err(y, oracle_gemm(p, w, x))
        assert err <= REL_TOL and err <= ARITH_TOL, (p.name, err)
    again, _ = _chain_outputs(wq, projs, M, flags, ws)
    one, _ = _chain_outputs(wq, projs, 1, flags, ws)
    for a, b, c in zip(ys, again, one):
        assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
        assert np.array_equal(a[:1].view(np.uint32), c.view(np.uint32))


def test_fused_workspace_serves_smaller_and_larger_sets():
    # The workspace layout depends on the descriptor set (the completion
    # counters sit after the split-K counters of the set's tiles), so a smaller
    # set's completion counters occupy a larger set's split-K counters: every
    # launch must leave them zeroed.  One layer, then two, then one again, on
    # one workspace sized for the two.
    import weight_only_bit_wq_gb300 as wq
    projs = _uniform_stack(5, 4, 128, layers=2)
    refs = [oracle_gemm(p, w, x) for p, w, x, d in projs]
    full = _descs(wq, projs, _layer_after(len(projs)))
    part = _descs(wq, projs[:6], _layer_after(6))
    ws = wq.new_step_workspace(full, wq.WQ_STEP_FUSED)
    for descs, n in ((part, 6), (full, 12), (part, 6), (full, 12)):
        for p, w, x, d in projs:
            d["y"].fill_(float("nan"))
        wq.wq_step_run(descs, ws, flags=wq.WQ_STEP_FUSED)
        torch.cuda.synchronize()
        wq.wq_check_workspace(ws)
        for (p, w, x, d), r in zip(projs[:n], refs[:n]):
            err = rel_err(d["y"].cpu().numpy(), r)
            assert err <= REL_TOL and err <= ARITH_TOL, (n, p.name, err)


@pytest.mark.parametrize("deps", [False, True], ids=["independent", "layer-chain"])
@pytest.mark.parametrize("M", [1, 12])
def test_fused_step_matches_oracle(M, deps):
    import weight_only_bit_wq_gb300 as wq
    projs = _stack(M)
    after = _layer_after(len(projs)) if deps else None
    descs = _descs(wq, projs, after)
    ws = wq.new_step_workspace(descs, wq.WQ_STEP_FUSED)
    for _ in range(2):  # the second run checks that counters were left clean
        for p, w, x, d in projs:
            d["y"].fill_(float("nan"))
        wq.wq_step_run(descs, ws, flags=wq.WQ_STEP_FUSED)
        torch.cuda.synchronize()
        wq.wq_check_workspace(ws)
        for p, w, x, d in projs:
            err = rel_err(d["y"].cpu().numpy(), oracle_gemm(p, w, x))
            assert err <= REL_TOL and err <= ARITH_TOL, (p.name, err)


def test_fused_graph_replays_bitwise_and_rows_are_batch_invariant():
    import weight_only_bit_wq_gb300 as wq
    M = 4
    projs = _uniform_stack(M, 4, 128)
    after = _layer_after(len(projs))
    descs = _descs(wq, projs, after)
    ws = wq.new_step_workspace(descs, wq.WQ_STEP_FUSED)
    wq.wq_step_run(descs, ws, flags=wq.WQ_STEP_FUSED)
    torch.cuda.synchronize()
    ref = [d["y"].cpu().numpy().copy() for p, w, x, d in projs]
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    g = wq.StepGraph(descs, ws, stream=stream, flags=wq.WQ_STEP_FUSED)
    for _ in range(3):
        for p, w, x, d in projs:
            d["y"].fill_(float("nan"))
        g.launch(stream=stream)
        stream.synchronize()
        for (p, w, x, d), r in zip(projs, ref):
            assert (d["y"].cpu().numpy().view(np.uint32) == r.view(np.uint32)).all(), p.name
    g.close()
    wq.wq_check_workspace(ws)
    # each row alone (M = 1, same projections otherwise) equals its row of the stack
    for row in (0, 3):
        alone = []
        for p, w, x, d in projs:
            xr = d["x"][row:row + 1].contiguous()
            alone.append(dict(x=xr, wq=d["wq"], scales=d["s"], zeros=d["z"],
                              y=torch.empty((1, p.N), dtype=torch.float32, device=dev()),
                              M=1, N=p.N, K=p.K, group=p.group, bits=p.bits))
        for i, a in enumerate(alone):
            a["after"] = after[i]
        d1 = wq.make_descs(alone)
        ws1 = wq.new_step_workspace(d1, wq.WQ_STEP_FUSED)
        wq.wq_step_run(d1, ws1, flags=wq.WQ_STEP_FUSED)
        torch.cuda.synchronize()
        for a, r in zip(alone, ref):
            assert (a["y"].cpu().numpy()[0].view(np.uint32) == r[row].view(np.uint32)).all()


def test_fused_step_bad_dependency_rejected():
    import weight_only_bit_wq_gb300 as wq
    projs = _stack(1)[:3]
    descs = _descs(wq, projs, [-1, 1, 0])  # projection 1 cannot wait for itself
    assert wq.wq_step_workspace_bytes(descs, wq.WQ_STEP_FUSED) == 0
    with pytest.raises(wq.WQError):
        wq.wq_step_run(descs, wq.new_workspace(1, 640, 640, 128, 4), flags=wq.WQ_STEP_FUSED)


def test_sequential_step_with_empty_projections_between_gemms():
    # Sequential mode launches a GEMM that follows another as a programmatic
    # dependent; a projection with K = 0 (Y zero-filled, no kernel) or M = 0
    # (nothing at all) between two GEMMs must break that chain cleanly.
    import weight_only_bit_wq_gb300 as wq
    shapes = [(640, 512, 4, 128), (640, 640, 2, 64), (1280, 640, 4, 64), (896, 1536, 3, 128)]
    projs = []
    for i, (K, N, bits, G) in enumerate(shapes):
        p = synth.Projection(f"e{i}", 5, N, K, bits, G, 500, index=i)
        w, x, d = to_dev_host_inputs(p)
        d["y"] = torch.full((p.M, p.N), float("nan"), dtype=torch.float32, device=dev())
        projs.append((p, w, x, d))
    ref = [wq.wq_gemm(d["x"], d["wq"], d["s"], d["z"], p.N, p.group, p.bits).cpu().numpy()
           for p, w, x, d in projs]
    p0, _, _, d0 = projs[0]
    y_k0 = torch.full((3, 700), float("nan"), dtype=torch.float32, device=dev())
    y_m0 = torch.full((1, 1), float("nan"), dtype=torch.float32, device=dev())
    entries = [dict(x=d["x"], wq=d["wq"], scales=d["s"], zeros=d["z"], y=d["y"], M=p.M, N=p.N,
                    K=p.K, group=p.group, bits=p.bits) for p, w, x, d in projs]
    k0 = dict(x=d0["x"], wq=d0["wq"], scales=d0["s"], zeros=d0["z"], y=y_k0, M=3, N=700, K=0,
              group=128, bits=4)
    m0 = dict(x=d0["x"], wq=d0["wq"], scales=d0["s"], zeros=d0["z"], y=y_m0, M=0, N=1, K=128,
              group=128, bits=4)
    order = [entries[0], entries[1], k0, entries[2], m0, entries[3]]
    descs = wq.make_descs(order)
    ws = wq.new_workspace(16, 1536, 1280, 32, 2)
    for graph in (False, True):
        for p, w, x, d in projs:
            d["y"].fill_(float("nan"))
        y_k0.fill_(float("nan"))
        if graph:
            stream = torch.cuda.Stream()
            stream.wait_stream(torch.cuda.current_stream())
            g = wq.StepGraph(descs, ws, stream=stream)
            g.launch(stream=stream)
            stream.synchronize()
            g.close()
        else:
            wq.wq_step_run(descs, ws)
            torch.cuda.synchronize()
        for (p, w, x, d), r in zip(projs, ref):
            assert (d["y"].cpu().numpy().view(np.uint32) == r.view(np.uint32)).all(), (p.name, graph)
        assert (y_k0.cpu().numpy() == 0).all()
        assert np.isnan(y_m0.cpu().numpy()).all()
    wq.wq_check_workspace(ws)
    p, w, x, d = projs[3]
    err = rel_err(d["y"].cpu().numpy(), oracle_gemm(p, w, x))
    assert err <= REL_TOL and err <= ARITH_TOL
