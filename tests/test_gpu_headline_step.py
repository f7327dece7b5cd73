"""The benchmarked decode step at full size: 64 layers x (q, k, v, o, gate/up,
down) with the real shapes (K = 5120 / 17408; N = 5120, 1024, 1024, 5120,
34816, 5120), 4-bit codes in groups of 128, run as ONE fused persistent launch
that honours the layer chain (q, k, v after the previous layer's down; o after
v; gate/up after o; down after gate/up) -- the launch the benchmark times.

Every one of the 384 projections is checked element by element against the
fp64 oracle on sampled weight rows (tile edges, the first and last rows, and
random rows; the oracle recomputes those rows from the same seeded generator),
at 16 rows (the benchmark's row count), 1 row and 24 rows (the 32-row kernel
build).  Rows are bitwise equal across the three row counts (batch
invariance: OpenJet news page, "新提示不会让所有人停摆").  The sequential mode
(one launch per projection) and the per-phase mode (one launch per dependency
phase, the bench's headline) are checked against the oracle on the same rows;
they split each tile's K range differently from the fused launch, so the modes
agree to rounding, not bit for bit.  The per-phase mode is also bitwise
batch-invariant (16 rows against 1).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from wqtest import ARITH_TOL, REL_TOL, dev, rel_err

pytestmark = pytest.mark.gpu

LAYERS = synth.STEP_LAYERS
ROW_COUNTS = (16, 1, 24)
MAX_ROWS = max(ROW_COUNTS)


def layer_after(n):
    """`after` of projection i in the layer chain (-1 for the first layer's q, k, v)."""
    out = []
    for i in range(n):
        base, j = i - i % 6, i % 6
        out.append(base - 1 if j < 3 else base + j - 1)
    return out


def sample_rows(N, seed):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 31, 32, 127, 128, 255, 256, N // 2, N - 129, N - 128, N - 1]
    rows = np.unique(np.concatenate([np.array(fixed), rng.integers(0, N, 12)]))
    return rows[(rows >= 0) & (rows < N)]


@pytest.fixture(scope="module")
def stack():
    import __graft_entry__
    __graft_entry__.build()
    import weight_only_bit_wq_gb300 as wq
    projs = synth.step_projections(MAX_ROWS, LAYERS)
    weights = []
    for p in projs:
        q, s, z = synth.gen_weights_torch(p, dev())
        weights.append((wq.wq_pack(q, p.bits), s, z))
        del q
    torch.cuda.synchronize()
    xs = [synth.gen_x(p) for p in projs]  # [MAX_ROWS][K] bf16 bits; row m never depends on M
    after = layer_after(len(projs))
    # oracle on the sampled rows of every projection, for all MAX_ROWS rows of X
    ref = []
    for i, p in enumerate(projs):
        rows = sample_rows(p.N, 1000 + i)
        w = synth.gen_weights(p, rows=rows)
        y = oracle.gemm_f64(xs[i], oracle.pack(w["q"], p.bits), w["s"], w["z"], p.K, p.group, p.bits)
        ref.append((rows, y))  # y: [MAX_ROWS][len(rows)]
    yield dict(projs=projs, weights=weights, xs=xs, after=after, ref=ref)
    del weights
    torch.cuda.empty_cache()


def _run(wq, st, M, flags):
    """One step at M rows; returns each projection's Y on the host."""
    descs, ys = [], []
    for i, (p, (wqw, s, z)) in enumerate(zip(st["projs"], st["weights"])):
        x = torch.from_numpy(np.ascontiguousarray(st["xs"][i][:M]).view(np.int16)).to(dev())
        y = torch.full((M, p.N), float("nan"), dtype=torch.float32, device=dev())
        ys.append(y)
        descs.append(dict(x=x, wq=wqw, scales=s, zeros=z, y=y, M=M, N=p.N, K=p.K, group=p.group,
                          bits=p.bits, after=st["after"][i]))
    cd = wq.make_descs(descs)
    ws = wq.new_step_workspace(cd, flags)
    wq.wq_step_run(cd, ws, flags=flags)
    torch.cuda.synchronize()
    wq.wq_check_workspace(ws)
    out = [y.cpu().numpy() for y in ys]
    del descs, ys, ws
    return out


def _check_oracle(st, ys, M, what):
    worst = 0.0
    for i, (p, y) in enumerate(zip(st["projs"], ys)):
        rows, y_ref = st["ref"][i]
        assert np.isfinite(y).all(), (what, p.name)
        err = rel_err(y[:, rows], y_ref[:M])
        assert err <= REL_TOL and err <= ARITH_TOL, (what, M, p.name, err)
        worst = max(worst, err)
    return worst


def test_fused_layer_chain_full_size_all_projections(stack):
    import weight_only_bit_wq_gb300 as wq
    res = {}
    for M in ROW_COUNTS:
        res[M] = _run(wq, stack, M, wq.WQ_STEP_FUSED)
        _check_oracle(stack, res[M], M, "fused")
    # batch invariance across row counts and kernel builds (16- and 32-row)
    for i in range(len(stack["projs"])):
        a16, a1, a24 = res[16][i], res[1][i], res[24][i]
        assert np.array_equal(a1[0].view(np.uint32), a16[0].view(np.uint32)), i
        assert np.array_equal(a24[:16].view(np.uint32), a16.view(np.uint32)), i


def test_sequential_and_phased_full_size_all_projections(stack):
    import weight_only_bit_wq_gb300 as wq
    ys = _run(wq, stack, 16, 0)
    _check_oracle(stack, ys, 16, "sequential")
    # one launch per dependency phase (the headline mode), at 16 rows and 1 row
    flags = wq.WQ_STEP_FUSED | wq.WQ_STEP_PHASES
    p16 = _run(wq, stack, 16, flags)
    _check_oracle(stack, p16, 16, "phased")
    p1 = _run(wq, stack, 1, flags)
    _check_oracle(stack, p1, 1, "phased")
    for i, (a, b) in enumerate(zip(p16, p1)):
        assert np.array_equal(b[0].view(np.uint32), a[0].view(np.uint32)), i
