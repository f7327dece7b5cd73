"""GPU parity of wq_gemm against the fp64 oracle, batch invariance, determinism
and edge cases.  All calls go through the C ABI."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
import synth
from wqtest import ARITH_TOL, REL_TOL, dev, oracle_gemm, proj, rel_err, to_dev_host_inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _wq():
    import weight_only_bit_wq_gb300 as wq
    return wq


FORMATS = [(4, 128), (4, 64), (4, 32), (2, 64), (2, 128), (2, 32), (3, 128), (3, 64), (3, 32)]
SHAPES = [(1, 1, 128), (3, 130, 384), (16, 300, 1280), (8, 257, 2048), (9, 128, 640),
          (12, 513, 4480), (5, 200, 1056)]


def _fid(f):
    return f"b{f[0]}g{f[1]}"


@pytest.mark.parametrize("fmt", FORMATS, ids=_fid)
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_gemm_matches_oracle(fmt, M, N, K):
    bits, G = fmt
    if K % G:
        pytest.skip("K must be a multiple of the group")
    p = synth.Projection("t", M, N, K, bits, G, 1000 + M + N + bits, s_range=(0.005, 0.04),
                         outlier_frac=0.01)
    w, x, d = to_dev_host_inputs(p)
    y = _wq().wq_gemm(d["x"], d["wq"], d["s"], d["z"], N, G, bits)
    y_ref = oracle_gemm(p, w, x)
    err = rel_err(y.cpu().numpy(), y_ref)
    assert err <= REL_TOL
    assert err <= ARITH_TOL, err


@pytest.mark.parametrize("name", ["C1", "C2"])
def test_config_full(name):
    p = synth.CONFIGS[name]
    w, x, d = to_dev_host_inputs(p)
    y = _wq().wq_gemm(d["x"], d["wq"], d["s"], d["z"], p.N, p.group, p.bits)
    err = rel_err(y.cpu().numpy(), oracle_gemm(p, w, x))
    assert err <= REL_TOL and err <= ARITH_TOL, err


def test_c2_rows_alone_equal_stacked_bitwise():
    # each agent's row computed alone is bit-identical to the 4-row stacked call
    p = synth.CONFIGS["C2"]
    w, x, d = to_dev_host_inputs(p)
    wq = _wq()
    y = wq.wq_gemm(d["x"], d["wq"], d["s"], d["z"], p.N, p.group, p.bits).cpu().numpy()
    for r in range(p.M):
        xr = torch.from_numpy(synth.gen_x(p.with_m(r + 1))[r:r + 1].view(np.int16)).to(dev())
        yr = wq.wq_gemm(xr, d["wq"], d["s"], d["z"], p.N, p.group, p.bits).cpu().numpy()
        assert (yr[0].view(np.uint32) == y[r].view(np.uint32)).all(), r


def _device_weights(p):
    q, s, z = synth.gen_weights_torch(p, dev())
    wq = _wq().wq_pack(q, p.bits)
    del q
    return wq, s, z


def _sample_rows(N, n=96, seed=0):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 7, 8, 127, 128, 129, N // 2, N - 129, N - 128, N - 2, N - 1]
    rows = np.unique(np.concatenate([np.array(fixed), rng.integers(0, N, n)]))
    return rows[(rows >= 0) & (rows < N)]


@pytest.mark.parametrize("name", ["C3", "C4a", "C4b", "C4c"])
def test_config_full_size_sampled_rows(name):
    # full-size launch (the benchmarked configuration); the oracle recomputes
    # sampled weight rows from the same seeded generator
    p = synth.CONFIGS[name]
    wqw, s, z = _device_weights(p)
    x = synth.gen_x(p)
    xd = torch.from_numpy(x.view(np.int16)).to(dev())
    y = _wq().wq_gemm(xd, wqw, s, z, p.N, p.group, p.bits).cpu().numpy()
    rows = _sample_rows(p.N)
    ws = synth.gen_weights(p, rows=rows)
    y_ref = oracle.gemm_f64(x, oracle.pack(ws["q"], p.bits), ws["s"], ws["z"], p.K, p.group, p.bits)
    err = rel_err(y[:, rows], y_ref)
    assert err <= REL_TOL and err <= ARITH_TOL, err
    assert np.isfinite(y).all()


def test_fused_qkv_projection_sampled_rows():
    # q, k and v of one layer concatenated along N (5120 + 1024 + 1024 rows)
    # stream as one projection; sampled rows against the oracle
    p = synth.Projection("qkv", 12, 7168, 5120, 4, 128, 11)
    wqw, s, z = _device_weights(p)
    x = synth.gen_x(p)
    xd = torch.from_numpy(x.view(np.int16)).to(dev())
    y = _wq().wq_gemm(xd, wqw, s, z, p.N, p.group, p.bits).cpu().numpy()
    rows = _sample_rows(p.N)
    rows = np.unique(np.concatenate([rows, [5119, 5120, 6143, 6144]]))
    ws = synth.gen_weights(p, rows=rows)
    y_ref = oracle.gemm_f64(x, oracle.pack(ws["q"], p.bits), ws["s"], ws["z"], p.K, p.group, p.bits)
    err = rel_err(y[:, rows], y_ref)
    assert err <= REL_TOL and err <= ARITH_TOL, err


def test_c3_row_subsets_bitwise():
    # rows of the 12-row call equal the same rows computed in 1-, 5- and 9-row calls
    p = synth.CONFIGS["C3"]
    wqw, s, z = _device_weights(p)
    x = torch.from_numpy(synth.gen_x(p).view(np.int16)).to(dev())
    wq = _wq()
    y = wq.wq_gemm(x, wqw, s, z, p.N, p.group, p.bits).cpu().numpy().view(np.uint32)
    for m in (1, 5, 8, 9, 12):
        ym = wq.wq_gemm(x[:m].contiguous(), wqw, s, z, p.N, p.group, p.bits).cpu().numpy().view(np.uint32)
        assert (ym == y[:m]).all(), m
    # a later row alone
    y7 = wq.wq_gemm(x[7:8].contiguous(), wqw, s, z, p.N, p.group, p.bits).cpu().numpy().view(np.uint32)
    assert (y7[0] == y[7]).all()


def test_repeat_calls_and_workspaces_bitwise():
    p = proj("C2", M=7, x_row_seeds=None)
    w, x, d = to_dev_host_inputs(p)
    wq = _wq()
    y1 = wq.wq_gemm(d["x"], d["wq"], d["s"], d["z"], p.N, p.group, p.bits).cpu().numpy()
    ws = wq.new_workspace(p.M, p.N, p.K, p.group, p.bits)
    y2 = wq.wq_gemm(d["x"], d["wq"], d["s"], d["z"], p.N, p.group, p.bits, workspace=ws).cpu().numpy()
    y3 = wq.wq_gemm(d["x"], d["wq"], d["s"], d["z"], p.N, p.group, p.bits, workspace=ws).cpu().numpy()
    assert (y1.view(np.uint32) == y2.view(np.uint32)).all()
    assert (y2.view(np.uint32) == y3.view(np.uint32)).all()
    wq.wq_check_workspace(ws)
    wq.wq_check_workspace()


def test_k_zero_gives_zeros_and_empty_calls():
    wq = _wq()
    d = dev()
    y = torch.full((3, 5), 7.0, device=d)
    x = torch.zeros((3, 0), dtype=torch.int16, device=d)
    wqw = torch.zeros((5, 0), dtype=torch.int32, device=d)
    s = torch.zeros((5, 0), dtype=torch.int16, device=d)
    z = torch.zeros((5, 0), dtype=torch.uint8, device=d)
    wq.wq_gemm(x, wqw, s, z, 5, 128, 4, out=y)
    assert (y.cpu() == 0).all()
    x0 = torch.zeros((0, 128), dtype=torch.int16, device=d)
    y0 = wq.wq_gemm(x0, wqw, s, z, 5, 128, 4)
    assert y0.shape == (0, 5)


def test_extreme_codes_and_zero_points():
    # q - z spans the full signed range [-(2^b - 1), 2^b - 1] with the largest scales
    wq = _wq()
    for bits in (2, 3, 4):
        top = (1 << bits) - 1
        N, K, G, M = 160, 1024, 64, 16
        q = np.zeros((N, K), dtype=np.uint8)
        q[::2] = top
        z = np.zeros((N, K // G), dtype=np.uint8)
        z[1::2] = top
        s = np.full((N, K // G), 0x4000, dtype=np.uint16)  # 2.0
        x = synth.gen_x(synth.Projection("t", M, N, K, bits, G, 77))
        d = dev()
        y = wq.wq_gemm(torch.from_numpy(x.view(np.int16)).to(d),
                       wq.wq_pack(torch.from_numpy(q).to(d), bits),
                       torch.from_numpy(s.view(np.int16)).to(d), torch.from_numpy(z).to(d), N, G, bits)
        y_ref = oracle.gemm_f64(x, oracle.pack(q, bits), s, z, K, G, bits)
        assert rel_err(y.cpu().numpy(), y_ref) <= ARITH_TOL


@pytest.mark.parametrize("fmt,M,N,K", [((4, 128), 16, 128, 65536), ((2, 32), 7, 160, 32768),
                                       ((3, 128), 12, 300160, 256)],
                         ids=["long-K-one-tile", "long-K-2bit", "tall-N"])
def test_extreme_shapes_sampled_rows(fmt, M, N, K):
    # one 128-row tile split over the most CTAs a tile may have (long K), and
    # thousands of tiles with a short K (tall N): sampled weight rows against
    # the oracle
    wq = _wq()
    bits, G = fmt
    p = proj("C3", M=M, N=N, K=K, bits=bits, group=G, outlier_frac=0.0)
    q, s, z = synth.gen_weights_torch(p, dev())
    wq_d = wq.wq_pack(q, bits)
    del q
    x = synth.gen_x(p)
    y = wq.wq_gemm(torch.from_numpy(x.view(np.int16)).to(dev()), wq_d, s, z, N, G, bits)
    torch.cuda.synchronize()
    wq.wq_check_workspace()
    rows = np.unique(np.linspace(0, N - 1, 24).astype(np.int64))
    w = synth.gen_weights(p, rows=rows)
    ref = oracle.gemm_f64(x, oracle.pack(w["q"], bits), w["s"], w["z"], K, G, bits)
    got = y.cpu().numpy()[:, rows]
    assert rel_err(got, ref) <= REL_TOL


@pytest.mark.parametrize("fmt", [(4, 128), (2, 64), (3, 32)], ids=_fid)
def test_largest_supported_zero_point(fmt):
    # z up to 127 is exact in every kernel build (128 + z is an 8-bit bf16
    # mantissa pattern); here every zero point is 120..127
    wq = _wq()
    bits, G = fmt
    p = proj("C3", M=6, N=260, K=1024, bits=bits, group=G, outlier_frac=0.0, z_range=(120, 127))
    w, x, d = to_dev_host_inputs(p)
    y = wq.wq_gemm(d["x"], d["wq"], d["s"], d["z"], p.N, G, bits)
    torch.cuda.synchronize()
    ref = oracle.gemm_f64(x, oracle.pack(w["q"], bits), w["s"], w["z"], p.K, G, bits)
    assert rel_err(y.cpu().numpy(), ref) <= REL_TOL
