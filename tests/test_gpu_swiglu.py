"""Fused gate/up activation: wq_gemm_swiglu, and the WQ_EPI_SWIGLU epilogue of a
decode step feeding the down projection's X.  The reference is the oracle's
fp64 GEMM followed by its fp64 SwiGLU and one bf16 rounding; the GPU rounds
its fp32 sums through fp32 arithmetic first, so single elements may differ by
one bf16 step where the exact value lies next to a rounding boundary."""
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


def _key(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> integers ordered like the values (+0 and -0 equal)."""
    b = bits.astype(np.int64)
    mag = b & 0x7FFF
    return np.where(b & 0x8000, -mag, mag)


def _ulps(a: np.ndarray, b: np.ndarray) -> int:
    return int(np.abs(_key(a) - _key(b)).max())


def _bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


CASES = [(5, 1280, 1280, 4, 128), (16, 600, 2048, 3, 64), (1, 2000, 17408, 4, 128),
         (8, 1536, 5120, 2, 32), (12, 256, 640, 2, 128)]


@pytest.mark.parametrize("M,N,K,bits,G", CASES, ids=lambda c: str(c))
def test_swiglu_matches_oracle(M, N, K, bits, G):
    import weight_only_bit_wq_gb300 as wq
    p = synth.Projection("gu", M, N, K, bits, G, 601)
    w, x, d = to_dev_host_inputs(p)
    out = wq.wq_gemm_swiglu(d["x"], d["wq"], d["s"], d["z"], N, G, bits)
    torch.cuda.synchronize()
    got = _bits(out)
    assert got.shape == (M, N // 2)
    check_activation(got, oracle_gemm(p, w, x))
    wq.wq_check_workspace()


def test_swiglu_is_the_activation_of_wq_gemm():
    # same fp32 sums as wq_gemm; the activation in fp32 on the host agrees to
    # one bf16 step (the device expf and the host exp may differ in the last bit)
    import weight_only_bit_wq_gb300 as wq
    M, N, K, bits, G = 7, 2 * 640, 2560, 4, 128
    p = synth.Projection("gu2", M, N, K, bits, G, 602)
    w, x, d = to_dev_host_inputs(p)
    y = wq.wq_gemm(d["x"], d["wq"], d["s"], d["z"], N, G, bits).cpu().numpy()
    got = _bits(wq.wq_gemm_swiglu(d["x"], d["wq"], d["s"], d["z"], N, G, bits))
    g, u = y[:, 0::2], y[:, 1::2]
    host = torch.from_numpy((g / (np.float32(1) + np.exp(-g)) * u).astype(np.float32))
    ref = _bits(host.to(torch.bfloat16))
    assert _ulps(got, ref) <= 1
    assert (got == ref).mean() > 0.99


def test_swiglu_rows_are_batch_invariant():
    import weight_only_bit_wq_gb300 as wq
    M, N, K, bits, G = 9, 2 * 512, 3072, 4, 64
    p = synth.Projection("gu3", M, N, K, bits, G, 603)
    w, x, d = to_dev_host_inputs(p)
    full = _bits(wq.wq_gemm_swiglu(d["x"], d["wq"], d["s"], d["z"], N, G, bits))
    for m in (0, 4, 8):
        alone = _bits(wq.wq_gemm_swiglu(d["x"][m:m + 1].contiguous(), d["wq"], d["s"], d["z"], N, G,
                                        bits))
        assert (alone[0] == full[m]).all(), m


def test_swiglu_saturating_gates():
    # Gate values from far below the fp32 exponential's range to well above
    # it.  Down to about -87 the result matches the oracle to one bf16 step;
    # below, the device's 1 + exp(-g) passes 2^126 and its quotient is zero,
    # where the exact value is under 1e-36 times |up| in magnitude.
    import weight_only_bit_wq_gb300 as wq
    targets = [-150.0, -100.0, -88.0, -87.5, -80.0, -10.0, 0.25, 60.0]
    F, K, G, M = len(targets), 256, 128, 2
    N = 2 * F
    q = np.full((N, K), 15, dtype=np.uint8)
    z = np.zeros((N, K // G), dtype=np.uint8)
    s32 = np.empty((N, K // G), dtype=np.float32)
    s32[0::2] = (np.array(targets, dtype=np.float32) / (15 * K))[:, None]
    s32[1::2] = np.float32(2.0 / (15 * K))
    s = synth.f32_to_bf16_bits(s32)
    x = synth.f32_to_bf16_bits(np.array([[1.0] * K, [0.5] * K], dtype=np.float32))
    d = dev()
    out = wq.wq_gemm_swiglu(torch.from_numpy(x.view(np.int16)).to(d),
                            wq.wq_pack(torch.from_numpy(q).to(d), 4),
                            torch.from_numpy(s.view(np.int16)).to(d), torch.from_numpy(z).to(d),
                            N, G, 4)
    got = _bits(out)
    y64 = oracle.gemm_f64(x, oracle.pack(q, 4), s, z, K, G, 4)
    ref = oracle.swiglu_bf16(y64)
    g = y64[:, 0::2]
    normal = g > -87.0
    assert normal.sum() >= 10 and (~normal).sum() >= 3
    assert _ulps(got[normal], ref[normal]) <= 1
    assert ((got[~normal] & 0x7FFF) == 0).all()
    ref_f = synth.bf16_bits_to_f32(ref[~normal])
    assert (np.abs(ref_f) < 1e-35).all()


def test_swiglu_rejects_odd_width_and_handles_empty_k():
    import weight_only_bit_wq_gb300 as wq
    p = synth.Projection("gu4", 2, 256, 256, 4, 128, 604)
    w, x, d = to_dev_host_inputs(p)
    with pytest.raises(wq.WQError):
        wq.wq_gemm_swiglu(d["x"], d["wq"], d["s"], d["z"], 255, 128, 4)
    empty = torch.full((2, 128), 7.0, dtype=torch.bfloat16, device=dev())
    wq.wq_gemm_swiglu(d["x"][:, :0].contiguous(), d["wq"], d["s"], d["z"], 256, 128, 4, out=empty)
    torch.cuda.synchronize()
    assert (_bits(empty) == 0).all()


@pytest.mark.parametrize("M", [6, 20])
@pytest.mark.parametrize("fused", [False, True], ids=["sequential", "fused"])
def test_gate_up_activation_feeds_down_in_a_step(fused, M):
    # gate/up with the activation epilogue writes the down projection's X;
    # down waits for it (fused: on the device; sequential: by stream order);
    # 20 rows run the 32-row build
    import weight_only_bit_wq_gb300 as wq
    F, H = 640, 1280  # features, hidden
    gu = synth.Projection("gu5", M, 2 * F, H, 4, 128, 605)
    dn = synth.Projection("dn5", M, H, F, 4, 128, 606, index=1)
    wg, xg, dg = to_dev_host_inputs(gu)
    wd, _xd_unused, dd = to_dev_host_inputs(dn)
    act = torch.full((M, F), float("nan"), dtype=torch.bfloat16, device=dev())
    y = torch.full((M, H), float("nan"), dtype=torch.float32, device=dev())
    descs = wq.make_descs([
        dict(x=dg["x"], wq=dg["wq"], scales=dg["s"], zeros=dg["z"], y=act, M=M, N=2 * F, K=H,
             group=128, bits=4, epilogue=wq.WQ_EPI_SWIGLU),
        dict(x=act, wq=dd["wq"], scales=dd["s"], zeros=dd["z"], y=y, M=M, N=H, K=F, group=128,
             bits=4, after=0),
    ])
    flags = wq.WQ_STEP_FUSED if fused else 0
    ws = wq.new_step_workspace(descs, flags)
    for _ in range(2):
        act.fill_(float("nan"))
        y.fill_(float("nan"))
        wq.wq_step_run(descs, ws, flags=flags)
        torch.cuda.synchronize()
        wq.wq_check_workspace(ws)
        a_bits = _bits(act)
        check_activation(a_bits, oracle_gemm(gu, wg, xg))
        # down against the oracle, fed the activation the GPU produced
        x_dn = a_bits.view(np.uint16)
        y_ref = oracle.gemm_f64(x_dn, oracle.pack(wd["q"], 4), wd["s"], wd["z"], F, 128, 4)
        err = rel_err(y.cpu().numpy(), y_ref)
        assert err <= REL_TOL and err <= ARITH_TOL, err
