"""GPU parity of wq_pack / wq_unpack / wq_dequant: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from wqtest import dev, u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


SHAPES = [(1, 1), (3, 7), (5, 10), (130, 257), (64, 384), (17, 1000), (256, 5120)]


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("N,K", SHAPES)
def test_pack_bit_exact(bits, N, K):
    import weight_only_bit_wq_gb300 as wq
    rng = np.random.default_rng(N * 1000 + K + bits)
    q = rng.integers(0, 256, size=(N, K), dtype=np.uint8)  # high bits must be ignored
    wq_d = wq.wq_pack(torch.from_numpy(q).to(dev()), bits)
    assert (u32(wq_d) == oracle.pack(q, bits)).all()
    back = wq.wq_unpack(wq_d, K, bits)
    assert (back.cpu().numpy() == oracle.unpack(oracle.pack(q, bits), K, bits)).all()


@pytest.mark.parametrize("bits,G", [(4, 128), (4, 32), (3, 128), (3, 64), (2, 64), (2, 32)])
@pytest.mark.parametrize("N,K", [(3, 128), (130, 384), (200, 1280)])
def test_dequant_bit_exact(bits, G, N, K):
    import weight_only_bit_wq_gb300 as wq
    p = synth.Projection("t", 1, N, K, bits, G, 7 + bits, s_range=(0.005, 0.04))
    w = synth.gen_weights(p)
    wq_ref = oracle.pack(w["q"], bits)
    d = dev()
    wq_d = wq.wq_pack(torch.from_numpy(w["q"]).to(d), bits)
    out = wq.wq_dequant(wq_d, torch.from_numpy(w["s"].view(np.int16)).to(d),
                        torch.from_numpy(w["z"]).to(d), K, G, bits)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert (got == oracle.dequant_bf16(wq_ref, w["s"], w["z"], K, G, bits)).all()


def test_dequant_rounding_ties_bit_exact():
    # scales with full 7-bit mantissas times every (q - z) hit every tie case
    import weight_only_bit_wq_gb300 as wq
    N, K, G = 128, 32 * 16, 32
    q = np.tile(np.arange(16, dtype=np.uint8), (N, K // 16))
    s = (0x3F80 + (np.arange(N * (K // G)) % 128)).astype(np.uint16).reshape(N, K // G)
    z = (np.arange(N * (K // G)) % 16).astype(np.uint8).reshape(N, K // G)
    d = dev()
    wq_d = wq.wq_pack(torch.from_numpy(q).to(d), 4)
    out = wq.wq_dequant(wq_d, torch.from_numpy(s.view(np.int16)).to(d), torch.from_numpy(z).to(d),
                        K, G, 4)
    got = out.view(torch.int16).cpu().numpy().view(np.uint16)
    assert (got == oracle.dequant_bf16(oracle.pack(q, 4), s, z, K, G, 4)).all()
