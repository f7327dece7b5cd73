"""The seeded input generators: the torch path that builds device inputs gives
the same bits as the numpy path that feeds the oracle (checked here with torch
on the CPU, so the GPU tests and the bench draw exactly the oracle's inputs),
and the draws follow their stated ranges."""
import dataclasses

import numpy as np
import pytest
import torch

import synth


@pytest.mark.parametrize("bits,group,N,K", [(4, 128, 70, 256), (3, 64, 33, 320), (2, 32, 5, 96)])
def test_weights_torch_equal_numpy(bits, group, N, K):
    p = synth.Projection("t", 1, N, K, bits, group, 11, s_range=(0.005, 0.04))
    w = synth.gen_weights(p)
    q, s, z = synth.gen_weights_torch(p, torch.device("cpu"), row_chunk=16)
    assert (q.numpy() == w["q"]).all()
    assert (s.numpy().view(np.uint16) == w["s"]).all()
    assert (z.numpy() == w["z"]).all()


def test_weight_draws_stay_in_range():
    p = synth.Projection("t", 1, 64, 512, 3, 128, 12, s_range=(0.005, 0.04))
    w = synth.gen_weights(p)
    assert w["q"].min() == 0 and w["q"].max() == 7
    assert w["z"].max() <= 7
    s = synth.bf16_bits_to_f32(w["s"])
    # bf16 rounding of U(a, b) may reach one bf16 step past either end
    assert s.min() >= 0.005 * (1 - 2 ** -8) and s.max() <= 0.04 * (1 + 2 ** -8)


def test_rows_subset_equals_full_generation():
    p = synth.Projection("t", 1, 40, 256, 4, 128, 13)
    full = synth.gen_weights(p)
    part = synth.gen_weights(p, rows=[3, 17, 39])
    for k in ("q", "s", "z"):
        assert (part[k] == full[k][[3, 17, 39]]).all()
