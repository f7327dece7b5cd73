"""Pins of the fp64 CPU oracle against facts that do not come from the oracle.

Each test fixes the oracle to something independent of its own code: values
printed on the pages or derived by hand from the layout (golden files),
closed forms, invariants, exact rational brute force on tiny inputs, and one
special case that reduces to a library routine (torch's float64 matmul and
torch's float32 -> bfloat16 cast).  A dropped term, a wrong sign, a wrong
group index or a transposed operand in the oracle fails at least one of them.
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth


# ------------------------------------------------------------------ fixtures
def _read_golden(path, parts=3):
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([part.split() for part in line.split("|", parts - 1)])
    return rows


def _bf16(v: float) -> int:
    """bf16 bits of a value that is exactly representable in bf16."""
    b = np.array([v], dtype=np.float32).view(np.uint32)[0]
    assert b & 0xFFFF == 0, v
    return int(b >> 16)


def _bf16_value(bits: int) -> Fraction:
    f = np.array([bits << 16], dtype=np.uint32).view(np.float32)[0]
    return Fraction(float(f))


# --------------------------------------------------------------- packing
@pytest.mark.parametrize("K,bits,W", [
    (1024, 4, 128), (5120, 4, 640), (17408, 4, 2176), (17408, 3, 1744),
    (17408, 2, 1088), (11, 3, 4), (1, 2, 4), (33, 4, 8), (40, 3, 4), (41, 3, 8)])
def test_words_per_row_closed_form(K, bits, W):
    # ceil(K / values-per-word) rounded up to a multiple of 4 words (16 bytes)
    assert oracle.words_per_row(K, bits) == W


def test_pack_golden_words(golden_dir):
    rows = _read_golden(os.path.join(golden_dir, "pack_words.txt"))
    assert len(rows) >= 10
    for (hdr, codes, words) in rows:
        bits, K = int(hdr[0]), int(hdr[1])
        q = np.array([[int(c) for c in codes]], dtype=np.uint8)
        assert q.shape[1] == K
        expect = np.array([[int(w, 16) for w in words]], dtype=np.uint32)
        got = oracle.pack(q, bits)
        assert got.shape == expect.shape, (hdr, got.shape)
        assert (got == expect).all(), (hdr, [hex(v) for v in got[0]])
        assert (oracle.unpack(expect, K, bits) == q).all()


@pytest.mark.parametrize("bits", [2, 3, 4])
@pytest.mark.parametrize("K", [1, 7, 10, 31, 64, 160, 257, 384])
def test_pack_unpack_every_value_every_slot(bits, K):
    # Row n holds (n + k) mod 2^b, so across the 2^b rows every value sits in
    # every slot of every word, including partial last words and words that
    # straddle a group boundary (3-bit).
    nv = 1 << bits
    n = np.arange(nv)[:, None]
    k = np.arange(K)[None, :]
    q = ((n + k) % nv).astype(np.uint8)
    wq = oracle.pack(q, bits)
    assert wq.shape == (nv, oracle.words_per_row(K, bits))
    assert (oracle.unpack(wq, K, bits) == q).all()
    # pad slots, pad bits and pad words are zero: the popcount of a row equals
    # the popcount of its codes
    pc_words = np.array([sum(bin(int(w)).count("1") for w in row) for row in wq])
    pc_codes = np.array([sum(bin(int(c)).count("1") for c in row) for row in q])
    assert (pc_words == pc_codes).all()
    if bits == 3:
        # bits 15 and 31 of every word are pad bits
        assert ((wq & np.uint32(0x80008000)) == 0).all()


def test_pack_keeps_low_bits_only():
    q = np.array([[0xF7, 0x13]], dtype=np.uint8)
    assert (oracle.unpack(oracle.pack(q, 3), 2, 3) == np.array([[7, 3]])).all()
    assert (oracle.unpack(oracle.pack(q, 2), 2, 2) == np.array([[3, 3]])).all()


def test_bad_bits_rejected():
    with pytest.raises(ValueError):
        oracle.pack(np.zeros((1, 8), dtype=np.uint8), 5)


# ------------------------------------------------------------ bf16 rounding
def test_bf16_rne_golden(golden_dir):
    rows = _read_golden(os.path.join(golden_dir, "dequant_bf16.txt"))
    assert len(rows) >= 8
    for (inp, out, _why) in rows:
        s_bits, qv, zv = int(inp[0], 16), int(inp[1]), int(inp[2])
        expect = int(out[0], 16)
        exact = (qv - zv) * float(_bf16_value(s_bits))
        assert oracle.bf16_rne(exact) == expect, (inp, hex(oracle.bf16_rne(exact)))
        # the same through the packed dequantisation path (K = G = 32, one group)
        q = np.full((1, 32), qv, dtype=np.uint8)
        wq = oracle.pack(q, 4)
        s = np.array([[s_bits]], dtype=np.uint16)
        z = np.array([[zv]], dtype=np.uint8)
        w = oracle.dequant_bf16(wq, s, z, 32, 32, 4)
        assert (w == expect).all()


def test_bf16_rne_matches_torch_cast():
    # torch's float32 -> bfloat16 cast is an independent round-to-nearest-even
    rng = np.random.default_rng(123)
    mant = rng.integers(0, 1 << 23, size=4000)
    expo = rng.integers(100, 150, size=4000)
    sign = rng.integers(0, 2, size=4000)
    bits = (sign << 31) | (expo << 23) | mant
    # include exact ties: low 16 bits = 0x8000
    bits[:500] = (bits[:500] & ~0xFFFF) | 0x8000
    f = bits.astype(np.uint32).view(np.float32)
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_rne(float(v)) for v in f], dtype=np.uint16)
    assert (got == ref).all()


# ---------------------------------------------------------- dequantisation
def test_dequant_group_index_and_sign():
    # scale of group g is 2^-(g+1); q - z = +1 in even groups, -2 in odd groups
    K, G, bits = 256, 32, 4
    ng = K // G
    s = np.array([[_bf16(2.0 ** -(g + 1)) for g in range(ng)]], dtype=np.uint16)
    z = np.array([[3 if g % 2 == 0 else 5 for g in range(ng)]], dtype=np.uint8)
    q = np.array([[4 if (k // G) % 2 == 0 else 3 for k in range(K)]], dtype=np.uint8)
    w = oracle.dequant_f64(oracle.pack(q, bits), s, z, K, G, bits)
    expect = np.array([(1.0 if (k // G) % 2 == 0 else -2.0) * 2.0 ** -((k // G) + 1)
                       for k in range(K)])
    assert (w[0] == expect).all()


def test_dequant_unit_scale_is_code_minus_zero():
    p = synth.Projection("t", 1, 3, 384, 3, 128, 11)
    wts = synth.gen_weights(p)
    s = np.full_like(wts["s"], _bf16(1.0))
    w = oracle.dequant_f64(oracle.pack(wts["q"], 3), s, wts["z"], p.K, p.group, 3)
    zz = np.repeat(wts["z"].astype(np.int64), p.group, axis=1)
    assert (w == (wts["q"].astype(np.int64) - zz)).all()


# ----------------------------------------------------------------- GEMM
def _exact_gemm(x_bits, q, s_bits, z, G):
    """Exact rational Y and sum of |terms| from the raw codes (brute force, tiny sizes)."""
    M, K = x_bits.shape
    N = q.shape[0]
    xv = [[_bf16_value(int(b)) for b in row] for row in x_bits]
    sv = [[_bf16_value(int(b)) for b in row] for row in s_bits]
    y = [[None] * N for _ in range(M)]
    mag = [[None] * N for _ in range(M)]
    for m in range(M):
        for n in range(N):
            acc, a = Fraction(0), Fraction(0)
            for k in range(K):
                t = xv[m][k] * (int(q[n][k]) - int(z[n][k // G])) * sv[n][k // G]
                acc += t
                a += abs(t)
            y[m][n], mag[m][n] = acc, a
    return y, mag


@pytest.mark.parametrize("bits,G,K,N,M", [(4, 32, 64, 3, 1), (3, 32, 96, 5, 3), (2, 64, 128, 2, 16),
                                          (4, 128, 256, 4, 5), (3, 64, 192, 2, 2), (4, 64, 128, 2, 32),
                                          (2, 32, 64, 3, 24)])
def test_gemm_brute_force_exact(bits, G, K, N, M):
    p = synth.Projection("t", M, N, K, bits, G, 100 + bits)
    w = synth.gen_weights(p)
    x = synth.gen_x(p)
    y = oracle.gemm_f64(x, oracle.pack(w["q"], bits), w["s"], w["z"], K, G, bits)
    ye, mag = _exact_gemm(x, w["q"], w["s"], w["z"], G)
    nonzero = 0
    for m in range(M):
        for n in range(N):
            # a sequential fp64 sum of K exact products errs by at most (K-1) 2^-53 sum|t|
            assert abs(Fraction(float(y[m, n])) - ye[m][n]) <= (K - 1) * Fraction(1, 2 ** 53) * mag[m][n]
            nonzero += ye[m][n] != 0
    assert nonzero == M * N


def test_gemm_identity_tile():
    K = N = 128
    q = np.eye(N, K, dtype=np.uint8)
    s = np.full((N, 1), _bf16(1.0), dtype=np.uint16)
    z = np.zeros((N, 1), dtype=np.uint8)
    p = synth.Projection("t", 5, N, K, 4, 128, 3)
    x = synth.gen_x(p)
    y = oracle.gemm_f64(x, oracle.pack(q, 4), s, z, K, 128, 4)
    assert (y == synth.bf16_bits_to_f32(x).astype(np.float64)).all()


def test_gemm_one_hot():
    M, N, K, G, bits = 3, 7, 256, 64, 4
    p = synth.Projection("t", M, N, K, bits, G, 9)
    w = synth.gen_weights(p)
    x = synth.gen_x(p)
    zz = np.repeat(w["z"], G, axis=1)
    q = zz.copy()  # q == z everywhere ...
    n0, k0 = 5, 130  # ... except one code (n0 != k0, group 2)
    q[n0, k0] = (int(zz[n0, k0]) + 6) % 16
    d = int(q[n0, k0]) - int(zz[n0, k0])
    y = oracle.gemm_f64(x, oracle.pack(q, bits), w["s"], w["z"], K, G, bits)
    col = synth.bf16_bits_to_f32(x[:, k0]).astype(np.float64) * d * float(
        synth.bf16_bits_to_f32(w["s"][n0, k0 // G]))
    assert (y[:, n0] == col).all()
    y[:, n0] = 0
    assert (y == 0).all()


def test_gemm_codes_equal_zero_points_give_zero():
    p = synth.Projection("t", 4, 9, 384, 3, 128, 21)
    w = synth.gen_weights(p)
    q = np.repeat(w["z"], p.group, axis=1)
    y = oracle.gemm_f64(synth.gen_x(p), oracle.pack(q, 3), w["s"], w["z"], p.K, p.group, 3)
    assert (y == 0).all()


def test_gemm_constant_weight_closed_form():
    # x == 1 and w == c * s everywhere  ->  y == K * c * s exactly
    M, N, K, G = 2, 3, 512, 128
    x = np.full((M, K), _bf16(1.0), dtype=np.uint16)
    q = np.full((N, K), 11, dtype=np.uint8)
    z = np.full((N, K // G), 4, dtype=np.uint8)
    s = np.full((N, K // G), _bf16(0.015625), dtype=np.uint16)
    y = oracle.gemm_f64(x, oracle.pack(q, 4), s, z, K, G, 4)
    assert (y == K * 7 * 0.015625).all()


def test_gemm_matches_torch_float64_matmul():
    # special case reducing to a library routine: dequantise, then X @ W^T
    p = synth.CONFIGS["C4b"]
    import dataclasses
    p = dataclasses.replace(p, N=48, K=1280)
    w = synth.gen_weights(p)
    x = synth.gen_x(p)
    wq = oracle.pack(w["q"], p.bits)
    wd = oracle.dequant_f64(wq, w["s"], w["z"], p.K, p.group, p.bits)
    ref = (torch.from_numpy(synth.bf16_bits_to_f32(x).astype(np.float64))
           @ torch.from_numpy(wd).T).numpy()
    y = oracle.gemm_f64(x, wq, w["s"], w["z"], p.K, p.group, p.bits)
    assert np.abs(y - ref).max() <= 1e-11 * np.abs(ref).max()


def test_gemm_rows_independent_and_thread_count_independent():
    # the oracle is row-independent: a row's result alone == stacked, bitwise
    p = synth.CONFIGS["C2"]
    import dataclasses
    p = dataclasses.replace(p, N=96, K=1024)
    w = synth.gen_weights(p)
    x = synth.gen_x(p)
    wq = oracle.pack(w["q"], 4)
    y = oracle.gemm_f64(x, wq, w["s"], w["z"], p.K, 128, 4, threads=3)
    for m in range(p.M):
        ym = oracle.gemm_f64(x[m:m + 1], wq, w["s"], w["z"], p.K, 128, 4, threads=1)
        assert (ym[0] == y[m]).all()


# ------------------------------------------------------- step-time floor
def test_step_floor_matches_printed_figure(golden_dir):
    (inp, out), = [(r[0], r[1]) for r in _read_golden(os.path.join(golden_dir, "step_floor.txt"), 2)]
    t_ms = oracle.step_floor_seconds(float(inp[0]), float(inp[1])) * 1e3
    assert abs(t_ms - float(out[0])) <= float(out[1])
    assert abs(t_ms - 17.842) < 1e-3


# ------------------------------------------------------------ fused SwiGLU
def test_swiglu_golden_values(golden_dir):
    rows = _read_golden(os.path.join(golden_dir, "swiglu_bf16.txt"))
    assert len(rows) >= 6
    for (inp, out, _why) in rows:
        g, u = float(inp[0]), float(inp[1])
        y = np.array([[g, u]], dtype=np.float64)
        assert int(oracle.swiglu_bf16(y)[0, 0]) == int(out[0], 16), (inp, hex(int(oracle.swiglu_bf16(y)[0, 0])))


def test_silu_closed_forms():
    # silu(x) - silu(-x) = x (sigmoid(x) + sigmoid(-x) = 1); silu(0) = 0;
    # silu(x) -> x and silu(-x) -> -x e^-x as x grows
    for x in (0.25, 1.0, 3.5, 7.0, 12.0):
        assert abs((oracle.silu_f64(x) - oracle.silu_f64(-x)) - x) <= 4e-16 * x
    assert oracle.silu_f64(0.0) == 0.0
    assert oracle.silu_f64(40.0) == 40.0
    assert abs(oracle.silu_f64(-40.0) / (-40.0 * np.exp(-40.0)) - 1.0) < 1e-15
    # sigmoid(x) = silu(x) / x is the logistic function: 1/2 at 0+, e/(1+e) at 1
    assert abs(oracle.silu_f64(1.0) - np.e / (1.0 + np.e)) < 1e-16


def test_swiglu_layout_pairs_rows_and_rejects_odd_widths():
    # column 2j is the gate and 2j + 1 the up value of feature j; swapping them
    # changes the result, and an odd width is refused
    y = np.array([[2.0, 1.0, 1.0, 2.0], [-3.0, 0.25, 0.0, 9.0]])
    out = oracle.swiglu_bf16(y)
    assert out.shape == (2, 2)
    assert out[0, 0] == oracle.bf16_rne(oracle.silu_f64(2.0) * 1.0)
    assert out[0, 1] == oracle.bf16_rne(oracle.silu_f64(1.0) * 2.0)
    assert out[0, 0] != out[0, 1]
    assert out[1, 1] == 0  # silu(0) * 9 = 0
    with pytest.raises(ValueError):
        oracle.swiglu_bf16(np.zeros((1, 3)))
