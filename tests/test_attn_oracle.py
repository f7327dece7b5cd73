"""CPU pins of the decode-attention oracle (paged q8_0 KV pool): the binary16
and q8_0 decodings against hand-derived values and numpy's half type,
closed forms of softmax attention, invariance to where pages sit in the pool
and to duplicated key/value heads, the causal view of draft rows, and a dense
numpy computation as an independent library routine."""
import dataclasses
import os

import numpy as np
import pytest

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "fp16_q8_0.txt")


def _golden():
    fp16, q8 = [], []
    for line in open(GOLDEN):
        t = line.split()
        if not t or t[0].startswith("#"):
            continue
        if t[0] == "fp16":
            fp16.append((int(t[1], 16), float(t[2])))
        else:
            q8.append((int(t[1], 16), int(t[2]), float(t[3])))
    return fp16, q8


def test_fp16_golden_values():
    fp16, _ = _golden()
    assert len(fp16) >= 8
    for bits, v in fp16:
        got = oracle.fp16_value(bits)
        assert got == v and np.signbit(got) == np.signbit(v), hex(bits)


def test_fp16_every_finite_pattern_matches_numpy_half():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    finite = np.isfinite(ref)
    got = np.array([oracle.fp16_value(int(b)) for b in bits[finite]])
    assert (got == ref[finite]).all()


def test_q8_0_golden_values():
    _, q8 = _golden()
    for d, c, v in q8:
        codes = np.zeros(32, dtype=np.int8)
        codes[5] = c
        got = oracle.q8_0_dequant(codes, np.array([d], dtype=np.uint16))
        assert got[5] == v and (np.delete(got, 5) == 0).all()


def test_q8_0_blocks_take_their_own_scale():
    codes = np.arange(-64, 64, dtype=np.int8)  # 4 blocks
    scales = np.array([0x3C00, 0x3800, 0xC000, 0x0400], dtype=np.uint16)
    got = oracle.q8_0_dequant(codes, scales)
    ref = codes.astype(np.float64) * np.repeat(scales.view(np.float16).astype(np.float64), 32)
    assert (got == ref).all()


CASE = synth.PagedAttention("pa", (37, 100, 64), 3, 8, 2, 64, 16, 5, shared_prefix=32)


def _run(d, **over):
    a = dict(d)
    a.update(over)
    return oracle.paged_attention_f64(a["q"], a["kc"], a["kd"], a["vc"], a["vd"], a["page_table"],
                                      a["seq_len"], a["row_seq"], a["row_pos"])


def _dense(d, Hq, Hkv, D, T):
    """Independent dense computation with numpy: gather each row's keys and
    values through its page table, dequantise with numpy's half type, softmax
    with np.exp, weighted sum with einsum."""
    k = d["kc"].astype(np.float64) * np.repeat(d["kd"].view(np.float16).astype(np.float64), 32, -1)
    v = d["vc"].astype(np.float64) * np.repeat(d["vd"].view(np.float16).astype(np.float64), 32, -1)
    q = synth.bf16_bits_to_f32(d["q"]).astype(np.float64)
    out = np.zeros(q.shape)
    for i, (b, pos) in enumerate(zip(d["row_seq"], d["row_pos"])):
        t = np.arange(pos + 1)
        pg = d["page_table"][b][t // T]
        kk = k[pg, :, t % T, :]  # [n][Hkv][D]
        vv = v[pg, :, t % T, :]
        for h in range(Hq):
            g = h // (Hq // Hkv)
            s = kk[:, g, :] @ q[i, h] / np.sqrt(D)
            w = np.exp(s - s.max())
            out[i, h] = np.einsum("t,td->d", w / w.sum(), vv[:, g, :])
    return out


def test_matches_dense_numpy():
    d = synth.gen_paged_attention(CASE)
    got = _run(d)
    ref = _dense(d, CASE.Hq, CASE.Hkv, CASE.D, CASE.T)
    assert np.abs(got - ref).max() <= 1e-12 * np.abs(ref).max()


def test_single_position_returns_its_value():
    p = dataclasses.replace(CASE, seq_lens=(1, 5), rows_per_seq=1, shared_prefix=0)
    d = synth.gen_paged_attention(p)
    got = _run(d, row_pos=np.array([0, 0], dtype=np.int32))
    v = oracle.q8_0_dequant(d["vc"], d["vd"])
    for i, b in enumerate((0, 1)):
        page = d["page_table"][b][0]
        for h in range(p.Hq):
            assert (got[i, h] == v[page, h // (p.Hq // p.Hkv), 0]).all()


def test_identical_keys_average_the_values():
    d = synth.gen_paged_attention(CASE)
    kc = d["kc"].copy()
    kc[:] = kc[0:1, :, 0:1, :]  # one key everywhere
    kd = d["kd"].copy()
    kd[:] = kd[0:1, :, 0:1, :]
    got = _run(d, kc=kc, kd=kd)
    v = oracle.q8_0_dequant(d["vc"], d["vd"])
    for i, (b, pos) in enumerate(zip(d["row_seq"], d["row_pos"])):
        t = np.arange(pos + 1)
        vv = v[d["page_table"][b][t // CASE.T], :, t % CASE.T, :]
        for h in range(CASE.Hq):
            ref = vv[:, h // (CASE.Hq // CASE.Hkv), :].mean(axis=0)
            assert np.abs(got[i, h] - ref).max() <= 1e-12 * max(np.abs(ref).max(), 1e-300)


def test_draft_rows_see_only_earlier_positions():
    d = synth.gen_paged_attention(CASE)
    got = _run(d)
    for i, (b, pos) in enumerate(zip(d["row_seq"], d["row_pos"])):
        sl = d["seq_len"].copy()
        sl[b] = pos + 1  # the cache cut right after this row
        one = _run(d, q=d["q"][i:i + 1], seq_len=sl, row_seq=d["row_seq"][i:i + 1],
                   row_pos=d["row_pos"][i:i + 1])
        assert (one[0] == got[i]).all()


def test_page_placement_does_not_matter():
    d = synth.gen_paged_attention(CASE)
    got = _run(d)
    pages = d["kc"].shape[0]
    perm = np.random.default_rng(3).permutation(pages)  # new physical page of old page j
    moved = {}
    for key in ("kc", "kd", "vc", "vd"):
        a = np.empty_like(d[key])
        a[perm] = d[key]
        moved[key] = a
    table = perm[d["page_table"]].astype(np.int32)
    got2 = _run(d, page_table=table, **moved)
    assert (got2 == got).all()


def test_sequence_and_row_order_do_not_matter():
    # relabelling the sequences (page-table rows and lengths) and listing the
    # query rows in another order moves each row's result with it
    d = synth.gen_paged_attention(CASE)
    got = _run(d)
    B = len(CASE.seq_lens)
    sp = np.array([2, 0, 1])[:B]             # new label of old sequence b
    inv = np.argsort(sp)                      # old sequence of new label
    rp = np.random.default_rng(4).permutation(len(d["row_seq"]))  # new row i = old row rp[i]
    got2 = _run(d, page_table=np.ascontiguousarray(d["page_table"][inv]),
                seq_len=np.ascontiguousarray(d["seq_len"][inv]),
                row_seq=np.ascontiguousarray(sp[d["row_seq"][rp]].astype(np.int32)),
                row_pos=np.ascontiguousarray(d["row_pos"][rp]),
                q=np.ascontiguousarray(d["q"][rp]))
    assert (got2 == got[rp]).all()


def test_duplicated_kv_heads_give_the_same_attention():
    d = synth.gen_paged_attention(CASE)
    got = _run(d)
    rep = CASE.Hq // CASE.Hkv
    wide = {k: np.repeat(d[k], rep, axis=1) for k in ("kc", "kd", "vc", "vd")}  # Hkv = Hq
    got2 = _run(d, **wide)
    assert (got2 == got).all()


def test_one_dominant_key_selects_its_value():
    p = dataclasses.replace(CASE, seq_lens=(20,), rows_per_seq=1, shared_prefix=0, Hq=2, Hkv=2)
    d = synth.gen_paged_attention(p)
    kc = np.zeros_like(d["kc"])
    kd = np.full_like(d["kd"], 0x3C00)
    q = np.zeros_like(d["q"])
    q[0, :, 0] = 0x4000  # q = 2 e_0 in every head
    t0 = 11  # the key that wins: component 0 = 100, all other keys 0
    page = d["page_table"][0][t0 // p.T]
    kc[page, :, t0 % p.T, 0] = 100
    got = _run(d, kc=kc, kd=kd, q=q)
    v = oracle.q8_0_dequant(d["vc"], d["vd"])
    # weight of every other key: e^(-200 / sqrt(D)) = e^-25 ~ 1.4e-11
    for h in range(2):
        ref = v[page, h, t0 % p.T]
        assert np.abs(got[0, h] - ref).max() <= 1e-9 * np.abs(v).max()


def test_rejects_bad_arguments():
    d = synth.gen_paged_attention(CASE)
    with pytest.raises(ValueError):
        _run(d, row_pos=d["seq_len"][d["row_seq"]])  # a position past the cache
    bad = d["page_table"].copy()
    bad[1, 0] = d["kc"].shape[0]  # a page outside the pool
    with pytest.raises(ValueError):
        _run(d, page_table=bad)
    with pytest.raises(ValueError):  # 8 query heads over 3 key/value heads
        _run(d, **{k: np.repeat(d[k], 3, axis=1)[:, :3] for k in ("kc", "kd", "vc", "vd")})
