"""Pins for the CPU oracle: each test ties it to something other than itself.

What pins what (a plausible mistake and the test that catches it):
  fp16 decoding wrong                -> test_half_decoding_matches_numpy
  transposed operand / wrong scale / wrong softmax / wrong gather
                                     -> test_dense_sdpa_special_case, test_hand_cases,
                                        test_brute_force_high_precision
  KV head h % Hkv instead of h / G   -> test_gqa_head_mapping
  page index t/BS and t%BS swapped   -> test_page_permutation_invariance,
                                        test_dense_sdpa_special_case
  tail of the last page read         -> test_poison_never_read, test_hand_cases (NaN rows)
  log2-space partials / reduce wrong -> test_hand_cases (partials), test_split_invariance
  online update wrong (rescale)      -> test_online_log2_equals_definition
  length 0 / length 1                -> test_zero_length, test_length_one_returns_v
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_03_gb300.workloads import make_custom

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_cases.json")


def _np(w):
    return dict(q=w.q.numpy(), k_cache=w.k_cache.numpy(), v_cache=w.v_cache.numpy(),
                block_tables=w.block_tables.numpy(), seq_lens=w.seq_lens.numpy())


def _small(seed=0, Hq=8, Hkv=2, D=16, BS=4, lens=(1, 7, 13), poison=True, std=1.0,
           scale=None):
    return make_custom(S=len(lens), Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=list(lens), seed=seed,
                       device="cpu", poison=poison, std=std, scale=scale,
                       NB=int(sum((l + BS - 1) // BS for l in lens)) + 5)


def _dense(w):
    """Dense K, V [S][Hkv][Lmax][D] gathered from the generator's own record
    of which physical page holds which logical page (not the page table)."""
    S, Hkv, BS, D = w.S, w.Hkv, w.BS, w.D
    lens = w.lens
    Lmax = int(lens.max())
    K = np.zeros((S, Hkv, Lmax, D))
    V = np.zeros((S, Hkv, Lmax, D))
    kc = w.k_cache.numpy().astype(np.float64)
    vc = w.v_cache.numpy().astype(np.float64)
    for s in range(S):
        own = w.page_ids[w.page_offsets[s]:w.page_offsets[s + 1]].numpy()
        for t in range(int(lens[s])):
            K[s, :, t] = kc[own[t // BS], :, t % BS]
            V[s, :, t] = vc[own[t // BS], :, t % BS]
    return K, V


# ---------------------------------------------------------------- decoding
def test_half_decoding_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.half_to_double(bits)
    ref = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


# ---------------------------------------------------------------- golden
def _parse(x):
    if isinstance(x, list):
        return [_parse(y) for y in x]
    if isinstance(x, str):
        if x == "nan":
            return float("nan")
        if x.startswith("log2("):
            return math.log2(float(x[5:-1]))
        return float(Fraction(x))
    return float(x)


def _case_inputs(c):
    f16 = lambda a: np.asarray(_parse(a), dtype=np.float16)
    scale = {"ln3": math.log(3.0), "ln2": math.log(2.0)}[c["scale"]]
    return dict(q=f16(c["q"]), k_cache=f16(c["k_cache"]), v_cache=f16(c["v_cache"]),
                block_tables=np.asarray(c["block_tables"], dtype=np.int32),
                seq_lens=np.asarray(c["seq_lens"], dtype=np.int32)), scale


@pytest.mark.parametrize("idx", [0, 1])
def test_hand_cases(idx):
    c = json.load(open(GOLDEN))["cases"][idx]
    inp, scale = _case_inputs(c)
    out = oracle.decode(**inp, scale=scale)
    np.testing.assert_allclose(out, np.asarray(_parse(c["out"])), rtol=0, atol=1e-13)
    wt = c["weights"]
    w = oracle.weights(inp["q"], inp["k_cache"], inp["block_tables"], inp["seq_lens"],
                       scale, wt["s"], wt["h"])
    np.testing.assert_allclose(w, wt["w"], rtol=0, atol=1e-15)
    pt = c["partials"]
    m, l, o = oracle.split_partials(**inp, scale=scale, P=pt["P"])
    np.testing.assert_allclose(m, np.asarray(_parse(pt["m"])), rtol=0, atol=1e-13)
    np.testing.assert_allclose(l, np.asarray(_parse(pt["l"])), rtol=0, atol=1e-13)
    np.testing.assert_allclose(o, np.asarray(_parse(pt["o"])), rtol=0, atol=1e-13)
    np.testing.assert_allclose(oracle.merge_partials(m, l, o), out, rtol=0, atol=1e-13)
    if "page_reads" in c:
        reads = oracle.page_reads(inp["block_tables"], inp["seq_lens"], c["Hkv"], c["BS"],
                                  c["NB"])
        assert reads.tolist() == c["page_reads"]


# ---------------------------------------------------------------- library special case
@pytest.mark.parametrize("Hq,Hkv", [(8, 2), (4, 4), (6, 1)])
@pytest.mark.parametrize("BS", [4, 8])
def test_dense_sdpa_special_case(Hq, Hkv, BS):
    w = _small(seed=11 + Hq + BS, Hq=Hq, Hkv=Hkv, BS=BS, lens=(1, 9, 23, 16))
    out = oracle.decode(**_np(w), scale=w.scale)
    K, V = _dense(w)
    G = Hq // Hkv
    q = torch.from_numpy(w.q.numpy().astype(np.float64))
    for s in range(w.S):
        L = int(w.lens[s])
        Kd = torch.from_numpy(K[s, :, :L]).repeat_interleave(G, dim=0)  # [Hq, L, D]
        Vd = torch.from_numpy(V[s, :, :L]).repeat_interleave(G, dim=0)
        ref = torch.nn.functional.scaled_dot_product_attention(
            q[s][:, None, :], Kd, Vd, scale=w.scale)[:, 0, :]
        np.testing.assert_allclose(out[s], ref.numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------- brute force
def test_brute_force_high_precision():
    """Every length 0..40 for BS in {8, 16, 32}, tiny D, against 40-digit
    arithmetic on the same fp16 values (independent dense formulation)."""
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 40
    for BS in (8, 16, 32):
        lens = list(range(0, 41))
        w = make_custom(S=len(lens), Hq=4, Hkv=2, D=4, BS=BS, lens=lens, seed=BS,
                        device="cpu", NB=200)
        out = oracle.decode(**_np(w), scale=w.scale)
        K, V = _dense(w) if max(lens) else (None, None)
        qf = w.q.numpy().astype(np.float64)
        for s, L in enumerate(lens):
            for h in range(4):
                g = h // 2
                if L == 0:
                    assert np.all(out[s, h] == 0.0)
                    continue
                z = [mp.mpf(w.scale) * mp.fsum(mp.mpf(qf[s, h, d]) * mp.mpf(K[s, g, t, d])
                                               for d in range(4)) for t in range(L)]
                zm = max(z)
                e = [mp.e ** (x - zm) for x in z]
                den = mp.fsum(e)
                for d in range(4):
                    ref = mp.fsum(e[t] * mp.mpf(V[s, g, t, d]) for t in range(L)) / den
                    assert abs(out[s, h, d] - float(ref)) <= 1e-13, (BS, L, h, d)


# ---------------------------------------------------------------- closed forms
def test_length_one_returns_v():
    w = _small(seed=3, lens=(1, 1, 1))
    out = oracle.decode(**_np(w), scale=w.scale)
    _, V = _dense(w)
    G = w.Hq // w.Hkv
    for s in range(w.S):
        for h in range(w.Hq):
            assert np.array_equal(out[s, h], V[s, h // G, 0])


def test_constant_v():
    w = _small(seed=4, lens=(5, 17, 40))
    inp = _np(w)
    inp["v_cache"] = np.full_like(inp["v_cache"], np.float16(-1.75))
    out = oracle.decode(**inp, scale=w.scale)
    np.testing.assert_allclose(out, -1.75, rtol=0, atol=1e-14)


def test_weights_sum_to_one():
    w = _small(seed=5, lens=(3, 30, 64), std=2.0)
    inp = _np(w)
    for s in range(w.S):
        for h in (0, 3, 7):
            wt = oracle.weights(inp["q"], inp["k_cache"], inp["block_tables"],
                                inp["seq_lens"], w.scale, s, h)
            assert len(wt) == w.lens[s]
            assert np.all(wt >= 0)
            assert abs(wt.sum() - 1.0) <= 1e-12


def test_weights_match_dense_softmax():
    """The weights of every (sequence, query head) against a numpy softmax of
    the densely gathered keys of KV head h / G."""
    w = _small(seed=19, Hq=8, Hkv=2, lens=(1, 9, 23))
    inp = _np(w)
    K, _ = _dense(w)
    G = w.Hq // w.Hkv
    q = w.q.numpy().astype(np.float64)
    for s in range(w.S):
        L = int(w.lens[s])
        for h in range(w.Hq):
            z = w.scale * (K[s, h // G, :L] @ q[s, h])
            e = np.exp(z - z.max())
            ours = oracle.weights(inp["q"], inp["k_cache"], inp["block_tables"], inp["seq_lens"],
                                  w.scale, s, h)
            np.testing.assert_allclose(ours, e / e.sum(), rtol=0, atol=1e-13)


def test_scale_zero_gives_mean():
    w = _small(seed=6, lens=(2, 11, 29), scale=0.0)
    out = oracle.decode(**_np(w), scale=0.0)
    _, V = _dense(w)
    G = w.Hq // w.Hkv
    for s in range(w.S):
        L = int(w.lens[s])
        for h in range(w.Hq):
            np.testing.assert_allclose(out[s, h], V[s, h // G, :L].mean(axis=0), rtol=0,
                                       atol=1e-14)


def test_gqa_head_mapping():
    """V of KV head g is the constant g: query head h must output h // G."""
    for Hq, Hkv in [(8, 2), (12, 4), (6, 3), (4, 1)]:
        w = _small(seed=7, Hq=Hq, Hkv=Hkv, lens=(4, 9, 21))
        inp = _np(w)
        v = inp["v_cache"].copy()
        for g in range(Hkv):
            v[:, g] = np.float16(g)
        inp["v_cache"] = v
        out = oracle.decode(**inp, scale=w.scale)
        G = Hq // Hkv
        for h in range(Hq):
            np.testing.assert_allclose(out[:, h], float(h // G), rtol=0, atol=1e-14,
                                       err_msg=f"Hq={Hq} Hkv={Hkv} h={h}")


def test_zero_length():
    w = _small(seed=8, lens=(0, 5, 0))
    out = oracle.decode(**_np(w), scale=w.scale)
    assert np.all(out[0] == 0) and np.all(out[2] == 0)
    assert np.all(np.isfinite(out[1])) and np.any(out[1] != 0)
    reads = oracle.page_reads(w.block_tables.numpy(), w.seq_lens.numpy(), w.Hkv, w.BS, w.NB)
    assert np.all(reads[0] == -1) and np.all(reads[2] == -1)


# ---------------------------------------------------------------- invariants
def test_page_permutation_invariance():
    w = _small(seed=9, lens=(13, 33, 7), BS=4)
    inp = _np(w)
    out = oracle.decode(**inp, scale=w.scale)
    rng = np.random.default_rng(1)
    perm = rng.permutation(w.NB)               # physical page p moves to perm[p]
    k2 = np.empty_like(inp["k_cache"])
    v2 = np.empty_like(inp["v_cache"])
    k2[perm] = inp["k_cache"]
    v2[perm] = inp["v_cache"]
    bt2 = perm[inp["block_tables"]].astype(np.int32)
    out2 = oracle.decode(q=inp["q"], k_cache=k2, v_cache=v2, block_tables=bt2,
                         seq_lens=inp["seq_lens"], scale=w.scale)
    assert np.array_equal(out, out2)


def test_poison_never_read():
    """NaN tail rows, NaN unowned pages and random page-table entries past
    the last page change nothing."""
    w = _small(seed=10, lens=(5, 14, 31), BS=8, poison=True)
    assert w.meta["poison"]
    out = oracle.decode(**_np(w), scale=w.scale)
    assert np.all(np.isfinite(out))
    clean = _small(seed=10, lens=(5, 14, 31), BS=8, poison=False)
    out_clean = oracle.decode(**_np(clean), scale=clean.scale)
    assert np.array_equal(out, out_clean)
    reads = oracle.page_reads(w.block_tables.numpy(), w.seq_lens.numpy(), w.Hkv, w.BS, w.NB)
    for s in range(w.S):
        own = w.page_ids[w.page_offsets[s]:w.page_offsets[s + 1]].numpy()
        for g in range(w.Hkv):
            assert reads[s, g, :len(own)].tolist() == own.tolist()
            assert np.all(reads[s, g, len(own):] == -1)


def test_online_log2_equals_definition():
    w = _small(seed=12, lens=(1, 50, 97), std=1.5)
    inp = _np(w)
    a = oracle.decode(**inp, scale=w.scale)
    b = oracle.online_log2(**inp, scale=w.scale)
    np.testing.assert_allclose(a, b, rtol=0, atol=1e-12)


@pytest.mark.parametrize("P", [1, 4, 7, 16, 100, 256, 512, 4096])
def test_split_invariance(P):
    w = _small(seed=13, lens=(1, 37, 300, 700), BS=4, std=1.5, Hq=4, Hkv=2)
    inp = _np(w)
    ref = oracle.decode(**inp, scale=w.scale)
    m, l, o = oracle.split_partials(**inp, scale=w.scale, P=P)
    assert np.all(l[np.isfinite(m)] >= 1.0)       # the max token contributes exactly 1
    out = oracle.merge_partials(m, l, o)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_merge_skips_empty_partitions():
    w = _small(seed=14, lens=(3, 40), BS=4, Hq=2, Hkv=1)
    inp = _np(w)
    m, l, o = oracle.split_partials(**inp, scale=w.scale, P=8, NPmax=9)
    assert np.all(l[0, :, 1:] == 0) and np.all(np.isneginf(m[0, :, 1:]))
    np.testing.assert_allclose(oracle.merge_partials(m, l, o),
                               oracle.decode(**inp, scale=w.scale), rtol=0, atol=1e-12)


def test_rejects_bad_inputs():
    w = _small(seed=15, lens=(5, 9, 2))
    inp = _np(w)
    bt = inp["block_tables"].copy()
    bt[1, 0] = w.NB                       # a page that must be read is out of range
    with pytest.raises(ValueError):
        oracle.decode(**{**inp, "block_tables": bt}, scale=w.scale)
    sl = inp["seq_lens"].copy()
    sl[0] = w.MB * w.BS + 1               # longer than the page table row
    with pytest.raises(ValueError):
        oracle.decode(**{**inp, "seq_lens": sl}, scale=w.scale)
    bt = inp["block_tables"].copy()
    bt[2, 1:] = -5                        # entries past the last page are not read
    oracle.decode(**{**inp, "block_tables": bt}, scale=w.scale)


# ---------------------------------------------------------------- KV-cache append
def _new_kv(w, seed):
    g = torch.Generator().manual_seed(seed)
    kn = torch.randn((w.S, w.Hkv, w.D), generator=g).to(torch.float16).numpy()
    vn = torch.randn((w.S, w.Hkv, w.D), generator=g).to(torch.float16).numpy()
    return kn, vn


def test_append_writes_only_the_newest_rows():
    w = _small(seed=21, lens=(0, 1, 8, 13), BS=4)
    kn, vn = _new_kv(w, 1)
    inp = _np(w)
    k2, v2 = oracle.append_kv(inp["k_cache"], inp["v_cache"], kn, vn, inp["block_tables"],
                              inp["seq_lens"])
    expect_k = inp["k_cache"].view(np.uint16).copy()
    expect_v = inp["v_cache"].view(np.uint16).copy()
    for s in range(w.S):          # where the generator placed token L-1
        L = int(w.lens[s])
        if L == 0:
            continue
        page = int(w.page_ids[w.page_offsets[s] + (L - 1) // w.BS])
        expect_k[page, :, (L - 1) % w.BS] = kn[s].view(np.uint16)
        expect_v[page, :, (L - 1) % w.BS] = vn[s].view(np.uint16)
    assert np.array_equal(k2.view(np.uint16), expect_k)
    assert np.array_equal(v2.view(np.uint16), expect_v)


def test_append_then_decode_closed_forms():
    # L = 1: the output is the appended value; poison in the slot is overwritten
    w = _small(seed=22, lens=(1, 1, 1), BS=8)
    inp = _np(w)
    for s in range(w.S):
        page = int(w.page_ids[w.page_offsets[s]])
        inp["k_cache"][page, :, 0] = np.float16("nan")
        inp["v_cache"][page, :, 0] = np.float16("nan")
    kn, vn = _new_kv(w, 2)
    out = oracle.decode_append(inp["q"], kn, vn, inp["k_cache"], inp["v_cache"],
                               inp["block_tables"], inp["seq_lens"], w.scale)
    G = w.Hq // w.Hkv
    for s in range(w.S):
        for h in range(w.Hq):
            assert np.array_equal(out[s, h], vn[s, h // G].astype(np.float64))
    # longer: equals the plain decode of caches holding the new rows
    w = _small(seed=23, lens=(5, 16, 33), BS=4)
    inp = _np(w)
    kn, vn = _new_kv(w, 3)
    k2, v2 = inp["k_cache"].copy(), inp["v_cache"].copy()
    for s in range(w.S):
        L = int(w.lens[s])
        page = int(w.page_ids[w.page_offsets[s] + (L - 1) // w.BS])
        k2[page, :, (L - 1) % w.BS] = kn[s]
        v2[page, :, (L - 1) % w.BS] = vn[s]
    a = oracle.decode_append(inp["q"], kn, vn, inp["k_cache"], inp["v_cache"],
                             inp["block_tables"], inp["seq_lens"], w.scale)
    b = oracle.decode(inp["q"], k2, v2, inp["block_tables"], inp["seq_lens"], w.scale)
    assert np.array_equal(a, b)


# ---------------------------------------------------------------- cache layouts
def _layouts(inp):
    """The same cache in three layouts, as (name, k_flat, v_flat, strides):
    token-major [NB][BS][Hkv][D] (a numpy transpose), pages padded with NaN
    between them, and rows padded with NaN to D + 8 halves."""
    k, v = inp["k_cache"], inp["v_cache"]
    NB, Hkv, BS, D = k.shape
    tm = lambda a: np.ascontiguousarray(a.transpose(0, 2, 1, 3))
    pad_page = 24

    def padded_pages(a):
        b = np.full((NB, Hkv * BS * D + pad_page), np.float16("nan"), dtype=np.float16)
        b[:, :Hkv * BS * D] = a.reshape(NB, -1)
        return b

    def padded_rows(a):
        b = np.full((NB, Hkv, BS, D + 8), np.float16("nan"), dtype=np.float16)
        b[..., :D] = a
        return b

    return [
        ("token_major", tm(k), tm(v), (BS * Hkv * D, D, Hkv * D)),
        ("padded_pages", padded_pages(k), padded_pages(v), (Hkv * BS * D + pad_page, BS * D, D)),
        ("padded_rows", padded_rows(k), padded_rows(v),
         (Hkv * BS * (D + 8), BS * (D + 8), D + 8)),
        ("head_major", k, v, (Hkv * BS * D, BS * D, D)),
    ]


def test_strided_layouts_equal_head_major():
    """The strided form reads the same numbers whatever the layout: bitwise
    equal to the head-major decode (layouts built by numpy, not the oracle;
    a swapped head/token stride or a read of the padding fails here)."""
    w = _small(seed=31, Hq=8, Hkv=2, D=16, BS=4, lens=(0, 1, 7, 13, 16))
    inp = _np(w)
    ref = oracle.decode(**inp, scale=w.scale)
    NB, Hkv, BS, D = inp["k_cache"].shape
    for name, kf, vf, strides in _layouts(inp):
        out = oracle.decode_strided(inp["q"], kf, vf, inp["block_tables"], inp["seq_lens"],
                                    w.scale, Hkv, BS, NB, strides)
        assert np.array_equal(out, ref), name


def test_strided_append_equals_head_major_append():
    w = _small(seed=32, lens=(0, 1, 8, 13), BS=4)
    inp = _np(w)
    kn, vn = _new_kv(w, 4)
    k_ref, v_ref = oracle.append_kv(inp["k_cache"], inp["v_cache"], kn, vn,
                                    inp["block_tables"], inp["seq_lens"])
    NB, Hkv, BS, D = inp["k_cache"].shape
    kf, vf = (np.ascontiguousarray(a.transpose(0, 2, 1, 3)) for a in (inp["k_cache"],
                                                                      inp["v_cache"]))
    k2, v2 = oracle.append_kv_strided(kf, vf, kn, vn, inp["block_tables"], inp["seq_lens"], Hkv,
                                      BS, NB, (BS * Hkv * D, D, Hkv * D))
    back = lambda a: np.ascontiguousarray(a.reshape(NB, BS, Hkv, D).transpose(0, 2, 1, 3))
    assert np.array_equal(back(k2).view(np.uint16), k_ref.view(np.uint16))
    assert np.array_equal(back(v2).view(np.uint16), v_ref.view(np.uint16))
