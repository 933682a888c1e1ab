"""Pins for the oracle's paged variable-length attention (several query tokens
per sequence, causal over the cached tokens up to each query's position).

What pins what:
  position of query i (L - n + i) or the causal bound wrong
        -> test_hand_case, test_dense_causal_sdpa, test_each_row_is_a_decode_of_its_prefix
  query rows read from the wrong place (row / sequence confusion)
        -> test_hand_case, test_dense_causal_sdpa
  decode not the n = 1 case -> test_single_token_rows_equal_decode
  page table / layout       -> test_page_permutation_invariance, test_dense_causal_sdpa
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_03_gb300.workloads import make_varlen

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "varlen_cases.json")


def _parse(x):
    if isinstance(x, list):
        return [_parse(y) for y in x]
    if isinstance(x, str):
        return float("nan") if x == "nan" else float(Fraction(x))
    return float(x)


def _inp(w):
    c = w.compact()
    return dict(q=c["q"], cu_seqlens_q=c["cu_seqlens_q"], k_cache=c["k_cache"],
                v_cache=c["v_cache"], block_tables=c["block_tables"], seq_lens=c["seq_lens"],
                scale=c["scale"])


def _small(seed, ctx, n, Hq=8, Hkv=2, D=16, BS=4, poison=True):
    return make_varlen(S=len(n), Hq=Hq, Hkv=Hkv, D=D, BS=BS, ctx=list(ctx), n=list(n),
                       seed=seed, device="cpu", poison=poison)


def test_hand_case():
    c = json.load(open(GOLDEN))["cases"][0]
    f16 = lambda a: np.asarray(_parse(a), dtype=np.float16)
    out = oracle.varlen(f16(c["q"]), np.asarray(c["cu_seqlens_q"], dtype=np.int32),
                        f16(c["k_cache"]), f16(c["v_cache"]),
                        np.asarray(c["block_tables"], dtype=np.int32),
                        np.asarray(c["seq_lens"], dtype=np.int32), math.log(3.0))
    np.testing.assert_allclose(out, np.asarray(_parse(c["out"])), rtol=0, atol=1e-13)


def _dense(w):
    """Dense K, V per sequence [Hkv, L, D] from the generator's record of
    which physical page holds which logical page (not the page table)."""
    base = w.base
    kc = base.k_cache.numpy().astype(np.float64)
    vc = base.v_cache.numpy().astype(np.float64)
    out = []
    for s in range(w.S):
        L = int(base.lens[s])
        own = base.page_ids[base.page_offsets[s]:base.page_offsets[s + 1]].numpy()
        K = np.stack([kc[own[t // w.BS], :, t % w.BS] for t in range(L)], axis=1)
        V = np.stack([vc[own[t // w.BS], :, t % w.BS] for t in range(L)], axis=1)
        out.append((K, V))
    return out


@pytest.mark.parametrize("Hq,Hkv,BS", [(8, 2, 4), (6, 3, 8), (4, 4, 4)])
def test_dense_causal_sdpa(Hq, Hkv, BS):
    """Against torch's scaled_dot_product_attention in float64 with an
    explicit causal mask aligned to the end of each sequence."""
    w = _small(5 + Hq + BS, ctx=[0, 3, 9, 30], n=[5, 1, 7, 12], Hq=Hq, Hkv=Hkv, BS=BS)
    out = oracle.varlen(**_inp(w))
    G = Hq // Hkv
    cu = w.cu_seqlens_q.numpy()
    q = torch.from_numpy(w.q.numpy().astype(np.float64))
    for s, (K, V) in enumerate(_dense(w)):
        n, L = int(w.q_lens[s]), int(w.base.lens[s])
        Kd = torch.from_numpy(K).repeat_interleave(G, dim=0)   # [Hq, L, D]
        Vd = torch.from_numpy(V).repeat_interleave(G, dim=0)
        qs = q[cu[s]:cu[s + 1]].transpose(0, 1)                  # [Hq, n, D]
        mask = torch.arange(L)[None, :] <= (L - n + torch.arange(n))[:, None]
        ref = torch.nn.functional.scaled_dot_product_attention(qs, Kd, Vd, attn_mask=mask,
                                                               scale=w.scale)
        np.testing.assert_allclose(out[cu[s]:cu[s + 1]], ref.transpose(0, 1).numpy(), rtol=0,
                                   atol=1e-12)


def test_each_row_is_a_decode_of_its_prefix():
    """Query i of sequence s equals a one-token decode of the same query over
    the sequence cut to its first L - n + i + 1 tokens."""
    w = _small(7, ctx=[0, 5, 20], n=[6, 3, 9])
    inp = _inp(w)
    out = oracle.varlen(**inp)
    cu = inp["cu_seqlens_q"]
    for s in range(w.S):
        n, L = int(w.q_lens[s]), int(inp["seq_lens"][s])
        for i in range(n):
            r = cu[s] + i
            one = oracle.decode(inp["q"][r:r + 1], inp["k_cache"], inp["v_cache"],
                                inp["block_tables"][s:s + 1],
                                np.array([L - n + i + 1], dtype=np.int32), inp["scale"])
            np.testing.assert_allclose(out[r], one[0], rtol=0, atol=1e-13)


def test_single_token_rows_equal_decode():
    w = _small(8, ctx=[0, 4, 17, 40], n=[1, 1, 1, 1])
    inp = _inp(w)
    out = oracle.varlen(**inp)
    ref = oracle.decode(inp["q"], inp["k_cache"], inp["v_cache"], inp["block_tables"],
                        inp["seq_lens"], inp["scale"])
    assert np.array_equal(out, ref)


def test_prompt_first_row_is_v0():
    """A whole prompt (n = L): its first query attends token 0 alone."""
    w = _small(9, ctx=[0, 0], n=[5, 9], poison=True)
    inp = _inp(w)
    out = oracle.varlen(**inp)
    G = w.Hq // w.Hkv
    for s in range(w.S):
        page = int(inp["block_tables"][s, 0])
        r = inp["cu_seqlens_q"][s]
        for h in range(w.Hq):
            assert np.array_equal(out[r, h], inp["v_cache"][page, h // G, 0].astype(np.float64))


def test_page_permutation_invariance():
    w = _small(10, ctx=[3, 11], n=[4, 6])
    inp = _inp(w)
    a = oracle.varlen(**inp)
    NB = inp["k_cache"].shape[0]
    perm = np.random.default_rng(0).permutation(NB)
    k2 = np.empty_like(inp["k_cache"])
    v2 = np.empty_like(inp["v_cache"])
    k2[perm] = inp["k_cache"]
    v2[perm] = inp["v_cache"]
    bt = np.where(inp["block_tables"] >= 0, perm[np.maximum(inp["block_tables"], 0)], -1)
    b = oracle.varlen(**{**inp, "k_cache": k2, "v_cache": v2,
                         "block_tables": bt.astype(np.int32)})
    assert np.array_equal(a, b)


def test_token_major_layout_equal():
    w = _small(11, ctx=[2, 13], n=[3, 5])
    inp = _inp(w)
    a = oracle.varlen(**inp)
    NB, Hkv, BS, D = inp["k_cache"].shape
    tm = lambda x: np.ascontiguousarray(x.transpose(0, 2, 1, 3))
    b = oracle.varlen(**{**inp, "k_cache": tm(inp["k_cache"]), "v_cache": tm(inp["v_cache"])},
                      layout=(Hkv, BS, NB, (BS * Hkv * D, D, Hkv * D)))
    assert np.array_equal(a, b)


def test_rejects_bad_inputs():
    w = _small(12, ctx=[0, 2], n=[3, 2])
    inp = _inp(w)
    bad = inp["cu_seqlens_q"].copy()
    bad[1] = 4                                   # 4 query tokens in a 3-token sequence
    bad_q = np.concatenate([inp["q"], inp["q"][:1]])
    bad[2] = 6
    with pytest.raises(ValueError):
        oracle.varlen(**{**inp, "cu_seqlens_q": bad, "q": bad_q})
