"""Pins for the oracle's quantised-KV decode (8-bit codes, affine group-64
format with bf16 (scale, bias)).

  dequantisation formula           -> test_worked_example (the pages' numbers)
  bf16 decoding                    -> test_bf16_decoding_matches_torch
  code / metadata addressing, K/V  -> test_equals_fp16_decode_on_exact_values,
                                      test_dense_sdpa_on_dequantised_values
  strided layouts (codes, pairs)   -> test_strided_q8_equals_head_major,
                                      test_strided_q8_append_equals_head_major
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from paged_gqa_decode_03_gb300.workloads import make_custom, make_q8

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "affine_dequant.json")


def _bf16_bits(x):
    return torch.tensor(x, dtype=torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_worked_example():
    for c in json.load(open(GOLDEN))["cases"]:
        meta = _bf16_bits([[c["scale"], c["bias"]]])
        got = oracle.dequant_affine(np.array(c["codes"], dtype=np.uint8), meta,
                                    group=len(c["codes"]))
        assert got.tolist() == c["values"]


def test_bf16_decoding_matches_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_double(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])


def _q8(seed, Hq=8, Hkv=2, D=128, BS=8, lens=(1, 9, 23, 40)):
    w = make_custom(S=len(lens), Hq=Hq, Hkv=Hkv, D=D, BS=BS, lens=list(lens), seed=seed,
                    device="cpu", NB=int(sum((l + BS - 1) // BS for l in lens)) + 3)
    return w, make_q8(w)


def _np(t):
    return t.numpy() if t.dtype != torch.int16 else t.numpy().view(np.uint16)


def test_equals_fp16_decode_on_exact_values():
    """With scale 2^-5 and biases on the 2^-5 grid every dequantised value is
    exact in fp16: the quantised decode must equal the fp16 decode of those
    values bit for bit (same fp64 arithmetic on the same numbers)."""
    w, c = _q8(31)
    rng = np.random.default_rng(0)
    out = []
    for codes, meta in ((c.k_codes, c.k_meta), (c.v_codes, c.v_meta)):
        m = meta.view(torch.bfloat16).clone()
        m[..., 0] = 2.0 ** -5
        m[..., 1] = torch.from_numpy(rng.integers(-160, -96, size=m.shape[:-1]) / 32.0).to(
            torch.bfloat16)
        vals = (codes.double() * m[..., 0].double().repeat_interleave(64, -1)
                + m[..., 1].double().repeat_interleave(64, -1))
        out.append((codes.numpy(), m.view(torch.int16).numpy().view(np.uint16),
                    vals.to(torch.float16).numpy()))
        assert torch.equal(vals.to(torch.float16).double(), vals)     # exact in fp16
    (kc, km, kf), (vc, vm, vf) = out
    bt, sl, q = w.block_tables.numpy(), w.seq_lens.numpy(), w.q.numpy()
    a = oracle.decode_q8(q, kc, km, vc, vm, bt, sl, w.scale)
    b = oracle.decode(q, kf, vf, bt, sl, w.scale)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("Hq,Hkv,BS", [(8, 2, 8), (4, 4, 16)])
def test_dense_sdpa_on_dequantised_values(Hq, Hkv, BS):
    """Against torch's scaled_dot_product_attention (float64) on rows
    dequantised with torch and gathered by the generator's page record."""
    w, c = _q8(40 + Hq, Hq=Hq, Hkv=Hkv, BS=BS)
    out = oracle.decode_q8(w.q.numpy(), c.k_codes.numpy(), _np(c.k_meta), c.v_codes.numpy(),
                           _np(c.v_meta), w.block_tables.numpy(), w.seq_lens.numpy(), w.scale)

    def deq(codes, meta):
        m = meta.view(torch.bfloat16).double()
        return codes.double() * m[..., 0].repeat_interleave(64, -1) + m[..., 1].repeat_interleave(64, -1)
    K, V = deq(c.k_codes, c.k_meta), deq(c.v_codes, c.v_meta)
    G = Hq // Hkv
    q = w.q.double()
    for s in range(w.S):
        L = int(w.lens[s])
        own = w.page_ids[w.page_offsets[s]:w.page_offsets[s + 1]]
        idx = torch.arange(L)
        Kd = K[own[idx // BS], :, idx % BS].transpose(0, 1).repeat_interleave(G, 0)
        Vd = V[own[idx // BS], :, idx % BS].transpose(0, 1).repeat_interleave(G, 0)
        ref = torch.nn.functional.scaled_dot_product_attention(q[s][:, None], Kd, Vd,
                                                               scale=w.scale)[:, 0]
        np.testing.assert_allclose(out[s], ref.numpy(), rtol=0, atol=1e-12)


def test_poison_metadata_never_read():
    w, c = _q8(50)
    out = oracle.decode_q8(w.q.numpy(), c.k_codes.numpy(), _np(c.k_meta), c.v_codes.numpy(),
                           _np(c.v_meta), w.block_tables.numpy(), w.seq_lens.numpy(), w.scale)
    assert np.all(np.isfinite(out))


def _q8_layouts(codes, meta, pad_row=16, pad_page=48):
    """One quantised array pair in three layouts built by numpy, as (name,
    codes_flat, meta_flat, code_strides, meta_strides): token-major
    [NB][BS][Hkv][...], rows padded (codes by pad_row bytes, pairs by one
    extra pair, both padded with 0xFF / NaN bits), pages padded."""
    NB, Hkv, BS, D = codes.shape
    NM = (D // 64) * 2
    m = meta.reshape(NB, Hkv, BS, NM)
    tm = lambda a: np.ascontiguousarray(a.transpose(0, 2, 1, 3))
    pc = np.full((NB, Hkv, BS, D + pad_row), 0xFF, dtype=np.uint8)
    pc[..., :D] = codes
    pm = np.full((NB, Hkv, BS, NM + 2), 0x7FC1, dtype=np.uint16)
    pm[..., :NM] = m
    gc = np.full((NB, Hkv * BS * D + pad_page), 0xFF, dtype=np.uint8)
    gc[:, :Hkv * BS * D] = codes.reshape(NB, -1)
    gm = np.full((NB, Hkv * BS * NM + 8), 0x7FC1, dtype=np.uint16)
    gm[:, :Hkv * BS * NM] = m.reshape(NB, -1)
    return [
        ("token_major", tm(codes), tm(m), (BS * Hkv * D, D, Hkv * D), (BS * Hkv * NM, NM, Hkv * NM)),
        ("padded_rows", pc, pm, (Hkv * BS * (D + pad_row), BS * (D + pad_row), D + pad_row),
         (Hkv * BS * (NM + 2), BS * (NM + 2), NM + 2)),
        ("padded_pages", gc, gm, (Hkv * BS * D + pad_page, BS * D, D),
         (Hkv * BS * NM + 8, BS * NM, NM)),
    ]


@pytest.mark.parametrize("D,BS", [(128, 8), (256, 16)])
def test_strided_q8_equals_head_major(D, BS):
    """The strided quantised decode reads the same numbers whatever the
    layout: bitwise equal to the head-major one (layouts built by numpy; a
    swapped head/token stride or a read of the padding fails here)."""
    w, c = _q8(61 + D, D=D, BS=BS, lens=(0, 1, 9, 23, 40))
    args = (w.block_tables.numpy(), w.seq_lens.numpy(), w.scale)
    ref = oracle.decode_q8(w.q.numpy(), c.k_codes.numpy(), _np(c.k_meta), c.v_codes.numpy(),
                           _np(c.v_meta), *args)
    NB, Hkv = c.k_codes.shape[:2]
    lk = _q8_layouts(c.k_codes.numpy(), _np(c.k_meta))
    lv = _q8_layouts(c.v_codes.numpy(), _np(c.v_meta))
    for (name, kc, km, cs, ms), (_, vc, vm, _, _) in zip(lk, lv):
        out = oracle.decode_q8_strided(w.q.numpy(), kc, km, vc, vm, *args, Hkv, BS, NB, cs, ms)
        assert np.array_equal(out, ref), name


def test_strided_q8_append_equals_head_major():
    w, c = _q8(71, D=128, BS=8, lens=(0, 1, 8, 23))
    rng = np.random.default_rng(3)
    kn = rng.standard_normal((w.S, w.Hkv, 128)).astype(np.float16)
    vn = rng.standard_normal((w.S, w.Hkv, 128)).astype(np.float16)
    bt, sl = w.block_tables.numpy(), w.seq_lens.numpy()
    kc, km, vc, vm = c.k_codes.numpy(), _np(c.k_meta), c.v_codes.numpy(), _np(c.v_meta)
    ref = oracle.append_kv_q8(kc, km, vc, vm, kn, vn, bt, sl)
    NB, Hkv, BS, D = kc.shape
    tm = lambda a: np.ascontiguousarray(a.reshape(NB, Hkv, BS, -1).transpose(0, 2, 1, 3))
    got = oracle.append_kv_q8_strided(tm(kc), tm(km), tm(vc), tm(vm), kn, vn, bt, sl, Hkv, BS,
                                      NB, (BS * Hkv * D, D, Hkv * D), (BS * Hkv * 4, 4, Hkv * 4))
    back = lambda a, n: np.ascontiguousarray(a.reshape(NB, BS, Hkv, n).transpose(0, 2, 1, 3))
    assert np.array_equal(back(got[0], D), ref[0])
    assert np.array_equal(back(got[1], 4), ref[1].reshape(NB, Hkv, BS, 4))
    assert np.array_equal(back(got[2], D), ref[2])
    assert np.array_equal(back(got[3], 4), ref[3].reshape(NB, Hkv, BS, 4))
