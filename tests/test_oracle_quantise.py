"""Pins for the oracle's quantiser (binary16 rows -> 8-bit codes with a bf16
(scale, bias) pair per group of 64, the reading side of which is the
Kapitsa series' affine group format).  The pages give no quantiser; the
reading taken is bias = bf16(min), scale = bf16((max - min) / 255),
code = clamp(rint((x - bias) / scale), 0, 255), every step in binary32.

  inverse of the pages' worked example     -> test_worked_example_inverted
  exact grid (codes recovered exactly)      -> test_exact_grid
  rounding rule (ties to even)              -> test_ties_go_to_even
  scale 0 / constant group                  -> test_constant_group
  error bound of the round trip             -> test_round_trip_bound
  bf16 rounding of the pair                 -> test_pair_is_bf16_of_min_and_step
  codes counted from the stored bias        -> test_codes_count_from_the_stored_bias
  row addressing of the cache writes        -> test_rows_land_at_their_slots,
                                               test_append_is_the_newest_row
"""
import json
import os

import numpy as np
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "affine_dequant.json")


def _bf16(x):
    """bf16 bits of float values, nearest with ties to even (torch)."""
    return torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16).view(
        torch.int16).numpy().view(np.uint16)


def _f32(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).astype(np.uint32).view(np.float32)


def test_worked_example_inverted():
    """A group whose minimum is the example's bias and whose range is 255
    steps of its scale holds the example's values at the example's codes."""
    for c in json.load(open(GOLDEN))["cases"]:
        s, b = c["scale"], c["bias"]
        k = np.concatenate([[0, 255], c["codes"], np.arange(60) * 4 + 2])[:64]
        x = (b + s * k).astype(np.float16)
        assert np.array_equal(x.astype(np.float64), b + s * k)  # exact in binary16
        codes, pair = oracle.quantise_affine(x)
        assert np.array_equal(pair[0], _bf16([s, b]))
        assert codes[2:2 + len(c["codes"])].tolist() == c["codes"]
        got = oracle.dequant_affine(codes[2:2 + len(c["codes"])], pair, group=len(c["codes"]))
        assert got.tolist() == c["values"]


def test_exact_grid():
    rng = np.random.default_rng(5)
    for b, s in [(-2.0, 2.0 ** -6), (0.5, 2.0 ** -9), (-0.75, 2.0 ** -8)]:
        k = np.concatenate([[0, 255], rng.integers(0, 256, 62)])
        rng.shuffle(k)
        x = (b + s * k).astype(np.float16)
        assert np.array_equal(x.astype(np.float64), b + s * k)
        codes, pair = oracle.quantise_affine(x)
        assert np.array_equal(codes, k.astype(np.uint8))
        assert np.array_equal(pair[0], _bf16([s, b]))


def test_ties_go_to_even():
    # bias 0, scale 1/64: x = (2j + 1) / 128 sits half-way between codes j, j+1
    j = np.arange(62)
    x = np.concatenate([[0.0, 255 / 64], (2 * j + 1) / 128]).astype(np.float16)
    codes, pair = oracle.quantise_affine(x)
    assert np.array_equal(pair[0], _bf16([1 / 64, 0.0]))
    want = np.where(j % 2 == 0, j, j + 1)
    assert np.array_equal(codes[2:], want.astype(np.uint8))


def test_constant_group():
    for v in [0.0, 0.1, -3.5, 1000.0]:
        x = np.full(64, v, dtype=np.float16)
        codes, pair = oracle.quantise_affine(x)
        assert not codes.any()
        assert pair[0, 0] == 0
        assert pair[0, 1] == _bf16([np.float32(np.float16(v))])[0]


def test_pair_is_bf16_of_min_and_step():
    rng = np.random.default_rng(9)
    x = (rng.standard_normal(64 * 50) * 3 + rng.standard_normal(50).repeat(64)).astype(np.float16)
    codes, pairs = oracle.quantise_affine(x)
    g = x.astype(np.float32).reshape(50, 64)
    mn, mx = g.min(1), g.max(1)
    step = ((mx - mn).astype(np.float32) / np.float32(255)).astype(np.float32)
    assert np.array_equal(pairs[:, 0], _bf16(step))
    assert np.array_equal(pairs[:, 1], _bf16(mn))


def test_round_trip_bound():
    rng = np.random.default_rng(11)
    x = (rng.standard_normal(64 * 200) * rng.uniform(0.01, 50, 200).repeat(64)).astype(np.float16)
    codes, pairs = oracle.quantise_affine(x)
    back = oracle.dequant_affine(codes, pairs).reshape(200, 64)
    g = x.astype(np.float64).reshape(200, 64)
    S = _f32(pairs[:, 0]).astype(np.float64)[:, None]
    mn, mx = np.abs(g.min(1))[:, None], np.abs(g.max(1))[:, None]
    # half a step, plus what bf16 rounding of bias and step can move the ends
    bound = S / 2 + 2.0 ** -8 * (mn + mx) + 1e-6
    assert np.all(np.abs(back - g) <= bound)
    # the codes span the range: within a few steps of 0 and 255 (bf16 rounding
    # of the pair moves the ends by up to 2^-9 of |min| and 255 * 2^-9 steps)
    c = codes.reshape(200, 64).astype(int)
    lo = np.ceil(2.0 ** -9 * mn[:, 0] / S[:, 0] + 0.5)
    assert np.all(c.min(1) <= lo)
    assert np.all(c.max(1) >= 255 - np.ceil(255 * 2.0 ** -9 + lo))


def test_rows_land_at_their_slots():
    rng = np.random.default_rng(13)
    NB, Hkv, BS, D = 6, 2, 4, 128
    codes = rng.integers(0, 256, (NB, Hkv, BS, D)).astype(np.uint8)
    meta = rng.integers(0, 65536, (NB, Hkv, BS, D // 64, 2)).astype(np.uint16)
    src = rng.standard_normal((3, Hkv, D)).astype(np.float16)
    slots = np.array([5, -1, 4 * 5 + 3], dtype=np.int32)  # page 1 row 1, skipped, page 5 row 3
    c2, m2 = oracle.quantise_rows(codes, meta, src, slots)
    touched = np.zeros((NB, BS), dtype=bool)
    for n, slot in enumerate(slots):
        if slot < 0:
            continue
        p, r = divmod(int(slot), BS)
        touched[p, r] = True
        for h in range(Hkv):
            want_c, want_m = oracle.quantise_affine(src[n, h])
            assert np.array_equal(c2[p, h, r], want_c)
            assert np.array_equal(m2[p, h, r], want_m)
    for p in range(NB):
        for r in range(BS):
            if not touched[p, r]:
                assert np.array_equal(c2[p, :, r], codes[p, :, r])
                assert np.array_equal(m2[p, :, r], meta[p, :, r])


def test_append_is_the_newest_row():
    rng = np.random.default_rng(17)
    NB, Hkv, BS, D, S, MB = 10, 2, 8, 256, 3, 3
    kc = rng.integers(0, 256, (NB, Hkv, BS, D)).astype(np.uint8)
    vc = rng.integers(0, 256, (NB, Hkv, BS, D)).astype(np.uint8)
    km = rng.integers(0, 65536, (NB, Hkv, BS, D // 64, 2)).astype(np.uint16)
    vm = rng.integers(0, 65536, (NB, Hkv, BS, D // 64, 2)).astype(np.uint16)
    bt = np.array([[7, 2, 0], [3, 0, 0], [9, 8, 1]], dtype=np.int32)
    lens = np.array([11, 0, 17], dtype=np.int32)
    kn = rng.standard_normal((S, Hkv, D)).astype(np.float16)
    vn = rng.standard_normal((S, Hkv, D)).astype(np.float16)
    got = oracle.append_kv_q8(kc, km, vc, vm, kn, vn, bt, lens)
    slots = np.array([2 * BS + 2, -1, 1 * BS + 0], dtype=np.int32)  # page 2 row 2; -; page 1 row 0
    want_k = oracle.quantise_rows(kc, km, kn, slots)
    want_v = oracle.quantise_rows(vc, vm, vn, slots)
    for a, b in zip(got, want_k + want_v):
        assert np.array_equal(a, b)


def test_codes_count_from_the_stored_bias():
    """The minimum 1 + 2^-10 is not a bf16 value (it is stored as 1.0), the
    step 2^-10 is: values on the stored grid 1.0 + c * 2^-10 come back
    exactly, so the codes are counted from the stored bias, not the minimum
    (the maximum, one step past code 255, clamps)."""
    k = np.arange(64)
    x = (1 + 2.0 ** -10 + 2.0 ** -10 * np.concatenate([[255], k[:63] * 4])).astype(np.float16)
    codes, pair = oracle.quantise_affine(x)
    assert np.array_equal(pair[0], _bf16([2.0 ** -10, 1.0]))
    back = oracle.dequant_affine(codes, pair)
    assert np.array_equal(back[1:], x[1:].astype(np.float64))
    assert codes[0] == 255 and back[0] == 1 + 255 * 2.0 ** -10
