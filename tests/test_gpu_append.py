"""GPU parity of the fused KV-cache append + decode (paged_gqa_decode_append)
against the oracle's append_kv + decode; the cache afterwards must hold the
new rows bit-exactly and nothing else may change."""
import numpy as np
import pytest
import torch

import oracle
import paged_gqa_decode_03_gb300 as pgd
from paged_gqa_decode_03_gb300.workloads import make_custom, make_workload
from parity_util import assert_parity

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    yield
    assert pgd.pgd_check_device_error() == 0


def _slot(w, s):
    """(physical page, row) of token seq_lens[s] - 1, from the generator's record."""
    L = int(w.lens[s])
    return int(w.page_ids[w.page_offsets[s] + (L - 1) // w.BS]), (L - 1) % w.BS


def check_append(w, P=None, seed=0):
    g = torch.Generator(device=DEV).manual_seed(seed)
    kn = torch.randn((w.S, w.Hkv, w.D), generator=g, device=DEV).to(torch.float16)
    vn = torch.randn((w.S, w.Hkv, w.D), generator=g, device=DEV).to(torch.float16)
    for s in range(w.S):     # the slot holds garbage before the call
        if w.lens[s]:
            page, row = _slot(w, s)
            w.k_cache[page, :, row] = float("nan")
            w.v_cache[page, :, row] = float("nan")
    before_k, before_v = w.k_cache.clone(), w.v_cache.clone()
    c = w.compact()
    ref = oracle.decode_append(c["q"], kn.cpu().numpy(), vn.cpu().numpy(), c["k_cache"],
                               c["v_cache"], c["block_tables"], c["seq_lens"], c["scale"])
    out = torch.full((w.S, w.Hq, w.D), float("nan"), dtype=torch.float32, device=DEV)
    pgd.paged_gqa_decode_append(out, w.q, kn, vn, w.k_cache, w.v_cache, w.block_tables,
                                w.seq_lens, w.scale, w.P if P is None else P)
    torch.cuda.synchronize()
    assert_parity(out.cpu().numpy(), ref, f"{w.name} append")
    # the cache: new rows written, everything else unchanged (bitwise)
    expect_k, expect_v = before_k.view(torch.int16), before_v.view(torch.int16)
    for s in range(w.S):
        if w.lens[s]:
            page, row = _slot(w, s)
            expect_k[page, :, row] = kn[s].view(torch.int16)
            expect_v[page, :, row] = vn[s].view(torch.int16)
    assert torch.equal(w.k_cache.view(torch.int16), expect_k)
    assert torch.equal(w.v_cache.view(torch.int16), expect_v)
    assert pgd.pgd_check_device_error() == 0
    return out, kn, vn


@pytest.mark.parametrize("name", ["batch_decode", "long_context", "ragged_tails", "serving_mix"])
def test_append_workloads_reduced(name):
    check_append(make_workload(name, device=DEV, S=8, seed=41), seed=1)


def test_append_batch_decode_full():
    check_append(make_workload("batch_decode", device=DEV), seed=2)


@pytest.mark.parametrize("D", [128, 256])
@pytest.mark.parametrize("BS", [8, 16, 32])
def test_append_edge_lengths(D, BS):
    lens = [0, 1, 2, 7, 8, 9, 15, 16, 17, 33, 255, 256, 257, 511, 512, 513, 1000]
    w = make_custom(S=len(lens), Hq=16, Hkv=2, D=D, BS=BS, lens=lens, seed=D + BS,
                    device=DEV, MB=(1024 + BS - 1) // BS)
    for P in (256, 512):
        out, kn, vn = check_append(w, P=P, seed=P)
        assert torch.all(out[0] == 0)
        for h in range(w.Hq):        # length 1: the output is the appended value
            assert torch.equal(out[1, h], vn[1, h // (w.Hq // w.Hkv)].float())
