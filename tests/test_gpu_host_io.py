"""paged_gqa_decode_host: the decode step with the step's inputs (q, page
tables, lengths) and its output in host memory, the K/V cache resident on
the device.  Checked against the oracle and bit for bit against
paged_gqa_decode on the same inputs (the same kernels run on the staged
copies)."""
import ctypes

import numpy as np
import pytest
import torch

import paged_gqa_decode_03_gb300 as pgd
from paged_gqa_decode_03_gb300.workloads import make_custom, make_workload
from parity_util import assert_parity, oracle_out, run

pytestmark = pytest.mark.gpu

DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()
    torch.cuda.set_device(0)
    pgd.pgd_check_device_error()
    yield


def host_inputs(w, pinned=True):
    pin = (lambda t: t.pin_memory()) if pinned else (lambda t: t)
    return (pin(torch.empty((w.S, w.Hq, w.D), dtype=torch.float32)), pin(w.q.cpu()),
            pin(w.block_tables.cpu()), pin(w.seq_lens.cpu()))


@pytest.mark.parametrize("name,P,kw", [
    ("batch_decode", 512, dict(S=20, seed=81)),
    ("ragged_tails", 256, dict(S=24, seed=82)),
    ("long_context", 256, dict(S=3, seed=83)),
    ("tiny", 512, {}),
])
@pytest.mark.parametrize("pinned", [True, False])
def test_host_entry_matches_device_entry_and_oracle(name, P, kw, pinned):
    w = make_workload(name, device=DEV, **kw)
    out_h, q_h, bt_h, sl_h = host_inputs(w, pinned)
    staging = torch.empty(pgd.pgd_host_staging_bytes(w.S, w.Hq, w.D, w.MB), dtype=torch.uint8,
                          device=DEV)
    staging.fill_(0xFF)                # stale contents must not matter
    ref = run(w, P=P).cpu().numpy()
    for call in range(2):
        out_h.fill_(float("nan"))
        pgd.paged_gqa_decode_host(out_h, q_h, bt_h, sl_h, w.k_cache, w.v_cache, w.scale,
                                  staging, P)
        got = out_h.numpy()            # valid on return: the call waited for its stream
        assert np.array_equal(got, ref), f"{name} call {call}: differs from paged_gqa_decode"
    assert_parity(got, oracle_out(w), f"{name} against the oracle")
    assert pgd.pgd_check_device_error() == 0


def test_host_entry_on_a_side_stream():
    w = make_custom(S=5, Hq=16, Hkv=2, D=128, BS=16, lens=[0, 1, 17, 700, 1300], seed=84,
                    device=DEV)
    out_h, q_h, bt_h, sl_h = host_inputs(w)
    staging = torch.empty(pgd.pgd_host_staging_bytes(w.S, w.Hq, w.D, w.MB), dtype=torch.uint8,
                          device=DEV)
    s = torch.cuda.Stream()
    pgd.paged_gqa_decode_host(out_h, q_h, bt_h, sl_h, w.k_cache, w.v_cache, w.scale, staging,
                              256, stream=s)
    got = out_h.numpy()
    assert np.all(got[0] == 0)         # an empty sequence gives zeros
    assert_parity(got, oracle_out(w), "side stream")


def test_host_entry_rejects_small_staging():
    w = make_workload("batch_decode", device=DEV, S=4, seed=85)
    out_h, q_h, bt_h, sl_h = host_inputs(w)
    need = pgd.pgd_host_staging_bytes(w.S, w.Hq, w.D, w.MB)
    staging = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    out_h.fill_(7.0)
    with pytest.raises(pgd.PGDError, match="staging"):
        pgd.paged_gqa_decode_host(out_h, q_h, bt_h, sl_h, w.k_cache, w.v_cache, w.scale,
                                  staging, 512)
    assert torch.all(out_h == 7.0)     # nothing copied back
