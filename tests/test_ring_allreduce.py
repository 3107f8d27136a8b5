"""Tile-centric ring AllReduce over logical ranks, GPU against the CPU oracle.

The kernel performs the same binary32 additions in the same ring order as
the oracle, so every rank's output must match it bit for bit; every flag
must hold the epoch; the input must be left untouched.
"""
import numpy as np
import pytest
import torch

import oracle
from overlap_producer_warps_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from overlap_producer_warps_gb300 import api as _api
    _api.lib()
    return _api


def _run(api, d, epochs=1):
    R, n = d["R"], d["n"]
    heap = torch.from_numpy(d["heap"]).cuda()
    F = api.ring_num_flags(R, n)
    sig = api.Signal(F)
    for _ in range(epochs):
        e = sig.next_epoch()
        api.ring_allreduce(heap, d["rank_off"], d["data_off"], d["recv_off"], d["out_off"], n, sig, e)
        st = sig.status()
        assert st[0] == api.OK, st
        if R > 1:
            assert np.all(sig.flags().cpu().numpy()[:F] == e)
    return heap.cpu().numpy(), sig


@pytest.mark.parametrize("R,n,order", [
    (2, 2 * 1024, None),
    (3, 3 * 400, (2, 0, 1)),          # chunk 400: one partial piece
    (4, 4 * 1024 * 3 + 4 * 36, (1, 3, 0, 2)),  # several pieces and a ragged tail
    (8, 8 * 4096, None),
    (1, 64, None),                    # single rank: output = input
    (5, 5 * 2052, (4, 3, 2, 1, 0)),
])
def test_matches_oracle_bit_for_bit(api, R, n, order):
    d = inputs.ring_inputs(R, n, seed=R + n, slot_order=order)
    got, _ = _run(api, d)
    ref = oracle.ring_allreduce(d["heap"], d["rank_off"], R, d["data_off"], d["out_off"], n)
    for j in range(R):
        o = int(d["rank_off"][j])
        out = got[o + d["out_off"]:o + d["out_off"] + n * 4]
        assert np.array_equal(out, ref[o + d["out_off"]:o + d["out_off"] + n * 4]), f"rank {j}"
        data = got[o + d["data_off"]:o + d["data_off"] + n * 4]
        assert np.array_equal(data, d["heap"][o + d["data_off"]:o + d["data_off"] + n * 4])


def test_epochs_reused_without_reset(api):
    R, n = 4, 4 * 2048
    d = inputs.ring_inputs(R, n, seed=7)
    got, sig = _run(api, d, epochs=5)
    ref = oracle.ring_allreduce(d["heap"], d["rank_off"], R, d["data_off"], d["out_off"], n)
    o = int(d["rank_off"][1]) + d["out_off"]
    assert np.array_equal(got[o:o + n * 4], ref[o:o + n * 4])


def test_large_ring(api):
    """8 ranks of 4 Mi fp32 values (16 MiB each): several waves of pieces per warp."""
    R, n = 8, 8 * (1 << 19)
    d = inputs.ring_inputs(R, n, seed=11)
    got, _ = _run(api, d, epochs=2)
    ref = oracle.ring_allreduce(d["heap"], d["rank_off"], R, d["data_off"], d["out_off"], n)
    for j in (0, 5):
        o = int(d["rank_off"][j]) + d["out_off"]
        assert np.array_equal(got[o:o + n * 4], ref[o:o + n * 4])
