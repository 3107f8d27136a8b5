"""Logical-rank all-to-all with put + signal + epoch, GPU against the oracle.

A byte copy: every receive buffer must match the oracle bit for bit, every
peer flag must hold the epoch, and the send buffers must be untouched."""
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


@pytest.mark.parametrize("R,B,order", [
    (2, 4096, None),
    (3, 48, (1, 2, 0)),               # less than one piece per slice
    (4, 3 * 32768 + 1040, (3, 0, 2, 1)),  # several pieces and a ragged tail
    (8, 65536, None),
    (1, 1024, None),
])
def test_matches_oracle_bit_for_bit(api, R, B, order):
    d = inputs.alltoall_inputs(R, B, seed=R * 3 + B, slot_order=order)
    heap = torch.from_numpy(d["heap"]).cuda()
    F = api.alltoall_num_flags(R, B)
    sig = api.Signal(F)
    for _ in range(3):
        e = sig.next_epoch()
        api.alltoall(heap, d["rank_off"], d["send_off"], d["recv_off"], B, sig, e)
        assert sig.status()[0] == api.OK
        flags = sig.flags().cpu().numpy()[:F].reshape(R, R, -1)
        for j in range(R):
            for r in range(R):
                if r != j:
                    assert np.all(flags[j, r] == e)
    got = heap.cpu().numpy()
    ref = oracle.alltoall(d["heap"], d["rank_off"], R, d["send_off"], d["recv_off"], B)
    assert np.array_equal(got, ref)
