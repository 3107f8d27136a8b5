"""Failure detection without a GPU fault.

A tile whose flag is never published (or published with a stale epoch) must
make the consumer's bounded wait run out: the kernel latches TIMEOUT with the
rank and flag slot in the signal object's status word and returns, leaving
the context usable.  Host-side argument and epoch errors come back at once.
"""
import numpy as np
import pytest
import torch

from overlap_producer_warps_gb300 import inputs
from tests.helpers import AgProblem, assert_gemm_close, host_bits

pytestmark = pytest.mark.gpu

TIMEOUT_NS = 50_000_000  # 50 ms


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from overlap_producer_warps_gb300 import api as _api
    _api.lib()
    return _api


def _problem(seed=40):
    return AgProblem(inputs.ag_inputs(dict(R=4, M_r=128, K=256, N=512, dist="normal", scale=0.5),
                                      seed=seed))


@pytest.mark.parametrize("kind", ["drop", "stale"])
def test_missing_flag_times_out_and_recovers(api, kind):
    prob = _problem()
    F = api.ag_num_flags(4, 128, 256)
    sig = api.Signal(F)
    slot = 5
    fk = api.FAULT_DROP_TILE if kind == "drop" else api.FAULT_STALE_EPOCH
    prob.run(api, sig, sig.next_epoch(), api.make_opts(timeout_ns=TIMEOUT_NS, fault_kind=fk,
                                                       fault_arg=slot))
    status, rank, where = sig.status()
    assert status == api.ERR_TIMEOUT
    assert (rank, where) == (slot // (F // 4), slot)
    # the error is latched: further launches are refused until reset
    assert api.ag_gemm_status(prob.heap, prob.rank_off, prob.a_off, prob.M_r, prob.N, prob.K,
                              prob.B, prob.G, prob.C, sig, sig.next_epoch()) == api.ERR_NOT_READY
    # the context is still usable: reset and run correctly
    sig.reset()
    prob.run(api, sig, sig.next_epoch())
    assert sig.status()[0] == api.OK
    assert np.all(sig.flags().cpu().numpy() == 1)
    _, C_ref = prob.oracle_full()
    assert_gemm_close(host_bits(prob.C), C_ref)


def test_bad_epoch_is_refused_on_the_host(api):
    prob = _problem()
    sig = api.Signal(api.ag_num_flags(4, 128, 256))
    args = (prob.heap, prob.rank_off, prob.a_off, prob.M_r, prob.N, prob.K, prob.B, prob.G, prob.C)
    assert api.ag_gemm_status(*args, sig, 2) == api.ERR_BAD_EPOCH   # must be 1
    assert api.ag_gemm_status(*args, sig, 0) == api.ERR_BAD_EPOCH
    consumer = api.make_opts(role=api.ROLE_CONSUMER)
    assert api.ag_gemm_status(*args, sig, 1, consumer) == api.ERR_BAD_EPOCH  # nothing published yet
    assert api.ag_gemm_status(*args, sig, 1) == api.OK
    assert sig.status()[0] == api.OK
    assert api.ag_gemm_status(*args, sig, 1) == api.ERR_BAD_EPOCH   # epochs only move forward


def test_too_few_slots_and_misalignment(api):
    prob = _problem()
    small = api.Signal(3)
    args = (prob.heap, prob.rank_off, prob.a_off, prob.M_r, prob.N, prob.K, prob.B, prob.G, prob.C)
    assert api.ag_gemm_status(*args, small, 1) == api.ERR_INVALID_ARG
    sig = api.Signal(api.ag_num_flags(4, 128, 256))
    assert api.ag_gemm_status(prob.heap, prob.rank_off, 8, prob.M_r, prob.N, prob.K, prob.B,
                              prob.G, prob.C, sig, 1) == api.ERR_MISALIGNED


def test_row_add_missing_increment_times_out(api):
    prob = _problem()
    n_rows = api.ag_num_row_counters(4, 128, 256)
    sig = api.Signal(n_rows)
    # tile slot 5 = rank 2, row tile 0, k-tile 1: its row counter (slot 2) never completes
    prob.run(api, sig, sig.next_epoch(), api.make_opts(timeout_ns=TIMEOUT_NS,
                                                       fault_kind=api.FAULT_DROP_TILE, fault_arg=5,
                                                       signal_mode=api.SIGNAL_ROW_ADD))
    status, rank, where = sig.status()
    assert (status, rank, where) == (api.ERR_TIMEOUT, 2, 2)
