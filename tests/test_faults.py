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


def _plant(sig, slot, value):
    """Write `value` into one flag slot behind the kernels' back."""
    flags = sig.flags()
    flags[slot] = value
    torch.cuda.synchronize()


@pytest.mark.parametrize("mode", ["set", "row_add"])
def test_checked_publish_finds_the_previous_epoch(api, mode):
    """OPW_SYNC_CHECKED publishes by exchange (SET) or fetch-add (ROW_ADD) and
    requires the previous epoch's value; a planted value is reported as
    FLAG_PROTOCOL with the producing rank and the slot, and the signal object
    recovers after a reset."""
    prob = _problem(seed=41)
    row_add = mode == "row_add"
    F = api.ag_num_row_counters(4, 128, 256) if row_add else api.ag_num_flags(4, 128, 256)
    sm = api.SIGNAL_ROW_ADD if row_add else api.SIGNAL_TILE_SET
    sig = api.Signal(F)

    def opts():
        return api.make_opts(sync_mode=api.SYNC_CHECKED, signal_mode=sm, timeout_ns=TIMEOUT_NS)

    for _ in range(3):
        prob.run(api, sig, sig.next_epoch(), opts())
        assert sig.status()[0] == api.OK
    _, C_ref = prob.oracle_full()
    assert_gemm_close(host_bits(prob.C), C_ref)
    e = sig.next_epoch()
    # flag tiles are 128x128 here: 4 ranks x 1 row x 2 k-columns (T_k = 2)
    if row_add:
        slot, rank = 2, 2
        _plant(sig, slot, e * 2 + 3)      # outside this epoch's window [(e-1)*2, e*2)
    else:
        slot, rank = 5, 2
        _plant(sig, slot, e + 3)          # not e - 1
    prob.run(api, sig, e, opts())
    assert sig.status() == (api.ERR_FLAG_PROTOCOL, rank, slot)
    sig.reset()
    prob.run(api, sig, sig.next_epoch(), opts())
    assert sig.status()[0] == api.OK


def test_gemm_rs_checked_publish_finds_the_previous_epoch(api):
    from tests.helpers import RsProblem
    d = inputs.rs_inputs(dict(R=2, M=256, K_r=128, N=256, dist="normal", scale=0.5), seed=50)
    prob = RsProblem(d)
    F = api.rs_num_flags(2, 256, 256)          # 2 ranks x 1 x 2 output tiles
    sig = api.Signal(F)
    opts = api.make_opts(sync_mode=api.SYNC_CHECKED, timeout_ns=TIMEOUT_NS)
    for _ in range(3):
        prob.run(api, sig, sig.next_epoch(), opts)
        assert sig.status()[0] == api.OK
    e = sig.next_epoch()
    _plant(sig, 3, e + 3)
    prob.run(api, sig, e, opts)
    assert sig.status() == (api.ERR_FLAG_PROTOCOL, 1, 3)  # slot 3 belongs to rank 1
    sig.reset()
    prob.run(api, sig, sig.next_epoch(), opts)
    assert sig.status()[0] == api.OK


def test_local_rank_tiles_are_not_waited_for(api):
    """The consumer reads its own rank's shard in place: a flag of that rank
    that is never published delays nobody (the launch completes and C is
    right), while the same drop with local_rank=-1 times out."""
    prob = _problem(seed=42)
    F = api.ag_num_flags(4, 128, 256)
    slot = 1                                  # rank 0's second flag tile
    sig = api.Signal(F)
    prob.run(api, sig, sig.next_epoch(), api.make_opts(timeout_ns=TIMEOUT_NS, local_rank=0,
                                                       fault_kind=api.FAULT_DROP_TILE,
                                                       fault_arg=slot))
    assert sig.status()[0] == api.OK
    flags = sig.flags().cpu().numpy()
    assert flags[slot] == 0 and np.all(np.delete(flags, slot) == 1)
    G_ref, C_ref = prob.oracle_full()
    assert np.array_equal(host_bits(prob.G), G_ref)
    assert_gemm_close(host_bits(prob.C), C_ref)
    sig2 = api.Signal(F)
    prob.run(api, sig2, sig2.next_epoch(), api.make_opts(timeout_ns=TIMEOUT_NS, local_rank=-1,
                                                         fault_kind=api.FAULT_DROP_TILE,
                                                         fault_arg=slot))
    assert sig2.status() == (api.ERR_TIMEOUT, 0, slot)
