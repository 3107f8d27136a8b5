"""GEMM -> ReduceScatter on the GPU against the CPU oracle, through the C ABI.

Each rank j's output block must match rows [j*M/R, (j+1)*M/R) of the oracle's
fp64 sum of partials (rounded to bf16) within rel-Frobenius 1e-3 and
per-element 1e-2*max|ref|; every flag must equal the epoch; repeated runs
must be bit-identical (fixed-order fp32 reduction).
"""
import numpy as np
import pytest
import torch

import oracle
from overlap_producer_warps_gb300 import inputs
from tests.helpers import RsProblem, assert_gemm_close, quarter_rows, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from overlap_producer_warps_gb300 import api as _api
    _api.lib()
    return _api


def _cfg(R, M, K_r, N, scale=0.5):
    return dict(R=R, M=M, K_r=K_r, N=N, dist="normal", scale=scale)


def _check_all(api, prob, rows=None):
    R, Mb = prob.R, prob.Mb
    if rows is None:
        rows = np.arange(prob.M)
    S = prob.oracle_rows(rows)
    for j in range(R):
        sel = (rows >= j * Mb) & (rows < (j + 1) * Mb)
        if not np.any(sel):
            continue
        got = prob.out_bits(j)[rows[sel] - j * Mb]
        assert_gemm_close(got, S[sel], what=f"out_{j}")


@pytest.mark.parametrize("R,M,K_r,N,order", [
    (2, 256, 128, 256, None),
    (3, 384, 200, 328, (2, 0, 1)),     # ragged K_r and N, permuted rank table
    (8, 1024, 64, 512, None),
    (1, 256, 320, 264, None),          # single rank: plain GEMM
    (4, 1024, 448, 1024, (3, 1, 2, 0)),
    (2, 256, 8, 256, None),            # K_r = 8: one k-stage, almost all of it zero fill
    (3, 384, 136, 200, None),          # a second k-stage holding 8 of K
])
def test_shapes(api, R, M, K_r, N, order):
    d = inputs.rs_inputs(_cfg(R, M, K_r, N), seed=R * 5 + K_r, slot_order=order)
    prob = RsProblem(d)
    F = api.rs_num_flags(R, M, N)
    sig = api.Signal(F)
    e = sig.next_epoch()
    prob.run(api, sig, e)
    st = sig.status()
    assert st[0] == api.OK, st
    assert np.array_equal(sig.flags().cpu().numpy(), oracle.expected_flags(F, e))
    _check_all(api, prob)


def test_legs_alone(api):
    """The GEMM leg alone (producer role) stores and publishes nothing and
    leaves the epoch unused; the scatter leg alone (consumer role) stores
    bf16 zeros into every rank's block and publishes every flag; a fused
    launch after both gives the oracle's result."""
    R, M, K_r, N = 3, 768, 192, 328   # ragged last column tile
    d = inputs.rs_inputs(_cfg(R, M, K_r, N), seed=53)
    prob = RsProblem(d)
    F = api.rs_num_flags(R, M, N)
    sig = api.Signal(F)
    out_bytes = prob.Mb * N * 2
    regions = [prob.heap[int(prob.rank_off[j]) + d["out_off"]:
                         int(prob.rank_off[j]) + d["out_off"] + out_bytes] for j in range(R)]
    for reg in regions:
        reg.fill_(0x7F)
    e = sig.next_epoch()
    prob.run(api, sig, e, api.make_opts(role=api.ROLE_PRODUCER))
    torch.cuda.synchronize()
    assert sig.status()[0] == api.OK
    assert sig.next_epoch() == e
    assert not sig.flags().any()
    for reg in regions:
        assert bool((reg == 0x7F).all())

    prob.run(api, sig, e, api.make_opts(role=api.ROLE_CONSUMER))
    torch.cuda.synchronize()
    assert sig.status()[0] == api.OK
    assert np.array_equal(sig.flags().cpu().numpy(), oracle.expected_flags(F, e))
    for reg in regions:
        assert not bool(reg.any())

    e2 = sig.next_epoch()
    assert e2 == e + 1
    prob.run(api, sig, e2, api.make_opts(sync_mode=api.SYNC_CHECKED))
    assert sig.status()[0] == api.OK
    assert np.array_equal(sig.flags().cpu().numpy(), oracle.expected_flags(F, e2))
    _check_all(api, prob)


@pytest.mark.parametrize("num_ctas", [1, 2, 5, 6])
def test_pair_counts(api, num_ctas):
    """CTAs run in pairs: 1 and 2 CTAs give one pair, 5 gives two.  With 15
    pair tiles (M = 4 x 256 + 128, so the last row of pair tiles is ragged)
    every pair does several tiles and one CTA of each last-row pair holds
    rows past M."""
    R, M, K_r, N = 3, 1152, 192, 768
    d = inputs.rs_inputs(_cfg(R, M, K_r, N), seed=41 + num_ctas)
    prob = RsProblem(d)
    F = api.rs_num_flags(R, M, N)
    sig = api.Signal(F)
    e = sig.next_epoch()
    prob.run(api, sig, e, api.make_opts(num_ctas=num_ctas))
    st = sig.status()
    assert st[0] == api.OK, st
    assert np.array_equal(sig.flags().cpu().numpy(), oracle.expected_flags(F, e))
    _check_all(api, prob)


def test_output_independent_of_pair_count(api):
    """Each pair reduces its tiles' partials in rank order in fp32, whatever
    the grid: 64 pair tiles on 8, 12, 13 and 21 pairs (0, 4, 12 and 1 tiles in
    the last partial wave) must give bit-identical outputs."""
    R, M, K_r, N = 4, 4096, 192, 1024
    d = inputs.rs_inputs(_cfg(R, M, K_r, N), seed=45)
    prob = RsProblem(d)
    F = api.rs_num_flags(R, M, N)
    outs = []
    for num_ctas in (16, 24, 26, 42):
        sig = api.Signal(F)
        for _ in range(2):
            e = sig.next_epoch()
            prob.run(api, sig, e, api.make_opts(num_ctas=num_ctas))
            st = sig.status()
            assert st[0] == api.OK, (num_ctas, st)
            assert np.all(sig.flags().cpu().numpy() == e)
        outs.append(np.concatenate([prob.out_bits(j) for j in range(R)]))
        sig.close()
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    rows = sample_rows(prob.M, 128, 1, seed=3)
    _check_all(api, prob, rows)


def test_deterministic_and_epochs(api):
    R, M, K_r, N = 4, 512, 256, 512
    d = inputs.rs_inputs(_cfg(R, M, K_r, N), seed=31)
    prob = RsProblem(d)
    F = api.rs_num_flags(R, M, N)
    sig = api.Signal(F)
    outs = []
    for _ in range(5):
        e = sig.next_epoch()
        prob.run(api, sig, e)
        assert sig.status()[0] == api.OK
        assert np.all(sig.flags().cpu().numpy() == e)
        outs.append(np.concatenate([prob.out_bits(j) for j in range(R)]))
    for o in outs[1:]:
        assert np.array_equal(o, outs[0])
    _check_all(api, prob)


def test_only_output_regions_are_written(api):
    R, M, K_r, N = 2, 256, 128, 256
    d = inputs.rs_inputs(_cfg(R, M, K_r, N), seed=32)
    prob = RsProblem(d)
    before = prob.heap.cpu().numpy().copy()
    sig = api.Signal(api.rs_num_flags(R, M, N))
    prob.run(api, sig, sig.next_epoch())
    assert sig.status()[0] == api.OK
    after = prob.heap.cpu().numpy()
    mask = np.ones(before.size, dtype=bool)
    for j in range(R):
        o = int(prob.rank_off[j]) + d["out_off"]
        mask[o:o + prob.Mb * N * 2] = False
    assert np.array_equal(before[mask], after[mask])


def test_full_size_tp_sampled(api):
    """GEMM-RS TP layer at full size (R=8, A_r 8192x1792, B_r 1792x4096), sampled rows."""
    cfg = inputs.CONFIGS["rs_tp"]
    d = inputs.rs_inputs(cfg, seed=0)
    prob = RsProblem(d)
    sig = api.Signal(api.rs_num_flags(prob.R, prob.M, prob.N))
    for _ in range(2):
        prob.run(api, sig, sig.next_epoch())
        assert sig.status()[0] == api.OK
    assert np.all(sig.flags().cpu().numpy() == 2)
    rows = sample_rows(prob.M, 128, 1, seed=2)
    _check_all(api, prob, rows)


# ---------------------------------------------------------------- receiving side

def _out_regions(prob):
    d, n = prob.d, prob.Mb * prob.N * 2
    return [prob.heap[int(prob.rank_off[j]) + d["out_off"]:int(prob.rank_off[j]) + d["out_off"] + n]
            for j in range(prob.R)]


def _consume(api, prob, sig, epoch, opts=None):
    """One GEMM-RS launch with the receiving side, into a NaN-filled recv
    buffer, with every rank's output block first filled with NaN bits too (a
    copy taken before a tile's store landed would show)."""
    d = prob.d
    for reg in _out_regions(prob):
        reg.fill_(0xFF)
    recv = torch.full((prob.M, prob.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    api.gemm_rs_consume(prob.heap, prob.rank_off, d["a_off"], d["b_off"], d["out_off"], prob.M,
                        prob.N, prob.K_r, recv, sig, epoch, opts)
    return recv


@pytest.mark.parametrize("R,M,K_r,N,num_ctas", [
    (3, 1152, 192, 328, 0),   # ragged last pair tile (the odd CTA has no rows) and ragged N
    (4, 1024, 448, 1024, 2),  # one pair: its odd CTA receives every tile the even one stores
    (2, 256, 128, 200, 0),
])
def test_receiving_side_acquires_every_tile_before_copying(api, R, M, K_r, N, num_ctas):
    d = inputs.rs_inputs(_cfg(R, M, K_r, N), seed=80 + R)
    prob = RsProblem(d)
    F = api.rs_num_flags(R, M, N)
    sig = api.Signal(F)
    trace = torch.full((2 * F,), -1, dtype=torch.int64, device="cuda")
    for _ in range(2):
        trace.fill_(-1)
        e = sig.next_epoch()
        recv = _consume(api, prob, sig, e, api.make_opts(trace=trace, num_ctas=num_ctas))
        st = sig.status()
        assert st[0] == api.OK, st
        assert np.array_equal(sig.flags().cpu().numpy(), oracle.expected_flags(F, e))
        # the receiver's copy is every rank's block, bit for bit
        got = recv.view(torch.int16).cpu().numpy().view(np.uint16)
        want = np.concatenate([prob.out_bits(j) for j in range(R)])
        assert np.array_equal(got, want)
        # every tile published, every tile acquired, never before its publish
        t = trace.cpu().numpy().view(np.uint64)
        pub, got_at = t[:F], t[F:2 * F]
        none = np.uint64(2 ** 64 - 1)
        assert np.all(pub != none) and np.all(got_at != none)
        assert np.all(pub <= got_at)
    _check_all(api, prob)


def test_receiving_side_with_checked_publish(api):
    R, M, K_r, N = 4, 1024, 256, 512
    d = inputs.rs_inputs(_cfg(R, M, K_r, N), seed=85)
    prob = RsProblem(d)
    F = api.rs_num_flags(R, M, N)
    sig = api.Signal(F)
    for _ in range(3):
        e = sig.next_epoch()
        recv = _consume(api, prob, sig, e, api.make_opts(sync_mode=api.SYNC_CHECKED))
        assert sig.status()[0] == api.OK
        got = recv.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, np.concatenate([prob.out_bits(j) for j in range(R)]))
    _check_all(api, prob)


def test_receiving_side_times_out_on_a_missing_flag_and_recovers(api):
    """A tile whose flag is never published: the receiving wait runs out and
    latches TIMEOUT with that tile's rank and slot; after a reset the next
    launch is correct."""
    R, M, K_r, N = 2, 512, 128, 512
    d = inputs.rs_inputs(_cfg(R, M, K_r, N), seed=86)
    prob = RsProblem(d)
    F = api.rs_num_flags(R, M, N)
    sig = api.Signal(F)
    slot = 9
    _consume(api, prob, sig, sig.next_epoch(),
             api.make_opts(timeout_ns=50_000_000, fault_kind=api.FAULT_DROP_TILE, fault_arg=slot))
    status, rank, where = sig.status()
    assert status == api.ERR_TIMEOUT
    assert (rank, where) == (slot // (F // R), slot)
    sig.reset()
    recv = _consume(api, prob, sig, sig.next_epoch())
    assert sig.status()[0] == api.OK
    got = recv.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, np.concatenate([prob.out_bits(j) for j in range(R)]))
    _check_all(api, prob)


def test_full_size_tp_with_receiving_side(api):
    """GEMM-RS TP at full size with the receiving side: recv bit-equal to the
    blocks, the blocks within the tolerance on sampled rows."""
    cfg = inputs.CONFIGS["rs_tp"]
    prob = RsProblem(inputs.rs_inputs(cfg, seed=0))
    F = api.rs_num_flags(prob.R, prob.M, prob.N)
    sig = api.Signal(F)
    trace = torch.full((2 * F,), -1, dtype=torch.int64, device="cuda")
    recv = _consume(api, prob, sig, sig.next_epoch(), api.make_opts(trace=trace))
    assert sig.status()[0] == api.OK
    got = recv.view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, np.concatenate([prob.out_bits(j) for j in range(prob.R)]))
    t = trace.cpu().numpy().view(np.uint64)
    assert np.all(t[:F] <= t[F:2 * F])
    _check_all(api, prob, quarter_rows(prob.M, seed=4))
