"""Hundreds of launches across modes reproduce the same bits: a race check.

Every element of AG-GEMM's C sums the same products in the same k order
whatever the schedule, pair-tile width, grid size, publish order, signal mode
or sync mode, and GEMM-RS adds the ranks' partials in rank order whatever the
grid.  So a race anywhere in the protocol (a tile loaded before its copy
landed, an accumulator reused before it was read out, a staging buffer
overwritten before its store read it, a flag published before its stores
completed) would show up as bits that differ from one launch to the next.

These tests launch back to back, cycling through the modes, with G, C and the
GEMM-RS output blocks set to a NaN pattern before every launch (so a region a
launch fails to write cannot pass by keeping the previous launch's bits).
Every launch's outputs are compared on the device with the first launch's,
every flag with its launch's epoch, and the first launch with the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from overlap_producer_warps_gb300 import inputs
from tests.helpers import AgProblem, RsProblem, assert_gemm_close, host_bits, quarter_rows

pytestmark = pytest.mark.gpu

NAN_BITS = -1  # int16 0xffff: a bf16 NaN


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from overlap_producer_warps_gb300 import api as _api
    _api.lib()
    return _api


def test_ag_gemm_modes_repeat_bit_for_bit(api):
    R, M_r, K, N = 8, 512, 1024, 1288   # 16 pair rows; 6 (or 3 wide) column tiles, ragged
    d = inputs.ag_inputs(dict(R=R, M_r=M_r, K=K, N=N, dist="normal", scale=0.5), seed=91)
    prob = AgProblem(d)
    F = api.ag_num_flags(R, M_r, K)
    sig = api.Signal(F)
    sig_add = api.Signal(api.ag_num_row_counters(R, M_r, K))
    T_k = K // api.ag_flag_tile(M_r, K)
    perm = (5, 2, 7, 0, 3, 6, 1, 4)
    modes = [
        ("default", dict()),
        ("static swizzle", dict(schedule=api.SCHED_SWIZZLE)),
        ("256x512 tiles", dict(tile_n=512)),
        ("8 pairs, 256x256", dict(num_ctas=16, tile_n=256)),
        ("3 pairs, 256x512", dict(num_ctas=6, tile_n=512)),
        ("permuted publish with delays", dict(publish_perm=perm,
                                              delay_ns=(0, 3000, 0, 1500, 0, 0, 4000, 500))),
        ("checked publish", dict(sync_mode=api.SYNC_CHECKED)),
        ("no local shard", dict(local_rank=-1)),
        ("producer then consumer", None),
        ("row-ADD signals", dict(signal_mode=api.SIGNAL_ROW_ADD)),
    ]
    opts = {name: (api.make_opts(**kw) if kw is not None else None) for name, kw in modes}
    prod, cons = api.make_opts(role=api.ROLE_PRODUCER), api.make_opts(role=api.ROLE_CONSUMER)

    G0 = C0 = None
    bad = torch.zeros((), dtype=torch.int64, device="cuda")
    flag_bad = torch.zeros((), dtype=torch.int64, device="cuda")
    launches = 0
    for rep in range(24):
        for name, _ in modes:
            prob.G.view(torch.int16).fill_(NAN_BITS)
            prob.C.view(torch.int16).fill_(NAN_BITS)
            if name == "row-ADD signals":
                e = sig_add.next_epoch()
                prob.run(api, sig_add, e, opts[name])
                flag_bad += (sig_add.flags() != e * T_k).sum()
            elif name == "producer then consumer":
                e = sig.next_epoch()
                prob.run(api, sig, e, prod)
                prob.run(api, sig, e, cons)
                flag_bad += (sig.flags() != e).sum()
            else:
                e = sig.next_epoch()
                prob.run(api, sig, e, opts[name])
                flag_bad += (sig.flags() != e).sum()
            launches += 1
            if G0 is None:
                torch.cuda.synchronize()
                assert sig.status()[0] == api.OK
                G0, C0 = prob.G.clone(), prob.C.clone()
                G_ref = oracle.allgather(d["heap"], d["rank_off"], R, d["a_off"], M_r, K)
                assert np.array_equal(host_bits(G0), G_ref)
                rows = quarter_rows(prob.M, seed=92)
                assert_gemm_close(host_bits(C0)[rows], prob.oracle_rows(rows))
                continue
            bad += (prob.G.view(torch.int16) != G0.view(torch.int16)).sum()
            bad += (prob.C.view(torch.int16) != C0.view(torch.int16)).sum()
    torch.cuda.synchronize()
    assert sig.status()[0] == api.OK and sig_add.status()[0] == api.OK
    assert launches == 24 * len(modes)
    assert int(flag_bad) == 0, f"{int(flag_bad)} flags not at their launch's epoch"
    assert int(bad) == 0, f"{int(bad)} elements of G or C differ from the first launch"
    sig.close()
    sig_add.close()


def test_gemm_rs_grids_repeat_bit_for_bit(api):
    R, M, K_r, N = 8, 2048, 200, 1288   # 8 pair rows x 6 column tiles, ragged K and N
    d = inputs.rs_inputs(dict(R=R, M=M, K_r=K_r, N=N, dist="normal", scale=0.5), seed=93)
    prob = RsProblem(d)
    F = api.rs_num_flags(R, M, N)
    sig = api.Signal(F)
    recv = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    out_slices = [prob.heap[int(prob.rank_off[j]) + d["out_off"]:
                            int(prob.rank_off[j]) + d["out_off"] + prob.Mb * N * 2]
                  for j in range(R)]
    grids = [dict(), dict(num_ctas=16), dict(num_ctas=26), dict(sync_mode=api.SYNC_CHECKED)]
    opts = [api.make_opts(**kw) for kw in grids]

    ref = None
    bad = torch.zeros((), dtype=torch.int64, device="cuda")
    flag_bad = torch.zeros((), dtype=torch.int64, device="cuda")
    for rep in range(30):
        for i, o in enumerate(opts):
            for s in out_slices:
                s.fill_(255)
            recv.view(torch.int16).fill_(NAN_BITS)
            e = sig.next_epoch()
            consume = (rep + i) % 2 == 1   # every other launch also runs the receiving side
            if consume:
                api.gemm_rs_consume(prob.heap, prob.rank_off, d["a_off"], d["b_off"], d["out_off"],
                                    M, N, K_r, recv, sig, e, o)
            else:
                prob.run(api, sig, e, o)
            flag_bad += (sig.flags() != e).sum()
            outs = torch.cat([s.view(torch.int16) for s in out_slices])
            if ref is None:
                torch.cuda.synchronize()
                assert sig.status()[0] == api.OK
                ref = outs.clone()
                rows = quarter_rows(M, seed=94)
                S = prob.oracle_rows(rows)
                got = np.concatenate([prob.out_bits(j) for j in range(R)])
                assert_gemm_close(got[rows], S)
                continue
            bad += (outs != ref).sum()
            if consume:
                bad += (recv.view(torch.int16).reshape(-1) != ref).sum()
    torch.cuda.synchronize()
    assert sig.status()[0] == api.OK
    assert int(flag_bad) == 0, f"{int(flag_bad)} flags not at their launch's epoch"
    assert int(bad) == 0, f"{int(bad)} output elements differ from the first launch"
    sig.close()


@pytest.mark.parametrize("name,launches", [("ag_tp", 40), ("ag_skew", 12), ("rs_tp", 30)])
def test_full_size_layers_repeat_bit_for_bit(api, name, launches):
    """The benchmark's layers at full size, in its launch configuration (the
    skew layer with its permuted publish order and delays): every launch
    reproduces the first one's bits.  Parity of that first result with the
    oracle at these sizes is the full-size parity tests' part."""
    cfg = inputs.CONFIGS[name]
    if name.startswith("rs"):
        d = inputs.rs_inputs(cfg, seed=0)
        prob = RsProblem(d)
        sig = api.Signal(api.rs_num_flags(prob.R, prob.M, prob.N))
        outs = [prob.heap[int(prob.rank_off[j]) + d["out_off"]:
                          int(prob.rank_off[j]) + d["out_off"] + prob.Mb * prob.N * 2]
                for j in range(prob.R)]
        opts = None
    else:
        d = inputs.ag_inputs(cfg, seed=0)
        prob = AgProblem(d)
        sig = api.Signal(api.ag_num_flags(prob.R, prob.M_r, prob.K))
        outs = [prob.G.view(torch.uint8).reshape(-1), prob.C.view(torch.uint8).reshape(-1)]
        opts = None
        if cfg.get("skew"):
            perm, delay = inputs.skew_schedule(0, prob.R)
            opts = api.make_opts(publish_perm=perm, delay_ns=delay)
    first = None
    bad = torch.zeros((), dtype=torch.int64, device="cuda")
    flag_bad = torch.zeros((), dtype=torch.int64, device="cuda")
    for i in range(launches):
        for t in outs:
            t.fill_(255)
        e = sig.next_epoch()
        prob.run(api, sig, e, opts)
        flag_bad += (sig.flags() != e).sum()
        if first is None:
            first = [t.clone() for t in outs]
            continue
        for t, f in zip(outs, first):
            bad += (t != f).sum()
    torch.cuda.synchronize()
    assert sig.status()[0] == api.OK
    assert int(flag_bad) == 0, f"{int(flag_bad)} flags not at their launch's epoch"
    assert int(bad) == 0, f"{int(bad)} output bytes differ from the first launch"
    # the first launch wrote every output byte (none kept the 0xff pattern of a
    # bf16 NaN: the inputs are finite)
    for f in first:
        assert not bool((f.view(torch.int16) == -1).any())
    sig.close()
