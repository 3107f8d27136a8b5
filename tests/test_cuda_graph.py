"""The signal-object calls inside CUDA graphs.

A launch's epoch and claim bases are host-side arguments, so a captured launch
replays the same ones.  Capturing opw_signal_reset (a kernel that zeroes the
flags, counters and status word on the stream) followed by the launch at epoch
1 makes every replay start from the state the capture saw: each replay
publishes epoch 1 again.  These tests replay such graphs on new inputs and
compare with the oracle.
"""
import numpy as np
import pytest
import torch

import oracle
from overlap_producer_warps_gb300 import inputs
from tests.helpers import AgProblem, RsProblem, assert_gemm_close, host_bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from overlap_producer_warps_gb300 import api as _api
    _api.lib()
    return _api


def _ag_cfg(R, M_r, K, N):
    return dict(R=R, M_r=M_r, K=K, N=N, dist="normal", scale=0.5)


def _rs_cfg(R, M, K_r, N):
    return dict(R=R, M=M, K_r=K_r, N=N, dist="normal", scale=0.5)


def _load_ag(prob, d):
    """New shard and B contents into the captured buffers (same layout)."""
    prob.heap.copy_(torch.from_numpy(d["heap"]).to("cuda"))
    prob.B.view(torch.int16).copy_(torch.from_numpy(d["B"].view(np.int16)).to("cuda"))
    prob.d = d
    prob.G.fill_(float("nan"))
    prob.C.fill_(float("nan"))


def _check_ag(api, prob, sig, F):
    st = sig.status()
    assert st[0] == api.OK, st
    assert np.array_equal(sig.flags().cpu().numpy(), oracle.expected_flags(F, 1))
    G_ref, C_ref = prob.oracle_full()
    assert np.array_equal(host_bits(prob.G), G_ref), "gathered buffer differs"
    assert_gemm_close(host_bits(prob.C), C_ref)


def _check_rs(api, prob, sig, F):
    st = sig.status()
    assert st[0] == api.OK, st
    assert np.array_equal(sig.flags().cpu().numpy(), oracle.expected_flags(F, 1))
    rows = np.arange(prob.M)
    S = prob.oracle_rows(rows)
    for j in range(prob.R):
        got = prob.out_bits(j)
        assert_gemm_close(got, S[j * prob.Mb:(j + 1) * prob.Mb], what=f"out_{j}")


def test_ag_gemm_reset_and_launch_replayed(api):
    """Reset, then AG-GEMM at epoch 1 (permuted publish order with delays),
    captured once and replayed on three new sets of inputs."""
    cfg = _ag_cfg(4, 256, 512, 1288)
    order = (2, 0, 3, 1)
    prob = AgProblem(inputs.ag_inputs(cfg, seed=71, slot_order=order))
    F = api.ag_num_flags(4, 256, 512)
    sig = api.Signal(F)
    opts = api.make_opts(publish_perm=(3, 1, 0, 2), delay_ns=(0, 5000, 0, 20000))
    prob.run(api, sig, sig.next_epoch(), opts)   # outside any capture: first-call set-up
    _check_ag(api, prob, sig, F)
    graph, side = torch.cuda.CUDAGraph(), torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.graph(graph, stream=side):
        sig.reset(stream=side)
        prob.run(api, sig, 1, opts, stream=side)
    for seed in (72, 73, 74):
        _load_ag(prob, inputs.ag_inputs(cfg, seed=seed, slot_order=order))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        _check_ag(api, prob, sig, F)
    sig.close()


def test_tp_layer_step_as_one_graph(api):
    """One graph holding a whole tensor-parallel step: AG-GEMM, then GEMM-RS,
    each behind the reset of its own signal object; two replays on new
    inputs, both outputs against the oracle."""
    ag = AgProblem(inputs.ag_inputs(_ag_cfg(4, 256, 384, 776), seed=75))
    rs = RsProblem(inputs.rs_inputs(_rs_cfg(4, 1024, 200, 328), seed=76))
    F_ag, F_rs = api.ag_num_flags(4, 256, 384), api.rs_num_flags(4, 1024, 328)
    sig_ag, sig_rs = api.Signal(F_ag), api.Signal(F_rs)
    ag.run(api, sig_ag, sig_ag.next_epoch())
    rs.run(api, sig_rs, sig_rs.next_epoch())
    torch.cuda.synchronize()
    graph, side = torch.cuda.CUDAGraph(), torch.cuda.Stream()
    with torch.cuda.graph(graph, stream=side):
        sig_ag.reset(stream=side)
        ag.run(api, sig_ag, 1, stream=side)
        sig_rs.reset(stream=side)
        rs.run(api, sig_rs, 1, stream=side)
    for seed in (77, 78):
        _load_ag(ag, inputs.ag_inputs(_ag_cfg(4, 256, 384, 776), seed=seed))
        d = inputs.rs_inputs(_rs_cfg(4, 1024, 200, 328), seed=seed + 10)
        rs.heap.copy_(torch.from_numpy(d["heap"]).to("cuda"))
        rs.d = d
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        _check_ag(api, ag, sig_ag, F_ag)
        _check_rs(api, rs, sig_rs, F_rs)
    sig_ag.close()
    sig_rs.close()
