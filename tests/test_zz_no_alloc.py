"""opw_ag_gemm_noalloc: the AllGather -> GEMM call for callers that cannot
allocate device memory (a framework that owns all device memory through its
own pool, or a serving loop that cannot afford cudaMalloc's implicit device
synchronisation).  It keeps its flags and counters in a fixed array inside
the library, so it must give the oracle's results, and the same results as
opw_ag_gemm, call after call, even though every call reuses that array: after
a call that failed on the device, with either signal mode, in the checked
publish mode, and at exactly the largest flag count the array holds.  And it
must allocate nothing.

This file is named so that pytest collects it last.
"""
import numpy as np
import pytest
import torch

import oracle
from overlap_producer_warps_gb300 import inputs
from tests.helpers import AgProblem, assert_gemm_close, host_bits


@pytest.fixture(scope="module")
def api():
    from overlap_producer_warps_gb300 import api as _api
    from overlap_producer_warps_gb300 import build as _b
    _b.build()
    _api.lib()
    return _api


class _Ptr:
    def __init__(self, v):
        self._v = v

    def data_ptr(self):
        return self._v


class _NoStream:
    cuda_stream = 0


def test_rejects_sizes_beyond_the_fixed_scratch_on_the_host(api):
    # Checked before any CUDA call, so stand-in addresses are enough.
    args = dict(heap=_Ptr(0x100000), B=_Ptr(0x200000), G=_Ptr(0x300000), C=_Ptr(0x400000),
                status=_Ptr(0x500000))

    def call(R, M_r, K, N=256, opts=None, status=None):
        return api.ag_gemm_noalloc_status(args["heap"], [r * (1 << 20) for r in range(R)], 0, M_r,
                                          N, K, args["B"], args["G"], args["C"],
                                          status or args["status"], opts, stream=_NoStream())

    assert api.NOALLOC_MAX_FLAGS == 65536
    assert api.ag_num_flags(8, 8192, 32768) > api.NOALLOC_MAX_FLAGS
    assert call(8, 8192, 32768) == api.ERR_UNSUPPORTED_SHAPE
    # twice the maximum, with either signal mode
    assert api.ag_num_flags(8, 2 * 524288, 64) == api.NOALLOC_MAX_FLAGS * 2
    assert call(8, 2 * 524288, 64) == api.ERR_UNSUPPORTED_SHAPE
    assert call(8, 2 * 524288, 64,
                opts=api.make_opts(signal_mode=api.SIGNAL_ROW_ADD)) == api.ERR_UNSUPPORTED_SHAPE
    assert call(2, 128, 256, opts=api.make_opts(role=api.ROLE_CONSUMER)) == api.ERR_INVALID_ARG
    assert call(2, 128, 256, status=_Ptr(0)) == api.ERR_INVALID_ARG
    assert call(2, 128, 256, status=_Ptr(0x500004)) == api.ERR_MISALIGNED


def test_binding_refuses_a_status_tensor_of_the_wrong_kind(api):
    # the library writes 4 int32 words from the current device
    heap = B = G = C = _Ptr(0x100000)
    for bad in (torch.zeros(4, dtype=torch.int32),          # host memory
                torch.zeros(4, dtype=torch.int64),
                torch.zeros(3, dtype=torch.int32),
                torch.zeros(8, dtype=torch.int32)[::2]):    # not contiguous
        assert api.ag_gemm_noalloc_status(heap, [0, 1 << 20], 0, 128, 256, 256, B, G, C, bad,
                                          stream=_NoStream()) == api.ERR_INVALID_ARG


def _gpu():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")


def _reference(api, prob, opts=None):
    """The existing entry point (with its own signal object) on the same inputs."""
    n = (api.ag_num_row_counters if opts is not None and opts.signal_mode == api.SIGNAL_ROW_ADD
         else api.ag_num_flags)(prob.R, prob.M_r, prob.K)
    sig = api.Signal(n)
    G0, C0 = prob.G.clone(), prob.C.clone()
    prob.run(api, sig, sig.next_epoch(), opts)
    st = sig.status()
    assert st[0] == api.OK, st
    out = host_bits(prob.G), host_bits(prob.C)
    prob.G.copy_(G0)
    prob.C.copy_(C0)
    sig.close()
    return out


def _noalloc(api, prob, status, opts=None):
    """One no-allocation call into fresh NaN-filled outputs (a stale or
    skipped tile shows); returns the device status word and G, C."""
    G = torch.full_like(prob.G, float("nan"))
    C = torch.full_like(prob.C, float("nan"))
    rc = api.ag_gemm_noalloc_status(prob.heap, prob.rank_off, prob.a_off, prob.M_r, prob.N,
                                    prob.K, prob.B, G, C, status, opts)
    assert rc == api.OK, api.status_str(rc)
    torch.cuda.synchronize()
    return status.cpu().tolist(), G, C


def _check_against_oracle(prob, G, C, what):
    G_ref, C_ref = prob.oracle_full()
    assert np.array_equal(host_bits(G), G_ref), f"{what}: gathered buffer differs from the oracle"
    assert_gemm_close(host_bits(C), C_ref, what=f"{what}: C")


@pytest.mark.gpu
def test_matches_oracle_and_ag_gemm_on_two_calls_in_a_row(api):
    _gpu()
    cfg = dict(R=4, M_r=256, K=512, N=776, dist="normal", scale=0.5)
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    for call, seed in enumerate((51, 52)):   # different inputs each call
        prob = AgProblem(inputs.ag_inputs(cfg, seed=seed, slot_order=(2, 0, 3, 1)))
        G_ref, C_ref = _reference(api, prob)
        st, G, C = _noalloc(api, prob, status)
        assert st[0] == api.OK, (call, st)
        _check_against_oracle(prob, G, C, f"call {call}")
        # and the existing entry point's results: G bit for bit, C within the tolerance
        assert np.array_equal(host_bits(G), G_ref), f"call {call}: G differs from opw_ag_gemm"
        assert_gemm_close(host_bits(C), oracle.bf16_to_f64(C_ref), what=f"call {call}: C")


@pytest.mark.gpu
@pytest.mark.parametrize("tile_n", [256, 512])
def test_pair_tile_widths_match_oracle(api, tile_n):
    """Both pair-tile widths through the no-allocation call, on a ragged N
    (1288 = 2 x 512 + 264) with several wide tiles per pair, against the
    oracle; the width is the one asked for."""
    _gpu()
    prob = AgProblem(inputs.ag_inputs(dict(R=4, M_r=384, K=448, N=1288, dist="normal", scale=0.5),
                                      seed=59, slot_order=(3, 1, 0, 2)))
    opts = api.make_opts(tile_n=tile_n, num_ctas=6)   # 3 pairs: several tiles each
    assert api.ag_tile_n(4, 384, 1288, opts) == tile_n
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    st, G, C = _noalloc(api, prob, status, opts)
    assert st[0] == api.OK, (tile_n, st)
    _check_against_oracle(prob, G, C, f"tile_n {tile_n}")


@pytest.mark.gpu
def test_captured_in_a_cuda_graph_and_replayed(api):
    """The call allocates nothing and launches the same kernels with the same
    arguments every time (it clears its own flags and publishes epoch 1), so a
    CUDA graph can capture it once and replay it.  Three replays, each on new
    shard and B contents copied into the captured buffers, match the oracle."""
    _gpu()
    cfg = dict(R=4, M_r=256, K=512, N=1288, dist="normal", scale=0.5)
    prob = AgProblem(inputs.ag_inputs(cfg, seed=61, slot_order=(1, 3, 0, 2)))
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    G = torch.full_like(prob.G, float("nan"))
    C = torch.full_like(prob.C, float("nan"))
    args = (prob.heap, prob.rank_off, prob.a_off, prob.M_r, prob.N, prob.K, prob.B, G, C, status)
    # the first call on the device, outside any capture, looks up the scratch array
    assert api.ag_gemm_noalloc_status(*args) == api.OK
    torch.cuda.synchronize()
    graph, side = torch.cuda.CUDAGraph(), torch.cuda.Stream()
    with torch.cuda.graph(graph, stream=side):
        rc = api.ag_gemm_noalloc_status(*args, stream=side)
    assert rc == api.OK, api.status_str(rc)
    for seed in (62, 63, 64):
        d = inputs.ag_inputs(cfg, seed=seed, slot_order=(1, 3, 0, 2))
        prob.heap.copy_(torch.from_numpy(d["heap"]).to("cuda"))
        prob.B.view(torch.int16).copy_(torch.from_numpy(d["B"].view(np.int16)).to("cuda"))
        G.fill_(float("nan"))
        status.fill_(-1)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert status.cpu().tolist()[0] == api.OK, seed
        ref = AgProblem.__new__(AgProblem)
        ref.d, ref.R, ref.M_r, ref.K, ref.N = d, prob.R, prob.M_r, prob.K, prob.N
        ref.rank_off, ref.a_off = d["rank_off"], d["a_off"]
        _check_against_oracle(ref, G, C, f"replay with seed {seed}")


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["row_add", "checked", "checked_row_add"])
def test_signal_modes_and_checked_publish(api, mode):
    """Batched row counters and the checked publish both need the shared
    array cleared by the call: the counters start from 0 and the checked
    exchange must find epoch - 1 = 0 in every slot."""
    _gpu()
    kw = {}
    if "row_add" in mode:
        kw["signal_mode"] = api.SIGNAL_ROW_ADD
    if "checked" in mode:
        kw["sync_mode"] = api.SYNC_CHECKED
    prob = AgProblem(inputs.ag_inputs(dict(R=3, M_r=192, K=320, N=264, dist="normal", scale=0.5),
                                      seed=57))
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    for call in range(2):
        st, G, C = _noalloc(api, prob, status, api.make_opts(**kw))
        assert st[0] == api.OK, (mode, call, st)
        _check_against_oracle(prob, G, C, f"{mode} call {call}")


@pytest.mark.gpu
def test_a_failed_call_leaves_the_next_one_clean(api):
    """A call whose tile is never published times out on the device; the
    next call clears the shared array and the status word and is correct."""
    _gpu()
    prob = AgProblem(inputs.ag_inputs(dict(R=4, M_r=128, K=256, N=512, dist="normal", scale=0.5),
                                      seed=58))
    F = api.ag_num_flags(4, 128, 256)
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    slot = 5
    st, _, _ = _noalloc(api, prob, status,
                        api.make_opts(timeout_ns=50_000_000, fault_kind=api.FAULT_DROP_TILE,
                                      fault_arg=slot))
    assert st[0] == api.ERR_TIMEOUT, st
    assert (st[1], st[2]) == (slot // (F // 4), slot)
    for call in range(2):
        st, G, C = _noalloc(api, prob, status)
        assert st[0] == api.OK, (call, st)
        _check_against_oracle(prob, G, C, f"clean call {call}")


@pytest.fixture(scope="module")
def largest(api):
    """R=8 shards of 524288 x 64 with 64 x 64 flag tiles: 8 * 8192 * 1 =
    65536 flags (and as many row counters), every word of the array's flag
    part; with the oracle's G and C for it."""
    _gpu()
    R, M_r, K, N = 8, 524288, 64, 8
    assert api.ag_num_flags(R, M_r, K) == api.NOALLOC_MAX_FLAGS
    assert api.ag_num_row_counters(R, M_r, K) == api.NOALLOC_MAX_FLAGS
    prob = AgProblem(inputs.ag_inputs(dict(R=R, M_r=M_r, K=K, N=N, dist="normal", scale=0.5),
                                      seed=59))
    return prob, prob.oracle_full()


@pytest.mark.gpu
@pytest.mark.parametrize("signal_mode", ["tile_set", "row_add"])
def test_exactly_the_largest_flag_count(api, largest, signal_mode):
    """The whole of G and C is compared with the oracle."""
    prob, (G_ref, C_ref) = largest
    mode = api.SIGNAL_ROW_ADD if signal_mode == "row_add" else api.SIGNAL_TILE_SET
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    st, G, C = _noalloc(api, prob, status, api.make_opts(signal_mode=mode))
    assert st[0] == api.OK, st
    assert np.array_equal(host_bits(G), G_ref), f"{signal_mode}: gathered buffer differs"
    assert_gemm_close(host_bits(C), C_ref, what=f"{signal_mode} at the maximum: C")
    del G, C
    torch.cuda.empty_cache()


@pytest.mark.gpu
def test_calls_allocate_no_device_memory(api):
    """Free device memory (cudaMemGetInfo) is the same before and after
    several calls; the first call, which looks up the array and loads the
    kernels, comes before the first reading."""
    _gpu()
    prob = AgProblem(inputs.ag_inputs(dict(R=2, M_r=128, K=256, N=256, dist="normal", scale=0.5),
                                      seed=60))
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    args = (prob.heap, prob.rank_off, prob.a_off, prob.M_r, prob.N, prob.K, prob.B, prob.G, prob.C,
            status)
    assert api.ag_gemm_noalloc_status(*args) == api.OK
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for _ in range(5):
        assert api.ag_gemm_noalloc_status(*args) == api.OK
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0, (free0, free1)
    assert status.cpu().tolist()[0] == api.OK
    _check_against_oracle(prob, prob.G, prob.C, "after five calls")
