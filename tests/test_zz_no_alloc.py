"""opw_ag_gemm_noalloc: the AllGather -> GEMM call for callers that cannot
allocate device memory (a framework that owns all device memory through its
own pool, or a serving loop that cannot afford cudaMalloc's implicit device
synchronisation).  It keeps its flags and counters in a fixed array inside
the library, so it must give the same results as opw_ag_gemm, call after
call, even though every call reuses that array.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

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

    assert api.ag_num_flags(8, 8192, 32768) > api.NOALLOC_MAX_FLAGS
    assert call(8, 8192, 32768) == api.ERR_UNSUPPORTED_SHAPE
    assert call(2, 128, 256, opts=api.make_opts(role=api.ROLE_CONSUMER)) == api.ERR_INVALID_ARG
    assert call(2, 128, 256, status=_Ptr(0)) == api.ERR_INVALID_ARG
    assert call(2, 128, 256, status=_Ptr(0x500004)) == api.ERR_MISALIGNED


def _reference(api, d):
    """The existing entry point (with its own signal object) on the same inputs."""
    prob = AgProblem(d)
    sig = api.Signal(api.ag_num_flags(prob.R, prob.M_r, prob.K))
    prob.run(api, sig, sig.next_epoch())
    st = sig.status()
    assert st[0] == api.OK, st
    out = host_bits(prob.G), host_bits(prob.C)
    sig.close()
    return prob, out


@pytest.mark.gpu
def test_matches_ag_gemm_on_two_calls_in_a_row(api):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    cfg = dict(R=4, M_r=256, K=512, N=776, dist="normal", scale=0.5)
    status = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    for call, seed in enumerate((51, 52)):   # different inputs each call
        d = inputs.ag_inputs(cfg, seed=seed, slot_order=(2, 0, 3, 1))
        prob, (G_ref, C_ref) = _reference(api, d)
        # fresh outputs filled with NaN bits, so a stale or skipped tile shows
        G = torch.full_like(prob.G, float("nan"))
        C = torch.full_like(prob.C, float("nan"))
        rc = api.ag_gemm_noalloc_status(prob.heap, prob.rank_off, prob.a_off, prob.M_r, prob.N,
                                        prob.K, prob.B, G, C, status)
        assert rc == api.OK, (call, api.status_str(rc))
        torch.cuda.synchronize()
        assert status.cpu().tolist()[0] == api.OK, (call, status.cpu().tolist())
        assert np.array_equal(host_bits(G), G_ref), f"call {call}: gathered buffer differs"
        # same tolerance as every other C check, with the existing entry's C as reference
        from oracle import bf16_to_f64
        assert_gemm_close(host_bits(C), bf16_to_f64(C_ref), what=f"call {call}: C")
