"""The C ABI on a machine without a GPU: it loads, exports every function
include/opw.h declares, has the struct layout a C compiler gives the header,
and rejects bad arguments on the host before touching CUDA."""
import ctypes
import os
import re
import subprocess

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "opw.h")


@pytest.fixture(scope="module")
def api():
    from overlap_producer_warps_gb300 import api as _api
    from overlap_producer_warps_gb300 import build as _b
    _b.build()
    _api.lib()
    return _api


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(opw_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_expected_calls():
    names = declared_functions()
    for required in ["opw_ag_gemm", "opw_gemm_rs", "opw_signal_alloc", "opw_signal_reset",
                     "opw_signal_free", "opw_signal_next_epoch", "opw_status_sync"]:
        assert required in names


def test_every_declared_symbol_is_exported(api):
    lib = api.lib()
    names = declared_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding covers exactly the declared set
    assert sorted(api.SIGNATURES) == names


def test_struct_layout_matches_c_compiler(api):
    src = r"""
#include <stddef.h>
#include <stdio.h>
#include "opw.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu %zu\n", sizeof(opw_opts),
    offsetof(opw_opts, timeout_ns), offsetof(opw_opts, sync_mode), offsetof(opw_opts, schedule),
    offsetof(opw_opts, role), offsetof(opw_opts, num_ctas), offsetof(opw_opts, publish_perm),
    offsetof(opw_opts, delay_ns), offsetof(opw_opts, trace_dev), offsetof(opw_opts, fault_kind),
    offsetof(opw_opts, fault_arg), offsetof(opw_opts, signal_mode), offsetof(opw_opts, local_rank),
    offsetof(opw_opts, tile_n));
  printf("%zu %zu %zu %zu %zu\n", sizeof(opw_symm), offsetof(opw_symm, heap_dev),
    offsetof(opw_symm, rank_off), offsetof(opw_symm, R), offsetof(opw_symm, reserved));
  return 0;
}
"""
    d = os.path.dirname(api.LIB_PATH)  # the library's build folder (not tracked)
    c = os.path.join(d, "layout.c")
    exe = os.path.join(d, "layout")
    open(c, "w").write(src)
    subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), c, "-o", exe], check=True)
    out = subprocess.run([exe], capture_output=True, text=True, check=True).stdout.split("\n")
    opts = [int(v) for v in out[0].split()]
    symm = [int(v) for v in out[1].split()]
    O, S = api.Opts, api.Symm
    assert opts == [ctypes.sizeof(O)] + [getattr(O, f).offset for f, _ in O._fields_]
    assert symm == [ctypes.sizeof(S)] + [getattr(S, f).offset for f, _ in S._fields_]


def test_binding_constants_match_the_header(api):
    """Every OPW_* enum value the binding uses equals the header's #define."""
    defs = dict(re.findall(r"^#define OPW_(\w+)\s+(-?\d+)", open(HEADER).read(), re.M))
    names = [n for n in dir(api) if n.isupper() and not n.startswith("_") and n in defs]
    for n in ("OK", "ERR_FLAG_PROTOCOL", "SYNC_CHECKED", "SCHED_SWIZZLE", "ROLE_CONSUMER",
              "FAULT_STALE_EPOCH", "SIGNAL_ROW_ADD", "MAX_RANKS", "TRACE_MAX_CTAS"):
        assert n in names, n
    for n in names:
        assert getattr(api, n) == int(defs[n]), n


def test_status_strings(api):
    for code, name in [(0, "OK"), (1, "INVALID_ARG"), (2, "UNSUPPORTED_SHAPE"), (3, "MISALIGNED"),
                       (4, "BAD_EPOCH"), (5, "CUDA_ERROR"), (6, "TIMEOUT"), (7, "FLAG_PROTOCOL"),
                       (8, "NOT_READY"), (99, "UNKNOWN")]:
        assert api.status_str(code) == name
    assert api.lib().opw_abi_version() == 2


def test_flag_geometry(api):
    assert api.ag_flag_tile(1024, 4096) == 128
    assert api.ag_flag_tile(64, 128) == 64
    assert api.ag_flag_tile(192, 320) == 64
    assert api.ag_flag_tile(96, 128) == -1
    assert api.ag_num_flags(2, 64, 128) == 4            # the tiny configuration
    assert api.ag_num_flags(8, 1024, 4096) == 2048      # 8 ranks x 8 x 32
    assert api.ag_num_flags(8, 4096, 8192) == 16384
    assert api.ag_num_flags(9, 128, 128) == -1
    assert api.ag_num_row_counters(8, 1024, 4096) == 64   # 8 ranks x 8 row tiles
    assert api.ag_num_row_counters(2, 64, 128) == 2
    assert api.rs_num_flags(8, 8192, 4096) == 2048      # 8 ranks x 8 x 32
    assert api.rs_num_flags(8, 8192 + 128, 4096) == -1
    assert api.ring_num_flags(8, 8 * 4096) == 8 * 14 * 4      # 4 pieces of 1024 per chunk
    assert api.ring_num_flags(3, 3 * 400) == 3 * 4 * 1
    assert api.ring_num_flags(3, 1001) == -1
    assert api.ring_recv_bytes(8, 8 * 4096) == 14 * 4096 * 4
    assert api.alltoall_num_flags(8, 65536) == 8 * 8 * 2       # 32 KiB pieces
    assert api.alltoall_num_flags(3, 48) == 9
    assert api.alltoall_num_flags(3, 40) == -1
    F, T = 2048, 32 * 16  # 256x256 pair tiles
    assert api.ag_trace_words(8, 1024, 4096, 4096) == 2 * F + 2 * T + api.TRACE_MAX_CTAS


class _Fake:
    """Host-side stand-ins: the calls below must fail validation before any
    pointer is used, so plain aligned integers do as device addresses."""

    def __init__(self, value):
        self._v = value

    def data_ptr(self):
        return self._v


def _fake_sig():
    buf = ctypes.create_string_buffer(512)  # num_slots reads as 0
    class S:
        handle = ctypes.cast(buf, ctypes.c_void_p)
    S._buf = buf
    return S


def _ag(api, R=2, M_r=128, N=256, K=256, heap=0x100000, rank_off=None, a_off=0, B=0x200000,
        G=0x300000, C=0x400000, sig=None, epoch=1, opts=None):
    rank_off = [i * 65536 for i in range(R)] if rank_off is None else rank_off
    sig = _fake_sig() if sig is None else sig
    return api.ag_gemm_status(_Fake(heap), rank_off, a_off, M_r, N, K, _Fake(B), _Fake(G), _Fake(C),
                              sig, epoch, opts, stream=_NoStream())


class _NoStream:
    cuda_stream = 0


def test_ag_gemm_rejects_bad_arguments_on_the_host(api):
    E = api
    assert _ag(api, R=0, rank_off=[]) == E.ERR_INVALID_ARG
    assert _ag(api, R=9) == E.ERR_INVALID_ARG
    assert _ag(api, heap=0) == E.ERR_INVALID_ARG
    assert _ag(api, B=0) == E.ERR_INVALID_ARG
    assert _ag(api, heap=0x100008) == E.ERR_MISALIGNED
    assert _ag(api, rank_off=[0, 65544]) == E.ERR_MISALIGNED
    assert _ag(api, a_off=8) == E.ERR_MISALIGNED
    assert _ag(api, C=0x400004) == E.ERR_MISALIGNED
    assert _ag(api, M_r=100) == E.ERR_UNSUPPORTED_SHAPE
    assert _ag(api, K=96) == E.ERR_UNSUPPORTED_SHAPE
    assert _ag(api, N=100) == E.ERR_UNSUPPORTED_SHAPE
    assert _ag(api, N=0) == E.ERR_UNSUPPORTED_SHAPE
    assert _ag(api, opts=api.make_opts(sync_mode=7)) == E.ERR_INVALID_ARG
    assert _ag(api, opts=api.make_opts(role=3)) == E.ERR_INVALID_ARG
    assert _ag(api, opts=api.make_opts(publish_perm=[0, 0])) == E.ERR_INVALID_ARG
    assert _ag(api, opts=api.make_opts(publish_perm=[0, 2])) == E.ERR_INVALID_ARG
    assert _ag(api, opts=api.make_opts(signal_mode=2)) == E.ERR_INVALID_ARG
    assert _ag(api, opts=api.make_opts(local_rank=-2)) == E.ERR_INVALID_ARG
    assert _ag(api, opts=api.make_opts(local_rank=2)) == E.ERR_INVALID_ARG   # R = 2
    for tn in (128, 384, 1024, -256):                   # pair tiles are 256 or 512 wide
        assert _ag(api, opts=api.make_opts(tile_n=tn)) == E.ERR_INVALID_ARG
    # an explicit tile width is returned as is, without a device
    assert api.ag_tile_n(2, 128, 1024, api.make_opts(tile_n=512)) == 512
    assert api.ag_tile_n(2, 128, 1024, api.make_opts(tile_n=256)) == 256
    assert api.ag_tile_n(2, 128, 1024, api.make_opts(tile_n=384)) == -1
    assert api.ag_tile_n(9, 128, 1024, api.make_opts(tile_n=256)) == -1
    # a signal object with too few slots (here: none)
    assert _ag(api) == E.ERR_INVALID_ARG


def test_gemm_rs_rejects_bad_arguments_on_the_host(api):
    E = api
    s = _fake_sig()
    ns = _NoStream()

    def rs(M=512, N=256, K_r=128, a_off=0, b_off=0, out_off=0, opts=None, R=2):
        return api.gemm_rs_status(_Fake(0x100000), [i * 65536 for i in range(R)], a_off, b_off,
                                  out_off, M, N, K_r, s, 1, opts, stream=ns)

    assert rs(M=384) == E.ERR_UNSUPPORTED_SHAPE        # M/R not a multiple of 128
    assert rs(N=12) == E.ERR_UNSUPPORTED_SHAPE
    assert rs(K_r=4) == E.ERR_UNSUPPORTED_SHAPE
    assert rs(b_off=8) == E.ERR_MISALIGNED
    assert rs(opts=api.make_opts(publish_perm=[1, 0])) == E.ERR_INVALID_ARG
    assert rs(opts=api.make_opts(role=3)) == E.ERR_INVALID_ARG
    assert rs(opts=api.make_opts(role=-1)) == E.ERR_INVALID_ARG
    assert rs(opts=api.make_opts(tile_n=512)) == E.ERR_INVALID_ARG   # AG-GEMM only
    assert rs(opts=api.make_opts(sync_mode=api.SYNC_SERIAL)) == E.ERR_INVALID_ARG
    assert rs(opts=api.make_opts(fault_kind=api.FAULT_STALE_EPOCH)) == E.ERR_INVALID_ARG
    assert rs() == E.ERR_INVALID_ARG                    # too few slots


def test_gemm_rs_consume_rejects_bad_arguments_on_the_host(api):
    s = _fake_sig()
    ns = _NoStream()

    def rsc(recv=_Fake(0x900000), opts=None, M=512, N=256, K_r=128, R=2):
        return api.gemm_rs_consume_status(_Fake(0x100000), [i * 65536 for i in range(R)], 0, 0,
                                          0, M, N, K_r, recv, s, 1, opts, stream=ns)

    assert rsc(recv=None) == api.ERR_INVALID_ARG
    assert rsc(recv=_Fake(0x900008)) == api.ERR_MISALIGNED
    # only a fused launch publishes results for the receiving side to wait on
    assert rsc(opts=api.make_opts(role=api.ROLE_PRODUCER)) == api.ERR_INVALID_ARG
    assert rsc(opts=api.make_opts(role=api.ROLE_CONSUMER)) == api.ERR_INVALID_ARG
    assert rsc(N=12) == api.ERR_UNSUPPORTED_SHAPE
    assert rsc() == api.ERR_INVALID_ARG                 # too few slots


@pytest.mark.skipif(torch.cuda.is_available(), reason="checks the no-GPU error path")
def test_signal_alloc_without_gpu_reports_cuda_error(api):
    h = ctypes.c_void_p()
    assert api.lib().opw_signal_alloc(ctypes.byref(h), 16, None) == api.ERR_CUDA
    assert h.value is None
    assert api.lib().opw_signal_alloc(None, 16, None) == api.ERR_INVALID_ARG
    assert api.lib().opw_signal_free(None) == api.OK


def test_ring_allreduce_rejects_bad_arguments_on_the_host(api):
    s = _fake_sig()

    def ring(n=4096, R=4, data_off=0, recv_off=65536, out_off=262144, opts=None):
        return api.ring_allreduce_status(_Fake(0x100000), [i * (1 << 20) for i in range(R)],
                                         data_off, recv_off, out_off, n, s, 1, opts,
                                         stream=_NoStream())

    assert ring(n=4098) == api.ERR_UNSUPPORTED_SHAPE     # not a multiple of 4R
    assert ring(n=0) == api.ERR_UNSUPPORTED_SHAPE
    assert ring(recv_off=8) == api.ERR_MISALIGNED
    assert ring(opts=api.make_opts(sync_mode=1)) == api.ERR_INVALID_ARG
    assert ring(R=9) == api.ERR_INVALID_ARG
    assert ring() == api.ERR_INVALID_ARG                   # too few slots


def test_alltoall_rejects_bad_arguments_on_the_host(api):
    s = _fake_sig()

    def a2a(B=4096, R=4, send_off=0, recv_off=65536, opts=None):
        return api.alltoall_status(_Fake(0x100000), [i * (1 << 20) for i in range(R)], send_off,
                                   recv_off, B, s, 1, opts, stream=_NoStream())

    assert a2a(B=40) == api.ERR_UNSUPPORTED_SHAPE
    assert a2a(send_off=4) == api.ERR_MISALIGNED
    assert a2a(opts=api.make_opts(role=1)) == api.ERR_INVALID_ARG
    assert a2a() == api.ERR_INVALID_ARG                    # too few slots
