"""Thin ctypes binding over the C ABI in ``include/opw.h`` (``libopw.so``).

Argument marshalling only: every step of the path runs in the library's
CUDA kernels.  PyTorch supplies device memory and streams.  There is no CPU
fallback: if the library is missing, every entry point raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_build", "libopw.so")

OK = 0
ERR_INVALID_ARG = 1
ERR_UNSUPPORTED_SHAPE = 2
ERR_MISALIGNED = 3
ERR_BAD_EPOCH = 4
ERR_CUDA = 5
ERR_TIMEOUT = 6
ERR_FLAG_PROTOCOL = 7
ERR_NOT_READY = 8

SYNC_OVERLAP, SYNC_SERIAL, SYNC_CHECKED = 0, 1, 2
SCHED_READY, SCHED_SWIZZLE = 0, 1
ROLE_FUSED, ROLE_PRODUCER, ROLE_CONSUMER = 0, 1, 2
FAULT_NONE, FAULT_DROP_TILE, FAULT_STALE_EPOCH = 0, 1, 2
SIGNAL_TILE_SET, SIGNAL_ROW_ADD = 0, 1
MAX_RANKS = 8
TRACE_MAX_CTAS = 1024

# Every symbol include/opw.h declares, with its ctypes signature.
_c_i64p = ctypes.POINTER(ctypes.c_int64)


class Symm(ctypes.Structure):
    _fields_ = [("heap_dev", ctypes.c_void_p), ("rank_off", _c_i64p),
                ("R", ctypes.c_int32), ("reserved", ctypes.c_int32)]


class Opts(ctypes.Structure):
    _fields_ = [("timeout_ns", ctypes.c_uint64), ("sync_mode", ctypes.c_int32),
                ("schedule", ctypes.c_int32), ("role", ctypes.c_int32),
                ("num_ctas", ctypes.c_int32),
                ("publish_perm", ctypes.POINTER(ctypes.c_int32)),
                ("delay_ns", ctypes.POINTER(ctypes.c_uint32)),
                ("trace_dev", ctypes.c_void_p), ("fault_kind", ctypes.c_int32),
                ("fault_arg", ctypes.c_int32), ("signal_mode", ctypes.c_int32),
                ("local_rank", ctypes.c_int32), ("tile_n", ctypes.c_int32)]


_vp = ctypes.c_void_p
SIGNATURES = {
    "opw_status_str": (ctypes.c_char_p, [ctypes.c_int32]),
    "opw_abi_version": (ctypes.c_int32, []),
    "opw_signal_alloc": (ctypes.c_int32, [ctypes.POINTER(_vp), ctypes.c_int64, _vp]),
    "opw_signal_reset": (ctypes.c_int32, [_vp, _vp]),
    "opw_signal_free": (ctypes.c_int32, [_vp]),
    "opw_signal_next_epoch": (ctypes.c_int32, [_vp, ctypes.POINTER(ctypes.c_uint64)]),
    "opw_signal_flags": (ctypes.c_int32, [_vp, ctypes.POINTER(_vp), _c_i64p]),
    "opw_status_sync": (ctypes.c_int32, [_vp, _vp, ctypes.POINTER(ctypes.c_int32),
                                         ctypes.POINTER(ctypes.c_int32)]),
    "opw_opts_default": (None, [ctypes.POINTER(Opts)]),
    "opw_ag_flag_tile": (ctypes.c_int64, [ctypes.c_int64, ctypes.c_int64]),
    "opw_ag_num_flags": (ctypes.c_int64, [ctypes.c_int32, ctypes.c_int64, ctypes.c_int64]),
    "opw_ag_num_row_counters": (ctypes.c_int64, [ctypes.c_int32, ctypes.c_int64,
                                                 ctypes.c_int64]),
    "opw_ag_trace_words": (ctypes.c_int64, [ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int64]),
    "opw_ag_tile_n": (ctypes.c_int32, [ctypes.c_int32, ctypes.c_int64, ctypes.c_int64,
                                       ctypes.POINTER(Opts)]),
    "opw_ag_gemm": (ctypes.c_int32, [ctypes.POINTER(Symm), ctypes.c_size_t, ctypes.c_int64,
                                     ctypes.c_int64, ctypes.c_int64, _vp, _vp, _vp, _vp,
                                     ctypes.c_uint64, ctypes.POINTER(Opts), _vp]),
    "opw_ag_gemm_noalloc": (ctypes.c_int32, [ctypes.POINTER(Symm), ctypes.c_size_t,
                                             ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, _vp,
                                             _vp, _vp, _vp, ctypes.POINTER(Opts), _vp]),
    "opw_rs_num_flags": (ctypes.c_int64, [ctypes.c_int32, ctypes.c_int64, ctypes.c_int64]),
    "opw_alltoall_num_flags": (ctypes.c_int64, [ctypes.c_int32, ctypes.c_int64]),
    "opw_alltoall": (ctypes.c_int32, [ctypes.POINTER(Symm), ctypes.c_size_t, ctypes.c_size_t,
                                      ctypes.c_int64, _vp, ctypes.c_uint64, ctypes.POINTER(Opts),
                                      _vp]),
    "opw_ring_num_flags": (ctypes.c_int64, [ctypes.c_int32, ctypes.c_int64]),
    "opw_ring_recv_bytes": (ctypes.c_int64, [ctypes.c_int32, ctypes.c_int64]),
    "opw_ring_allreduce": (ctypes.c_int32, [ctypes.POINTER(Symm), ctypes.c_size_t,
                                            ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int64,
                                            _vp, ctypes.c_uint64, ctypes.POINTER(Opts), _vp]),
    "opw_gemm_rs": (ctypes.c_int32, [ctypes.POINTER(Symm), ctypes.c_size_t, ctypes.c_size_t,
                                     ctypes.c_size_t, ctypes.c_int64, ctypes.c_int64,
                                     ctypes.c_int64, _vp, ctypes.c_uint64, ctypes.POINTER(Opts),
                                     _vp]),
    "opw_gemm_rs_consume": (ctypes.c_int32, [ctypes.POINTER(Symm), ctypes.c_size_t,
                                             ctypes.c_size_t, ctypes.c_size_t, ctypes.c_int64,
                                             ctypes.c_int64, ctypes.c_int64, _vp, _vp,
                                             ctypes.c_uint64, ctypes.POINTER(Opts), _vp]),
}

_lock = threading.Lock()
_lib = None


class OpwError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = int(status)
        super().__init__(f"{what}: {status_str(status)} ({status})")


def lib():
    """Load libopw.so (built by ``overlap_producer_warps_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "overlap_producer_warps_gb300.build.build()")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
        return _lib


def status_str(s: int) -> str:
    return lib().opw_status_str(int(s)).decode()


def _check(status: int, what: str):
    if status != OK:
        raise OpwError(status, what)


def _stream_ptr(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream or None


class _DevArray:
    """Zero-copy torch view of library-owned device memory."""

    def __init__(self, ptr: int, n: int, typestr: str):
        self.__cuda_array_interface__ = {"shape": (n,), "typestr": typestr,
                                         "data": (ptr, False), "version": 3}


class Signal:
    """A signal object: int64 flags, epoch counter and device status word."""

    def __init__(self, num_slots: int, stream=None):
        h = ctypes.c_void_p()
        _check(lib().opw_signal_alloc(ctypes.byref(h), int(num_slots), _stream_ptr(stream)),
               "opw_signal_alloc")
        self._h = h
        self.num_slots = int(num_slots)

    @property
    def handle(self):
        return self._h

    def reset(self, stream=None):
        _check(lib().opw_signal_reset(self._h, _stream_ptr(stream)), "opw_signal_reset")

    def next_epoch(self) -> int:
        e = ctypes.c_uint64()
        _check(lib().opw_signal_next_epoch(self._h, ctypes.byref(e)), "opw_signal_next_epoch")
        return int(e.value)

    def flags(self) -> torch.Tensor:
        """Device view (no copy) of the flag array."""
        p = ctypes.c_void_p()
        n = ctypes.c_int64()
        _check(lib().opw_signal_flags(self._h, ctypes.byref(p), ctypes.byref(n)),
               "opw_signal_flags")
        return torch.as_tensor(_DevArray(p.value, n.value, "<i8"), device="cuda")

    def status(self, stream=None):
        """(status, rank, slot) after synchronising the stream."""
        r = ctypes.c_int32()
        t = ctypes.c_int32()
        s = lib().opw_status_sync(self._h, _stream_ptr(stream), ctypes.byref(r), ctypes.byref(t))
        return int(s), int(r.value), int(t.value)

    def close(self):
        if getattr(self, "_h", None):
            lib().opw_signal_free(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def make_opts(timeout_ns=0, sync_mode=SYNC_OVERLAP, schedule=SCHED_READY, role=ROLE_FUSED,
              num_ctas=0, publish_perm=None, delay_ns=None, trace=None, fault_kind=FAULT_NONE,
              fault_arg=0, signal_mode=SIGNAL_TILE_SET, local_rank=0, tile_n=0):
    """Build an Opts struct; array arguments are kept alive on the struct."""
    o = Opts()
    lib().opw_opts_default(ctypes.byref(o))
    o.timeout_ns = int(timeout_ns)
    o.sync_mode = int(sync_mode)
    o.schedule = int(schedule)
    o.role = int(role)
    o.num_ctas = int(num_ctas)
    keep = []
    if publish_perm is not None:
        arr = (ctypes.c_int32 * len(publish_perm))(*[int(v) for v in publish_perm])
        keep.append(arr)
        o.publish_perm = ctypes.cast(arr, ctypes.POINTER(ctypes.c_int32))
    if delay_ns is not None:
        arr = (ctypes.c_uint32 * len(delay_ns))(*[int(v) for v in delay_ns])
        keep.append(arr)
        o.delay_ns = ctypes.cast(arr, ctypes.POINTER(ctypes.c_uint32))
    if trace is not None:
        o.trace_dev = trace.data_ptr()
    o.fault_kind = int(fault_kind)
    o.fault_arg = int(fault_arg)
    o.signal_mode = int(signal_mode)
    o.local_rank = int(local_rank)
    o.tile_n = int(tile_n)
    o._keep = keep
    return o


def _symm(heap: torch.Tensor, rank_off) -> Symm:
    ro = np.ascontiguousarray(np.asarray(rank_off, dtype=np.int64))
    s = Symm()
    s.heap_dev = heap.data_ptr()
    s.rank_off = ro.ctypes.data_as(_c_i64p)
    s.R = len(ro)
    s.reserved = 0
    s._keep = ro
    return s


def ag_flag_tile(M_r: int, K: int) -> int:
    return int(lib().opw_ag_flag_tile(M_r, K))


def ag_num_flags(R: int, M_r: int, K: int) -> int:
    return int(lib().opw_ag_num_flags(R, M_r, K))


def ag_num_row_counters(R: int, M_r: int, K: int) -> int:
    return int(lib().opw_ag_num_row_counters(R, M_r, K))


def ag_trace_words(R: int, M_r: int, N: int, K: int) -> int:
    return int(lib().opw_ag_trace_words(R, M_r, N, K))


def ag_tile_n(R: int, M_r: int, N: int, opts=None) -> int:
    """Pair tile columns (256 or 512) an AG-GEMM launch with these sizes and
    options uses on the current device (-1 on error)."""
    return int(lib().opw_ag_tile_n(int(R), int(M_r), int(N),
                                   ctypes.byref(opts) if opts is not None else None))


def rs_num_flags(R: int, M: int, N: int) -> int:
    return int(lib().opw_rs_num_flags(R, M, N))


def ag_gemm_status(heap, rank_off, a_off, M_r, N, K, B, G, C, sig: Signal, epoch, opts=None,
                   stream=None) -> int:
    """opw_ag_gemm, returning the raw status code."""
    s = _symm(heap, rank_off)
    return int(lib().opw_ag_gemm(ctypes.byref(s), int(a_off), int(M_r), int(N), int(K),
                                 B.data_ptr(), G.data_ptr(), C.data_ptr(), sig.handle,
                                 int(epoch), ctypes.byref(opts) if opts is not None else None,
                                 _stream_ptr(stream)))


def ag_gemm(heap, rank_off, a_off, M_r, N, K, B, G, C, sig: Signal, epoch, opts=None,
            stream=None):
    """AllGather -> GEMM (see opw_ag_gemm).  Asynchronous on `stream`."""
    _check(ag_gemm_status(heap, rank_off, a_off, M_r, N, K, B, G, C, sig, epoch, opts, stream),
           "opw_ag_gemm")


NOALLOC_MAX_FLAGS = 65536


def ag_gemm_noalloc_status(heap, rank_off, a_off, M_r, N, K, B, G, C, status, opts=None,
                           stream=None) -> int:
    """opw_ag_gemm_noalloc, for callers that cannot allocate device memory.

    Same result as ag_gemm, with its scratch in a fixed array inside the
    library instead of a signal object.  `status` is a caller-owned int32
    tensor of at least 4 contiguous elements on the current CUDA device (or
    any object whose data_ptr() is such a device address); it receives the
    device-side status.  Returns the host-side status code (ERR_INVALID_ARG
    for a status tensor of the wrong kind).
    """
    if isinstance(status, torch.Tensor):
        # the library writes 4 int32 words there from the current device
        if (not status.is_cuda or status.dtype != torch.int32 or status.numel() < 4
                or not status.is_contiguous()
                or status.device.index != torch.cuda.current_device()):
            return ERR_INVALID_ARG
    s = _symm(heap, rank_off)
    return int(lib().opw_ag_gemm_noalloc(ctypes.byref(s), int(a_off), int(M_r), int(N), int(K),
                                         B.data_ptr(), G.data_ptr(), C.data_ptr(),
                                         status.data_ptr(),
                                         ctypes.byref(opts) if opts is not None else None,
                                         _stream_ptr(stream)))


def gemm_rs_status(heap, rank_off, a_off, b_off, out_off, M, N, K_r, sig: Signal, epoch,
                   opts=None, stream=None) -> int:
    s = _symm(heap, rank_off)
    return int(lib().opw_gemm_rs(ctypes.byref(s), int(a_off), int(b_off), int(out_off), int(M),
                                 int(N), int(K_r), sig.handle, int(epoch),
                                 ctypes.byref(opts) if opts is not None else None,
                                 _stream_ptr(stream)))


def gemm_rs(heap, rank_off, a_off, b_off, out_off, M, N, K_r, sig: Signal, epoch, opts=None,
            stream=None):
    """GEMM -> ReduceScatter (see opw_gemm_rs).  Asynchronous on `stream`."""
    _check(gemm_rs_status(heap, rank_off, a_off, b_off, out_off, M, N, K_r, sig, epoch, opts,
                          stream), "opw_gemm_rs")


def gemm_rs_consume_status(heap, rank_off, a_off, b_off, out_off, M, N, K_r, recv,
                           sig: Signal, epoch, opts=None, stream=None) -> int:
    """opw_gemm_rs_consume, returning the raw status code."""
    s = _symm(heap, rank_off)
    return int(lib().opw_gemm_rs_consume(ctypes.byref(s), int(a_off), int(b_off), int(out_off),
                                         int(M), int(N), int(K_r),
                                         recv.data_ptr() if recv is not None else None,
                                         sig.handle, int(epoch),
                                         ctypes.byref(opts) if opts is not None else None,
                                         _stream_ptr(stream)))


def gemm_rs_consume(heap, rank_off, a_off, b_off, out_off, M, N, K_r, recv, sig: Signal, epoch,
                    opts=None, stream=None):
    """GEMM -> ReduceScatter with the receiving side in the same launch (see
    opw_gemm_rs_consume): `recv` ([M, N] bf16) gets every rank's block after
    its flags are acquired on the device.  Asynchronous on `stream`."""
    _check(gemm_rs_consume_status(heap, rank_off, a_off, b_off, out_off, M, N, K_r, recv, sig,
                                  epoch, opts, stream), "opw_gemm_rs_consume")


def ring_num_flags(R: int, n: int) -> int:
    return int(lib().opw_ring_num_flags(R, n))


def ring_recv_bytes(R: int, n: int) -> int:
    return int(lib().opw_ring_recv_bytes(R, n))


def ring_allreduce_status(heap, rank_off, data_off, recv_off, out_off, n, sig: Signal, epoch,
                          opts=None, stream=None) -> int:
    s = _symm(heap, rank_off)
    return int(lib().opw_ring_allreduce(ctypes.byref(s), int(data_off), int(recv_off),
                                        int(out_off), int(n), sig.handle, int(epoch),
                                        ctypes.byref(opts) if opts is not None else None,
                                        _stream_ptr(stream)))


def ring_allreduce(heap, rank_off, data_off, recv_off, out_off, n, sig: Signal, epoch,
                   opts=None, stream=None):
    """Tile-centric ring AllReduce over the logical ranks (see opw_ring_allreduce)."""
    _check(ring_allreduce_status(heap, rank_off, data_off, recv_off, out_off, n, sig, epoch,
                                 opts, stream), "opw_ring_allreduce")


def alltoall_num_flags(R: int, bytes_per_peer: int) -> int:
    return int(lib().opw_alltoall_num_flags(R, bytes_per_peer))


def alltoall_status(heap, rank_off, send_off, recv_off, bytes_per_peer, sig: Signal, epoch,
                    opts=None, stream=None) -> int:
    s = _symm(heap, rank_off)
    return int(lib().opw_alltoall(ctypes.byref(s), int(send_off), int(recv_off),
                                  int(bytes_per_peer), sig.handle, int(epoch),
                                  ctypes.byref(opts) if opts is not None else None,
                                  _stream_ptr(stream)))


def alltoall(heap, rank_off, send_off, recv_off, bytes_per_peer, sig: Signal, epoch, opts=None,
             stream=None):
    """All-to-all over the logical ranks with put + signal + epoch (see opw_alltoall)."""
    _check(alltoall_status(heap, rank_off, send_off, recv_off, bytes_per_peer, sig, epoch, opts,
                           stream), "opw_alltoall")
