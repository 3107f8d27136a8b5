"""CPU oracle for the AllGather->GEMM / GEMM->ReduceScatter hot path.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg (``cpu_baseline`` and ``--impl reference``)
may import this package.  The product path (the CUDA library and its Python
binding) never imports, links or runs anything here, and this package never
imports the product.

The arithmetic lives in ``opw_oracle.c`` (plain C, fp64, no BLAS); this module
only compiles it with gcc and marshals numpy arrays through ctypes.  Each
function cites the passage of the pages it follows:

* "Triton-distributed Semantics" -- sections "AllGather and GEMM Overlapping",
  "GEMM and ReduceScatter Overlapping", "Threadblock Swizzling", "Example: Ring
  AllReduce with Overlap".
* Aboleth README -- Tier-2 all-to-all (put, signal with epoch, wait).
* "Distributed Architecture Design" -- section 2.3 (SignalOp SET and ADD) and
  section 5.3 (how symm_at finds a remote address).

Parity pins: every function here is pinned by ``tests/test_oracle_pins.py``
against brute force on tiny inputs, closed forms, library routines on special
cases and hand-computed fixtures under ``tests/golden/``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# The test of the pins themselves (tests/test_oracle_mutations.py) plants one
# mistake in a copy of the C source and names the copy in OPW_ORACLE_SRC; the
# library is then built next to that copy, never over the real one.
_SRC = os.environ.get("OPW_ORACLE_SRC") or os.path.join(_HERE, "opw_oracle.c")
_BUILD_DIR = (os.path.join(os.path.dirname(os.path.abspath(_SRC)), "_build")
              if os.environ.get("OPW_ORACLE_SRC") else os.path.join(_HERE, "_build"))
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_i64p = ctypes.POINTER(ctypes.c_int64)
_u16p = ctypes.POINTER(ctypes.c_uint16)
_u8p = ctypes.POINTER(ctypes.c_uint8)
_f64p = ctypes.POINTER(ctypes.c_double)
_f32p = ctypes.POINTER(ctypes.c_float)


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, -O2, no FP contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
           "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        sig = {
            "opw_oracle_threads": (ctypes.c_int, []),
            "opw_oracle_bf16_to_f64": (ctypes.c_double, [ctypes.c_uint16]),
            "opw_oracle_f64_to_bf16": (ctypes.c_uint16, [ctypes.c_double]),
            "opw_oracle_bf16_decode_array": (None, [_u16p, _f64p, ctypes.c_int64]),
            "opw_oracle_bf16_encode_array": (None, [_f64p, _u16p, ctypes.c_int64]),
            "opw_oracle_symm_at": (ctypes.c_uint64, [ctypes.c_uint64] * 3),
            "opw_oracle_allgather": (None, [_u8p, _i64p, ctypes.c_int, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_int64, _u16p]),
            "opw_oracle_gemm_f64": (None, [_u16p, ctypes.c_int64, _u16p, ctypes.c_int64,
                                           ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                           _f64p, ctypes.c_int64]),
            "opw_oracle_ag_gemm": (None, [_u8p, _i64p, ctypes.c_int, ctypes.c_int64,
                                          ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                          _u16p, _u16p, _f64p]),
            "opw_oracle_ag_gemm_rows": (None, [_u8p, _i64p, ctypes.c_int, ctypes.c_int64,
                                               ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                               _u16p, ctypes.c_int64, _i64p, _f64p]),
            "opw_oracle_gemm_rs": (None, [_u8p, _i64p, ctypes.c_int, ctypes.c_int64,
                                          ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                          ctypes.c_int64, ctypes.c_int64, _f64p, _u8p]),
            "opw_oracle_gemm_rs_rows": (None, [_u8p, _i64p, ctypes.c_int, ctypes.c_int64,
                                               ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                               ctypes.c_int64, ctypes.c_int64, _i64p, _f64p]),
            "opw_oracle_gemm_rs_rows_f32": (None, [_u8p, _i64p, ctypes.c_int, ctypes.c_int64,
                                                   ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                                   ctypes.c_int64, ctypes.c_int64, _i64p, _f32p]),
            "opw_oracle_expected_flags": (None, [ctypes.c_int64, ctypes.c_int64, _i64p]),
            "opw_oracle_expected_row_counters": (None, [ctypes.c_int64, ctypes.c_int64,
                                                        ctypes.c_int64, _i64p]),
            "opw_oracle_ring_allreduce": (None, [_u8p, _i64p, ctypes.c_int, ctypes.c_int64,
                                                 ctypes.c_int64, ctypes.c_int64, _u8p]),
            "opw_oracle_alltoall": (None, [_u8p, _i64p, ctypes.c_int, ctypes.c_int64,
                                           ctypes.c_int64, ctypes.c_int64, _u8p]),
            "opw_oracle_swizzle_row": (ctypes.c_int64, [ctypes.c_int64] * 4),
            "opw_oracle_consumer_order": (ctypes.c_int64, [ctypes.c_int64] * 7 + [_i64p, _i64p]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _p(a: np.ndarray, ptr_t):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data_as(ptr_t)


def threads() -> int:
    """OpenMP threads the oracle uses (OMP_NUM_THREADS, else all cores)."""
    return int(_load().opw_oracle_threads())


# -- bf16 codec ---------------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    out = np.empty(bits.shape, dtype=np.float64)
    _load().opw_oracle_bf16_decode_array(_p(bits, _u16p), _p(out, _f64p), bits.size)
    return out


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """fp64 -> bf16 bits, one round-to-nearest-even step."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(x.shape, dtype=np.uint16)
    _load().opw_oracle_bf16_encode_array(_p(x, _f64p), _p(out, _u16p), x.size)
    return out


def f64_to_bf16_scalar(x: float) -> int:
    return int(_load().opw_oracle_f64_to_bf16(float(x)))


# -- symm_at ------------------------------------------------------------------

def symm_at(ptr: int, heap_base_self: int, heap_base_pe: int) -> int:
    return int(_load().opw_oracle_symm_at(ptr, heap_base_self, heap_base_pe))


# -- AllGather / GEMM ---------------------------------------------------------

def _heap_args(heap: np.ndarray, rank_off):
    heap = np.ascontiguousarray(heap, dtype=np.uint8)
    ro = np.ascontiguousarray(np.asarray(rank_off, dtype=np.int64))
    return heap, ro


def allgather(heap, rank_off, R, a_off, M_r, K) -> np.ndarray:
    heap, ro = _heap_args(heap, rank_off)
    G = np.empty((R * M_r, K), dtype=np.uint16)
    _load().opw_oracle_allgather(_p(heap, _u8p), _p(ro, _i64p), R, a_off, M_r, K, _p(G, _u16p))
    return G


def gemm_f64(A: np.ndarray, B: np.ndarray) -> np.ndarray:
    """C = A @ B for bf16 bit arrays, fp64 accumulate in ascending k."""
    A = np.ascontiguousarray(A, dtype=np.uint16)
    B = np.ascontiguousarray(B, dtype=np.uint16)
    M, K = A.shape
    K2, N = B.shape
    assert K == K2
    C = np.empty((M, N), dtype=np.float64)
    _load().opw_oracle_gemm_f64(_p(A, _u16p), K, _p(B, _u16p), N, M, N, K, _p(C, _f64p), N)
    return C


def ag_gemm(heap, rank_off, R, a_off, M_r, N, K, B):
    """Returns (G bf16 bits [R*M_r, K], C fp64 [R*M_r, N])."""
    heap, ro = _heap_args(heap, rank_off)
    B = np.ascontiguousarray(B, dtype=np.uint16)
    G = np.empty((R * M_r, K), dtype=np.uint16)
    C = np.empty((R * M_r, N), dtype=np.float64)
    _load().opw_oracle_ag_gemm(_p(heap, _u8p), _p(ro, _i64p), R, a_off, M_r, N, K,
                               _p(B, _u16p), _p(G, _u16p), _p(C, _f64p))
    return G, C


def ag_gemm_rows(heap, rank_off, R, a_off, M_r, N, K, B, rows) -> np.ndarray:
    heap, ro = _heap_args(heap, rank_off)
    B = np.ascontiguousarray(B, dtype=np.uint16)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((rows.size, N), dtype=np.float64)
    _load().opw_oracle_ag_gemm_rows(_p(heap, _u8p), _p(ro, _i64p), R, a_off, M_r, N, K,
                                    _p(B, _u16p), rows.size, _p(rows, _i64p), _p(out, _f64p))
    return out


# -- GEMM-RS ------------------------------------------------------------------

def gemm_rs(heap, rank_off, R, a_off, b_off, out_off, M, N, K_r):
    """Returns (S fp64 [M, N], heap_out uint8 with each rank's bf16 block)."""
    heap, ro = _heap_args(heap, rank_off)
    S = np.empty((M, N), dtype=np.float64)
    heap_out = heap.copy()
    _load().opw_oracle_gemm_rs(_p(heap, _u8p), _p(ro, _i64p), R, a_off, b_off, out_off,
                               M, N, K_r, _p(S, _f64p), _p(heap_out, _u8p))
    return S, heap_out


def gemm_rs_rows(heap, rank_off, R, a_off, b_off, M, N, K_r, rows) -> np.ndarray:
    heap, ro = _heap_args(heap, rank_off)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((rows.size, N), dtype=np.float64)
    _load().opw_oracle_gemm_rs_rows(_p(heap, _u8p), _p(ro, _i64p), R, a_off, b_off, M, N, K_r,
                                    rows.size, _p(rows, _i64p), _p(out, _f64p))
    return out


def gemm_rs_rows_f32(heap, rank_off, R, a_off, b_off, M, N, K_r, rows) -> np.ndarray:
    heap, ro = _heap_args(heap, rank_off)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    out = np.empty((rows.size, N), dtype=np.float32)
    _load().opw_oracle_gemm_rs_rows_f32(_p(heap, _u8p), _p(ro, _i64p), R, a_off, b_off, M, N,
                                        K_r, rows.size, _p(rows, _i64p), _p(out, _f32p))
    return out


# -- signals and schedule -----------------------------------------------------

def expected_flags(n_slots: int, epoch: int) -> np.ndarray:
    out = np.empty(n_slots, dtype=np.int64)
    _load().opw_oracle_expected_flags(n_slots, epoch, _p(out, _i64p))
    return out


def expected_row_counters(n_rows: int, epoch: int, T_k: int) -> np.ndarray:
    out = np.empty(n_rows, dtype=np.int64)
    _load().opw_oracle_expected_row_counters(n_rows, epoch, T_k, _p(out, _i64p))
    return out


def swizzle_row(pid_m: int, rank: int, tiles_per_pe: int, total_tiles: int) -> int:
    return int(_load().opw_oracle_swizzle_row(pid_m, rank, tiles_per_pe, total_tiles))


def consumer_order(T_M: int, T_N: int, G: int, c: int, group_rows: int, rank: int,
                   tiles_per_pe: int, visit=None) -> np.ndarray:
    """Visit order (tile indices q = m*T_N + n) of consumer c of rank `rank`;
    `visit` (optional) lists the ranks in the order their rows are taken."""
    T = T_M * T_N
    out = np.empty(max(1, (T + G - 1) // G), dtype=np.int64)
    v = None if visit is None else np.ascontiguousarray(np.asarray(visit, dtype=np.int64))
    n = _load().opw_oracle_consumer_order(T_M, T_N, G, c, group_rows, rank, tiles_per_pe,
                                          None if v is None else _p(v, _i64p), _p(out, _i64p))
    return out[:n].copy()


# -- ring AllReduce -------------------------------------------------------------

def ring_allreduce(heap, rank_off, R, data_off, out_off, n):
    """heap_out (uint8, laid out like the heap) with every rank's fp32 result."""
    heap, ro = _heap_args(heap, rank_off)
    heap_out = heap.copy()
    _load().opw_oracle_ring_allreduce(_p(heap, _u8p), _p(ro, _i64p), R, data_off, out_off, n,
                                      _p(heap_out, _u8p))
    return heap_out


# -- all-to-all -----------------------------------------------------------------

def alltoall(heap, rank_off, R, send_off, recv_off, B):
    """heap_out with every rank's receive buffer filled (B bytes per slice)."""
    heap, ro = _heap_args(heap, rank_off)
    heap_out = heap.copy()
    _load().opw_oracle_alltoall(_p(heap, _u8p), _p(ro, _i64p), R, send_off, recv_off, B,
                                _p(heap_out, _u8p))
    return heap_out
