"""Shared test helpers: device placement of the seeded inputs and the parity check.

Tolerance (floating point outputs): relative Frobenius error <= 1e-3 and
every |err| <= 1e-2 * max|C_ref|, where C_ref is the oracle's fp64 result
rounded once to bf16.  Gathered buffers, flags and epochs are compared
bit-exactly.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle

REL_FRO_TOL = 1e-3
ELEM_TOL = 1e-2


def dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def host_bits(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def heap_region_bits(heap_dev: torch.Tensor, off: int, rows: int, cols: int) -> np.ndarray:
    t = heap_dev[off:off + rows * cols * 2]
    return t.cpu().numpy().view(np.uint16).reshape(rows, cols)


def gemm_errors(got_bits: np.ndarray, ref64: np.ndarray):
    ref = oracle.bf16_to_f64(oracle.f64_to_bf16(ref64))
    got = oracle.bf16_to_f64(got_bits)
    err = got - ref
    nref = np.linalg.norm(ref)
    rel = float(np.linalg.norm(err) / nref) if nref > 0 else float(np.linalg.norm(err))
    mx = float(np.abs(err).max()) if err.size else 0.0
    scale = float(np.abs(ref).max()) if ref.size else 0.0
    return rel, mx, scale


def assert_gemm_close(got_bits: np.ndarray, ref64: np.ndarray, what: str = "C"):
    assert got_bits.shape == ref64.shape, (got_bits.shape, ref64.shape)
    rel, mx, scale = gemm_errors(got_bits, ref64)
    msg = f"{what}: rel_fro={rel:.3e} max_abs_err={mx:.3e} max|ref|={scale:.3e}"
    if not (rel <= REL_FRO_TOL and mx <= ELEM_TOL * scale):
        got = oracle.bf16_to_f64(got_bits)
        ref = oracle.bf16_to_f64(oracle.f64_to_bf16(ref64))
        bad = np.argwhere(np.abs(got - ref) > ELEM_TOL * scale)
        msg += f"; {len(bad)} elements out of tolerance, first {bad[:8].tolist()}"
        if len(bad):
            i, j = bad[0]
            msg += f" got={got[i, j]!r} ref={ref[i, j]!r}"
    assert rel <= REL_FRO_TOL and mx <= ELEM_TOL * scale, msg


class AgProblem:
    """Device buffers for one AllGather->GEMM problem built from inputs.ag_inputs()."""

    def __init__(self, d: dict):
        self.d = d
        self.R, self.M_r, self.K, self.N = d["R"], d["M_r"], d["K"], d["N"]
        self.M = self.R * self.M_r
        self.heap = dev_u8(d["heap"])
        self.B = dev_bf16(d["B"])
        self.G = torch.empty((self.M, self.K), dtype=torch.bfloat16, device="cuda")
        self.C = torch.empty((self.M, self.N), dtype=torch.bfloat16, device="cuda")
        self.rank_off = d["rank_off"]
        self.a_off = d["a_off"]

    def run(self, api, sig, epoch, opts=None, stream=None):
        api.ag_gemm(self.heap, self.rank_off, self.a_off, self.M_r, self.N, self.K, self.B,
                    self.G, self.C, sig, epoch, opts, stream)

    def oracle_full(self):
        return oracle.ag_gemm(self.d["heap"], self.rank_off, self.R, self.a_off, self.M_r,
                              self.N, self.K, self.d["B"])

    def oracle_rows(self, rows):
        return oracle.ag_gemm_rows(self.d["heap"], self.rank_off, self.R, self.a_off, self.M_r,
                                   self.N, self.K, self.d["B"], rows)


class RsProblem:
    """Device heap for one GEMM->ReduceScatter problem built from inputs.rs_inputs()."""

    def __init__(self, d: dict):
        self.d = d
        self.R, self.M, self.K_r, self.N = d["R"], d["M"], d["K_r"], d["N"]
        self.Mb = self.M // self.R
        self.heap = dev_u8(d["heap"])
        self.rank_off = d["rank_off"]

    def run(self, api, sig, epoch, opts=None, stream=None):
        d = self.d
        api.gemm_rs(self.heap, self.rank_off, d["a_off"], d["b_off"], d["out_off"], self.M,
                    self.N, self.K_r, sig, epoch, opts, stream)

    def out_bits(self, j: int) -> np.ndarray:
        return heap_region_bits(self.heap, int(self.rank_off[j]) + self.d["out_off"], self.Mb,
                                self.N)

    def oracle_rows(self, rows):
        d = self.d
        return oracle.gemm_rs_rows(d["heap"], self.rank_off, self.R, d["a_off"], d["b_off"],
                                   self.M, self.N, self.K_r, rows)


def sample_rows(M: int, tile: int, per_tile: int, seed: int) -> np.ndarray:
    """A few rows from every row tile (first, last and random ones)."""
    rng = np.random.default_rng(seed)
    rows = set()
    for t0 in range(0, M, tile):
        t1 = min(M, t0 + tile)
        rows.update([t0, t1 - 1])
        rows.update(rng.integers(t0, t1, size=per_tile).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def quarter_rows(M: int, seed: int) -> np.ndarray:
    """One random row from each 32-row quarter of every 128-row block: every
    epilogue warp of both CTAs of every pair tile writes one of them."""
    rng = np.random.default_rng(seed)
    base = np.arange(0, M, 32, dtype=np.int64)
    rows = base + rng.integers(0, 32, size=base.size)
    return np.minimum(rows, M - 1)
