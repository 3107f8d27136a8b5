"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds no arithmetic of the method: it only draws random values,
rounds the draws to bf16 bit patterns and lays tensors out in the logical
symmetric heap.  Both the CUDA path and the CPU oracle receive exactly these
bits.

Recipe (each tensor independently seeded, so shapes can change without
shifting other tensors' values):

* generator: ``numpy.random.default_rng([seed, tensor_id, rank])`` with
  tensor ids A = 1, B = 2 (the skew schedule uses ``[seed, 0x5E]``);
* values: fp32 draws (uniform[-1, 1] for the tiny case, normal(0, 0.02) for
  the tensor-parallel layers), rounded to bf16 with round-to-nearest-even;
* heap: one allocation with R equal slices; rank r's slice starts at
  ``rank_off[r]``; each symmetric tensor sits at the same offset in every
  slice ("Distributed Architecture Design", section 5: same size and layout
  on every rank).
"""
from __future__ import annotations

import numpy as np
import torch

TENSOR_A = 1
TENSOR_B = 2
TENSOR_SKEW = 0x5E
HEAP_ALIGN = 4096

# Workloads.  Shapes are those of the tensor-parallel layers the pages'
# overlap patterns target; "flag_tile" is the square A tile one flag guards.
CONFIGS = {
    # AllGather -> GEMM, tiny: 2 ranks of 64x128, B 128x128, 64x64 flag tiles.
    "ag_tiny": dict(kind="ag", R=2, M_r=64, K=128, N=128, flag_tile=64,
                    dist="uniform", scale=1.0, epochs=1),
    # AllGather -> GEMM, TP layer: 8 ranks of 1024x4096, B 4096x4096.
    "ag_tp": dict(kind="ag", R=8, M_r=1024, K=4096, N=4096, flag_tile=128,
                  dist="normal", scale=0.02, epochs=20),
    # GEMM -> ReduceScatter, TP layer: A_r 8192x1792, B_r 1792x4096, out 8x(1024x4096).
    "rs_tp": dict(kind="rs", R=8, M=8192, K_r=1792, N=4096, flag_tile=128,
                  dist="normal", scale=0.02, epochs=20),
    # AllGather -> GEMM, large MLP: 8 ranks of 2048x8192, B 8192x3584.
    "ag_mlp": dict(kind="ag", R=8, M_r=2048, K=8192, N=3584, flag_tile=128,
                   dist="normal", scale=0.02, epochs=20),
    # AllGather -> GEMM with skewed readiness: 8 ranks of 4096x8192, B 8192x8192,
    # ranks published in a seeded permutation with seeded 0-50 us delays.
    "ag_skew": dict(kind="ag", R=8, M_r=4096, K=8192, N=8192, flag_tile=128,
                    dist="normal", scale=0.02, epochs=20, skew=True),
}


def _round_bf16(x32: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 bit patterns (round-to-nearest-even, via torch's cast)."""
    t = torch.from_numpy(np.ascontiguousarray(x32, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def draw_bf16(shape, seed: int, tensor_id: int, rank: int, dist: str, scale: float) -> np.ndarray:
    rng = np.random.default_rng([seed, tensor_id, rank])
    if dist == "uniform":
        x = rng.uniform(-1.0, 1.0, size=shape).astype(np.float32) * np.float32(scale)
    elif dist == "normal":
        x = rng.standard_normal(size=shape, dtype=np.float32) * np.float32(scale)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return _round_bf16(x)


def _align(n: int, a: int = HEAP_ALIGN) -> int:
    return (n + a - 1) // a * a


def ag_layout(R: int, M_r: int, K: int):
    """Heap layout for AllGather->GEMM: A_r at offset 0 of each slice."""
    a_off = 0
    slice_bytes = _align(M_r * K * 2)
    return dict(a_off=a_off, slice_bytes=slice_bytes)


def rs_layout(R: int, M: int, K_r: int, N: int):
    """Heap layout for GEMM->ReduceScatter: A_r, B_r, out_r in each slice."""
    a_off = 0
    b_off = _align(M * K_r * 2)
    out_off = b_off + _align(K_r * N * 2)
    slice_bytes = out_off + _align((M // R) * N * 2)
    return dict(a_off=a_off, b_off=b_off, out_off=out_off, slice_bytes=slice_bytes)


def rank_offsets(R: int, slice_bytes: int, order=None) -> np.ndarray:
    """rank_off[r] = byte offset of rank r's slice.  `order` places rank
    order[i] in physical slot i, to exercise a non-identity table."""
    slots = np.arange(R) if order is None else np.argsort(np.asarray(order))
    return (slots.astype(np.int64) * slice_bytes).astype(np.int64)


def ag_inputs(cfg: dict, seed: int = 0, slot_order=None, M_r=None, K=None, N=None):
    """Host heap (uint8) with every shard placed, B (bf16 bits) and the layout."""
    R = cfg["R"]
    M_r = cfg["M_r"] if M_r is None else M_r
    K = cfg["K"] if K is None else K
    N = cfg["N"] if N is None else N
    lay = ag_layout(R, M_r, K)
    rank_off = rank_offsets(R, lay["slice_bytes"], slot_order)
    heap = np.zeros(R * lay["slice_bytes"], dtype=np.uint8)
    for r in range(R):
        A_r = draw_bf16((M_r, K), seed, TENSOR_A, r, cfg["dist"], cfg["scale"])
        o = int(rank_off[r]) + lay["a_off"]
        heap[o:o + A_r.nbytes] = A_r.view(np.uint8).reshape(-1)
    B = draw_bf16((K, N), seed, TENSOR_B, 0, cfg["dist"], cfg["scale"])
    return dict(heap=heap, rank_off=rank_off, B=B, R=R, M_r=M_r, K=K, N=N, **lay)


def rs_inputs(cfg: dict, seed: int = 0, slot_order=None, M=None, K_r=None, N=None):
    R = cfg["R"]
    M = cfg["M"] if M is None else M
    K_r = cfg["K_r"] if K_r is None else K_r
    N = cfg["N"] if N is None else N
    lay = rs_layout(R, M, K_r, N)
    rank_off = rank_offsets(R, lay["slice_bytes"], slot_order)
    heap = np.zeros(R * lay["slice_bytes"], dtype=np.uint8)
    for r in range(R):
        A_r = draw_bf16((M, K_r), seed, TENSOR_A, r, cfg["dist"], cfg["scale"])
        B_r = draw_bf16((K_r, N), seed, TENSOR_B, r, cfg["dist"], cfg["scale"])
        o = int(rank_off[r])
        heap[o + lay["a_off"]:o + lay["a_off"] + A_r.nbytes] = A_r.view(np.uint8).reshape(-1)
        heap[o + lay["b_off"]:o + lay["b_off"] + B_r.nbytes] = B_r.view(np.uint8).reshape(-1)
    return dict(heap=heap, rank_off=rank_off, R=R, M=M, K_r=K_r, N=N, **lay)


def skew_schedule(seed: int, R: int):
    """Rank publish permutation and per-rank start delays (0-50 us, as ns)."""
    rng = np.random.default_rng([seed, TENSOR_SKEW])
    perm = rng.permutation(R).astype(np.int32)
    delay_us = rng.integers(0, 51, size=R)
    return perm, (delay_us * 1000).astype(np.uint32)


def ring_layout(R: int, n: int):
    """Heap layout for the ring AllReduce: data, receive area, output."""
    data_off = 0
    recv_off = _align(n * 4)
    out_off = recv_off + _align(max(1, 2 * R - 2) * (n // R) * 4)
    slice_bytes = out_off + _align(n * 4)
    return dict(data_off=data_off, recv_off=recv_off, out_off=out_off, slice_bytes=slice_bytes)


def ring_inputs(R: int, n: int, seed: int = 0, slot_order=None, scale: float = 1.0):
    """fp32 normal(0, scale) data per rank (tensor id A), placed in the heap."""
    lay = ring_layout(R, n)
    rank_off = rank_offsets(R, lay["slice_bytes"], slot_order)
    heap = np.zeros(R * lay["slice_bytes"], dtype=np.uint8)
    for r in range(R):
        rng = np.random.default_rng([seed, TENSOR_A, r])
        x = rng.standard_normal(n, dtype=np.float32) * np.float32(scale)
        o = int(rank_off[r]) + lay["data_off"]
        heap[o:o + n * 4] = x.view(np.uint8)
    return dict(heap=heap, rank_off=rank_off, R=R, n=n, **lay)


def alltoall_inputs(R: int, bytes_per_peer: int, seed: int = 0, slot_order=None):
    """Random send buffers (uniform bytes, tensor id A) and an empty receive area."""
    B = bytes_per_peer
    send_off = 0
    recv_off = _align(R * B)
    slice_bytes = recv_off + _align(R * B)
    rank_off = rank_offsets(R, slice_bytes, slot_order)
    heap = np.zeros(R * slice_bytes, dtype=np.uint8)
    for r in range(R):
        rng = np.random.default_rng([seed, TENSOR_A, r])
        o = int(rank_off[r]) + send_off
        heap[o:o + R * B] = rng.integers(0, 256, R * B, dtype=np.uint8)
    return dict(heap=heap, rank_off=rank_off, R=R, B=B, send_off=send_off, recv_off=recv_off,
                slice_bytes=slice_bytes)
