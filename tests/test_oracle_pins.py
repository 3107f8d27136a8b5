"""Pins for the CPU oracle: each check ties it to something other than itself.

Pins used: a library routine on the decode (torch's bf16 widening) and on
fp32 inputs of the encoder, the nearest-value property of rounding checked
by brute force against both neighbours, hand-computed fixtures under
tests/golden/, exact brute force on small integer inputs, closed forms
(identity, all-ones, one-hot), numpy's fp64 matmul within the fp64 error
bound, and the concat-K identity for the reduce-scatter.
"""
import numpy as np
import pytest
import torch

import oracle
from overlap_producer_warps_gb300 import inputs


# ---------------------------------------------------------------- bf16 codec

def _torch_bf16_to_f64(bits):
    return torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).double().numpy()


def test_bf16_decode_every_pattern_matches_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f64(bits)
    ref = _torch_bf16_to_f64(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], ref[~nan])
    assert np.array_equal(np.signbit(ours[~nan]), np.signbit(ref[~nan]))


def test_bf16_encode_golden(golden):
    for case in golden("bf16_rne.json")["cases"]:
        x = float.fromhex(case["x"])
        assert oracle.f64_to_bf16_scalar(x) == int(case["bf16"], 16), case


def test_bf16_encode_matches_torch_on_binary32_inputs():
    # A binary32 input is rounded once by torch's fp32 -> bf16 cast, so the two agree.
    rng = np.random.default_rng(1234)
    mant = rng.integers(0, 1 << 23, size=200_000, dtype=np.uint32)
    expo = rng.integers(0, 255, size=200_000, dtype=np.uint32)  # includes subnormals (0)
    sign = rng.integers(0, 2, size=200_000, dtype=np.uint32)
    x32 = ((sign << 31) | (expo << 23) | mant).view(np.float32)
    ours = oracle.f64_to_bf16(x32.astype(np.float64))
    ref = torch.from_numpy(x32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_bf16_encode_is_nearest_with_ties_to_even():
    # Brute-force property: the result is at least as close as both neighbours,
    # and on an exact tie it has an even significand.
    rng = np.random.default_rng(99)
    x = np.concatenate([
        rng.standard_normal(50_000) * 0.02,
        rng.standard_normal(20_000) * 1e30,
        rng.standard_normal(20_000) * 1e-39,           # bf16 subnormal range
        (1.0 + rng.integers(0, 256, 10_000) / 256.0) * 2.0 ** rng.integers(-20, 20, 10_000),
    ])
    enc = oracle.f64_to_bf16(x)
    dec = oracle.bf16_to_f64(enc)
    finite = np.isfinite(dec)
    x, enc, dec = x[finite], enc[finite], dec[finite]
    mag = enc & 0x7FFF
    up = oracle.bf16_to_f64((enc & 0x8000) | np.minimum(mag + 1, 0x7F80).astype(np.uint16))
    dn = oracle.bf16_to_f64((enc & 0x8000) | np.maximum(mag.astype(np.int32) - 1, 0).astype(np.uint16))
    err = np.abs(x - dec)
    assert np.all(err <= np.abs(x - up))
    assert np.all(err <= np.abs(x - dn))
    tie = (err == np.abs(x - up)) | ((err == np.abs(x - dn)) & (mag > 0))
    assert np.all((enc[tie] & 1) == 0)


def test_bf16_encode_special_values_match_torch():
    # Infinities and signed zeros bit for bit against torch's binary32 -> bf16
    # cast; every NaN (any sign or payload) to a NaN, whose payload neither
    # side fixes (torch gives 0xffff here).  Plus fp64 values beyond binary32's
    # range, which overflow to infinity or flush to a signed zero.
    special = np.array([0x7F800000, 0xFF800000, 0x00000000, 0x80000000, 0x7FC00000, 0xFFC00000,
                        0x7F800001, 0xFF812345, 0x7FFFFFFF], dtype=np.uint32).view(np.float32)
    ours = oracle.f64_to_bf16(special.astype(np.float64))
    ref = torch.from_numpy(special).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(special)

    def is_nan_bits(b):
        return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)
    assert np.all(is_nan_bits(ours[nan])) and np.all(is_nan_bits(ref[nan]))
    assert np.array_equal(ours[~nan], ref[~nan])
    big = np.array([1e300, -1e300, 2.0 ** 128, -(2.0 ** 129), 1e-300, -1e-300])
    assert [hex(v) for v in oracle.f64_to_bf16(big)] == ["0x7f80", "0xff80", "0x7f80", "0xff80",
                                                        "0x0", "0x8000"]


# ---------------------------------------------------------------- symm_at

def test_symm_at_golden(golden):
    fx = golden("symm_at.json")
    base = fx["heap_base"]
    for c in fx["cases"]:
        assert oracle.symm_at(c["ptr"], base[c["self"]], base[c["pe"]]) == c["expect"], c


# ---------------------------------------------------------------- GEMM

def _bf16_ints(shape, rng, lo=-8, hi=8):
    v = rng.integers(lo, hi + 1, size=shape).astype(np.float32)
    return torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16), v


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (3, 5, 7), (17, 9, 33), (48, 47, 45)])
def test_gemm_exact_against_integer_brute_force(M, N, K):
    rng = np.random.default_rng(M * 1000 + N * 10 + K)
    A, Av = _bf16_ints((M, K), rng)
    B, Bv = _bf16_ints((K, N), rng)
    C = oracle.gemm_f64(A, B)
    Ai = Av.astype(np.int64).tolist()
    Bi = Bv.astype(np.int64).tolist()
    for i in range(M):
        for j in range(N):
            assert C[i, j] == sum(Ai[i][k] * Bi[k][j] for k in range(K))


def test_gemm_closed_forms():
    rng = np.random.default_rng(5)
    K = 40
    A = inputs.draw_bf16((24, K), 3, 1, 0, "normal", 1.0)
    eye = np.where(np.eye(K, dtype=bool), np.uint16(0x3F80), np.uint16(0)).astype(np.uint16)
    assert np.array_equal(oracle.gemm_f64(A, eye), oracle.bf16_to_f64(A))   # B = I gives A
    ones_a = np.full((5, 37), 0x3F80, dtype=np.uint16)
    ones_b = np.full((37, 6), 0x3F80, dtype=np.uint16)
    assert np.all(oracle.gemm_f64(ones_a, ones_b) == 37.0)                  # all-ones gives K
    B = inputs.draw_bf16((K, 19), 3, 2, 0, "normal", 1.0)
    onehot = np.zeros((K, K), dtype=np.uint16)
    perm = rng.permutation(K)
    onehot[np.arange(K), perm] = 0x3F80
    assert np.array_equal(oracle.gemm_f64(onehot, B), oracle.bf16_to_f64(B)[perm])  # row pick


def test_gemm_matches_numpy_within_fp64_bound():
    A = inputs.draw_bf16((64, 300), 7, 1, 0, "normal", 0.02)
    B = inputs.draw_bf16((300, 96), 7, 2, 0, "normal", 0.02)
    Ad, Bd = oracle.bf16_to_f64(A), oracle.bf16_to_f64(B)
    C = oracle.gemm_f64(A, B)
    ref = Ad @ Bd
    bound = 300 * 2.0 ** -52 * (np.abs(Ad) @ np.abs(Bd))
    assert np.all(np.abs(C - ref) <= bound)


# ---------------------------------------------------------------- AllGather / AG-GEMM

def _small_ag(R=3, M_r=16, K=24, N=20, order=(2, 0, 1), seed=11):
    cfg = dict(R=R, M_r=M_r, K=K, N=N, dist="normal", scale=0.5)
    return inputs.ag_inputs(cfg, seed=seed, slot_order=list(order))


def test_allgather_is_row_concatenation_through_rank_table():
    d = _small_ag()
    R, M_r, K = d["R"], d["M_r"], d["K"]
    shards = [inputs.draw_bf16((M_r, K), 11, inputs.TENSOR_A, r, "normal", 0.5) for r in range(R)]
    G = oracle.allgather(d["heap"], d["rank_off"], R, d["a_off"], M_r, K)
    assert np.array_equal(G, np.concatenate(shards, axis=0))
    # The table is honoured: a permuted table moves the shards.
    assert list(d["rank_off"]) != sorted(d["rank_off"])


def test_ag_gemm_worked_example(golden):
    ex = golden("worked_examples.json")["ag_gemm"]
    R, M_r, K = 2, 1, 2
    to_bits = lambda a: torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    heap = np.zeros(R * 64, dtype=np.uint8)
    rank_off = np.array([64, 0], dtype=np.int64)   # rank 0's slice placed second
    for r in range(R):
        heap[rank_off[r]:rank_off[r] + 4] = to_bits(ex["A"][r]).view(np.uint8).reshape(-1)
    G, C = oracle.ag_gemm(heap, rank_off, R, 0, M_r, 3, K, to_bits(ex["B"]))
    assert np.array_equal(oracle.bf16_to_f64(G), np.array(ex["G"], dtype=np.float64))
    assert np.array_equal(C, np.array(ex["C"], dtype=np.float64))


def test_ag_gemm_matches_numpy_on_concatenation_and_rows_agree():
    d = _small_ag()
    R, M_r, K, N = d["R"], d["M_r"], d["K"], d["N"]
    G, C = oracle.ag_gemm(d["heap"], d["rank_off"], R, d["a_off"], M_r, N, K, d["B"])
    Gd, Bd = oracle.bf16_to_f64(G), oracle.bf16_to_f64(d["B"])
    assert np.all(np.abs(C - Gd @ Bd) <= K * 2.0 ** -52 * (np.abs(Gd) @ np.abs(Bd)))
    rows = [0, 5, M_r, 2 * M_r + 3, R * M_r - 1]
    assert np.array_equal(oracle.ag_gemm_rows(d["heap"], d["rank_off"], R, d["a_off"], M_r, N, K,
                                              d["B"], rows), C[rows])


def test_ag_gemm_single_rank_is_plain_gemm():
    d = _small_ag(R=1, order=(0,))
    G, C = oracle.ag_gemm(d["heap"], d["rank_off"], 1, d["a_off"], d["M_r"], d["N"], d["K"], d["B"])
    A0 = inputs.draw_bf16((d["M_r"], d["K"]), 11, inputs.TENSOR_A, 0, "normal", 0.5)
    assert np.array_equal(G, A0)
    assert np.array_equal(C, oracle.gemm_f64(A0, d["B"]))


# ---------------------------------------------------------------- GEMM-RS

def _small_rs(R=3, M=24, K_r=10, N=18, order=(1, 2, 0), seed=21):
    cfg = dict(R=R, M=M, K_r=K_r, N=N, dist="normal", scale=0.5)
    return inputs.rs_inputs(cfg, seed=seed, slot_order=list(order))


def _rs_operands(d, seed=21):
    A = [inputs.draw_bf16((d["M"], d["K_r"]), seed, inputs.TENSOR_A, r, "normal", 0.5) for r in range(d["R"])]
    B = [inputs.draw_bf16((d["K_r"], d["N"]), seed, inputs.TENSOR_B, r, "normal", 0.5) for r in range(d["R"])]
    return A, B


def test_gemm_rs_worked_example(golden):
    ex = golden("worked_examples.json")["gemm_rs"]
    to_bits = lambda a: torch.tensor(a, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    R, M, K_r, N = 2, 2, 1, 2
    a_off, b_off, out_off, sl = 0, 16, 32, 64
    rank_off = np.array([sl, 0], dtype=np.int64)
    heap = np.zeros(R * sl, dtype=np.uint8)
    for r in range(R):
        o = rank_off[r]
        heap[o + a_off:o + a_off + 4] = to_bits(ex["A"][r]).view(np.uint8).reshape(-1)
        heap[o + b_off:o + b_off + 4] = to_bits(ex["B"][r]).view(np.uint8).reshape(-1)
    S, heap_out = oracle.gemm_rs(heap, rank_off, R, a_off, b_off, out_off, M, N, K_r)
    assert np.array_equal(S, np.array(ex["S"], dtype=np.float64))
    for j in range(R):
        o = rank_off[j] + out_off
        got = oracle.bf16_to_f64(heap_out[o:o + 4].view(np.uint16)).reshape(1, 2)
        assert np.array_equal(got, np.array(ex["out"][j], dtype=np.float64))


def test_gemm_rs_equals_concat_k_gemm():
    # sum_r A_r B_r = [A_0 ... A_{R-1}] [B_0; ...; B_{R-1}]  (block matrix identity)
    d = _small_rs()
    A, B = _rs_operands(d)
    S, _ = oracle.gemm_rs(d["heap"], d["rank_off"], d["R"], d["a_off"], d["b_off"], d["out_off"],
                          d["M"], d["N"], d["K_r"])
    Ac = oracle.bf16_to_f64(np.concatenate(A, axis=1))
    Bc = oracle.bf16_to_f64(np.concatenate(B, axis=0))
    Kt = d["R"] * d["K_r"]
    assert np.all(np.abs(S - Ac @ Bc) <= 2 * Kt * 2.0 ** -52 * (np.abs(Ac) @ np.abs(Bc)))


def test_gemm_rs_sum_then_scatter_equals_scatter_of_sums():
    d = _small_rs()
    R, M, N = d["R"], d["M"], d["N"]
    S, heap_out = oracle.gemm_rs(d["heap"], d["rank_off"], R, d["a_off"], d["b_off"], d["out_off"],
                                 M, N, d["K_r"])
    Mb = M // R
    for j in range(R):
        # scatter first: rank j's rows, reduced on their own
        rows = np.arange(j * Mb, (j + 1) * Mb)
        Sj = oracle.gemm_rs_rows(d["heap"], d["rank_off"], R, d["a_off"], d["b_off"], M, N,
                                 d["K_r"], rows)
        assert np.array_equal(Sj, S[rows])
        o = int(d["rank_off"][j]) + d["out_off"]
        out_j = heap_out[o:o + Mb * N * 2].view(np.uint16).reshape(Mb, N)
        assert np.array_equal(out_j, oracle.f64_to_bf16(Sj))


def test_gemm_rs_single_rank_is_plain_gemm():
    d = _small_rs(R=1, M=8, order=(0,))
    A, B = _rs_operands(d)
    S, _ = oracle.gemm_rs(d["heap"], d["rank_off"], 1, d["a_off"], d["b_off"], d["out_off"],
                          d["M"], d["N"], d["K_r"])
    assert np.array_equal(S, oracle.gemm_f64(A[0], B[0]))


def test_gemm_rs_fp32_variant_within_fp32_bound():
    d = _small_rs()
    A, B = _rs_operands(d)
    rows = np.arange(d["M"])
    S64 = oracle.gemm_rs_rows(d["heap"], d["rank_off"], d["R"], d["a_off"], d["b_off"], d["M"],
                              d["N"], d["K_r"], rows)
    S32 = oracle.gemm_rs_rows_f32(d["heap"], d["rank_off"], d["R"], d["a_off"], d["b_off"],
                                  d["M"], d["N"], d["K_r"], rows)
    absP = sum(np.abs(oracle.bf16_to_f64(A[r])) @ np.abs(oracle.bf16_to_f64(B[r])) for r in range(d["R"]))
    assert np.all(np.abs(S32 - S64) <= (2 * d["R"] + 1) * 2.0 ** -24 * absP + 1e-30)
    # one rank: just the partial rounded to binary32
    S1 = oracle.gemm_rs_rows_f32(d["heap"], d["rank_off"], 1, d["a_off"], d["b_off"], d["M"],
                                 d["N"], d["K_r"], rows)
    assert np.array_equal(S1, oracle.gemm_f64(A[0], B[0]).astype(np.float32))


# ---------------------------------------------------------------- flags and schedule

def test_expected_flags_set_semantics():
    f = oracle.expected_flags(7, 13)
    assert f.dtype == np.int64 and np.all(f == 13)


def test_row_counters_against_simulated_adds():
    # Brute force: replay every launch's per-k-tile ADD of 1 on zeroed counters.
    for n_rows, T_k, epochs in [(1, 1, 1), (3, 4, 2), (8, 32, 5), (2, 2, 20)]:
        counters = [0] * n_rows
        for e in range(1, epochs + 1):
            for row in range(n_rows):
                for _ in range(T_k):
                    counters[row] += 1
            assert list(oracle.expected_row_counters(n_rows, e, T_k)) == counters


def test_swizzle_golden(golden):
    fx = golden("swizzle.json")
    pf = fx["page_formula"]
    for rank, row in enumerate(pf["by_rank"]):
        got = [oracle.swizzle_row(p, rank, pf["tiles_per_pe"], pf["total_tiles"])
               for p in range(pf["total_tiles"])]
        assert got == row, rank
    for case in fx["consumer_orders"]:
        for c, want in enumerate(case["orders"]):
            got = oracle.consumer_order(case["T_M"], case["T_N"], case["G"], c,
                                        case["group_rows"], case["rank"], case["tiles_per_pe"],
                                        case.get("visit"))
            assert list(got) == want, (case["note"], c)


@pytest.mark.parametrize("T_M,T_N,G,GM,rank,tpp", [(32, 16, 76, 1, 0, 4), (64, 14, 76, 1, 3, 8),
                                                   (128, 32, 76, 8, 5, 16), (9, 3, 4, 8, 1, 1),
                                                   (16, 3, 7, 2, 3, 4), (8, 1, 3, 1, 7, 1)])
def test_consumer_order_is_a_partition_starting_at_own_rows(T_M, T_N, G, GM, rank, tpp):
    orders = [oracle.consumer_order(T_M, T_N, G, c, GM, rank, tpp) for c in range(G)]
    seen = np.concatenate(orders)
    assert sorted(seen.tolist()) == list(range(T_M * T_N))           # every tile exactly once
    assert max(len(o) for o in orders) == -(-T_M * T_N // G)          # balanced
    # consumer 0 starts on the PE's own first row, column 0
    assert orders[0][0] == ((rank * tpp) % T_M) * T_N
    # undoing the rename gives rows that never go backwards, group by group
    for o in orders:
        rows = [((q // T_N) - rank * tpp) % T_M for q in o]
        assert [r // GM for r in rows] == sorted(r // GM for r in rows)
    # the whole order (position p is consumer p mod G's (p div G)-th tile):
    # inside a row group the columns never go backwards in even groups and
    # never forwards in odd ones
    full = [orders[pos % G][pos // G] for pos in range(T_M * T_N)]
    for pos0 in range(0, T_M * T_N, GM * T_N):
        g = pos0 // (GM * T_N)
        cols = [q % T_N for q in full[pos0:pos0 + GM * T_N]]
        assert cols == (sorted(cols) if g % 2 == 0 else sorted(cols, reverse=True))
    # the rank visit order of a ring (own rank, then rank+1, rank+2, ...) is
    # the page's formula, whenever the row tiles split evenly over the ranks
    if T_M % tpp == 0:
        R = T_M // tpp
        ring = [(rank + k) % R for k in range(R)]
        for c in range(G):
            assert list(oracle.consumer_order(T_M, T_N, G, c, GM, rank, tpp, ring)) == \
                list(orders[c])


# ---------------------------------------------------------------- ring AllReduce

def _ring_heap(xs, pad=64):
    R, n = len(xs), len(xs[0])
    sl = ((2 * n * 4 + pad - 1) // pad) * pad
    heap = np.zeros(R * sl, dtype=np.uint8)
    rank_off = np.array([((r + 1) % R) * sl for r in range(R)], dtype=np.int64)  # permuted table
    for r in range(R):
        heap[rank_off[r]:rank_off[r] + n * 4] = np.asarray(xs[r], dtype=np.float32).view(np.uint8)
    return heap, rank_off, n * 4   # data at 0, out at n*4


def _ring_out(heap_out, rank_off, R, out_off, n):
    return [heap_out[rank_off[j] + out_off:rank_off[j] + out_off + n * 4].view(np.float32) for j in range(R)]


def test_ring_allreduce_worked_examples(golden):
    ex = golden("worked_examples.json")["ring_allreduce"]
    for case in (ex, ex["fp32_order_case"]):
        xs = case["x"]
        R, n = len(xs), len(xs[0])
        heap, ro, out_off = _ring_heap(xs)
        outs = _ring_out(oracle.ring_allreduce(heap, ro, R, 0, out_off, n), ro, R, out_off, n)
        for o in outs:
            assert np.array_equal(o, np.array(case["sum"], dtype=np.float32))


def test_ring_allreduce_exact_on_integers_and_identical_on_every_rank():
    rng = np.random.default_rng(3)
    for R in (1, 2, 3, 8):
        n = R * 12
        xs = [rng.integers(-1000, 1000, n).astype(np.float32) for _ in range(R)]
        heap, ro, out_off = _ring_heap(xs)
        outs = _ring_out(oracle.ring_allreduce(heap, ro, R, 0, out_off, n), ro, R, out_off, n)
        exact = np.sum(np.stack(xs).astype(np.int64), axis=0)
        for o in outs:
            assert np.array_equal(o.astype(np.int64), exact)


def test_ring_allreduce_within_binary32_bound():
    rng = np.random.default_rng(4)
    R, n = 8, 8 * 256
    xs = [rng.standard_normal(n).astype(np.float32) for _ in range(R)]
    heap, ro, out_off = _ring_heap(xs)
    out = _ring_out(oracle.ring_allreduce(heap, ro, R, 0, out_off, n), ro, R, out_off, n)[0]
    X = np.stack(xs).astype(np.float64)
    assert np.all(np.abs(out - X.sum(0)) <= R * 2.0 ** -24 * np.abs(X).sum(0))


# ---------------------------------------------------------------- all-to-all

def _a2a_heap(sends, B, pad=64):
    R = len(sends)
    sl = ((2 * R * B + pad - 1) // pad) * pad
    heap = np.zeros(R * sl, dtype=np.uint8)
    rank_off = np.array([((r + 2) % R) * sl for r in range(R)], dtype=np.int64)  # permuted
    for r in range(R):
        heap[rank_off[r]:rank_off[r] + R * B] = np.asarray(sends[r], dtype=np.uint8).reshape(-1)
    return heap, rank_off, R * B   # send at 0, recv at R*B


def test_alltoall_worked_example(golden):
    ex = golden("worked_examples.json")["alltoall"]
    R, B = 3, 1
    heap, ro, recv_off = _a2a_heap(ex["send"], B)
    out = oracle.alltoall(heap, ro, R, 0, recv_off, B)
    for j in range(R):
        got = out[ro[j] + recv_off:ro[j] + recv_off + R * B]
        assert list(got) == ex["recv"][j]


def test_alltoall_is_an_involution_and_a_permutation_of_bytes():
    rng = np.random.default_rng(8)
    for R, B in [(1, 16), (2, 48), (5, 32), (8, 64)]:
        sends = [rng.integers(0, 256, R * B, dtype=np.uint8) for _ in range(R)]
        heap, ro, recv_off = _a2a_heap(sends, B)
        once = oracle.alltoall(heap, ro, R, 0, recv_off, B)
        recvs = [once[ro[j] + recv_off:ro[j] + recv_off + R * B].copy() for j in range(R)]
        # every input byte appears exactly once
        assert sorted(np.concatenate(recvs).tolist()) == sorted(np.concatenate(sends).tolist())
        # applying it again to the receive buffers gives back the send buffers
        heap2, ro2, recv_off2 = _a2a_heap(recvs, B)
        twice = oracle.alltoall(heap2, ro2, R, 0, recv_off2, B)
        for j in range(R):
            assert np.array_equal(twice[ro2[j] + recv_off2:ro2[j] + recv_off2 + R * B], sends[j])
