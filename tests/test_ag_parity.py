"""AllGather -> GEMM on the GPU against the CPU oracle, through the C ABI.

Bit-exact: the gathered buffer G, every flag (== epoch) and the identity /
all-ones special cases.  Floating point C: rel-Frobenius <= 1e-3 and
per-element <= 1e-2 * max|C_ref| against the oracle's fp64 result rounded to
bf16.  Sizes span several tiles and ragged edges; the tensor-parallel
configuration is checked on sampled rows.
"""
import numpy as np
import pytest
import torch

import oracle
from overlap_producer_warps_gb300 import inputs
from tests.helpers import AgProblem, assert_gemm_close, host_bits, quarter_rows, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def api():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    from overlap_producer_warps_gb300 import api as _api
    _api.lib()
    return _api


def _cfg(R, M_r, K, N, dist="normal", scale=0.5):
    return dict(R=R, M_r=M_r, K=K, N=N, dist=dist, scale=scale)


def _run_and_check(api, d, epoch_runs=1, opts_fn=None, full=True):
    prob = AgProblem(d)
    F = api.ag_num_flags(prob.R, prob.M_r, prob.K)
    sig = api.Signal(F)
    for i in range(epoch_runs):
        e = sig.next_epoch()
        prob.run(api, sig, e, opts_fn(i) if opts_fn else None)
        st = sig.status()
        assert st[0] == api.OK, st
        flags = sig.flags().cpu().numpy()
        assert np.array_equal(flags, oracle.expected_flags(F, e)), f"flags after epoch {e}"
    G_ref, C_ref = prob.oracle_full() if full else (None, None)
    if full:
        assert np.array_equal(host_bits(prob.G), G_ref), "gathered buffer differs"
        assert_gemm_close(host_bits(prob.C), C_ref)
    sig.close()
    return prob


def test_tiny_config(api):
    """R=2, 64x128 shards, B 128x128, 64x64 flag tiles, uniform[-1,1] seed 0, epoch 1."""
    cfg = inputs.CONFIGS["ag_tiny"]
    d = inputs.ag_inputs(cfg, seed=0)
    assert api.ag_flag_tile(cfg["M_r"], cfg["K"]) == cfg["flag_tile"]
    assert api.ag_num_flags(cfg["R"], cfg["M_r"], cfg["K"]) == 4
    _run_and_check(api, d)


def test_identity_b_is_bit_exact_gather(api):
    # B = I makes C = bf16(G) exactly: pins the A operand path bit for bit.
    R, M_r, K = 2, 128, 256
    d = inputs.ag_inputs(_cfg(R, M_r, K, K), seed=3)
    d["B"] = np.where(np.eye(K, dtype=bool), np.uint16(0x3F80), np.uint16(0)).astype(np.uint16)
    prob = AgProblem(d)
    sig = api.Signal(api.ag_num_flags(R, M_r, K))
    prob.run(api, sig, sig.next_epoch())
    assert sig.status()[0] == api.OK
    G = host_bits(prob.G)
    assert np.array_equal(host_bits(prob.C), G)
    assert np.array_equal(G, oracle.allgather(d["heap"], d["rank_off"], R, d["a_off"], M_r, K))


def test_one_hot_a_picks_rows_of_b(api):
    # A one-hot (row i selects row perm[i] of B) pins the B operand layout.
    R, M_r, K, N = 2, 128, 256, 512
    d = inputs.ag_inputs(_cfg(R, M_r, K, N), seed=4)
    rng = np.random.default_rng(4)
    for r in range(R):
        A = np.zeros((M_r, K), dtype=np.uint16)
        A[np.arange(M_r), rng.integers(0, K, M_r)] = 0x3F80
        o = int(d["rank_off"][r])
        d["heap"][o:o + A.nbytes] = A.view(np.uint8).reshape(-1)
    prob = AgProblem(d)
    sig = api.Signal(api.ag_num_flags(R, M_r, K))
    prob.run(api, sig, sig.next_epoch())
    assert sig.status()[0] == api.OK
    G = oracle.allgather(d["heap"], d["rank_off"], R, d["a_off"], M_r, K)
    picks = np.argmax(G, axis=1)
    assert np.array_equal(host_bits(prob.C), d["B"][picks])


def test_all_ones_gives_k(api):
    R, M_r, K, N = 2, 128, 384, 256
    d = inputs.ag_inputs(_cfg(R, M_r, K, N), seed=5)
    for r in range(R):
        o = int(d["rank_off"][r])
        d["heap"][o:o + M_r * K * 2] = np.full(M_r * K, 0x3F80, dtype=np.uint16).view(np.uint8)
    d["B"] = np.full((K, N), 0x3F80, dtype=np.uint16)
    prob = AgProblem(d)
    sig = api.Signal(api.ag_num_flags(R, M_r, K))
    prob.run(api, sig, sig.next_epoch())
    assert sig.status()[0] == api.OK
    assert np.all(oracle.bf16_to_f64(host_bits(prob.C)) == float(K))


@pytest.mark.parametrize("R,M_r,K,N,order", [
    (3, 64, 192, 200, (2, 0, 1)),      # flag tile 64, GEMM tiles straddle ranks, ragged N
    (4, 256, 512, 776, (1, 3, 0, 2)),  # flag tile 128, ragged N, permuted rank table
    (1, 128, 128, 8, None),            # single rank, narrowest N
    (8, 128, 1024, 512, None),         # eight ranks, several k-blocks per flag
    (5, 192, 320, 264, (4, 3, 2, 1, 0)),  # ragged M (960 rows) and N
])
def test_shapes(api, R, M_r, K, N, order):
    d = inputs.ag_inputs(_cfg(R, M_r, K, N), seed=R * 7 + K, slot_order=order)
    _run_and_check(api, d)


@pytest.mark.parametrize("R,M_r,K,N", [
    (2, 256, 256, 512),     # one 512-wide tile column
    (4, 256, 512, 776),     # ragged N: the second wide column holds 264 columns
    (3, 64, 192, 200),      # flag tile 64, N narrower than one wide tile
    (5, 192, 320, 1032),    # ragged M (960 rows) and N (3 wide columns)
    (8, 128, 1024, 1024),   # eight ranks, several k-blocks per flag
])
def test_wide_pair_tiles_match_oracle_and_narrow_tiles(api, R, M_r, K, N):
    """256 x 512 pair tiles (two N = 256 MMAs per k step into one 512-column
    accumulator) against the oracle, and bit for bit against 256 x 256 tiles:
    every output element sums the same products in the same order."""
    d = inputs.ag_inputs(_cfg(R, M_r, K, N), seed=R * 11 + N)
    wide = _run_and_check(api, d, epoch_runs=2, opts_fn=lambda i: api.make_opts(tile_n=512))
    narrow = _run_and_check(api, d, full=False, opts_fn=lambda i: api.make_opts(tile_n=256))
    assert np.array_equal(host_bits(wide.G), host_bits(narrow.G))
    assert np.array_equal(host_bits(wide.C), host_bits(narrow.C))


def test_wide_tiles_many_per_pair(api):
    """Two CTA pairs take 16 wide tiles each, so the one TMEM accumulator is
    handed between MMA and epilogue many times per launch, over 3 epochs."""
    d = inputs.ag_inputs(_cfg(4, 512, 512, 2048), seed=77)
    p1 = _run_and_check(api, d, epoch_runs=3,
                        opts_fn=lambda i: api.make_opts(tile_n=512, num_ctas=4))
    p2 = _run_and_check(api, d, full=False,
                        opts_fn=lambda i: api.make_opts(tile_n=512, num_ctas=4,
                                                        schedule=api.SCHED_SWIZZLE))
    assert np.array_equal(host_bits(p1.C), host_bits(p2.C))


@pytest.mark.parametrize("mode", ["serial", "checked", "swizzle", "no_local", "row_add", "skew"])
def test_wide_tiles_in_every_mode(api, mode):
    """256 x 512 pair tiles under each synchronisation, signal and schedule
    option, over 2 epochs: G bit for bit and C against the oracle, the flags
    (or row counters) at their epoch values, and C bit for bit against the
    same option on 256 x 256 tiles."""
    R, M_r, K, N = 4, 256, 384, 1288
    d = inputs.ag_inputs(_cfg(R, M_r, K, N), seed=80 + len(mode))
    kw = {"serial": dict(sync_mode=api.SYNC_SERIAL), "checked": dict(sync_mode=api.SYNC_CHECKED),
          "swizzle": dict(schedule=api.SCHED_SWIZZLE), "no_local": dict(local_rank=-1),
          "row_add": dict(signal_mode=api.SIGNAL_ROW_ADD),
          "skew": dict(publish_perm=(2, 0, 3, 1), delay_ns=(0, 20000, 5000, 0))}[mode]
    ft = api.ag_flag_tile(M_r, K)
    row_add = mode == "row_add"
    n_slots = api.ag_num_row_counters(R, M_r, K) if row_add else api.ag_num_flags(R, M_r, K)
    out = {}
    for tile_n in (512, 256):
        prob = AgProblem(d)
        sig = api.Signal(n_slots)
        opts = api.make_opts(tile_n=tile_n, num_ctas=6, **kw)
        for _ in range(2):
            e = sig.next_epoch()
            prob.run(api, sig, e, opts)
            assert sig.status()[0] == api.OK, (mode, tile_n)
            want = (oracle.expected_row_counters(n_slots, e, K // ft) if row_add
                    else oracle.expected_flags(n_slots, e))
            assert np.array_equal(sig.flags().cpu().numpy(), want), (mode, tile_n, e)
        sig.close()
        out[tile_n] = prob
    G_ref, C_ref = out[512].oracle_full()
    assert np.array_equal(host_bits(out[512].G), G_ref)
    assert_gemm_close(host_bits(out[512].C), C_ref, what=f"{mode}: C")
    assert np.array_equal(host_bits(out[512].C), host_bits(out[256].C))


def test_tile_width_choice(api):
    """The library's width for the benchmark layers on the full grid follows
    its documented rule: 512 when whole waves of wide tiles, at 1.93 times a
    256-wide wave, take less time than the 256-wide waves."""
    pairs = torch.cuda.get_device_properties(0).multi_processor_count // 2
    for name in ("ag_tp", "ag_mlp", "ag_skew"):
        c = inputs.CONFIGS[name]
        M, N = c["R"] * c["M_r"], c["N"]
        tm = (M + 255) // 256
        w1 = -(-tm * (-(-N // 256)) // pairs)
        w2 = -(-tm * (-(-N // 512)) // pairs)
        want = 512 if w2 * 193 < w1 * 100 else 256
        assert api.ag_tile_n(c["R"], c["M_r"], N) == want, name
        assert api.ag_tile_n(c["R"], c["M_r"], N, api.make_opts(tile_n=256)) == 256
    if pairs == 76:   # a full GB300: TP stays 256 wide, MLP and skew go wide
        assert [api.ag_tile_n(inputs.CONFIGS[n]["R"], inputs.CONFIGS[n]["M_r"],
                              inputs.CONFIGS[n]["N"]) for n in ("ag_tp", "ag_mlp", "ag_skew")] == \
            [256, 512, 512]


def test_epochs_reused_without_reset(api):
    """20 launches on one signal object: flags == e after each (TP-style epochs 1..20)."""
    d = inputs.ag_inputs(_cfg(4, 128, 256, 512), seed=9)
    _run_and_check(api, d, epoch_runs=20)


def test_serial_mode_matches_overlap_bit_for_bit(api):
    d = inputs.ag_inputs(_cfg(4, 256, 512, 512), seed=10)
    p1 = _run_and_check(api, d)
    p2 = _run_and_check(api, d, opts_fn=lambda i: api.make_opts(sync_mode=api.SYNC_SERIAL))
    assert np.array_equal(host_bits(p1.C), host_bits(p2.C))


def test_ready_schedule_matches_swizzle_bit_for_bit(api):
    d = inputs.ag_inputs(_cfg(4, 256, 512, 768), seed=11)
    p1 = _run_and_check(api, d, opts_fn=lambda i: api.make_opts(schedule=api.SCHED_SWIZZLE))
    p2 = _run_and_check(api, d, epoch_runs=3,
                        opts_fn=lambda i: api.make_opts(schedule=api.SCHED_READY))
    assert np.array_equal(host_bits(p1.C), host_bits(p2.C))


def test_producer_then_consumer_roles(api):
    d = inputs.ag_inputs(_cfg(4, 128, 384, 512), seed=12)
    prob = AgProblem(d)
    F = api.ag_num_flags(4, 128, 384)
    sig = api.Signal(F)
    e = sig.next_epoch()
    prob.run(api, sig, e, api.make_opts(role=api.ROLE_PRODUCER))
    assert sig.status()[0] == api.OK
    assert np.all(sig.flags().cpu().numpy() == e)
    assert sig.next_epoch() == e + 1
    prob.run(api, sig, e, api.make_opts(role=api.ROLE_CONSUMER))
    assert sig.status()[0] == api.OK
    G_ref, C_ref = prob.oracle_full()
    assert np.array_equal(host_bits(prob.G), G_ref)
    assert_gemm_close(host_bits(prob.C), C_ref)


def test_fewer_ctas_than_sms(api):
    d = inputs.ag_inputs(_cfg(2, 256, 256, 512), seed=13)
    _run_and_check(api, d, opts_fn=lambda i: api.make_opts(num_ctas=5))


def test_one_pair_claims_every_tile(api):
    """num_ctas=2: a single CTA pair claims all 32 pair tiles from the ready
    counter while every CTA's producer warp (two of them) gathers."""
    d = inputs.ag_inputs(_cfg(4, 512, 256, 1024), seed=16)
    _run_and_check(api, d, epoch_runs=2, opts_fn=lambda i: api.make_opts(num_ctas=2))


def test_grouped_ready_order_with_ragged_group(api):
    """K*N*2 > 64 MiB switches the ready order to groups of 8 pair rows with
    the column index outermost; 9 pair rows leave a ragged last group of 1."""
    R, M_r, K, N = 3, 768, 8192, 4224            # M = 2304 rows = 9 pair rows
    assert K * N * 2 > 64 << 20
    d = inputs.ag_inputs(_cfg(R, M_r, K, N), seed=17)
    prob = AgProblem(d)
    sig = api.Signal(api.ag_num_flags(R, M_r, K))
    for _ in range(2):
        prob.run(api, sig, sig.next_epoch())
        assert sig.status()[0] == api.OK
    G = host_bits(prob.G)
    assert np.array_equal(G, oracle.allgather(d["heap"], d["rank_off"], R, d["a_off"], M_r, K))
    rows = sample_rows(prob.M, 128, 1, seed=5)
    C = host_bits(prob.C)
    assert_gemm_close(C[rows], prob.oracle_rows(rows), what="grouped order C")


@pytest.mark.parametrize("R,M_r,K,N", [(4, 512, 512, 768), (3, 192, 320, 264)])
def test_local_rank_choice_does_not_change_results(api, R, M_r, K, N):
    """Reading the local rank's shard in place (and taking its tiles first) or
    waiting on every rank's flags computes the same G, C and flags bit for bit."""
    d = inputs.ag_inputs(_cfg(R, M_r, K, N), seed=18 + R)
    outs = []
    for local in (-1, 0, R - 1):
        prob = _run_and_check(api, d, epoch_runs=2, full=(local == -1),
                              opts_fn=lambda i, local=local: api.make_opts(local_rank=local))
        outs.append((host_bits(prob.G), host_bits(prob.C)))
    for G, C in outs[1:]:
        assert np.array_equal(G, outs[0][0]) and np.array_equal(C, outs[0][1])


def _trace_views(api, prob, trace, grid, tile_n):
    F = api.ag_num_flags(prob.R, prob.M_r, prob.K)
    T = ((prob.M + 255) // 256) * ((prob.N + tile_n - 1) // tile_n)  # 256 x tile_n pair tiles
    t = trace.cpu().numpy().view(np.uint64)
    return dict(publish=t[:F], consume=t[F:2 * F], tile=t[2 * F:2 * F + T],
                tile_start=t[2 * F + T:2 * F + 2 * T], cta_start=t[2 * F + 2 * T:2 * F + 2 * T + grid],
                F=F, T=T)


@pytest.mark.parametrize("local,perm,tile_n", [(2, None, 256), (0, None, 256),
                                               (1, (3, 0, 2, 1), 256), (2, None, 512),
                                               (1, (3, 0, 2, 1), 512)])
def test_trace_publish_before_consume_and_swizzle_order(api, local, perm, tile_n):
    R, M_r, K, N = 4, 256, 512, 1024
    d = inputs.ag_inputs(_cfg(R, M_r, K, N), seed=14)
    prob = AgProblem(d)
    sig = api.Signal(api.ag_num_flags(R, M_r, K))
    words = api.ag_trace_words(R, M_r, N, K)
    trace = torch.full((words,), -1, dtype=torch.int64, device="cuda")
    grid = 6
    opts = api.make_opts(trace=trace, num_ctas=grid, local_rank=local, publish_perm=perm,
                         schedule=api.SCHED_SWIZZLE, tile_n=tile_n)
    assert api.ag_tile_n(R, M_r, N, opts) == tile_n
    prob.run(api, sig, sig.next_epoch(), opts)
    assert sig.status()[0] == api.OK
    v = _trace_views(api, prob, trace, grid, tile_n)
    # every tile published; every tile of another rank acquired no earlier than
    # its publish; the local rank's own tiles (read in place) never acquired
    per_rank = v["F"] // R
    remote = (np.arange(v["F"]) // per_rank) != local
    assert np.all(v["publish"] > 0)
    assert np.all(v["consume"][remote] != np.uint64(2 ** 64 - 1))
    assert np.all(v["publish"][remote] <= v["consume"][remote])
    assert np.all(v["consume"][~remote] == np.uint64(2 ** 64 - 1))
    # each consumer (a CTA pair) visited its 256 x tile_n tiles in the
    # oracle's order: the page's rotation by the PE's rank (tiles_per_pe =
    # M_r/256 = 1), or, with a publish order, the own rank first and then the
    # others in it
    T_M, T_N, pairs = prob.M // 256, (N + tile_n - 1) // tile_n, grid // 2
    visit = None if perm is None else [local] + [r for r in perm if r != local]
    pair = (v["tile"] >> np.uint64(32)).astype(np.int64)
    pos = (v["tile"] & np.uint64(0xFFFFFFFF)).astype(np.int64)
    for c in range(pairs):
        mine = np.nonzero(pair == c)[0]
        got = mine[np.argsort(pos[mine])]
        want = oracle.consumer_order(T_M, T_N, pairs, c, 1, local, M_r // 256, visit)
        assert list(got) == list(want), c
    if perm is not None:   # ranks published in the given order
        pub = v["publish"].reshape(R, per_rank)
        for i in range(1, R):
            assert pub[perm[i - 1]].max() <= pub[perm[i]].min()
    # the PE's first tile is on its own rows
    assert oracle.consumer_order(T_M, T_N, pairs, 0, 1, local, 1)[0] == local * T_N
    G_ref, C_ref = prob.oracle_full()
    assert_gemm_close(host_bits(prob.C), C_ref)


def test_skewed_readiness_order_and_delays(api):
    R, M_r, K, N = 8, 128, 512, 512
    d = inputs.ag_inputs(_cfg(R, M_r, K, N), seed=15)
    perm, delay = inputs.skew_schedule(0, R)
    prob = AgProblem(d)
    sig = api.Signal(api.ag_num_flags(R, M_r, K))
    words = api.ag_trace_words(R, M_r, N, K)
    trace = torch.full((words,), -1, dtype=torch.int64, device="cuda")
    opts = api.make_opts(publish_perm=perm, delay_ns=delay, trace=trace)
    tile_n = api.ag_tile_n(R, M_r, N, opts)
    for _ in range(2):
        trace.fill_(-1)
        prob.run(api, sig, sig.next_epoch(), opts)
        assert sig.status()[0] == api.OK
        v = _trace_views(api, prob, trace, torch.cuda.get_device_properties(0).multi_processor_count,
                         tile_n)
        per_rank = v["F"] // R
        pub = v["publish"].reshape(R, per_rank)
        for i in range(1, R):
            assert pub[perm[i - 1]].max() <= pub[perm[i]].min(), f"rank {perm[i]} before {perm[i - 1]}"
        t0 = v["cta_start"].min()
        for r in range(R):
            assert pub[r].min() >= t0 + delay[r], f"rank {r} published before its delay"
        assert np.all(v["publish"] <= v["consume"])
    G_ref, C_ref = prob.oracle_full()
    assert np.array_equal(host_bits(prob.G), G_ref)
    assert_gemm_close(host_bits(prob.C), C_ref)


@pytest.mark.parametrize("name", ["ag_tp", "ag_mlp", "ag_skew"])
def test_full_size_configs_sampled(api, name):
    """The benchmark's workloads at full size, in its launch configuration; sampled rows."""
    cfg = inputs.CONFIGS[name]
    d = inputs.ag_inputs(cfg, seed=0)
    prob = AgProblem(d)
    sig = api.Signal(api.ag_num_flags(prob.R, prob.M_r, prob.K))
    opts = None
    if cfg.get("skew"):
        perm, delay = inputs.skew_schedule(0, prob.R)
        opts = api.make_opts(publish_perm=perm, delay_ns=delay)
    for _ in range(2):
        prob.run(api, sig, sig.next_epoch(), opts)
        assert sig.status()[0] == api.OK
    assert np.all(sig.flags().cpu().numpy() == 2)
    # gathered buffer bit-exact (full), C on sampled rows of every row tile
    G = host_bits(prob.G)
    assert np.array_equal(G, oracle.allgather(d["heap"], d["rank_off"], prob.R, d["a_off"],
                                              prob.M_r, prob.K))
    # one row in every 32-row quarter of every 128-row block: each epilogue
    # warp of both CTAs of every pair tile, in every column tile
    rows = quarter_rows(prob.M, seed=1)
    assert len(rows) == prob.M // 32
    C = host_bits(prob.C)
    assert_gemm_close(C[rows], prob.oracle_rows(rows), what=f"{name} sampled C")


@pytest.mark.parametrize("R,M_r,K,N", [(4, 256, 512, 776), (2, 64, 128, 128), (3, 64, 192, 200)])
def test_row_add_batched_signals(api, R, M_r, K, N):
    """One ADD counter per flag row: counters == epoch * K/ft after each launch."""
    d = inputs.ag_inputs(_cfg(R, M_r, K, N), seed=60 + R)
    prob = AgProblem(d)
    ft = api.ag_flag_tile(M_r, K)
    n_rows = api.ag_num_row_counters(R, M_r, K)
    sig = api.Signal(n_rows)
    for _ in range(5):
        e = sig.next_epoch()
        prob.run(api, sig, e, api.make_opts(signal_mode=api.SIGNAL_ROW_ADD))
        assert sig.status()[0] == api.OK
        assert np.array_equal(sig.flags().cpu().numpy(),
                              oracle.expected_row_counters(n_rows, e, K // ft))
    G_ref, C_ref = prob.oracle_full()
    assert np.array_equal(host_bits(prob.G), G_ref)
    assert_gemm_close(host_bits(prob.C), C_ref)


def test_row_add_and_tile_set_do_not_mix_without_reset(api):
    d = inputs.ag_inputs(_cfg(2, 128, 256, 256), seed=70)
    prob = AgProblem(d)
    sig = api.Signal(api.ag_num_flags(2, 128, 256))
    args = (prob.heap, prob.rank_off, prob.a_off, prob.M_r, prob.N, prob.K, prob.B, prob.G, prob.C)
    assert api.ag_gemm_status(*args, sig, 1) == api.OK
    add = api.make_opts(signal_mode=api.SIGNAL_ROW_ADD)
    assert api.ag_gemm_status(*args, sig, 2, add) == api.ERR_INVALID_ARG
    sig.reset()
    assert api.ag_gemm_status(*args, sig, 1, add) == api.OK
    assert sig.status()[0] == api.OK
    _, C_ref = prob.oracle_full()
    assert_gemm_close(host_bits(prob.C), C_ref)


@pytest.mark.parametrize("perm", [None, (3, 1, 0, 2)])
def test_launch_behind_another_streams_gemm(api, perm):
    """The launch needs no co-residency: started while another stream's GEMMs
    still hold the SMs, its CTAs are placed as SMs free up, so producers and
    consumers start at different times (the trace records how far apart).
    Neither kernel waits on the other; the result must still be the oracle's
    and every flag the epoch."""
    R, M_r, K, N = 4, 1024, 1024, 2048
    d = inputs.ag_inputs(_cfg(R, M_r, K, N), seed=91)
    prob = AgProblem(d)
    F = api.ag_num_flags(R, M_r, K)
    sig = api.Signal(F)
    words = api.ag_trace_words(R, M_r, N, K)
    trace = torch.full((words,), -1, dtype=torch.int64, device="cuda")
    big = torch.randn(8192, 8192, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(big)
    other = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(other):
        for _ in range(4):
            torch.matmul(big, big, out=out)
    e = sig.next_epoch()
    opts = api.make_opts(trace=trace, publish_perm=perm)
    prob.run(api, sig, e, opts)
    torch.cuda.synchronize()
    assert sig.status()[0] == api.OK
    assert np.all(sig.flags().cpu().numpy() == e)
    G_ref, C_ref = prob.oracle_full()
    assert np.array_equal(host_bits(prob.G), G_ref)
    assert_gemm_close(host_bits(prob.C), C_ref)
    grid = torch.cuda.get_device_properties(0).multi_processor_count
    starts = _trace_views(api, prob, trace, grid, api.ag_tile_n(R, M_r, N, opts))["cta_start"]
    starts = starts.astype(np.float64)
    print(f"CTA start spread: {(starts.max() - starts.min()) / 1e3:.1f} us")
