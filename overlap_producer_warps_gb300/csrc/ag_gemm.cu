// AllGather -> GEMM, tile by tile, in one persistent warp-specialised kernel.
//
// Follows "Triton-distributed Semantics": the producer copies every tile of
// every rank's shard into the gathered buffer and signals it ("Producer-
// Consumer Model", "AllGather and GEMM Overlapping" steps 1-2); the consumer
// waits on each tile's signal, establishes the data dependency ("Token-Based
// Data Dependency") and computes at once (step 3); consumers start on their
// own rank's rows and rotate ("Threadblock Swizzling").
//
// CTAs work in pairs (clusters of 2) on 256 x 256 output tiles with one
// tcgen05 cta_group::2 MMA per k step: CTA c of the pair holds rows
// 128c..128c+127 of the tile's A rows and columns 128c..128c+127 of B in its
// shared memory and receives its 128 accumulator rows in its own TMEM.  With
// 256 x 512 pair tiles (below) each k step is two such MMAs, one per
// 256-column half of the tile.  8 warps per CTA (12 with 256 x 512 tiles):
//   warp 0     loader (both CTAs): takes tiles from the on-chip tile queue and
//              TMA-loads this CTA's half of their A k-blocks (from the gathered
//              buffer G, or in place from the local rank's own shard) and B
//              k-blocks into a 6-stage ring (4 stages of twice the B with
//              256 x 512 tiles); the bytes of both halves complete on the
//              even CTA's `full` barrier.
//   warp 1     MMA (even CTA only): lane 0 alone issues the pair's
//              tcgen05.mma (bf16 x bf16 -> fp32) into a double-buffered TMEM
//              accumulator (2 x 128 lanes x 256 columns in each CTA; one
//              128 lanes x 512 columns accumulator with 256 x 512 tiles).
//   warp 2     gather producer (every CTA): claims flag tiles of A_r from a
//              device counter in publish order, TMA-copies each into G through
//              shared memory, waits for the copy to complete, and publishes the
//              tile's flag with st.release.gpu.
//   warp 3     allocates / frees the pair's TMEM; in the even CTA it is also
//              the scheduler: it picks the next output tile, acquires
//              (ld.acquire.gpu) the flags of all the A rows that tile needs
//              (none for the local rank's rows, which are read in place), and
//              only then puts it on both CTAs' tile queues.  Acquiring ahead
//              of the loaders keeps every global-memory round trip off the
//              k-block loop.  In the odd CTA it forwards the release of each
//              queue slot to the even CTA (see pop_tile).
// The GPU plays the consumer of rank p.local_rank (or none, -1): that rank's
// shard is local, so its tiles are taken first and its own flags are never
// waited for; its producer copies still fill G, after every other rank's.
//   warps 4-7  epilogue (both CTAs): tcgen05.ld -> bf16 (round to nearest
//              even) -> swizzled shared memory -> TMA store of C; with
//              256 x 512 pair tiles warps 8-11 take the second column half.
// With the gather alone (OPW_ROLE_PRODUCER) there are no consumer roles:
// warps 0-6 of every CTA are producers, each with staging buffers of its own
// in the shared memory the ring and the epilogue would use.
// Every wait is bounded: on timeout the kernel latches an error in the
// signal object's status word, drains its own in-flight copies and MMAs,
// frees TMEM and returns.  Cluster barriers bracket the kernel, so neither CTA
// of a pair leaves while the other may still use its shared memory or TMEM.
#include <atomic>

#include "opw_device.cuh"
#include "opw_kernels.h"

namespace opw {
namespace {

constexpr int GATHER_BUFS = 2;    // the fused kernel's producer staging buffers
constexpr int PROD_BUFS = 4;      // per producer warp when the gather runs alone
constexpr int HALF_N = BN / 2;                  // B columns of one MMA held by each CTA
constexpr int B_HALF_BYTES = BK * HALF_N * 2;   // 16 KiB: 2 chunks of 64 columns

// Pair tiles are 256 x (256 * NW).
//   NW = 1: one N = 256 MMA per k step into a double-buffered TMEM accumulator
//           (2 x 256 columns), so the epilogue of one tile overlaps the MMAs of
//           the next; a 6-stage ring of 32 KiB stages.  With 2 gather staging
//           buffers it fits the budget (225 KiB); against 5 stages with 4
//           buffers it was 1.3-2.2 % faster fused in a burst.
//   NW = 2: two N = 256 MMAs per k step (B columns 0-255 and 256-511 of the
//           tile) into one 512-column accumulator; a 4-stage ring of 48 KiB
//           stages (against 3 stages, whose loads often landed after the MMA
//           needed them, 1-2 % faster in a burst).  The MMA waits for the
//           read-out of the accumulator, so 8 epilogue warps (384 threads)
//           read its two column halves at once into registers and release it
//           before they store: about 1.8k cycles per tile against 5.2k when
//           the stores came first.  A CTA reads a quarter less operand data
//           from L2 per FLOP.  In a probe GEMM with random operands and whole
//           waves it ran 3.7 % faster in a burst and 5-8 % faster under the
//           power cap, where the lower on-chip traffic bought a 9 % higher SM
//           clock.
// The host picks the width per launch (opts.tile_n, or from the wave counts).
template <int NW>
struct Shape {
    static constexpr int STAGES = NW == 1 ? 6 : 4;
    static constexpr int B_STAGE = NW * B_HALF_BYTES;   // this CTA's B bytes per stage
    static constexpr int OFF_B = STAGES * A_STAGE_BYTES;
    static constexpr int OFF_EPI = OFF_B + STAGES * B_STAGE;  // the ring ends here
    static constexpr int EPI_WARPS = 4 * NW;             // warps 4 .. 4 + EPI_WARPS - 1
    static constexpr int THREADS = 32 * (4 + EPI_WARPS);
    // one staging buffer per epilogue warp: 32 rows x 64 columns (128B swizzle),
    // or x 32 columns (64B swizzle) with 256 x 512 tiles, whose stores come
    // after the accumulator is released and so can be smaller and serial
    static constexpr int EPI_COLS = NW == 1 ? 64 : 32;
    static constexpr int EPI_BUF_BYTES = 32 * EPI_COLS * 2;
    static constexpr int EPI_END = OFF_EPI + EPI_WARPS * EPI_BUF_BYTES;
    static constexpr uint32_t TX = 2u * (A_STAGE_BYTES + B_STAGE);  // both CTAs' bytes per stage
    static constexpr int ACCS = NW == 1 ? 2 : 1;        // TMEM accumulators
    static constexpr int CHUNKS = NW * BN / 64;         // 64-column epilogue chunks per tile
};
static_assert(Shape<1>::EPI_END == Shape<2>::EPI_END, "both layouts end where the gather starts");
static_assert(Shape<1>::OFF_B % 1024 == 0 && Shape<2>::OFF_B % 1024 == 0 &&
                  Shape<1>::OFF_EPI % 1024 == 0 && Shape<2>::OFF_EPI % 1024 == 0 &&
                  A_STAGE_BYTES % 1024 == 0 && B_HALF_BYTES % 1024 == 0,
              "swizzled stages and staging buffers must be 1024-byte aligned");
constexpr int AG_STAGES_MAX = 6;

struct AgCtrl {
    uint64_t full[AG_STAGES_MAX];   // even CTA: both halves of a stage have landed
    uint64_t empty[AG_STAGES_MAX];  // each CTA: the pair MMA is done with its stage
    uint64_t tmem_full[2];      // each CTA: an accumulator is complete in its TMEM
    uint64_t tmem_empty[2];     // even CTA: both CTAs' epilogues have read it
    uint64_t gfull[GATHER_BUFS];
    uint64_t gprod[8 * PROD_BUFS];  // producer-only role: PROD_BUFS per producer warp
    uint64_t tq_full[TILE_Q];   // each CTA: a tile id is in its queue slot
    uint64_t tq_empty[TILE_Q];  // even CTA: its readers of the slot and the odd CTA's forwarder are done
    uint64_t tq_fwd[TILE_Q];    // odd CTA: its readers of the slot are done
    uint64_t need_next;         // even CTA, loader -> scheduler: claim the next tile now
    uint64_t mma_done;
    int32_t tile_q[TILE_Q];
    uint32_t tmem_base;
    int32_t abort;
};

constexpr int OFF_A = 0;
constexpr int OFF_GATHER = OFF_A + Shape<1>::EPI_END;
constexpr int OFF_CTRL = OFF_GATHER + GATHER_BUFS * GATHER_BUF_BYTES;
constexpr int SMEM_ALLOC = OFF_CTRL + static_cast<int>(sizeof(AgCtrl)) + 1024;
static_assert(SMEM_ALLOC <= 232448, "shared memory budget (227 KiB per CTA)");
// With the gather alone (OPW_ROLE_PRODUCER) the consumer warps are idle and
// their shared memory is free: warp w < PROD_WARPS gathers through its own
// PROD_BUFS staging buffers at OFF_A + w * PROD_BUFS * GATHER_BUF_BYTES.
constexpr int PROD_WARPS_FIT = OFF_CTRL / (PROD_BUFS * GATHER_BUF_BYTES);
constexpr int PROD_WARPS = PROD_WARPS_FIT < 8 ? PROD_WARPS_FIT : 8;
static_assert(PROD_WARPS >= 1, "room for at least one producer warp");
static_assert(OFF_GATHER % 1024 == 0, "swizzled buffers must be 1024-byte aligned");

// The loader asks for its next tile this many k-blocks before the end of the
// current one: late enough that a pair never holds more than one tile it has
// not started (the dynamic schedule stays greedy, so pairs that wait longer on
// the gather do not end up with fewer tiles), early enough to hide the flag
// acquire and the first TMA loads.
constexpr int CLAIM_LEAD_KB = 64;

// Arrivals that free a tile-queue slot on the even CTA's tq_empty: its
// loader, MMA and epilogue warps (4, or 8 with 256 x 512 tiles), and the odd
// CTA's forwarder, which arrives once the odd CTA's readers (loader and
// epilogue warps) have all arrived on its tq_fwd.
template <int NW>
constexpr uint32_t TQ_READERS = 1 + 1 + Shape<NW>::EPI_WARPS + 1;
template <int NW>
constexpr uint32_t TQ_ODD_READERS = 1 + Shape<NW>::EPI_WARPS;

constexpr uint32_t TMEM_COLS = 2 * BN;  // two 256-column accumulators, or one of 512
constexpr uint32_t IDESC = idesc_bf16_f32(PAIR_M, BN, /*B MN-major*/ true);

__device__ __forceinline__ uint8_t* align1024(uint8_t* p)
{
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Wait without giving up on an abort: used only to let this CTA's own
// in-flight copies or MMAs land before it exits.  Still time-bounded.
__device__ __forceinline__ void drain_bar(uint64_t* bar, uint32_t parity, const ErrCtx& e)
{
    if (mbar_try_wait(bar, parity)) return;
    const uint64_t t0 = globaltimer();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer() - t0 > e.timeout_ns) {
            raise_error(e, OPW_ERR_TIMEOUT, -1, SITE_DRAIN);
            return;
        }
    }
}

// Pair tile at position `pos` of the consumers' tile order, which both
// schedules share ("Threadblock Swizzling": a PE begins with its own rows, and
// the remote rows have usually arrived by the time it reaches them).
// Pair rows are taken in groups of p.group_rows; within a group the column
// index runs slowest, so when B is larger than L2 can hold next to
// everything else, the pairs working at the same time share B column tiles
// (group_rows = 1 when B fits).  Successive groups sweep the columns in
// alternating directions, so a group starts on the column tiles the previous
// one left in L2 (5 % fewer DRAM reads on the skew layer).  Row position mp is renamed through the rank
// visit order p.visit: the consumer's own rank first (read in place, no
// wait), then every other rank in the order its tiles are published.  With
// ranks published in ring order that renaming is the page's
// pid_m -> (pid_m + rank * tiles_per_pe) mod total_tiles.
__device__ __forceinline__ int ordered_tile(const AgParams& p, int pos)
{
    const int first = (pos / (p.group_rows * p.T_N)) * p.group_rows;
    const int rows = min(p.group_rows, p.T_M - first);
    const int local = pos - first * p.T_N;
    const int mp = first + local % rows;
    int n = local / rows;
    if ((first / p.group_rows) & 1) n = p.T_N - 1 - n;  // odd groups sweep the columns backwards
    const int m = p.tpr > 0 ? p.visit[mp / p.tpr] * p.tpr + mp % p.tpr : mp;
    return m * p.T_N + n;
}

// Wait (whole warp) until every rank's publish counter shows all of its
// tiles published for this epoch: the serial mode's grid-wide barrier.
__device__ bool wait_all_published(const AgParams& p, const ErrCtx& ec)
{
    const uint32_t lane = lane_id();
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 0;; ++it) {
        bool ok = true;
        if (lane < static_cast<uint32_t>(p.R))
            ok = ld_acquire_u64(p.counters + CTR_RANK_DONE + lane) >= p.rank_target[lane];
        if (__all_sync(0xffffffffu, ok)) break;
        __nanosleep(256);
        if ((it & 7u) == 7u) {
            if (aborted(ec)) return false;
            if (globaltimer() - t0 > ec.timeout_ns) {
                if (lane == 0) raise_error(ec, OPW_ERR_TIMEOUT, -1, SITE_SERIAL);
                return false;
            }
        }
    }
    __syncwarp();
    if (lane == 0) fence_acq_rel_gpu();
    __syncwarp();
    return true;
}

// One polling round over the flags of k-columns [ready_kt, ready_kt + 32):
// lane i acquires column ready_kt + i in each flag row the tile covers.
// Returns how many leading columns are published (>= epoch).
__device__ __forceinline__ int poll_flags(const AgParams& p, int base0, int base1, int ready_kt)
{
    const uint32_t lane = lane_id();
    const int kt = ready_kt + static_cast<int>(lane);
    bool ready = true;
    if (kt < p.T_k) {
        const int64_t e = static_cast<int64_t>(p.epoch);
        ready = ld_acquire(p.flags + base0 + kt) >= e;
        if (base1 >= 0) ready = ready && (ld_acquire(p.flags + base1 + kt) >= e);
    }
    const uint32_t mask = __ballot_sync(0xffffffffu, ready);
    int n = (mask == 0xffffffffu) ? 32 : (__ffs(~mask) - 1);
    if (ready_kt + n > p.T_k) n = p.T_k - ready_kt;
    if (n > 0 && p.trace != nullptr && static_cast<int>(lane) < n) {
        const uint64_t now = globaltimer();
        const int F = p.R * p.T_mr * p.T_k;
        atomicMin(reinterpret_cast<unsigned long long*>(p.trace + F + base0 + kt), now);
        if (base1 >= 0)
            atomicMin(reinterpret_cast<unsigned long long*>(p.trace + F + base1 + kt), now);
    }
    return n;
}

// Batched signals: every column of the tile's flag row(s) is published once
// the row counter reaches epoch * T_k.  Returns the columns newly ready
// (all remaining ones, or 0).
__device__ __forceinline__ int poll_rows(const AgParams& p, int base0, int base1, int ready_kt)
{
    const int64_t target = static_cast<int64_t>(p.epoch) * p.T_k;
    bool ready = ld_acquire(p.flags + base0 / p.T_k) >= target;
    if (base1 >= 0) ready = ready && (ld_acquire(p.flags + base1 / p.T_k) >= target);
    ready = __all_sync(0xffffffffu, ready);
    return ready ? p.T_k - ready_kt : 0;
}

__device__ __forceinline__ int poll_any(const AgParams& p, int base0, int base1, int ready_kt)
{
    return p.signal_mode == OPW_SIGNAL_ROW_ADD ? poll_rows(p, base0, base1, ready_kt)
                                               : poll_flags(p, base0, base1, ready_kt);
}

// Acquire at least one more flag column of the tile (bounded wait): on
// return ready_kt has advanced past every column already published.
__device__ __noinline__ bool acquire_flags(const AgParams& p, const ErrCtx& ec, int base0,
                                           int base1, int& ready_kt)
{
    const uint32_t lane = lane_id();
    uint64_t t0 = 0;
    for (uint32_t spins = 0;; ++spins) {
        const int n = poll_any(p, base0, base1, ready_kt);
        if (n > 0) {
            ready_kt += n;
            // take any further columns that are already published, without waiting
            while (ready_kt < p.T_k) {
                const int more = poll_any(p, base0, base1, ready_kt);
                if (more == 0) break;
                ready_kt += more;
            }
            return true;
        }
        if (spins == 0) t0 = globaltimer();
        __nanosleep(128);
        if ((spins & 7u) == 7u) {
            if (aborted(ec)) return false;
            if (globaltimer() - t0 > ec.timeout_ns) {
                if (lane == 0) {
                    if (p.signal_mode == OPW_SIGNAL_ROW_ADD) {
                        const int row = base0 / p.T_k;  // the row counter waited on
                        raise_error(ec, OPW_ERR_TIMEOUT, row / p.T_mr, row);
                    } else {
                        const int slot = base0 + ready_kt;  // first missing slot
                        raise_error(ec, OPW_ERR_TIMEOUT, slot / (p.T_mr * p.T_k), slot);
                    }
                }
                return false;
            }
        }
    }
}

// ------------------------------------------------------------------ scheduler

// Flag rows covered by output rows [m0, m0 + BM): one for 128-row flag tiles,
// two for 64-row ones (base1 = -1 when there is no second row).
__device__ __forceinline__ void flag_rows(const AgParams& p, int m0, int& base0, int& base1)
{
    const int r = m0 / p.M_r;
    const int mt = (m0 - r * p.M_r) / p.ft;
    base0 = (r * p.T_mr + mt) * p.T_k;
    base1 = -1;
    if (p.ft < BM && m0 + p.ft < p.M) {
        const int g = m0 + p.ft;
        const int r1 = g / p.M_r;
        const int mt1 = (g - r1 * p.M_r) / p.ft;
        base1 = (r1 * p.T_mr + mt1) * p.T_k;
    }
}

// Rows [m0, m0 + 128) all belong to the consumer's own rank: read them from
// its shard in place, without any flag.
__device__ __forceinline__ bool local_half(const AgParams& p, int m0)
{
    if (p.local_rank < 0) return false;
    const int last = (m0 + BM <= p.M ? m0 + BM : p.M) - 1;
    return m0 / p.M_r == p.local_rank && last / p.M_r == p.local_rank;
}

struct LoaderRing {
    uint32_t stage = 0, sphase = 0, filled = 0, last_par = 0;
};

// Issue the TMA loads of this CTA's half of k-blocks [kb0, kb1) of a pair
// tile (A rows from m0; B columns n0 + 256 h .. + 127 for each MMA h of the
// k step): the plain GEMM pipeline, with nothing else in the loop.
template <int NW>
__device__ __forceinline__ bool issue_kblocks(const AgParams& p, uint8_t* smem, AgCtrl* ctrl,
                                              const ErrCtx& ec, LoaderRing& rg,
                                              const CUtensorMap* amap, int m0, int n0,
                                              int kb0, int kb1, uint32_t crank)
{
    const uint32_t lane = lane_id();
    for (int kb = kb0; kb < kb1; ++kb) {
        if (!wait_bar(&ctrl->empty[rg.stage], rg.sphase ^ 1u, ec, SITE_LOADER_EMPTY)) return false;
        if (lane == 0) {
            const uint32_t fb = mapa_shared(smem_u32(&ctrl->full[rg.stage]), 0);
            if (crank == 0) mbar_arrive_expect_tx(&ctrl->full[rg.stage], Shape<NW>::TX);
            tma_load_2d_pair(smem + OFF_A + rg.stage * A_STAGE_BYTES, amap, fb, kb * BK, m0);
            uint8_t* bs = smem + Shape<NW>::OFF_B + rg.stage * Shape<NW>::B_STAGE;
#pragma unroll
            for (int h = 0; h < NW; ++h)
#pragma unroll
                for (int j = 0; j < HALF_N / 64; ++j)
                    tma_load_2d_pair(bs + h * B_HALF_BYTES + j * B_CHUNK_BYTES, &p.b_load, fb,
                                     n0 + h * BN + 64 * j, kb * BK);
        }
        __syncwarp();
        rg.filled |= 1u << rg.stage;
        rg.last_par = (rg.last_par & ~(1u << rg.stage)) | (rg.sphase << rg.stage);
        if (++rg.stage == Shape<NW>::STAGES) { rg.stage = 0; rg.sphase ^= 1u; }
    }
    return true;
}

// Take the next tile id from this CTA's queue and release the slot (-2 when
// the wait failed).  The release is a local arrive with CTA-scope release
// semantics: on the even CTA's tq_empty, or on the odd CTA's tq_fwd, from
// which the odd CTA's warp 3 forwards it (run_forwarder).  A cluster-scope
// release arrive here cost about 1000 cycles per pop, and the loader and MMA
// threads pop at every tile boundary.
__device__ __forceinline__ int pop_tile(AgCtrl* ctrl, const ErrCtx& ec, uint32_t& tq,
                                        uint32_t& tqphase, uint32_t crank)
{
    if (!wait_bar_cluster(&ctrl->tq_full[tq], tqphase, ec, SITE_TILE_QUEUE)) return -2;
    const int q = reinterpret_cast<volatile int32_t*>(ctrl->tile_q)[tq];
    __syncwarp();
    if (lane_id() == 0) mbar_arrive(crank == 0 ? &ctrl->tq_empty[tq] : &ctrl->tq_fwd[tq]);
    __syncwarp();
    if (++tq == TILE_Q) { tq = 0; tqphase ^= 1u; }
    return q;
}

// pop_tile for a single thread (the MMA issuer): the same wait, read and
// release, with no warp to synchronise.
__device__ __forceinline__ int pop_tile_thread(AgCtrl* ctrl, const ErrCtx& ec, uint32_t& tq,
                                               uint32_t& tqphase)
{
    if (!wait_bar_cluster(&ctrl->tq_full[tq], tqphase, ec, SITE_TILE_QUEUE)) return -2;
    const int q = reinterpret_cast<volatile int32_t*>(ctrl->tile_q)[tq];
    mbar_arrive(&ctrl->tq_empty[tq]);
    if (++tq == TILE_Q) { tq = 0; tqphase ^= 1u; }
    return q;
}

// Odd CTA, warp 3: for each queue slot in turn, wait until the odd CTA's
// readers have taken it (tq_fwd), then free it on the even CTA's tq_empty
// with one cluster-scope release arrive.  That release is cumulative: it
// carries the readers' CTA-scope releases, so their reads of the slot come
// before the scheduler overwrites it.  Stops after the end-of-work entry.
__device__ void run_forwarder(AgCtrl* ctrl, const ErrCtx& ec)
{
    const uint32_t empty0 = mapa_shared(smem_u32(&ctrl->tq_empty[0]), 0);
    uint32_t tq = 0, tqphase = 0;
    while (true) {
        if (!wait_bar_cluster(&ctrl->tq_full[tq], tqphase, ec, SITE_TILE_QUEUE)) return;
        const int q = reinterpret_cast<volatile int32_t*>(ctrl->tile_q)[tq];
        if (!wait_bar(&ctrl->tq_fwd[tq], tqphase, ec, SITE_TILE_QUEUE)) return;
        __syncwarp();
        if (lane_id() == 0) mbar_arrive_cluster(empty0 + 8u * tq);
        __syncwarp();
        if (++tq == TILE_Q) { tq = 0; tqphase ^= 1u; }
        if (q < 0) return;
    }
}

// Even CTA, warp 3.
__device__ void run_scheduler(const AgParams& p, AgCtrl* ctrl, const ErrCtx& ec)
{
    const uint32_t lane = lane_id();
    const int G = static_cast<int>(nclusters_x());
    const int c = static_cast<int>(cluster_id_x());
    const int T = p.T_M * p.T_N;

    // Static schedule: pair c takes positions c, c + G, c + 2G, ... of the
    // tile order; the dynamic one claims positions from a device counter.

    const uint32_t peer_tq_full0 = mapa_shared(smem_u32(&ctrl->tq_full[0]), 1);
    const uint32_t peer_tile_q0 = mapa_shared(smem_u32(&ctrl->tile_q[0]), 1);
    uint32_t tq = 0, tqphase = 0;
    bool serial_pending = (p.sync_mode == OPW_SYNC_SERIAL);
    for (int s = 0;; ++s) {
        // Claim tile s only when the loader asks for it (it has reached the
        // last CLAIM_LEAD_KB k-blocks of tile s-1; phases cannot alias, since
        // the loader has popped at most s tiles) and the queue slot is free
        // in both CTAs.
        if (s > 0 && !wait_bar(&ctrl->need_next, (s - 1) & 1u, ec, SITE_TILE_QUEUE)) return;
        if (!wait_bar_cluster(&ctrl->tq_empty[tq], tqphase ^ 1u, ec, SITE_TILE_QUEUE)) return;
        int q;
        if (p.schedule == OPW_SCHED_READY) {
            long long idx = 0;
            if (lane == 0)
                idx = static_cast<long long>(atomicAdd(p.counters + CTR_CLAIM, 1ull) - p.claim_base);
            idx = __shfl_sync(0xffffffffu, idx, 0);
            q = idx < T ? ordered_tile(p, static_cast<int>(idx)) : -1;
        } else {
            const long long pos = c + static_cast<long long>(s) * G;
            q = pos < T ? ordered_tile(p, static_cast<int>(pos)) : -1;
        }
        if (q >= 0) {
            if (p.trace != nullptr && lane == 0) {
                const int F = p.R * p.T_mr * p.T_k;
                p.trace[2 * F + q] = (static_cast<uint64_t>(c) << 32) | static_cast<uint32_t>(s);
                p.trace[2 * F + T + q] = globaltimer();
            }
            if (serial_pending) {
                if (!wait_all_published(p, ec)) return;
                serial_pending = false;
            }
            // Acquire: no load of this tile's A rows (both 128-row halves)
            // before all their flags show the epoch.
            for (int half = 0; half < 2; ++half) {
                const int m0 = (q / p.T_N) * PAIR_M + half * BM;
                if (m0 >= p.M) break;
                if (local_half(p, m0)) continue;  // read in place: nothing to wait for
                int base0, base1;
                flag_rows(p, m0, base0, base1);
                int ready_kt = 0;
                while (ready_kt < p.T_k)
                    if (!acquire_flags(p, ec, base0, base1, ready_kt)) return;
            }
            // every lane's acquire precedes lane 0's release through the queues
            __syncwarp();
            if (lane == 0) fence_acq_rel_gpu();
            __syncwarp();
        }
        // Hand the tile over to both CTAs (-1 = no more work).
        if (lane == 0) {
            reinterpret_cast<volatile int32_t*>(ctrl->tile_q)[tq] = q;
            st_shared_cluster_s32(peer_tile_q0 + 4u * tq, q);
            mbar_arrive(&ctrl->tq_full[tq]);                    // release: the acquires above come first
            mbar_arrive_cluster(peer_tq_full0 + 8u * tq);
        }
        __syncwarp();
        if (++tq == TILE_Q) { tq = 0; tqphase ^= 1u; }
        if (q < 0) return;
    }
}

// ------------------------------------------------------------------ loader

// Warp 0 of both CTAs: takes tiles from the queue (their flags already
// acquired) and streams this CTA's half of their k-blocks through the ring.
template <int NW>
__device__ void run_loader(const AgParams& p, uint8_t* smem, AgCtrl* ctrl, const ErrCtx& ec,
                           uint32_t crank)
{
    const uint32_t lane = lane_id();
    const int KB = p.K / BK;
    LoaderRing rg;
    uint32_t tq = 0, tqphase = 0;
    while (true) {
        const int q = pop_tile(ctrl, ec, tq, tqphase, crank);
        if (q < 0) break;
        // consume_token: the scheduler's flag acquires reach this thread
        // through the queue barrier; order them before the async-proxy
        // reads of the tile.
        if (lane == 0) fence_async_global();
        __syncwarp();
        const int m0 = (q / p.T_N) * PAIR_M + static_cast<int>(crank) * BM;
        const int n0 = (q % p.T_N) * (NW * BN) + static_cast<int>(crank) * HALF_N;
        const bool loc = local_half(p, m0);
        const CUtensorMap* amap = loc ? &p.a_local_load : &p.g_load;
        const int ay = loc ? m0 - p.local_rank * p.M_r : m0;
        const int kb_ask = KB > CLAIM_LEAD_KB ? KB - CLAIM_LEAD_KB : 0;
        if (!issue_kblocks<NW>(p, smem, ctrl, ec, rg, amap, ay, n0, 0, kb_ask, crank)) break;
        if (crank == 0 && lane == 0) mbar_arrive(&ctrl->need_next);
        if (!issue_kblocks<NW>(p, smem, ctrl, ec, rg, amap, ay, n0, kb_ask, KB, crank)) break;
    }
    // The even CTA's `full` phases cover both CTAs' loads: every armed one
    // must complete before the pair may exit.
    if (crank == 0)
        for (int st = 0; st < Shape<NW>::STAGES; ++st)
            if (rg.filled & (1u << st)) drain_bar(&ctrl->full[st], (rg.last_par >> st) & 1u, ec);
}

// ------------------------------------------------------------------ MMA

// Even CTA, warp 1, lane 0 alone.  The tensor pipe takes an MMA only a
// little ahead of executing it, so whatever this thread does between one
// k-block's MMAs and the next lands on the pipe's critical path: one thread
// with no per-k-block warp synchronisation, stage counters instead of
// divisions, and descriptors stepped by addition (the start-address field
// is the shared address >> 4) kept the k-block at about 515 cycles against
// 570 for the same loop run by a whole warp.
template <int NW>
__device__ void run_mma(const AgParams& p, uint8_t* smem, AgCtrl* ctrl, uint32_t tmem,
                        const ErrCtx& ec)
{
    const int KB = p.K / BK;
    // A: K-major, rows 128 B apart, 8-row groups 1024 B apart; k steps of 16
    //    elements advance 32 B inside the swizzled row.
    const uint64_t a_desc0 = sdesc_sw128(smem_u32(smem + OFF_A), 16, 1024);
    // B: N-major, 64-column chunks 8 KiB apart (LBO), 8-row K groups 1024 B
    //    apart (SBO); k steps of 16 rows advance 2 KiB.
    const uint64_t b_desc0 = sdesc_sw128(smem_u32(smem + Shape<NW>::OFF_B), B_CHUNK_BYTES, 1024);
    uint32_t stage = 0, sphase = 0, acc = 0, aphase = 0, tq = 0, tqphase = 0;
    bool ok = true;
    while (ok) {
        const int q = pop_tile_thread(ctrl, ec, tq, tqphase);
        if (q < 0) break;

        // both CTAs' epilogues have read this accumulator
        if (!wait_bar_cluster(&ctrl->tmem_empty[acc], aphase ^ 1u, ec, SITE_MMA_TMEM_EMPTY)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * BN;
        for (int kb = 0; kb < KB; ++kb) {
            if (!wait_bar(&ctrl->full[stage], sphase, ec, SITE_MMA_FULL)) { ok = false; break; }
            tc_fence_after();
            const uint64_t ad = a_desc0 + stage * (A_STAGE_BYTES >> 4);
            const uint64_t bd = b_desc0 + stage * (Shape<NW>::B_STAGE >> 4);
#pragma unroll
            for (int k = 0; k < BK / UMMA_K; ++k)
#pragma unroll
                for (int h = 0; h < NW; ++h)  // MMA h: tile columns 256 h .. 256 h + 255
                    mma_bf16_pair(d + h * BN, ad + k * ((UMMA_K * 2) >> 4),
                                  bd + h * (B_HALF_BYTES >> 4) + k * ((UMMA_K * 128) >> 4), IDESC,
                                  (kb | k) != 0 ? 1u : 0u);
            mma_commit_pair(&ctrl->empty[stage], 0x3);  // frees both CTAs' stage when done
            if (++stage == Shape<NW>::STAGES) { stage = 0; sphase ^= 1u; }
        }
        if (!ok) break;
        mma_commit_pair(&ctrl->tmem_full[acc], 0x3);
        if (++acc == Shape<NW>::ACCS) { acc = 0; aphase ^= 1u; }
    }
    // Every MMA issued must complete before TMEM is released.
    mma_commit_pair(&ctrl->mma_done, 0x1);
    drain_bar(&ctrl->mma_done, 0, ec);
}

// ------------------------------------------------------------------ epilogue

// One warp stores 32 rows x COLS columns of C (w: this lane's row as COLS / 2
// packed bf16 pairs) through its staging buffer: swizzled st.shared, then one
// TMA store in a bulk group of its own, once the previous store has finished
// reading the buffer.  The C tensor map's box and swizzle match COLS: 64
// columns with the 128-byte swizzle (16-byte chunk j of row r at j ^ (r & 7)),
// 32 columns with the 64-byte swizzle (at j ^ ((r >> 1) & 3)).
template <int COLS>
__device__ __forceinline__ void store_chunk(const AgParams& p, uint8_t* buf, const uint32_t* w,
                                            int x, int row0)
{
    const uint32_t lane = lane_id();
    const uint32_t row_addr = smem_u32(buf) + lane * (COLS * 2u);
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
    const uint32_t sw = COLS == 64 ? (lane & 7u) : ((lane >> 1) & 3u);
#pragma unroll
    for (int j = 0; j < COLS / 8; ++j)
        st_shared_v4(row_addr + ((static_cast<uint32_t>(j) ^ sw) << 4), w[4 * j], w[4 * j + 1],
                     w[4 * j + 2], w[4 * j + 3]);
    fence_async_shared();
    __syncwarp();
    if (lane == 0) {
        tma_store_2d(&p.c_store, buf, x, row0);
        bulk_commit();
    }
    __syncwarp();
}

// Epilogue warps 4 .. 4 + EPI_WARPS - 1 of both CTAs: this CTA's 128 rows of
// each pair tile.  Warp w reads TMEM lanes 32 * (w % 4) .. + 31; with 8
// warps (NW = 2) warps 4-7 take columns 0-255 and warps 8-11 columns 256-511.
// NW = 1: each 64-column chunk goes TMEM -> registers -> bf16 -> swizzled
// staging rows -> TMA store, with the next chunk's TMEM load in flight
// meanwhile (chunks outside C are read from TMEM and dropped); the other
// accumulator keeps the MMA busy.  NW = 2: the one accumulator holds up the
// next tile's MMAs until it is read, so each warp reads its whole part into
// registers, releases it, and then stores it 32 columns at a time.
template <int NW>
__device__ void run_epilogue(const AgParams& p, uint8_t* smem, AgCtrl* ctrl, uint32_t tmem,
                             const ErrCtx& ec, int warp, uint32_t crank)
{
    using S = Shape<NW>;
    constexpr int CPW = S::CHUNKS / (S::EPI_WARPS / 4);  // chunks per warp and tile
    const uint32_t lane = lane_id();
    const int quarter = warp & 3;  // TMEM lanes 32*quarter .. +31 belong to this warp
    const int ch0 = ((warp - 4) >> 2) * CPW;  // this warp's first chunk of a tile
    uint8_t* buf = smem + S::OFF_EPI + (warp - 4) * S::EPI_BUF_BYTES;
    // the even CTA's tmem_empty[0], [1] (adjacent 8-byte barriers)
    const uint32_t empty_caddr0 = mapa_shared(smem_u32(&ctrl->tmem_empty[0]), 0);
    uint32_t acc = 0, aphase = 0, tq = 0, tqphase = 0;
    while (true) {
        const int q = pop_tile(ctrl, ec, tq, tqphase, crank);
        if (q < 0) break;

        const int m0 = (q / p.T_N) * PAIR_M + static_cast<int>(crank) * BM;
        const int n0 = (q % p.T_N) * (NW * BN);
        const int row0 = m0 + quarter * 32;
        if (!wait_bar(&ctrl->tmem_full[acc], aphase, ec, SITE_EPI_TMEM_FULL)) break;
        tc_fence_after();
        const uint32_t taddr =
            tmem + (static_cast<uint32_t>(quarter * 32) << 16) + acc * BN + ch0 * 64;
        if constexpr (NW == 2) {
            // The one accumulator holds up the next tile's MMAs until it is
            // read, so read this warp's whole 32 x 256 part into registers
            // first (packed to bf16: 128 registers a lane), release it, and
            // only then store, while the next tile's MMAs run.
            uint32_t pk[CPW][32];
#pragma unroll
            for (int c = 0; c < CPW; ++c) {
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t v[16];
                    tmem_ld16(taddr + c * 64 + h * 16, v);
                    tmem_ld_wait(v);
#pragma unroll
                    for (int i = 0; i < 8; ++i) pk[c][8 * h + i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(empty_caddr0 + 8u * acc);
#pragma unroll
            for (int c = 0; c < CPW; ++c)
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int x = n0 + (ch0 + c) * 64 + h * 32;
                    if (row0 < p.M && x < p.N)  // the same for the whole warp
                        store_chunk<S::EPI_COLS>(p, buf, &pk[c][16 * h], x, row0);
                }
            if (++acc == S::ACCS) { acc = 0; aphase ^= 1u; }
            continue;
        }
        uint32_t v0[32], v1[32];
        tmem_ld32(taddr, v0);
        tmem_ld32(taddr + 32, v1);
        tmem_ld_wait(v0);
        tmem_ld_wait(v1);
#pragma unroll
        for (int c = 0; c < CPW; ++c) {
            const int ch = ch0 + c;
            uint32_t n0v[32], n1v[32];
            if (c + 1 < CPW) {
                tmem_ld32(taddr + (c + 1) * 64, n0v);
                tmem_ld32(taddr + (c + 1) * 64 + 32, n1v);
            } else {
                // accumulator fully read: the MMA may reuse it
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_cluster(empty_caddr0 + 8u * acc);
            }
            if (row0 < p.M && n0 + ch * 64 < p.N) {  // the same for the whole warp
                uint32_t w[32];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    w[i] = pack_bf16x2(v0[2 * i], v0[2 * i + 1]);
                    w[16 + i] = pack_bf16x2(v1[2 * i], v1[2 * i + 1]);
                }
                store_chunk<S::EPI_COLS>(p, buf, w, n0 + ch * 64, row0);
            }
            if (c + 1 < CPW) {
                tmem_ld_wait(n0v);
                tmem_ld_wait(n1v);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    v0[i] = n0v[i];
                    v1[i] = n1v[i];
                }
            }
        }
        if (++acc == S::ACCS) { acc = 0; aphase ^= 1u; }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
}

// ------------------------------------------------------------------ gather producer

// Flag tile at position `pidx` of the publish order, and the position of its
// rank in a permuted publish order (0 without one).
struct GatherItem {
    int r, mt, kt, ip;
};

__device__ __forceinline__ GatherItem gather_item(const AgParams& p, int pidx)
{
    const int per_rank = p.T_mr * p.T_k;
    GatherItem g;
    g.ip = 0;
    if (p.has_perm) {
        // rank-major in publish order
        g.ip = pidx / per_rank;
        g.r = p.perm[g.ip];
        const int rem = pidx - g.ip * per_rank;
        g.mt = rem / p.T_k;
        g.kt = rem - g.mt * p.T_k;
    } else {
        // rank by rank in ring order after the consumer's own rank (the order
        // a ring AllGather delivers them, and the order the swizzled consumers
        // visit them), row block by row block, k fastest; the consumer's own
        // rank (read in place) last
        const int others = p.local_rank >= 0 ? (p.R - 1) * per_rank : p.R * per_rank;
        if (pidx < others) {
            const int ip = pidx / per_rank;
            g.r = p.local_rank >= 0 ? (p.local_rank + 1 + ip) % p.R : ip;
            const int rem = pidx - ip * per_rank;
            g.mt = rem / p.T_k;
            g.kt = rem - g.mt * p.T_k;
        } else {
            const int j = pidx - others;
            g.r = p.local_rank;
            g.mt = j / p.T_k;
            g.kt = j - g.mt * p.T_k;
        }
    }
    return g;
}

// Lane 0: the tile's copy into G is complete (every bulk store committed so
// far has been written), so publish its flag: SET the epoch with a release
// (or, with batched signals, ADD 1 to its row counter), then count it in its
// rank's publish counter.
__device__ __forceinline__ void publish_tile(const AgParams& p, const ErrCtx& ec, const GatherItem& g)
{
    bulk_wait<0>();
    fence_async_global();
    const int slot = (g.r * p.T_mr + g.mt) * p.T_k + g.kt;
    int64_t v = static_cast<int64_t>(p.epoch);
    bool skip = false;
    if (p.fault_kind == OPW_FAULT_DROP_TILE && slot == p.fault_arg) skip = true;
    if (p.fault_kind == OPW_FAULT_STALE_EPOCH && slot == p.fault_arg) v -= 1;
    // the publish time is read before the release, so no consumer can
    // observe the flag earlier than the recorded time
    const uint64_t t_pub = p.trace != nullptr ? globaltimer() : 0;
    const bool checked = p.sync_mode == OPW_SYNC_CHECKED;
    if (p.signal_mode == OPW_SIGNAL_ROW_ADD) {
        // batched signal: one counter per flag row, +1 per k-tile
        if (!skip && v == static_cast<int64_t>(p.epoch)) {
            unsigned long long* ctr =
                reinterpret_cast<unsigned long long*>(p.flags) + g.r * p.T_mr + g.mt;
            if (checked) {
                // this epoch's adds take the counter from (e-1)*T_k to e*T_k
                const uint64_t old = atom_add_release(ctr, 1ull);
                const uint64_t lo = (p.epoch - 1) * static_cast<uint64_t>(p.T_k);
                if (old < lo || old >= lo + static_cast<uint64_t>(p.T_k))
                    raise_error(ec, OPW_ERR_FLAG_PROTOCOL, g.r, g.r * p.T_mr + g.mt);
            } else {
                red_release_add(ctr, 1ull);
            }
        }
    } else if (!skip) {
        if (checked) {
            if (atom_exch_release(p.flags + slot, v) != static_cast<int64_t>(p.epoch) - 1)
                raise_error(ec, OPW_ERR_FLAG_PROTOCOL, g.r, slot);
        } else {
            st_release(p.flags + slot, v);
        }
    }
    red_release_add(p.counters + CTR_RANK_DONE + g.r, 1ull);
    if (p.trace != nullptr) p.trace[slot] = t_pub;
}

// A producer warp: warp 2 of every CTA in the fused kernel, or every warp
// that fits in the idle shared memory when the gather runs alone.  Flag
// tiles are claimed one at a time from a device counter, in publish order, by
// whichever producer warps are running, so no wait anywhere in the grid
// depends on a CTA that has not started: the launch needs no co-residency
// guarantee.  A tile is copied 32 rows at a time: TMA loads of A_r rows into
// the staging buffers, then a TMA store of each into G as it lands, with a
// buffer refilled as soon as its store has read it.  The next tile's loads
// are issued before the previous tile's stores are waited for and its flag
// published, and the next claim is made while the current tile is in flight.
// buf0 / gfull: this warp's nb staging buffers (GATHER_BUF_BYTES each) and
// their barriers.
__device__ void run_gather(const AgParams& p, uint8_t* buf0, uint64_t* gfull, int nb,
                           const ErrCtx& ec, uint64_t t_start)
{
    const uint32_t lane = lane_id();
    const int n_items = p.R * p.T_mr * p.T_k;
    const int subs = p.ft / GATHER_SUB_ROWS;  // 2 or 4
    const uint32_t unb = static_cast<uint32_t>(nb);
    const uint32_t sub_bytes = static_cast<uint32_t>(p.ft) * GATHER_SUB_ROWS * 2u;
    unsigned long long* claim_ctr = p.counters + CTR_GATHER;

    auto claimed = [&](unsigned long long raw) -> int {
        const long long v = static_cast<long long>(__shfl_sync(0xffffffffu, raw, 0) - p.gather_base);
        return v < n_items ? static_cast<int>(v) : -1;
    };
    unsigned long long raw = 0;
    if (lane == 0) raw = atomicAdd(claim_ctr, 1ull);
    int cur = claimed(raw);

    int ordered_upto = 0;  // rank positions whose predecessors are known complete
    uint32_t seq = 0;      // sub-box sequence number: buffer seq % nb
    bool pending = false;  // `pend` is copied (stores committed) but not yet published
    GatherItem pend{0, 0, 0, 0};
    bool ok = true;

    while (cur >= 0 && ok) {
        const GatherItem g = gather_item(p, cur);
        // the next claim travels while this tile is copied
        raw = 0;
        if (lane == 0) raw = atomicAdd(claim_ctr, 1ull);

        // Skewed readiness: rank r starts no earlier than delay_ns[r] after
        // this CTA started, and only after every tile of the rank published
        // before it.  Never wait while holding an unpublished tile: it may be
        // one the wait is for.
        uint32_t need_delay = 0;
        uint64_t d = 0;
        if (p.has_delay) {
            d = p.delay_ns[g.r] < ec.timeout_ns ? p.delay_ns[g.r] : ec.timeout_ns;
            if (lane == 0) need_delay = globaltimer() - t_start < d ? 1u : 0u;
            need_delay = __shfl_sync(0xffffffffu, need_delay, 0);
        }
        const bool need_order = p.has_perm && g.ip > 0 && ordered_upto < g.ip;
        if ((need_delay || need_order) && pending) {
            if (lane == 0) publish_tile(p, ec, pend);
            __syncwarp();
            pending = false;
        }
        if (need_delay)
            while (globaltimer() - t_start < d) __nanosleep(256);
        if (need_order) {
            const uint64_t target = p.rank_target[p.perm[g.ip - 1]];
            const unsigned long long* ctr = p.counters + CTR_RANK_DONE + p.perm[g.ip - 1];
            const uint64_t t0 = globaltimer();
            for (uint32_t s = 0;; ++s) {
                uint32_t done = 0;
                if (lane == 0) done = ld_acquire_u64(ctr) >= target ? 1u : 0u;
                done = __shfl_sync(0xffffffffu, done, 0);
                if (done) break;
                __nanosleep(256);
                if ((s & 7u) == 7u) {
                    if (aborted(ec)) { ok = false; break; }
                    if (globaltimer() - t0 > ec.timeout_ns) {
                        if (lane == 0) raise_error(ec, OPW_ERR_TIMEOUT, p.perm[g.ip - 1], SITE_SKEW_ORDER);
                        ok = false;
                        break;
                    }
                }
            }
            if (!ok) break;
            ordered_upto = g.ip;
        }

        // Loads of this tile, as many as there are staging buffers.  The
        // buffers were last read by the previous tile's stores: those must
        // have finished reading shared memory.
        const int x = g.kt * p.ft;
        const int y_src = g.mt * p.ft;
        const int y_dst = g.r * p.M_r + g.mt * p.ft;
        auto issue_load = [&](int sub) {  // lane 0
            const uint32_t sq = seq + static_cast<uint32_t>(sub);
            uint64_t* fb = &gfull[sq % unb];
            mbar_arrive_expect_tx(fb, sub_bytes);
            tma_load_2d(buf0 + (sq % unb) * GATHER_BUF_BYTES, &p.shard[g.r], fb, x,
                        y_src + sub * GATHER_SUB_ROWS);
        };
        const int ahead = subs < nb ? subs : nb;
        if (lane == 0) {
            bulk_wait_read<0>();
            for (int sub = 0; sub < ahead; ++sub) issue_load(sub);
        }
        __syncwarp();
        // The previous tile's stores are the only ones committed: wait for
        // them and publish it while this tile's loads are in flight.
        if (pending) {
            if (lane == 0) publish_tile(p, ec, pend);
            __syncwarp();
            pending = false;
        }
        // Store each sub-box into G as it lands; refill its buffer with a
        // later sub-box of the tile once the store has read it.
        for (int sub = 0; sub < subs; ++sub) {
            const uint32_t sq = seq + static_cast<uint32_t>(sub);
            if (!wait_bar(&gfull[sq % unb], (sq / unb) & 1u, ec, SITE_GATHER_LOAD)) {
                // every outstanding load must land before the CTA may exit
                const int issued = sub + nb < subs ? sub + nb : subs;
                for (int k = sub; k < issued; ++k) {
                    const uint32_t sk = seq + static_cast<uint32_t>(k);
                    drain_bar(&gfull[sk % unb], (sk / unb) & 1u, ec);
                }
                ok = false;
                break;
            }
            if (lane == 0) {
                tma_store_2d(&p.g_store, buf0 + (sq % unb) * GATHER_BUF_BYTES, x,
                             y_dst + sub * GATHER_SUB_ROWS);
                bulk_commit();
                if (sub + nb < subs) {
                    bulk_wait_read<0>();
                    issue_load(sub + nb);
                }
            }
            __syncwarp();
        }
        if (!ok) break;
        seq += static_cast<uint32_t>(subs);
        pending = true;
        pend = g;
        cur = claimed(raw);
    }
    if (pending && ok && lane == 0) publish_tile(p, ec, pend);
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
}

// ------------------------------------------------------------------ kernel

template <int NW>
__global__ void __launch_bounds__(Shape<NW>::THREADS, 1) ag_gemm_kernel(const __grid_constant__ AgParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    AgCtrl* ctrl = reinterpret_cast<AgCtrl*>(smem + OFF_CTRL);
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
    const uint32_t crank = cluster_ctarank();
    const bool consumer = p.role != OPW_ROLE_PRODUCER;
    const bool producer = p.role != OPW_ROLE_CONSUMER;

    if (threadIdx.x == 0) {
        for (int i = 0; i < Shape<NW>::STAGES; ++i) {
            mbar_init(&ctrl->full[i], 1);
            mbar_init(&ctrl->empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctrl->tmem_full[i], 1);
            mbar_init(&ctrl->tmem_empty[i], 2 * Shape<NW>::EPI_WARPS);  // epilogue warps of both CTAs
        }
        for (int i = 0; i < GATHER_BUFS; ++i) mbar_init(&ctrl->gfull[i], 1);
        for (int i = 0; i < PROD_WARPS * PROD_BUFS; ++i) mbar_init(&ctrl->gprod[i], 1);
        for (int i = 0; i < TILE_Q; ++i) {
            mbar_init(&ctrl->tq_full[i], 1);
            mbar_init(&ctrl->tq_empty[i], TQ_READERS<NW>);
            mbar_init(&ctrl->tq_fwd[i], TQ_ODD_READERS<NW>);
        }
        mbar_init(&ctrl->need_next, 1);
        mbar_init(&ctrl->mma_done, 1);
        // A device error latched by an earlier launch: do nothing.
        ctrl->abort = ld_relaxed_s32(p.status) != 0 ? 1 : 0;
        fence_barrier_init();
    }
    // Both CTAs' barriers exist before either CTA signals the other's.
    cluster_sync();
    if (warp == 3 && consumer) {
        tmem_alloc_pair(&ctrl->tmem_base, TMEM_COLS);
        tmem_relinquish_pair();
    }
    if (threadIdx.x == 32) {
        prefetch_tmap(&p.g_load);
        prefetch_tmap(&p.b_load);
        prefetch_tmap(&p.c_store);
        prefetch_tmap(&p.g_store);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    const ErrCtx ec{p.status, &ctrl->abort, p.timeout_ns};
    const uint64_t t_start = globaltimer();
    if (p.trace != nullptr && threadIdx.x == 0) {
        const int F = p.R * p.T_mr * p.T_k;
        const int T = p.T_M * p.T_N;
        if (blockIdx.x < OPW_TRACE_MAX_CTAS) p.trace[2 * F + 2 * T + blockIdx.x] = t_start;
    }
    // The pair follows the even CTA's start-up decision, so both run or neither does.
    const bool skip = ld_shared_cluster_u32(mapa_shared(smem_u32(&ctrl->abort), 0)) != 0;

    if (!skip && !consumer) {
        // the gather alone: every warp that has room in the idle shared memory
        if (warp < PROD_WARPS)
            run_gather(p, smem + OFF_A + warp * PROD_BUFS * GATHER_BUF_BYTES,
                       &ctrl->gprod[warp * PROD_BUFS], PROD_BUFS, ec, t_start);
    } else if (!skip) {
        if (warp == 0) {
            if (consumer) run_loader<NW>(p, smem, ctrl, ec, crank);
        } else if (warp == 1) {
            if (consumer && crank == 0 && lane_id() == 0) run_mma<NW>(p, smem, ctrl, tmem, ec);
        } else if (warp == 2) {
            if (producer)
                run_gather(p, smem + OFF_GATHER, ctrl->gfull, GATHER_BUFS, ec, t_start);
        } else if (warp == 3) {
            if (consumer && crank == 0) run_scheduler(p, ctrl, ec);
            if (consumer && crank == 1) run_forwarder(ctrl, ec);
        } else {
            if (consumer) run_epilogue<NW>(p, smem, ctrl, tmem, ec, warp, crank);
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 3 && consumer) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, TMEM_COLS);
    }
}

cudaLaunchConfig_t pair_config(unsigned pairs, unsigned threads, cudaStream_t s,
                               cudaLaunchAttribute* attr)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2u * pairs);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = SMEM_ALLOC;
    cfg.stream = s;
    // Clusters of 2 only.  No cross-CTA wait depends on a CTA that has not
    // started (producers claim flag tiles dynamically; consumers wait only on
    // flags), so the launch needs no co-residency guarantee.
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

bool set_smem_attr()
{
    static std::atomic<bool> attr_set[64] = {};  // per device; set once, benign repeats
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (!attr_set[dev]) {
        if (cudaFuncSetAttribute(ag_gemm_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_ALLOC) != cudaSuccess ||
            cudaFuncSetAttribute(ag_gemm_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 SMEM_ALLOC) != cudaSuccess)
            return false;
        attr_set[dev] = true;
    }
    return true;
}

}  // namespace

size_t ag_smem_bytes() { return SMEM_ALLOC; }

int ag_producer_warps(int role) { return role == OPW_ROLE_PRODUCER ? PROD_WARPS : 1; }

int ag_max_pairs()
{
    static std::atomic<int> cached[64] = {};  // per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (const int c = cached[dev].load(); c > 0) return c;
    if (!set_smem_attr()) return 0;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cudaLaunchAttribute attr1[1], attr2[1];
    const unsigned pairs = static_cast<unsigned>(sms / 2);
    const cudaLaunchConfig_t cfg1 = pair_config(pairs, Shape<1>::THREADS, nullptr, attr1);
    const cudaLaunchConfig_t cfg2 = pair_config(pairs, Shape<2>::THREADS, nullptr, attr2);
    // both widths use the same shared memory and cluster shape: one CTA per SM
    int n1 = 0, n2 = 0;
    if (cudaOccupancyMaxActiveClusters(&n1, ag_gemm_kernel<1>, &cfg1) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&n2, ag_gemm_kernel<2>, &cfg2) != cudaSuccess)
        return 0;
    const int n = n1 < n2 ? n1 : n2;
    cached[dev] = n;
    return n;
}

cudaError_t launch_ag_gemm(const AgParams& p, int pairs, cudaStream_t s)
{
    if (!set_smem_attr()) return cudaErrorInvalidDevice;
    cudaLaunchAttribute attr[1];
    const bool wide = p.tile_n == 2 * BN;
    const cudaLaunchConfig_t cfg = pair_config(static_cast<unsigned>(pairs),
                                               wide ? Shape<2>::THREADS : Shape<1>::THREADS, s, attr);
    return wide ? cudaLaunchKernelEx(&cfg, ag_gemm_kernel<2>, p)
                : cudaLaunchKernelEx(&cfg, ag_gemm_kernel<1>, p);
}

}  // namespace opw
