// GEMM -> ReduceScatter, tile by tile, in one persistent warp-specialised kernel.
//
// Follows "Triton-distributed Semantics", "GEMM and ReduceScatter
// Overlapping": the producer (the GEMM) computes each rank's partial output
// tile and signals it; the consumer (the ReduceScatter) waits for partial
// tiles as they appear, reduces them and scatters the result to the rank that
// owns the rows.  On one GPU the signal between GEMM and reduction is an
// on-chip mbarrier on a TMEM accumulator; the finished row block is written
// into its logical rank's slice and published there with st.release.gpu.
//
// CTAs work in pairs (clusters of 2) on 256 x 256 output tiles with one
// tcgen05 cta_group::2 MMA: CTA c of the pair holds rows 128c..128c+127 of
// A_r and columns 128c..128c+127 of B_r in its shared memory and receives rows
// 128c.. of the accumulator in its own TMEM.  Against one CTA per 128 x 256
// tile this moves a third less operand data from L2 per FLOP.  Each stage of
// the 3-stage ring holds 128 of K (two 128-byte swizzle atoms of A, 128-row
// chunks of B), so one barrier round trip and one commit cover 8 MMAs: with
// 64 of K per stage and 6 stages the same ring ran about 1 % slower and used
// 5 % more cycles per FLOP.  12 warps per CTA:
//   warp 0      loader (both CTAs): TMA-loads this CTA's half of every A_r / B_r
//               k-block, for rank r = 0..R-1 in order; the bytes of both
//               halves complete on the even CTA's `full` barrier.
//   warp 1      MMA (even CTA only): one thread issues the pair's MMAs; each
//               rank's partial P_r = A_r * B_r goes into a fresh fp32 TMEM
//               accumulator, alternating between two 256-column buffers.
//   warp 2      allocates / frees the pair's TMEM.
//   warp 3      the receiving side, when the caller asks for it (recv != NULL):
//               for each pair tile it acquires the flags of the OTHER CTA's
//               rows (step 3: it waits until a tile is ready) and copies each
//               finished 128x128 tile from its rank's block into recv.  The
//               other CTA runs on another SM, so every copy reads data that a
//               different SM's TMA stores wrote and released.  Otherwise idle.
//   warps 4-11  reduction (both CTAs): warp w reads TMEM lanes 32*(w&3).. and
//               columns 128*((w-4)>>2)..+127 of each partial and adds it into a
//               running fp32 sum held in registers, in rank order 0..R-1
//               (S = ((0 + P_0) + P_1) + ...); then rounds S to bf16, stores
//               the rows to rank j = row / (M/R) with TMA, and publishes the
//               128x128 output tiles' flags.
// For overlap timing the two legs also run alone: OPW_ROLE_PRODUCER runs the
// GEMM leg (loads, MMAs, the rank-order sums in registers) and stores and
// publishes nothing; OPW_ROLE_CONSUMER runs the scatter leg alone (no loads,
// no MMAs: S stays 0, so every output tile is stored as zeros and published).
#include <atomic>

#include "opw_device.cuh"
#include "opw_kernels.h"

namespace opw {
namespace {

constexpr int RS_THREADS = 384;
constexpr int RED_WARPS = 8;
constexpr int RS_STAGES = 3;
constexpr int RBK = 128;                                // K per stage: two 128-byte swizzle atoms
constexpr int HALF_N = BN / 2;                          // B columns held by each CTA
constexpr int RA_STAGE = BM * RBK * 2;                  // 32 KiB
constexpr int RB_CHUNK = RBK * 64 * 2;                  // 16 KiB: 128 K-rows x 64 N-columns
constexpr int B_HALF_BYTES = RBK * HALF_N * 2;          // 32 KiB: 2 chunks of 64 columns
constexpr uint32_t PAIR_TX_BYTES = 2u * (RA_STAGE + B_HALF_BYTES);

struct RsCtrl {
    uint64_t full[RS_STAGES];   // even CTA: both halves of a stage have landed
    uint64_t empty[RS_STAGES];  // each CTA: the pair MMA is done with its stage
    uint64_t tmem_full[2];      // each CTA: a partial is in its TMEM
    uint64_t tmem_empty[2];     // even CTA: both CTAs' reductions consumed it
    uint64_t mma_done;
    uint32_t tmem_base;
    int32_t abort;
};

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + RS_STAGES * RA_STAGE;
constexpr int OFF_EPI = OFF_B + RS_STAGES * B_HALF_BYTES;
constexpr int OFF_CTRL = OFF_EPI + RED_WARPS * EPI_WARP_BYTES;
constexpr int SMEM_ALLOC = OFF_CTRL + static_cast<int>(sizeof(RsCtrl)) + 1024;
static_assert(SMEM_ALLOC <= 232448, "shared memory budget (227 KiB per CTA)");
static_assert(OFF_B % 1024 == 0 && OFF_EPI % 1024 == 0, "swizzled buffers must be 1024-byte aligned");

constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint32_t IDESC = idesc_bf16_f32(PAIR_M, BN, /*B MN-major*/ true);

__device__ __forceinline__ uint8_t* align1024(uint8_t* p)
{
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

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

// Named barrier over the reduction warps that also ANDs a flag across them,
// so they agree on whether the tile succeeded.  Every reduction warp reaches
// it exactly once per tile, whatever happened before.
__device__ __forceinline__ bool red_bar_and(bool v)
{
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, %2, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "n"(RED_WARPS * 32)
        : "memory");
    return r != 0;
}

// Pair tiles of this cluster: positions cid + i * nc of the tile order, the
// same sequence in both CTAs.
struct PairSched {
    int cid, nc, nt;
};

// The pair tile (row tile m, column tile n; 256 x 256) at position `pos` of
// the tile order: pair rows in groups of p.group_rows, the column index
// outermost inside a group, so that the pairs working at the same time read
// fewer distinct B_r column tiles; successive groups sweep the columns in
// alternating directions, so a group starts on the B_r column tiles the
// previous one left in L2 (6 % fewer DRAM reads on the TP layer).
__device__ __forceinline__ void rs_tile(const RsParams& p, int pos, int& m, int& n)
{
    const int first = (pos / (p.group_rows * p.T_N)) * p.group_rows;
    const int rows = min(p.group_rows, p.T_M - first);
    const int local = pos - first * p.T_N;
    m = first + local % rows;
    n = local / rows;
    if ((first / p.group_rows) & 1) n = p.T_N - 1 - n;  // odd groups sweep the columns backwards
}

__device__ __forceinline__ PairSched pair_sched(const RsParams& p)
{
    PairSched s;
    s.cid = static_cast<int>(cluster_id_x());
    s.nc = static_cast<int>(nclusters_x());
    const int T = p.T_M * p.T_N;
    s.nt = s.cid < T ? (T - s.cid + s.nc - 1) / s.nc : 0;
    return s;
}

__device__ void rs_loader(const RsParams& p, uint8_t* smem, RsCtrl* ctrl, const ErrCtx& ec,
                          uint32_t crank)
{
    if (p.role == OPW_ROLE_CONSUMER) return;
    const uint32_t lane = lane_id();
    const PairSched ps = pair_sched(p);
    const int KB = (p.K_r + RBK - 1) / RBK;
    uint32_t stage = 0, sphase = 0, filled = 0, last_par = 0;
    bool ok = true;
    for (int i = 0; i < ps.nt && ok; ++i) {
        int tm, tn;
        rs_tile(p, ps.cid + i * ps.nc, tm, tn);
        const int m0 = tm * PAIR_M + static_cast<int>(crank) * BM;
        const int n0 = tn * BN + static_cast<int>(crank) * HALF_N;
        for (int r = 0; r < p.R && ok; ++r) {
            for (int kb = 0; kb < KB; ++kb) {
                if (!wait_bar(&ctrl->empty[stage], sphase ^ 1u, ec, SITE_LOADER_EMPTY)) { ok = false; break; }
                if (lane == 0) {
                    // The even CTA's `full` barrier counts the bytes of both halves.
                    const uint32_t fb = mapa_shared(smem_u32(&ctrl->full[stage]), 0);
                    if (crank == 0) mbar_arrive_expect_tx(&ctrl->full[stage], PAIR_TX_BYTES);
                    uint8_t* as_ = smem + OFF_A + stage * RA_STAGE;
                    tma_load_2d_pair(as_, &p.a_load[r], fb, kb * RBK, m0);
                    tma_load_2d_pair(as_ + RA_STAGE / 2, &p.a_load[r], fb, kb * RBK + 64, m0);
                    uint8_t* bs = smem + OFF_B + stage * B_HALF_BYTES;
#pragma unroll
                    for (int j = 0; j < HALF_N / 64; ++j)
                        tma_load_2d_pair(bs + j * RB_CHUNK, &p.b_load[r], fb, n0 + 64 * j, kb * RBK);
                }
                __syncwarp();
                filled |= 1u << stage;
                last_par = (last_par & ~(1u << stage)) | (sphase << stage);
                if (++stage == RS_STAGES) { stage = 0; sphase ^= 1u; }
            }
        }
    }
    // The even CTA's `full` phases cover both CTAs' loads: let every armed
    // one complete before the pair may exit.
    if (crank == 0)
        for (int st = 0; st < RS_STAGES; ++st)
            if (filled & (1u << st)) drain_bar(&ctrl->full[st], (last_par >> st) & 1u, ec);
}

// Even CTA, warp 1, lane 0 alone: the MMA issue loop (one thread, no warp
// synchronisation per stage, descriptors stepped by addition), since the
// issuing thread's work between one stage's MMAs and the next is on the
// tensor pipe's critical path.
__device__ void rs_mma(const RsParams& p, uint8_t* smem, RsCtrl* ctrl, uint32_t tmem,
                       const ErrCtx& ec)
{
    if (p.role == OPW_ROLE_CONSUMER) return;
    const PairSched ps = pair_sched(p);
    const int KB = (p.K_r + RBK - 1) / RBK;
    // A: K-major, two 128-row x 64-K atoms 16 KiB apart; k steps of 16
    //    elements advance 32 B inside an atom's swizzled rows.
    const uint64_t a_desc0 = sdesc_sw128(smem_u32(smem + OFF_A), 16, 1024);
    // B: N-major, 64-column chunks of 128 K-rows 16 KiB apart (LBO), 8-row K
    //    groups 1024 B apart (SBO); k steps advance 2 KiB.
    const uint64_t b_desc0 = sdesc_sw128(smem_u32(smem + OFF_B), RB_CHUNK, 1024);
    uint32_t stage = 0, sphase = 0, acc = 0, aphase = 0;
    bool ok = true;
    for (int i = 0; i < ps.nt && ok; ++i) {
        for (int r = 0; r < p.R && ok; ++r) {
            // a fresh accumulator for each rank's partial, once both CTAs'
            // reductions have read the previous contents
            if (!wait_bar_cluster(&ctrl->tmem_empty[acc], aphase ^ 1u, ec, SITE_MMA_TMEM_EMPTY)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d = tmem + acc * BN;
            for (int kb = 0; kb < KB; ++kb) {
                if (!wait_bar(&ctrl->full[stage], sphase, ec, SITE_MMA_FULL)) { ok = false; break; }
                tc_fence_after();
                const uint64_t ad = a_desc0 + stage * (RA_STAGE >> 4);
                const uint64_t bd = b_desc0 + stage * (B_HALF_BYTES >> 4);
#pragma unroll
                for (int k = 0; k < RBK / UMMA_K; ++k)
                    mma_bf16_pair(d, ad + ((k >> 2) * (RA_STAGE / 2) + (k & 3) * (UMMA_K * 2)) / 16,
                                  bd + k * ((UMMA_K * 128) >> 4), IDESC, (kb | k) != 0 ? 1u : 0u);
                mma_commit_pair(&ctrl->empty[stage], 0x3);  // both CTAs' stage is free
                if (++stage == RS_STAGES) { stage = 0; sphase ^= 1u; }
            }
            if (!ok) break;
            mma_commit_pair(&ctrl->tmem_full[acc], 0x3);  // partial P_r is ready
            if (++acc == 2) { acc = 0; aphase ^= 1u; }
        }
    }
    mma_commit_pair(&ctrl->mma_done, 0x1);
    drain_bar(&ctrl->mma_done, 0, ec);
}

__device__ void rs_reduce(const RsParams& p, uint8_t* smem, RsCtrl* ctrl, uint32_t tmem,
                          const ErrCtx& ec, int warp, uint32_t crank)
{
    const uint32_t lane = lane_id();
    const PairSched ps = pair_sched(p);
    const int quarter = warp & 3;
    const int half = (warp - 4) >> 2;
    uint8_t* buf = smem + OFF_EPI + (warp - 4) * EPI_WARP_BYTES;
    const uint32_t row_addr = smem_u32(buf) + lane * 128u;
    uint32_t empty_caddr[2];
    for (int a = 0; a < 2; ++a) empty_caddr[a] = mapa_shared(smem_u32(&ctrl->tmem_empty[a]), 0);
    uint32_t acc = 0, aphase = 0;
    const bool reduce = p.role != OPW_ROLE_CONSUMER;
    const bool scatter = p.role != OPW_ROLE_PRODUCER;
    for (int i = 0; i < ps.nt; ++i) {
        bool ok = true;
        int tm, tn;
        rs_tile(p, ps.cid + i * ps.nc, tm, tn);
        const int m0 = tm * PAIR_M + static_cast<int>(crank) * BM;
        const int n0 = tn * BN;
        float S[128];
#pragma unroll
        for (int e = 0; e < 128; ++e) S[e] = 0.0f;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        for (int r = 0; r < p.R && reduce; ++r) {
            if (!wait_bar(&ctrl->tmem_full[acc], aphase, ec, SITE_EPI_TMEM_FULL)) { ok = false; break; }
            tc_fence_after();
            const uint32_t taddr = tmem + lane_off + acc * BN + half * 128;
#pragma unroll
            for (int ch = 0; ch < 8; ++ch) {
                uint32_t v[16];
                tmem_ld16(taddr + ch * 16, v);
                tmem_ld_wait(v);
#pragma unroll
                for (int e = 0; e < 16; ++e) S[ch * 16 + e] = S[ch * 16 + e] + __uint_as_float(v[e]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive_cluster(empty_caddr[acc]);  // partial consumed
            if (++acc == 2) { acc = 0; aphase ^= 1u; }
        }

        // Scatter: these rows belong to rank j; store them in its slice.  In a
        // ragged last pair tile the odd CTA's rows may lie past M: it reduced
        // zeros and stores nothing.
        const bool rows_in = scatter && m0 < p.M;
        const int j = rows_in ? m0 / p.Mb : 0;
        const int row_in_block = m0 - j * p.Mb + quarter * 32;
#pragma unroll
        for (int ch = 0; ch < 2 && ok && rows_in; ++ch) {
            uint32_t w[32];
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                const int col = ch * 64 + 2 * e;
                w[e] = pack_bf16x2(__float_as_uint(S[col]), __float_as_uint(S[col + 1]));
            }
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
#pragma unroll
            for (int k = 0; k < 8; ++k)
                st_shared_v4(row_addr + ((static_cast<uint32_t>(k) ^ (lane & 7u)) << 4), w[4 * k],
                             w[4 * k + 1], w[4 * k + 2], w[4 * k + 3]);
            fence_async_shared();
            __syncwarp();
            const int x = n0 + half * 128 + ch * 64;
            if (lane == 0 && x < p.N) {
                tma_store_2d(&p.out_store[j], buf, x, row_in_block);
                bulk_commit();
            }
            __syncwarp();
        }
        // Publish the tile's 128x128 flags once every reduction warp's rows have landed.
        if (lane == 0) bulk_wait<0>();
        __syncwarp();
        if (!red_bar_and(ok)) break;
        if (warp == 4 && lane == 0 && rows_in) {
            fence_async_global();
            const int mt = (m0 - j * p.Mb) / 128;
            for (int t = 0; t < BN / 128; ++t) {
                const int ntile = n0 / 128 + t;
                if (ntile < p.T_fn) {
                    const int slot = (j * p.T_fm + mt) * p.T_fn + ntile;
                    if (p.fault_kind == OPW_FAULT_DROP_TILE && slot == p.fault_arg) continue;
                    const uint64_t t_pub = p.trace != nullptr ? globaltimer() : 0;
                    if (p.checked) {
                        if (atom_exch_release(p.flags + slot, static_cast<int64_t>(p.epoch)) !=
                            static_cast<int64_t>(p.epoch) - 1)
                            raise_error(ec, OPW_ERR_FLAG_PROTOCOL, j, slot);
                    } else {
                        st_release(p.flags + slot, static_cast<int64_t>(p.epoch));
                    }
                    if (p.trace != nullptr) p.trace[slot] = t_pub;
                }
            }
        }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
}

// Warp 3 of both CTAs, when recv is given: the receiving ranks' side.  For
// each pair tile, in the pair's order, acquire (bounded, >= epoch) the flag of
// each 128x128 output tile that the OTHER CTA of the pair reduced and stored,
// then copy that tile from its rank's block out_j into recv (rows as in S).
// Every lane acquires the flag itself, so each lane's loads are ordered after
// it; the writer made its TMA stores visible (bulk wait, proxy fence) before
// its release.
__device__ void rs_receive(const RsParams& p, const ErrCtx& ec, uint32_t crank)
{
    if (p.recv == nullptr) return;
    const uint32_t lane = lane_id();
    const PairSched ps = pair_sched(p);
    const int F = p.R * p.T_fm * p.T_fn;
    const int64_t e = static_cast<int64_t>(p.epoch);
    for (int i = 0; i < ps.nt; ++i) {
        int tm, tn;
        rs_tile(p, ps.cid + i * ps.nc, tm, tn);
        const int m0 = tm * PAIR_M + static_cast<int>(crank ^ 1u) * BM;
        if (m0 >= p.M) continue;  // a ragged last pair tile: the other CTA has no rows
        const int j = m0 / p.Mb;
        const int mt = (m0 - j * p.Mb) / 128;
        const int n_first = (tn * BN) / 128;
        for (int t = 0; t < BN / 128; ++t) {
            const int ntile = n_first + t;
            if (ntile >= p.T_fn) break;
            const int slot = (j * p.T_fm + mt) * p.T_fn + ntile;
            const uint64_t t0 = globaltimer();
            for (uint32_t spin = 0;; ++spin) {
                if (__all_sync(0xffffffffu, ld_acquire(p.flags + slot) >= e)) break;
                __nanosleep(128);
                if ((spin & 7u) == 7u) {
                    if (aborted(ec)) return;
                    if (globaltimer() - t0 > ec.timeout_ns) {
                        if (lane == 0) raise_error(ec, OPW_ERR_TIMEOUT, j, slot);
                        return;
                    }
                }
            }
            if (p.trace != nullptr && lane == 0) p.trace[F + slot] = globaltimer();
            // 128 rows of up to 128 columns, 16 bytes per lane and step
            const int col0 = ntile * 128;
            const int vecs = (p.N - col0 < 128 ? p.N - col0 : 128) / 8;
            const uint16_t* src = p.out_rank[j] + static_cast<int64_t>(m0 - j * p.Mb) * p.N + col0;
            uint16_t* dst = p.recv + static_cast<int64_t>(m0) * p.N + col0;
            for (int v = static_cast<int>(lane); v < 128 * vecs; v += 32) {
                const int row = v / vecs;
                const int c = (v - row * vecs) * 8;
                const uint4 x = *reinterpret_cast<const uint4*>(src + static_cast<int64_t>(row) * p.N + c);
                *reinterpret_cast<uint4*>(dst + static_cast<int64_t>(row) * p.N + c) = x;
            }
        }
    }
}

__global__ void __launch_bounds__(RS_THREADS, 1) gemm_rs_kernel(const __grid_constant__ RsParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    RsCtrl* ctrl = reinterpret_cast<RsCtrl*>(smem + OFF_CTRL);
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);
    const uint32_t crank = cluster_ctarank();

    if (threadIdx.x == 0) {
        for (int i = 0; i < RS_STAGES; ++i) {
            mbar_init(&ctrl->full[i], 1);
            mbar_init(&ctrl->empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctrl->tmem_full[i], 1);
            mbar_init(&ctrl->tmem_empty[i], 2 * RED_WARPS);
        }
        mbar_init(&ctrl->mma_done, 1);
        // A device error latched by an earlier launch: do nothing.
        ctrl->abort = ld_relaxed_s32(p.status) != 0 ? 1 : 0;
        fence_barrier_init();
    }
    // Both CTAs' barriers exist before either CTA signals the other's.
    cluster_sync();
    if (warp == 2) {
        tmem_alloc_pair(&ctrl->tmem_base, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    const ErrCtx ec{p.status, &ctrl->abort, p.timeout_ns};
    // The pair follows the even CTA's start-up decision, so both run or neither does.
    const bool skip = ld_shared_cluster_u32(mapa_shared(smem_u32(&ctrl->abort), 0)) != 0;

    if (!skip) {
        if (warp == 0) {
            rs_loader(p, smem, ctrl, ec, crank);
        } else if (warp == 1) {
            if (crank == 0 && lane_id() == 0) rs_mma(p, smem, ctrl, tmem, ec);
        } else if (warp == 3) {
            rs_receive(p, ec, crank);
        } else if (warp >= 4) {
            rs_reduce(p, smem, ctrl, tmem, ec, warp, crank);
        }
    }

    // No CTA of the pair leaves (or frees TMEM) while the other may still
    // use its shared memory, barriers or TMEM.
    tc_fence_before();
    __syncthreads();
    cluster_sync();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc_pair(tmem, TMEM_COLS);
    }
}

}  // namespace

size_t rs_smem_bytes() { return SMEM_ALLOC; }

// Clusters of this kernel that can be resident at once (0 on error).
int rs_max_pairs()
{
    static std::atomic<int> cached[64] = {};  // per device
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (const int c = cached[dev].load(); c > 0) return c;
    if (cudaFuncSetAttribute(gemm_rs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_ALLOC) != cudaSuccess)
        return 0;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms & ~1));
    cfg.blockDim = dim3(RS_THREADS);
    cfg.dynamicSmemBytes = SMEM_ALLOC;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_rs_kernel, &cfg) != cudaSuccess) return 0;
    cached[dev] = n;
    return n;
}

cudaError_t launch_gemm_rs(const RsParams& p, int pairs, cudaStream_t s)
{
    static std::atomic<bool> attr_set[64] = {};  // per device; set once, benign repeats
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_set[dev]) {
        err = cudaFuncSetAttribute(gemm_rs_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   SMEM_ALLOC);
        if (err != cudaSuccess) return err;
        attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(2 * pairs));
    cfg.blockDim = dim3(RS_THREADS);
    cfg.dynamicSmemBytes = SMEM_ALLOC;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_rs_kernel, p);
}

}  // namespace opw
