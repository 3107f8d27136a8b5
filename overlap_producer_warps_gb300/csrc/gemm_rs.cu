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
// One CTA per SM, 12 warps:
//   warp 0      loader: TMA-loads A_r / B_r k-blocks for rank r = 0..R-1 in
//               order into a 4-stage shared-memory ring.
//   warp 1      MMA: one thread issues tcgen05.mma; each rank's partial
//               P_r = A_r * B_r goes into a fresh fp32 TMEM accumulator,
//               alternating between two 256-column buffers.
//   warp 2      allocates / frees TMEM.
//   warp 3      idle.
//   warps 4-11  reduction: warp w reads TMEM lanes 32*(w&3).. and columns
//               128*((w-4)>>2)..+127 of each partial and adds it into a
//               running fp32 sum held in registers, in rank order 0..R-1
//               (S = ((0 + P_0) + P_1) + ...); then rounds S to bf16, stores
//               the rows to rank j = row / (M/R) with TMA, and publishes the
//               128x128 output tiles' flags.
#include "opw_device.cuh"
#include "opw_kernels.h"

namespace opw {
namespace {

constexpr int RS_THREADS = 384;
constexpr int RED_WARPS = 8;

struct RsCtrl {
    uint64_t full[STAGES];
    uint64_t empty[STAGES];
    uint64_t tmem_full[2];
    uint64_t tmem_empty[2];
    uint64_t mma_done;
    uint32_t tmem_base;
    int32_t abort;
};

constexpr int OFF_A = 0;
constexpr int OFF_B = OFF_A + STAGES * A_STAGE_BYTES;
constexpr int OFF_EPI = OFF_B + STAGES * B_STAGE_BYTES;
constexpr int OFF_CTRL = OFF_EPI + RED_WARPS * EPI_WARP_BYTES;
constexpr int SMEM_ALLOC = OFF_CTRL + static_cast<int>(sizeof(RsCtrl)) + 1024;
static_assert(SMEM_ALLOC <= 232448, "shared memory budget (227 KiB per CTA)");

constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, /*B MN-major*/ true);

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

// Output tiles of this CTA: q = c + i*G (row tiles of the full M, 256 columns).
__device__ __forceinline__ int n_tiles_of(const RsParams& p)
{
    const int T = p.T_M * p.T_N;
    const int c = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
    return c < T ? (T - c + G - 1) / G : 0;
}

__device__ void rs_loader(const RsParams& p, uint8_t* smem, RsCtrl* ctrl, const ErrCtx& ec)
{
    const uint32_t lane = lane_id();
    const int c = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
    const int KB = (p.K_r + BK - 1) / BK;
    const int nt = n_tiles_of(p);
    uint32_t stage = 0, sphase = 0, filled = 0, last_par = 0;
    bool ok = true;
    for (int i = 0; i < nt && ok; ++i) {
        const int q = c + i * G;
        const int m0 = (q / p.T_N) * BM, n0 = (q % p.T_N) * BN;
        for (int r = 0; r < p.R && ok; ++r) {
            for (int kb = 0; kb < KB; ++kb) {
                if (!wait_bar(&ctrl->empty[stage], sphase ^ 1u, ec, SITE_LOADER_EMPTY)) { ok = false; break; }
                if (lane == 0) {
                    uint64_t* fb = &ctrl->full[stage];
                    mbar_arrive_expect_tx(fb, A_STAGE_BYTES + B_STAGE_BYTES);
                    tma_load_2d(smem + OFF_A + stage * A_STAGE_BYTES, &p.a_load[r], fb, kb * BK, m0);
                    uint8_t* bs = smem + OFF_B + stage * B_STAGE_BYTES;
#pragma unroll
                    for (int j = 0; j < BN / 64; ++j)
                        tma_load_2d(bs + j * B_CHUNK_BYTES, &p.b_load[r], fb, n0 + 64 * j, kb * BK);
                }
                __syncwarp();
                filled |= 1u << stage;
                last_par = (last_par & ~(1u << stage)) | (sphase << stage);
                if (++stage == STAGES) { stage = 0; sphase ^= 1u; }
            }
        }
    }
    for (int st = 0; st < STAGES; ++st)
        if (filled & (1u << st)) drain_bar(&ctrl->full[st], (last_par >> st) & 1u, ec);
}

__device__ void rs_mma(const RsParams& p, uint8_t* smem, RsCtrl* ctrl, uint32_t tmem,
                       const ErrCtx& ec)
{
    const uint32_t lane = lane_id();
    const int KB = (p.K_r + BK - 1) / BK;
    const int nt = n_tiles_of(p);
    const uint32_t a_base = smem_u32(smem + OFF_A);
    const uint32_t b_base = smem_u32(smem + OFF_B);
    uint32_t stage = 0, sphase = 0, acc = 0, aphase = 0;
    bool ok = true;
    for (int i = 0; i < nt && ok; ++i) {
        for (int r = 0; r < p.R && ok; ++r) {
            // a fresh accumulator for each rank's partial
            if (!wait_bar(&ctrl->tmem_empty[acc], aphase ^ 1u, ec, SITE_MMA_TMEM_EMPTY)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d = tmem + acc * BN;
            for (int kb = 0; kb < KB; ++kb) {
                if (!wait_bar(&ctrl->full[stage], sphase, ec, SITE_MMA_FULL)) { ok = false; break; }
                tc_fence_after();
                if (lane == 0) {
                    const uint32_t as = a_base + stage * A_STAGE_BYTES;
                    const uint32_t bs = b_base + stage * B_STAGE_BYTES;
#pragma unroll
                    for (int k = 0; k < BK / UMMA_K; ++k) {
                        const uint64_t ad = sdesc_sw128(as + k * (UMMA_K * 2), 16, 1024);
                        const uint64_t bd = sdesc_sw128(bs + k * (UMMA_K * 128), B_CHUNK_BYTES, 1024);
                        mma_bf16(d, ad, bd, IDESC, (kb | k) != 0 ? 1u : 0u);
                    }
                    mma_commit(&ctrl->empty[stage]);
                }
                __syncwarp();
                if (++stage == STAGES) { stage = 0; sphase ^= 1u; }
            }
            if (!ok) break;
            if (lane == 0) mma_commit(&ctrl->tmem_full[acc]);  // partial P_r is ready
            __syncwarp();
            if (++acc == 2) { acc = 0; aphase ^= 1u; }
        }
    }
    if (lane == 0) mma_commit(&ctrl->mma_done);
    __syncwarp();
    drain_bar(&ctrl->mma_done, 0, ec);
}

__device__ void rs_reduce(const RsParams& p, uint8_t* smem, RsCtrl* ctrl, uint32_t tmem,
                          const ErrCtx& ec, int warp)
{
    const uint32_t lane = lane_id();
    const int c = static_cast<int>(blockIdx.x), G = static_cast<int>(gridDim.x);
    const int quarter = warp & 3;
    const int half = (warp - 4) >> 2;
    const int nt = n_tiles_of(p);
    uint8_t* buf = smem + OFF_EPI + (warp - 4) * EPI_WARP_BYTES;
    const uint32_t row_addr = smem_u32(buf) + lane * 128u;
    uint32_t acc = 0, aphase = 0;
    for (int i = 0; i < nt; ++i) {
        bool ok = true;
        const int q = c + i * G;
        const int m0 = (q / p.T_N) * BM, n0 = (q % p.T_N) * BN;
        float S[128];
#pragma unroll
        for (int e = 0; e < 128; ++e) S[e] = 0.0f;
        const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
        for (int r = 0; r < p.R; ++r) {
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
            if (lane == 0) mbar_arrive(&ctrl->tmem_empty[acc]);  // partial consumed
            if (++acc == 2) { acc = 0; aphase ^= 1u; }
        }

        // Scatter: these rows belong to rank j; store them in its slice.
        const int j = m0 / p.Mb;
        const int row_in_block = m0 - j * p.Mb + quarter * 32;
#pragma unroll
        for (int ch = 0; ch < 2 && ok; ++ch) {
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
        if (warp == 4 && lane == 0) {
            fence_async_global();
            const int mt = (m0 - j * p.Mb) / 128;
            for (int t = 0; t < BN / 128; ++t) {
                const int ntile = n0 / 128 + t;
                if (ntile < p.T_fn) {
                    const int slot = (j * p.T_fm + mt) * p.T_fn + ntile;
                    const uint64_t t_pub = p.trace != nullptr ? globaltimer() : 0;
                    st_release(p.flags + slot, static_cast<int64_t>(p.epoch));
                    if (p.trace != nullptr) p.trace[slot] = t_pub;
                }
            }
        }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
}

__global__ void __launch_bounds__(RS_THREADS, 1) gemm_rs_kernel(const __grid_constant__ RsParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    RsCtrl* ctrl = reinterpret_cast<RsCtrl*>(smem + OFF_CTRL);
    const int warp = __shfl_sync(0xffffffffu, static_cast<int>(threadIdx.x >> 5), 0);

    if (threadIdx.x == 0) {
        for (int i = 0; i < STAGES; ++i) {
            mbar_init(&ctrl->full[i], 1);
            mbar_init(&ctrl->empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&ctrl->tmem_full[i], 1);
            mbar_init(&ctrl->tmem_empty[i], RED_WARPS);
        }
        mbar_init(&ctrl->mma_done, 1);
        ctrl->abort = ld_relaxed_s32(p.status) != 0 ? 1 : 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (ctrl->abort) return;
    if (warp == 2) {
        tmem_alloc(&ctrl->tmem_base, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = ctrl->tmem_base;
    const ErrCtx ec{p.status, &ctrl->abort, p.timeout_ns};

    if (warp == 0) {
        rs_loader(p, smem, ctrl, ec);
    } else if (warp == 1) {
        rs_mma(p, smem, ctrl, tmem, ec);
    } else if (warp >= 4) {
        rs_reduce(p, smem, ctrl, tmem, ec, warp);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

}  // namespace

size_t rs_smem_bytes() { return SMEM_ALLOC; }

cudaError_t launch_gemm_rs(const RsParams& p, int grid, cudaStream_t s)
{
    static bool attr_set[64] = {};
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
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(RS_THREADS);
    cfg.dynamicSmemBytes = SMEM_ALLOC;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, gemm_rs_kernel, p);
}

}  // namespace opw
