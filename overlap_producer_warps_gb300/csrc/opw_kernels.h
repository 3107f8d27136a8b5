// Internal interface between the C-ABI host code (opw_host.cu) and the
// kernels: parameter blocks passed by value as __grid_constant__ and the
// launch entry points.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/opw.h"

namespace opw {

// GEMM tiling shared by both kernels: CTAs work in pairs (clusters of 2, one
// CTA per SM, tcgen05 cta_group::2) on PAIR_M x BN output tiles.
constexpr int BM = 128;       // output rows per CTA = TMEM lanes
constexpr int PAIR_M = 2 * BM;  // output rows per pair tile
constexpr int BN = 256;       // columns per output tile = fp32 TMEM columns per accumulator
constexpr int BK = 64;        // K per pipeline stage = one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;    // K per tcgen05.mma (kind::f16)
constexpr int TILE_Q = 4;     // depth of the tile-id queue (loader -> MMA, epilogue)

constexpr int A_STAGE_BYTES = BM * BK * 2;       // 16 KiB
constexpr int B_CHUNK_BYTES = BK * 64 * 2;       // 8 KiB: 64 K-rows x 64 N-columns
constexpr int EPI_WARP_BYTES = 32 * 64 * 2;      // 4 KiB: 32 rows x 64 columns bf16
constexpr int GATHER_SUB_ROWS = 32;              // producer copies a flag tile 32 rows at a time
constexpr int GATHER_BUF_BYTES = GATHER_SUB_ROWS * 128 * 2;  // 8 KiB (flag tile <= 128 wide)

// Counter words in the signal object after the flags: per-rank publish
// counts, the tile-claim counter of the dynamic consumer schedule, and the
// flag-tile claim counter of the producer warps.
constexpr int CTR_RANK_DONE = 0;
constexpr int CTR_CLAIM = OPW_MAX_RANKS;
constexpr int CTR_GATHER = OPW_MAX_RANKS + 1;
constexpr int CTR_WORDS = OPW_MAX_RANKS + 8;

// Error-site tags written to status[2] when an on-chip wait times out.
enum WaitSite : int32_t {
    SITE_LOADER_EMPTY = 1001,
    SITE_MMA_FULL = 1002,
    SITE_MMA_TMEM_EMPTY = 1003,
    SITE_EPI_TMEM_FULL = 1004,
    SITE_TILE_QUEUE = 1005,
    SITE_GATHER_LOAD = 1006,
    SITE_DRAIN = 1007,
    SITE_SKEW_ORDER = 1008,
    SITE_SERIAL = 1009,
};

// Trace words of GEMM-RS: [0, F) publish time of each output flag slot,
// [F, 2F) the time the receiving side acquired it.

struct AgParams {
    CUtensorMap shard[OPW_MAX_RANKS];  // A_r [M_r, K], box {ft, 32}, no swizzle (producer load)
    CUtensorMap g_store;               // G [M, K], box {ft, 32}, no swizzle (producer store)
    CUtensorMap g_load;                // G [M, K], box {64, 128}, 128B swizzle (consumer A)
    CUtensorMap b_load;                // B [K, N], box {64, 64}, 128B swizzle (consumer B)
    CUtensorMap c_store;               // C [M, N], box {64, 32}, 128B swizzle (epilogue);
                                       // {32, 32}, 64B swizzle with 256 x 512 tiles
    CUtensorMap a_local_load;          // A_local [M_r, K], box {64, 128}, 128B swizzle (consumer A)
    int64_t* flags;
    int32_t* status;
    unsigned long long* counters;
    uint64_t* trace;
    uint64_t epoch;
    uint64_t timeout_ns;
    uint64_t claim_base;      // claim-counter value before this launch
    uint64_t gather_base;     // producer claim-counter value before this launch
    int32_t R, M_r, M, N, K;
    int32_t ft;               // flag tile edge (64 or 128)
    int32_t T_mr, T_k;        // flag tiles per rank along M, along K
    int32_t T_M, T_N;         // PAIR_M x tile_n pair tiles along M, along N
    int32_t tile_n;           // pair tile columns: BN or 2 * BN (host's choice per launch)
    int32_t role, sync_mode, schedule;
    int32_t group_rows;       // both schedules: pair rows per rasterisation group
    int32_t tpr;              // pair rows per rank (M_r / 256), 0 when a rank's rows are
                              // not whole pair rows (then rows are taken in order)
    int32_t visit[OPW_MAX_RANKS];  // ranks in the order the consumer takes their rows
    int32_t signal_mode;      // OPW_SIGNAL_TILE_SET or OPW_SIGNAL_ROW_ADD
    int32_t local_rank;       // the consumer's own rank (read in place, no flag wait), or -1
    int32_t has_perm, has_delay;
    int32_t fault_kind, fault_arg;
    int32_t perm[OPW_MAX_RANKS];
    uint32_t delay_ns[OPW_MAX_RANKS];
    // rank r's publish counter once every tile of this epoch is published
    uint64_t rank_target[OPW_MAX_RANKS];
};

struct RsParams {
    CUtensorMap a_load[OPW_MAX_RANKS];  // A_r [M, K_r], box {64, 128}, 128B swizzle
    CUtensorMap b_load[OPW_MAX_RANKS];  // B_r [K_r, N], box {64, 128}, 128B swizzle
    CUtensorMap out_store[OPW_MAX_RANKS];  // out_j [M/R, N], box {64, 32}, 128B swizzle
    int64_t* flags;
    int32_t* status;
    uint64_t* trace;
    uint64_t epoch;
    uint64_t timeout_ns;
    int32_t R, M, N, K_r, Mb;
    int32_t T_M, T_N;         // 256 x 256 pair tiles along M, along N
    int32_t group_rows;       // pair rows per rasterisation group of the tile order
    int32_t T_fm, T_fn;       // 128x128 flag tiles per rank block along M, along N
    int32_t checked;          // OPW_SYNC_CHECKED: publish by exchange, expect epoch-1
    int32_t role;             // OPW_ROLE_*: FUSED, PRODUCER (GEMM leg), CONSUMER (scatter leg)
    int32_t fault_kind, fault_arg;  // OPW_FAULT_DROP_TILE: never publish flag slot fault_arg
    // Receiving side (NULL recv: none): warp 3 of each CTA acquires the flags
    // of the other CTA's output tiles and copies each into recv [M, N].
    const uint16_t* out_rank[OPW_MAX_RANKS];  // out_j, [M/R, N] bf16
    uint16_t* recv;
};

struct RingParams {
    char* heap;
    int64_t rank_off[OPW_MAX_RANKS];
    int64_t data_off, recv_off, out_off;  // byte offsets inside every rank's slice
    int64_t chunk;                        // fp32 values per chunk (n / R)
    int32_t R, P;                         // ranks, pieces per chunk
    int64_t* flags;
    int32_t* status;
    uint64_t epoch;
    uint64_t timeout_ns;
};

constexpr int RING_PIECE = 1024;  // fp32 values one warp moves per ring action

// Shared memory each kernel asks for (dynamic, includes 1 KiB alignment slack).
size_t ag_smem_bytes();
size_t rs_smem_bytes();

int ag_max_pairs();  // clusters of 2 AG-GEMM CTAs that fit at once (0 on error)
int ag_producer_warps(int role);  // gathering warps per CTA for OPW_ROLE_* role

// AG-GEMM host set-up shared by the two entry points (opw_host.cu).
// ag_check_args: every argument check that needs no CUDA call; *ft = flag tile.
opw_status ag_check_args(const opw_symm* symm, size_t a_off, int64_t M_r, int64_t N, int64_t K,
                         const void* B_dev, const void* G_dev, const void* C_dev,
                         const opw_opts& o, int64_t* ft);
// CTA pairs to launch for these options on device `dev` (0 on error).
int ag_pairs_for(const opw_opts& o, int dev);
// Pair tile columns (BN or 2 * BN) for a launch of `pairs` pairs on an M x N output.
int ag_tile_n_for(const opw_opts& o, int pairs, int64_t M, int64_t N);
// Tensor maps, shapes and options of the launch; the caller sets flags,
// status, counters, epoch, claim_base and rank_target.
opw_status ag_fill_params(const opw_symm* symm, size_t a_off, int64_t M_r, int64_t N, int64_t K,
                          int64_t ft, const void* B_dev, void* G_dev, void* C_dev,
                          const opw_opts& o, int tile_n, AgParams* p);
cudaError_t launch_ag_gemm(const AgParams& p, int pairs, cudaStream_t s);
int rs_max_pairs();  // clusters of 2 GEMM-RS CTAs that fit at once (0 on error)
cudaError_t launch_gemm_rs(const RsParams& p, int pairs, cudaStream_t s);
cudaError_t launch_ring_allreduce(const RingParams& p, int sms, cudaStream_t s);

}  // namespace opw

// Signal object behind the opaque opw_signal handle (host side).

struct opw_signal {
    int device;
    int64_t num_slots;
    void* mem;                     // one device allocation: flags | status | counters
    int64_t* flags;                // [num_slots]
    int32_t* status;               // [4]: code, rank, slot, reserved
    unsigned long long* counters;  // [CTR_WORDS]
    uint64_t epoch_last;           // last epoch published (host view)
    uint64_t rank_done[OPW_MAX_RANKS];       // expected rank counters after all enqueued launches
    uint64_t rank_target_last[OPW_MAX_RANKS];  // targets of the last producing launch
    uint64_t claim_next;           // claim counter value after all enqueued launches
    uint64_t gather_next;          // producer claim counter value after all enqueued launches
    bool latched;                  // opw_status_sync saw a device error
    int32_t mode;                  // signal mode since the last reset (-1: none yet)
    int64_t mode_tk;               // K/ft used with OPW_SIGNAL_ROW_ADD since the last reset
};


