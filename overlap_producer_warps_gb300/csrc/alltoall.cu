// Logical-rank all-to-all with put + signal + epoch (Aboleth README, Tier-2
// all-to-all: one program per peer puts its slice into the peer's receive
// buffer at position RANK, signals the peer's flag for RANK with the epoch,
// and waits until each peer's slice has arrived in its own buffer).
//
// On one GPU every rank's send and receive buffers are slices of the heap.
// A slice of B bytes is cut into 32 KiB pieces; a warp copies one piece, 8 KiB
// at a time (16-byte loads and stores that bypass L1), and, for a peer, releases the
// flag of (receiver j, sender r, piece) with the epoch.  The receiving side
// then acquires every incoming flag (>= epoch, bounded wait): the
// "wait_signal" of the page.  All warps are co-resident (cooperative launch)
// and finish their puts before they wait, so no wait can block a put.
#include <cstring>

#include "opw_device.cuh"
#include "opw_kernels.h"

namespace opw {
namespace {

constexpr int A2A_THREADS = 256;
constexpr int A2A_PIECE = 32768;               // bytes per warp action (one flag)
constexpr int A2A_CHUNK = 8192;                // bytes one warp holds in registers at once
constexpr int A2A_VEC = A2A_CHUNK / 16 / 32;   // uint4 per lane (16)

struct A2aParams {
    char* heap;
    int64_t rank_off[OPW_MAX_RANKS];
    int64_t send_off, recv_off;
    int64_t B;      // bytes per slice
    int32_t R, P;   // ranks, pieces per slice
    int64_t* flags;
    int32_t* status;
    uint64_t epoch;
    uint64_t timeout_ns;
};

__device__ __forceinline__ void copy_chunk(const char* src, char* dst, int len)
{
    const uint32_t lane = lane_id();
    uint4 v[A2A_VEC];
#pragma unroll
    for (int k = 0; k < A2A_VEC; ++k) {
        const int idx = static_cast<int>(lane) + 32 * k;
        if (16 * idx < len) v[k] = __ldcg(reinterpret_cast<const uint4*>(src) + idx);
    }
#pragma unroll
    for (int k = 0; k < A2A_VEC; ++k) {
        const int idx = static_cast<int>(lane) + 32 * k;
        if (16 * idx < len) __stcg(reinterpret_cast<uint4*>(dst) + idx, v[k]);
    }
}

// One release per 32 KiB rather than per 8 KiB: each release waits for the
// warp's stores to be performed, so fewer of them keep more bytes in flight.
__device__ __forceinline__ void copy_piece(const char* src, char* dst, int len)
{
    for (int o = 0; o < len; o += A2A_CHUNK)
        copy_chunk(src + o, dst + o, len - o < A2A_CHUNK ? len - o : A2A_CHUNK);
}

__global__ void __launch_bounds__(A2A_THREADS) alltoall_kernel(const __grid_constant__ A2aParams p)
{
    __shared__ int32_t cta_abort;
    if (threadIdx.x == 0) cta_abort = ld_relaxed_s32(p.status) != 0 ? 1 : 0;
    __syncthreads();
    if (cta_abort) return;  // a device error is latched from an earlier launch
    const ErrCtx ec{p.status, &cta_abort, p.timeout_ns};
    const int warps = A2A_THREADS / 32;
    const int gw = static_cast<int>(blockIdx.x) * warps + static_cast<int>(threadIdx.x >> 5);
    const int GW = static_cast<int>(gridDim.x) * warps;
    const int items = p.R * p.R * p.P;

    // put + signal: item (sender r, receiver j, piece)
    for (int i = gw; i < items; i += GW) {
        const int r = i / (p.R * p.P);
        const int j = (i / p.P) % p.R;
        const int piece = i % p.P;
        const int64_t off = static_cast<int64_t>(piece) * A2A_PIECE;
        const int64_t rest = p.B - off;
        const int len = rest < A2A_PIECE ? static_cast<int>(rest) : A2A_PIECE;
        const char* src = p.heap + p.rank_off[r] + p.send_off + j * p.B + off;
        char* dst = p.heap + p.rank_off[j] + p.recv_off + r * p.B + off;
        copy_piece(src, dst, len);
        if (r != j) {
            __syncwarp();  // every lane's stores precede lane 0's release
            if (lane_id() == 0)
                st_release(p.flags + (static_cast<int64_t>(j) * p.R + r) * p.P + piece,
                           static_cast<int64_t>(p.epoch));
            __syncwarp();
        }
    }

    // wait_signal: item (receiver j, sender r, piece), peers only
    const int64_t e = static_cast<int64_t>(p.epoch);
    for (int i = gw; i < items; i += GW) {
        const int j = i / (p.R * p.P);
        const int r = (i / p.P) % p.R;
        if (r == j) continue;
        const int64_t slot = (static_cast<int64_t>(j) * p.R + r) * p.P + i % p.P;
        if (ld_acquire(p.flags + slot) >= e) continue;
        const uint64_t t0 = globaltimer();
        for (uint32_t it = 1;; ++it) {
            __nanosleep(64);
            if (ld_acquire(p.flags + slot) >= e) break;
            if ((it & 15u) == 0) {
                if (aborted(ec)) return;
                if (globaltimer() - t0 > ec.timeout_ns) {
                    if (lane_id() == 0) raise_error(ec, OPW_ERR_TIMEOUT, j, static_cast<int32_t>(slot));
                    return;
                }
            }
        }
    }
}

cudaError_t launch_alltoall(const A2aParams& p, int sms, cudaStream_t s)
{
    int per_sm = 0;
    cudaError_t err =
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, alltoall_kernel, A2A_THREADS, 0);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    if (per_sm > 4) per_sm = 4;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms * per_sm));
    cfg.blockDim = dim3(A2A_THREADS);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, alltoall_kernel, p);
}

}  // namespace
}  // namespace opw

// ---------------------------------------------------------------- C ABI

extern "C" {

int64_t opw_alltoall_num_flags(int32_t R, int64_t bytes_per_peer)
{
    if (R < 1 || R > OPW_MAX_RANKS || bytes_per_peer <= 0 || bytes_per_peer % 16 != 0) return -1;
    const int64_t P = (bytes_per_peer + opw::A2A_PIECE - 1) / opw::A2A_PIECE;
    return static_cast<int64_t>(R) * R * P;
}

opw_status opw_alltoall(const opw_symm* symm, size_t send_off, size_t recv_off,
                        int64_t bytes_per_peer, opw_signal* sig, uint64_t epoch,
                        const opw_opts* opts, void* stream)
{
    if (symm == nullptr || symm->heap_dev == nullptr || symm->rank_off == nullptr ||
        symm->R < 1 || symm->R > OPW_MAX_RANKS || symm->reserved != 0 || sig == nullptr)
        return OPW_ERR_INVALID_ARG;
    opw_opts o;
    opw_opts_default(&o);
    if (opts != nullptr) o = *opts;
    if (o.sync_mode != 0 || o.schedule != 0 || o.role != 0 || o.publish_perm != nullptr ||
        o.delay_ns != nullptr || o.fault_kind != 0 || o.num_ctas < 0 || o.signal_mode != 0 ||
        o.local_rank < -1 || o.local_rank > 0 || o.trace_dev != nullptr || o.tile_n != 0)
        return OPW_ERR_INVALID_ARG;
    const int R = symm->R;
    if (bytes_per_peer <= 0 || bytes_per_peer % 16 != 0 || bytes_per_peer > (int64_t(1) << 40))
        return OPW_ERR_UNSUPPORTED_SHAPE;
    if ((reinterpret_cast<uintptr_t>(symm->heap_dev) & 15u) != 0 || (send_off & 15u) != 0 ||
        (recv_off & 15u) != 0)
        return OPW_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r) {
        if (symm->rank_off[r] < 0) return OPW_ERR_INVALID_ARG;
        if ((symm->rank_off[r] & 15) != 0) return OPW_ERR_MISALIGNED;
    }
    const int64_t F = opw_alltoall_num_flags(R, bytes_per_peer);
    if (F < 0 || F > (int64_t(1) << 31)) return OPW_ERR_UNSUPPORTED_SHAPE;
    if (sig->num_slots < F) return OPW_ERR_INVALID_ARG;
    if (sig->mode >= 0 && sig->mode != OPW_SIGNAL_TILE_SET) return OPW_ERR_INVALID_ARG;
    if (sig->latched) return OPW_ERR_NOT_READY;
    if (epoch != sig->epoch_last + 1) return OPW_ERR_BAD_EPOCH;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != sig->device) return OPW_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return OPW_ERR_CUDA;
    if (o.num_ctas > 0 && o.num_ctas < sms) sms = o.num_ctas;

    opw::A2aParams p;
    std::memset(&p, 0, sizeof p);
    p.heap = static_cast<char*>(symm->heap_dev);
    for (int r = 0; r < R; ++r) p.rank_off[r] = symm->rank_off[r];
    p.send_off = static_cast<int64_t>(send_off);
    p.recv_off = static_cast<int64_t>(recv_off);
    p.B = bytes_per_peer;
    p.R = R;
    p.P = static_cast<int32_t>((bytes_per_peer + opw::A2A_PIECE - 1) / opw::A2A_PIECE);
    p.flags = sig->flags;
    p.status = sig->status;
    p.epoch = epoch;
    p.timeout_ns = o.timeout_ns != 0 ? o.timeout_ns : 2000000000ull;
    if (opw::launch_alltoall(p, sms, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return OPW_ERR_CUDA;
    sig->mode = OPW_SIGNAL_TILE_SET;
    sig->epoch_last = epoch;
    return OPW_OK;
}

}  // extern "C"
