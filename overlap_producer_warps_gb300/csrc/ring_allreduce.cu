// Tile-centric ring AllReduce over R logical ranks ("Triton-distributed
// Semantics", "Example: Ring AllReduce with Overlap").
//
// Every rank's n fp32 values form R chunks.  Reduce-scatter: in R-1 steps a
// rank adds its own copy of a chunk to the partial sum the previous rank sent
// it (reduced = local + incoming) and sends the result on; all-gather: R-1
// more steps pass every finished chunk around the ring.  Each chunk is split
// into pieces of RING_PIECE values; a piece moves by itself through the
// steps, guarded by one flag per (receiving rank, step, piece) that holds the
// epoch once the piece has landed in that rank's receive slot.  So a piece of
// step s+1 starts as soon as the same piece of step s has arrived, with no
// barrier across ranks: every tile has its own wait and notify ("Example:
// Ring AllReduce with Overlap").
//
// On one GPU the "send" is a store into the next rank's receive slot (its
// slice of the heap) and the "notify" a st.release.gpu of that slot's flag.
// Work item (rank r, piece p) runs 2R-1 actions in order; each warp walks its
// items action by action, so every wait is on an earlier action of another
// item and all warps (co-resident, cooperative launch) make progress.
#include <cstring>

#include "opw_device.cuh"
#include "opw_kernels.h"

namespace opw {
namespace {

constexpr int RING_THREADS = 256;
constexpr int VEC = RING_PIECE / 4 / 32;  // float4 per lane per piece (8)

struct PieceRegs {
    float4 v[VEC];
};

__device__ __forceinline__ void load_piece(const float* src, int len, PieceRegs& out)
{
    const uint32_t lane = lane_id();
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
        const int idx = static_cast<int>(lane) + 32 * k;
        if (4 * idx < len) out.v[k] = __ldcg(reinterpret_cast<const float4*>(src) + idx);
    }
}

__device__ __forceinline__ void store_piece(float* dst, int len, const PieceRegs& in)
{
    const uint32_t lane = lane_id();
#pragma unroll
    for (int k = 0; k < VEC; ++k) {
        const int idx = static_cast<int>(lane) + 32 * k;
        if (4 * idx < len) __stcg(reinterpret_cast<float4*>(dst) + idx, in.v[k]);
    }
}

// Bounded wait (whole warp) until *flag >= epoch.  Every lane performs the
// acquire itself, so each lane's following loads are ordered after it.
__device__ bool wait_flag(const RingParams& p, const ErrCtx& ec, const int64_t* flag, int rank,
                          int64_t slot)
{
    const int64_t e = static_cast<int64_t>(p.epoch);
    if (ld_acquire(flag) >= e) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(64);
        if (ld_acquire(flag) >= e) return true;
        if ((it & 15u) == 0) {
            if (aborted(ec)) return false;
            if (globaltimer() - t0 > ec.timeout_ns) {
                if (lane_id() == 0) raise_error(ec, OPW_ERR_TIMEOUT, rank, static_cast<int32_t>(slot));
                return false;
            }
        }
    }
}

// Publish after every lane's stores of the piece: the warp barrier orders
// them before lane 0's release.
__device__ __forceinline__ void publish(int64_t* flag, uint64_t epoch)
{
    __syncwarp();
    if (lane_id() == 0) st_release(flag, static_cast<int64_t>(epoch));
    __syncwarp();
}

__device__ bool ring_action(const RingParams& p, const ErrCtx& ec, int a, int r, int piece)
{
    const int R = p.R;
    const int64_t off = static_cast<int64_t>(piece) * RING_PIECE;
    const int64_t rest = p.chunk - off;
    const int len = rest < RING_PIECE ? static_cast<int>(rest) : RING_PIECE;
    const int next = (r + 1) % R;
    char* base_r = p.heap + p.rank_off[r];
    char* base_n = p.heap + p.rank_off[next];
    auto X = [&](int c) { return reinterpret_cast<float*>(base_r + p.data_off) + c * p.chunk + off; };
    auto OUT = [&](int c) { return reinterpret_cast<float*>(base_r + p.out_off) + c * p.chunk + off; };
    auto RECV = [&](char* base, int g) {
        return reinterpret_cast<float*>(base + p.recv_off) + static_cast<int64_t>(g) * p.chunk + off;
    };
    auto SLOT = [&](int rank, int g) {
        return (static_cast<int64_t>(rank) * (2 * R - 2) + g) * p.P + piece;
    };

    PieceRegs v;
    if (R == 1) {  // nothing to exchange: the sum is the rank's own data
        load_piece(X(0), len, v);
        store_piece(OUT(0), len, v);
        return true;
    }
    if (a == 0) {  // send my own chunk r to the next rank
        load_piece(X(r), len, v);
        store_piece(RECV(base_n, 0), len, v);
        publish(p.flags + SLOT(next, 0), p.epoch);
        return true;
    }
    if (a <= R - 1) {  // reduce-scatter step s
        const int s = a - 1;
        const int c = (r - s - 1 + 2 * R) % R;
        const int64_t slot = SLOT(r, s);
        if (!wait_flag(p, ec, p.flags + slot, r, slot)) return false;
        PieceRegs in;
        load_piece(X(c), len, v);
        load_piece(RECV(base_r, s), len, in);
#pragma unroll
        for (int k = 0; k < VEC; ++k) {  // reduced = local + incoming
            v.v[k].x = v.v[k].x + in.v[k].x;
            v.v[k].y = v.v[k].y + in.v[k].y;
            v.v[k].z = v.v[k].z + in.v[k].z;
            v.v[k].w = v.v[k].w + in.v[k].w;
        }
        if (s < R - 2) {
            store_piece(RECV(base_n, s + 1), len, v);
            publish(p.flags + SLOT(next, s + 1), p.epoch);
        } else {  // chunk c is complete here: keep it and start the all-gather
            store_piece(OUT(c), len, v);
            store_piece(RECV(base_n, R - 1), len, v);
            publish(p.flags + SLOT(next, R - 1), p.epoch);
        }
        return true;
    }
    // all-gather step s: receive finished chunk (r - s), keep it, pass it on
    const int s = a - R;
    const int g = R - 1 + s;
    const int c = (r - s + 2 * R) % R;
    const int64_t slot = SLOT(r, g);
    if (!wait_flag(p, ec, p.flags + slot, r, slot)) return false;
    load_piece(RECV(base_r, g), len, v);
    store_piece(OUT(c), len, v);
    if (s < R - 2) {
        store_piece(RECV(base_n, g + 1), len, v);
        publish(p.flags + SLOT(next, g + 1), p.epoch);
    }
    return true;
}

__global__ void __launch_bounds__(RING_THREADS) ring_allreduce_kernel(const __grid_constant__ RingParams p)
{
    __shared__ int32_t cta_abort;
    if (threadIdx.x == 0) cta_abort = ld_relaxed_s32(p.status) != 0 ? 1 : 0;
    __syncthreads();
    if (cta_abort) return;  // a device error is latched from an earlier launch
    const ErrCtx ec{p.status, &cta_abort, p.timeout_ns};
    const int warps = RING_THREADS / 32;
    const int gw = static_cast<int>(blockIdx.x) * warps + static_cast<int>(threadIdx.x >> 5);
    const int GW = static_cast<int>(gridDim.x) * warps;
    const int items = p.R * p.P;
    const int actions = p.R == 1 ? 1 : 2 * p.R - 1;
    for (int a = 0; a < actions; ++a) {
        for (int i = gw; i < items; i += GW) {
            if (!ring_action(p, ec, a, i / p.P, i % p.P)) return;
        }
    }
}

}  // namespace

cudaError_t launch_ring_allreduce(const RingParams& p, int sms, cudaStream_t s)
{
    int per_sm = 0;
    cudaError_t err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ring_allreduce_kernel,
                                                                    RING_THREADS, 0);
    if (err != cudaSuccess) return err;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    if (per_sm > 4) per_sm = 4;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms * per_sm));
    cfg.blockDim = dim3(RING_THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, ring_allreduce_kernel, p);
}

}  // namespace opw

// ---------------------------------------------------------------- C ABI

extern "C" {

int64_t opw_ring_num_flags(int32_t R, int64_t n)
{
    if (R < 1 || R > OPW_MAX_RANKS || n <= 0 || n % (4 * R) != 0) return -1;
    const int64_t chunk = n / R;
    const int64_t P = (chunk + opw::RING_PIECE - 1) / opw::RING_PIECE;
    const int64_t f = static_cast<int64_t>(R) * (2 * R - 2) * P;
    return f > 0 ? f : 1;
}

int64_t opw_ring_recv_bytes(int32_t R, int64_t n)
{
    if (R < 1 || R > OPW_MAX_RANKS || n <= 0 || n % (4 * R) != 0) return -1;
    return static_cast<int64_t>(2 * R - 2) * (n / R) * 4;
}

opw_status opw_ring_allreduce(const opw_symm* symm, size_t data_off, size_t recv_off,
                              size_t out_off, int64_t n, opw_signal* sig, uint64_t epoch,
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
    if (n <= 0 || n % (4 * R) != 0 || n / R > (int64_t(1) << 40)) return OPW_ERR_UNSUPPORTED_SHAPE;
    if ((reinterpret_cast<uintptr_t>(symm->heap_dev) & 15u) != 0 || (data_off & 15u) != 0 ||
        (recv_off & 15u) != 0 || (out_off & 15u) != 0)
        return OPW_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r) {
        if (symm->rank_off[r] < 0) return OPW_ERR_INVALID_ARG;
        if ((symm->rank_off[r] & 15) != 0) return OPW_ERR_MISALIGNED;
    }
    const int64_t F = opw_ring_num_flags(R, n);
    if (F < 0 || sig->num_slots < F) return OPW_ERR_INVALID_ARG;
    if (sig->mode >= 0 && sig->mode != OPW_SIGNAL_TILE_SET) return OPW_ERR_INVALID_ARG;
    if (sig->latched) return OPW_ERR_NOT_READY;
    if (epoch != sig->epoch_last + 1) return OPW_ERR_BAD_EPOCH;
    if (static_cast<int64_t>(2 * R - 2) * ((n / R + opw::RING_PIECE - 1) / opw::RING_PIECE) * R >
        (int64_t(1) << 31))
        return OPW_ERR_UNSUPPORTED_SHAPE;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != sig->device) return OPW_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return OPW_ERR_CUDA;
    if (o.num_ctas > 0 && o.num_ctas < sms) sms = o.num_ctas;

    opw::RingParams p;
    std::memset(&p, 0, sizeof p);
    p.heap = static_cast<char*>(symm->heap_dev);
    for (int r = 0; r < R; ++r) p.rank_off[r] = symm->rank_off[r];
    p.data_off = static_cast<int64_t>(data_off);
    p.recv_off = static_cast<int64_t>(recv_off);
    p.out_off = static_cast<int64_t>(out_off);
    p.chunk = n / R;
    p.R = R;
    p.P = static_cast<int32_t>((p.chunk + opw::RING_PIECE - 1) / opw::RING_PIECE);
    p.flags = sig->flags;
    p.status = sig->status;
    p.epoch = epoch;
    p.timeout_ns = o.timeout_ns != 0 ? o.timeout_ns : 2000000000ull;
    if (opw::launch_ring_allreduce(p, sms, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return OPW_ERR_CUDA;
    sig->mode = OPW_SIGNAL_TILE_SET;
    sig->epoch_last = epoch;
    return OPW_OK;
}

}  // extern "C"
