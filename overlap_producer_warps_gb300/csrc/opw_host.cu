// Host side of the C ABI declared in include/opw.h: argument validation,
// signal objects (flags, epochs, status word, counters), tensor-map
// encoding and the launches.  Nothing here prints, throws or
// allocates except opw_signal_alloc.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <new>

#include "../../include/opw.h"
#include "opw_kernels.h"

using namespace opw;

namespace {

constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;

__global__ void signal_reset_kernel(int64_t* flags, int64_t n, int32_t* status,
                                    unsigned long long* counters)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        flags[i] = 0;
    if (blockIdx.x == 0) {
        if (threadIdx.x < 4) status[threadIdx.x] = 0;
        if (threadIdx.x < CTR_WORDS) counters[threadIdx.x] = 0;
    }
}

opw_status reset_device(opw_signal* s, cudaStream_t st)
{
    int blocks = static_cast<int>((s->num_slots + 255) / 256);
    if (blocks < 1) blocks = 1;
    if (blocks > 1024) blocks = 1024;
    signal_reset_kernel<<<blocks, 256, 0, st>>>(s->flags, s->num_slots, s->status, s->counters);
    if (cudaGetLastError() != cudaSuccess) return OPW_ERR_CUDA;
    s->epoch_last = 0;
    for (int r = 0; r < OPW_MAX_RANKS; ++r) s->rank_done[r] = s->rank_target_last[r] = 0;
    s->claim_next = 0;
    s->gather_next = 0;
    s->latched = false;
    s->mode = -1;
    s->mode_tk = 0;
    return OPW_OK;
}

// ---------------------------------------------------------------- CUDA helpers

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D bf16 row-major tensor [rows, cols] (row stride = cols elements).
bool make_map(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint32_t box_cols,
              uint32_t box_rows, CUtensorMapSwizzle sw)
{
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {cols * 2};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count(int dev)
{
    static std::atomic<int> cache[64] = {};  // per device
    if (dev < 0 || dev >= 64) return 0;
    if (const int c = cache[dev].load(); c > 0) return c;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
    return n;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned16(int64_t v) { return (v & 15) == 0; }

const opw_opts& opts_or_default(const opw_opts* o, opw_opts& tmp)
{
    if (o != nullptr) return *o;
    opw_opts_default(&tmp);
    return tmp;
}

opw_status check_symm(const opw_symm* s)
{
    if (s == nullptr || s->heap_dev == nullptr || s->rank_off == nullptr) return OPW_ERR_INVALID_ARG;
    if (s->R < 1 || s->R > OPW_MAX_RANKS || s->reserved != 0) return OPW_ERR_INVALID_ARG;
    if (!aligned16(s->heap_dev)) return OPW_ERR_MISALIGNED;
    for (int r = 0; r < s->R; ++r) {
        if (s->rank_off[r] < 0) return OPW_ERR_INVALID_ARG;
        if (!aligned16(s->rank_off[r])) return OPW_ERR_MISALIGNED;
    }
    return OPW_OK;
}

int grid_for(const opw_opts& o, int dev)
{
    const int sms = sm_count(dev);
    if (sms <= 0) return 0;
    if (o.num_ctas > 0 && o.num_ctas < sms) return o.num_ctas;
    return sms;
}

}  // namespace

// ---------------------------------------------------------------- AG-GEMM set-up
// Shared by opw_ag_gemm and opw_ag_gemm_noalloc.

namespace opw {

opw_status ag_check_args(const opw_symm* symm, size_t a_off, int64_t M_r, int64_t N, int64_t K,
                         const void* B_dev, const void* G_dev, const void* C_dev,
                         const opw_opts& o, int64_t* ft_out)
{
    opw_status st = check_symm(symm);
    if (st != OPW_OK) return st;
    if (B_dev == nullptr || G_dev == nullptr || C_dev == nullptr) return OPW_ERR_INVALID_ARG;
    if (o.sync_mode != OPW_SYNC_OVERLAP && o.sync_mode != OPW_SYNC_SERIAL &&
        o.sync_mode != OPW_SYNC_CHECKED)
        return OPW_ERR_INVALID_ARG;
    if (o.schedule != OPW_SCHED_SWIZZLE && o.schedule != OPW_SCHED_READY) return OPW_ERR_INVALID_ARG;
    if (o.role < OPW_ROLE_FUSED || o.role > OPW_ROLE_CONSUMER) return OPW_ERR_INVALID_ARG;
    if (o.fault_kind < OPW_FAULT_NONE || o.fault_kind > OPW_FAULT_STALE_EPOCH) return OPW_ERR_INVALID_ARG;
    if (o.num_ctas < 0) return OPW_ERR_INVALID_ARG;
    if (o.signal_mode != OPW_SIGNAL_TILE_SET && o.signal_mode != OPW_SIGNAL_ROW_ADD)
        return OPW_ERR_INVALID_ARG;
    if (o.tile_n != 0 && o.tile_n != BN && o.tile_n != 2 * BN) return OPW_ERR_INVALID_ARG;
    const int R = symm->R;
    if (o.local_rank < -1 || o.local_rank >= R) return OPW_ERR_INVALID_ARG;
    if (o.publish_perm != nullptr) {
        bool seen[OPW_MAX_RANKS] = {};
        for (int i = 0; i < R; ++i) {
            const int r = o.publish_perm[i];
            if (r < 0 || r >= R || seen[r]) return OPW_ERR_INVALID_ARG;
            seen[r] = true;
        }
    }
    const int64_t ft = opw_ag_flag_tile(M_r, K);
    if (ft < 0 || N <= 0 || N % 8 != 0) return OPW_ERR_UNSUPPORTED_SHAPE;
    const int64_t M = static_cast<int64_t>(R) * M_r;
    if (M > (int64_t(1) << 31) || N > (int64_t(1) << 31) || K > (int64_t(1) << 31))
        return OPW_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(B_dev) || !aligned16(G_dev) || !aligned16(C_dev) ||
        !aligned16(static_cast<int64_t>(a_off)) ||
        (o.trace_dev != nullptr && (reinterpret_cast<uintptr_t>(o.trace_dev) & 7u) != 0))
        return OPW_ERR_MISALIGNED;
    *ft_out = ft;
    return OPW_OK;
}

int ag_pairs_for(const opw_opts& o, int dev)
{
    // CTAs work in pairs: num_ctas (or the SM count) is rounded down to an
    // even number, at least 2, and capped at what can be resident.
    const int grid = grid_for(o, dev);
    if (grid <= 0) return 0;
    const int max_pairs = ag_max_pairs();
    if (max_pairs <= 0) return 0;
    const int pairs = grid / 2 > 0 ? grid / 2 : 1;
    return pairs < max_pairs ? pairs : max_pairs;
}

int ag_tile_n_for(const opw_opts& o, int pairs, int64_t M, int64_t N)
{
    if (o.tile_n != 0) return o.tile_n;
    if (pairs <= 0) return BN;
    // Whole waves of pair tiles: a 256 x 512 tile takes about 1.93 times as
    // long as a 256 x 256 one (its epilogue is not overlapped), so it pays
    // only when it needs fewer than that many times the 256-wide waves.  On
    // the TP layer (512 tiles of 256 x 256 on 76 pairs) 7 waves beat 4 x 1.93;
    // on the MLP and skew layers (12 and 54 waves) the wide tiles win.
    const int64_t tm = (M + PAIR_M - 1) / PAIR_M;
    const int64_t w1 = (tm * ((N + BN - 1) / BN) + pairs - 1) / pairs;
    const int64_t w2 = (tm * ((N + 2 * BN - 1) / (2 * BN)) + pairs - 1) / pairs;
    return w2 * 193 < w1 * 100 ? 2 * BN : BN;
}

opw_status ag_fill_params(const opw_symm* symm, size_t a_off, int64_t M_r, int64_t N, int64_t K,
                          int64_t ft, const void* B_dev, void* G_dev, void* C_dev,
                          const opw_opts& o, int tile_n, AgParams* pp)
{
    AgParams& p = *pp;
    std::memset(&p, 0, sizeof p);
    const int R = symm->R;
    const int64_t M = static_cast<int64_t>(R) * M_r;
    char* heap = static_cast<char*>(symm->heap_dev);
    for (int r = 0; r < R; ++r) {
        if (!make_map(&p.shard[r], heap + symm->rank_off[r] + a_off, K, M_r, static_cast<uint32_t>(ft),
                      GATHER_SUB_ROWS, CU_TENSOR_MAP_SWIZZLE_NONE))
            return OPW_ERR_CUDA;
    }
    if (!make_map(&p.g_store, G_dev, K, M, static_cast<uint32_t>(ft), GATHER_SUB_ROWS,
                  CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&p.g_load, G_dev, K, M, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&p.b_load, B_dev, N, K, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&p.c_store, C_dev, N, M, tile_n == 2 * BN ? 32 : 64, 32,
                  tile_n == 2 * BN ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B))
        return OPW_ERR_CUDA;
    p.local_rank = o.local_rank;
    if (o.local_rank >= 0 &&
        !make_map(&p.a_local_load, heap + symm->rank_off[o.local_rank] + a_off, K, M_r, 64, BM,
                  CU_TENSOR_MAP_SWIZZLE_128B))
        return OPW_ERR_CUDA;
    p.trace = o.trace_dev;
    p.timeout_ns = o.timeout_ns != 0 ? o.timeout_ns : kDefaultTimeoutNs;
    p.R = R;
    p.M_r = static_cast<int32_t>(M_r);
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.ft = static_cast<int32_t>(ft);
    p.T_mr = static_cast<int32_t>(M_r / ft);
    p.T_k = static_cast<int32_t>(K / ft);
    p.T_M = static_cast<int32_t>((M + PAIR_M - 1) / PAIR_M);
    p.tile_n = tile_n;
    p.T_N = static_cast<int32_t>((N + tile_n - 1) / tile_n);
    p.role = o.role;
    p.sync_mode = o.sync_mode;
    p.schedule = o.schedule;
    // Row groups only pay when B (K x N bf16) is too big to stay in L2.  On
    // the skew layer (B 128 MiB) groups of 8 pair rows read 4.3 GB from DRAM
    // per launch; groups of 12, 16 and 24 were slower, and 16 read 5.5 GB.
    p.group_rows = (K * N * 2 > (int64_t(64) << 20)) ? 8 : 1;
    // Ranks in the order the consumers take their rows: the local rank's own
    // first, then the others in publish order (ring order after the local
    // rank unless a publish order is given).  Rows are renamed rank by rank
    // only when a rank's rows fill whole pair rows.
    p.tpr = static_cast<int32_t>((M_r % PAIR_M == 0) ? M_r / PAIR_M : 0);
    {
        const int own = o.local_rank;
        int k = 0;
        if (own >= 0) p.visit[k++] = own;
        for (int i = 0; i < R; ++i) {
            const int r = o.publish_perm != nullptr ? o.publish_perm[i]
                                                    : (own >= 0 ? (own + 1 + i) % R : i);
            if (r != own && k < R) p.visit[k++] = r;
        }
    }
    p.signal_mode = o.signal_mode;
    p.has_perm = o.publish_perm != nullptr;
    p.has_delay = o.delay_ns != nullptr;
    p.fault_kind = o.fault_kind;
    p.fault_arg = o.fault_arg;
    for (int i = 0; i < R; ++i) {
        p.perm[i] = o.publish_perm != nullptr ? o.publish_perm[i] : i;
        p.delay_ns[i] = o.delay_ns != nullptr ? o.delay_ns[i] : 0u;
    }
    return OPW_OK;
}

}  // namespace opw

// ---------------------------------------------------------------- C ABI

extern "C" {

const char* opw_status_str(opw_status s)
{
    switch (s) {
    case OPW_OK: return "OK";
    case OPW_ERR_INVALID_ARG: return "INVALID_ARG";
    case OPW_ERR_UNSUPPORTED_SHAPE: return "UNSUPPORTED_SHAPE";
    case OPW_ERR_MISALIGNED: return "MISALIGNED";
    case OPW_ERR_BAD_EPOCH: return "BAD_EPOCH";
    case OPW_ERR_CUDA: return "CUDA_ERROR";
    case OPW_ERR_TIMEOUT: return "TIMEOUT";
    case OPW_ERR_FLAG_PROTOCOL: return "FLAG_PROTOCOL";
    case OPW_ERR_NOT_READY: return "NOT_READY";
    default: return "UNKNOWN";
    }
}

int32_t opw_abi_version(void) { return OPW_ABI_VERSION; }

void opw_opts_default(opw_opts* o)
{
    if (o != nullptr) std::memset(o, 0, sizeof(*o));
}

opw_status opw_signal_alloc(opw_signal** out, int64_t num_slots, void* stream)
{
    if (out == nullptr) return OPW_ERR_INVALID_ARG;
    *out = nullptr;
    if (num_slots < 1 || num_slots > (int64_t(1) << 40)) return OPW_ERR_INVALID_ARG;
    opw_signal* s = new (std::nothrow) opw_signal();
    if (s == nullptr) return OPW_ERR_CUDA;
    if (cudaGetDevice(&s->device) != cudaSuccess) {
        delete s;
        return OPW_ERR_CUDA;
    }
    const size_t flag_bytes = static_cast<size_t>(num_slots) * sizeof(int64_t);
    const size_t status_off = (flag_bytes + 255) & ~size_t(255);
    const size_t ctr_off = status_off + 256;
    const size_t total = ctr_off + CTR_WORDS * sizeof(unsigned long long);
    if (cudaMalloc(&s->mem, total) != cudaSuccess) {
        delete s;
        return OPW_ERR_CUDA;
    }
    s->num_slots = num_slots;
    s->flags = static_cast<int64_t*>(s->mem);
    s->status = reinterpret_cast<int32_t*>(static_cast<char*>(s->mem) + status_off);
    s->counters = reinterpret_cast<unsigned long long*>(static_cast<char*>(s->mem) + ctr_off);
    if (reset_device(s, static_cast<cudaStream_t>(stream)) != OPW_OK) {
        cudaFree(s->mem);
        delete s;
        return OPW_ERR_CUDA;
    }
    *out = s;
    return OPW_OK;
}

opw_status opw_signal_reset(opw_signal* sig, void* stream)
{
    if (sig == nullptr) return OPW_ERR_INVALID_ARG;
    return reset_device(sig, static_cast<cudaStream_t>(stream));
}

opw_status opw_signal_free(opw_signal* sig)
{
    if (sig == nullptr) return OPW_OK;
    const cudaError_t e = cudaFree(sig->mem);
    delete sig;
    return e == cudaSuccess ? OPW_OK : OPW_ERR_CUDA;
}

opw_status opw_signal_next_epoch(const opw_signal* sig, uint64_t* epoch)
{
    if (sig == nullptr || epoch == nullptr) return OPW_ERR_INVALID_ARG;
    *epoch = sig->epoch_last + 1;
    return OPW_OK;
}

opw_status opw_signal_flags(const opw_signal* sig, int64_t** flags_dev, int64_t* num_slots)
{
    if (sig == nullptr) return OPW_ERR_INVALID_ARG;
    if (flags_dev != nullptr) *flags_dev = sig->flags;
    if (num_slots != nullptr) *num_slots = sig->num_slots;
    return OPW_OK;
}

opw_status opw_status_sync(opw_signal* sig, void* stream, int32_t* rank, int32_t* tile)
{
    if (sig == nullptr) return OPW_ERR_INVALID_ARG;
    if (rank != nullptr) *rank = -1;
    if (tile != nullptr) *tile = -1;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return OPW_ERR_CUDA;
    int32_t h[4] = {0, 0, 0, 0};
    if (cudaMemcpy(h, sig->status, sizeof h, cudaMemcpyDeviceToHost) != cudaSuccess)
        return OPW_ERR_CUDA;
    if (h[0] != OPW_OK) {
        sig->latched = true;
        if (rank != nullptr) *rank = h[1];
        if (tile != nullptr) *tile = h[2];
    }
    return h[0];
}

int64_t opw_ag_flag_tile(int64_t M_r, int64_t K)
{
    if (M_r <= 0 || K <= 0) return -1;
    if (M_r % 128 == 0 && K % 128 == 0) return 128;
    if (M_r % 64 == 0 && K % 64 == 0) return 64;
    return -1;
}

int64_t opw_ag_num_flags(int32_t R, int64_t M_r, int64_t K)
{
    const int64_t ft = opw_ag_flag_tile(M_r, K);
    if (ft < 0 || R < 1 || R > OPW_MAX_RANKS) return -1;
    return static_cast<int64_t>(R) * (M_r / ft) * (K / ft);
}

int64_t opw_ag_num_row_counters(int32_t R, int64_t M_r, int64_t K)
{
    const int64_t ft = opw_ag_flag_tile(M_r, K);
    if (ft < 0 || R < 1 || R > OPW_MAX_RANKS) return -1;
    return static_cast<int64_t>(R) * (M_r / ft);
}

int64_t opw_ag_trace_words(int32_t R, int64_t M_r, int64_t N, int64_t K)
{
    const int64_t F = opw_ag_num_flags(R, M_r, K);
    if (F < 0 || N <= 0) return -1;
    const int64_t T = ((R * M_r + PAIR_M - 1) / PAIR_M) * ((N + BN - 1) / BN);
    return 2 * F + 2 * T + OPW_TRACE_MAX_CTAS;
}

int32_t opw_ag_tile_n(int32_t R, int64_t M_r, int64_t N, const opw_opts* opts_in)
{
    opw_opts tmp;
    const opw_opts& o = opts_or_default(opts_in, tmp);
    if (R < 1 || R > OPW_MAX_RANKS || M_r <= 0 || N <= 0 || o.num_ctas < 0) return -1;
    if (o.tile_n != 0) return (o.tile_n == BN || o.tile_n == 2 * BN) ? o.tile_n : -1;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    const int pairs = opw::ag_pairs_for(o, dev);
    if (pairs <= 0) return -1;
    return opw::ag_tile_n_for(o, pairs, static_cast<int64_t>(R) * M_r, N);
}

opw_status opw_ag_gemm(const opw_symm* symm, size_t a_off, int64_t M_r, int64_t N, int64_t K,
                       const void* B_dev, void* G_dev, void* C_dev, opw_signal* sig,
                       uint64_t epoch, const opw_opts* opts_in, void* stream)
{
    // ---- arguments (no CUDA call before every check has passed)
    if (sig == nullptr) return OPW_ERR_INVALID_ARG;
    opw_opts tmp;
    const opw_opts& o = opts_or_default(opts_in, tmp);
    int64_t ft = 0;
    opw_status st = opw::ag_check_args(symm, a_off, M_r, N, K, B_dev, G_dev, C_dev, o, &ft);
    if (st != OPW_OK) return st;
    const int R = symm->R;
    const bool row_add = o.signal_mode == OPW_SIGNAL_ROW_ADD;
    const int64_t F = static_cast<int64_t>(R) * (M_r / ft) * (row_add ? 1 : K / ft);
    if (sig->num_slots < F) return OPW_ERR_INVALID_ARG;
    // Row counters are cumulative: one mode (and one K/ft) until the next reset.
    if (sig->mode >= 0 && (sig->mode != o.signal_mode || (row_add && sig->mode_tk != K / ft)))
        return OPW_ERR_INVALID_ARG;
    if (sig->latched) return OPW_ERR_NOT_READY;
    const bool produces = o.role != OPW_ROLE_CONSUMER;
    if (produces ? epoch != sig->epoch_last + 1 : (epoch != sig->epoch_last || epoch == 0))
        return OPW_ERR_BAD_EPOCH;

    // ---- launch
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != sig->device) return OPW_ERR_CUDA;
    const int pairs = opw::ag_pairs_for(o, dev);
    if (pairs <= 0) return OPW_ERR_CUDA;
    AgParams p;
    const int tile_n = opw::ag_tile_n_for(o, pairs, static_cast<int64_t>(R) * M_r, N);
    st = opw::ag_fill_params(symm, a_off, M_r, N, K, ft, B_dev, G_dev, C_dev, o, tile_n, &p);
    if (st != OPW_OK) return st;
    p.flags = sig->flags;
    p.status = sig->status;
    p.counters = sig->counters;
    p.epoch = epoch;
    p.claim_base = sig->claim_next;
    p.gather_base = sig->gather_next;
    const uint64_t per_rank = static_cast<uint64_t>(p.T_mr) * p.T_k;
    for (int r = 0; r < R; ++r)
        p.rank_target[r] = produces ? sig->rank_done[r] + per_rank : sig->rank_target_last[r];

    if (launch_ag_gemm(p, pairs, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return OPW_ERR_CUDA;

    // ---- host bookkeeping for the next launch on this object
    sig->mode = o.signal_mode;
    sig->mode_tk = K / ft;
    if (produces) {
        sig->epoch_last = epoch;
        // every flag tile is claimed once, and every producer warp makes one
        // claim past the end
        sig->gather_next += per_rank * static_cast<uint64_t>(R) +
                            2u * static_cast<uint64_t>(pairs) *
                                static_cast<uint64_t>(ag_producer_warps(o.role));
        for (int r = 0; r < R; ++r) {
            sig->rank_target_last[r] = p.rank_target[r];
            sig->rank_done[r] = p.rank_target[r];
        }
    }
    if (o.role != OPW_ROLE_PRODUCER && o.schedule == OPW_SCHED_READY)
        sig->claim_next += static_cast<uint64_t>(p.T_M) * p.T_N + static_cast<uint64_t>(pairs);
    return OPW_OK;
}

int64_t opw_rs_num_flags(int32_t R, int64_t M, int64_t N)
{
    if (R < 1 || R > OPW_MAX_RANKS || M <= 0 || N <= 0 || M % (128 * R) != 0) return -1;
    return static_cast<int64_t>(R) * (M / R / 128) * ((N + 127) / 128);
}

}  // extern "C"

namespace {

// GEMM-RS launch shared by opw_gemm_rs and opw_gemm_rs_consume (recv_dev
// NULL for the former).
opw_status gemm_rs_launch(const opw_symm* symm, size_t a_off, size_t b_off, size_t out_off,
                          int64_t M, int64_t N, int64_t K_r, void* recv_dev, opw_signal* sig,
                          uint64_t epoch, const opw_opts* opts_in, void* stream)
{
    opw_status st = check_symm(symm);
    if (st != OPW_OK) return st;
    if (sig == nullptr) return OPW_ERR_INVALID_ARG;
    opw_opts tmp;
    const opw_opts& o = opts_or_default(opts_in, tmp);
    if ((o.sync_mode != OPW_SYNC_OVERLAP && o.sync_mode != OPW_SYNC_CHECKED) || o.schedule != 0 ||
        o.role < OPW_ROLE_FUSED || o.role > OPW_ROLE_CONSUMER || o.publish_perm != nullptr ||
        o.delay_ns != nullptr || (o.fault_kind != OPW_FAULT_NONE && o.fault_kind != OPW_FAULT_DROP_TILE) ||
        o.num_ctas < 0 || o.signal_mode != 0 || o.local_rank < -1 || o.local_rank > 0 ||
        o.tile_n != 0)
        return OPW_ERR_INVALID_ARG;
    // the receiving side waits on published tiles: only a fused launch publishes results
    if (recv_dev != nullptr && o.role != OPW_ROLE_FUSED) return OPW_ERR_INVALID_ARG;
    const int R = symm->R;
    if (M <= 0 || N <= 0 || K_r <= 0 || M % (128 * R) != 0 || N % 8 != 0 || K_r % 8 != 0)
        return OPW_ERR_UNSUPPORTED_SHAPE;
    if (M > (int64_t(1) << 31) || N > (int64_t(1) << 31) || K_r > (int64_t(1) << 31))
        return OPW_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(static_cast<int64_t>(a_off)) || !aligned16(static_cast<int64_t>(b_off)) ||
        !aligned16(static_cast<int64_t>(out_off)) ||
        (recv_dev != nullptr && !aligned16(recv_dev)) ||
        (o.trace_dev != nullptr && (reinterpret_cast<uintptr_t>(o.trace_dev) & 7u) != 0))
        return OPW_ERR_MISALIGNED;
    const int64_t F = opw_rs_num_flags(R, M, N);
    if (F < 0 || sig->num_slots < F) return OPW_ERR_INVALID_ARG;
    if (sig->latched) return OPW_ERR_NOT_READY;
    if (epoch != sig->epoch_last + 1) return OPW_ERR_BAD_EPOCH;

    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != sig->device) return OPW_ERR_CUDA;
    // CTAs work in pairs: num_ctas (or the SM count) is rounded down to an
    // even number, at least 2, and capped at what can be resident.
    const int grid = grid_for(o, dev);
    if (grid <= 0) return OPW_ERR_CUDA;
    const int max_pairs = rs_max_pairs();
    if (max_pairs <= 0) return OPW_ERR_CUDA;
    int pairs = grid / 2 > 0 ? grid / 2 : 1;
    if (pairs > max_pairs) pairs = max_pairs;

    RsParams p;
    std::memset(&p, 0, sizeof p);
    const int64_t Mb = M / R;
    char* heap = static_cast<char*>(symm->heap_dev);
    for (int r = 0; r < R; ++r) {
        char* base = heap + symm->rank_off[r];
        if (!make_map(&p.a_load[r], base + a_off, K_r, M, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map(&p.b_load[r], base + b_off, N, K_r, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_map(&p.out_store[r], base + out_off, N, Mb, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B))
            return OPW_ERR_CUDA;
        p.out_rank[r] = reinterpret_cast<const uint16_t*>(base + out_off);
    }
    p.recv = static_cast<uint16_t*>(recv_dev);
    p.flags = sig->flags;
    p.status = sig->status;
    p.trace = o.trace_dev;
    p.epoch = epoch;
    p.timeout_ns = o.timeout_ns != 0 ? o.timeout_ns : kDefaultTimeoutNs;
    p.R = R;
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K_r = static_cast<int32_t>(K_r);
    p.Mb = static_cast<int32_t>(Mb);
    p.T_M = static_cast<int32_t>((M + 2 * BM - 1) / (2 * BM));
    p.T_N = static_cast<int32_t>((N + BN - 1) / BN);
    // Groups of 8 pair rows: the pairs running at the same time (76 on a
    // GB300) cover about 8 x 9 tiles instead of 5 x 16, reading fewer B_r
    // column tiles per wave (measured on the tensor-parallel layer: 4 % fewer
    // DRAM reads, 2.4 % faster than row order; groups of 16 read more).
    p.group_rows = 8;
    p.T_fm = static_cast<int32_t>(Mb / 128);
    p.T_fn = static_cast<int32_t>((N + 127) / 128);
    p.checked = o.sync_mode == OPW_SYNC_CHECKED;
    p.role = o.role;
    p.fault_kind = o.fault_kind;
    p.fault_arg = o.fault_arg;
    if (launch_gemm_rs(p, pairs, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return OPW_ERR_CUDA;
    // The GEMM leg alone publishes nothing: the epoch stays the next one.
    if (o.role != OPW_ROLE_PRODUCER) sig->epoch_last = epoch;
    return OPW_OK;
}

}  // namespace

extern "C" {

opw_status opw_gemm_rs(const opw_symm* symm, size_t a_off, size_t b_off, size_t out_off, int64_t M,
                       int64_t N, int64_t K_r, opw_signal* sig, uint64_t epoch,
                       const opw_opts* opts_in, void* stream)
{
    return gemm_rs_launch(symm, a_off, b_off, out_off, M, N, K_r, nullptr, sig, epoch, opts_in,
                          stream);
}

opw_status opw_gemm_rs_consume(const opw_symm* symm, size_t a_off, size_t b_off, size_t out_off,
                               int64_t M, int64_t N, int64_t K_r, void* recv_dev, opw_signal* sig,
                               uint64_t epoch, const opw_opts* opts_in, void* stream)
{
    if (recv_dev == nullptr) return OPW_ERR_INVALID_ARG;
    return gemm_rs_launch(symm, a_off, b_off, out_off, M, N, K_r, recv_dev, sig, epoch, opts_in,
                          stream);
}

}  // extern "C"
