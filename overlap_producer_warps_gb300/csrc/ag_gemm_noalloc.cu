// opw_ag_gemm_noalloc: the AllGather -> GEMM launch for callers that cannot
// allocate device memory.
//
// opw_ag_gemm needs a signal object, and creating one calls cudaMalloc.  Some
// callers cannot do that: code running under a framework that owns every
// byte of device memory through its own pool (a raw allocation would bypass
// its accounting or fail against its memory cap), and latency-critical
// serving loops where cudaMalloc's implicit device synchronisation is not
// acceptable.  This entry point keeps the kernel's scratch -- the per-tile
// flags and the per-rank / claim counters -- in a fixed array compiled into
// the library instead, so a call allocates nothing.  The caller still passes
// every input and output, plus a small device status word of its own.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (about 512 KiB) until the process exits.  Host code only
// sees a stand-in for its name, never its device address, so the address is
// looked up with cudaGetSymbolAddress once per device and passed to the
// kernels.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/opw.h"
#include "opw_kernels.h"

using namespace opw;

namespace {

// Largest flag count one call may use (OPW_NOALLOC_MAX_FLAGS in opw.h).
constexpr int64_t kMaxFlags = OPW_NOALLOC_MAX_FLAGS;
constexpr int64_t kCounterWords = 32;
static_assert(CTR_WORDS <= kCounterWords, "counter block too small");

// Flags in words [0, kMaxFlags), counters in the next kCounterWords words.
static __device__ __align__(256) unsigned long long opw_noalloc_scratch[kMaxFlags + kCounterWords];

// Per-device address of the scratch array, found once with the device current.
std::mutex g_mu;
void* g_scratch[64] = {};

cudaError_t scratch_for_device(int dev, void** out)
{
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_scratch[dev] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, opw_noalloc_scratch);
        if (e != cudaSuccess) return e;
        if (p == nullptr) return cudaErrorInvalidSymbol;
        g_scratch[dev] = p;
    }
    *out = g_scratch[dev];
    return cudaSuccess;
}

// Every call starts from zero: flags, counters and the caller's status word.
__global__ void noalloc_clear_kernel(int64_t* flags, int64_t n_flags, unsigned long long* counters,
                                     int32_t* status)
{
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n_flags;
         i += stride)
        flags[i] = 0;
    if (blockIdx.x == 0) {
        if (threadIdx.x < kCounterWords) counters[threadIdx.x] = 0;
        if (threadIdx.x < 4) status[threadIdx.x] = 0;
    }
}

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

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" opw_status opw_ag_gemm_noalloc(const opw_symm* symm, size_t a_off, int64_t M_r,
                                          int64_t N, int64_t K, const void* B_dev, void* G_dev,
                                          void* C_dev, int32_t* status_dev, const opw_opts* opts_in,
                                          void* stream)
{
    // ---- arguments, all before any CUDA call
    if (symm == nullptr || symm->heap_dev == nullptr || symm->rank_off == nullptr ||
        symm->R < 1 || symm->R > OPW_MAX_RANKS || symm->reserved != 0)
        return OPW_ERR_INVALID_ARG;
    if (B_dev == nullptr || G_dev == nullptr || C_dev == nullptr || status_dev == nullptr)
        return OPW_ERR_INVALID_ARG;
    opw_opts o;
    std::memset(&o, 0, sizeof o);
    if (opts_in != nullptr) o = *opts_in;
    if (o.role != OPW_ROLE_FUSED) return OPW_ERR_INVALID_ARG;  // no epochs persist between calls
    if (o.sync_mode != OPW_SYNC_OVERLAP && o.sync_mode != OPW_SYNC_SERIAL &&
        o.sync_mode != OPW_SYNC_CHECKED)
        return OPW_ERR_INVALID_ARG;
    if (o.schedule != OPW_SCHED_SWIZZLE && o.schedule != OPW_SCHED_READY) return OPW_ERR_INVALID_ARG;
    if (o.fault_kind < OPW_FAULT_NONE || o.fault_kind > OPW_FAULT_STALE_EPOCH) return OPW_ERR_INVALID_ARG;
    if (o.num_ctas < 0) return OPW_ERR_INVALID_ARG;
    if ((o.signal_mode != OPW_SIGNAL_TILE_SET && o.signal_mode != OPW_SIGNAL_ROW_ADD) ||
        o.reserved != 0)
        return OPW_ERR_INVALID_ARG;
    const int R = symm->R;
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
    const int64_t F = static_cast<int64_t>(R) * (M_r / ft) * (K / ft);
    if (F > kMaxFlags) return OPW_ERR_UNSUPPORTED_SHAPE;  // beyond the fixed scratch
    if (!aligned16(symm->heap_dev) || !aligned16(B_dev) || !aligned16(G_dev) || !aligned16(C_dev) ||
        !aligned16(status_dev) || (a_off & 15u) != 0 ||
        (o.trace_dev != nullptr && (reinterpret_cast<uintptr_t>(o.trace_dev) & 7u) != 0))
        return OPW_ERR_MISALIGNED;
    for (int r = 0; r < R; ++r) {
        if (symm->rank_off[r] < 0) return OPW_ERR_INVALID_ARG;
        if ((symm->rank_off[r] & 15) != 0) return OPW_ERR_MISALIGNED;
    }

    // ---- set-up for this device (first call only), then the launches
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return OPW_ERR_CUDA;
    void* scratch = nullptr;
    if (scratch_for_device(dev, &scratch) != cudaSuccess) return OPW_ERR_CUDA;
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return OPW_ERR_CUDA;
    const int grid = (o.num_ctas > 0 && o.num_ctas < sms) ? o.num_ctas : sms;
    const int max_pairs = ag_max_pairs();
    if (max_pairs <= 0) return OPW_ERR_CUDA;
    int pairs = grid / 2 > 0 ? grid / 2 : 1;
    if (pairs > max_pairs) pairs = max_pairs;

    int64_t* flags = static_cast<int64_t*>(scratch);
    unsigned long long* counters = static_cast<unsigned long long*>(scratch) + kMaxFlags;

    AgParams p;
    std::memset(&p, 0, sizeof p);
    char* heap = static_cast<char*>(symm->heap_dev);
    for (int r = 0; r < R; ++r)
        if (!make_map(&p.shard[r], heap + symm->rank_off[r] + a_off, K, M_r, static_cast<uint32_t>(ft),
                      GATHER_SUB_ROWS, CU_TENSOR_MAP_SWIZZLE_NONE))
            return OPW_ERR_CUDA;
    if (!make_map(&p.g_store, G_dev, K, M, static_cast<uint32_t>(ft), GATHER_SUB_ROWS,
                  CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&p.g_load, G_dev, K, M, 64, BM, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&p.b_load, B_dev, N, K, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&p.c_store, C_dev, N, M, 64, 32, CU_TENSOR_MAP_SWIZZLE_128B))
        return OPW_ERR_CUDA;
    p.flags = flags;
    p.status = status_dev;
    p.counters = counters;
    p.trace = o.trace_dev;
    p.epoch = 1;  // flags were just cleared to 0
    p.timeout_ns = o.timeout_ns != 0 ? o.timeout_ns : 2000000000ull;
    p.claim_base = 0;
    p.R = R;
    p.M_r = static_cast<int32_t>(M_r);
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.ft = static_cast<int32_t>(ft);
    p.T_mr = static_cast<int32_t>(M_r / ft);
    p.T_k = static_cast<int32_t>(K / ft);
    p.T_M = static_cast<int32_t>((M + PAIR_M - 1) / PAIR_M);
    p.T_N = static_cast<int32_t>((N + BN - 1) / BN);
    p.role = OPW_ROLE_FUSED;
    p.sync_mode = o.sync_mode;
    p.schedule = o.schedule;
    // Row groups only pay when B (K x N bf16) is too big to stay in L2.
    p.group_rows = (K * N * 2 > (int64_t(64) << 20)) ? 8 : 1;
    p.signal_mode = o.signal_mode;
    p.has_perm = o.publish_perm != nullptr;
    p.has_delay = o.delay_ns != nullptr;
    p.fault_kind = o.fault_kind;
    p.fault_arg = o.fault_arg;
    for (int i = 0; i < R; ++i) {
        p.perm[i] = o.publish_perm != nullptr ? o.publish_perm[i] : i;
        p.delay_ns[i] = o.delay_ns != nullptr ? o.delay_ns[i] : 0u;
        p.rank_target[i] = static_cast<uint64_t>(p.T_mr) * p.T_k;
    }

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int blocks = static_cast<int>((F + 255) / 256);
    if (blocks < 1) blocks = 1;
    noalloc_clear_kernel<<<blocks, 256, 0, st>>>(flags, F, counters, status_dev);
    if (cudaGetLastError() != cudaSuccess) return OPW_ERR_CUDA;
    if (launch_ag_gemm(p, pairs, st) != cudaSuccess) return OPW_ERR_CUDA;
    return OPW_OK;
}
