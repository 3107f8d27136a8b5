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

#include <cstdint>
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

// True if `ptr` is device (or managed) memory that device `dev` owns.  A
// failed query leaves no error pending for the caller's next CUDA call.
bool on_device(const void* ptr, int dev)
{
    cudaPointerAttributes a;
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) && a.device == dev;
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


}  // namespace

extern "C" opw_status opw_ag_gemm_noalloc(const opw_symm* symm, size_t a_off, int64_t M_r,
                                          int64_t N, int64_t K, const void* B_dev, void* G_dev,
                                          void* C_dev, int32_t* status_dev, const opw_opts* opts_in,
                                          void* stream)
{
    // ---- arguments, all before any CUDA call
    opw_opts o;
    opw_opts_default(&o);
    if (opts_in != nullptr) o = *opts_in;
    if (status_dev == nullptr) return OPW_ERR_INVALID_ARG;
    if (o.role != OPW_ROLE_FUSED) return OPW_ERR_INVALID_ARG;  // no epochs persist between calls
    int64_t ft = 0;
    const opw_status st_args = ag_check_args(symm, a_off, M_r, N, K, B_dev, G_dev, C_dev, o, &ft);
    if (st_args != OPW_OK) return st_args;
    const int R = symm->R;
    const bool row_add = o.signal_mode == OPW_SIGNAL_ROW_ADD;
    const int64_t F = static_cast<int64_t>(R) * (M_r / ft) * (row_add ? 1 : K / ft);
    if (F > kMaxFlags) return OPW_ERR_UNSUPPORTED_SHAPE;  // beyond the fixed scratch
    if ((reinterpret_cast<uintptr_t>(status_dev) & 15u) != 0) return OPW_ERR_MISALIGNED;

    // ---- set-up for this device (first call only), then the launches
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return OPW_ERR_CUDA;
    // The kernels run with this device's scratch: every buffer must be this
    // device's memory too.
    if (!on_device(status_dev, dev) || !on_device(symm->heap_dev, dev) || !on_device(B_dev, dev) ||
        !on_device(G_dev, dev) || !on_device(C_dev, dev))
        return OPW_ERR_INVALID_ARG;
    void* scratch = nullptr;
    if (scratch_for_device(dev, &scratch) != cudaSuccess) return OPW_ERR_CUDA;
    const int pairs = ag_pairs_for(o, dev);
    if (pairs <= 0) return OPW_ERR_CUDA;

    int64_t* flags = static_cast<int64_t*>(scratch);
    unsigned long long* counters = static_cast<unsigned long long*>(scratch) + kMaxFlags;
    AgParams p;
    const int tile_n = ag_tile_n_for(o, pairs, static_cast<int64_t>(symm->R) * M_r, N);
    const opw_status st_params =
        ag_fill_params(symm, a_off, M_r, N, K, ft, B_dev, G_dev, C_dev, o, tile_n, &p);
    if (st_params != OPW_OK) return st_params;
    p.flags = flags;
    p.status = status_dev;
    p.counters = counters;
    p.epoch = 1;  // flags were just cleared to 0
    p.claim_base = 0;
    p.gather_base = 0;
    for (int i = 0; i < R; ++i) p.rank_target[i] = static_cast<uint64_t>(p.T_mr) * p.T_k;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int blocks = static_cast<int>((F + 255) / 256);
    if (blocks < 1) blocks = 1;
    noalloc_clear_kernel<<<blocks, 256, 0, st>>>(flags, F, counters, status_dev);
    if (cudaGetLastError() != cudaSuccess) return OPW_ERR_CUDA;
    if (launch_ag_gemm(p, pairs, st) != cudaSuccess) return OPW_ERR_CUDA;
    return OPW_OK;
}
