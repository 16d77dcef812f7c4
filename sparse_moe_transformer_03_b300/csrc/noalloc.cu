// noalloc.cu -- flint_permute_static: the expert permutation (a stable
// counting sort of the (token, slot) pairs by expert) with its scratch in one
// fixed array of device memory that this file declares, instead of in a
// layer handle's workspace.
//
// It serves callers that may not allocate device memory at the point where
// they route: an allocator-free serving loop that reserves all of its memory
// up front, or a caller running under an external memory pool that forbids
// cudaMalloc in the request path.  Nothing here calls cudaMalloc, cudaFree or
// any routine that allocates; the scratch is a module global, sized for the
// largest request (FLINT_CHUNK tokens), and all calls on a device share it.
#include <mutex>

#include "../../include/flint_moe.h"
#include "flint_common.cuh"
#include "flint_internal.h"

using namespace flint;

namespace {

constexpr int NA_MAX_T = FLINT_CHUNK;
constexpr int NA_MAX_BLK = (NA_MAX_T + PERM_BLOCK_TOKENS - 1) / PERM_BLOCK_TOKENS;

// byte offsets inside the scratch array (each 256-byte aligned)
constexpr size_t NA_STATUS = 0;                                          // uint32 status word
constexpr size_t NA_RANK = 256;                                          // int32 [NA_MAX_T * TOPK]
constexpr size_t NA_COUNTS = NA_RANK + (size_t)NA_MAX_T * TOPK * 4;      // int32 [NA_MAX_BLK * E]
constexpr size_t NA_BASE = NA_COUNTS + (size_t)NA_MAX_BLK * E * 4;       // int32 [NA_MAX_BLK * E]
constexpr size_t NA_BYTES = NA_BASE + (size_t)NA_MAX_BLK * E * 4;        // 327,936 bytes
static_assert(NA_RANK % 256 == 0 && NA_COUNTS % 256 == 0 && NA_BASE % 256 == 0, "scratch carve alignment");

// Zero at module load.  Only the status word has to start at zero: the
// counting sort writes every rank, count and base it later reads.
static __device__ __align__(256) unsigned char g_perm_scratch[NA_BYTES];

constexpr int NA_MAX_DEVICES = 64;
std::mutex g_setup_mu;
unsigned char* g_scratch_ptr[NA_MAX_DEVICES] = {};

// Device address of the scratch array on the current device, looked up once
// per device (the lookup loads the module on that device).
cudaError_t scratch_for_current_device(unsigned char** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= NA_MAX_DEVICES) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (!g_scratch_ptr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_perm_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = static_cast<unsigned char*>(p);
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" flint_status_t flint_permute_static(const int32_t* idx, int T, int32_t* offsets, int32_t* gather_idx,
                                               cudaStream_t s) {
    if (!idx || !offsets || !gather_idx || T < 1) return FLINT_ERR_INVALID_ARG;
    if (T > NA_MAX_T) return FLINT_ERR_INVALID_ARG;   // beyond the fixed scratch
    if (!aligned4(idx) || !aligned4(offsets) || !aligned4(gather_idx)) return FLINT_ERR_INVALID_ARG;

    unsigned char* base = nullptr;
    if (scratch_for_current_device(&base) != cudaSuccess) return FLINT_ERR_CUDA;
    uint32_t* status = reinterpret_cast<uint32_t*>(base + NA_STATUS);

    LaunchCtx L;
    L.stream = s;
    L.status = status;
    L.wait_limit_ns = 1000000000ull;
    L.num_sms = 0;
    L.pdl = true;
    L.prof_kernel = -1;
    L.prof_start = L.prof_stop = nullptr;
    cudaError_t e = launch_permutation(L, idx, T, reinterpret_cast<int32_t*>(base + NA_RANK),
                                       reinterpret_cast<int32_t*>(base + NA_COUNTS),
                                       reinterpret_cast<int32_t*>(base + NA_BASE), offsets, gather_idx);
    uint32_t st = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&st, status, sizeof st, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return FLINT_ERR_CUDA;
    if (st != 0) {
        // clear it for the next call
        if (cudaMemsetAsync(status, 0, sizeof st, s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess)
            return FLINT_ERR_CUDA;
        return st == ST_BADINDEX ? FLINT_ERR_DEVICE_BADINDEX : FLINT_ERR_CUDA;
    }
    return FLINT_OK;
}
