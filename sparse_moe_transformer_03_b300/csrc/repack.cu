// repack.cu -- layouts the handle owns, built once at create time.
//
// Tiled copy of every bf16 expert matrix for the tensor-core path.  The
// matrix [R][K] is cut into tiles of 128 rows x 64 columns, stored one after
// another in (row block, column chunk) order; inside a tile row r's 16-byte
// chunk c sits at r*128 + ((c ^ (r % 8)) * 16), which is the 128-byte-swizzled
// K-major layout the tensor core reads from shared memory.  A pipeline stage
// is then one contiguous 16 KiB cp.async.bulk copy per tile, streamed from
// HBM in full.
#include "flint_common.cuh"
#include "flint_internal.h"

namespace flint {

// one thread per 16-byte chunk of the output
__global__ void __launch_bounds__(256) repack_tiled_kernel(const __nv_bfloat16* __restrict__ in,
                                                          __nv_bfloat16* __restrict__ out, int R, int K) {
    const size_t n16 = (size_t)R * K / 8;
    const int KC = K / 64;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n16; i += (size_t)gridDim.x * blockDim.x) {
        const int cd = (int)(i & 7), r = (int)((i >> 3) & 127);
        const size_t t = i >> 10;
        const size_t kc = t % KC, rb = t / KC;
        const int c = cd ^ (r & 7);   // source chunk stored at swizzled position cd
        const size_t row = rb * 128 + r, col = kc * 64 + (size_t)c * 8;
        reinterpret_cast<uint4*>(out)[i] = reinterpret_cast<const uint4*>(in + row * K + col)[0];
    }
}

cudaError_t launch_repack_tiled(const __nv_bfloat16* in, __nv_bfloat16* out, int R, int K, cudaStream_t s) {
    const size_t n16 = (size_t)R * K / 8;
    int grid = (int)((n16 + 255) / 256);
    if (grid > 148 * 32) grid = 148 * 32;
    repack_tiled_kernel<<<grid, 256, 0, s>>>(in, out, R, K);
    return cudaGetLastError();
}

}  // namespace flint
