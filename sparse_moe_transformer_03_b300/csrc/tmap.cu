// tmap.cu -- host-side encoding of TMA tensor maps (2-D bf16, 128-byte
// swizzle) through the driver entry point, so the library does not link
// libcuda directly.
#include <cudaTypedefs.h>

#include "flint_internal.h"

namespace flint {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// A row-major bf16 matrix [rows][cols] (row pitch in elements); boxes of
// box_rows x box_cols elements, 128-byte swizzle (box_cols * 2 must be 128).
bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t pitch,
                    uint32_t box_rows, uint32_t box_cols) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[2] = {cols, rows};
    cuuint64_t gstride[1] = {pitch * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estride[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), gdim, gstride, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The handle's tiled experts (repack.cu) as a 4-D bf16 tensor whose
// innermost line is four tile rows (512 bytes, contiguous in a tile): 256
// elements x 32 row quads x 384 tiles (256 gate/up tiles, then 128 down
// tiles) x 257 experts, no swizzle (the bytes are already in the tensor
// core's order).  A box of box_quads quads x box_tiles consecutive tiles
// lands in shared memory as [tile][quad][512 bytes]; each 512-byte line is
// one request of the copy engine.
bool encode_tiled_experts_4d(CUtensorMap* map, const void* tiled, uint32_t box_quads, uint32_t box_tiles) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[4] = {256, 32, 384, 257};
    cuuint64_t gstride[3] = {512, 16384, (cuuint64_t)384 * 16384};
    cuuint32_t box[4] = {256, box_quads, box_tiles, 1};
    cuuint32_t estride[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(tiled), gdim, gstride, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The owned NVFP4 experts (decode_nvfp4.cu) viewed as 32-bit words, so a
// 512-byte line of codes is one 128-element box row.  Gate/up view: 1152
// words of a 4608-byte chunk x 4 chunks of a unit x 64 units x 257 experts;
// a box of box_words x 1 chunk x box_units units.  Down view: 1152 words x
// 128 units x 257 experts from the down part of expert 0; a box of box_words
// x box_units units.  No swizzle: the bytes land as stored.
static bool encode_u32(CUtensorMap* map, const void* base, int rank, const cuuint64_t* gdim,
                       const cuuint64_t* gstride, const cuuint32_t* box) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint32_t estride[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, rank, const_cast<void*>(base), gdim, gstride, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_u32_rows(CUtensorMap* map, const void* base, uint64_t rows, uint32_t row_words, uint32_t box_rows) {
    const cuuint64_t gdim[2] = {row_words, rows};
    const cuuint64_t gstride[1] = {(cuuint64_t)row_words * 4};
    const cuuint32_t box[2] = {row_words, box_rows};
    return encode_u32(map, base, 2, gdim, gstride, box);
}

bool encode_nvfp4_gateup(CUtensorMap* map, const uint8_t* nv, uint32_t box_words, uint32_t box_units) {
    const cuuint64_t gdim[4] = {NV_CHUNK / 4, NV_GU_CHUNKS, NV_GU_UNITS, NEXP};
    const cuuint64_t gstride[3] = {NV_CHUNK, (cuuint64_t)NV_GU_CHUNKS * NV_CHUNK, NV_EXPERT_BYTES};
    const cuuint32_t box[4] = {box_words, 1, box_units, 1};
    return encode_u32(map, nv, 4, gdim, gstride, box);
}

bool encode_nvfp4_down(CUtensorMap* map, const uint8_t* nv, uint32_t box_words, uint32_t box_units) {
    const cuuint64_t gdim[3] = {NV_CHUNK / 4, NV_DN_UNITS, NEXP};
    const cuuint64_t gstride[2] = {NV_CHUNK, NV_EXPERT_BYTES};
    const cuuint32_t box[3] = {box_words, box_units, 1};
    return encode_u32(map, nv + NV_GU_BYTES, 3, gdim, gstride, box);
}

}  // namespace flint
