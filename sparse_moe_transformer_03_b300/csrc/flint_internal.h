// flint_internal.h -- host-side declarations shared by the library's .cu files.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "flint_common.cuh"

namespace flint {

// Launch context of one API call.
struct LaunchCtx {
    cudaStream_t stream;
    uint32_t* status;      // device view of the handle's host-mapped status word
    uint64_t wait_limit_ns;
    int num_sms;
    bool pdl;              // launch kernels as programmatic dependents
    int prof_kernel;       // flint_kernel_t whose launch is bracketed by the events below, or -1
    cudaEvent_t prof_start, prof_stop;
};

// Launch `kern` on L.stream, as a programmatic dependent of the previous
// kernel on the stream when L.pdl is set.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(const LaunchCtx& L, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// launch_pdl, with the launch bracketed by L's profiling events when `kid`
// is the kernel the caller asked to time.
template <typename... KArgs, typename... Args>
cudaError_t launch_hooked(const LaunchCtx& L, int kid, void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          Args... args) {
    const bool hook = L.prof_kernel == kid;
    if (hook) {
        const cudaError_t e = cudaEventRecord(L.prof_start, L.stream);
        if (e != cudaSuccess) return e;
    }
    const cudaError_t e = launch_pdl(L, kern, grid, block, smem, args...);
    if (e != cudaSuccess || !hook) return e;
    return cudaEventRecord(L.prof_stop, L.stream);
}

// router.cu
constexpr int PERM_BLOCK_TOKENS = 128;   // tokens per block of the permutation's counting sort
cudaError_t launch_router_logits_decode(const LaunchCtx& L, const __nv_bfloat16* x, int T,
                                        const __nv_bfloat16* Wr, const float* bias, float* logits);
cudaError_t launch_select(const LaunchCtx& L, const float* logits, int T, int32_t* idx, float* w);
cudaError_t launch_permutation(const LaunchCtx& L, const int32_t* idx, int T, int32_t* local_rank,
                               int32_t* blk_counts, int32_t* blk_base, int32_t* offsets, int32_t* gather);
// scan + scatter only (block-local ranks and counts already computed)
cudaError_t launch_perm_scan_scatter(const LaunchCtx& L, const int32_t* idx, int T, const int32_t* local_rank,
                                     const int32_t* blk_counts, int32_t* blk_base, int32_t* offsets,
                                     int32_t* gather, int32_t* pair_slot);

// tmap.cu
bool encode_bf16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t pitch,
                    uint32_t box_rows, uint32_t box_cols);

bool encode_tiled_experts_4d(CUtensorMap* map, const void* tiled, uint32_t box_quads, uint32_t box_tiles);

// repack.cu
cudaError_t launch_repack_tiled(const __nv_bfloat16* in, __nv_bfloat16* out, int R, int K, cudaStream_t s);

// prefill.cu
cudaError_t prefill_set_attributes();
cudaError_t launch_prefill_router(const LaunchCtx& L, const CUtensorMap& x_map, const CUtensorMap& wr_map, int T,
                                  const float* bias, float* logits, int32_t* idx, float* w, int32_t* local_rank,
                                  int32_t* blk_counts);
cudaError_t launch_prefill_experts(const LaunchCtx& L, const __nv_bfloat16* x, const CUtensorMap& h_map, int T,
                                   const int32_t* offsets, const int32_t* gather, const int32_t* pair_slot,
                                   const float* w_route, const __nv_bfloat16* tiled, __nv_bfloat16* h_perm,
                                   __nv_bfloat16* o_perm, __nv_bfloat16* y);
// y[t] = routed slots' outputs x routing weights + the shared slot, fixed order
cudaError_t launch_prefill_combine(const LaunchCtx& L, const __nv_bfloat16* o_perm, const int32_t* pair_slot,
                                   const float* w_route, int T, __nv_bfloat16* y);

// decode_nvfp4.cu -- owned NVFP4 expert layout.  A chunk holds 16 matrix
// rows x 512 columns (32 blocks of 16 columns): 32 x 128 bytes of E2M1 codes
// in mma.sync A-fragment order, then 32 x 16 bytes of E4M3 block scales.
// Per expert: 64 gate/up units (gate rows 8u..8u+7 and up rows 8u..8u+7) of
// 4 chunks each (K = 2048), then 128 down units (rows 16v..16v+15) of one
// chunk (K = 512).
constexpr int NV_CHUNK_KB = 32;                          // 16-column blocks per chunk
constexpr int NV_CODES = NV_CHUNK_KB * 128;              // 4096
constexpr int NV_CHUNK = NV_CODES + NV_CHUNK_KB * 16;    // 4608
constexpr int NV_GU_UNITS = I / 8;                       // 64
constexpr int NV_GU_CHUNKS = H / (16 * NV_CHUNK_KB);     // 4
constexpr int NV_DN_UNITS = H / 16;                      // 128
constexpr size_t NV_GU_BYTES = (size_t)NV_GU_UNITS * NV_GU_CHUNKS * NV_CHUNK;   // 1,179,648
constexpr size_t NV_DN_BYTES = (size_t)NV_DN_UNITS * NV_CHUNK;                 // 589,824
constexpr size_t NV_EXPERT_BYTES = NV_GU_BYTES + NV_DN_BYTES;                  // 1,769,472

// kind 0: a gate_up matrix, 1: a down matrix, 2: any [rows][H] matrix (rows a
// multiple of 16) as rows/16 units of 16 straight rows x 4 chunks
cudaError_t launch_repack_nvfp4(const uint8_t* packed, const uint8_t* scales, int kind, int rows, uint8_t* out,
                                cudaStream_t s);
cudaError_t decode_nvfp4_set_attributes();
cudaError_t launch_decode_experts_nvfp4(const LaunchCtx& L, const uint8_t* nv, const float* nv_ts,
                                        const float* logits, const __nv_bfloat16* x, int T, DecodeTables* tables,
                                        int32_t* idx, float* w, __nv_bfloat16* a_buf, __nv_bfloat16* y);

// tmap.cu: the owned NVFP4 experts as TMA tensors of 32-bit words
bool encode_nvfp4_gateup(CUtensorMap* map, const uint8_t* nv, uint32_t box_words, uint32_t box_units);
bool encode_nvfp4_down(CUtensorMap* map, const uint8_t* nv, uint32_t box_words, uint32_t box_units);
// a [rows][row_words] array of 32-bit words, boxes of row_words x box_rows, no swizzle
bool encode_u32_rows(CUtensorMap* map, const void* base, uint64_t rows, uint32_t row_words, uint32_t box_rows);

// prefill_nvfp4.cu -- grouped tcgen05 GEMMs with the NVFP4 weight operand
// dequantised in shared memory.  maps: gate/up codes, gate/up scales, down
// codes, down scales (encode_nvfp4_prefill_maps).
cudaError_t prefill_nvfp4_set_attributes();
bool encode_nvfp4_prefill_maps(CUtensorMap (&maps)[4], const uint8_t* nv);
cudaError_t launch_prefill_experts_nvfp4(const LaunchCtx& L, const __nv_bfloat16* x, const CUtensorMap& h_map,
                                         const CUtensorMap (&maps)[4], int T, const int32_t* offsets,
                                         const int32_t* gather, const int32_t* pair_slot, const float* w_route,
                                         const float* nv_ts, __nv_bfloat16* h_perm, __nv_bfloat16* o_perm,
                                         __nv_bfloat16* y);

// stack_decode.cu -- every layer of a stack in one persistent launch (bf16 or
// NVFP4 experts, T <= STACK_MAX_T).  Layer l reads x of its own and writes its y; layer l
// starts only after every CTA finished layer l - 1, so x[l] may be y[l - 1].
constexpr int STACK_MAX_T = 8;
constexpr int STACK_MAX_LAYERS = 64;
struct StackLayerArgs {
    const CUtensorMap* maps;         // bf16: the layer's tiled experts as 4-D tensor maps (device memory):
                                     // [0] gate/up boxes (8 rows x 16 tiles), [1] down boxes (16 rows x 8 tiles)
    const uint8_t* nv;               // NVFP4: the layer's owned experts (NV_EXPERT_BYTES each)
    const float* nv_ts;              // NVFP4: tensor scales [NEXP][2] (gate_up, down)
    const __nv_bfloat16* router;     // [E][H]
    const float* bias;               // [E] or null
    const __nv_bfloat16* x;          // [T][H]
    __nv_bfloat16* y;                // [T][H]
};
struct StackParams {
    StackLayerArgs layer[STACK_MAX_LAYERS];
    int n_layers, T;
    int nvfp4;                       // the layers' expert format: 0 bf16, 1 NVFP4
    uint32_t smem_bytes;             // the device's opt-in shared memory per block
    float* logits;                   // [STACK_MAX_T][E] router logits (scratch)
    __nv_bfloat16* act;              // [STACK_MAX_T * 7][I] activations, chunk-swizzled rows (scratch)
    unsigned long long* bar;         // grid barrier counter (scratch)
    uint32_t* abort_flag;            // set by a CTA whose bounded wait ran out
    uint32_t* status;
    uint64_t limit_ns;
};
// scratch of a stack launch inside a handle's workspace: logits,
// activations, barrier counter and abort flag, contiguous (cleared together
// after a device error)
constexpr size_t STACK_LOGITS_BYTES = (size_t)STACK_MAX_T * E * 4;
constexpr size_t STACK_ACT_BYTES = (size_t)STACK_MAX_T * (TOPK + 1) * I * 2;
constexpr size_t STACK_CLEAR_BYTES = STACK_LOGITS_BYTES + STACK_ACT_BYTES + 16;
cudaError_t stack_decode_set_attributes(int max_optin);
cudaError_t launch_stack_decode(const LaunchCtx& L, StackParams& p, int max_optin);

// decode_mma.cu -- bf16 decode (T <= DEC_T) on mma.sync, from the tiled copy
cudaError_t decode_mma_set_attributes();
cudaError_t launch_decode_experts_mma(const LaunchCtx& L, const uint8_t* tiled, const float* logits,
                                      const __nv_bfloat16* x, int T, DecodeTables* tables, int32_t* idx, float* w,
                                      __nv_bfloat16* a_buf, __nv_bfloat16* y);

}  // namespace flint
