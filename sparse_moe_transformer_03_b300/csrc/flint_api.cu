// flint_api.cu -- the C ABI (include/flint_moe.h): handle creation, argument
// checking, workspace, dispatch between the decode and the grouped
// tensor-core paths, and the device status word.
#include <cstdlib>
#include <cstring>
#include <new>

#include "../../include/flint_moe.h"
#include "flint_common.cuh"
#include "flint_internal.h"

using namespace flint;

struct flint_moe {
    flint_dtype_t dtype;
    int device;
    int num_sms;
    int smem_optin;                // opt-in shared memory per block of the device
    uint64_t wait_limit_ns;
    int prof_kernel;               // profiling hook (flint_moe_set_kernel_events), -1 when unset
    cudaEvent_t prof_start, prof_stop;

    // weights
    const __nv_bfloat16* router_W;
    const float* router_b;
    // owned tiled copies of the expert matrices for the tensor-core path
    // (per expert: gate_up tiles then down tiles, see repack.cu); bf16 only
    __nv_bfloat16* tiled;
    // NVFP4: owned repacked experts (NV_EXPERT_BYTES each) and tensor scales [NEXP][2]
    uint8_t* nv;
    float* nv_ts;
    CUtensorMap nv_maps[4];        // NVFP4: gate/up codes and scales, down codes and scales (prefill boxes)
    CUtensorMap wr_map;            // router, boxes 64 x 256
    CUtensorMap h_map;             // h_perm, boxes 64 x 256

    // status word in host-mapped memory
    uint32_t* status_host;
    uint32_t* status_dev;

    // workspace
    void* ws_base;
    size_t ws_bytes;
    float* logits;                 // [CHUNK][E]
    int32_t* idx;                  // [CHUNK][TOPK]
    float* w;                      // [CHUNK][TOPK]
    DecodeTables* dec_tables;
    __nv_bfloat16* a_dec;          // decode activations (act_index layout)
    int32_t* local_rank;           // [CHUNK][TOPK]
    int32_t* blk_counts;           // [CHUNK/128][E]
    int32_t* blk_base;             // [CHUNK/128][E]
    int32_t* offsets;              // [E+1]
    int32_t* gather;               // [CHUNK*TOPK]
    int32_t* pair_slot;            // [CHUNK*TOPK] slot of each (token, choice) pair
    __nv_bfloat16* h_perm;         // [(TOPK+1)*CHUNK][I]
    __nv_bfloat16* o_perm;         // [(TOPK+1)*CHUNK][H]
    // scratch of flint_moe_forward_layers when this handle is layers[0]
    unsigned char* stack_clear;    // tagged logits and activations, barrier counter, abort flag
    CUtensorMap* stack_maps;       // [2] this layer's tiled experts as 4-D tensor maps (bf16 handles)
};

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

flint_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? FLINT_OK : FLINT_ERR_CUDA; }

// Take (and clear) a device status left by an earlier call.
flint_status_t take_device_status(flint_moe* h) {
    volatile uint32_t* s = h->status_host;
    const uint32_t v = *s;
    if (v == 0) return FLINT_OK;
    *s = 0;
    if (v == ST_TIMEOUT) return FLINT_ERR_DEVICE_TIMEOUT;
    if (v == ST_BADINDEX) return FLINT_ERR_DEVICE_BADINDEX;
    if (v == ST_INTERNAL) return FLINT_ERR_INTERNAL;
    return FLINT_ERR_CUDA;
}

LaunchCtx ctx_of(const flint_moe* h, cudaStream_t s) {
    LaunchCtx L;
    L.stream = s;
    L.status = h->status_dev;
    L.wait_limit_ns = h->wait_limit_ns;
    L.num_sms = h->num_sms;
    L.pdl = true;
    L.prof_kernel = h->prof_kernel;
    L.prof_start = h->prof_start;
    L.prof_stop = h->prof_stop;
    return L;
}

// Bump allocator over one cudaMalloc.
struct Carve {
    char* base;
    size_t off;
    template <typename T>
    T* take(size_t count) {
        off = (off + 255) & ~size_t(255);
        T* p = reinterpret_cast<T*>(base + off);
        off += count * sizeof(T);
        return p;
    }
};

void free_handle(flint_moe* h) {
    if (!h) return;
    if (h->ws_base) cudaFree(h->ws_base);
    if (h->tiled) cudaFree(h->tiled);
    if (h->nv) cudaFree(h->nv);
    if (h->nv_ts) cudaFree(h->nv_ts);
    if (h->status_host) cudaFreeHost(h->status_host);
    delete h;
}

void carve_workspace(flint_moe* h, char* base, size_t* bytes_out) {
    Carve c{base, 0};
    h->logits = c.take<float>((size_t)CHUNK * E);
    h->idx = c.take<int32_t>((size_t)CHUNK * TOPK);
    h->w = c.take<float>((size_t)CHUNK * TOPK);
    h->dec_tables = c.take<DecodeTables>(1);
    h->a_dec = c.take<__nv_bfloat16>(DEC_ACT_BYTES / 2);
    h->local_rank = c.take<int32_t>((size_t)CHUNK * TOPK);
    h->blk_counts = c.take<int32_t>((size_t)(CHUNK / 128) * E);
    h->blk_base = c.take<int32_t>((size_t)(CHUNK / 128) * E);
    h->offsets = c.take<int32_t>(E + 1);
    h->gather = c.take<int32_t>((size_t)CHUNK * TOPK);
    h->pair_slot = c.take<int32_t>((size_t)CHUNK * TOPK);
    h->h_perm = c.take<__nv_bfloat16>((size_t)(TOPK + 1) * CHUNK * I);
    h->o_perm = c.take<__nv_bfloat16>((size_t)(TOPK + 1) * CHUNK * H);
    h->stack_clear = c.take<unsigned char>(STACK_CLEAR_BYTES);
    h->stack_maps = c.take<CUtensorMap>(2);
    *bytes_out = c.off;
}

}  // namespace

extern "C" {

const char* flint_status_string(flint_status_t st) {
    switch (st) {
        case FLINT_OK: return "FLINT_OK";
        case FLINT_ERR_INVALID_ARG: return "FLINT_ERR_INVALID_ARG";
        case FLINT_ERR_CUDA: return "FLINT_ERR_CUDA";
        case FLINT_ERR_OOM: return "FLINT_ERR_OOM";
        case FLINT_ERR_DEVICE_TIMEOUT: return "FLINT_ERR_DEVICE_TIMEOUT";
        case FLINT_ERR_DEVICE_BADINDEX: return "FLINT_ERR_DEVICE_BADINDEX";
        case FLINT_ERR_UNSUPPORTED: return "FLINT_ERR_UNSUPPORTED";
        case FLINT_ERR_INTERNAL: return "FLINT_ERR_INTERNAL";
    }
    return "FLINT_ERR_UNKNOWN";
}

flint_status_t flint_moe_create(flint_moe_t* out, const void* router_W, const float* router_b,
                                const void* const* gate_up_W, const void* const* down_W,
                                const void* const* shared_W, flint_dtype_t dtype) {
    if (!out) return FLINT_ERR_INVALID_ARG;
    *out = nullptr;
    if (!router_W || !gate_up_W || !down_W || !shared_W) return FLINT_ERR_INVALID_ARG;
    if (dtype != FLINT_BF16 && dtype != FLINT_NVFP4) return FLINT_ERR_INVALID_ARG;
    if (!aligned16(router_W) || (router_b && !aligned16(router_b))) return FLINT_ERR_INVALID_ARG;
    for (int e = 0; e < NEXP; ++e) {
        const void* gu = e < E ? gate_up_W[e] : shared_W[0];
        const void* dn = e < E ? down_W[e] : shared_W[1];
        if (!gu || !dn) return FLINT_ERR_INVALID_ARG;
        if (dtype == FLINT_BF16 && (!aligned16(gu) || !aligned16(dn))) return FLINT_ERR_INVALID_ARG;
        if (dtype == FLINT_NVFP4) {
            const flint_nvfp4_t* mg = static_cast<const flint_nvfp4_t*>(gu);
            const flint_nvfp4_t* md = static_cast<const flint_nvfp4_t*>(dn);
            if (!mg->packed || !mg->block_scales || !md->packed || !md->block_scales) return FLINT_ERR_INVALID_ARG;
        }
    }

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FLINT_ERR_CUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return FLINT_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return FLINT_ERR_UNSUPPORTED;

    flint_moe* h = new (std::nothrow) flint_moe();
    if (!h) return FLINT_ERR_OOM;
    std::memset(h, 0, sizeof(*h));
    h->dtype = dtype;
    h->device = dev;
    h->num_sms = prop.multiProcessorCount;
    h->smem_optin = (int)prop.sharedMemPerBlockOptin;
    h->wait_limit_ns = 1000000000ull;   // one second
    h->prof_kernel = -1;
    h->router_W = static_cast<const __nv_bfloat16*>(router_W);
    h->router_b = router_b;

    flint_status_t st = FLINT_OK;
    {
        if (cudaHostAlloc(reinterpret_cast<void**>(&h->status_host), 64, cudaHostAllocMapped) != cudaSuccess)
            st = FLINT_ERR_OOM;
        else {
            *h->status_host = 0;
            if (cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->status_dev), h->status_host, 0) !=
                cudaSuccess)
                st = FLINT_ERR_CUDA;
        }
    }
    if (st == FLINT_OK) {
        size_t bytes = 0;
        carve_workspace(h, nullptr, &bytes);
        if (cudaMalloc(&h->ws_base, bytes) != cudaSuccess)
            st = FLINT_ERR_OOM;
        else {
            h->ws_bytes = bytes;
            carve_workspace(h, static_cast<char*>(h->ws_base), &bytes);
            if (cudaMemset(h->ws_base, 0, bytes) != cudaSuccess) st = FLINT_ERR_CUDA;
        }
    }
    const size_t expert_elems = (size_t)3 * H * I;   // gate_up + down
    if (st == FLINT_OK && dtype == FLINT_NVFP4) {
        // repack every expert into the owned chunk layout; keep the tensor scales
        float ts[NEXP * 2];
        if (cudaMalloc(&h->nv, (size_t)NEXP * NV_EXPERT_BYTES) != cudaSuccess ||
            cudaMalloc(&h->nv_ts, sizeof ts) != cudaSuccess)
            st = FLINT_ERR_OOM;
        for (int e = 0; st == FLINT_OK && e < NEXP; ++e) {
            const flint_nvfp4_t* mg = static_cast<const flint_nvfp4_t*>(e < E ? gate_up_W[e] : shared_W[0]);
            const flint_nvfp4_t* md = static_cast<const flint_nvfp4_t*>(e < E ? down_W[e] : shared_W[1]);
            ts[2 * e] = mg->tensor_scale;
            ts[2 * e + 1] = md->tensor_scale;
            uint8_t* b = h->nv + (size_t)e * NV_EXPERT_BYTES;
            if (launch_repack_nvfp4(mg->packed, mg->block_scales, 0, 0, b, 0) != cudaSuccess ||
                launch_repack_nvfp4(md->packed, md->block_scales, 1, 0, b + NV_GU_BYTES, 0) != cudaSuccess)
                st = FLINT_ERR_CUDA;
        }
        if (st == FLINT_OK && cudaMemcpy(h->nv_ts, ts, sizeof ts, cudaMemcpyHostToDevice) != cudaSuccess)
            st = FLINT_ERR_CUDA;
        if (st == FLINT_OK && !encode_nvfp4_prefill_maps(h->nv_maps, h->nv)) st = FLINT_ERR_CUDA;
    }
    if (st == FLINT_OK && dtype == FLINT_BF16) {
        if (cudaMalloc(&h->tiled, (size_t)NEXP * expert_elems * sizeof(__nv_bfloat16)) != cudaSuccess)
            st = FLINT_ERR_OOM;
        // the caller's matrices are read here only
        for (int e = 0; st == FLINT_OK && e < NEXP; ++e) {
            __nv_bfloat16* b = h->tiled + (size_t)e * expert_elems;
            const auto* gu = static_cast<const __nv_bfloat16*>(e < E ? gate_up_W[e] : shared_W[0]);
            const auto* dn = static_cast<const __nv_bfloat16*>(e < E ? down_W[e] : shared_W[1]);
            if (launch_repack_tiled(gu, b, 2 * I, H, 0) != cudaSuccess ||
                launch_repack_tiled(dn, b + (size_t)2 * I * H, H, I, 0) != cudaSuccess)
                st = FLINT_ERR_CUDA;
        }
    }
    if (st == FLINT_OK) {
        // tensor maps of the router and of h_perm
        const bool enc = encode_bf16_2d(&h->wr_map, h->router_W, E, H, H, E, 64) &&
                         encode_bf16_2d(&h->h_map, h->h_perm, (uint64_t)(TOPK + 1) * CHUNK, I, I, 256, 64);
        if (!enc) st = FLINT_ERR_CUDA;
    }
    if (st == FLINT_OK && dtype == FLINT_BF16) {
        // the tiled experts as 4-D tensors for the persistent stack kernel
        CUtensorMap maps[2];
        if (!encode_tiled_experts_4d(&maps[0], h->tiled, 2, 16) || !encode_tiled_experts_4d(&maps[1], h->tiled, 4, 8) ||
            cudaMemcpy(h->stack_maps, maps, sizeof maps, cudaMemcpyHostToDevice) != cudaSuccess)
            st = FLINT_ERR_CUDA;
    }
    if (st == FLINT_OK) st = from_cuda(prefill_set_attributes());
    if (st == FLINT_OK) st = from_cuda(decode_nvfp4_set_attributes());
    if (st == FLINT_OK) st = from_cuda(prefill_nvfp4_set_attributes());
    if (st == FLINT_OK) st = from_cuda(decode_mma_set_attributes());
    if (st == FLINT_OK) st = from_cuda(stack_decode_set_attributes(h->smem_optin));
    if (st == FLINT_OK) st = from_cuda(cudaDeviceSynchronize());
    if (st != FLINT_OK) {
        cudaGetLastError();
        free_handle(h);
        return st;
    }
    *out = h;
    return FLINT_OK;
}

flint_status_t flint_moe_forward(flint_moe_t h, const void* x, int T, void* y, cudaStream_t s) {
    if (!h || !x || !y || T < 1) return FLINT_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(y)) return FLINT_ERR_INVALID_ARG;
    const char* xb = static_cast<const char*>(x);
    const char* yb = static_cast<const char*>(y);
    const size_t bytes = (size_t)T * H * 2;
    if (xb < yb + bytes && yb < xb + bytes) return FLINT_ERR_INVALID_ARG;
    flint_status_t st = take_device_status(h);
    if (st != FLINT_OK) return st;

    const LaunchCtx L = ctx_of(h, s);
    const __nv_bfloat16* xs = static_cast<const __nv_bfloat16*>(x);
    __nv_bfloat16* ys = static_cast<__nv_bfloat16*>(y);
    if (h->dtype == FLINT_NVFP4 && T <= DEC_T) {
        cudaError_t e = launch_router_logits_decode(L, xs, T, h->router_W, h->router_b, h->logits);
        if (e == cudaSuccess)
            e = launch_decode_experts_nvfp4(L, h->nv, h->nv_ts, h->logits, xs, T, h->dec_tables, h->idx, h->w,
                                            h->a_dec, ys);
        return from_cuda(e);
    }
    if (T <= DEC_T) {
        cudaError_t e = launch_router_logits_decode(L, xs, T, h->router_W, h->router_b, h->logits);
        if (e == cudaSuccess)
            e = launch_decode_experts_mma(L, reinterpret_cast<const uint8_t*>(h->tiled), h->logits, xs, T,
                                          h->dec_tables, h->idx, h->w, h->a_dec, ys);
        return from_cuda(e);
    }
    // grouped tensor-core path, chunks of CHUNK tokens
    for (int t0 = 0; t0 < T; t0 += CHUNK) {
        const int Tc = T - t0 < CHUNK ? T - t0 : CHUNK;
        const __nv_bfloat16* xc = xs + (size_t)t0 * H;
        CUtensorMap xmap;
        if (!encode_bf16_2d(&xmap, xc, Tc, H, H, 128, 64)) return FLINT_ERR_CUDA;
        cudaError_t e = launch_prefill_router(L, xmap, h->wr_map, Tc, h->router_b, nullptr, h->idx, h->w,
                                              h->local_rank, h->blk_counts);
        if (e == cudaSuccess)
            e = launch_perm_scan_scatter(L, h->idx, Tc, h->local_rank, h->blk_counts, h->blk_base, h->offsets,
                                         h->gather, h->pair_slot);
        if (e == cudaSuccess) {
            if (h->dtype == FLINT_NVFP4)
                e = launch_prefill_experts_nvfp4(L, xc, h->h_map, h->nv_maps, Tc, h->offsets, h->gather,
                                                 h->pair_slot, h->w, h->nv_ts, h->h_perm, h->o_perm,
                                                 ys + (size_t)t0 * H);
            else
                e = launch_prefill_experts(L, xc, h->h_map, Tc, h->offsets, h->gather, h->pair_slot, h->w,
                                           h->tiled, h->h_perm, h->o_perm, ys + (size_t)t0 * H);
        }
        if (e != cudaSuccess) return FLINT_ERR_CUDA;
    }
    return FLINT_OK;
}

flint_status_t flint_moe_forward_layers(const flint_moe_t* layers, int n, const void* const* x, int T,
                                        void* const* y, cudaStream_t s) {
    if (!layers || !x || !y || n < 1 || T < 1) return FLINT_ERR_INVALID_ARG;
    flint_moe* h0 = layers[0];
    if (!h0) return FLINT_ERR_INVALID_ARG;
    const size_t bytes = (size_t)T * H * 2;
    for (int l = 0; l < n; ++l) {
        const flint_moe* h = layers[l];
        if (!h || h->dtype != h0->dtype || h->device != h0->device) return FLINT_ERR_INVALID_ARG;
        if (!x[l] || !y[l] || !aligned16(x[l]) || !aligned16(y[l])) return FLINT_ERR_INVALID_ARG;
        const char* xb = static_cast<const char*>(x[l]);
        const char* yb = static_cast<const char*>(y[l]);
        if (xb < yb + bytes && yb < xb + bytes) return FLINT_ERR_INVALID_ARG;
    }
    flint_status_t st = take_device_status(h0);
    if (st != FLINT_OK) {
        // a stack launch that gave up may have left its barrier counter and
        // tagged logits mid-way: start the next one from a clean scratch
        if (cudaMemsetAsync(h0->stack_clear, 0, STACK_CLEAR_BYTES, s) != cudaSuccess) return FLINT_ERR_CUDA;
        return st;
    }
    const bool persistent = T <= STACK_MAX_T && h0->num_sms >= 128 && h0->num_sms <= E;
    if (!persistent) {
        // larger batches: one forward per layer, in order
        for (int l = 0; l < n; ++l) {
            st = flint_moe_forward(layers[l], x[l], T, y[l], s);
            if (st != FLINT_OK) return st;
        }
        return FLINT_OK;
    }
    const LaunchCtx L = ctx_of(h0, s);
    for (int l0 = 0; l0 < n; l0 += STACK_MAX_LAYERS) {
        StackParams p;
        std::memset(&p, 0, sizeof p);
        p.n_layers = n - l0 < STACK_MAX_LAYERS ? n - l0 : STACK_MAX_LAYERS;
        p.T = T;
        p.nvfp4 = h0->dtype == FLINT_NVFP4 ? 1 : 0;
        for (int i = 0; i < p.n_layers; ++i) {
            const flint_moe* h = layers[l0 + i];
            p.layer[i].maps = h->stack_maps;
            p.layer[i].nv = h->nv;
            p.layer[i].nv_ts = h->nv_ts;
            p.layer[i].router = h->router_W;
            p.layer[i].bias = h->router_b;
            p.layer[i].x = static_cast<const __nv_bfloat16*>(x[l0 + i]);
            p.layer[i].y = static_cast<__nv_bfloat16*>(y[l0 + i]);
        }
        p.logits = reinterpret_cast<float*>(h0->stack_clear);
        p.act = reinterpret_cast<__nv_bfloat16*>(h0->stack_clear + STACK_LOGITS_BYTES);
        p.bar = reinterpret_cast<unsigned long long*>(h0->stack_clear + STACK_LOGITS_BYTES + STACK_ACT_BYTES);
        p.abort_flag = reinterpret_cast<uint32_t*>(h0->stack_clear + STACK_LOGITS_BYTES + STACK_ACT_BYTES + 8);
        p.status = h0->status_dev;
        p.limit_ns = h0->wait_limit_ns;
        if (launch_stack_decode(L, p, h0->smem_optin) != cudaSuccess) return FLINT_ERR_CUDA;
    }
    return FLINT_OK;
}

flint_status_t flint_moe_route_only(flint_moe_t h, const void* x, float* logits, int T, int32_t* idx,
                                    float* w, int32_t* offsets, int32_t* gather_idx, cudaStream_t s) {
    if (!h || !idx || !w || T < 1 || T > CHUNK) return FLINT_ERR_INVALID_ARG;
    if (!x && !logits) return FLINT_ERR_INVALID_ARG;
    if ((x && !aligned16(x)) || (logits && !aligned16(logits))) return FLINT_ERR_INVALID_ARG;
    flint_status_t st = take_device_status(h);
    if (st != FLINT_OK) return st;

    const LaunchCtx L = ctx_of(h, s);
    cudaError_t e = cudaSuccess;
    if (x) {
        float* lg = logits ? logits : h->logits;
        const __nv_bfloat16* xs = static_cast<const __nv_bfloat16*>(x);
        if (T <= DEC_T) {
            e = launch_router_logits_decode(L, xs, T, h->router_W, h->router_b, lg);
            if (e == cudaSuccess) e = launch_select(L, lg, T, idx, w);
        } else {
            CUtensorMap xmap;
            if (!encode_bf16_2d(&xmap, xs, T, H, H, 128, 64)) return FLINT_ERR_CUDA;
            e = launch_prefill_router(L, xmap, h->wr_map, T, h->router_b, logits, idx, w, h->local_rank,
                                      h->blk_counts);
            if (e == cudaSuccess && (offsets || gather_idx))
                e = launch_perm_scan_scatter(L, idx, T, h->local_rank, h->blk_counts, h->blk_base,
                                             offsets ? offsets : h->offsets, gather_idx, nullptr);
            if (e == cudaSuccess) e = cudaStreamSynchronize(s);
            if (e != cudaSuccess) return FLINT_ERR_CUDA;
            return take_device_status(h);
        }
    } else {
        e = launch_select(L, logits, T, idx, w);
    }
    if (e == cudaSuccess && (offsets || gather_idx)) {
        int32_t* off = offsets ? offsets : h->offsets;
        e = launch_permutation(L, idx, T, h->local_rank, h->blk_counts, h->blk_base, off, gather_idx);
    }
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return FLINT_ERR_CUDA;
    return take_device_status(h);
}

flint_status_t flint_moe_set_kernel_events(flint_moe_t h, int kernel, cudaEvent_t start, cudaEvent_t stop) {
    if (!h) return FLINT_ERR_INVALID_ARG;
    if (kernel == -1) {
        h->prof_kernel = -1;
        h->prof_start = h->prof_stop = nullptr;
        return FLINT_OK;
    }
    if (kernel < FLINT_KERNEL_ROUTER || kernel > FLINT_KERNEL_COMBINE || !start || !stop)
        return FLINT_ERR_INVALID_ARG;
    h->prof_kernel = kernel;
    h->prof_start = start;
    h->prof_stop = stop;
    return FLINT_OK;
}

flint_status_t flint_moe_destroy(flint_moe_t h) {
    if (!h) return FLINT_OK;
    cudaError_t e = cudaDeviceSynchronize();
    flint_status_t st = take_device_status(h);
    free_handle(h);
    if (st == FLINT_OK && e != cudaSuccess) st = FLINT_ERR_CUDA;
    return st;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// test hook: a bounded wait that nothing satisfies
// ---------------------------------------------------------------------------

__global__ void bounded_wait_probe_kernel(uint64_t limit_ns, uint32_t* result) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    // nothing arrives on the barrier: phase 0 never completes
    const bool ok = __syncthreads_and(mbar_wait_bounded(&bar, 0, limit_ns));
    if (threadIdx.x == 0) *result = ok ? 0u : ST_TIMEOUT;
}

extern "C" flint_status_t flint_debug_bounded_wait(uint64_t timeout_ns, cudaStream_t s) {
    if (timeout_ns == 0 || timeout_ns > 10000000000ull) return FLINT_ERR_INVALID_ARG;
    uint32_t* d = nullptr;
    if (cudaMalloc(&d, sizeof(uint32_t)) != cudaSuccess) return FLINT_ERR_OOM;
    uint32_t r = 0xFFFFFFFFu;
    bounded_wait_probe_kernel<<<1, 32, 0, s>>>(timeout_ns, d);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess) e = cudaMemcpyAsync(&r, d, sizeof r, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    cudaFree(d);
    if (e != cudaSuccess) return FLINT_ERR_CUDA;
    if (r == ST_TIMEOUT) return FLINT_ERR_DEVICE_TIMEOUT;
    return r == 0 ? FLINT_OK : FLINT_ERR_CUDA;
}
