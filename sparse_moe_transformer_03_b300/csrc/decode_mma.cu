// decode_mma.cu -- bf16 weight-streaming decode kernels (T <= 32) on the
// warp-level tensor core (mma.sync m16n8k16).
//
// Layer definition: RecursiveSI/flint (vLLM recipe page), "Overview" (256
// experts, top-6 sigmoid routing plus a shared expert); SwiGLU experts with
// H = 2048, I = 512 are this library's reading (the pages name neither).
//
// At decode sizes each expert weight meets only a few tokens, so the layer is
// bound by reading the touched experts' weights from HBM once: (U + 1)
// experts x 6 MiB, U = distinct routed experts of the batch.  The expert
// matrices are dotted with the tokens on the tensor core all the same: one
// MMA instruction does 2048 multiply-adds for the warp, so the kernels keep
// pace with HBM when every weight meets 8 or more tokens (the shared expert
// meets all of them), and at one token they measured faster than CUDA-core
// dot products as well.  After the router kernel has written the
// fp32 logits, two kernels run, chained with programmatic dependent launch;
// each ranks the experts of every token from the logits and builds the
// (expert slot, token) tables in its own shared memory (slot 0 = the shared
// expert), and the shared expert's first weights are requested before the
// kernel waits on the router.
//
// They read the handle's tiled copy of the experts (repack.cu): tiles of 128
// rows x 64 columns in the 128-byte-swizzled layout.  Eight consecutive rows
// of a tile are 1 KiB of contiguous bytes, so a unit's operands arrive by
// cp.async.bulk in 1 KiB (gate/up) or 2 KiB (down) pieces, and ldmatrix
// reads them without bank conflicts (the swizzle spreads the eight rows of an
// 8x8 matrix over all banks).
//
//   gateup_mma   Unit = 8 gate rows + the 8 matching up rows of one expert
//                (the MMA's 16 rows); item = a unit against one tile of up
//                to 8 of the expert's tokens (the N columns).  The CTA takes
//                one item at a time: warp w streams columns 256w .. 256w +
//                255 (8 KiB) into its ring and multiplies them by x
//                fragments it fetched into registers during the item before;
//                the eight partial sums are added in warp order in smem, then
//                a = silu(g) * u is written as bf16.
//   down_mma     CTA c owns output rows 16c .. 16c + 15 (one M tile).  Its
//                work items are (slot, column half, tile of 8 tokens): 256
//                columns of the slot's 16 rows (4 pieces of 2 KiB) against up
//                to 8 of its tokens; item j goes to warp j % 8, so the shared
//                slot's tiles and halves spread over the warps.  An item's
//                activations (8 pairs x 256 columns, contiguous in the
//                act_index layout the gate/up kernel writes) arrive in the
//                same ring slot as its weights, by one more bulk copy.  w * D
//                accumulates per (token, row) in the warp's own buffer and
//                the eight buffers are summed in warp order: deterministic.
//
// The down kernel routes for itself, like the NVFP4 one, and starts its
// weight chunks before waiting on the gate/up kernel.
#include "flint_common.cuh"
#include "../../include/flint_moe.h"
#include "flint_internal.h"
#include "mma_sync.cuh"
#include "routing.cuh"

namespace flint {

constexpr size_t MM_TILE = 16384;                         // one 128 x 64 bf16 tile
constexpr size_t MM_EXPERT_BYTES = (size_t)3 * H * I * 2; // one expert in the tiled copy
constexpr size_t MM_DOWN_OFF = (size_t)2 * I * H * 2;     // its down tiles follow the gate/up tiles
constexpr int MM_GU_KT = H / 64;                          // 32 column tiles per gate/up row block
constexpr int MM_DN_KT = I / 64;                          // 8 column tiles per down row block
constexpr int MM_CHUNK = 8192;
constexpr int MM_WARPS = 8;

// ---------------------------------------------------------------------------
// gate/up + SwiGLU
// ---------------------------------------------------------------------------

constexpr int MG_UNITS = DEC_UNITS;      // 64 units per expert

struct GateUpMmaParams {
    const uint8_t* tiled;         // the handle's tiled experts
    const float* logits;
    const __nv_bfloat16* x;
    int T;
    DecodeTables* tables_out;
    int32_t* idx_out;
    float* w_out;
    __nv_bfloat16* a;             // activations, act_index layout
    uint32_t* status;
    uint64_t limit_ns;
};

// Work item = (slot u, unit r, tile nt of 8 tokens), packed u << 8 | r << 2 |
// nt; item j of the grid goes to CTA j % G.  Each warp fetches its B
// fragments (x rows of the tile's tokens, its 256 columns) into registers
// while the item before runs, so x needs no shared memory and the weight ring
// holds three chunks per warp.  A unit with several token tiles (the shared
// expert's for T > 8) reads its weights once per tile; the repeats hit L2.

constexpr int MI_NS = 3;                            // ring chunks per warp
constexpr int MI_PART = 2 * MM_WARPS * 32 * 4;      // partial sums: [item parity][warp][lane][4]

static inline size_t mi_smem_bytes() {
    return (size_t)MM_WARPS * MI_NS * MM_CHUNK + (size_t)MI_PART * 4 + (size_t)MM_WARPS * MI_NS * 8 +
           sizeof(DecodeTables) + DEC_T * TOPK * 8 + 2 * E * 4 + DEC_MAX_CTA_ITEMS * 4;
}

__global__ void __launch_bounds__(MM_WARPS * 32, 1) gateup_mma_kernel(GateUpMmaParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int T = p.T, G = gridDim.x, c = blockIdx.x;
    uint8_t* ring = smem + (size_t)warp * MI_NS * MM_CHUNK;
    float* part = reinterpret_cast<float*>(smem + (size_t)MM_WARPS * MI_NS * MM_CHUNK);
    uint64_t* bar = reinterpret_cast<uint64_t*>(part + MI_PART) + warp * MI_NS;
    DecodeTables* tab = reinterpret_cast<DecodeTables*>(reinterpret_cast<uint64_t*>(part + MI_PART) + MM_WARPS * MI_NS);
    int* sel_e = reinterpret_cast<int*>(tab + 1);
    float* sel_w = reinterpret_cast<float*>(sel_e + DEC_T * TOPK);
    uint32_t* tmask = reinterpret_cast<uint32_t*>(sel_w + DEC_T * TOPK);
    int* pair0 = reinterpret_cast<int*>(tmask + E);
    int* list = pair0 + E;                           // this CTA's items c, c + G, ...

    if (lane == 0) {
        for (int s = 0; s < MI_NS; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    const int nt0 = (T + 7) >> 3;                    // token tiles of the shared slot (slot 0)
    // this warp's chunk of an item: 4 column tiles x (gate piece, up piece)
    auto issue = [&](int i, int it, int expert) {
        const int s = i % MI_NS, r = (it >> 2) & (MG_UNITS - 1);
        uint8_t* dst = ring + (size_t)s * MM_CHUNK;
        const uint8_t* src = p.tiled + (size_t)expert * MM_EXPERT_BYTES + (size_t)(r & 15) * 1024;
        mbar_arrive_expect_tx(&bar[s], MM_CHUNK);
#pragma unroll
        for (int kt = 0; kt < 4; ++kt) {
            const int kc = warp * 4 + kt;
            bulk_g2s(dst + (2 * kt) * 1024, src + ((size_t)(r >> 4) * MM_GU_KT + kc) * MM_TILE, 1024, &bar[s]);
            bulk_g2s(dst + (2 * kt + 1) * 1024, src + ((size_t)((r >> 4) + 4) * MM_GU_KT + kc) * MM_TILE, 1024,
                     &bar[s]);
        }
    };

    // ---- before the router has finished: the shared slot's items (their
    // tile count is ceil(T / 8) whatever the routing) ----
    int issued = 0;
    if (lane == 0) {
        for (int i = 0; i < MI_NS && c + G * i < MG_UNITS * nt0; ++i) {
            const int j = c + G * i;
            issue(i, ((j / nt0) << 2) | (j % nt0), SHARED);
            issued = i + 1;
        }
    }
    pdl_wait();     // router logits are complete (and x is ready)
    pdl_trigger();

    // ---- top-6 of every token, then the (slot, token) tables ----
    select_tokens_warps(p.logits, T, warp, lane, sel_e, sel_w, c == 0 ? p.idx_out : nullptr,
                        c == 0 ? p.w_out : nullptr);
    __syncthreads();
    if (warp == 0) build_decode_tables_warp(T, sel_e, sel_w, tmask, pair0, tab, lane);
    __syncthreads();
    if (c == 0) {
        const int* src = reinterpret_cast<const int*>(tab);
        int* dst = reinterpret_cast<int*>(p.tables_out);
        for (int k = threadIdx.x; k < (int)(sizeof(DecodeTables) / 4); k += blockDim.x) dst[k] = src[k];
    }
    int my_items = list_gateup_items(tab, c, G, list);
    if (my_items < 0) {   // ruled out by the grid size (DEC_MIN_GRID); drained below
        if (threadIdx.x == 0) report_status(p.status, ST_INTERNAL);
        my_items = 0;
    }
    __syncthreads();
    if (lane == 0) {
        for (int i = issued; i < MI_NS && i < my_items; ++i) {
            issue(i, list[i], tab->slot_expert[list[i] >> 8]);
            issued = i + 1;
        }
    }

    const int mi = lane >> 3, li = lane & 7;
    const uint32_t lrow = (uint32_t)((mi & 1) * 1024 + li * 128);
    const int lkh = mi >> 1;
    const int g = lane >> 2, cq = lane & 3;
    // B fragments of an item: x row of the tile's token g (the last token past
    // the slot's end), this warp's columns
    auto load_b = [&](int it, uint32_t (&b)[16][2]) {
        const int u = it >> 8, pb = tab->slot_pair0[u], np = tab->slot_pair0[u + 1] - pb;
        const int n = (it & 3) * 8 + g;
        const int tok = tab->pair_token[pb + (n < np ? n : np - 1)];
        const unsigned int* x0 = reinterpret_cast<const unsigned int*>(p.x + (size_t)tok * H + warp * 256 + 2 * cq);
#pragma unroll
        for (int kb = 0; kb < 16; ++kb) {
            b[kb][0] = __ldg(x0 + kb * 8);
            b[kb][1] = __ldg(x0 + kb * 8 + 4);
        }
    };
    uint32_t bq[16][2];
    if (my_items > 0) load_b(list[0], bq);
    bool ok = true;
    int i = 0;
    for (; i < my_items; ++i) {
        const int it = list[i];
        uint32_t bn[16][2];
        if (i + 1 < my_items) load_b(list[i + 1], bn);
        const int s = i % MI_NS;
        const bool got = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&bar[s], (i / MI_NS) & 1, p.limit_ns));
        float* pw = part + (((i & 1) * MM_WARPS + warp) * 32 + lane) * 4;
        if (got) {
            const uint8_t* buf = ring + (size_t)s * MM_CHUNK;
            float acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int kb = 0; kb < 16; kb += 2) {
                uint32_t a[4], a2[4];
                const int kt = kb >> 2, j0 = 2 * (kb & 3) + lkh;
                ldmatrix_x4(a, buf + kt * 2048 + lrow + ((j0 ^ li) << 4));
                ldmatrix_x4(a2, buf + kt * 2048 + lrow + (((j0 + 2) ^ li) << 4));
                mma_bf16_16816(acc, a, bq[kb][0], bq[kb][1]);
                mma_bf16_16816(acc2, a2, bq[kb + 1][0], bq[kb + 1][1]);
            }
            __syncwarp();   // every lane is done reading slot s
            if (lane == 0 && i + MI_NS < my_items) {
                fence_proxy_async_smem();
                issue(i + MI_NS, list[i + MI_NS], tab->slot_expert[list[i + MI_NS] >> 8]);
                issued = i + MI_NS + 1;
            }
            *reinterpret_cast<float4*>(pw) = make_float4(acc[0] + acc2[0], acc[1] + acc2[1], acc[2] + acc2[2],
                                                         acc[3] + acc2[3]);
        }
        if (!__syncthreads_and(got)) {
            ok = false;
            break;
        }
        // warp i % 8 adds the item's eight partial sums in warp order; lane
        // (g, cq) then holds gate (x, y) and up (z, w) of row 8r + g for
        // tokens 2cq, 2cq + 1 of the tile.  The buffer of parity i & 1 is
        // next written after the barrier of item i + 1, which this warp
        // reaches only after the sum.
        if (warp == (i & (MM_WARPS - 1))) {
            const float* pb0 = part + ((i & 1) * MM_WARPS * 32 + lane) * 4;
            float4 sum = *reinterpret_cast<const float4*>(pb0);
#pragma unroll
            for (int w = 1; w < MM_WARPS; ++w) {
                const float4 v = *reinterpret_cast<const float4*>(pb0 + w * 32 * 4);
                sum.x += v.x;
                sum.y += v.y;
                sum.z += v.z;
                sum.w += v.w;
            }
            const int u = it >> 8, r = (it >> 2) & (MG_UNITS - 1);
            const int pb = tab->slot_pair0[u], np = tab->slot_pair0[u + 1] - pb;
            const int j = 8 * r + g, n0 = (it & 3) * 8 + 2 * cq;
            if (n0 < np) p.a[act_index(pb + n0, j)] = __float2bfloat16_rn(silu_f(sum.x) * sum.z);
            if (n0 + 1 < np) p.a[act_index(pb + n0 + 1, j)] = __float2bfloat16_rn(silu_f(sum.y) * sum.w);
        }
#pragma unroll
        for (int kb = 0; kb < 16; ++kb) {
            bq[kb][0] = bn[kb][0];
            bq[kb][1] = bn[kb][1];
        }
    }
    if (lane == 0) {
        if (!ok) report_status(p.status, ST_TIMEOUT);
        // copies still in flight into this warp's ring (after a timeout, or the
        // shared slot's prefetched items when the item list came out empty):
        // wait for them, bounded, before the CTA exits
        for (int k = i; k < issued; ++k) mbar_wait_bounded(&bar[k % MI_NS], (k / MI_NS) & 1, p.limit_ns);
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// down projection + weighted combine
// ---------------------------------------------------------------------------

constexpr int MD_CTAS = H / 16;          // 128
constexpr int MD_NS = 2;                 // ring slots per warp
constexpr int MD_ACT = 8 * 256 * 2;      // an item's activation tile: 8 pairs x 256 columns, bf16
constexpr int MD_SLOT = MM_CHUNK + MD_ACT;

struct DownMmaParams {
    const uint8_t* tiled;
    const float* logits;          // [T][E] (final before this kernel starts)
    const __nv_bfloat16* a;       // activations, act_index layout
    __nv_bfloat16* y;
    int T;
    uint32_t* status;
    uint64_t limit_ns;
};

static inline size_t md_smem_bytes(int T) {
    return (size_t)MM_WARPS * MD_NS * (MD_SLOT + 8) + (size_t)MM_WARPS * T * 16 * 4 + sizeof(DecodeTables) +
           DEC_T * TOPK * 8 + 2 * E * 4 + (DEC_MAX_DOWN_ITEMS + 1) * 4;
}

__global__ void __launch_bounds__(MM_WARPS * 32, 1) down_mma_kernel(DownMmaParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, Tk = p.T;
    uint8_t* ring = smem + (size_t)warp * MD_NS * MD_SLOT;
    float* yw_all = reinterpret_cast<float*>(smem + (size_t)MM_WARPS * MD_NS * MD_SLOT);
    float* yw = yw_all + warp * Tk * 16;
    uint64_t* bars = reinterpret_cast<uint64_t*>(yw_all + MM_WARPS * Tk * 16);
    uint64_t* bar = bars + warp * MD_NS;
    DecodeTables* tab = reinterpret_cast<DecodeTables*>(bars + MM_WARPS * MD_NS);
    int* sel_e = reinterpret_cast<int*>(tab + 1);
    float* sel_w = reinterpret_cast<float*>(sel_e + DEC_T * TOPK);
    uint32_t* tmask = reinterpret_cast<uint32_t*>(sel_w + DEC_T * TOPK);
    int* pair0 = reinterpret_cast<int*>(tmask + E);
    int* items = pair0 + E;
    int* n_items_s = items + DEC_MAX_DOWN_ITEMS;

    if (lane == 0) {
        for (int s = 0; s < MD_NS; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    // the warp's k-th item is items[warp + 8k]; its weights: columns 256 half
    // .. + 255 of rows 16c .. 16c + 15 of the slot's expert; its activations:
    // the tile's 8 pairs in that half (pairs past the slot's end come along
    // and are not used)
    auto item_of = [&](int k) { return items[warp + MM_WARPS * k]; };
    auto copy_w = [&](int k) {
        const int it = item_of(k), s = k % MD_NS;
        const int expert = tab->slot_expert[it >> 3];
        const uint8_t* base = p.tiled + (size_t)expert * MM_EXPERT_BYTES + MM_DOWN_OFF + (size_t)(c & 7) * 2048;
        const int rb = c >> 3, kc0 = ((it >> 2) & 1) * 4;
        uint8_t* dst = ring + (size_t)s * MD_SLOT;
#pragma unroll
        for (int kt = 0; kt < 4; ++kt)
            bulk_g2s(dst + kt * 2048, base + ((size_t)rb * MM_DN_KT + kc0 + kt) * MM_TILE, 2048, &bar[s]);
    };
    auto copy_a = [&](int k) {
        const int it = item_of(k), s = k % MD_NS;
        const int p0 = tab->slot_pair0[it >> 3] + (it & 3) * 8;
        bulk_g2s(ring + (size_t)s * MD_SLOT + MM_CHUNK, p.a + ((size_t)((it >> 2) & 1) * DEC_ACT_ROWS + p0) * 256,
                 MD_ACT, &bar[s]);
    };
    // The router grid completed before any gate/up CTA passed its dependency
    // wait, and this launch is triggered only after those waits: the logits
    // are final here.  Route for ourselves and start the weight chunks while
    // the gate/up kernel still runs.
    select_tokens_warps(p.logits, Tk, warp, lane, sel_e, sel_w, nullptr, nullptr);
    for (int k = threadIdx.x; k < MM_WARPS * Tk * 16; k += blockDim.x) yw_all[k] = 0.f;
    __syncthreads();
    if (warp == 0) {
        build_decode_tables_warp(Tk, sel_e, sel_w, tmask, pair0, tab, lane);
        const int n = build_down_items_warp(tab, items, lane);
        if (lane == 0) *n_items_s = n;
    }
    __syncthreads();
    const int n_items = *n_items_s;
    const int my_items = n_items > warp ? (n_items - warp + MM_WARPS - 1) / MM_WARPS : 0;
    // weights of the first items now (the phase waits for its arrival, which
    // comes with the activations after the dependency wait)
    int issued = 0;
    if (lane == 0) {
        for (int k = 0; k < MD_NS && k < my_items; ++k) {
            mbar_expect_tx(&bar[k], MM_CHUNK);
            copy_w(k);
            issued = k + 1;
        }
    }
    pdl_wait();     // the gate/up kernel is complete: activations are visible
    pdl_trigger();
    if (lane == 0) {
        for (int k = 0; k < issued; ++k) {
            mbar_arrive_expect_tx(&bar[k], MD_ACT);
            copy_a(k);
        }
    }

    const int mi = lane >> 3, li = lane & 7;
    const int lr = (mi & 1) * 8 + li;               // row 0..15 of the M tile
    const uint32_t lrow = (uint32_t)lr * 128;
    const int lkh = mi >> 1;
    const int g = lane >> 2, cq = lane & 3;
    bool ok = true;
    int k = 0;
    for (; k < my_items; ++k) {
        const int it = item_of(k), u = it >> 3, nt = it & 3;
        const int pb = tab->slot_pair0[u], np = tab->slot_pair0[u + 1] - pb;
        const int s = k % MD_NS;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&bar[s], (k / MD_NS) & 1, p.limit_ns))) {
            ok = false;
            break;
        }
        const uint8_t* buf = ring + (size_t)s * MD_SLOT;
        // row g of the activation tile; chunk q of it sits at q ^ (pair % 8)
        const uint8_t* ar = buf + MM_CHUNK + g * 512 + 4 * cq;
        const int sw = (pb + nt * 8 + g) & 7;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kb = 0; kb < 16; ++kb) {
            uint32_t a[4];
            const int kt = kb >> 2, j = 2 * (kb & 3) + lkh;
            ldmatrix_x4(a, buf + kt * 2048 + lrow + ((j ^ li) << 4));
            mma_bf16_16816(acc[kb & 1], a, *reinterpret_cast<const uint32_t*>(ar + (((2 * kb) ^ sw) << 4)),
                           *reinterpret_cast<const uint32_t*>(ar + (((2 * kb + 1) ^ sw) << 4)));
        }
        __syncwarp();
        if (lane == 0 && k + MD_NS < my_items) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bar[s], MM_CHUNK + MD_ACT);
            copy_w(k + MD_NS);
            copy_a(k + MD_NS);
            issued = k + MD_NS + 1;
        }
        // lane (g, cq) holds rows g, g + 8 of tokens 2cq, 2cq + 1 of the tile
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int n = nt * 8 + 2 * cq + hh;
            if (n < np) {
                const int pr = pb + n, t = tab->pair_token[pr];
                const float wgt = tab->pair_weight[pr];
                yw[t * 16 + g] = fmaf(wgt, acc[0][hh] + acc[1][hh], yw[t * 16 + g]);
                yw[t * 16 + g + 8] = fmaf(wgt, acc[0][2 + hh] + acc[1][2 + hh], yw[t * 16 + g + 8]);
            }
        }
    }
    if (!ok && lane == 0) {
        report_status(p.status, ST_TIMEOUT);
        for (int q = k; q < issued; ++q) mbar_wait_bounded(&bar[q % MD_NS], (q / MD_NS) & 1, p.limit_ns);
    }
    __syncthreads();
    for (int q = threadIdx.x; q < Tk * 16; q += blockDim.x) {
        const int t = q >> 4, rr = q & 15;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < MM_WARPS; ++w) sum += yw_all[w * Tk * 16 + t * 16 + rr];
        p.y[(size_t)t * H + 16 * c + rr] = __float2bfloat16_rn(sum);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

cudaError_t decode_mma_set_attributes() {
    size_t dmax = 0;
    for (int T = 1; T <= DEC_T; ++T) dmax = md_smem_bytes(T) > dmax ? md_smem_bytes(T) : dmax;
    cudaError_t e =
        cudaFuncSetAttribute(gateup_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)mi_smem_bytes());
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(down_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dmax);
}

cudaError_t launch_decode_experts_mma(const LaunchCtx& L, const uint8_t* tiled, const float* logits,
                                      const __nv_bfloat16* x, int T, DecodeTables* tables, int32_t* idx, float* w,
                                      __nv_bfloat16* a_buf, __nv_bfloat16* y) {
    if (T < 1 || T > DEC_T) return cudaErrorInvalidValue;
    __nv_bfloat16* a16 = a_buf;
    GateUpMmaParams gp{tiled, logits, x, T, tables, idx, w, a16, L.status, L.wait_limit_ns};
    // at most 64 x (257 + 28) items over the grid: 72 CTAs or more keep every
    // CTA's list within its 256 entries
    const int gi = L.num_sms >= DEC_MIN_GRID ? L.num_sms : DEC_MIN_GRID;
    cudaError_t e = launch_hooked(L, FLINT_KERNEL_GATE_UP, gateup_mma_kernel, dim3(gi), dim3(MM_WARPS * 32),
                                  mi_smem_bytes(), gp);
    if (e != cudaSuccess) return e;
    DownMmaParams dp{tiled, logits, a16, y, T, L.status, L.wait_limit_ns};
    return launch_hooked(L, FLINT_KERNEL_DOWN, down_mma_kernel, dim3(MD_CTAS), dim3(MM_WARPS * 32),
                         md_smem_bytes(T), dp);
}

}  // namespace flint
