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
//                slot's tiles and halves spread over the warps.  The
//                activations are staged in smem when the batch has at most 64
//                (token, expert) pairs, else each item's B fragments are
//                fetched into registers while the item before it computes.
//                w * D accumulates per (token, row) in the warp's own buffer
//                and the eight buffers are summed in warp order: deterministic.
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

constexpr int MG_UNITS = I / 8;          // 64 units per expert

struct GateUpMmaParams {
    const uint8_t* tiled;         // the handle's tiled experts
    const float* logits;
    const __nv_bfloat16* x;
    int T;
    DecodeTables* tables_out;
    int32_t* idx_out;
    float* w_out;
    __nv_bfloat16* a;             // [pairs][I]
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
constexpr int MI_MAX_CTA_ITEMS = 256;               // items of one CTA (grid >= 72 CTAs)
constexpr int MI_PART = 2 * MM_WARPS * 32 * 4;      // partial sums: [item parity][warp][lane][4]

static inline size_t mi_smem_bytes() {
    return (size_t)MM_WARPS * MI_NS * MM_CHUNK + (size_t)MI_PART * 4 + (size_t)MM_WARPS * MI_NS * 8 +
           sizeof(DecodeTables) + DEC_T * TOPK * 8 + 2 * E * 4 + (NEXP + 1) * 4 + MI_MAX_CTA_ITEMS * 4;
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
    int* slot_item0 = pair0 + E;                     // first item of each slot (+ the total)
    int* list = slot_item0 + NEXP + 1;               // this CTA's items c, c + G, ...

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
    for (int t = warp; t < T; t += MM_WARPS) {
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __ldcg(p.logits + (size_t)t * E + lane + 32 * k);
        int sel[TOPK];
        float wt[TOPK];
        warp_top6(v, lane, sel, wt);
        if (lane < TOPK) {
            const int se = pick6(sel, lane);
            const float sw = pick6(wt, lane);
            sel_e[t * TOPK + lane] = se;
            sel_w[t * TOPK + lane] = sw;
            if (c == 0) {
                p.idx_out[t * TOPK + lane] = se;
                p.w_out[t * TOPK + lane] = sw;
            }
        }
    }
    __syncthreads();
    if (warp == 0) {
        build_decode_tables_warp(T, sel_e, sel_w, tmask, pair0, tab, lane);
        // slot_item0: exclusive prefix of 64 * ceil(np / 8) over the slots
        int base = 0;
        for (int u0 = 0; u0 < tab->n_slots; u0 += 32) {
            const int u = u0 + lane;
            const int n = u < tab->n_slots ? MG_UNITS * ((tab->slot_pair0[u + 1] - tab->slot_pair0[u] + 7) >> 3) : 0;
            int inc = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xFFFFFFFFu, inc, o);
                if (lane >= o) inc += v;
            }
            if (u < tab->n_slots) slot_item0[u] = base + inc - n;
            base += __shfl_sync(0xFFFFFFFFu, inc, 31);
        }
        if (lane == 0) slot_item0[tab->n_slots] = base;
    }
    __syncthreads();
    if (c == 0) {
        const int* src = reinterpret_cast<const int*>(tab);
        int* dst = reinterpret_cast<int*>(p.tables_out);
        for (int k = threadIdx.x; k < (int)(sizeof(DecodeTables) / 4); k += blockDim.x) dst[k] = src[k];
    }
    const int n_slots = tab->n_slots, total = slot_item0[n_slots];
    int my_items = c < total ? (total - c + G - 1) / G : 0;
    if (my_items > MI_MAX_CTA_ITEMS) {   // the launcher sizes the grid so that this cannot happen
        if (threadIdx.x == 0) report_status(p.status, ST_BADINDEX);
        my_items = 0;
    }
    for (int i = threadIdx.x; i < my_items; i += blockDim.x) {
        const int j = c + G * i;
        int lo = 0, hi = n_slots - 1;     // the last slot u with slot_item0[u] <= j
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (slot_item0[mid] <= j) lo = mid;
            else hi = mid - 1;
        }
        const int l = j - slot_item0[lo];
        const int ntu = (tab->slot_pair0[lo + 1] - tab->slot_pair0[lo] + 7) >> 3;
        list[i] = (lo << 8) | ((l / ntu) << 2) | (l % ntu);
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
            if (n0 < np) p.a[(size_t)(pb + n0) * I + j] = __float2bfloat16_rn(silu_f(sum.x) * sum.z);
            if (n0 + 1 < np) p.a[(size_t)(pb + n0 + 1) * I + j] = __float2bfloat16_rn(silu_f(sum.y) * sum.w);
        }
#pragma unroll
        for (int kb = 0; kb < 16; ++kb) {
            bq[kb][0] = bn[kb][0];
            bq[kb][1] = bn[kb][1];
        }
    }
    if (!ok) {
        if (lane == 0) {
            report_status(p.status, ST_TIMEOUT);
            for (int k = i; k < issued; ++k) mbar_wait_bounded(&bar[k % MI_NS], (k / MI_NS) & 1, p.limit_ns);
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// down projection + weighted combine
// ---------------------------------------------------------------------------

constexpr int MD_CTAS = H / 16;          // 128
constexpr int MD_APAIRS = 64;            // activation rows staged in smem up to this many pairs
constexpr int MD_AROW = I * 2 + 16;      // bytes per staged row
// items: 2 column halves x the N tiles of every slot (sum of ceil(np / 8) over
// the slots is below slots + pairs / 8)
constexpr int MD_MAX_ITEMS = 2 * (NEXP + DEC_PAIRS / 8);

struct DownMmaParams {
    const uint8_t* tiled;
    const float* logits;          // [T][E] (final before this kernel starts)
    const __nv_bfloat16* a;       // [pairs][I]
    __nv_bfloat16* y;
    int ns;
    int T;
    uint32_t* status;
    uint64_t limit_ns;
};

static inline int md_ns(int T) { return T <= 9 ? 2 : 3; }
__host__ __device__ inline bool md_staged(int T) { return (TOPK + 1) * T <= MD_APAIRS; }
static inline size_t md_smem_bytes(int T) {
    return (size_t)MM_WARPS * md_ns(T) * MM_CHUNK + (md_staged(T) ? (size_t)(TOPK + 1) * T * MD_AROW : 0) +
           (size_t)MM_WARPS * T * 16 * 4 + (MM_WARPS * md_ns(T) + 1) * 8 + sizeof(DecodeTables) +
           DEC_T * TOPK * 8 + 2 * E * 4 + (MD_MAX_ITEMS + 1) * 4;
}

// Lists the down kernel's work items in slot order, each slot's first column
// half before its second and the N tiles in order within a half; packed as
// slot << 3 | half << 2 | tile.  One warp; returns the count on every lane.
__device__ __forceinline__ int build_down_items_warp(const DecodeTables* tab, int* items, int lane) {
    int base = 0;
    for (int u0 = 0; u0 < tab->n_slots; u0 += 32) {
        const int u = u0 + lane;
        const int nt = u < tab->n_slots ? (tab->slot_pair0[u + 1] - tab->slot_pair0[u] + 7) >> 3 : 0;
        int inc = nt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if (lane >= o) inc += v;
        }
        const int off = base + 2 * (inc - nt);
        for (int hk = 0; hk < 2; ++hk)
            for (int t = 0; t < nt; ++t) items[off + hk * nt + t] = (u << 3) | (hk << 2) | t;
        base += 2 * __shfl_sync(0xFFFFFFFFu, inc, 31);
    }
    __syncwarp();
    return base;
}

__global__ void __launch_bounds__(MM_WARPS * 32, 1) down_mma_kernel(DownMmaParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, NS = p.ns, Tk = p.T;
    const bool staged = md_staged(Tk);
    uint8_t* ring = smem + (size_t)warp * NS * MM_CHUNK;
    uint8_t* astage = smem + (size_t)MM_WARPS * NS * MM_CHUNK;
    float* yw_all = reinterpret_cast<float*>(astage + (staged ? (size_t)(TOPK + 1) * Tk * MD_AROW : 0));
    float* yw = yw_all + warp * Tk * 16;
    uint64_t* bars = reinterpret_cast<uint64_t*>(yw_all + MM_WARPS * Tk * 16);
    uint64_t* bar = bars + warp * NS;
    uint64_t* abar = bars + MM_WARPS * NS;
    DecodeTables* tab = reinterpret_cast<DecodeTables*>(abar + 1);
    int* sel_e = reinterpret_cast<int*>(tab + 1);
    float* sel_w = reinterpret_cast<float*>(sel_e + DEC_T * TOPK);
    uint32_t* tmask = reinterpret_cast<uint32_t*>(sel_w + DEC_T * TOPK);
    int* pair0 = reinterpret_cast<int*>(tmask + E);
    int* items = pair0 + E;
    int* n_items_s = items + MD_MAX_ITEMS;

    if (lane == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&bar[s], 1);
        if (warp == 0) mbar_init(abar, 1);
        fence_mbar_init();
    }
    // the warp's k-th item is items[warp + 8k]; its weights: columns 256 half
    // .. + 255 of rows 16c .. 16c + 15 of the slot's expert
    auto item_of = [&](int k) { return items[warp + MM_WARPS * k]; };
    auto issue = [&](int k) {
        const int it = item_of(k), s = k % NS;
        const int expert = tab->slot_expert[it >> 3];
        const uint8_t* base = p.tiled + (size_t)expert * MM_EXPERT_BYTES + MM_DOWN_OFF + (size_t)(c & 7) * 2048;
        const int rb = c >> 3, kc0 = ((it >> 2) & 1) * 4;
        uint8_t* dst = ring + (size_t)s * MM_CHUNK;
        mbar_arrive_expect_tx(&bar[s], MM_CHUNK);
#pragma unroll
        for (int kt = 0; kt < 4; ++kt)
            bulk_g2s(dst + kt * 2048, base + ((size_t)rb * MM_DN_KT + kc0 + kt) * MM_TILE, 2048, &bar[s]);
    };
    // The router grid completed before any gate/up CTA passed its dependency
    // wait, and this launch is triggered only after those waits: the logits
    // are final here.  Route for ourselves and start the weight chunks while
    // the gate/up kernel still runs.
    for (int t = warp; t < Tk; t += MM_WARPS) {
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = __ldcg(p.logits + (size_t)t * E + lane + 32 * k);
        int sel[TOPK];
        float wt[TOPK];
        warp_top6(v, lane, sel, wt);
        if (lane < TOPK) {
            sel_e[t * TOPK + lane] = pick6(sel, lane);
            sel_w[t * TOPK + lane] = pick6(wt, lane);
        }
    }
    for (int k = threadIdx.x; k < MM_WARPS * Tk * 16; k += blockDim.x) yw_all[k] = 0.f;
    __syncthreads();
    if (warp == 0) {
        build_decode_tables_warp(Tk, sel_e, sel_w, tmask, pair0, tab, lane);
        const int n = build_down_items_warp(tab, items, lane);
        if (lane == 0) *n_items_s = n;
    }
    __syncthreads();
    const int n_items = *n_items_s, n_pairs = tab->n_pairs;
    const int my_items = n_items > warp ? (n_items - warp + MM_WARPS - 1) / MM_WARPS : 0;
    int issued = 0;
    if (lane == 0) {
        for (int k = 0; k < NS && k < my_items; ++k) {
            issue(k);
            issued = k + 1;
        }
    }
    pdl_wait();     // the gate/up kernel is complete: activations are visible
    pdl_trigger();
    if (staged && threadIdx.x == 0) {
        mbar_arrive_expect_tx(abar, n_pairs * I * 2);
        for (int pr = 0; pr < n_pairs; ++pr) bulk_g2s(astage + (size_t)pr * MD_AROW, p.a + (size_t)pr * I, I * 2, abar);
    }
    bool ok = true;
    if (staged && my_items > 0) ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(abar, 0, p.limit_ns));

    const int mi = lane >> 3, li = lane & 7;
    const int lr = (mi & 1) * 8 + li;               // row 0..15 of the M tile
    const uint32_t lrow = (uint32_t)lr * 128;
    const int lkh = mi >> 1;
    const int g = lane >> 2, cq = lane & 3;
    // this lane's B row of item k: pair pb + 8 tile + g (the last pair past np)
    auto b_row = [&](int it) {
        const int u = it >> 3, pb = tab->slot_pair0[u], np = tab->slot_pair0[u + 1] - pb;
        const int n = (it & 3) * 8 + g;
        return pb + (n < np ? n : np - 1);
    };
    // B fragments of the warp's k-th item from the activations in global
    // memory (read-only here; written by the previous grid)
    auto load_b = [&](int k, uint32_t (&b)[16][2]) {
        const int it = item_of(k);
        const unsigned int* a0 = reinterpret_cast<const unsigned int*>(p.a + (size_t)b_row(it) * I +
                                                                       ((it >> 2) & 1) * 256 + 2 * cq);
#pragma unroll
        for (int kb = 0; kb < 16; ++kb) {
            b[kb][0] = __ldg(a0 + kb * 8);
            b[kb][1] = __ldg(a0 + kb * 8 + 4);
        }
    };
    uint32_t bq[16][2];
    if (!staged && my_items > 0) load_b(0, bq);
    int k = 0;
    for (; ok && k < my_items; ++k) {
        const int it = item_of(k), u = it >> 3, hk = (it >> 2) & 1, nt = it & 3;
        const int pb = tab->slot_pair0[u], np = tab->slot_pair0[u + 1] - pb;
        uint32_t bn[16][2];
        if (!staged && k + 1 < my_items) load_b(k + 1, bn);
        const int s = k % NS;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&bar[s], (k / NS) & 1, p.limit_ns))) {
            ok = false;
            break;
        }
        const uint8_t* buf = ring + (size_t)s * MM_CHUNK;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        if (staged) {
            const uint8_t* ar = astage + (size_t)b_row(it) * MD_AROW + (hk * 256 + 2 * cq) * 2;
#pragma unroll
            for (int kb = 0; kb < 16; ++kb) {
                uint32_t a[4];
                const int kt = kb >> 2, j = 2 * (kb & 3) + lkh;
                ldmatrix_x4(a, buf + kt * 2048 + lrow + ((j ^ li) << 4));
                mma_bf16_16816(acc[kb & 1], a, *reinterpret_cast<const uint32_t*>(ar + kb * 32),
                               *reinterpret_cast<const uint32_t*>(ar + kb * 32 + 16));
            }
        } else {
#pragma unroll
            for (int kb = 0; kb < 16; ++kb) {
                uint32_t a[4];
                const int kt = kb >> 2, j = 2 * (kb & 3) + lkh;
                ldmatrix_x4(a, buf + kt * 2048 + lrow + ((j ^ li) << 4));
                mma_bf16_16816(acc[kb & 1], a, bq[kb][0], bq[kb][1]);
            }
        }
        __syncwarp();
        if (lane == 0 && k + NS < my_items) {
            fence_proxy_async_smem();
            issue(k + NS);
            issued = k + NS + 1;
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
        if (!staged) {
#pragma unroll
            for (int kb = 0; kb < 16; ++kb) {
                bq[kb][0] = bn[kb][0];
                bq[kb][1] = bn[kb][1];
            }
        }
    }
    if (!ok && lane == 0) {
        report_status(p.status, ST_TIMEOUT);
        for (int q = k; q < issued; ++q) mbar_wait_bounded(&bar[q % NS], (q / NS) & 1, p.limit_ns);
        if (staged && warp == 0) mbar_wait_bounded(abar, 0, p.limit_ns);
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
                                      float* a_buf, __nv_bfloat16* y) {
    if (T < 1 || T > DEC_T) return cudaErrorInvalidValue;
    __nv_bfloat16* a16 = reinterpret_cast<__nv_bfloat16*>(a_buf);
    GateUpMmaParams gp{tiled, logits, x, T, tables, idx, w, a16, L.status, L.wait_limit_ns};
    // at most 64 x (257 + 28) items over the grid: 72 CTAs or more keep every
    // CTA's list within its 256 entries
    const int gi = L.num_sms >= 72 ? L.num_sms : 72;
    cudaError_t e = launch_hooked(L, FLINT_KERNEL_GATE_UP, gateup_mma_kernel, dim3(gi), dim3(MM_WARPS * 32),
                                  mi_smem_bytes(), gp);
    if (e != cudaSuccess) return e;
    DownMmaParams dp{tiled, logits, a16, y, md_ns(T), T, L.status, L.wait_limit_ns};
    return launch_hooked(L, FLINT_KERNEL_DOWN, down_mma_kernel, dim3(MD_CTAS), dim3(MM_WARPS * 32),
                         md_smem_bytes(T), dp);
}

}  // namespace flint
