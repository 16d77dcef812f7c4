// prefill.cu -- the many-token path (T > 32) on the 5th-generation tensor
// cores: tcgen05.mma with fp32 accumulators in TMEM, operands staged in smem
// by bulk copies of pre-tiled weights, TMA tiled loads and cp.async gathers.
//
//   prefill_router   logits[128 tokens][256 experts] per CTA (K = 2048); the
//                    epilogue (one thread per token) adds the bias, selects the
//                    top-6 with equal logits going to the lower expert id,
//                    renormalises the sigmoid weights and computes each
//                    (token, slot) pair's rank among the block's pairs of the
//                    same expert plus the block's per-expert counts.
//   (scan, scatter)  offsets[257] and the expert-grouped pair list (router.cu)
//   prefill_gateup   grouped GEMM, "swapped": M = 128 rows of an expert's gate
//                    (and, in a second accumulator, the matching up) matrix,
//                    N = up to 256 of the expert's tokens gathered from x by
//                    cp.async (16-byte chunks into the swizzled tile),
//                    K = 2048.  Epilogue: h = silu(gate) * up, bf16, into
//                    h_perm[slot][512] (routed slots in expert order, then the
//                    shared expert's T slots).
//   prefill_down     grouped GEMM: M = 128 rows of the expert's down matrix,
//                    N = up to 256 slots of h_perm, K = 512.  Epilogue: the
//                    expert output of every slot, bf16, into o_perm[slot][2048].
//   combine          y[t] = sum of the token's six routed slots times their
//                    routing weights plus its shared slot, fp32, fixed order.
//
// Warp roles in every GEMM kernel: warp 0 issues TMA (one elected thread),
// warp 1 allocates TMEM and issues MMAs (one thread), warps 2..5 drain TMEM in
// the epilogue (warp w reads TMEM lanes 32*(w%4)..+31; the grouped GEMMs use
// two epilogue warps per lane quarter).  The grouped GEMMs are persistent:
// CTA c takes units c, c + grid, ... of the list ordered by (expert, row
// block, token pass).  Every wait is bounded; a timeout sets an
// abort flag the other roles observe, reports FLINT_ERR_DEVICE_TIMEOUT and the
// CTA still frees its TMEM.
//
// Layer definition: RecursiveSI/flint (vLLM recipe page), "Overview"; SwiGLU
// experts with H = 2048, I = 512 are this library's reading.
#include "../../include/flint_moe.h"
#include "flint_common.cuh"
#include "flint_internal.h"
#include "tc_ptx.cuh"
#include "prefill_common.cuh"

namespace flint {

// ===========================================================================
// router GEMM + top-6 + block-local permutation ranks
// ===========================================================================

constexpr int RG_STAGES = 4;
constexpr int RG_B_BYTES = E * PF_BK * 2;                  // 32 KiB: all 256 router rows
constexpr int RG_STAGE = PF_TILE_BYTES + RG_B_BYTES;       // 48 KiB
constexpr int RG_SMEM = 1024 + RG_STAGES * RG_STAGE + 256 + E * 4 * 4;

struct RouterGemmParams {
    int T;
    const float* bias;        // [E] or null
    float* logits;            // [T][E] or null (route-only output)
    int32_t* idx;             // [T][6]
    float* w;                 // [T][6]
    int32_t* local_rank;      // [T][6]
    int32_t* blk_counts;      // [nblk][E]
    uint32_t* status;
    uint64_t limit_ns;
};

__global__ void __launch_bounds__(PF_THREADS, 1)
    prefill_router_kernel(const __grid_constant__ CUtensorMap x_map, const __grid_constant__ CUtensorMap wr_map,
                          RouterGemmParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + RG_STAGES * RG_STAGE);
    uint64_t* empty = full + RG_STAGES;
    uint64_t* tfull = empty + RG_STAGES;
    uint64_t* mdone = tfull + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdone + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    uint32_t* mask = reinterpret_cast<uint32_t*>(smem + RG_STAGES * RG_STAGE + 256);   // [E][4]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int blk = blockIdx.x, row0 = blk * PF_TILE;

    if (threadIdx.x == 0) {
        for (int s = 0; s < RG_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(mdone, 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 256);
        tc::tmem_relinquish();
    }
    for (int k = threadIdx.x; k < E * 4; k += PF_THREADS) mask[k] = 0u;
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    pdl_wait();      // x may come from the previous kernel
    pdl_trigger();

    constexpr int KC = H / PF_BK;   // 32
    if (warp == 0 && lane == 0) {
        tc::prefetch_tensormap(&x_map);
        tc::prefetch_tensormap(&wr_map);
        for (int kc = 0; kc < KC; ++kc) {
            const int s = kc % RG_STAGES;
            if (!pf_wait(&empty[s], ((kc / RG_STAGES) & 1) ^ 1, p.limit_ns, abort)) break;
            uint8_t* st = smem + s * RG_STAGE;
            mbar_arrive_expect_tx(&full[s], RG_STAGE);
            tc::tma_load_2d(st, &x_map, kc * PF_BK, row0, &full[s]);
            tc::tma_load_2d(st + PF_TILE_BYTES, &wr_map, kc * PF_BK, 0, &full[s]);
        }
    } else if (warp == 1 && lane == 0) {
        constexpr uint32_t idesc = tc::idesc_bf16_f32(128, 256);
        for (int kc = 0; kc < KC; ++kc) {
            const int s = kc % RG_STAGES;
            if (!pf_wait(&full[s], (kc / RG_STAGES) & 1, p.limit_ns, abort)) break;
            tc::fence_after_sync();
            const uint8_t* st = smem + s * RG_STAGE;
            const uint64_t a = tc::smem_desc_sw128(st), b = tc::smem_desc_sw128(st + PF_TILE_BYTES);
#pragma unroll
            for (int kk = 0; kk < PF_BK / 16; ++kk)
                tc::mma_bf16(tmem, a + 2 * kk, b + 2 * kk, idesc, (kc | kk) != 0);
            tc::mma_commit(&empty[s]);
        }
        tc::mma_commit(tfull);
        tc::mma_commit(mdone);
        mbar_wait_bounded(mdone, 0, p.limit_ns);
    } else if (warp >= 2) {
        const int q = warp & 3, row = 32 * q + lane, t = row0 + row;
        // tcgen05.ld is warp-collective: the warp decides together
        const bool ok = __all_sync(0xFFFFFFFFu, pf_wait(tfull, 0, p.limit_ns, abort));
        tc::fence_after_sync();
        float tv[TOPK];
        int ti[TOPK];
#pragma unroll
        for (int r = 0; r < TOPK; ++r) {
            tv[r] = -INFINITY;
            ti[r] = r;
        }
        if (ok) {
#pragma unroll 1
            for (int c = 0; c < E / 32; ++c) {
                uint32_t v[32];
                tc::tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + 32 * c, v);
                tc::tmem_ld_wait();
                float l[32];
#pragma unroll
                for (int m = 0; m < 32; ++m) l[m] = __uint_as_float(v[m]) + (p.bias ? __ldg(p.bias + 32 * c + m) : 0.f);
                if (p.logits && t < p.T) {
                    float4* dst = reinterpret_cast<float4*>(p.logits + (size_t)t * E + 32 * c);
#pragma unroll
                    for (int m = 0; m < 8; ++m) dst[m] = make_float4(l[4 * m], l[4 * m + 1], l[4 * m + 2], l[4 * m + 3]);
                }
                // insertion into the sorted top-6; experts arrive in increasing
                // id, so a strict comparison keeps the lower id on equal logits
#pragma unroll
                for (int m = 0; m < 32; ++m) {
                    const float x = l[m];
                    if (x > tv[TOPK - 1]) {
                        tv[TOPK - 1] = x;
                        ti[TOPK - 1] = 32 * c + m;
#pragma unroll
                        for (int r = TOPK - 1; r > 0; --r) {
                            if (tv[r] > tv[r - 1]) {
                                const float a = tv[r];
                                tv[r] = tv[r - 1];
                                tv[r - 1] = a;
                                const int b = ti[r];
                                ti[r] = ti[r - 1];
                                ti[r - 1] = b;
                            }
                        }
                    }
                }
            }
        }
        float s[TOPK], sum = 0.f;
#pragma unroll
        for (int r = 0; r < TOPK; ++r) {
            s[r] = sigmoid_f(tv[r]);
            sum += s[r];
        }
        if (t < p.T) {
#pragma unroll
            for (int r = 0; r < TOPK; ++r) {
                p.idx[t * TOPK + r] = ti[r];
                p.w[t * TOPK + r] = s[r] / sum;
                atomicOr(&mask[ti[r] * 4 + (row >> 5)], 1u << (row & 31));
            }
        }
        epi_sync();
        if (t < p.T) {
#pragma unroll
            for (int r = 0; r < TOPK; ++r) {
                const uint32_t* m = mask + ti[r] * 4;
                int rank = __popc(m[row >> 5] & ((1u << (row & 31)) - 1u));
                for (int wd = 0; wd < (row >> 5); ++wd) rank += __popc(m[wd]);
                p.local_rank[t * TOPK + r] = rank;
            }
        }
        for (int e = row; e < E; e += 128)
            p.blk_counts[blk * E + e] = __popc(mask[e * 4]) + __popc(mask[e * 4 + 1]) + __popc(mask[e * 4 + 2]) +
                                        __popc(mask[e * 4 + 3]);
        if (!ok && row == 0) report_status(p.status, ST_TIMEOUT);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 256);
    }
}

// ---------------------------------------------------------------------------
// GEMM 1: gate/up + SwiGLU
// ---------------------------------------------------------------------------

constexpr int G1_STAGES = 3;
constexpr int G1_STAGE = 2 * PF_TILE_BYTES + GP_B_BYTES;    // gate, up, tokens: 64 KiB
constexpr int G1_BLOCKS = I / PF_TILE;                      // 4 row blocks of 128
constexpr int G1_SMEM = 1024 + G1_STAGES * G1_STAGE + 512 + GP_N * 4 + (int)sizeof(Sched) + 16 + GP_EPI_WARPS * STG_WARP;

__global__ void __launch_bounds__(G1_THREADS, 1)
    prefill_gateup_kernel(const __nv_bfloat16* __restrict__ x, GroupedParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + G1_STAGES * G1_STAGE);
    uint64_t* empty = full + G1_STAGES;
    uint64_t* tfull = empty + G1_STAGES;
    uint64_t* tempty = tfull + 1;
    uint64_t* mdone = tempty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdone + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* tok = reinterpret_cast<int*>(smem + G1_STAGES * G1_STAGE + 512);           // [GP_N]
    Sched* S = reinterpret_cast<Sched*>(tok + GP_N);
    uint8_t* stg_all = align16(reinterpret_cast<uint8_t*>(S + 1));                            // [8][STG_WARP]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = G1_THREADS / 32;
    // gather warps: warp 0 (which also issues the weight TMA) and the last warp
    const bool gather_warp = warp == 0 || warp == nwarps - 1;
    const int gw = warp == 0 ? 0 : 1;

    if (threadIdx.x == 0) {
        for (int s = 0; s < G1_STAGES; ++s) {
            // one arrive.expect_tx for the weight tiles + one cp.async arrival per gather thread
            mbar_init(&full[s], 1 + 32 * GP_GATHER_WARPS);
            mbar_init(&empty[s], 1);
        }
        mbar_init(tfull, 1);
        mbar_init(tempty, GP_EPI_WARPS);
        mbar_init(mdone, 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;   // gate accumulator: columns 0..255, up: 256..511
    pdl_wait();     // routing, permutation and x are complete
    pdl_trigger();
    build_sched(S, p, G1_BLOCKS);
    const int total = S->upre[NEXP];
    const int sixT = TOPK * p.T;
    constexpr int KC = H / PF_BK;   // 32

    if (gather_warp) {
        // Thread g of the 64 gather threads copies 16-byte chunk c = g % 8 of
        // token rows n = g / 8 + 8 i: eight lanes cover one 128-byte row, so a
        // warp-wide copy reads four whole rows.
        const int g = 32 * gw + lane, c = g & 7, r0 = g >> 3;
        const uint32_t dst_off = (uint32_t)r0 * 128u + ((uint32_t)(c ^ r0) << 4);   // n & 7 == r0
        int kc_all = 0;
        for (int u = blockIdx.x; u < total && !__shfl_sync(0xFFFFFFFFu, *abort, 0); u += gridDim.x) {
            const Unit U = decode_unit(S, u);
            // token of each of this thread's rows (padding rows repeat the last
            // valid token); npad is a multiple of 16, so rows i < npad / 8 are in
            const int nrows = U.npad >> 3;
            int tk[GP_N / 8];
#pragma unroll
            for (int i = 0; i < GP_N / 8; ++i) {
                const int slot = U.base + min(r0 + 8 * i, U.nvalid - 1);
                tk[i] = i < nrows ? (U.e < E ? __ldg(p.gather + slot) / TOPK : slot - sixT) : 0;
            }
            // gate tiles of row block blk, up tiles of row block 4 + blk
            const uint8_t* wt = reinterpret_cast<const uint8_t*>(p.tiled + (size_t)U.e * EXPERT_ELEMS);
            for (int kc = 0; kc < KC; ++kc, ++kc_all) {
                const int s = kc_all % G1_STAGES;
                bool ok = true;
                if (lane == 0) ok = pf_wait(&empty[s], ((kc_all / G1_STAGES) & 1) ^ 1, p.limit_ns, abort);
                if (!__shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0)) break;
                uint8_t* st = smem + s * G1_STAGE;
                if (warp == 0 && lane == 0) {
                    mbar_arrive_expect_tx(&full[s], 2 * PF_TILE_BYTES);
                    bulk_g2s(st, wt + (size_t)(U.blk * KC + kc) * PF_TILE_BYTES, PF_TILE_BYTES, &full[s]);
                    bulk_g2s(st + PF_TILE_BYTES, wt + (size_t)((I / PF_TILE + U.blk) * KC + kc) * PF_TILE_BYTES,
                             PF_TILE_BYTES, &full[s]);
                }
                // token rows into the 128-byte-swizzled K-major tile: 16-byte
                // chunk c of row n lands at n*128 + ((c ^ (n & 7)) * 16)
                uint8_t* bt = st + 2 * PF_TILE_BYTES + dst_off;
                const __nv_bfloat16* xk = x + kc * PF_BK + 8 * c;
#pragma unroll
                for (int i = 0; i < GP_N / 8; ++i)
                    if (i < nrows) tc::cp_async16(bt + i * 1024, xk + (size_t)tk[i] * H);
                tc::cp_async_arrive_noinc(&full[s]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int kc_all = 0, lu = 0;
            for (int u = blockIdx.x; u < total && !*abort; u += gridDim.x, ++lu) {
                const Unit U = decode_unit(S, u);
                if (!pf_wait(tempty, (lu & 1) ^ 1, p.limit_ns, abort)) break;
                tc::fence_after_sync();
                const uint32_t idesc = tc::idesc_bf16_f32(128, U.npad);
                for (int kc = 0; kc < KC; ++kc, ++kc_all) {
                    const int s = kc_all % G1_STAGES;
                    if (!pf_wait(&full[s], (kc_all / G1_STAGES) & 1, p.limit_ns, abort)) break;
                    // the token rows were written by cp.async (generic proxy); the
                    // tensor core reads smem through the async proxy
                    fence_proxy_async_smem();
                    tc::fence_after_sync();
                    const uint8_t* st = smem + s * G1_STAGE;
                    const uint64_t ag = tc::smem_desc_sw128(st), au = tc::smem_desc_sw128(st + PF_TILE_BYTES);
                    const uint64_t bx = tc::smem_desc_sw128(st + 2 * PF_TILE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < PF_BK / 16; ++kk) {
                        tc::mma_bf16(tmem, ag + 2 * kk, bx + 2 * kk, idesc, (kc | kk) != 0);
                        tc::mma_bf16(tmem + GP_N, au + 2 * kk, bx + 2 * kk, idesc, (kc | kk) != 0);
                    }
                    tc::mma_commit(&empty[s]);
                }
                tc::mma_commit(tfull);
            }
            // every MMA this thread issued has finished before TMEM is freed
            tc::mma_commit(mdone);
            mbar_wait_bounded(mdone, 0, p.limit_ns);
        }
        __syncwarp();
    } else {
        const int ew = warp - 2, q = warp & 3, half = ew >> 2;
        uint8_t* stg = stg_all + ew * STG_WARP;
        int lu = 0;
        for (int u = blockIdx.x; u < total; u += gridDim.x, ++lu) {
            const Unit U = decode_unit(S, u);
            if (!__all_sync(0xFFFFFFFFu, pf_wait(tfull, lu & 1, p.limit_ns, abort))) break;
            tc::fence_after_sync();
            const int j0 = U.blk * PF_TILE + 32 * q;   // this warp's 32 rows of h
            const uint32_t tg = tmem + ((uint32_t)(32 * q) << 16);
            // the two warps of a lane quarter take alternate 32-column chunks
            for (int c0 = 32 * half; c0 < U.npad; c0 += 64) {
                uint32_t g[32], up[32];
                tc::tmem_ld32(tg + c0, g);
                tc::tmem_ld32(tg + GP_N + c0, up);
                tc::tmem_ld_wait();
                float h[32];
#pragma unroll
                for (int m = 0; m < 32; ++m) h[m] = silu_fast(__uint_as_float(g[m])) * __uint_as_float(up[m]);
                stage_store_32x32(stg, lane, h, U.nvalid - c0, [&](int n) {
                    return p.h_perm + (size_t)(U.base + c0 + n) * I + j0;
                });
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty);
        }
    }
    if (*abort && threadIdx.x == 0) report_status(p.status, ST_TIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// ---------------------------------------------------------------------------
// GEMM 2: down projection + weighted scatter-add
// ---------------------------------------------------------------------------

constexpr int G2_STAGES = 4;
constexpr int G2_STAGE = PF_TILE_BYTES + GP_B_BYTES;   // down tile, activation tile: 48 KiB
constexpr int G2_BLOCKS = H / PF_TILE;                 // 16 row blocks of 128
constexpr int G2_SMEM = 1024 + G2_STAGES * G2_STAGE + 512 + (int)sizeof(Sched) + 16 + GP_EPI_WARPS * STG_WARP;

__global__ void __launch_bounds__(GP_THREADS, 1)
    prefill_down_kernel(const __grid_constant__ CUtensorMap h_map, GroupedParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + G2_STAGES * G2_STAGE);
    uint64_t* empty = full + G2_STAGES;
    uint64_t* tfull = empty + G2_STAGES;    // [2]
    uint64_t* tempty = tfull + 2;           // [2]
    uint64_t* mdone = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdone + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    Sched* S = reinterpret_cast<Sched*>(smem + G2_STAGES * G2_STAGE + 512);
    uint8_t* stg_all = align16(reinterpret_cast<uint8_t*>(S + 1));                           // [8][STG_WARP]
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < G2_STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], GP_EPI_WARPS);
        }
        mbar_init(mdone, 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(tmem_slot, 512);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;   // two accumulators of 256 columns
    pdl_wait();     // h_perm is complete
    pdl_trigger();
    build_sched(S, p, G2_BLOCKS);
    const int total = S->upre[NEXP];
    constexpr int KC = I / PF_BK;   // 8

    if (warp == 0) {
        if (lane == 0) {
            tc::prefetch_tensormap(&h_map);
            int kc_all = 0;
            for (int u = blockIdx.x; u < total && !*abort; u += gridDim.x) {
                const Unit U = decode_unit(S, u);
                const uint8_t* wt = reinterpret_cast<const uint8_t*>(p.tiled + (size_t)U.e * EXPERT_ELEMS +
                                                                     (size_t)2 * I * H);
                for (int kc = 0; kc < KC; ++kc, ++kc_all) {
                    const int s = kc_all % G2_STAGES;
                    if (!pf_wait(&empty[s], ((kc_all / G2_STAGES) & 1) ^ 1, p.limit_ns, abort)) break;
                    uint8_t* st = smem + s * G2_STAGE;
                    mbar_arrive_expect_tx(&full[s], PF_TILE_BYTES + GP_B_BYTES);
                    bulk_g2s(st, wt + (size_t)(U.blk * KC + kc) * PF_TILE_BYTES, PF_TILE_BYTES, &full[s]);
                    tc::tma_load_2d(st + PF_TILE_BYTES, &h_map, kc * PF_BK, U.base, &full[s]);
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            int kc_all = 0, lu = 0;
            for (int u = blockIdx.x; u < total && !*abort; u += gridDim.x, ++lu) {
                const Unit U = decode_unit(S, u);
                const int b = lu & 1;
                if (!pf_wait(&tempty[b], ((lu >> 1) & 1) ^ 1, p.limit_ns, abort)) break;
                tc::fence_after_sync();
                const uint32_t idesc = tc::idesc_bf16_f32(128, U.npad);
                const uint32_t d = tmem + b * GP_N;
                for (int kc = 0; kc < KC; ++kc, ++kc_all) {
                    const int s = kc_all % G2_STAGES;
                    if (!pf_wait(&full[s], (kc_all / G2_STAGES) & 1, p.limit_ns, abort)) break;
                    tc::fence_after_sync();
                    const uint8_t* st = smem + s * G2_STAGE;
                    const uint64_t a = tc::smem_desc_sw128(st), bh = tc::smem_desc_sw128(st + PF_TILE_BYTES);
#pragma unroll
                    for (int kk = 0; kk < PF_BK / 16; ++kk)
                        tc::mma_bf16(d, a + 2 * kk, bh + 2 * kk, idesc, (kc | kk) != 0);
                    tc::mma_commit(&empty[s]);
                }
                tc::mma_commit(&tfull[b]);
            }
            tc::mma_commit(mdone);
            mbar_wait_bounded(mdone, 0, p.limit_ns);
        }
        __syncwarp();
    } else {
        const int ew = warp - 2, q = warp & 3, half = ew >> 2;
        uint8_t* stg = stg_all + ew * STG_WARP;
        int lu = 0;
        for (int u = blockIdx.x; u < total; u += gridDim.x, ++lu) {
            const Unit U = decode_unit(S, u);
            const int b = lu & 1;
            if (!__all_sync(0xFFFFFFFFu, pf_wait(&tfull[b], (lu >> 1) & 1, p.limit_ns, abort))) break;
            tc::fence_after_sync();
            const int h0 = U.blk * PF_TILE + 32 * q;   // this warp's 32 rows of the output
            const uint32_t td = tmem + ((uint32_t)(32 * q) << 16) + b * GP_N;
            for (int c0 = 32 * half; c0 < U.npad; c0 += 64) {
                uint32_t v[32];
                tc::tmem_ld32(td + c0, v);
                tc::tmem_ld_wait();
                float o[32];
#pragma unroll
                for (int m = 0; m < 32; ++m) o[m] = __uint_as_float(v[m]);
                stage_store_32x32(stg, lane, o, U.nvalid - c0, [&](int n) {
                    return p.o_perm + (size_t)(U.base + c0 + n) * H + h0;
                });
            }
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[b]);
        }
    }
    if (*abort && threadIdx.x == 0) report_status(p.status, ST_TIMEOUT);
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, 512);
    }
}

// y[t] = sum_j w[t][j] * o_perm[slot(t, j)] + o_perm[6T + t], summed in fp32 in
// slot order (the six routed experts by decreasing logit, then the shared
// expert): deterministic.  One thread per 8 output columns of a token.
__global__ void __launch_bounds__(256) combine_kernel(const __nv_bfloat16* __restrict__ o_perm,
                                                     const int32_t* __restrict__ pair_slot,
                                                     const float* __restrict__ w_route, int T,
                                                     __nv_bfloat16* __restrict__ y) {
    pdl_wait();
    pdl_trigger();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= T * (H / 8)) return;
    const int t = i / (H / 8), c = (i % (H / 8)) * 8;
    float acc[8];
    {
        const uint4 v = __ldcg(reinterpret_cast<const uint4*>(o_perm + ((size_t)TOPK * T + t) * H + c));
        acc[0] = bf_lo(v.x); acc[1] = bf_hi(v.x); acc[2] = bf_lo(v.y); acc[3] = bf_hi(v.y);
        acc[4] = bf_lo(v.z); acc[5] = bf_hi(v.z); acc[6] = bf_lo(v.w); acc[7] = bf_hi(v.w);
    }
    float r[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) r[k] = 0.f;
#pragma unroll
    for (int j = 0; j < TOPK; ++j) {
        const int slot = __ldg(pair_slot + t * TOPK + j);
        const float wj = __ldg(w_route + t * TOPK + j);
        const uint4 v = __ldcg(reinterpret_cast<const uint4*>(o_perm + (size_t)slot * H + c));
        r[0] = fmaf(wj, bf_lo(v.x), r[0]); r[1] = fmaf(wj, bf_hi(v.x), r[1]);
        r[2] = fmaf(wj, bf_lo(v.y), r[2]); r[3] = fmaf(wj, bf_hi(v.y), r[3]);
        r[4] = fmaf(wj, bf_lo(v.z), r[4]); r[5] = fmaf(wj, bf_hi(v.z), r[5]);
        r[6] = fmaf(wj, bf_lo(v.w), r[6]); r[7] = fmaf(wj, bf_hi(v.w), r[7]);
    }
    __nv_bfloat162 out[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) out[k] = __floats2bfloat162_rn(r[2 * k] + acc[2 * k], r[2 * k + 1] + acc[2 * k + 1]);
    *reinterpret_cast<uint4*>(y + (size_t)t * H + c) = *reinterpret_cast<const uint4*>(out);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

cudaError_t prefill_set_attributes() {
    cudaError_t e = cudaFuncSetAttribute(prefill_router_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, RG_SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(prefill_gateup_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, G1_SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(prefill_down_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, G2_SMEM);
    return e;
}

cudaError_t launch_prefill_router(const LaunchCtx& L, const CUtensorMap& x_map, const CUtensorMap& wr_map, int T,
                                  const float* bias, float* logits, int32_t* idx, float* w, int32_t* local_rank,
                                  int32_t* blk_counts) {
    RouterGemmParams rp{T, bias, logits, idx, w, local_rank, blk_counts, L.status, L.wait_limit_ns};
    return launch_hooked(L, FLINT_KERNEL_ROUTER, prefill_router_kernel, dim3((T + PF_TILE - 1) / PF_TILE), dim3(PF_THREADS), RG_SMEM, x_map,
                      wr_map, rp);
}

cudaError_t launch_prefill_experts(const LaunchCtx& L, const __nv_bfloat16* x, const CUtensorMap& h_map, int T,
                                   const int32_t* offsets, const int32_t* gather, const int32_t* pair_slot,
                                   const float* w_route, const __nv_bfloat16* tiled, __nv_bfloat16* h_perm,
                                   __nv_bfloat16* o_perm, __nv_bfloat16* y) {
    GroupedParams gp{T, offsets, gather, w_route, tiled, h_perm, o_perm, L.status, L.wait_limit_ns};
    cudaError_t e = launch_hooked(L, FLINT_KERNEL_GATE_UP, prefill_gateup_kernel, dim3(L.num_sms), dim3(G1_THREADS), G1_SMEM, x, gp);
    if (e != cudaSuccess) return e;
    e = launch_hooked(L, FLINT_KERNEL_DOWN, prefill_down_kernel, dim3(L.num_sms), dim3(GP_THREADS), G2_SMEM, h_map, gp);
    if (e != cudaSuccess) return e;
    return launch_prefill_combine(L, o_perm, pair_slot, w_route, T, y);
}

cudaError_t launch_prefill_combine(const LaunchCtx& L, const __nv_bfloat16* o_perm, const int32_t* pair_slot,
                                   const float* w_route, int T, __nv_bfloat16* y) {
    const int n8 = T * (H / 8);
    return launch_hooked(L, FLINT_KERNEL_COMBINE, combine_kernel, dim3((n8 + 255) / 256), dim3(256), 0, o_perm,
                         pair_slot, w_route, T, y);
}

}  // namespace flint
