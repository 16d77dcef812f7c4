// prefill_nvfp4.cu -- the many-token path (T > 32) for NVFP4 experts, run as
// W4A16: the grouped tcgen05 GEMMs of prefill.cu with the weight operand
// dequantised on chip.
//
// Per K step of 64 columns of a unit's 128 weight rows:
//   * one elected thread copies, by TMA, the step's E2M1 codes and E4M3
//     block scales straight out of the owned NVFP4 layout (decode_nvfp4.cu:
//     4608-byte chunks of 16 rows x 512 columns, codes in mma.sync A-fragment
//     order) into a raw ring: 576 bytes per 16 rows;
//   * eight dequantising warps turn them into a bf16 tile in the canonical
//     128-byte-swizzle K-major layout the MMA reads.  code x block scale is
//     exact in bf16 (at most 6 significant bits); the fp32 tensor scale
//     multiplies the accumulator in the epilogue;
//   * the tokens (gate/up: rows of x gathered by cp.async; down: h_perm
//     tiles by TMA), the single MMA-issuing thread, the TMEM epilogues, the
//     persistent unit schedule and the combine are those of the bf16 path.
// The weight bytes streamed from HBM are 4.5 bits per weight instead of 16.
//
// NVFP4 weights: e2m1(q) * e4m3(s_block) * s_tensor with one block scale per
// 16 consecutive columns of a row; the checkpoint is run as W4A16
// (RecursiveSI/flint vLLM recipe page, "Overview").
#include <cuda_fp16.h>

#include "../../include/flint_moe.h"
#include "flint_common.cuh"
#include "flint_internal.h"
#include "nvfp4_frag.cuh"
#include "prefill_common.cuh"
#include "tc_ptx.cuh"

namespace flint {

constexpr int NQ_WARPS = 8;      // dequantising warps
constexpr int NQ_WBUF = 2;       // bf16 weight stages

// Raw ring entry of one K step (4 K blocks) of a 128-row block made of
// `units` owned units of 16 rows: the codes ([unit][4 x 128 bytes]) then the
// scales ([unit][4 x 16 bytes]), as the two TMA boxes land them.
__host__ __device__ constexpr int nq_raw_codes(int units) { return units * 4 * 128; }
__host__ __device__ constexpr int nq_raw_bytes(int units) { return units * 4 * (128 + 16); }

// One 16 x 16 block (K block kbl of the step) of an owned unit, dequantised
// by the warp into the swizzled bf16 tile: A-fragment rows g and g + 8 go to
// the tile rows at row_lo and row_hi (both with row % 8 == g, so the
// 16-byte chunk of columns 16 kbl + 8 h lands at chunk (2 kbl + h) ^ g and
// the 32 lanes' 4-byte stores hit 32 different banks).
__device__ __forceinline__ void nq_dequant_block(const uint8_t* codes, const uint8_t* scales, int kbl, int lane,
                                                 uint8_t* row_lo, uint8_t* row_hi) {
    const int g = lane >> 2, c = lane & 3;
    uint32_t a[4];
    nv_a_frag(*reinterpret_cast<const uint32_t*>(codes + kbl * 128 + 4 * lane),
              *reinterpret_cast<const uint16_t*>(scales + kbl * 16 + 2 * g), a);
    const int c0 = (((2 * kbl) ^ g) << 4) + 4 * c, c1 = (((2 * kbl + 1) ^ g) << 4) + 4 * c;
    *reinterpret_cast<uint32_t*>(row_lo + c0) = f16x2_to_bf16x2(a[0]);
    *reinterpret_cast<uint32_t*>(row_hi + c0) = f16x2_to_bf16x2(a[1]);
    *reinterpret_cast<uint32_t*>(row_lo + c1) = f16x2_to_bf16x2(a[2]);
    *reinterpret_cast<uint32_t*>(row_hi + c1) = f16x2_to_bf16x2(a[3]);
}

// Copies still in flight after an abort: wait (briefly) for the last stages
// the producer issued before the CTA exits.
__device__ __forceinline__ void nq_drain(uint64_t* bars, int stages, int issued) {
    for (int q = issued > stages ? issued - stages : 0; q < issued; ++q)
        mbar_wait_bounded(&bars[q % stages], (q / stages) & 1, 10000000ull);
}

// ---------------------------------------------------------------------------
// GEMM 1: gate/up + SwiGLU
// ---------------------------------------------------------------------------
// Warps: 0 = TMA of the raw weights (lane 0) and token gather, 1 = TMEM and
// MMA issue, 2..9 = epilogue, 10 = token gather, 11..18 = dequantisation.
// Rings: NQ_WBUF bf16 weight stages (gate tile, up tile), N1_STAGES stages of
// (token tile, raw weights).

constexpr int N1_UNITS = PF_TILE / 8;                         // owned gate/up units per 128-row block
constexpr int N1_RAW = nq_raw_bytes(N1_UNITS);                // 9 KiB
constexpr int N1_STAGES = 3;
constexpr int N1_STAGE = GP_B_BYTES + N1_RAW;                 // 41 KiB
constexpr int N1_WSTAGE = 2 * PF_TILE_BYTES;                  // 32 KiB
constexpr int N1_BLOCKS = I / PF_TILE;                        // 4 row blocks
constexpr int N1_THREADS = G1_THREADS + 32 * NQ_WARPS;        // 608
constexpr int N1_UPW = N1_UNITS / NQ_WARPS;                   // owned units per dequantising warp
constexpr int N1_DQ0 = G1_THREADS / 32;                       // first dequantising warp
constexpr int N1_SMEM =
    1024 + NQ_WBUF * N1_WSTAGE + N1_STAGES * N1_STAGE + 512 + (int)sizeof(Sched) + 16 + GP_EPI_WARPS * STG_WARP;
static_assert(N1_STAGE % 1024 == 0, "token tiles must stay 1024-byte aligned");
static_assert(N1_SMEM <= 232448, "shared memory per block");

__global__ void __launch_bounds__(N1_THREADS, 1)
    prefill_gateup_nvfp4_kernel(const __nv_bfloat16* __restrict__ x, const __grid_constant__ CUtensorMap code_map,
                                const __grid_constant__ CUtensorMap scale_map, GroupedParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* wring = smem;                                    // [NQ_WBUF][gate | up]
    uint8_t* sring = smem + NQ_WBUF * N1_WSTAGE;              // [N1_STAGES][tokens | raw]
    uint64_t* sfull = reinterpret_cast<uint64_t*>(sring + N1_STAGES * N1_STAGE);
    uint64_t* sempty = sfull + N1_STAGES;
    uint64_t* rfull = sempty + N1_STAGES;
    uint64_t* wfull = rfull + N1_STAGES;
    uint64_t* wempty = wfull + NQ_WBUF;
    uint64_t* tfull = wempty + NQ_WBUF;
    uint64_t* tempty = tfull + 1;
    uint64_t* mdone = tempty + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdone + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    Sched* S = reinterpret_cast<Sched*>(sring + N1_STAGES * N1_STAGE + 512);
    uint8_t* stg_all = align16(reinterpret_cast<uint8_t*>(S + 1));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < N1_STAGES; ++s) {
            mbar_init(&sfull[s], 32 * GP_GATHER_WARPS);   // one cp.async arrival per gather thread
            mbar_init(&sempty[s], 1);
            mbar_init(&rfull[s], 1);
        }
        for (int w = 0; w < NQ_WBUF; ++w) {
            mbar_init(&wfull[w], NQ_WARPS);
            mbar_init(&wempty[w], 1);
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
    build_sched(S, p, N1_BLOCKS);
    const int total = S->upre[NEXP];
    const int sixT = TOPK * p.T;
    constexpr int KC = H / PF_BK;   // 32

    if (warp == 0 || warp == N1_DQ0 - 1) {
        // token gather (as in the bf16 kernel); warp 0's lane 0 also issues the
        // raw weight copies of the stage
        const int gw = warp == 0 ? 0 : 1;
        const int g = 32 * gw + lane, c = g & 7, r0 = g >> 3;
        const uint32_t dst_off = (uint32_t)r0 * 128u + ((uint32_t)(c ^ r0) << 4);
        if (warp == 0 && lane == 0) {
            tc::prefetch_tensormap(&code_map);
            tc::prefetch_tensormap(&scale_map);
        }
        int kc_all = 0;
        for (int u = blockIdx.x; u < total && !__shfl_sync(0xFFFFFFFFu, *abort, 0); u += gridDim.x) {
            const Unit U = decode_unit(S, u);
            const int nrows = U.npad >> 3;
            int tk[GP_N / 8];
#pragma unroll
            for (int i = 0; i < GP_N / 8; ++i) {
                const int slot = U.base + min(r0 + 8 * i, U.nvalid - 1);
                tk[i] = i < nrows ? (U.e < E ? __ldg(p.gather + slot) / TOPK : slot - sixT) : 0;
            }
            bool ok = true;
            for (int kc = 0; kc < KC; ++kc, ++kc_all) {
                const int s = kc_all % N1_STAGES;
                if (lane == 0) ok = pf_wait(&sempty[s], ((kc_all / N1_STAGES) & 1) ^ 1, p.limit_ns, abort);
                if (!__shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0)) break;
                uint8_t* st = sring + s * N1_STAGE;
                if (warp == 0 && lane == 0) {
                    uint8_t* raw = st + GP_B_BYTES;
                    mbar_arrive_expect_tx(&rfull[s], N1_RAW);
                    tc::tma_load_4d(raw, &code_map, 128 * (kc & 7), kc >> 3, N1_UNITS * U.blk, U.e, &rfull[s]);
                    tc::tma_load_4d(raw + nq_raw_codes(N1_UNITS), &scale_map, 1024 + 16 * (kc & 7), kc >> 3,
                                    N1_UNITS * U.blk, U.e, &rfull[s]);
                }
                uint8_t* bt = st + dst_off;
                const __nv_bfloat16* xk = x + kc * PF_BK + 8 * c;
#pragma unroll
                for (int i = 0; i < GP_N / 8; ++i)
                    if (i < nrows) tc::cp_async16(bt + i * 1024, xk + (size_t)tk[i] * H);
                tc::cp_async_arrive_noinc(&sfull[s]);
            }
            if (!__shfl_sync(0xFFFFFFFFu, ok ? 1 : 0, 0)) break;
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (warp == 0 && lane == 0 && *abort) nq_drain(rfull, N1_STAGES, kc_all);
        __syncwarp();
    } else if (warp == 1) {
        if (lane == 0) {
            int kc_all = 0, lu = 0;
            for (int u = blockIdx.x; u < total && !*abort; u += gridDim.x, ++lu) {
                const Unit U = decode_unit(S, u);
                if (!pf_wait(tempty, (lu & 1) ^ 1, p.limit_ns, abort)) break;
                tc::fence_after_sync();
                const uint32_t idesc = tc::idesc_bf16_f32(128, U.npad);
                for (int kc = 0; kc < KC; ++kc, ++kc_all) {
                    const int s = kc_all % N1_STAGES, w = kc_all % NQ_WBUF;
                    if (!pf_wait(&sfull[s], (kc_all / N1_STAGES) & 1, p.limit_ns, abort)) break;
                    if (!pf_wait(&wfull[w], (kc_all / NQ_WBUF) & 1, p.limit_ns, abort)) break;
                    // token rows (cp.async) and weight tiles (st.shared) were written
                    // through the generic proxy; the tensor core reads the async proxy
                    fence_proxy_async_smem();
                    tc::fence_after_sync();
                    const uint8_t* wt = wring + w * N1_WSTAGE;
                    const uint64_t ag = tc::smem_desc_sw128(wt), au = tc::smem_desc_sw128(wt + PF_TILE_BYTES);
                    const uint64_t bx = tc::smem_desc_sw128(sring + s * N1_STAGE);
#pragma unroll
                    for (int kk = 0; kk < PF_BK / 16; ++kk) {
                        tc::mma_bf16(tmem, ag + 2 * kk, bx + 2 * kk, idesc, (kc | kk) != 0);
                        tc::mma_bf16(tmem + GP_N, au + 2 * kk, bx + 2 * kk, idesc, (kc | kk) != 0);
                    }
                    tc::mma_commit(&sempty[s]);
                    tc::mma_commit(&wempty[w]);
                }
                tc::mma_commit(tfull);
            }
            tc::mma_commit(mdone);
            mbar_wait_bounded(mdone, 0, p.limit_ns);
        }
        __syncwarp();
    } else if (warp >= N1_DQ0) {
        // dequantisation: warp d takes owned units N1_UPW d .. N1_UPW (d + 1) - 1
        // of the block (gate and up rows 8 N1_UPW d ..)
        const int d = warp - N1_DQ0, g = lane >> 2;
        int kc_all = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < total; u += gridDim.x) {
            for (int kc = 0; kc < KC; ++kc, ++kc_all) {
                const int s = kc_all % N1_STAGES, w = kc_all % NQ_WBUF;
                ok = __all_sync(0xFFFFFFFFu, pf_wait(&rfull[s], (kc_all / N1_STAGES) & 1, p.limit_ns, abort) &&
                                                 pf_wait(&wempty[w], ((kc_all / NQ_WBUF) & 1) ^ 1, p.limit_ns, abort));
                if (!ok) break;
                const uint8_t* raw = sring + s * N1_STAGE + GP_B_BYTES;
                uint8_t* gt = wring + w * N1_WSTAGE;
#pragma unroll
                for (int qi = 0; qi < N1_UPW; ++qi) {
                    const int ql = N1_UPW * d + qi;
                    const uint8_t* codes = raw + ql * 512;
                    const uint8_t* scales = raw + nq_raw_codes(N1_UNITS) + ql * 64;
                    uint8_t* row_g = gt + (8 * ql + g) * 128;            // gate row 8 ql + g of the block
                    uint8_t* row_u = row_g + PF_TILE_BYTES;             // up row 8 ql + g
#pragma unroll
                    for (int kbl = 0; kbl < 4; ++kbl) nq_dequant_block(codes, scales, kbl, lane, row_g, row_u);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&wfull[w]);
            }
        }
    } else {
        const int ew = warp - 2, q = warp & 3, half = ew >> 2;
        uint8_t* stg = stg_all + ew * STG_WARP;
        int lu = 0;
        for (int u = blockIdx.x; u < total; u += gridDim.x, ++lu) {
            const Unit U = decode_unit(S, u);
            if (!__all_sync(0xFFFFFFFFu, pf_wait(tfull, lu & 1, p.limit_ns, abort))) break;
            tc::fence_after_sync();
            const float ts = __ldg(p.nv_ts + 2 * U.e);    // gate_up tensor scale
            const int j0 = U.blk * PF_TILE + 32 * q;
            const uint32_t tg = tmem + ((uint32_t)(32 * q) << 16);
            for (int c0 = 32 * half; c0 < U.npad; c0 += 64) {
                uint32_t gr[32], up[32];
                tc::tmem_ld32(tg + c0, gr);
                tc::tmem_ld32(tg + GP_N + c0, up);
                tc::tmem_ld_wait();
                float h[32];
#pragma unroll
                for (int m = 0; m < 32; ++m)
                    h[m] = silu_fast(ts * __uint_as_float(gr[m])) * (ts * __uint_as_float(up[m]));
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
// GEMM 2: down projection
// ---------------------------------------------------------------------------
// Warps: 0 = TMA of activation tiles and raw weights (lane 0), 1 = TMEM and
// MMA issue, 2..9 = epilogue (two TMEM accumulators), 10..17 = dequantisation.

constexpr int N2_UNITS = PF_TILE / 16;                        // owned down units per 128-row block
constexpr int N2_RAW = nq_raw_bytes(N2_UNITS);                // 4.5 KiB
constexpr int N2_STAGES = 4;
constexpr int N2_STAGE = GP_B_BYTES + 5 * 1024;               // activations, raw (padded): 37 KiB
constexpr int N2_WSTAGE = PF_TILE_BYTES;                      // 16 KiB
constexpr int N2_BLOCKS = H / PF_TILE;                        // 16 row blocks
constexpr int N2_THREADS = GP_THREADS + 32 * NQ_WARPS;        // 576
constexpr int N2_UPW = N2_UNITS / NQ_WARPS;
constexpr int N2_DQ0 = GP_THREADS / 32;
constexpr int N2_SMEM =
    1024 + NQ_WBUF * N2_WSTAGE + N2_STAGES * N2_STAGE + 512 + (int)sizeof(Sched) + 16 + GP_EPI_WARPS * STG_WARP;
static_assert(N2_RAW <= N2_STAGE - GP_B_BYTES, "raw entry fits its stage");
static_assert(N2_STAGE % 1024 == 0, "activation tiles must stay 1024-byte aligned");
static_assert(N2_SMEM <= 232448, "shared memory per block");

__global__ void __launch_bounds__(N2_THREADS, 1)
    prefill_down_nvfp4_kernel(const __grid_constant__ CUtensorMap h_map, const __grid_constant__ CUtensorMap code_map,
                              const __grid_constant__ CUtensorMap scale_map, GroupedParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = align1024(smem_raw);
    uint8_t* wring = smem;                                    // [NQ_WBUF][down tile]
    uint8_t* sring = smem + NQ_WBUF * N2_WSTAGE;              // [N2_STAGES][activations | raw]
    uint64_t* sfull = reinterpret_cast<uint64_t*>(sring + N2_STAGES * N2_STAGE);
    uint64_t* sempty = sfull + N2_STAGES;
    uint64_t* rfull = sempty + N2_STAGES;
    uint64_t* wfull = rfull + N2_STAGES;
    uint64_t* wempty = wfull + NQ_WBUF;
    uint64_t* tfull = wempty + NQ_WBUF;     // [2]
    uint64_t* tempty = tfull + 2;           // [2]
    uint64_t* mdone = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mdone + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    Sched* S = reinterpret_cast<Sched*>(sring + N2_STAGES * N2_STAGE + 512);
    uint8_t* stg_all = align16(reinterpret_cast<uint8_t*>(S + 1));
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < N2_STAGES; ++s) {
            mbar_init(&sfull[s], 1);
            mbar_init(&sempty[s], 1);
            mbar_init(&rfull[s], 1);
        }
        for (int w = 0; w < NQ_WBUF; ++w) {
            mbar_init(&wfull[w], NQ_WARPS);
            mbar_init(&wempty[w], 1);
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
    build_sched(S, p, N2_BLOCKS);
    const int total = S->upre[NEXP];
    constexpr int KC = I / PF_BK;   // 8

    if (warp == 0) {
        if (lane == 0) {
            tc::prefetch_tensormap(&h_map);
            tc::prefetch_tensormap(&code_map);
            tc::prefetch_tensormap(&scale_map);
            int kc_all = 0;
            for (int u = blockIdx.x; u < total && !*abort; u += gridDim.x) {
                const Unit U = decode_unit(S, u);
                for (int kc = 0; kc < KC; ++kc) {
                    const int s = kc_all % N2_STAGES;
                    if (!pf_wait(&sempty[s], ((kc_all / N2_STAGES) & 1) ^ 1, p.limit_ns, abort)) break;
                    uint8_t* st = sring + s * N2_STAGE;
                    uint8_t* raw = st + GP_B_BYTES;
                    mbar_arrive_expect_tx(&rfull[s], N2_RAW);
                    tc::tma_load_3d(raw, &code_map, 128 * kc, N2_UNITS * U.blk, U.e, &rfull[s]);
                    tc::tma_load_3d(raw + nq_raw_codes(N2_UNITS), &scale_map, 1024 + 16 * kc, N2_UNITS * U.blk, U.e,
                                    &rfull[s]);
                    mbar_arrive_expect_tx(&sfull[s], GP_B_BYTES);
                    tc::tma_load_2d(st, &h_map, kc * PF_BK, U.base, &sfull[s]);
                    ++kc_all;
                }
            }
            if (*abort) {
                nq_drain(rfull, N2_STAGES, kc_all);
                nq_drain(sfull, N2_STAGES, kc_all);
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
                const uint32_t dacc = tmem + b * GP_N;
                for (int kc = 0; kc < KC; ++kc, ++kc_all) {
                    const int s = kc_all % N2_STAGES, w = kc_all % NQ_WBUF;
                    if (!pf_wait(&sfull[s], (kc_all / N2_STAGES) & 1, p.limit_ns, abort)) break;
                    if (!pf_wait(&wfull[w], (kc_all / NQ_WBUF) & 1, p.limit_ns, abort)) break;
                    fence_proxy_async_smem();   // the weight tile was written through the generic proxy
                    tc::fence_after_sync();
                    const uint64_t a = tc::smem_desc_sw128(wring + w * N2_WSTAGE);
                    const uint64_t bh = tc::smem_desc_sw128(sring + s * N2_STAGE);
#pragma unroll
                    for (int kk = 0; kk < PF_BK / 16; ++kk)
                        tc::mma_bf16(dacc, a + 2 * kk, bh + 2 * kk, idesc, (kc | kk) != 0);
                    tc::mma_commit(&sempty[s]);
                    tc::mma_commit(&wempty[w]);
                }
                tc::mma_commit(&tfull[b]);
            }
            tc::mma_commit(mdone);
            mbar_wait_bounded(mdone, 0, p.limit_ns);
        }
        __syncwarp();
    } else if (warp >= N2_DQ0) {
        // dequantisation: warp d takes owned units N2_UPW d .. (rows 16 N2_UPW d ..)
        const int d = warp - N2_DQ0, g = lane >> 2;
        int kc_all = 0;
        bool ok = true;
        for (int u = blockIdx.x; ok && u < total; u += gridDim.x) {
            for (int kc = 0; kc < KC; ++kc, ++kc_all) {
                const int s = kc_all % N2_STAGES, w = kc_all % NQ_WBUF;
                ok = __all_sync(0xFFFFFFFFu, pf_wait(&rfull[s], (kc_all / N2_STAGES) & 1, p.limit_ns, abort) &&
                                                 pf_wait(&wempty[w], ((kc_all / NQ_WBUF) & 1) ^ 1, p.limit_ns, abort));
                if (!ok) break;
                const uint8_t* raw = sring + s * N2_STAGE + GP_B_BYTES;
                uint8_t* tile = wring + w * N2_WSTAGE;
#pragma unroll
                for (int vi = 0; vi < N2_UPW; ++vi) {
                    const int v = N2_UPW * d + vi;
                    const uint8_t* codes = raw + v * 512;
                    const uint8_t* scales = raw + nq_raw_codes(N2_UNITS) + v * 64;
                    uint8_t* row_lo = tile + (16 * v + g) * 128;
#pragma unroll
                    for (int kbl = 0; kbl < 4; ++kbl) nq_dequant_block(codes, scales, kbl, lane, row_lo, row_lo + 1024);
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(&wfull[w]);
            }
        }
    } else {
        const int ew = warp - 2, q = warp & 3, half = ew >> 2;
        uint8_t* stg = stg_all + ew * STG_WARP;
        int lu = 0;
        for (int u = blockIdx.x; u < total; u += gridDim.x, ++lu) {
            const Unit U = decode_unit(S, u);
            const int b = lu & 1;
            if (!__all_sync(0xFFFFFFFFu, pf_wait(&tfull[b], (lu >> 1) & 1, p.limit_ns, abort))) break;
            tc::fence_after_sync();
            const float ts = __ldg(p.nv_ts + 2 * U.e + 1);    // down tensor scale
            const int h0 = U.blk * PF_TILE + 32 * q;
            const uint32_t td = tmem + ((uint32_t)(32 * q) << 16) + b * GP_N;
            for (int c0 = 32 * half; c0 < U.npad; c0 += 64) {
                uint32_t v[32];
                tc::tmem_ld32(td + c0, v);
                tc::tmem_ld_wait();
                float o[32];
#pragma unroll
                for (int m = 0; m < 32; ++m) o[m] = ts * __uint_as_float(v[m]);
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

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

cudaError_t prefill_nvfp4_set_attributes() {
    cudaError_t e =
        cudaFuncSetAttribute(prefill_gateup_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, N1_SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(prefill_down_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, N2_SMEM);
    return e;
}

bool encode_nvfp4_prefill_maps(CUtensorMap (&maps)[4], const uint8_t* nv) {
    return encode_nvfp4_gateup(&maps[0], nv, 128, N1_UNITS) && encode_nvfp4_gateup(&maps[1], nv, 16, N1_UNITS) &&
           encode_nvfp4_down(&maps[2], nv, 128, N2_UNITS) && encode_nvfp4_down(&maps[3], nv, 16, N2_UNITS);
}

cudaError_t launch_prefill_experts_nvfp4(const LaunchCtx& L, const __nv_bfloat16* x, const CUtensorMap& h_map,
                                         const CUtensorMap (&maps)[4], int T, const int32_t* offsets,
                                         const int32_t* gather, const int32_t* pair_slot, const float* w_route,
                                         const float* nv_ts, __nv_bfloat16* h_perm, __nv_bfloat16* o_perm,
                                         __nv_bfloat16* y) {
    GroupedParams gp{T, offsets, gather, w_route, nullptr, h_perm, o_perm, L.status, L.wait_limit_ns, nv_ts};
    cudaError_t e = launch_hooked(L, FLINT_KERNEL_GATE_UP, prefill_gateup_nvfp4_kernel, dim3(L.num_sms),
                                  dim3(N1_THREADS), N1_SMEM, x, maps[0], maps[1], gp);
    if (e != cudaSuccess) return e;
    e = launch_hooked(L, FLINT_KERNEL_DOWN, prefill_down_nvfp4_kernel, dim3(L.num_sms), dim3(N2_THREADS), N2_SMEM,
                      h_map, maps[2], maps[3], gp);
    if (e != cudaSuccess) return e;
    return launch_prefill_combine(L, o_perm, pair_slot, w_route, T, y);
}

}  // namespace flint
