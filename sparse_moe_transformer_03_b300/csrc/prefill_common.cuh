// prefill_common.cuh -- pieces shared by the grouped tensor-core GEMMs of
// the many-token path (bf16 experts in prefill.cu, NVFP4 experts in
// prefill_nvfp4.cu): tile sizes, the bounded waits, the persistent unit
// schedule over (expert, row block, token pass) and the epilogue's staged
// stores.
#pragma once

#include "flint_common.cuh"
#include "flint_internal.h"
#include "tc_ptx.cuh"

namespace flint {

constexpr int PF_THREADS = 192;
constexpr int PF_TILE = 128;                 // rows of every operand tile
constexpr int PF_BK = 64;                    // K per stage: 128 bytes of bf16
constexpr int PF_TILE_BYTES = PF_TILE * PF_BK * 2;   // 16 KiB
constexpr size_t EXPERT_ELEMS = (size_t)3 * H * I;   // one expert's gate_up + down

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ uint8_t* align16(uint8_t* p) {
    return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 15) & ~uintptr_t(15));
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// Named barrier of the 128 epilogue threads that also ANDs a predicate, so a
// decision to give up is taken by all of them together.
__device__ __forceinline__ bool epi_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.cta.red.and.pred q, 1, 128, p;\n"
        " selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(v ? 1u : 0u)
        : "memory");
    return r != 0;
}

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool pf_wait(uint64_t* bar, uint32_t parity, uint64_t limit, volatile int* abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 16; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*abort) return false;
        if (globaltimer_ns() - t0 > limit) {
            *abort = 1;
            return false;
        }
    }
}

// ===========================================================================
// grouped expert GEMMs
// ===========================================================================
// A unit is (expert, row block, token pass): 128 rows of one expert matrix
// against up to GP_N (256) of its tokens.  Most experts receive fewer than
// 256 tokens, so each weight tile is streamed from HBM once and used for all
// of the expert's tokens; passes of one row block are adjacent in the unit
// order so larger experts share the tile through L2.

constexpr int GP_N = 256;                        // tokens per pass (MMA N <= 256)
constexpr int GP_EPI_WARPS = 8;                  // two per TMEM lane quarter
constexpr int GP_GATHER_WARPS = 2;               // token-row gathers of the gate/up GEMM
constexpr int GP_THREADS = 64 + 32 * GP_EPI_WARPS;   // producer + MMA + epilogue
constexpr int G1_THREADS = GP_THREADS + 32;      // + a second gather warp (the last warp)
constexpr int GP_B_BYTES = GP_N * PF_BK * 2;     // 32 KiB

__device__ __forceinline__ void gp_epi_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(32 * GP_EPI_WARPS) : "memory");
}
__device__ __forceinline__ bool gp_epi_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n barrier.cta.red.and.pred q, 1, %2, p;\n"
        " selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "n"(32 * GP_EPI_WARPS)
        : "memory");
    return r != 0;
}

// Epilogue staging: each epilogue warp holds a 32 (tokens) x 32 (rows) bf16
// tile, written column-wise from TMEM lanes and read back row-wise so every
// lane stores 64 contiguous bytes of one token row (rows padded to 80 bytes
// so both phases are free of bank conflicts).
constexpr int STG_ROW = 80;                       // bytes per staged token row
constexpr int STG_WARP = 32 * STG_ROW;            // 2.5 KiB per epilogue warp

// lane = row r of a 32-row block holding 32 token values v[n] (fp32): stage
// them as bf16 and let lane n write its 64-byte token row to dst(n).
template <typename DstFn>
__device__ __forceinline__ void stage_store_32x32(uint8_t* stg, int lane, const float (&v)[32], int nvalid_here,
                                                  DstFn dst) {
#pragma unroll
    for (int m = 0; m < 32; ++m)
        *reinterpret_cast<__nv_bfloat16*>(stg + m * STG_ROW + 2 * lane) = __float2bfloat16_rn(v[m]);
    __syncwarp();
    if (lane < nvalid_here) {
        const uint4* src = reinterpret_cast<const uint4*>(stg + lane * STG_ROW);
        uint4* d = reinterpret_cast<uint4*>(dst(lane));
        d[0] = src[0];
        d[1] = src[1];
        d[2] = src[2];
        d[3] = src[3];
    }
    __syncwarp();
}

struct GroupedParams {
    int T;
    const int32_t* offsets;      // [E+1] slot base of each routed expert (6T total)
    const int32_t* gather;       // [6T] pair ids t*6+j grouped by expert
    const float* w_route;        // [T][6]
    const __nv_bfloat16* tiled;  // [NEXP] x (gate_up tiles, down tiles), 16 KiB tiles (repack.cu)
    __nv_bfloat16* h_perm;       // [7T][I]
    __nv_bfloat16* o_perm;       // [7T][H] per-slot expert outputs
    uint32_t* status;
    uint64_t limit_ns;
    const float* nv_ts;          // NVFP4 experts: tensor scales [NEXP][2] (gate_up, down)
};

// Per-CTA copy of the unit schedule: expert e covers units
// [upre[e], upre[e+1]); its slots start at base[e] and number cnt[e].
struct Sched {
    int base[NEXP + 1];
    int cnt[NEXP];
    int upre[NEXP + 1];
};

__device__ inline void build_sched(Sched* S, const GroupedParams& p, int blocks) {
    const int tid = threadIdx.x;
    for (int e = tid; e < NEXP; e += blockDim.x) {
        const int b = e < E ? p.offsets[e] : TOPK * p.T;
        const int n = e < E ? p.offsets[e + 1] - b : p.T;
        S->base[e] = b;
        S->cnt[e] = n;
    }
    __syncthreads();
    if (tid < 32) {
        // exclusive scan of units over the 257 experts, 9 per lane
        int loc[9], sum = 0;
#pragma unroll
        for (int k = 0; k < 9; ++k) {
            const int e = tid * 9 + k;
            loc[k] = e < NEXP ? blocks * ((S->cnt[e] + GP_N - 1) / GP_N) : 0;
            sum += loc[k];
        }
        int inc = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int a = __shfl_up_sync(0xFFFFFFFFu, inc, o);
            if (tid >= o) inc += a;
        }
        int run = inc - sum;
#pragma unroll
        for (int k = 0; k < 9; ++k) {
            const int e = tid * 9 + k;
            if (e < NEXP) S->upre[e] = run;
            run += loc[k];
        }
        if (tid == 31) S->upre[NEXP] = run;
    }
    __syncthreads();
}

// expert of unit u (binary search over the prefix)
__device__ __forceinline__ int unit_expert(const Sched* S, int u) {
    int lo = 0, hi = NEXP - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (S->upre[mid] <= u) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

struct Unit {
    int e, blk, pass, base, nvalid, npad;
};

// unit order within an expert: (row block, pass)
__device__ __forceinline__ Unit decode_unit(const Sched* S, int u) {
    Unit U;
    U.e = unit_expert(S, u);
    const int np = (S->cnt[U.e] + GP_N - 1) / GP_N;
    const int r = u - S->upre[U.e];
    U.blk = r / np;
    U.pass = r - U.blk * np;
    U.base = S->base[U.e] + U.pass * GP_N;
    U.nvalid = min(GP_N, S->cnt[U.e] - U.pass * GP_N);
    U.npad = (U.nvalid + 15) & ~15;
    return U;
}

}  // namespace flint
