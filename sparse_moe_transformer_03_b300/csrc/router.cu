// router.cu -- router logits, sigmoid top-6 selection with renormalisation,
// the decode routing tables and the token->expert permutation.
//
// RecursiveSI/flint (vLLM recipe page), "Overview": 256 experts with top-6
// sigmoid routing plus a shared expert.  The selection ranks experts by the
// fp32 logit (the sigmoid is increasing, so this is the ranking by score
// without its fp32 saturation), keeps the lower expert index on equal logits,
// and renormalises the six sigmoid scores to sum to one.
#include "flint_common.cuh"
#include "../../include/flint_moe.h"
#include "flint_internal.h"
#include "routing.cuh"

namespace flint {

// ---------------------------------------------------------------------------
// decode router: logits for T <= 32
// ---------------------------------------------------------------------------

constexpr int RT_WARPS = 4;                    // one expert per warp
constexpr int RT_CTAS = E / RT_WARPS;          // 64

// Logits only (the expert kernels of the forward select for themselves).
// Grid: (64 expert groups of 4, token groups of RL_TOK).  Each warp keeps its
// expert's 4 KiB router row in registers (loaded before the dependency wait);
// the CTA stages its tokens' x rows in smem with one bulk copy, so a token
// costs shared-memory reads instead of an L2 round trip.
constexpr int RL_TOK = 8;

__global__ void __launch_bounds__(RT_WARPS * 32) router_logits_decode_kernel(const __nv_bfloat16* x, int T,
                                                                           const __nv_bfloat16* Wr,
                                                                           const float* bias, float* logits,
                                                                           uint32_t* status, uint64_t limit_ns) {
    __shared__ __align__(128) __nv_bfloat16 xs[RL_TOK * H];   // 32 KiB
    __shared__ __align__(8) uint64_t xbar;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * RT_WARPS + warp;
    const int t0 = blockIdx.y * RL_TOK, nt = min(RL_TOK, T - t0);
    uint4 wr[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) wr[i] = ldg16(Wr + (size_t)e * H + 8 * (lane + 32 * i));
    const float b = bias ? __ldg(bias + e) : 0.f;
    if (threadIdx.x == 0) {
        mbar_init(&xbar, 1);
        fence_mbar_init();
    }
    __syncthreads();
    pdl_trigger();
    pdl_wait();
    if (threadIdx.x == 0) {
        mbar_arrive_expect_tx(&xbar, nt * H * 2);
        bulk_g2s(xs, x + (size_t)t0 * H, nt * H * 2, &xbar);
    }
    const bool ok = __syncthreads_and(mbar_wait_bounded(&xbar, 0, limit_ns));
    if (!ok) {         // the copy did not complete in time: the logits are not written
        if (threadIdx.x == 0) report_status(status, ST_TIMEOUT);
        return;
    }
    for (int t = 0; t < nt; ++t) {
        const __nv_bfloat16* xr = xs + t * H;
        float acc = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint4 xv = *reinterpret_cast<const uint4*>(xr + 8 * (lane + 32 * i));
            acc = fmaf(bf_lo(wr[i].x), bf_lo(xv.x), acc);
            acc = fmaf(bf_hi(wr[i].x), bf_hi(xv.x), acc);
            acc = fmaf(bf_lo(wr[i].y), bf_lo(xv.y), acc);
            acc = fmaf(bf_hi(wr[i].y), bf_hi(xv.y), acc);
            acc = fmaf(bf_lo(wr[i].z), bf_lo(xv.z), acc);
            acc = fmaf(bf_hi(wr[i].z), bf_hi(xv.z), acc);
            acc = fmaf(bf_lo(wr[i].w), bf_lo(xv.w), acc);
            acc = fmaf(bf_hi(wr[i].w), bf_hi(xv.w), acc);
        }
        acc = warp_sum(acc);
        if (lane == 0) logits[(size_t)(t0 + t) * E + e] = acc + b;
    }
}

// ---------------------------------------------------------------------------
// selection from given fp32 logits (route-only fed with logits): one warp per
// token, the same warp top-6 as the forward path
// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(128) select_kernel(const float* logits, int T, int32_t* idx, float* w) {
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int t = blockIdx.x * 4 + warp;
    if (t >= T) return;
    float v[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __ldcg(logits + (size_t)t * E + lane + 32 * i);
    int sel[TOPK];
    float wt[TOPK];
    warp_top6(v, lane, sel, wt);
    if (lane < TOPK) {
        idx[t * TOPK + lane] = pick6(sel, lane);
        w[t * TOPK + lane] = pick6(wt, lane);
    }
}

// ---------------------------------------------------------------------------
// permutation: stable counting sort of the (token, slot) pairs by expert
// ---------------------------------------------------------------------------
// Blocks of PB_TOK tokens.  perm_local: per block, each pair's rank among the
// block's earlier pairs of the same expert (from per-expert token bitmasks,
// so the result is deterministic) and the block's per-expert counts.
// perm_scan: offsets[e] and each block's base per expert.  perm_scatter:
// gather[offsets[e] + base[b][e] + rank] = pair id.

constexpr int PB_TOK = PERM_BLOCK_TOKENS;

__global__ void __launch_bounds__(PB_TOK) perm_local_kernel(const int32_t* idx, int T, int32_t* local_rank,
                                                           int32_t* blk_counts, uint32_t* status) {
    pdl_wait();
    __shared__ uint32_t mask[E][PB_TOK / 32];
    const int b = blockIdx.x, tid = threadIdx.x;
    for (int i = tid; i < E * (PB_TOK / 32); i += PB_TOK) (&mask[0][0])[i] = 0u;
    __syncthreads();
    const int t = b * PB_TOK + tid;
    int sel[TOPK];
    if (t < T) {
#pragma unroll
        for (int j = 0; j < TOPK; ++j) {
            int e = idx[t * TOPK + j];
            if (e < 0 || e >= E) {
                report_status(status, ST_BADINDEX);
                e = 0;
            }
            sel[j] = e;
            atomicOr(&mask[e][tid >> 5], 1u << (tid & 31));
        }
    }
    __syncthreads();
    if (t < T) {
#pragma unroll
        for (int j = 0; j < TOPK; ++j) {
            const int e = sel[j];
            int r = 0;
            for (int wd = 0; wd < (tid >> 5); ++wd) r += __popc(mask[e][wd]);
            r += __popc(mask[e][tid >> 5] & ((1u << (tid & 31)) - 1u));
            local_rank[t * TOPK + j] = r;
        }
    }
    for (int e = tid; e < E; e += PB_TOK) {
        int c = 0;
#pragma unroll
        for (int wd = 0; wd < PB_TOK / 32; ++wd) c += __popc(mask[e][wd]);
        blk_counts[b * E + e] = c;
    }
}

__global__ void __launch_bounds__(E) perm_scan_kernel(const int32_t* __restrict__ blk_counts, int nblk,
                                                     int32_t* __restrict__ blk_base, int32_t* __restrict__ offsets) {
    pdl_wait();
    const int e = threadIdx.x;
    int run = 0;
    // independent loads, 16 in flight at a time
    for (int b0 = 0; b0 < nblk; b0 += 16) {
        int c[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) c[k] = b0 + k < nblk ? __ldcg(blk_counts + (b0 + k) * E + e) : 0;
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            if (b0 + k < nblk) blk_base[(b0 + k) * E + e] = run;
            run += c[k];
        }
    }
    // exclusive scan of run over the 256 experts
    __shared__ int warp_tot[E / 32];
    const int lane = e & 31, wid = e >> 5;
    int incl = run;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += a;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    int before = 0;
    for (int i = 0; i < wid; ++i) before += warp_tot[i];
    offsets[e] = before + incl - run;
    if (e == E - 1) offsets[E] = before + incl;
}

__global__ void __launch_bounds__(256) perm_scatter_kernel(const int32_t* idx, const int32_t* local_rank, int T,
                                                          const int32_t* blk_base, const int32_t* offsets,
                                                          int32_t* gather, int32_t* pair_slot) {
    pdl_wait();
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= T * TOPK) return;
    const int t = p / TOPK;
    const int b = t / PB_TOK;
    const int e = idx[p];
    if (e < 0 || e >= E) return;
    const int slot = offsets[e] + blk_base[b * E + e] + local_rank[p];
    gather[slot] = p;
    if (pair_slot) pair_slot[p] = slot;
}

// ---------------------------------------------------------------------------
// host launchers
// ---------------------------------------------------------------------------

cudaError_t launch_router_logits_decode(const LaunchCtx& L, const __nv_bfloat16* x, int T,
                                        const __nv_bfloat16* Wr, const float* bias, float* logits) {
    return launch_hooked(L, FLINT_KERNEL_ROUTER, router_logits_decode_kernel,
                         dim3(RT_CTAS, (T + RL_TOK - 1) / RL_TOK), dim3(RT_WARPS * 32), 0, x, T, Wr, bias, logits,
                         L.status, L.wait_limit_ns);
}

cudaError_t launch_select(const LaunchCtx& L, const float* logits, int T, int32_t* idx, float* w) {
    return launch_pdl(L, select_kernel, dim3((T + 3) / 4), dim3(128), 0, logits, T, idx, w);
}

cudaError_t launch_permutation(const LaunchCtx& L, const int32_t* idx, int T, int32_t* local_rank,
                               int32_t* blk_counts, int32_t* blk_base, int32_t* offsets, int32_t* gather) {
    const int nblk = (T + PB_TOK - 1) / PB_TOK;
    cudaError_t err = launch_pdl(L, perm_local_kernel, dim3(nblk), dim3(PB_TOK), 0, idx, T, local_rank,
                                 blk_counts, L.status);
    if (err != cudaSuccess) return err;
    err = launch_pdl(L, perm_scan_kernel, dim3(1), dim3(E), 0, (const int32_t*)blk_counts, nblk, blk_base,
                     offsets);
    if (err != cudaSuccess) return err;
    if (!gather) return cudaSuccess;
    return launch_pdl(L, perm_scatter_kernel, dim3((T * TOPK + 255) / 256), dim3(256), 0, idx,
                      (const int32_t*)local_rank, T, (const int32_t*)blk_base, (const int32_t*)offsets, gather,
                      (int32_t*)nullptr);
}

cudaError_t launch_perm_scan_scatter(const LaunchCtx& L, const int32_t* idx, int T, const int32_t* local_rank,
                                     const int32_t* blk_counts, int32_t* blk_base, int32_t* offsets,
                                     int32_t* gather, int32_t* pair_slot) {
    const int nblk = (T + PB_TOK - 1) / PB_TOK;
    cudaError_t err = launch_pdl(L, perm_scan_kernel, dim3(1), dim3(E), 0, blk_counts, nblk, blk_base, offsets);
    if (err != cudaSuccess || !gather) return err;
    return launch_pdl(L, perm_scatter_kernel, dim3((T * TOPK + 255) / 256), dim3(256), 0, idx, local_rank, T,
                      (const int32_t*)blk_base, (const int32_t*)offsets, gather, pair_slot);
}

}  // namespace flint
