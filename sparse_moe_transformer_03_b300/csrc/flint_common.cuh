// flint_common.cuh -- shapes, workspace layout and inline-PTX helpers shared
// by the sm_103a kernels of the Flint MoE layer.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace flint {

constexpr int H = 2048;          // model width
constexpr int I = 512;           // expert intermediate width
constexpr int E = 256;           // routed experts
constexpr int TOPK = 6;          // routed experts per token
constexpr int SHARED = 256;      // expert index of the shared expert
constexpr int NEXP = 257;        // routed + shared
constexpr int CHUNK = 8192;      // tokens per internal chunk
constexpr int DEC_T = 32;        // decode path: T <= DEC_T
constexpr int DEC_PAIRS = DEC_T * (TOPK + 1);

// device status codes (mirrors flint_status_t)
constexpr uint32_t ST_TIMEOUT = 4;
constexpr uint32_t ST_BADINDEX = 5;
constexpr uint32_t ST_INTERNAL = 7;   // an internal capacity check failed (a library defect)

// Per-call routing tables of the decode path, written by the router's last
// CTA.  Slot 0 is the shared expert (all T tokens, weight 1); slots 1..U are
// the routed experts touched by the batch in increasing expert id, each with
// its tokens in increasing token id.  A "pair" is one (expert slot, token).
struct DecodeTables {
    int n_slots;                  // U + 1
    int n_pairs;                  // 7T
    int T;
    int pad_;
    int slot_expert[NEXP];        // expert id of each slot (256 = shared)
    int slot_pair0[NEXP + 1];     // first pair of each slot
    int slot_tile0[NEXP + 1];     // first 8-token tile of each slot (tiles = ceil(pairs / 8))
    int pair_token[DEC_PAIRS];    // token of each pair
    float pair_weight[DEC_PAIRS]; // routing weight of each pair (shared: 1)
};

// The decode activations a = silu(g) * u (bf16), written by the gate/up
// kernels and read by the down kernels, in two column halves: half h holds
// columns 256h .. 256h + 255 of every pair as [DEC_ACT_ROWS][256], so the
// 8 pairs of one token tile are 4 KiB of contiguous bytes (one bulk copy).
// Within a row the 16-byte chunk k sits at k ^ (pair % 8): the 8 rows of a
// tile read the same column through different banks.  DEC_ACT_ROWS leaves 8
// rows of slack after the last pair so a tile's copy stays inside its half.
constexpr int DEC_ACT_ROWS = DEC_PAIRS + 8;
constexpr size_t DEC_ACT_BYTES = (size_t)2 * DEC_ACT_ROWS * 256 * 2;
__host__ __device__ __forceinline__ size_t act_index(int pair, int j) {
    const int h = j >> 8, k = (j >> 3) & 31;
    return ((size_t)h * DEC_ACT_ROWS + pair) * 256 + ((k ^ (pair & 7)) << 3) + (j & 7);
}

// ---------------------------------------------------------------------------
// small helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Record a device error in the status word (host-mapped memory): the last
// writer wins, any non-zero value is an error.
__device__ __forceinline__ void report_status(uint32_t* status, uint32_t code) {
    if (status) {
        *reinterpret_cast<volatile uint32_t*>(status) = code;
        __threadfence_system();
    }
}

// bf16 pair in a 32-bit word -> two floats (exact)
__device__ __forceinline__ float bf_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ float silu_f(float z) { return z / (1.0f + expf(-z)); }
__device__ __forceinline__ float sigmoid_f(float z) { return 1.0f / (1.0f + expf(-z)); }
// silu through the hardware base-2 exponential and reciprocal approximations:
// exp(-z) = 2^(-z log2(e)).  Relative error a few 1e-7 (far below bf16
// rounding); z -> -inf gives 2^+inf = inf, 1/inf = 0 and the result -0.
__device__ __forceinline__ float silu_fast(float z) {
    float e, r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(e) : "f"(z * -1.4426950408889634f));
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(1.0f + e));
    return z * r;
}

// ---------------------------------------------------------------------------
// programmatic dependent launch
// ---------------------------------------------------------------------------

// Block until the grids this grid depends on have completed and their memory
// is visible.  A no-op when the kernel was not launched as a dependent.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel on the stream to be scheduled early (it must itself
// call pdl_wait before touching anything this grid writes).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// mbarrier + bulk asynchronous copies
// ---------------------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

// Make mbarrier initialisation visible to the asynchronous proxy.
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// Raise the phase's expected transaction bytes without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, giving up after
// limit_ns nanoseconds of %globaltimer.  Returns false on timeout.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
}

// One bulk copy global -> shared (contiguous bytes), completing on `bar`.
// dst and src 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Hint: bring [src, src+bytes) into L2 (bytes a multiple of 16).
__device__ __forceinline__ void bulk_prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 16-byte read-only global load
__device__ __forceinline__ uint4 ldg16(const void* p) { return __ldg(reinterpret_cast<const uint4*>(p)); }

// 16-byte load that bypasses L1 (data written by other CTAs of this grid)
__device__ __forceinline__ float4 ldcg_f4(const float* p) { return __ldcg(reinterpret_cast<const float4*>(p)); }

}  // namespace flint
