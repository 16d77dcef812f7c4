// lm_head.cu -- the 4-bit output layer: logits[t][v] = sum_h x[t][h] W[v][h]
// for a decode batch (T <= 32), W an NVFP4 matrix [V][2048] run as W4A16.
// The pages report that Flint's output head was quantised to 4 bits too
// (mrchatgpt.org article, section 4, the quantisation item; qantcore.space
// review, section 04, the quantised variants); V is not on the pages.
//
// Design (HBM-bound weight streaming, one launch):
//   * the handle owns W repacked into the chunk layout of the NVFP4 expert
//     kernels (decode_nvfp4.cu, kind 2): units of 16 rows x 2048 columns, four
//     4608-byte chunks each (codes in mma.sync A-fragment order, then the E4M3
//     block scales), 1152 bytes per row;
//   * one persistent CTA per SM takes a balanced contiguous range of units;
//     a producer warp streams their chunks by bulk copy into a ring of
//     4608-byte slots, issued round-robin over the consumer warps (chunk c of
//     every warp's unit, then chunk c + 1, ...), so each warp has its next
//     chunk in flight while it works on the current one;
//   * 16 consumer warps: warp w multiplies whole units (16 rows x K 2048) by
//     the tokens, dequantising each 16 x 16 block straight into an f16 A
//     fragment (nvfp4_frag.cuh) and multiplying it with x staged in shared
//     memory as f16 (token t scaled by 2^e_t so that its largest |x| lies in
//     [2^14, 2^15): exact for every bf16 value within 28 binades of it); the
//     fp32 accumulators get s_tensor * 2^-e_t at the end and the warp writes
//     its 16 logits per token;
//   * a slot's sequence word (release / acquire in shared memory) tells a
//     consumer that the producer armed the slot for that use before it waits
//     on the slot's barrier parity, so warps that share a slot at different
//     uses never see each other's phase.
// Every wait is bounded by %globaltimer; a wait that gives up sets the CTA's
// abort flag, reports FLINT_ERR_DEVICE_TIMEOUT through the status word and
// the producer drains its copies in flight before the CTA exits.
#include <cuda_fp16.h>

#include <new>

#include "../../include/flint_moe.h"
#include "flint_common.cuh"
#include "flint_internal.h"
#include "mma_sync.cuh"
#include "nvfp4_frag.cuh"

namespace flint {
namespace {

constexpr int LH_NW = 16;                          // consumer warps
constexpr int LH_THREADS = 32 * (LH_NW + 1);       // + the producer warp
constexpr int LH_XSTRIDE = 2 * H + 16;             // bytes per staged token row (bank spread)
constexpr int LH_UNIT = NV_GU_CHUNKS * NV_CHUNK;   // 18432 bytes: 16 rows x 2048
constexpr int LH_MAX_SLOTS = 64;

struct LmParams {
    const uint8_t* nv;          // owned layout, units * LH_UNIT bytes
    float ts;                   // tensor scale
    const __nv_bfloat16* x;     // [T][H]
    float* logits;              // [T][V]
    int T, V, units, nslot;
    uint32_t* status;
    uint64_t limit_ns;
};

// dynamic shared memory: ring | x (8 NT rows) | xinv[32] | seq[nslot] | full | empty | abort
__host__ __device__ constexpr uint32_t lh_x_off(int nslot) { return (uint32_t)nslot * NV_CHUNK; }
__host__ __device__ constexpr uint32_t lh_xinv_off(int nslot, int nt) {
    return lh_x_off(nslot) + (uint32_t)(8 * nt) * LH_XSTRIDE;
}
__host__ __device__ constexpr uint32_t lh_seq_off(int nslot, int nt) { return lh_xinv_off(nslot, nt) + 32 * 4; }
__host__ __device__ constexpr uint32_t lh_bar_off(int nslot, int nt) {
    return (lh_seq_off(nslot, nt) + (uint32_t)nslot * 4 + 7) & ~7u;
}
__host__ __device__ constexpr uint32_t lh_smem_bytes(int nslot, int nt) {
    return lh_bar_off(nslot, nt) + (uint32_t)nslot * 16 + 16;
}

__device__ __forceinline__ void lh_st_release(uint32_t* p, uint32_t v) {
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t lh_ld_acquire(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
    return v;
}

struct LmState {
    uint8_t* ring;
    uint32_t* seq;
    uint64_t* full;
    uint64_t* empty;
    volatile uint32_t* abort;
    int nslot;
    uint64_t limit;
};

__device__ __forceinline__ void lh_fail(const LmState& s, uint32_t* status) {
    *s.abort = 1;
    report_status(status, ST_TIMEOUT);
}

// bounded parity wait that also gives up once another warp aborted
__device__ __forceinline__ bool lh_wait(const LmState& s, uint64_t* bar, uint32_t parity, uint32_t* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*s.abort) return false;
        if (globaltimer_ns() - t0 > s.limit) {
            lh_fail(s, status);
            return false;
        }
    }
}

// ring entry q has landed: first the producer's arming of slot q % nslot for
// use q / nslot (sequence word q + 1), then that use's barrier phase
__device__ __forceinline__ bool lh_wait_full(const LmState& s, uint32_t q, uint32_t* status) {
    const int slot = (int)(q % (uint32_t)s.nslot);
    if (lh_ld_acquire(&s.seq[slot]) != q + 1u) {
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
            bool armed = false;
#pragma unroll 1
            for (int i = 0; i < 64 && !armed; ++i) armed = lh_ld_acquire(&s.seq[slot]) == q + 1u;
            if (armed) break;
            if (*s.abort) return false;
            if (globaltimer_ns() - t0 > s.limit) {
                lh_fail(s, status);
                return false;
            }
        }
    }
    return lh_wait(s, &s.full[slot], (q / (uint32_t)s.nslot) & 1, status);
}

// Ring entry of chunk c of the unit that warp w takes in round r (n units in
// the CTA): rounds before r hold 4 LH_NW entries each; round r holds
// 4 nw_r, chunk-major over its nw_r active warps.
__device__ __forceinline__ uint32_t lh_entry(int r, int c, int w, int n) {
    const int nw = min(LH_NW, n - r * LH_NW);
    return (uint32_t)(4 * LH_NW * r + c * nw + w);
}

template <int NT>   // token tiles of 8: T <= 8 NT
__global__ void __launch_bounds__(LH_THREADS, 1) lm_head_nvfp4_kernel(LmParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    LmState s;
    s.nslot = p.nslot;
    s.limit = p.limit_ns;
    s.ring = smem;
    uint8_t* xs = smem + lh_x_off(p.nslot);
    float* xinv = reinterpret_cast<float*>(smem + lh_xinv_off(p.nslot, NT));
    s.seq = reinterpret_cast<uint32_t*>(smem + lh_seq_off(p.nslot, NT));
    s.full = reinterpret_cast<uint64_t*>(smem + lh_bar_off(p.nslot, NT));
    s.empty = s.full + p.nslot;
    s.abort = reinterpret_cast<volatile uint32_t*>(s.empty + p.nslot);
    // the CTA's units: a balanced contiguous range
    const int G = gridDim.x, c = blockIdx.x;
    const int u0 = (int)((long long)p.units * c / G), u1 = (int)((long long)p.units * (c + 1) / G);
    const int n = u1 - u0, rounds = (n + LH_NW - 1) / LH_NW;
    const uint32_t nslot = (uint32_t)p.nslot;

    if (threadIdx.x == 0) {
        for (int i = 0; i < p.nslot; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
            s.seq[i] = 0;
        }
        *s.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == LH_NW) {
        // producer: chunk entries in ring order (round, chunk, warp)
        if (lane == 0) {
            uint32_t q = 0;
            bool ok = true;
            for (int r = 0; ok && r < rounds; ++r) {
                const int nw = min(LH_NW, n - r * LH_NW);
                for (int cc = 0; ok && cc < NV_GU_CHUNKS; ++cc) {
                    for (int w = 0; w < nw; ++w) {
                        const uint32_t slot = q % nslot;
                        if (q >= nslot && !lh_wait(s, &s.empty[slot], (q / nslot - 1) & 1, p.status)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(&s.full[slot], NV_CHUNK);
                        lh_st_release(&s.seq[slot], q + 1u);
                        bulk_g2s(s.ring + (size_t)slot * NV_CHUNK,
                                 p.nv + (size_t)(u0 + r * LH_NW + w) * LH_UNIT + (size_t)cc * NV_CHUNK, NV_CHUNK,
                                 &s.full[slot]);
                        ++q;
                    }
                }
            }
            // after an abort: the copies in flight land before the CTA exits
            if (*s.abort)
                for (uint32_t k = q > nslot ? q - nslot : 0u; k < q; ++k)
                    mbar_wait_bounded(&s.full[k % nslot], (k / nslot) & 1, 10000000ull);
        }
        return;
    }

    // consumers: x -> f16 x 2^e_t, token t on warp t % LH_NW (rows past T zero)
    for (int t = warp; t < 8 * NT; t += LH_NW) {
        uint4* row = reinterpret_cast<uint4*>(xs + (size_t)t * LH_XSTRIDE);
        if (t < p.T) {
            const uint4* src = reinterpret_cast<const uint4*>(p.x + (size_t)t * H);
            uint4 v[8];
            float mx = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                v[k] = __ldg(src + lane + 32 * k);
                mx = fmaxf(mx, fmaxf(fmaxf(fabsf(bf_lo(v[k].x)), fabsf(bf_hi(v[k].x))),
                                     fmaxf(fabsf(bf_lo(v[k].y)), fabsf(bf_hi(v[k].y)))));
                mx = fmaxf(mx, fmaxf(fmaxf(fabsf(bf_lo(v[k].z)), fabsf(bf_hi(v[k].z))),
                                     fmaxf(fabsf(bf_lo(v[k].w)), fabsf(bf_hi(v[k].w)))));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
            int e = mx > 0.f ? 14 - ilogbf(mx) : 0;
            e = e > 126 ? 126 : e;
            const float sc = ldexpf(1.f, e);
            if (lane == 0) xinv[t] = ldexpf(1.f, -e);
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const __half2 h0 = __floats2half2_rn(bf_lo(v[k].x) * sc, bf_hi(v[k].x) * sc);
                const __half2 h1 = __floats2half2_rn(bf_lo(v[k].y) * sc, bf_hi(v[k].y) * sc);
                const __half2 h2 = __floats2half2_rn(bf_lo(v[k].z) * sc, bf_hi(v[k].z) * sc);
                const __half2 h3 = __floats2half2_rn(bf_lo(v[k].w) * sc, bf_hi(v[k].w) * sc);
                uint4 o;
                o.x = *reinterpret_cast<const uint32_t*>(&h0);
                o.y = *reinterpret_cast<const uint32_t*>(&h1);
                o.z = *reinterpret_cast<const uint32_t*>(&h2);
                o.w = *reinterpret_cast<const uint32_t*>(&h3);
                row[lane + 32 * k] = o;
            }
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) row[lane + 32 * k] = make_uint4(0, 0, 0, 0);
            if (lane == 0) xinv[t] = 0.f;
        }
    }
    asm volatile("bar.sync 1, %0;" ::"n"(32 * LH_NW) : "memory");   // the consumer warps only

    // units: warp w takes unit r LH_NW + w of the range in round r
    constexpr int ACC = NT >= 4 ? 1 : (NT == 1 ? 4 : 2);   // independent accumulator chains per tile
    const int g = lane >> 2, cq = lane & 3;
    bool ok = true;
    for (int r = 0; ok && r < rounds; ++r) {
        const int nw = min(LH_NW, n - r * LH_NW);
        if (warp >= nw) break;                  // only the last round is partial
        float acc[ACC][NT][4];
#pragma unroll
        for (int a = 0; a < ACC; ++a)
#pragma unroll
            for (int j = 0; j < NT; ++j) acc[a][j][0] = acc[a][j][1] = acc[a][j][2] = acc[a][j][3] = 0.f;
        for (int cc = 0; cc < NV_GU_CHUNKS; ++cc) {
            const uint32_t q = lh_entry(r, cc, warp, n);
            if (!__all_sync(0xFFFFFFFFu, lh_wait_full(s, q, p.status))) {
                ok = false;
                break;
            }
            const uint8_t* buf = s.ring + (size_t)(q % nslot) * NV_CHUNK;
            // B: token 8 j + g, columns 512 cc + 16 kb + 2 cq (and + 8)
            const uint8_t* xb = xs + (size_t)g * LH_XSTRIDE + cc * 1024 + 4 * cq;
#pragma unroll
            for (int kb = 0; kb < NV_CHUNK_KB; ++kb) {
                uint32_t a[4];
                nv_a_frag(*reinterpret_cast<const uint32_t*>(buf + kb * 128 + 4 * lane),
                          *reinterpret_cast<const uint16_t*>(buf + NV_CODES + kb * 16 + 2 * g), a);
#pragma unroll
                for (int j = 0; j < NT; ++j) {
                    const uint8_t* xj = xb + (size_t)j * 8 * LH_XSTRIDE + kb * 32;
                    mma_f16_16816(acc[kb % ACC][j], a, *reinterpret_cast<const uint32_t*>(xj),
                                  *reinterpret_cast<const uint32_t*>(xj + 16));
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.empty[q % nslot]);
        }
        if (!ok) break;
        // lane (g, cq): rows v0 and v0 + 8, tokens 8 j + 2 cq and + 1
        const size_t v0 = (size_t)16 * (u0 + r * LH_NW + warp) + g;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            float d[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                d[i] = acc[0][j][i];
#pragma unroll
                for (int a = 1; a < ACC; ++a) d[i] += acc[a][j][i];
            }
            const int t0 = 8 * j + 2 * cq, t1 = t0 + 1;
            if (t0 < p.T) {
                const float f = p.ts * xinv[t0];
                p.logits[(size_t)t0 * p.V + v0] = d[0] * f;
                p.logits[(size_t)t0 * p.V + v0 + 8] = d[2] * f;
            }
            if (t1 < p.T) {
                const float f = p.ts * xinv[t1];
                p.logits[(size_t)t1 * p.V + v0] = d[1] * f;
                p.logits[(size_t)t1 * p.V + v0 + 8] = d[3] * f;
            }
        }
    }
}

// largest ring (<= LH_MAX_SLOTS chunk slots) that fits the opt-in shared memory
int lh_nslot(int nt, int smem_optin) {
    int k = LH_MAX_SLOTS;
    while (k > 0 && lh_smem_bytes(k, nt) > (uint32_t)smem_optin) --k;
    return k;
}

template <int NT>
cudaError_t lh_launch(const LmParams& p0, int grid, int smem_optin, cudaStream_t s) {
    LmParams p = p0;
    p.nslot = lh_nslot(NT, smem_optin);
    if (p.nslot < 1) return cudaErrorInvalidConfiguration;
    lm_head_nvfp4_kernel<NT><<<grid, LH_THREADS, lh_smem_bytes(p.nslot, NT), s>>>(p);
    return cudaGetLastError();
}

template <int NT>
cudaError_t lh_set_attr(int smem_optin) {
    return cudaFuncSetAttribute(lm_head_nvfp4_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_optin);
}

}  // namespace
}  // namespace flint

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------

struct flint_lm_head {
    int device, num_sms, smem_optin;
    int V, units;
    uint8_t* nv;                 // owned repacked W
    float ts;
    uint32_t* status_host;       // host-mapped status word
    uint32_t* status_dev;
    uint64_t limit_ns;
};

namespace {

void lh_free(flint_lm_head* h) {
    if (h->nv) cudaFree(h->nv);
    if (h->status_host) cudaFreeHost(h->status_host);
    delete h;
}

flint_status_t lh_take_status(flint_lm_head* h) {
    volatile uint32_t* s = h->status_host;
    const uint32_t v = *s;
    if (v == 0) return FLINT_OK;
    *s = 0;
    if (v == flint::ST_TIMEOUT) return FLINT_ERR_DEVICE_TIMEOUT;
    if (v == flint::ST_INTERNAL) return FLINT_ERR_INTERNAL;
    return FLINT_ERR_CUDA;
}

}  // namespace

extern "C" {

flint_status_t flint_lm_head_create(flint_lm_head_t* out, const flint_nvfp4_t* W, int V) {
    using namespace flint;
    if (!out) return FLINT_ERR_INVALID_ARG;
    *out = nullptr;
    if (!W || !W->packed || !W->block_scales) return FLINT_ERR_INVALID_ARG;
    if (V <= 0 || V % 16 != 0 || V > (1 << 24)) return FLINT_ERR_INVALID_ARG;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return FLINT_ERR_CUDA;
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return FLINT_ERR_CUDA;
    if (prop.major != 10 || prop.minor != 3) return FLINT_ERR_UNSUPPORTED;

    flint_lm_head* h = new (std::nothrow) flint_lm_head();
    if (!h) return FLINT_ERR_OOM;
    h->device = dev;
    h->num_sms = prop.multiProcessorCount;
    h->smem_optin = (int)prop.sharedMemPerBlockOptin;
    h->V = V;
    h->units = V / 16;
    h->ts = W->tensor_scale;
    h->limit_ns = 1000000000ull;   // one second
    flint_status_t st = FLINT_OK;
    if (cudaHostAlloc(reinterpret_cast<void**>(&h->status_host), 64, cudaHostAllocMapped) != cudaSuccess) {
        st = FLINT_ERR_OOM;
    } else {
        *h->status_host = 0;
        if (cudaHostGetDevicePointer(reinterpret_cast<void**>(&h->status_dev), h->status_host, 0) != cudaSuccess)
            st = FLINT_ERR_CUDA;
    }
    if (st == FLINT_OK && cudaMalloc(&h->nv, (size_t)h->units * LH_UNIT) != cudaSuccess) st = FLINT_ERR_OOM;
    if (st == FLINT_OK && launch_repack_nvfp4(W->packed, W->block_scales, 2, V, h->nv, 0) != cudaSuccess)
        st = FLINT_ERR_CUDA;
    if (st == FLINT_OK) {
        const cudaError_t e = cudaSuccess == lh_set_attr<1>(h->smem_optin) &&
                                      cudaSuccess == lh_set_attr<2>(h->smem_optin) &&
                                      cudaSuccess == lh_set_attr<3>(h->smem_optin) &&
                                      cudaSuccess == lh_set_attr<4>(h->smem_optin)
                                  ? cudaDeviceSynchronize()
                                  : cudaErrorInvalidValue;
        if (e != cudaSuccess) st = FLINT_ERR_CUDA;
    }
    if (st != FLINT_OK) {
        cudaGetLastError();
        lh_free(h);
        return st;
    }
    *out = h;
    return FLINT_OK;
}

flint_status_t flint_lm_head_forward(flint_lm_head_t h, const void* x, int T, float* logits, cudaStream_t s) {
    using namespace flint;
    if (!h || !x || !logits || T < 1 || T > FLINT_LM_HEAD_MAX_T) return FLINT_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(logits) & 15u))
        return FLINT_ERR_INVALID_ARG;
    const char* xb = static_cast<const char*>(x);
    const char* lb = reinterpret_cast<const char*>(logits);
    if (xb < lb + (size_t)T * h->V * 4 && lb < xb + (size_t)T * H * 2) return FLINT_ERR_INVALID_ARG;
    const flint_status_t st = lh_take_status(h);
    if (st != FLINT_OK) return st;
    LmParams p{h->nv, h->ts, static_cast<const __nv_bfloat16*>(x), logits, T, h->V, h->units, 0, h->status_dev,
               h->limit_ns};
    const int grid = h->units < h->num_sms ? h->units : h->num_sms;
    cudaError_t e;
    switch ((T + 7) / 8) {
        case 1: e = lh_launch<1>(p, grid, h->smem_optin, s); break;
        case 2: e = lh_launch<2>(p, grid, h->smem_optin, s); break;
        case 3: e = lh_launch<3>(p, grid, h->smem_optin, s); break;
        default: e = lh_launch<4>(p, grid, h->smem_optin, s); break;
    }
    return e == cudaSuccess ? FLINT_OK : FLINT_ERR_CUDA;
}

flint_status_t flint_lm_head_destroy(flint_lm_head_t h) {
    if (!h) return FLINT_OK;
    const cudaError_t e = cudaDeviceSynchronize();
    flint_status_t st = lh_take_status(h);
    lh_free(h);
    if (st == FLINT_OK && e != cudaSuccess) st = FLINT_ERR_CUDA;
    return st;
}

}  // extern "C"
