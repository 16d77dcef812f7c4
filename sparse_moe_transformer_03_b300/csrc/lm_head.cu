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
//     consumer warp w takes units w, w + NW, ... of it and streams their
//     chunks itself: its lane 0 keeps D chunks in flight in the warp's own D
//     ring slots (one 2-D TMA box of 9 x 512 bytes per chunk) and issues
//     chunk k + D into the slot of chunk k once the warp has read it.  No
//     warp waits on another: an earlier design with one producer thread
//     feeding every warp in a fixed order streamed at 2.8 TB/s with the
//     arithmetic removed, each slot waiting on the slowest warp;
//   * NW consumer warps (16; 8 when T > 16, where x takes more shared
//     memory): warp w multiplies whole units (16 rows x K 2048) by
//     the tokens, dequantising each 16 x 16 block straight into an f16 A
//     fragment (nvfp4_frag.cuh) and multiplying it with x staged in shared
//     memory as f16 (token t scaled by 2^e_t so that its largest |x| lies in
//     [2^14, 2^15): exact for every bf16 value within 28 binades of it); the
//     fp32 accumulators get s_tensor * 2^-e_t at the end and the warp writes
//     its 16 logits per token.
// Every wait is bounded by %globaltimer; a wait that gives up sets the CTA's
// abort flag, reports FLINT_ERR_DEVICE_TIMEOUT through the status word and
// each warp lets its copies in flight land before the CTA exits.
#include <cuda_fp16.h>

#include <new>

#include "../../include/flint_moe.h"
#include "flint_common.cuh"
#include "flint_internal.h"
#include "mma_sync.cuh"
#include "nvfp4_frag.cuh"
#include "tc_ptx.cuh"

namespace flint {
namespace {

template <int NT>
struct LhCfg {
    // consumer warps, each with two ring slots beside x (T <= 16: 16 warps,
    // 32 slots; T <= 32: 8 warps, 16 slots).  Measured at T = 1: 16 x 2 slots
    // 37.5 us, 20 x 2 37.4, 14 x 3 42.0, 8 x 5 41.6
    static constexpr int NW = NT <= 2 ? 16 : 8;
    static constexpr int THREADS = 32 * NW;
};
constexpr int LH_XSTRIDE = 2 * H + 16;             // bytes per staged token row (bank spread)
constexpr int LH_UNIT = NV_GU_CHUNKS * NV_CHUNK;   // 18432 bytes: 16 rows x 2048
constexpr int LH_MAX_SLOTS = 64;
constexpr int LH_BOX_ROWS = NV_CHUNK / 512;        // a chunk as 9 rows of 512 bytes (one TMA box)

struct LmParams {
    float ts;                   // tensor scale
    const __nv_bfloat16* x;     // [T][H]
    float* logits;              // [T][V]
    int T, V, units, nslot;
    uint32_t* status;
    uint64_t limit_ns;
};

// dynamic shared memory: ring | x (8 NT rows) | xinv[32] | uses[nslot] | full[nslot] | abort
__host__ __device__ constexpr uint32_t lh_x_off(int nslot) { return (uint32_t)nslot * NV_CHUNK; }
__host__ __device__ constexpr uint32_t lh_xinv_off(int nslot, int nt) {
    return lh_x_off(nslot) + (uint32_t)(8 * nt) * LH_XSTRIDE;
}
__host__ __device__ constexpr uint32_t lh_uses_off(int nslot, int nt) { return lh_xinv_off(nslot, nt) + 32 * 4; }
__host__ __device__ constexpr uint32_t lh_bar_off(int nslot, int nt) {
    return (lh_uses_off(nslot, nt) + (uint32_t)nslot * 4 + 7) & ~7u;
}
__host__ __device__ constexpr uint32_t lh_smem_bytes(int nslot, int nt) {
    return lh_bar_off(nslot, nt) + (uint32_t)nslot * 8 + 16;
}

struct LmState {
    uint8_t* ring;
    uint32_t* uses;         // per slot: how many copies were issued into it
    uint64_t* full;
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

template <int NT>   // token tiles of 8: T <= 8 NT
__global__ void __launch_bounds__(LhCfg<NT>::THREADS, 1)
    lm_head_nvfp4_kernel(const __grid_constant__ CUtensorMap map, LmParams p) {
    constexpr int NW = LhCfg<NT>::NW;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    LmState s;
    s.nslot = p.nslot;
    s.limit = p.limit_ns;
    s.ring = smem;
    uint8_t* xs = smem + lh_x_off(p.nslot);
    float* xinv = reinterpret_cast<float*>(smem + lh_xinv_off(p.nslot, NT));
    s.uses = reinterpret_cast<uint32_t*>(smem + lh_uses_off(p.nslot, NT));
    s.full = reinterpret_cast<uint64_t*>(smem + lh_bar_off(p.nslot, NT));
    s.abort = reinterpret_cast<volatile uint32_t*>(s.full + p.nslot);
    // the CTA's units: a balanced contiguous range; warp w takes units
    // w, w + NW, ... of it, i.e. chunks k = 0 .. 4 m - 1 (unit w + (k / 4) NW,
    // chunk k % 4), streamed through its own D slots (chunk k in slot
    // w D + k % D, that slot's use k / D)
    const int G = gridDim.x, c = blockIdx.x;
    const int u0 = (int)((long long)p.units * c / G), u1 = (int)((long long)p.units * (c + 1) / G);
    const int n = u1 - u0;
    const int D = p.nslot / NW;
    const int m = warp < n ? (n - warp + NW - 1) / NW : 0;
    const int nch = NV_GU_CHUNKS * m;
    uint64_t* full = s.full + warp * D;
    uint8_t* ring = s.ring + (size_t)warp * D * NV_CHUNK;
    uint32_t* uses = s.uses + warp * D;

    if (lane == 0) {
        for (int i = 0; i < D; ++i) {
            mbar_init(&full[i], 1);
            uses[i] = 0;
        }
        if (warp == 0) *s.abort = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // lane 0: chunk k into its slot (one 2-D box of 9 x 512 bytes)
    auto issue = [&](int k) {
        const int sl = k % D;
        mbar_arrive_expect_tx(&full[sl], NV_CHUNK);
        uses[sl] = (uint32_t)(k / D) + 1u;
        const int chunk = (u0 + warp + (k / NV_GU_CHUNKS) * NW) * NV_GU_CHUNKS + k % NV_GU_CHUNKS;
        tc::tma_load_2d(ring + (size_t)sl * NV_CHUNK, &map, 0, LH_BOX_ROWS * chunk, &full[sl]);
    };
    if (lane == 0) {
        tc::prefetch_tensormap(&map);
        for (int k = 0; k < D && k < nch; ++k) issue(k);
    }

    // x -> f16 x 2^e_t, token t on warp t % NW (rows past T zero)
    for (int t = warp; t < 8 * NT; t += NW) {
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
    __syncthreads();

    constexpr int ACC = NT >= 4 ? 1 : (NT == 1 ? 4 : 2);   // independent accumulator chains per tile
    const int g = lane >> 2, cq = lane & 3;
    float acc[ACC][NT][4];
    for (int k = 0; k < nch; ++k) {
        const int cc = k % NV_GU_CHUNKS;
        if (cc == 0) {
#pragma unroll
            for (int a = 0; a < ACC; ++a)
#pragma unroll
                for (int j = 0; j < NT; ++j) acc[a][j][0] = acc[a][j][1] = acc[a][j][2] = acc[a][j][3] = 0.f;
        }
        const int sl = k % D;
        if (!__all_sync(0xFFFFFFFFu, lh_wait(s, &full[sl], (uint32_t)(k / D) & 1, p.status))) break;
        const uint8_t* buf = ring + (size_t)sl * NV_CHUNK;
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
        // the slot's reads are done (generic proxy) before the next copy into it (async proxy)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0 && k + D < nch) issue(k + D);
        if (cc != NV_GU_CHUNKS - 1) continue;
        // lane (g, cq): rows v0 and v0 + 8, tokens 8 j + 2 cq and + 1
        const size_t v0 = (size_t)16 * (u0 + warp + (k / NV_GU_CHUNKS) * NW) + g;
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
    // after an abort: this warp's copies in flight land before the CTA exits
    if (lane == 0 && *s.abort)
        for (int i = 0; i < D; ++i)
            if (uses[i]) mbar_wait_bounded(&full[i], (uses[i] - 1) & 1, 10000000ull);
}

// largest ring that fits the opt-in shared memory: a multiple of the
// consumer warps, at most LH_MAX_SLOTS; 0 when not even two slots per warp fit
int lh_nslot(int nt, int nw, int smem_optin) {
    int k = LH_MAX_SLOTS / nw * nw;
    while (k >= 2 * nw && lh_smem_bytes(k, nt) > (uint32_t)smem_optin) k -= nw;
    return k >= 2 * nw ? k : 0;
}

template <int NT>
cudaError_t lh_launch(const CUtensorMap& map, const LmParams& p0, int grid, int smem_optin, cudaStream_t s) {
    LmParams p = p0;
    p.nslot = lh_nslot(NT, LhCfg<NT>::NW, smem_optin);
    if (p.nslot == 0) return cudaErrorInvalidConfiguration;
    lm_head_nvfp4_kernel<NT><<<grid, LhCfg<NT>::THREADS, lh_smem_bytes(p.nslot, NT), s>>>(map, p);
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
    CUtensorMap map;             // nv as [units x 4 x 9] rows of 128 32-bit words
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
    if (st == FLINT_OK &&
        !encode_u32_rows(&h->map, h->nv, (uint64_t)h->units * NV_GU_CHUNKS * LH_BOX_ROWS, 128, LH_BOX_ROWS))
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
    LmParams p{h->ts, static_cast<const __nv_bfloat16*>(x), logits, T, h->V, h->units, 0, h->status_dev,
               h->limit_ns};
    const int grid = h->units < h->num_sms ? h->units : h->num_sms;
    cudaError_t e;
    switch ((T + 7) / 8) {
        case 1: e = lh_launch<1>(h->map, p, grid, h->smem_optin, s); break;
        case 2: e = lh_launch<2>(h->map, p, grid, h->smem_optin, s); break;
        case 3: e = lh_launch<3>(h->map, p, grid, h->smem_optin, s); break;
        default: e = lh_launch<4>(h->map, p, grid, h->smem_optin, s); break;
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
