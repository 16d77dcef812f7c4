// decode_nvfp4.cu -- the weight-streaming decode kernels (T <= 32) for
// NVFP4 expert weights run as W4A16 (RecursiveSI/flint vLLM recipe page,
// "Overview": the NVFP4 checkpoint is repacked at load and run as W4A16).
//
// A weight is e2m1(q) * e4m3(s_block) * s_tensor with one E4M3 scale per 16
// consecutive columns of a row and one fp32 scale per matrix.  Sixteen
// columns are exactly one k-step of the legacy tensor-core MMA m16n8k16, so
// the kernels dequantise in registers straight into MMA A fragments: each
// lane converts its four bytes of codes (cvt.rn.f16x2.e2m1x2, exact) and
// multiplies them by the block scale of its two rows in f16 (exact: an E2M1
// value times an E4M3 value has at most 6 significant bits and lies in
// [2^-10, 2688]).  The MMAs accumulate in fp32; the tensor scale and the
// activation scale are applied once per output.  At decode sizes the tensor
// core is otherwise idle; it replaces about 40 CUDA-core instructions per
// weight block and token.
//
//   gateup_nvfp4  Unit = 8 gate rows + the 8 matching up rows of one expert
//                 (the MMA's 16 rows), K = 2048 in 4 chunks of 4608 bytes;
//                 a quad of warps takes a unit, each warp streaming one
//                 chunk by cp.async.bulk into its ring, and the four partial
//                 sums are added in warp order.  The tokens are the N
//                 columns (tiles of 8).  x is staged in
//                 shared memory as f16 times a power of two per token
//                 (chosen so the token's largest |x| lies in [2^14, 2^15):
//                 exact for every bf16 value not 28 binades below it); the
//                 factor is divided out of the result.  Each lane ends with
//                 gate and up of the same (row, token), so a = silu(g) * u is
//                 formed in registers and written as bf16.
//   down_nvfp4    CTA c owns output rows 16c..16c+15 (one MMA M tile).  Warp
//                 w takes expert slots w, w + 8, ... (one 4608-byte chunk
//                 each); the activations arrive as bf16 (written so by the
//                 gate/up kernel; bf16 has fp32's range) for a bf16 MMA,
//                 staged in smem when the batch is small; w * s_tensor * D is
//                 accumulated per (token, row) in the warp's own buffer and
//                 the eight buffers are summed in warp order: deterministic.
//
// Routing, tables and the shared-expert prefetch are those of the bf16
// decode kernels (decode_mma.cu).
#include <cuda_fp16.h>

#include "flint_common.cuh"
#include "../../include/flint_moe.h"
#include "flint_internal.h"
#include "mma_sync.cuh"
#include "routing.cuh"

namespace flint {

// ---------------------------------------------------------------------------
// create-time repack into the owned layout
// ---------------------------------------------------------------------------

// kind 0: gate_up [2I][H] -> 64 units x 4 chunks; kind 1: down [H][I] -> 128 units.
// In a chunk, K block kb, lane t = 4g + c holds at 4t the code bytes of
// (row g, cols 2c..2c+1), (row g+8, same), (row g, cols 8+2c..9+2c),
// (row g+8, same) -- the m16n8k16 A fragment, low nibble = lower column;
// the scales of (row g, row g+8) sit at NV_CODES + 16 kb + 2g.
__global__ void repack_nvfp4_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scales,
                                    int kind, uint8_t* __restrict__ out) {
    const int K = kind == 0 ? H : I;
    const int nchunks = kind == 0 ? NV_GU_UNITS * NV_GU_CHUNKS : NV_DN_UNITS;
    const int total = nchunks * NV_CHUNK_KB * 32;
    const size_t prow = K / 2, srow = K / 16;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
        const int lane = i & 31, kb = (i >> 5) & (NV_CHUNK_KB - 1), ch = i >> 10;
        const int unit = kind == 0 ? ch / NV_GU_CHUNKS : ch;
        const int kbg = (kind == 0 ? ch % NV_GU_CHUNKS : 0) * NV_CHUNK_KB + kb;
        auto row_of = [&](int arow) {
            return kind == 0 ? (arow < 8 ? 8 * unit + arow : I + 8 * unit + (arow - 8)) : 16 * unit + arow;
        };
        const int g = lane >> 2, c = lane & 3;
        const size_t rg = row_of(g), rg8 = row_of(g + 8);
        uint8_t* dst = out + (size_t)ch * NV_CHUNK;
        uchar4 v;
        v.x = packed[rg * prow + kbg * 8 + c];
        v.y = packed[rg8 * prow + kbg * 8 + c];
        v.z = packed[rg * prow + kbg * 8 + 4 + c];
        v.w = packed[rg8 * prow + kbg * 8 + 4 + c];
        *reinterpret_cast<uchar4*>(dst + kb * 128 + 4 * lane) = v;
        if (lane < 8) {
            dst[NV_CODES + kb * 16 + 2 * lane] = scales[(size_t)row_of(lane) * srow + kbg];
            dst[NV_CODES + kb * 16 + 2 * lane + 1] = scales[(size_t)row_of(lane + 8) * srow + kbg];
        }
    }
}

cudaError_t launch_repack_nvfp4(const uint8_t* packed, const uint8_t* scales, int kind, uint8_t* out,
                                cudaStream_t s) {
    const int nchunks = kind == 0 ? NV_GU_UNITS * NV_GU_CHUNKS : NV_DN_UNITS;
    const int total = nchunks * NV_CHUNK_KB * 32;
    repack_nvfp4_kernel<<<(total + 255) / 256, 256, 0, s>>>(packed, scales, kind, out);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// fragments and MMAs
// ---------------------------------------------------------------------------

// A fragment (f16) of one 16 x 16 block: codes = this lane's 4 code bytes,
// sc2 = E4M3 scales of its rows (g, g + 8).
__device__ __forceinline__ void nv_a_frag(uint32_t codes, uint16_t sc2, uint32_t (&a)[4]) {
    uint32_t s;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(s) : "h"(sc2));
    const __half2 s2 = *reinterpret_cast<const __half2*>(&s);
    const __half2 sg = __low2half2(s2), s8 = __high2half2(s2);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        uint32_t h;
        asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}\n" : "=r"(h) : "r"(codes >> (8 * k)));
        const __half2 q = *reinterpret_cast<const __half2*>(&h);
        const __half2 r = __hmul2(q, (k & 1) ? s8 : sg);
        a[k] = *reinterpret_cast<const uint32_t*>(&r);
    }
}

__device__ __forceinline__ uint32_t f16x2_to_bf16x2(uint32_t v) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&v));
    const __nv_bfloat162 b = __float22bfloat162_rn(f);   // exact: at most 6 significant bits
    return *reinterpret_cast<const uint32_t*>(&b);
}

// ---------------------------------------------------------------------------
// gate/up + SwiGLU
// ---------------------------------------------------------------------------

constexpr int GN_WARPS = 8;
constexpr int GN_XROW = H + 8;   // f16 per staged token row (+8: conflict-free B loads)

struct GateUpNvParams {
    const uint8_t* nv;            // owned experts, NV_EXPERT_BYTES each
    const float* ts;              // [NEXP][2] tensor scales (gate_up, down)
    const float* logits;          // [T][E]
    const __nv_bfloat16* x;       // [T][H]
    int T;
    int ns;                       // ring chunks per warp
    DecodeTables* tables_out;
    int32_t* idx_out;
    float* w_out;
    __nv_bfloat16* a;             // [pairs][I] bf16 (the down kernel's MMA operand)
    uint32_t* status;
    uint64_t limit_ns;
};

constexpr int GN_QUADS = GN_WARPS / 4;                 // a quad of warps works on one unit
constexpr int GN_PART = GN_QUADS * 4 * 4 * 32 * 4;      // partial sums [quad][warp][N tile][lane][4]

// ring chunks per warp (one chunk = the warp's quarter of a unit): deep while
// x is small; one when x fills the shared memory (the next chunk then goes to L2)
static inline int gn_ns(int T) { return T <= 8 ? 4 : (T <= 24 ? 2 : 1); }

static inline size_t gn_smem_bytes(int T) {
    return (size_t)GN_WARPS * gn_ns(T) * NV_CHUNK + (size_t)T * GN_XROW * 2 + DEC_T * 4 + (size_t)GN_PART * 4 +
           (size_t)GN_WARPS * gn_ns(T) * 8 + sizeof(DecodeTables) + DEC_T * TOPK * 8 + 2 * E * 4;
}

// barrier (and AND of a predicate) of the 128 threads of quad q
__device__ __forceinline__ bool quad_all(int q, bool v) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, t;\n setp.ne.u32 p, %1, 0;\n barrier.cta.red.and.pred t, %2, 128, p;\n"
        " selp.u32 %0, 1, 0, t;\n}\n"
        : "=r"(r)
        : "r"(v ? 1u : 0u), "r"(1 + q)
        : "memory");
    return r != 0;
}
__device__ __forceinline__ void quad_sync(int q) { asm volatile("bar.sync %0, 128;" ::"r"(1 + q) : "memory"); }

// Quad q of CTA c takes units c + G q, c + G (q + 2), ...; warp k of the quad
// streams and multiplies chunk k (columns 512k .. 512k + 511) of each, and the
// four partial sums are added in warp order.  A unit then costs each warp a
// quarter of the dequantise -> MMA chain it used to cost one warp.
__global__ void __launch_bounds__(GN_WARPS * 32, 1) gateup_nvfp4_kernel(GateUpNvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp >> 2, wq = warp & 3;
    const int NS = p.ns, T = p.T, G = gridDim.x, c = blockIdx.x;
    uint8_t* ring = smem + (size_t)warp * NS * NV_CHUNK;
    __half* xh = reinterpret_cast<__half*>(smem + (size_t)GN_WARPS * NS * NV_CHUNK);
    float* xinv = reinterpret_cast<float*>(xh + (size_t)T * GN_XROW);
    float* part = xinv + DEC_T;
    uint64_t* bars = reinterpret_cast<uint64_t*>(part + GN_PART);
    uint64_t* bar = bars + warp * NS;
    DecodeTables* tab = reinterpret_cast<DecodeTables*>(bars + GN_WARPS * NS);
    int* sel_e = reinterpret_cast<int*>(tab + 1);
    float* sel_w = reinterpret_cast<float*>(sel_e + DEC_T * TOPK);
    uint32_t* tmask = reinterpret_cast<uint32_t*>(sel_w + DEC_T * TOPK);
    int* pair0 = reinterpret_cast<int*>(tmask + E);

    if (lane == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // the quad's i-th unit; this warp's chunk of it is chunk wq
    auto unit_of = [&](int i) { return c + G * (quad + GN_QUADS * i); };
    auto chunk_ptr = [&](int i, int expert) {
        const int r = unit_of(i) & (NV_GU_UNITS - 1);
        return p.nv + (size_t)expert * NV_EXPERT_BYTES + ((size_t)r * NV_GU_CHUNKS + wq) * NV_CHUNK;
    };
    auto issue = [&](int i, int expert) {
        const int s = i % NS;
        mbar_arrive_expect_tx(&bar[s], NV_CHUNK);
        bulk_g2s(ring + (size_t)s * NV_CHUNK, chunk_ptr(i, expert), NV_CHUNK, &bar[s]);
    };

    // ---- before the router has finished: the shared expert's chunks ----
    int issued = 0;
    if (lane == 0) {
        for (int i = 0; i < NS && unit_of(i) < NV_GU_UNITS; ++i) {
            issue(i, SHARED);
            issued = i + 1;
        }
    }
    pdl_wait();     // router logits are complete (and x is ready)
    pdl_trigger();

    // ---- x -> f16 times 2^e_t per token ----
    for (int t = warp; t < T; t += GN_WARPS) {
        uint4 v[8];
        float mx = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            v[k] = ldg16(p.x + (size_t)t * H + 8 * (lane + 32 * k));
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
            *reinterpret_cast<uint4*>(xh + (size_t)t * GN_XROW + 8 * (lane + 32 * k)) = o;
        }
    }

    // ---- top-6 of every token, then the (slot, token) tables ----
    for (int t = warp; t < T; t += GN_WARPS) {
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
    if (warp == 0) build_decode_tables_warp(T, sel_e, sel_w, tmask, pair0, tab, lane);
    __syncthreads();
    if (c == 0) {
        const int* src = reinterpret_cast<const int*>(tab);
        int* dst = reinterpret_cast<int*>(p.tables_out);
        for (int k = threadIdx.x; k < (int)(sizeof(DecodeTables) / 4); k += blockDim.x) dst[k] = src[k];
    }
    const int total_units = tab->n_slots * NV_GU_UNITS;
    int my_units = 0;
    while (unit_of(my_units) < total_units) ++my_units;
    auto expert_of = [&](int i) { return tab->slot_expert[unit_of(i) / NV_GU_UNITS]; };
    if (lane == 0) {
        for (int i = issued; i < NS && i < my_units; ++i) {
            issue(i, expert_of(i));
            issued = i + 1;
        }
        if (NS == 1 && my_units > 1) bulk_prefetch_l2(chunk_ptr(1, expert_of(1)), NV_CHUNK);
    }

    const int g = lane >> 2, cq = lane & 3;
    float* qpart = part + quad * (4 * 4 * 32 * 4);
    bool ok = true;
    int i = 0;
    for (; i < my_units; ++i) {
        const int q = unit_of(i), u = q / NV_GU_UNITS, r = q & (NV_GU_UNITS - 1);
        const int pb = tab->slot_pair0[u], np = tab->slot_pair0[u + 1] - pb;   // 1..32 tokens
        const int ntile = (np + 7) >> 3;
        int xo[4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int n = nt * 8 + g;
            xo[nt] = tab->pair_token[pb + (n < np ? n : np - 1)] * GN_XROW + 2 * cq + wq * 512;
        }
        const int s = i % NS;
        const bool got = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&bar[s], (i / NS) & 1, p.limit_ns));
        if (got) {
            // four accumulators per N tile (K block kb goes to chain kb % 4)
            float acc[4][4][4];
#pragma unroll
            for (int ch = 0; ch < 4; ++ch)
#pragma unroll
                for (int nt = 0; nt < 4; ++nt)
#pragma unroll
                    for (int k = 0; k < 4; ++k) acc[ch][nt][k] = 0.f;
            const uint8_t* buf = ring + (size_t)s * NV_CHUNK;
#pragma unroll 2
            for (int kb = 0; kb < NV_CHUNK_KB; kb += 4) {
                uint32_t a[4][4];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    nv_a_frag(*reinterpret_cast<const uint32_t*>(buf + (kb + ch) * 128 + 4 * lane),
                              *reinterpret_cast<const uint16_t*>(buf + NV_CODES + (kb + ch) * 16 + 2 * g), a[ch]);
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    if (nt < ntile) {
                        const __half* xb = xh + xo[nt] + kb * 16;
#pragma unroll
                        for (int ch = 0; ch < 4; ++ch)
                            mma_f16_16816(acc[ch][nt], a[ch], *reinterpret_cast<const uint32_t*>(xb + 16 * ch),
                                          *reinterpret_cast<const uint32_t*>(xb + 16 * ch + 8));
                    }
                }
            }
            __syncwarp();   // every lane is done reading slot s
            if (lane == 0) {
                if (i + NS < my_units) {
                    fence_proxy_async_smem();
                    issue(i + NS, expert_of(i + NS));
                    issued = i + NS + 1;
                }
                if (NS == 1 && i + 2 < my_units) bulk_prefetch_l2(chunk_ptr(i + 2, expert_of(i + 2)), NV_CHUNK);
            }
#pragma unroll
            for (int nt = 0; nt < 4; ++nt)
                if (nt < ntile)
                    *reinterpret_cast<float4*>(qpart + ((wq * 4 + nt) * 32 + lane) * 4) = make_float4(
                        acc[0][nt][0] + acc[1][nt][0] + (acc[2][nt][0] + acc[3][nt][0]),
                        acc[0][nt][1] + acc[1][nt][1] + (acc[2][nt][1] + acc[3][nt][1]),
                        acc[0][nt][2] + acc[1][nt][2] + (acc[2][nt][2] + acc[3][nt][2]),
                        acc[0][nt][3] + acc[1][nt][3] + (acc[2][nt][3] + acc[3][nt][3]));
        }
        // the decision to go on is taken by the whole quad
        if (!quad_all(quad, got)) {
            ok = false;
            break;
        }
        // warp nt of the quad adds tile nt's four partial sums in warp order;
        // lane (g, cq) then holds gate (0, 1) and up (2, 3) of row j = 8r + g
        if (wq < ntile) {
            float4 sum = *reinterpret_cast<const float4*>(qpart + (wq * 32 + lane) * 4);
#pragma unroll
            for (int w = 1; w < 4; ++w) {
                const float4 v = *reinterpret_cast<const float4*>(qpart + ((w * 4 + wq) * 32 + lane) * 4);
                sum.x += v.x;
                sum.y += v.y;
                sum.z += v.z;
                sum.w += v.w;
            }
            const float tsg = __ldg(p.ts + 2 * tab->slot_expert[u]);
            const int j = 8 * r + g, n0 = wq * 8 + 2 * cq;
            if (n0 < np) {
                const float f = tsg * xinv[tab->pair_token[pb + n0]];
                p.a[(size_t)(pb + n0) * I + j] = __float2bfloat16_rn(silu_f(sum.x * f) * (sum.z * f));
            }
            if (n0 + 1 < np) {
                const float f = tsg * xinv[tab->pair_token[pb + n0 + 1]];
                p.a[(size_t)(pb + n0 + 1) * I + j] = __float2bfloat16_rn(silu_f(sum.y * f) * (sum.w * f));
            }
        }
        quad_sync(quad);   // the partial sums are read before the next unit writes them
    }
    if (!ok) {
        if (lane == 0) {
            report_status(p.status, ST_TIMEOUT);
            // drain copies still in flight into this warp's ring (bounded)
            for (int k = i; k < issued; ++k) mbar_wait_bounded(&bar[k % NS], (k / NS) & 1, p.limit_ns);
        }
        __syncwarp();
    }
}

// ---------------------------------------------------------------------------
// down projection + weighted combine
// ---------------------------------------------------------------------------

constexpr int DV_WARPS = 8;
constexpr int DV_CTAS = H / 16;        // 128: CTA c owns rows 16c .. 16c + 15
constexpr int DV_APAIRS = 64;          // activation rows staged in smem when the batch has at most this many
constexpr int DV_AROW = I * 2 + 16;    // bytes per staged row (+16: conflict-free B loads)

struct DownNvParams {
    const uint8_t* nv;
    const float* ts;
    const float* logits;          // [T][E] router logits (final before this kernel starts)
    const __nv_bfloat16* a;       // [pairs][I] bf16
    __nv_bfloat16* y;             // [T][H]
    int ns;                       // ring chunks per warp
    int T;
    uint32_t* status;
    uint64_t limit_ns;
};

// small batches keep the kernel small, so the next layer's gate/up CTAs fit beside it
static inline int dv_ns(int T) { return T <= 2 ? 1 : (T <= 8 ? 2 : 4); }
__host__ __device__ inline bool dv_staged(int T) { return (TOPK + 1) * T <= DV_APAIRS; }

static inline size_t dv_smem_bytes(int T) {
    return (size_t)DV_WARPS * dv_ns(T) * NV_CHUNK + (dv_staged(T) ? (size_t)(TOPK + 1) * T * DV_AROW : 0) +
           (size_t)DV_WARPS * T * 16 * 4 + (DV_WARPS * dv_ns(T) + 1) * 8 + sizeof(DecodeTables) +
           DEC_T * TOPK * 8 + 2 * E * 4;
}

__global__ void __launch_bounds__(DV_WARPS * 32, 1) down_nvfp4_kernel(DownNvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, NS = p.ns, Tk = p.T;
    const bool staged = dv_staged(Tk);
    uint8_t* ring = smem + (size_t)warp * NS * NV_CHUNK;
    uint8_t* astage = smem + (size_t)DV_WARPS * NS * NV_CHUNK;                           // [7T][DV_AROW]
    float* yw_all = reinterpret_cast<float*>(astage + (staged ? (size_t)(TOPK + 1) * Tk * DV_AROW : 0));
    float* yw = yw_all + warp * Tk * 16;                                                  // [8][T][16]
    uint64_t* bars = reinterpret_cast<uint64_t*>(yw_all + DV_WARPS * Tk * 16);
    uint64_t* bar = bars + warp * NS;
    uint64_t* abar = bars + DV_WARPS * NS;
    DecodeTables* tab = reinterpret_cast<DecodeTables*>(abar + 1);
    int* sel_e = reinterpret_cast<int*>(tab + 1);
    float* sel_w = reinterpret_cast<float*>(sel_e + DEC_T * TOPK);
    uint32_t* tmask = reinterpret_cast<uint32_t*>(sel_w + DEC_T * TOPK);
    int* pair0 = reinterpret_cast<int*>(tmask + E);

    if (lane == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&bar[s], 1);
        if (warp == 0) mbar_init(abar, 1);
        fence_mbar_init();
    }
    auto issue = [&](int i, int expert) {
        const int s = i % NS;
        const uint8_t* src = p.nv + (size_t)expert * NV_EXPERT_BYTES + NV_GU_BYTES + (size_t)c * NV_CHUNK;
        mbar_arrive_expect_tx(&bar[s], NV_CHUNK);
        bulk_g2s(ring + (size_t)s * NV_CHUNK, src, NV_CHUNK, &bar[s]);
    };
    // Every gate/up CTA triggers this launch only after its own dependency
    // wait, which returns once the router grid has completed: the logits are
    // final here although the gate/up kernel may still be running.  Select
    // each token's experts and build the same tables the gate/up kernel
    // builds, and start the weight chunks of this warp's first slots now, so
    // they stream while the gate/up kernel runs.
    for (int t = warp; t < Tk; t += DV_WARPS) {
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
    for (int k = threadIdx.x; k < DV_WARPS * Tk * 16; k += blockDim.x) yw_all[k] = 0.f;
    __syncthreads();
    if (warp == 0) build_decode_tables_warp(Tk, sel_e, sel_w, tmask, pair0, tab, lane);
    __syncthreads();
    const int n_slots = tab->n_slots, n_pairs = tab->n_pairs;
    const int my_slots = n_slots > warp ? (n_slots - warp + DV_WARPS - 1) / DV_WARPS : 0;
    int issued = 0;
    if (lane == 0) {
        for (int i = 0; i < NS && i < my_slots; ++i) {
            issue(i, tab->slot_expert[warp + DV_WARPS * i]);
            issued = i + 1;
        }
    }
    pdl_wait();     // the gate/up kernel is complete: activations are visible
    pdl_trigger();
    if (staged && threadIdx.x == 0) {
        // every activation row, one bulk copy per row (padded rows in smem)
        mbar_arrive_expect_tx(abar, n_pairs * I * 2);
        for (int pr = 0; pr < n_pairs; ++pr) bulk_g2s(astage + (size_t)pr * DV_AROW, p.a + (size_t)pr * I, I * 2, abar);
    }
    bool ok = true;
    if (staged && my_slots > 0) ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(abar, 0, p.limit_ns));

    const int g = lane >> 2, cq = lane & 3;
    int i = 0;
    for (; ok && i < my_slots; ++i) {
        const int u = warp + DV_WARPS * i, s = i % NS;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&bar[s], (i / NS) & 1, p.limit_ns))) {
            ok = false;
            break;
        }
        const uint8_t* buf = ring + (size_t)s * NV_CHUNK;
        const int pb = tab->slot_pair0[u], np = tab->slot_pair0[u + 1] - pb;
        const int ntile = (np + 7) >> 3;
        int prow[4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
            const int n = nt * 8 + g;
            prow[nt] = pb + (n < np ? n : np - 1);
        }
        float acc[4][4];
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) acc[nt][0] = acc[nt][1] = acc[nt][2] = acc[nt][3] = 0.f;
        if (staged) {
#pragma unroll 4
            for (int kb = 0; kb < NV_CHUNK_KB; ++kb) {
                uint32_t a[4];
                nv_a_frag(*reinterpret_cast<const uint32_t*>(buf + kb * 128 + 4 * lane),
                          *reinterpret_cast<const uint16_t*>(buf + NV_CODES + kb * 16 + 2 * g), a);
#pragma unroll
                for (int k = 0; k < 4; ++k) a[k] = f16x2_to_bf16x2(a[k]);
#pragma unroll
                for (int nt = 0; nt < 4; ++nt) {
                    if (nt < ntile) {
                        const uint8_t* ar = astage + (size_t)prow[nt] * DV_AROW + (kb * 16 + 2 * cq) * 2;
                        mma_bf16_16816(acc[nt], a, *reinterpret_cast<const uint32_t*>(ar),
                                       *reinterpret_cast<const uint32_t*>(ar + 16));
                    }
                }
            }
        } else {
            // activations through L1 (read-only here; written by the previous
            // grid): the first N tile's operands for 16 blocks are requested
            // at once, the other tiles' as they are used
#pragma unroll 1
            for (int kh = 0; kh < NV_CHUNK_KB; kh += 16) {
                uint32_t bq[16][2];
                const unsigned int* a0 =
                    reinterpret_cast<const unsigned int*>(p.a + (size_t)prow[0] * I + kh * 16 + 2 * cq);
#pragma unroll
                for (int kb = 0; kb < 16; ++kb) {
                    bq[kb][0] = __ldg(a0 + kb * 8);
                    bq[kb][1] = __ldg(a0 + kb * 8 + 4);
                }
#pragma unroll
                for (int kb = 0; kb < 16; ++kb) {
                    uint32_t a[4];
                    nv_a_frag(*reinterpret_cast<const uint32_t*>(buf + (kh + kb) * 128 + 4 * lane),
                              *reinterpret_cast<const uint16_t*>(buf + NV_CODES + (kh + kb) * 16 + 2 * g), a);
#pragma unroll
                    for (int k = 0; k < 4; ++k) a[k] = f16x2_to_bf16x2(a[k]);
                    mma_bf16_16816(acc[0], a, bq[kb][0], bq[kb][1]);
#pragma unroll
                    for (int nt = 1; nt < 4; ++nt) {
                        if (nt < ntile) {
                            const unsigned int* ar = reinterpret_cast<const unsigned int*>(
                                p.a + (size_t)prow[nt] * I + (kh + kb) * 16 + 2 * cq);
                            mma_bf16_16816(acc[nt], a, __ldg(ar), __ldg(ar + 4));
                        }
                    }
                }
            }
        }
        __syncwarp();
        if (lane == 0 && i + NS < my_slots) {
            fence_proxy_async_smem();
            issue(i + NS, tab->slot_expert[warp + DV_WARPS * (i + NS)]);
            issued = i + NS + 1;
        }
        // lane (g, cq): rows g and g + 8 of this CTA's 16, tile columns 2cq, 2cq + 1
        const float tsd = __ldg(p.ts + 2 * tab->slot_expert[u] + 1);
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                const int n = nt * 8 + 2 * cq + hh;
                if (nt < ntile && n < np) {
                    const int pr = pb + n, t = tab->pair_token[pr];
                    const float wgt = tab->pair_weight[pr] * tsd;
                    yw[t * 16 + g] = fmaf(wgt, acc[nt][hh], yw[t * 16 + g]);
                    yw[t * 16 + g + 8] = fmaf(wgt, acc[nt][2 + hh], yw[t * 16 + g + 8]);
                }
            }
        }
    }
    if (!ok && lane == 0) {
        report_status(p.status, ST_TIMEOUT);
        for (int k = i; k < issued; ++k) mbar_wait_bounded(&bar[k % NS], (k / NS) & 1, p.limit_ns);
        if (staged && warp == 0) mbar_wait_bounded(abar, 0, p.limit_ns);
    }
    __syncthreads();
    // y rows 16c .. 16c + 15: the eight warps' partial sums in warp order
    for (int k = threadIdx.x; k < Tk * 16; k += blockDim.x) {
        const int t = k >> 4, rr = k & 15;
        float sum = 0.f;
#pragma unroll
        for (int w = 0; w < DV_WARPS; ++w) sum += yw_all[w * Tk * 16 + t * 16 + rr];
        p.y[(size_t)t * H + 16 * c + rr] = __float2bfloat16_rn(sum);
    }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

cudaError_t decode_nvfp4_set_attributes() {
    cudaError_t e = cudaFuncSetAttribute(gateup_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)(gn_smem_bytes(DEC_T) > gn_smem_bytes(8) ? gn_smem_bytes(DEC_T)
                                                                                       : gn_smem_bytes(8)));
    if (e != cudaSuccess) return e;
    size_t dmax = 0;
    for (int T = 1; T <= DEC_T; ++T) dmax = dv_smem_bytes(T) > dmax ? dv_smem_bytes(T) : dmax;
    return cudaFuncSetAttribute(down_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dmax);
}

cudaError_t launch_decode_experts_nvfp4(const LaunchCtx& L, const uint8_t* nv, const float* nv_ts,
                                        const float* logits, const __nv_bfloat16* x, int T, DecodeTables* tables,
                                        int32_t* idx, float* w, float* a_buf, __nv_bfloat16* y) {
    // the activations are kept as bf16 in the (fp32-sized) activation buffer
    __nv_bfloat16* a16 = reinterpret_cast<__nv_bfloat16*>(a_buf);
    GateUpNvParams gp{nv, nv_ts, logits, x, T, gn_ns(T), tables, idx, w, a16, L.status, L.wait_limit_ns};
    cudaError_t e = launch_hooked(L, FLINT_KERNEL_GATE_UP, gateup_nvfp4_kernel, dim3(L.num_sms),
                                  dim3(GN_WARPS * 32), gn_smem_bytes(T), gp);
    if (e != cudaSuccess) return e;
    DownNvParams dp{nv, nv_ts, logits, a16, y, dv_ns(T), T, L.status, L.wait_limit_ns};
    return launch_hooked(L, FLINT_KERNEL_DOWN, down_nvfp4_kernel, dim3(DV_CTAS), dim3(DV_WARPS * 32),
                         dv_smem_bytes(T), dp);
}

}  // namespace flint
