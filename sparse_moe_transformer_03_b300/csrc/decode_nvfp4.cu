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
//                 item = a unit against one tile of up to 8 of the expert's
//                 tokens (the N columns).  The CTA takes one item at a time:
//                 warp w streams half of chunk w / 2 (16 K blocks: 2 KiB of
//                 codes, 256 bytes of scales) by cp.async.bulk into its ring,
//                 and the eight partial sums are added in warp order.  x is
//                 staged in shared memory as f16 times a power of two per
//                 token (chosen so the token's largest |x| lies in [2^14,
//                 2^15): exact for every bf16 value not 28 binades below it);
//                 the factor is divided out of the result.  The lane that
//                 adds the partial sums holds gate and up of the same (row,
//                 token), so a = silu(g) * u is formed in registers and
//                 written as bf16.
//   down_nvfp4    CTA c owns output rows 16c..16c+15 (one MMA M tile).  Its
//                 items are (slot, column half, tile of 8 tokens), item j to
//                 warp j % 8, each half of the slot's 4608-byte chunk; the
//                 activations arrive as bf16 (written so by the gate/up
//                 kernel; bf16 has fp32's range) for a bf16 MMA, in the same
//                 ring slot as the weights (one 4 KiB bulk copy per item);
//                 w * s_tensor * D is accumulated per (token, row) in the
//                 warp's own buffer and the eight buffers are summed in warp
//                 order: deterministic.
//
// Routing, tables and the shared-expert prefetch are those of the bf16
// decode kernels (decode_mma.cu).
#include <cuda_fp16.h>

#include "flint_common.cuh"
#include "../../include/flint_moe.h"
#include "flint_internal.h"
#include "mma_sync.cuh"
#include "nvfp4_frag.cuh"
#include "routing.cuh"

namespace flint {

// ---------------------------------------------------------------------------
// create-time repack into the owned layout
// ---------------------------------------------------------------------------

// kind 0: gate_up [2I][H] -> 64 units x 4 chunks; kind 1: down [H][I] -> 128
// units of one chunk; kind 2: any [R][H] (the output layer) -> R/16 units of
// 16 straight rows x 4 chunks.
// In a chunk, K block kb, lane t = 4g + c holds at 4t the code bytes of
// (row g, cols 2c..2c+1), (row g+8, same), (row g, cols 8+2c..9+2c),
// (row g+8, same) -- the m16n8k16 A fragment, low nibble = lower column;
// the scales of (row g, row g+8) sit at NV_CODES + 16 kb + 2g.
__global__ void repack_nvfp4_kernel(const uint8_t* __restrict__ packed, const uint8_t* __restrict__ scales,
                                    int kind, int nchunks, uint8_t* __restrict__ out) {
    const int K = kind == 1 ? I : H;
    const int cpu = kind == 1 ? 1 : NV_GU_CHUNKS;          // chunks per unit
    const size_t total = (size_t)nchunks * NV_CHUNK_KB * 32;
    const size_t prow = K / 2, srow = K / 16;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const int lane = (int)(i & 31), kb = (int)((i >> 5) & (NV_CHUNK_KB - 1));
        const int ch = (int)(i >> 10);
        const int unit = ch / cpu;
        const int kbg = (ch % cpu) * NV_CHUNK_KB + kb;
        auto row_of = [&](int arow) -> size_t {
            return kind == 0 ? (arow < 8 ? 8 * unit + arow : I + 8 * unit + (arow - 8)) : (size_t)16 * unit + arow;
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
            dst[NV_CODES + kb * 16 + 2 * lane] = scales[row_of(lane) * srow + kbg];
            dst[NV_CODES + kb * 16 + 2 * lane + 1] = scales[row_of(lane + 8) * srow + kbg];
        }
    }
}

cudaError_t launch_repack_nvfp4(const uint8_t* packed, const uint8_t* scales, int kind, int rows, uint8_t* out,
                                cudaStream_t s) {
    const int nchunks = kind == 0 ? NV_GU_UNITS * NV_GU_CHUNKS : kind == 1 ? NV_DN_UNITS : rows / 16 * NV_GU_CHUNKS;
    const size_t total = (size_t)nchunks * NV_CHUNK_KB * 32;
    const size_t blocks = (total + 255) / 256;
    repack_nvfp4_kernel<<<(unsigned)(blocks < 65535 * 16 ? blocks : 65535 * 16), 256, 0, s>>>(packed, scales, kind,
                                                                                              nchunks, out);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// gate/up + SwiGLU
// ---------------------------------------------------------------------------

constexpr int GN_WARPS = 8;
constexpr int GN_XROW = H + 8;                   // f16 per staged token row (+8: conflict-free B loads)
constexpr int NV_PIECE = NV_CHUNK / 2;           // half a chunk: 16 K blocks of codes, then their scales
constexpr int NV_PIECE_CODES = NV_CODES / 2;     // 2048
constexpr int NV_SMEM_BUDGET = 227 * 1024;       // dynamic shared memory of one CTA
constexpr int GN_PART = 2 * GN_WARPS * 32 * 4;   // partial sums [item parity][warp][lane][4]
static_assert(NV_PIECE % 16 == 0 && NV_PIECE_CODES % 16 == 0, "bulk copies want 16-byte pieces");

struct GateUpNvParams {
    const uint8_t* nv;            // owned experts, NV_EXPERT_BYTES each
    const float* ts;              // [NEXP][2] tensor scales (gate_up, down)
    const float* logits;          // [T][E]
    const __nv_bfloat16* x;       // [T][H]
    int T;
    int ns;                       // ring pieces per warp
    DecodeTables* tables_out;
    int32_t* idx_out;
    float* w_out;
    __nv_bfloat16* a;             // activations, act_index layout (the down kernel's MMA operand)
    uint32_t* status;
    uint64_t limit_ns;
};

static inline size_t gn_fixed_bytes(int T) {
    return (size_t)T * GN_XROW * 2 + DEC_T * 4 + (size_t)GN_PART * 4 + sizeof(DecodeTables) + DEC_T * TOPK * 8 +
           2 * E * 4 + DEC_MAX_CTA_ITEMS * 4 + 8;
}
// ring pieces per warp: what the shared memory left beside x holds, at most 8
// (4 for one or two tokens, whose CTAs have about three items each)
static inline int gn_ns(int T) {
    const int room = (int)(((size_t)NV_SMEM_BUDGET - gn_fixed_bytes(T)) / ((size_t)GN_WARPS * (NV_PIECE + 8)));
    const int cap = T <= 2 ? 4 : 8;
    return room < cap ? room : cap;
}
static inline size_t gn_smem_bytes(int T) {
    return (size_t)GN_WARPS * gn_ns(T) * (NV_PIECE + 8) + gn_fixed_bytes(T);
}

// Work items as in the bf16 kernel: (slot, unit of 8 gate + 8 up rows, tile of
// up to 8 tokens), one at a time per CTA.  Warp w takes K blocks 16w .. 16w +
// 15 (half of chunk w / 2 of the unit: 2 KiB of codes and 256 bytes of
// scales); the eight partial sums are added in warp order.
__global__ void __launch_bounds__(GN_WARPS * 32, 1) gateup_nvfp4_kernel(GateUpNvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int NS = p.ns, T = p.T, G = gridDim.x, c = blockIdx.x;
    uint8_t* ring = smem + (size_t)warp * NS * NV_PIECE;
    __half* xh = reinterpret_cast<__half*>(smem + (size_t)GN_WARPS * NS * NV_PIECE);
    float* xinv = reinterpret_cast<float*>(xh + (size_t)T * GN_XROW);
    float* part = xinv + DEC_T;
    uint64_t* bar = reinterpret_cast<uint64_t*>(part + GN_PART) + warp * NS;
    uint64_t* xbar = reinterpret_cast<uint64_t*>(part + GN_PART) + GN_WARPS * NS;   // the raw x rows
    DecodeTables* tab = reinterpret_cast<DecodeTables*>(xbar + 1);
    int* sel_e = reinterpret_cast<int*>(tab + 1);
    float* sel_w = reinterpret_cast<float*>(sel_e + DEC_T * TOPK);
    uint32_t* tmask = reinterpret_cast<uint32_t*>(sel_w + DEC_T * TOPK);
    int* pair0 = reinterpret_cast<int*>(tmask + E);
    int* list = pair0 + E;                           // this CTA's items c, c + G, ...

    if (lane == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&bar[s], 1);
        if (warp == 0) mbar_init(xbar, 1);
        fence_mbar_init();
    }
    __syncthreads();

    const int nt0 = (T + 7) >> 3;                    // token tiles of the shared slot (slot 0)
    auto issue = [&](int i, int it, int expert) {
        const int s = i % NS, r = (it >> 2) & (NV_GU_UNITS - 1);
        const uint8_t* chunk =
            p.nv + (size_t)expert * NV_EXPERT_BYTES + ((size_t)r * NV_GU_CHUNKS + (warp >> 1)) * NV_CHUNK;
        uint8_t* dst = ring + (size_t)s * NV_PIECE;
        mbar_arrive_expect_tx(&bar[s], NV_PIECE);
        bulk_g2s(dst, chunk + (warp & 1) * NV_PIECE_CODES, NV_PIECE_CODES, &bar[s]);
        bulk_g2s(dst + NV_PIECE_CODES, chunk + NV_CODES + (warp & 1) * (NV_PIECE - NV_PIECE_CODES),
                 NV_PIECE - NV_PIECE_CODES, &bar[s]);
    };

    // ---- before the router has finished: the shared slot's items ----
    int issued = 0;
    if (lane == 0) {
        for (int i = 0; i < NS && c + G * i < NV_GU_UNITS * nt0; ++i) {
            const int j = c + G * i;
            issue(i, ((j / nt0) << 2) | (j % nt0), SHARED);
            issued = i + 1;
        }
    }
    pdl_wait();     // router logits are complete (and x is ready)
    pdl_trigger();

    // ---- the raw bf16 x rows into their padded smem rows (lane t of warp 0
    // copies token t; T <= 32), landing while the CTA ranks the experts ----
    if (warp == 0) {
        if (lane == 0) mbar_arrive_expect_tx(xbar, (uint32_t)T * H * 2);
        __syncwarp();
        if (lane < T) bulk_g2s(xh + (size_t)lane * GN_XROW, p.x + (size_t)lane * H, H * 2, xbar);
    }

    // ---- top-6 of every token, then the (slot, token) tables and the items ----
    select_tokens_warps(p.logits, T, warp, lane, sel_e, sel_w, c == 0 ? p.idx_out : nullptr,
                        c == 0 ? p.w_out : nullptr);
    __syncthreads();
    bool xok = true;
    if (warp == 0) {
        build_decode_tables_warp(T, sel_e, sel_w, tmask, pair0, tab, lane);
    } else {
        // meanwhile: x -> f16 times 2^e_t per token, in place
        xok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(xbar, 0, p.limit_ns));
        for (int t = warp - 1; xok && t < T; t += GN_WARPS - 1) {
            uint4* row = reinterpret_cast<uint4*>(xh + (size_t)t * GN_XROW);
            uint4 v[8];
            float mx = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                v[k] = row[lane + 32 * k];
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
        }
    }
    bool ok = __syncthreads_and(xok);
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
        for (int i = issued; i < NS && i < my_items; ++i) {
            issue(i, list[i], tab->slot_expert[list[i] >> 8]);
            issued = i + 1;
        }
    }

    const int g = lane >> 2, cq = lane & 3;
    int i = 0;
    for (; ok && i < my_items; ++i) {
        const int it = list[i], u = it >> 8;
        const int pb = tab->slot_pair0[u], np = tab->slot_pair0[u + 1] - pb;
        const int n = (it & 3) * 8 + g;
        const __half* xb = xh + tab->pair_token[pb + (n < np ? n : np - 1)] * GN_XROW + warp * 256 + 2 * cq;
        const int s = i % NS;
        const bool got = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(&bar[s], (i / NS) & 1, p.limit_ns));
        float* pw = part + (((i & 1) * GN_WARPS + warp) * 32 + lane) * 4;
        if (got) {
            // four accumulators (K block kb goes to chain kb % 4)
            float acc[4][4];
#pragma unroll
            for (int ch = 0; ch < 4; ++ch) acc[ch][0] = acc[ch][1] = acc[ch][2] = acc[ch][3] = 0.f;
            const uint8_t* buf = ring + (size_t)s * NV_PIECE;
#pragma unroll
            for (int kb = 0; kb < 16; kb += 4) {
                uint32_t a[4][4];
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    nv_a_frag(*reinterpret_cast<const uint32_t*>(buf + (kb + ch) * 128 + 4 * lane),
                              *reinterpret_cast<const uint16_t*>(buf + NV_PIECE_CODES + (kb + ch) * 16 + 2 * g),
                              a[ch]);
#pragma unroll
                for (int ch = 0; ch < 4; ++ch)
                    mma_f16_16816(acc[ch], a[ch], *reinterpret_cast<const uint32_t*>(xb + (kb + ch) * 16),
                                  *reinterpret_cast<const uint32_t*>(xb + (kb + ch) * 16 + 8));
            }
            __syncwarp();   // every lane is done reading slot s
            if (lane == 0 && i + NS < my_items) {
                fence_proxy_async_smem();
                issue(i + NS, list[i + NS], tab->slot_expert[list[i + NS] >> 8]);
                issued = i + NS + 1;
            }
            *reinterpret_cast<float4*>(pw) = make_float4(acc[0][0] + acc[1][0] + (acc[2][0] + acc[3][0]),
                                                         acc[0][1] + acc[1][1] + (acc[2][1] + acc[3][1]),
                                                         acc[0][2] + acc[1][2] + (acc[2][2] + acc[3][2]),
                                                         acc[0][3] + acc[1][3] + (acc[2][3] + acc[3][3]));
        }
        if (!__syncthreads_and(got)) {
            ok = false;
            break;
        }
        // warp i % 8 adds the item's eight partial sums in warp order; lane
        // (g, cq) then holds gate (x, y) and up (z, w) of row 8r + g for tokens
        // 2cq, 2cq + 1 of the tile.  The buffer of parity i & 1 is next written
        // after the barrier of item i + 1, which this warp reaches only after
        // the sum.
        if (warp == (i & (GN_WARPS - 1))) {
            const float* pb0 = part + ((i & 1) * GN_WARPS * 32 + lane) * 4;
            float4 sum = *reinterpret_cast<const float4*>(pb0);
#pragma unroll
            for (int w = 1; w < GN_WARPS; ++w) {
                const float4 v = *reinterpret_cast<const float4*>(pb0 + w * 32 * 4);
                sum.x += v.x;
                sum.y += v.y;
                sum.z += v.z;
                sum.w += v.w;
            }
            const float tsg = __ldg(p.ts + 2 * tab->slot_expert[u]);
            const int j = 8 * ((it >> 2) & (NV_GU_UNITS - 1)) + g, n0 = (it & 3) * 8 + 2 * cq;
            if (n0 < np) {
                const float f = tsg * xinv[tab->pair_token[pb + n0]];
                p.a[act_index(pb + n0, j)] = __float2bfloat16_rn(silu_f(sum.x * f) * (sum.z * f));
            }
            if (n0 + 1 < np) {
                const float f = tsg * xinv[tab->pair_token[pb + n0 + 1]];
                p.a[act_index(pb + n0 + 1, j)] = __float2bfloat16_rn(silu_f(sum.y * f) * (sum.w * f));
            }
        }
    }
    if (lane == 0) {
        if (!ok) {
            report_status(p.status, ST_TIMEOUT);
            if (warp == 0) mbar_wait_bounded(xbar, 0, p.limit_ns);
        }
        // copies still in flight into this warp's ring (after a timeout, or the
        // shared slot's prefetched pieces when the item list came out empty):
        // wait for them, bounded, before the CTA exits
        for (int k = i; k < issued; ++k) mbar_wait_bounded(&bar[k % NS], (k / NS) & 1, p.limit_ns);
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// down projection + weighted combine
// ---------------------------------------------------------------------------

constexpr int DV_WARPS = 8;
constexpr int DV_CTAS = H / 16;        // 128: CTA c owns rows 16c .. 16c + 15
constexpr int DV_ACT = 8 * 256 * 2;    // an item's activation tile: 8 pairs x 256 columns, bf16
constexpr int DV_SLOT = NV_PIECE + DV_ACT;
static_assert(DV_SLOT % 16 == 0, "ring slots stay 16-byte aligned");

struct DownNvParams {
    const uint8_t* nv;
    const float* ts;
    const float* logits;          // [T][E] router logits (final before this kernel starts)
    const __nv_bfloat16* a;       // activations, act_index layout
    __nv_bfloat16* y;             // [T][H]
    int ns;                       // ring slots per warp
    int T;
    uint32_t* status;
    uint64_t limit_ns;
};

static inline size_t dv_fixed_bytes(int T) {
    return (size_t)DV_WARPS * T * 16 * 4 + sizeof(DecodeTables) + DEC_T * TOPK * 8 + 2 * E * 4 +
           (DEC_MAX_DOWN_ITEMS + 1) * 4;
}
// ring slots per warp: a warp has about 2 (T + 1) / 8 + 1 items at small T;
// small batches keep the kernel small, so the next layer's gate/up CTAs fit
// beside it
static inline int dv_ns(int T) {
    const int room = (int)(((size_t)NV_SMEM_BUDGET - dv_fixed_bytes(T)) / ((size_t)DV_WARPS * (DV_SLOT + 8)));
    const int cap = T <= 2 ? 2 : 4;
    return room < cap ? room : cap;
}
static inline size_t dv_smem_bytes(int T) { return (size_t)DV_WARPS * dv_ns(T) * (DV_SLOT + 8) + dv_fixed_bytes(T); }

// Work items as in the bf16 down kernel: (slot, column half, tile of 8
// tokens), item j to warp j % 8.  A ring slot holds half of the slot's
// 16-row chunk (2 KiB of codes and 256 bytes of scales) and the tile's
// activations (4 KiB, one bulk copy from the act_index layout).
__global__ void __launch_bounds__(DV_WARPS * 32, 1) down_nvfp4_kernel(DownNvParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int c = blockIdx.x, NS = p.ns, Tk = p.T;
    uint8_t* ring = smem + (size_t)warp * NS * DV_SLOT;
    float* yw_all = reinterpret_cast<float*>(smem + (size_t)DV_WARPS * NS * DV_SLOT);
    float* yw = yw_all + warp * Tk * 16;                                                  // [8][T][16]
    uint64_t* bars = reinterpret_cast<uint64_t*>(yw_all + DV_WARPS * Tk * 16);
    uint64_t* bar = bars + warp * NS;
    DecodeTables* tab = reinterpret_cast<DecodeTables*>(bars + DV_WARPS * NS);
    int* sel_e = reinterpret_cast<int*>(tab + 1);
    float* sel_w = reinterpret_cast<float*>(sel_e + DEC_T * TOPK);
    uint32_t* tmask = reinterpret_cast<uint32_t*>(sel_w + DEC_T * TOPK);
    int* pair0 = reinterpret_cast<int*>(tmask + E);
    int* items = pair0 + E;
    int* n_items_s = items + DEC_MAX_DOWN_ITEMS;

    if (lane == 0) {
        for (int s = 0; s < NS; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    auto item_of = [&](int k) { return items[warp + DV_WARPS * k]; };
    auto copy_w = [&](int k) {
        const int it = item_of(k), s = k % NS, hk = (it >> 2) & 1;
        const uint8_t* chunk =
            p.nv + (size_t)tab->slot_expert[it >> 3] * NV_EXPERT_BYTES + NV_GU_BYTES + (size_t)c * NV_CHUNK;
        uint8_t* dst = ring + (size_t)s * DV_SLOT;
        bulk_g2s(dst, chunk + hk * NV_PIECE_CODES, NV_PIECE_CODES, &bar[s]);
        bulk_g2s(dst + NV_PIECE_CODES, chunk + NV_CODES + hk * (NV_PIECE - NV_PIECE_CODES),
                 NV_PIECE - NV_PIECE_CODES, &bar[s]);
    };
    auto copy_a = [&](int k) {
        const int it = item_of(k), s = k % NS;
        const int p0 = tab->slot_pair0[it >> 3] + (it & 3) * 8;
        bulk_g2s(ring + (size_t)s * DV_SLOT + NV_PIECE, p.a + ((size_t)((it >> 2) & 1) * DEC_ACT_ROWS + p0) * 256,
                 DV_ACT, &bar[s]);
    };
    // Every gate/up CTA triggers this launch only after its own dependency
    // wait, which returns once the router grid has completed: the logits are
    // final here although the gate/up kernel may still be running.  Select
    // each token's experts and build the same tables the gate/up kernel
    // builds, and start the weight pieces of this warp's first items now, so
    // they stream while the gate/up kernel runs.
    select_tokens_warps(p.logits, Tk, warp, lane, sel_e, sel_w, nullptr, nullptr);
    for (int k = threadIdx.x; k < DV_WARPS * Tk * 16; k += blockDim.x) yw_all[k] = 0.f;
    __syncthreads();
    if (warp == 0) {
        build_decode_tables_warp(Tk, sel_e, sel_w, tmask, pair0, tab, lane);
        const int n = build_down_items_warp(tab, items, lane);
        if (lane == 0) *n_items_s = n;
    }
    __syncthreads();
    const int n_items = *n_items_s;
    const int my_items = n_items > warp ? (n_items - warp + DV_WARPS - 1) / DV_WARPS : 0;
    // weights of the first items now (the phase waits for its arrival, which
    // comes with the activations after the dependency wait)
    int issued = 0;
    if (lane == 0) {
        for (int k = 0; k < NS && k < my_items; ++k) {
            mbar_expect_tx(&bar[k], NV_PIECE);
            copy_w(k);
            issued = k + 1;
        }
    }
    pdl_wait();     // the gate/up kernel is complete: activations are visible
    pdl_trigger();
    if (lane == 0) {
        for (int k = 0; k < issued; ++k) {
            mbar_arrive_expect_tx(&bar[k], DV_ACT);
            copy_a(k);
        }
    }

    const int g = lane >> 2, cq = lane & 3;
    bool ok = true;
    int k = 0;
    for (; k < my_items; ++k) {
        const int it = item_of(k), u = it >> 3, nt = it & 3;
        const int pb = tab->slot_pair0[u], np = tab->slot_pair0[u + 1] - pb;
        const int s = k % NS;
        if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&bar[s], (k / NS) & 1, p.limit_ns))) {
            ok = false;
            break;
        }
        const uint8_t* buf = ring + (size_t)s * DV_SLOT;
        // row g of the activation tile; chunk q of it sits at q ^ (pair % 8)
        const uint8_t* ar = buf + NV_PIECE + g * 512 + 4 * cq;
        const int sw = (pb + nt * 8 + g) & 7;
        float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kb = 0; kb < 16; ++kb) {
            uint32_t a[4];
            nv_a_frag(*reinterpret_cast<const uint32_t*>(buf + kb * 128 + 4 * lane),
                      *reinterpret_cast<const uint16_t*>(buf + NV_PIECE_CODES + kb * 16 + 2 * g), a);
#pragma unroll
            for (int q = 0; q < 4; ++q) a[q] = f16x2_to_bf16x2(a[q]);
            mma_bf16_16816(acc[kb & 1], a, *reinterpret_cast<const uint32_t*>(ar + (((2 * kb) ^ sw) << 4)),
                           *reinterpret_cast<const uint32_t*>(ar + (((2 * kb + 1) ^ sw) << 4)));
        }
        __syncwarp();
        if (lane == 0 && k + NS < my_items) {
            fence_proxy_async_smem();
            mbar_arrive_expect_tx(&bar[s], NV_PIECE + DV_ACT);
            copy_w(k + NS);
            copy_a(k + NS);
            issued = k + NS + 1;
        }
        // lane (g, cq): rows g and g + 8 of this CTA's 16, tokens 2cq, 2cq + 1 of the tile
        const float tsd = __ldg(p.ts + 2 * tab->slot_expert[u] + 1);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
            const int n = nt * 8 + 2 * cq + hh;
            if (n < np) {
                const int pr = pb + n, t = tab->pair_token[pr];
                const float wgt = tab->pair_weight[pr] * tsd;
                yw[t * 16 + g] = fmaf(wgt, acc[0][hh] + acc[1][hh], yw[t * 16 + g]);
                yw[t * 16 + g + 8] = fmaf(wgt, acc[0][2 + hh] + acc[1][2 + hh], yw[t * 16 + g + 8]);
            }
        }
    }
    if (!ok && lane == 0) {
        report_status(p.status, ST_TIMEOUT);
        for (int q = k; q < issued; ++q) mbar_wait_bounded(&bar[q % NS], (q / NS) & 1, p.limit_ns);
    }
    __syncthreads();
    // y rows 16c .. 16c + 15: the eight warps' partial sums in warp order
    for (int q = threadIdx.x; q < Tk * 16; q += blockDim.x) {
        const int t = q >> 4, rr = q & 15;
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
    size_t gmax = 0, dmax = 0;
    for (int T = 1; T <= DEC_T; ++T) {
        gmax = gn_smem_bytes(T) > gmax ? gn_smem_bytes(T) : gmax;
        dmax = dv_smem_bytes(T) > dmax ? dv_smem_bytes(T) : dmax;
    }
    cudaError_t e = cudaFuncSetAttribute(gateup_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gmax);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(down_nvfp4_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)dmax);
}

cudaError_t launch_decode_experts_nvfp4(const LaunchCtx& L, const uint8_t* nv, const float* nv_ts,
                                        const float* logits, const __nv_bfloat16* x, int T, DecodeTables* tables,
                                        int32_t* idx, float* w, __nv_bfloat16* a_buf, __nv_bfloat16* y) {
    __nv_bfloat16* a16 = a_buf;
    if (T < 1 || T > DEC_T) return cudaErrorInvalidValue;
    GateUpNvParams gp{nv, nv_ts, logits, x, T, gn_ns(T), tables, idx, w, a16, L.status, L.wait_limit_ns};
    // at most 64 x (257 + 28) items over the grid: 72 CTAs or more keep every
    // CTA's list within DEC_MAX_CTA_ITEMS
    const int gi = L.num_sms >= DEC_MIN_GRID ? L.num_sms : DEC_MIN_GRID;
    cudaError_t e = launch_hooked(L, FLINT_KERNEL_GATE_UP, gateup_nvfp4_kernel, dim3(gi), dim3(GN_WARPS * 32),
                                  gn_smem_bytes(T), gp);
    if (e != cudaSuccess) return e;
    DownNvParams dp{nv, nv_ts, logits, a16, y, dv_ns(T), T, L.status, L.wait_limit_ns};
    return launch_hooked(L, FLINT_KERNEL_DOWN, down_nvfp4_kernel, dim3(DV_CTAS), dim3(DV_WARPS * 32),
                         dv_smem_bytes(T), dp);
}

}  // namespace flint
