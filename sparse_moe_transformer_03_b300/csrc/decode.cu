// decode.cu -- weight-streaming expert kernels for small batches (T <= 32).
//
// At decode sizes each expert weight is used by only a few tokens, so the
// layer is bound by reading the touched experts' weights from HBM once:
// (U + 1) experts x 6 MiB, U = distinct routed experts of the batch.  After
// the router kernel has written the fp32 logits, two kernels run, chained
// with programmatic dependent launch:
//
//   gateup_decode  Every CTA selects the top-6 of each token from the logits
//                  and builds the (expert slot, token) tables in its own
//                  shared memory (slot 0 = the shared expert).  Work units
//                  are one (gate row j, up row I+j) pair of one expert: 8 KiB
//                  streamed by cp.async.bulk into a per-warp smem ring, dotted
//                  with each of the expert's tokens (x staged in smem), and
//                  a = silu(g) * u written per (expert, token) pair.  Units
//                  are dealt to CTAs cyclically so every SM streams the same
//                  number of bytes and the many-token shared expert is spread
//                  over all of them.  The shared expert does not depend on the
//                  routing: its first units are requested before the kernel
//                  waits on the router.
//   down_decode    CTA c owns output rows [h0, h1) of y.  It reads rows
//                  [h0, h1) of every touched expert's down matrix and the
//                  activations of each slot (staged in
//                  smem with one bulk copy per chunk of slots) and accumulates
//                  w * (Wd a) per token in a fixed order (shared expert first,
//                  then routed experts by id): the combine is fused and
//                  deterministic.  It keeps its smem small so the next
//                  layer's gateup_decode CTAs fit beside it and start
//                  streaming.
//
// Layer definition: RecursiveSI/flint (vLLM recipe page), "Overview" (256
// experts, top-6 sigmoid routing plus a shared expert); SwiGLU experts with
// H = 2048, I = 512 are this library's reading (the pages name neither).
#include "flint_common.cuh"
#include "../../include/flint_moe.h"
#include "flint_internal.h"
#include "routing.cuh"

namespace flint {

constexpr int GU_WARPS = 8;
constexpr int GU_NS = 2;                              // ring slots per warp
constexpr int GU_UNIT = 2 * H * 2;                    // one (gate row, up row) pair
constexpr int GU_XS_T = 4;                            // tokens whose x is staged in smem
constexpr int GU_RING = GU_WARPS * GU_NS * GU_UNIT;   // 128 KiB
constexpr int GU_XS = GU_XS_T * H * 2;                // 16 KiB
constexpr int GU_NBAR = GU_WARPS * GU_NS + 1;
constexpr int GU_SMEM = GU_RING + GU_XS + GU_NBAR * 8 + NEXP * 8 + (int)sizeof(DecodeTables) + DEC_T * TOPK * 8 + 2 * E * 4;

constexpr int DN_WARPS = 8;
constexpr int DN_APAIRS = DEC_T;   // activation vectors staged per chunk (>= pairs of any slot)
constexpr int DN_GROUP = 4;        // expert slots whose down rows are loaded together
constexpr int DN_REG_T = 4;        // up to this many tokens the partial sums stay in registers

// grid of the down kernel (>= 128 so a CTA owns at most 16 rows, 2 per warp)
inline int down_grid(int num_sms) { return num_sms < 128 ? 128 : num_sms; }

struct GateUpParams {
    const ExpertTables* experts;
    const float* logits;          // [T][E] fp32 router logits (bias included)
    const __nv_bfloat16* x;       // [T][H]
    int T;
    DecodeTables* tables_out;     // written by CTA 0 for the down kernel
    int32_t* idx_out;             // [T][6], written by CTA 0
    float* w_out;                 // [T][6], written by CTA 0
    float* a;                     // [pairs][I]
    uint32_t* status;
    uint64_t limit_ns;
};

// At most 128 registers (and the down kernel at most 128): 8 warps of each fit
// in the SM's 64K registers together, so the next layer's gate/up CTAs can
// start streaming while the down kernel still runs.
__global__ void __launch_bounds__(GU_WARPS * 32, 2) gateup_decode_kernel(GateUpParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ring = smem + warp * GU_NS * GU_UNIT;
    __nv_bfloat16* xs = reinterpret_cast<__nv_bfloat16*>(smem + GU_RING);
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + GU_RING + GU_XS);
    uint64_t* bar = bars + warp * GU_NS;
    uint64_t* xbar = bars + GU_WARPS * GU_NS;
    const __nv_bfloat16** wptr = reinterpret_cast<const __nv_bfloat16**>(bars + GU_NBAR);   // [NEXP]
    DecodeTables* tab = reinterpret_cast<DecodeTables*>(wptr + NEXP);
    int* sel_e = reinterpret_cast<int*>(tab + 1);
    float* sel_w = reinterpret_cast<float*>(sel_e + DEC_T * TOPK);
    uint32_t* tmask = reinterpret_cast<uint32_t*>(sel_w + DEC_T * TOPK);
    int* pair0 = reinterpret_cast<int*>(tmask + E);
    const int G = gridDim.x, c = blockIdx.x, T = p.T;

    // the experts' gate/up pointers (immutable) into smem, so issuing a unit
    // never waits on a dependent global load
    for (int e = threadIdx.x; e < NEXP; e += blockDim.x) wptr[e] = p.experts->gate_up[e];
    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < GU_NS; ++s) mbar_init(&bar[s], 1);
        if (warp == 0) mbar_init(xbar, 1);
        fence_mbar_init();
    }
    __syncthreads();

    auto unit_of = [&](int i) { return c + G * (warp + GU_WARPS * i); };
    auto issue = [&](int i, int expert) {
        const int q = unit_of(i), j = q & (I - 1), s = i % GU_NS;
        const __nv_bfloat16* W = wptr[expert];
        mbar_arrive_expect_tx(&bar[s], GU_UNIT);
        bulk_g2s(ring + s * GU_UNIT, W + (size_t)j * H, H * 2, &bar[s]);
        bulk_g2s(ring + s * GU_UNIT + H * 2, W + (size_t)(I + j) * H, H * 2, &bar[s]);
    };

    // ---- before the router has finished: routing-independent traffic ----
    int issued = 0;
    if (lane == 0) {
        for (int i = 0; i < GU_NS && unit_of(i) < I; ++i) {   // shared-expert units
            issue(i, SHARED);
            issued = i + 1;
        }
    }
    pdl_wait();     // router logits are complete and visible (and x is ready)
    pdl_trigger();  // the down kernel may be scheduled

    const bool x_in_smem = T <= GU_XS_T;
    if (threadIdx.x == 0 && x_in_smem) {
        mbar_arrive_expect_tx(xbar, T * H * 2);
        bulk_g2s(xs, p.x, T * H * 2, xbar);
    }

    // ---- top-6 of every token, then the (slot, token) tables, in smem ----
    for (int t = warp; t < T; t += GU_WARPS) {
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
        // publish the tables for the down kernel
        const int* src = reinterpret_cast<const int*>(tab);
        int* dst = reinterpret_cast<int*>(p.tables_out);
        for (int k = threadIdx.x; k < (int)(sizeof(DecodeTables) / 4); k += blockDim.x) dst[k] = src[k];
    }
    const int n_slots = tab->n_slots;
    const int total = n_slots * I;
    if (lane == 0) {
        for (int i = issued; i < GU_NS && unit_of(i) < total; ++i) {
            issue(i, tab->slot_expert[unit_of(i) >> 9]);
            issued = i + 1;
        }
    }
    bool ok = true;
    if (x_in_smem) ok = __all_sync(0xFFFFFFFFu, mbar_wait_bounded(xbar, 0, p.limit_ns));

    int i = 0;
    for (; ok && unit_of(i) < total; ++i) {
        const int q = unit_of(i), s = i % GU_NS;
        // every lane waits; the decision to give up is taken by the whole warp
        if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&bar[s], (i / GU_NS) & 1, p.limit_ns))) {
            ok = false;
            break;
        }
        const uint8_t* buf = ring + s * GU_UNIT;
        const int u = q >> 9, j = q & (I - 1);
        const int pb = tab->slot_pair0[u], pe = tab->slot_pair0[u + 1];
        for (int pr = pb; pr < pe; ++pr) {
            const int t = tab->pair_token[pr];
            float g = 0.f, up = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int off = 8 * (lane + 32 * k);
                const uint4 wg = *reinterpret_cast<const uint4*>(buf + 2 * off);
                const uint4 wu = *reinterpret_cast<const uint4*>(buf + H * 2 + 2 * off);
                const uint4 xv = x_in_smem ? *reinterpret_cast<const uint4*>(xs + t * H + off)
                                           : ldg16(p.x + (size_t)t * H + off);
                const float x0 = bf_lo(xv.x), x1 = bf_hi(xv.x), x2 = bf_lo(xv.y), x3 = bf_hi(xv.y);
                const float x4 = bf_lo(xv.z), x5 = bf_hi(xv.z), x6 = bf_lo(xv.w), x7 = bf_hi(xv.w);
                g = fmaf(bf_lo(wg.x), x0, g);
                g = fmaf(bf_hi(wg.x), x1, g);
                g = fmaf(bf_lo(wg.y), x2, g);
                g = fmaf(bf_hi(wg.y), x3, g);
                g = fmaf(bf_lo(wg.z), x4, g);
                g = fmaf(bf_hi(wg.z), x5, g);
                g = fmaf(bf_lo(wg.w), x6, g);
                g = fmaf(bf_hi(wg.w), x7, g);
                up = fmaf(bf_lo(wu.x), x0, up);
                up = fmaf(bf_hi(wu.x), x1, up);
                up = fmaf(bf_lo(wu.y), x2, up);
                up = fmaf(bf_hi(wu.y), x3, up);
                up = fmaf(bf_lo(wu.z), x4, up);
                up = fmaf(bf_hi(wu.z), x5, up);
                up = fmaf(bf_lo(wu.w), x6, up);
                up = fmaf(bf_hi(wu.w), x7, up);
            }
            g = warp_sum(g);
            up = warp_sum(up);
            if (lane == 0) p.a[(size_t)pr * I + j] = silu_f(g) * up;
        }
        __syncwarp();   // every lane is done reading slot s
        if (lane == 0 && unit_of(i + GU_NS) < total) {
            fence_proxy_async_smem();
            issue(i + GU_NS, tab->slot_expert[unit_of(i + GU_NS) >> 9]);
        }
    }
    if (!ok) {
        if (lane == 0) {
            report_status(p.status, ST_TIMEOUT);
            // drain copies still in flight into this warp's ring (bounded)
            for (int k = i; k < i + GU_NS && k < issued + 64 && unit_of(k) < total; ++k)
                mbar_wait_bounded(&bar[k % GU_NS], (k / GU_NS) & 1, p.limit_ns);
        }
        __syncwarp();
    }
}

struct DownParams {
    const ExpertTables* experts;
    const DecodeTables* tables;
    const float* a;         // [pairs][I]
    __nv_bfloat16* y;       // [T][H]
    int rows_max;           // ceil(H / gridDim.x) <= 16
    int apairs;             // activation vectors the smem buffer holds
    uint32_t* status;
    uint64_t limit_ns;
};

__global__ void __launch_bounds__(DN_WARPS * 32, 2) down_decode_kernel(DownParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, c = blockIdx.x;
    const int h0 = (c * H) / G, h1 = ((c + 1) * H) / G, nrows = h1 - h0;
    float* a_s = reinterpret_cast<float*>(smem);                          // [apairs][I]
    uint64_t* bar = reinterpret_cast<uint64_t*>(a_s + (size_t)p.apairs * I);
    const __nv_bfloat16** dptr = reinterpret_cast<const __nv_bfloat16**>(bar + 1);   // [NEXP]
    DecodeTables* tab = reinterpret_cast<DecodeTables*>(dptr + NEXP);
    float* yacc = reinterpret_cast<float*>(tab + 1);                      // [T][rows_max]

    // the experts' down pointers (immutable) into smem before waiting
    for (int e = threadIdx.x; e < NEXP; e += blockDim.x) dptr[e] = p.experts->down[e];
    pdl_wait();       // the gate/up kernel is complete: tables and activations are visible
    pdl_trigger();    // the next kernel on the stream may be scheduled
    if (threadIdx.x == 0) {
        mbar_init(bar, 1);
        fence_mbar_init();
        // small batches: all activation vectors fit, start their copy at once
        const int np = __ldcg(&p.tables->n_pairs);
        if (np <= p.apairs) {
            mbar_arrive_expect_tx(bar, np * I * 4);
            bulk_g2s(a_s, p.a, np * I * 4, bar);
        }
    }
    {
        const int* src = reinterpret_cast<const int*>(p.tables);
        int* dst = reinterpret_cast<int*>(tab);
        for (int k = threadIdx.x; k < (int)(sizeof(DecodeTables) / 4); k += blockDim.x) dst[k] = __ldcg(src + k);
    }
    __syncthreads();
    const int T = tab->T, n_slots = tab->n_slots;
    const bool one_chunk = tab->n_pairs <= p.apairs;
    for (int k = threadIdx.x; k < T * p.rows_max; k += blockDim.x) yacc[k] = 0.f;
    const int r0 = warp, r1 = warp + DN_WARPS;
    const bool has0 = r0 < nrows, has1 = r1 < nrows;
    float acc[DN_REG_T][2];
#pragma unroll
    for (int tt = 0; tt < DN_REG_T; ++tt) acc[tt][0] = acc[tt][1] = 0.f;

    bool ok = true;
    int chunk = 0;
    for (int u0 = 0; u0 < n_slots; ++chunk) {
        // the next chunk of slots whose activation vectors fit in smem
        int u1 = u0 + 1;
        while (u1 < n_slots && tab->slot_pair0[u1 + 1] - tab->slot_pair0[u0] <= p.apairs) ++u1;
        const int p0 = tab->slot_pair0[u0], p1 = tab->slot_pair0[u1];
        if (threadIdx.x == 0 && !one_chunk) {
            mbar_arrive_expect_tx(bar, (p1 - p0) * I * 4);
            bulk_g2s(a_s, p.a + (size_t)p0 * I, (p1 - p0) * I * 4, bar);
        }
        if (!__syncthreads_and(mbar_wait_bounded(bar, chunk & 1, p.limit_ns))) {
            ok = false;
            break;
        }
        for (int g = u0; g < u1; g += DN_GROUP) {
            uint4 wv[DN_GROUP][2][2];
#pragma unroll
            for (int jj = 0; jj < DN_GROUP; ++jj) {
                if (g + jj < u1) {
                    const __nv_bfloat16* W = dptr[tab->slot_expert[g + jj]];
                    if (has0) {
                        wv[jj][0][0] = ldg16(W + (size_t)(h0 + r0) * I + 8 * lane);
                        wv[jj][0][1] = ldg16(W + (size_t)(h0 + r0) * I + 256 + 8 * lane);
                    }
                    if (has1) {
                        wv[jj][1][0] = ldg16(W + (size_t)(h0 + r1) * I + 8 * lane);
                        wv[jj][1][1] = ldg16(W + (size_t)(h0 + r1) * I + 256 + 8 * lane);
                    }
                }
            }
#pragma unroll
            for (int jj = 0; jj < DN_GROUP; ++jj) {
                const int u = g + jj;
                if (u >= u1) break;
                for (int pr = tab->slot_pair0[u]; pr < tab->slot_pair0[u + 1]; ++pr) {
                    const float* ar = a_s + (size_t)(pr - p0) * I;
                    const float4 a0 = *reinterpret_cast<const float4*>(ar + 8 * lane);
                    const float4 a1 = *reinterpret_cast<const float4*>(ar + 8 * lane + 4);
                    const float4 a2 = *reinterpret_cast<const float4*>(ar + 256 + 8 * lane);
                    const float4 a3 = *reinterpret_cast<const float4*>(ar + 256 + 8 * lane + 4);
                    const int t = tab->pair_token[pr];
                    const float wgt = tab->pair_weight[pr];
                    float d[2];
#pragma unroll
                    for (int rr = 0; rr < 2; ++rr) {
                        const uint4 w0 = wv[jj][rr][0], w1 = wv[jj][rr][1];
                        float x = bf_lo(w0.x) * a0.x;
                        x = fmaf(bf_hi(w0.x), a0.y, x);
                        x = fmaf(bf_lo(w0.y), a0.z, x);
                        x = fmaf(bf_hi(w0.y), a0.w, x);
                        x = fmaf(bf_lo(w0.z), a1.x, x);
                        x = fmaf(bf_hi(w0.z), a1.y, x);
                        x = fmaf(bf_lo(w0.w), a1.z, x);
                        x = fmaf(bf_hi(w0.w), a1.w, x);
                        float z = bf_lo(w1.x) * a2.x;
                        z = fmaf(bf_hi(w1.x), a2.y, z);
                        z = fmaf(bf_lo(w1.y), a2.z, z);
                        z = fmaf(bf_hi(w1.y), a2.w, z);
                        z = fmaf(bf_lo(w1.z), a3.x, z);
                        z = fmaf(bf_hi(w1.z), a3.y, z);
                        z = fmaf(bf_lo(w1.w), a3.z, z);
                        z = fmaf(bf_hi(w1.w), a3.w, z);
                        d[rr] = x + z;
                    }
                    if (T <= DN_REG_T) {
                        // weighted partial sums stay in registers; one warp
                        // reduction per (row, token) after the last slot
#pragma unroll
                        for (int tt = 0; tt < DN_REG_T; ++tt) {
                            if (t == tt) {
                                acc[tt][0] = fmaf(wgt, d[0], acc[tt][0]);
                                acc[tt][1] = fmaf(wgt, d[1], acc[tt][1]);
                            }
                        }
                    } else {
                        const float d0 = has0 ? warp_sum(d[0]) : 0.f;
                        const float d1 = has1 ? warp_sum(d[1]) : 0.f;
                        if (lane == 0) {
                            if (has0) yacc[t * p.rows_max + r0] += wgt * d0;
                            if (has1) yacc[t * p.rows_max + r1] += wgt * d1;
                        }
                    }
                }
            }
        }
        __syncthreads();   // every warp is done with a_s
        u0 = u1;
    }
    if (!ok) {
        if (threadIdx.x == 0) report_status(p.status, ST_TIMEOUT);
        return;
    }
    if (T <= DN_REG_T) {
#pragma unroll
        for (int tt = 0; tt < DN_REG_T; ++tt) {
            if (tt < T) {
                const float s0 = warp_sum(acc[tt][0]);
                const float s1 = warp_sum(acc[tt][1]);
                if (lane == 0) {
                    if (has0) yacc[tt * p.rows_max + r0] = s0;
                    if (has1) yacc[tt * p.rows_max + r1] = s1;
                }
            }
        }
        __syncthreads();
    }
    for (int k = threadIdx.x; k < T * nrows; k += blockDim.x) {
        const int t = k / nrows, r = k % nrows;
        p.y[(size_t)t * H + h0 + r] = __float2bfloat16_rn(yacc[t * p.rows_max + r]);
    }
}

static int down_smem_bytes(int T, int rows_max, int apairs) {
    return apairs * I * 4 + 8 + NEXP * 8 + (int)sizeof(DecodeTables) + T * rows_max * 4;
}

cudaError_t decode_set_attributes() {
    cudaError_t e = cudaFuncSetAttribute(gateup_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GU_SMEM);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(down_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                down_smem_bytes(DEC_T, 16, DN_APAIRS));
}

cudaError_t launch_decode_experts(const LaunchCtx& L, const ExpertTables* experts, const float* logits,
                                  const __nv_bfloat16* x, int T, DecodeTables* tables, int32_t* idx, float* w,
                                  float* a_buf, __nv_bfloat16* y) {
    const int Gd = down_grid(L.num_sms);
    GateUpParams gp{experts, logits, x, T, tables, idx, w, a_buf, L.status, L.wait_limit_ns};
    cudaError_t e = launch_hooked(L, FLINT_KERNEL_GATE_UP, gateup_decode_kernel, dim3(L.num_sms), dim3(GU_WARPS * 32), GU_SMEM, gp);
    if (e != cudaSuccess) return e;
    const int rows_max = (H + Gd - 1) / Gd;
    const int apairs = (TOPK + 1) * T < DN_APAIRS ? (TOPK + 1) * T : DN_APAIRS;
    DownParams dp{experts, tables, a_buf, y, rows_max, apairs, L.status, L.wait_limit_ns};
    return launch_hooked(L, FLINT_KERNEL_DOWN, down_decode_kernel, dim3(Gd), dim3(DN_WARPS * 32), down_smem_bytes(T, rows_max, apairs),
                      dp);
}

}  // namespace flint
