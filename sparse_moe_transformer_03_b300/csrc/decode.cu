// decode.cu -- weight-streaming expert kernels for small batches (T <= 32).
//
// At decode sizes each expert weight is used by only a few tokens, so the
// layer is bound by reading the touched experts' weights from HBM once:
// (U + 1) experts x 6 MiB, U = distinct routed experts of the batch.  Two
// kernels, chained with programmatic dependent launch:
//
//   gateup_decode  units of one (gate row j, up row I+j) pair of an expert:
//                  8 KiB streamed by cp.async.bulk into a per-warp smem ring,
//                  dotted with each of the expert's tokens (bf16 x, fp32 sums),
//                  a = silu(g) * u written per (expert, token) pair.  Units
//                  are dealt to CTAs cyclically so every SM streams the same
//                  number of bytes and the many-token shared expert is spread
//                  over all of them.  The shared expert (slot 0) does not
//                  depend on the routing: its first units are requested
//                  before the kernel waits on the router.
//   down_decode    CTA c owns output rows [h0, h1) of y.  It streams rows
//                  [h0, h1) of every touched expert's down matrix (one bulk
//                  copy per expert) and accumulates w * (Wd a) per token in a
//                  fixed order (shared expert first, then routed experts by
//                  id), so the combine is fused and deterministic.  Its first
//                  stages are requested while gateup_decode still runs.
//
// Layer definition: RecursiveSI/flint (vLLM recipe page), "Overview" (256
// experts, top-6 sigmoid routing plus a shared expert); SwiGLU experts with
// H = 2048, I = 512 are this library's reading (the pages name neither).
#include "flint_common.cuh"
#include "flint_internal.h"

namespace flint {

constexpr int GU_WARPS = 8;
constexpr int GU_NS = 2;              // ring slots per warp
constexpr int GU_UNIT = 2 * H * 2;    // bytes of one (gate row, up row) pair
constexpr int GU_SMEM = GU_WARPS * GU_NS * GU_UNIT + GU_WARPS * GU_NS * 8;

constexpr int DN_WARPS = 8;
constexpr int DN_NS = 6;              // ring slots
constexpr int DN_PREFETCH = 16;       // further stages hinted into L2

struct GateUpParams {
    const ExpertTables* experts;
    const DecodeTables* tables;
    const __nv_bfloat16* x;  // [T][H]
    float* a;                // [pairs][I]
    uint32_t* status;
    uint64_t limit_ns;
};

// at most 168 registers: 8 warps x 168 plus a down_decode CTA (8 warps x 80)
// still fit in the SM's 64K registers, so the two kernels can overlap
__global__ void __maxnreg__(168) gateup_decode_kernel(GateUpParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t* ring = smem + warp * GU_NS * GU_UNIT;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + GU_WARPS * GU_NS * GU_UNIT) + warp * GU_NS;
    const int G = gridDim.x, c = blockIdx.x;

    if (lane == 0) {
#pragma unroll
        for (int s = 0; s < GU_NS; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncwarp();

    // i-th unit of this warp
    auto unit_of = [&](int i) { return c + G * (warp + GU_WARPS * i); };
    auto issue = [&](int i, int expert) {
        const int q = unit_of(i), j = q & (I - 1), s = i % GU_NS;
        const __nv_bfloat16* W = p.experts->gate_up[expert];
        mbar_arrive_expect_tx(&bar[s], GU_UNIT);
        bulk_g2s(ring + s * GU_UNIT, W + (size_t)j * H, H * 2, &bar[s]);
        bulk_g2s(ring + s * GU_UNIT + H * 2, W + (size_t)(I + j) * H, H * 2, &bar[s]);
    };

    // shared-expert units (q < I) do not depend on the routing
    int issued = 0;
    if (lane == 0) {
        for (int i = 0; i < GU_NS && unit_of(i) < I; ++i) {
            issue(i, SHARED);
            issued = i + 1;
        }
    }
    pdl_wait();      // router done: tables are visible (and x is ready)
    pdl_trigger();   // the down kernel may start streaming its rows

    const int n_slots = p.tables->n_slots;
    const int total = n_slots * I;
    if (lane == 0) {
        for (int i = issued; i < GU_NS && unit_of(i) < total; ++i) {
            issue(i, p.tables->slot_expert[unit_of(i) >> 9]);
            issued = i + 1;
        }
    }

    bool ok = true;
    int i = 0;
    for (; unit_of(i) < total; ++i) {
        const int q = unit_of(i), s = i % GU_NS;
        // every lane waits; the decision to give up is taken by the whole warp
        if (!__all_sync(0xFFFFFFFFu, mbar_wait_bounded(&bar[s], (i / GU_NS) & 1, p.limit_ns))) {
            ok = false;
            break;
        }
        const uint8_t* buf = ring + s * GU_UNIT;
        uint4 wg[8], wu[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            wg[k] = *reinterpret_cast<const uint4*>(buf + 16 * (lane + 32 * k));
            wu[k] = *reinterpret_cast<const uint4*>(buf + H * 2 + 16 * (lane + 32 * k));
        }
        __syncwarp();
        if (lane == 0 && unit_of(i + GU_NS) < total) {
            fence_proxy_async_smem();
            issue(i + GU_NS, p.tables->slot_expert[unit_of(i + GU_NS) >> 9]);
        }
        const int u = q >> 9, j = q & (I - 1);
        const int pb = p.tables->slot_pair0[u], pe = p.tables->slot_pair0[u + 1];
        for (int pr = pb; pr < pe; ++pr) {
            const int t = p.tables->pair_token[pr];
            const __nv_bfloat16* xr = p.x + (size_t)t * H;
            float g = 0.f, up = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const uint4 xv = ldg16(xr + 8 * (lane + 32 * k));
                const float x0 = bf_lo(xv.x), x1 = bf_hi(xv.x), x2 = bf_lo(xv.y), x3 = bf_hi(xv.y);
                const float x4 = bf_lo(xv.z), x5 = bf_hi(xv.z), x6 = bf_lo(xv.w), x7 = bf_hi(xv.w);
                g = fmaf(bf_lo(wg[k].x), x0, g);
                g = fmaf(bf_hi(wg[k].x), x1, g);
                g = fmaf(bf_lo(wg[k].y), x2, g);
                g = fmaf(bf_hi(wg[k].y), x3, g);
                g = fmaf(bf_lo(wg[k].z), x4, g);
                g = fmaf(bf_hi(wg[k].z), x5, g);
                g = fmaf(bf_lo(wg[k].w), x6, g);
                g = fmaf(bf_hi(wg[k].w), x7, g);
                up = fmaf(bf_lo(wu[k].x), x0, up);
                up = fmaf(bf_hi(wu[k].x), x1, up);
                up = fmaf(bf_lo(wu[k].y), x2, up);
                up = fmaf(bf_hi(wu[k].y), x3, up);
                up = fmaf(bf_lo(wu[k].z), x4, up);
                up = fmaf(bf_hi(wu[k].z), x5, up);
                up = fmaf(bf_lo(wu[k].w), x6, up);
                up = fmaf(bf_hi(wu[k].w), x7, up);
            }
            g = warp_sum(g);
            up = warp_sum(up);
            if (lane == 0) p.a[(size_t)pr * I + j] = silu_f(g) * up;
        }
    }
    if (!ok) {
        if (lane == 0) {
            report_status(p.status, ST_TIMEOUT);
            // drain copies still in flight into this warp's ring (bounded)
            for (int k = i; k < i + GU_NS && unit_of(k) < total; ++k)
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
    int rows_max;           // ceil(H / gridDim.x)
    uint32_t* status;
    uint64_t limit_ns;
};

__global__ void __launch_bounds__(DN_WARPS * 32, 1) down_decode_kernel(DownParams p) {
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = gridDim.x, c = blockIdx.x;
    const int h0 = (c * H) / G, h1 = ((c + 1) * H) / G, nrows = h1 - h0;
    const int slot_bytes = p.rows_max * I * 2;
    uint8_t* ring = smem;
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + DN_NS * slot_bytes);
    float* yacc = reinterpret_cast<float*>(bar + DN_NS);   // [T][rows_max]

    if (threadIdx.x == 0) {
#pragma unroll
        for (int s = 0; s < DN_NS; ++s) mbar_init(&bar[s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // The routing tables were complete before gateup_decode (our primary)
    // passed its own wait, so they can be read ahead of ours; the down rows
    // are immutable.  Only the activations `a` need the wait.
    const int n_slots = p.tables->n_slots;
    const int T = p.tables->T;
    auto issue = [&](int u) {
        const int s = u % DN_NS;
        const __nv_bfloat16* W = p.experts->down[p.tables->slot_expert[u]] + (size_t)h0 * I;
        mbar_arrive_expect_tx(&bar[s], nrows * I * 2);
        bulk_g2s(ring + s * slot_bytes, W, nrows * I * 2, &bar[s]);
    };
    if (threadIdx.x == 0) {
        for (int u = 0; u < DN_NS && u < n_slots; ++u) issue(u);
        for (int u = DN_NS; u < DN_NS + DN_PREFETCH && u < n_slots; ++u)
            bulk_prefetch_l2(p.experts->down[p.tables->slot_expert[u]] + (size_t)h0 * I, nrows * I * 2);
    }
    for (int k = threadIdx.x; k < T * p.rows_max; k += blockDim.x) yacc[k] = 0.f;
    pdl_wait();       // gate/up activations are complete
    pdl_trigger();
    __syncthreads();

    bool ok = true;
    int u = 0;
    for (; u < n_slots; ++u) {
        const int s = u % DN_NS;
        // the decision to give up is taken by the whole CTA
        if (!__syncthreads_and(mbar_wait_bounded(&bar[s], (u / DN_NS) & 1, p.limit_ns))) {
            ok = false;
            break;
        }
        const int pb = p.tables->slot_pair0[u], pe = p.tables->slot_pair0[u + 1];
        const uint8_t* buf = ring + s * slot_bytes;
        for (int r = warp; r < nrows; r += DN_WARPS) {
            const uint4 w0 = *reinterpret_cast<const uint4*>(buf + r * I * 2 + 16 * lane);
            const uint4 w1 = *reinterpret_cast<const uint4*>(buf + r * I * 2 + 16 * (lane + 32));
            for (int pr = pb; pr < pe; ++pr) {
                const float* ar = p.a + (size_t)pr * I;
                const float4 a0 = __ldcg(reinterpret_cast<const float4*>(ar + 8 * lane));
                const float4 a1 = __ldcg(reinterpret_cast<const float4*>(ar + 8 * lane + 4));
                const float4 a2 = __ldcg(reinterpret_cast<const float4*>(ar + 256 + 8 * lane));
                const float4 a3 = __ldcg(reinterpret_cast<const float4*>(ar + 256 + 8 * lane + 4));
                float d = 0.f;
                d = fmaf(bf_lo(w0.x), a0.x, d);
                d = fmaf(bf_hi(w0.x), a0.y, d);
                d = fmaf(bf_lo(w0.y), a0.z, d);
                d = fmaf(bf_hi(w0.y), a0.w, d);
                d = fmaf(bf_lo(w0.z), a1.x, d);
                d = fmaf(bf_hi(w0.z), a1.y, d);
                d = fmaf(bf_lo(w0.w), a1.z, d);
                d = fmaf(bf_hi(w0.w), a1.w, d);
                d = fmaf(bf_lo(w1.x), a2.x, d);
                d = fmaf(bf_hi(w1.x), a2.y, d);
                d = fmaf(bf_lo(w1.y), a2.z, d);
                d = fmaf(bf_hi(w1.y), a2.w, d);
                d = fmaf(bf_lo(w1.z), a3.x, d);
                d = fmaf(bf_hi(w1.z), a3.y, d);
                d = fmaf(bf_lo(w1.w), a3.z, d);
                d = fmaf(bf_hi(w1.w), a3.w, d);
                d = warp_sum(d);
                if (lane == 0) {
                    const int t = p.tables->pair_token[pr];
                    yacc[t * p.rows_max + r] += p.tables->pair_weight[pr] * d;
                }
            }
        }
        __syncthreads();   // every warp is done with slot s
        if (threadIdx.x == 0 && u + DN_NS < n_slots) {
            fence_proxy_async_smem();
            issue(u + DN_NS);
        }
    }
    if (!ok) {
        if (threadIdx.x == 0) {
            report_status(p.status, ST_TIMEOUT);
            for (int k = u; k < u + DN_NS && k < n_slots; ++k)
                mbar_wait_bounded(&bar[k % DN_NS], (k / DN_NS) & 1, p.limit_ns);
        }
        __syncthreads();
        return;
    }
    __syncthreads();
    for (int k = threadIdx.x; k < T * nrows; k += blockDim.x) {
        const int t = k / nrows, r = k % nrows;
        p.y[(size_t)t * H + h0 + r] = __float2bfloat16_rn(yacc[t * p.rows_max + r]);
    }
}

cudaError_t decode_set_attributes() {
    cudaError_t e = cudaFuncSetAttribute(gateup_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, GU_SMEM);
    if (e != cudaSuccess) return e;
    // down kernel: sized for the smallest plausible grid (ceil(2048/132) rows)
    const int rows_max = 16;
    const int smem = DN_NS * rows_max * I * 2 + DN_NS * 8 + DEC_T * rows_max * 4;
    return cudaFuncSetAttribute(down_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
}

cudaError_t launch_decode_experts(const LaunchCtx& L, const ExpertTables* experts, const DecodeTables* tables,
                                  const __nv_bfloat16* x, float* a_buf, __nv_bfloat16* y, int T) {
    GateUpParams gp{experts, tables, x, a_buf, L.status, L.wait_limit_ns};
    cudaError_t e = launch_pdl(L, gateup_decode_kernel, dim3(L.num_sms), dim3(GU_WARPS * 32), GU_SMEM, gp);
    if (e != cudaSuccess) return e;
    const int G = L.num_sms;
    const int rows_max = (H + G - 1) / G;
    DownParams dp{experts, tables, a_buf, y, rows_max, L.status, L.wait_limit_ns};
    const int smem = DN_NS * rows_max * I * 2 + DN_NS * 8 + T * rows_max * 4;
    return launch_pdl(L, down_decode_kernel, dim3(G), dim3(DN_WARPS * 32), smem, dp);
}

}  // namespace flint
