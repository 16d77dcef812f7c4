// routing.cuh -- device helpers shared by the router and the decode expert
// kernels: warp-wide sigmoid top-6 with renormalisation, and the per-batch
// (expert slot, token) tables of the decode path.
//
// RecursiveSI/flint (vLLM recipe page), "Overview": top-6 sigmoid routing
// over 256 experts plus an always-active shared expert.
#pragma once

#include "flint_common.cuh"

namespace flint {

// ---------------------------------------------------------------------------
// warp-wide top-6 of one token's 256 logits
// ---------------------------------------------------------------------------

// Order-preserving map of an fp32 value to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t f32_key(float v) {
    const uint32_t u = __float_as_uint(v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_f32(uint32_t k) {
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Lane l holds logits of experts l, l+32, ..., l+224.  On return every lane
// has the six chosen expert ids (decreasing logit, equal logits: lower id
// first) and their renormalised sigmoid weights.  Each round takes the warp
// maximum of the lanes' best remaining keys (one redux), then the lowest
// expert id among the lanes holding that key (a second redux).
__device__ __forceinline__ void warp_top6(const float (&v)[8], int lane, int (&sel)[TOPK], float (&wt)[TOPK]) {
    uint32_t key[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) key[i] = f32_key(v[i]);
    uint32_t taken = 0;
    float selv[TOPK];
#pragma unroll
    for (int r = 0; r < TOPK; ++r) {
        uint32_t bk = 0;
        int bi = 0x7FFFFFFF;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            // ids grow with i, so a strict comparison keeps the lower id
            if (!((taken >> i) & 1u) && key[i] > bk) {
                bk = key[i];
                bi = lane + 32 * i;
            }
        }
        const uint32_t mk = __reduce_max_sync(0xFFFFFFFFu, bk);
        const int mi = (int)__reduce_min_sync(0xFFFFFFFFu, (uint32_t)(bk == mk ? bi : 0x7FFFFFFF));
        sel[r] = mi;
        selv[r] = key_f32(mk);
        if (lane == (mi & 31)) taken |= 1u << (mi >> 5);
    }
    float s[TOPK], sum = 0.f;
#pragma unroll
    for (int r = 0; r < TOPK; ++r) {
        s[r] = sigmoid_f(selv[r]);
        sum += s[r];
    }
#pragma unroll
    for (int r = 0; r < TOPK; ++r) wt[r] = s[r] / sum;
}

// Value of a register array at a lane-dependent index without local memory.
template <typename T>
__device__ __forceinline__ T pick6(const T (&a)[TOPK], int i) {
    T r = a[0];
#pragma unroll
    for (int k = 1; k < TOPK; ++k)
        if (i == k) r = a[k];
    return r;
}

// Build the decode tables from sel_e/sel_w (token-major, T <= 32), by the
// calling warp alone.  tmask[e] collects the tokens choosing expert e as a
// bitmask, so a token's position in its expert's list (its popcount rank)
// and the slot order (increasing expert id) are the same in every CTA.
// tmask and pair0 are E-entry scratch arrays.
__device__ __forceinline__ void build_decode_tables_warp(int T, const int* sel_e, const float* sel_w,
                                                         uint32_t* tmask, int* pair0, DecodeTables* tab,
                                                         int lane) {
#pragma unroll
    for (int k = 0; k < 8; ++k) tmask[lane * 8 + k] = 0u;
    __syncwarp();
    for (int p = lane; p < T * TOPK; p += 32) atomicOr(&tmask[sel_e[p]], 1u << (p / TOPK));
    __syncwarp();
    uint32_t m[8];
    int pres = 0, sum = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        m[k] = tmask[lane * 8 + k];
        pres += m[k] != 0u;
        sum += __popc(m[k]);
    }
    int ip = pres, is = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xFFFFFFFFu, ip, o);
        const int b = __shfl_up_sync(0xFFFFFFFFu, is, o);
        if (lane >= o) {
            ip += a;
            is += b;
        }
    }
    int slot = 1 + ip - pres;   // slot 0 is the shared expert
    int pr = T + is - sum;      // pairs 0..T-1 are the shared expert's
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int e = lane * 8 + k;
        pair0[e] = pr;
        if (m[k]) {
            tab->slot_expert[slot] = e;
            tab->slot_pair0[slot] = pr;
            ++slot;
            pr += __popc(m[k]);
        }
    }
    if (lane == 31) {
        tab->n_slots = slot;
        tab->n_pairs = pr;
        tab->slot_pair0[slot] = pr;
        tab->T = T;
        tab->slot_expert[0] = SHARED;
        tab->slot_pair0[0] = 0;
    }
    for (int t = lane; t < T; t += 32) {
        tab->pair_token[t] = t;
        tab->pair_weight[t] = 1.0f;
    }
    __syncwarp();
    for (int p = lane; p < T * TOPK; p += 32) {
        const int t = p / TOPK, e = sel_e[p];
        const int q = pair0[e] + __popc(tmask[e] & ((1u << t) - 1u));
        tab->pair_token[q] = t;
        tab->pair_weight[q] = sel_w[p];
    }
    __syncwarp();
}

}  // namespace flint
