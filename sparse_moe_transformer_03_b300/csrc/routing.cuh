// routing.cuh -- device helpers shared by the router and the decode expert
// kernels: warp-wide sigmoid top-6 with renormalisation, the per-batch
// (expert slot, token) tables of the decode path, and the decode kernels'
// work-item lists.
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

// Top-6 of tokens warp, warp + 8, ..., warp + 24 (T <= 32, eight warps):
// every one of the warp's tokens has its logits requested before the first
// selection.  idx_out / w_out (global, or null) receive the choices too.
__device__ __forceinline__ void select_tokens_warps(const float* logits, int T, int warp, int lane, int* sel_e,
                                                    float* sel_w, int32_t* idx_out, float* w_out) {
    float v[4][8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int t = warp + 8 * q;
#pragma unroll
        for (int k = 0; k < 8; ++k) v[q][k] = t < T ? __ldcg(logits + (size_t)t * E + lane + 32 * k) : 0.f;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const int t = warp + 8 * q;
        if (t < T) {
            int sel[TOPK];
            float wt[TOPK];
            warp_top6(v[q], lane, sel, wt);
            if (lane < TOPK) {
                const int se = pick6(sel, lane);
                const float sw = pick6(wt, lane);
                sel_e[t * TOPK + lane] = se;
                sel_w[t * TOPK + lane] = sw;
                if (idx_out) {
                    idx_out[t * TOPK + lane] = se;
                    w_out[t * TOPK + lane] = sw;
                }
            }
        }
    }
}

// Build the decode tables from sel_e/sel_w (token-major, T <= 32), by the
// calling warp alone.  tmask[e] collects the tokens choosing expert e as a
// bitmask, so a token's position in its expert's list (its popcount rank)
// and the slot order (increasing expert id) are the same in every CTA.  One
// warp scan gives each slot its first pair and its first 8-token tile.
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
    int pres = 0, sum = 0, tiles = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        m[k] = tmask[lane * 8 + k];
        pres += m[k] != 0u;
        sum += __popc(m[k]);
        tiles += (__popc(m[k]) + 7) >> 3;
    }
    int ip = pres, is = sum, it = tiles;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xFFFFFFFFu, ip, o);
        const int b = __shfl_up_sync(0xFFFFFFFFu, is, o);
        const int c = __shfl_up_sync(0xFFFFFFFFu, it, o);
        if (lane >= o) {
            ip += a;
            is += b;
            it += c;
        }
    }
    int slot = 1 + ip - pres;               // slot 0 is the shared expert
    int pr = T + is - sum;                  // pairs 0..T-1 are the shared expert's
    int tile = ((T + 7) >> 3) + it - tiles; // and its ceil(T / 8) tiles come first
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int e = lane * 8 + k;
        pair0[e] = pr;
        if (m[k]) {
            tab->slot_expert[slot] = e;
            tab->slot_pair0[slot] = pr;
            tab->slot_tile0[slot] = tile;
            ++slot;
            pr += __popc(m[k]);
            tile += (__popc(m[k]) + 7) >> 3;
        }
    }
    if (lane == 31) {
        tab->n_slots = slot;
        tab->n_pairs = pr;
        tab->slot_pair0[slot] = pr;
        tab->slot_tile0[slot] = tile;
        tab->T = T;
        tab->slot_expert[0] = SHARED;
        tab->slot_pair0[0] = 0;
        tab->slot_tile0[0] = 0;
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

// ---------------------------------------------------------------------------
// work items of the decode expert kernels
// ---------------------------------------------------------------------------

// Gate/up items: (slot u, unit r of the slot's DEC_UNITS, tile nt of 8 of
// the slot's tokens), packed u << 8 | r << 2 | nt; in slot order, units in
// order within a slot, tiles in order within a unit: slot u's items start at
// DEC_UNITS x slot_tile0[u].  Item j of the grid goes to CTA j % G.
constexpr int DEC_UNITS = 64;              // 8 gate + 8 up rows per unit, I = 512
constexpr int DEC_MAX_CTA_ITEMS = 256;     // per CTA
constexpr int DEC_MIN_GRID = 72;           // the gate/up grids have at least this many CTAs
static_assert(DEC_UNITS * 4 <= 256, "unit and tile fit in the low byte");
// Most 8-token tiles a batch can have: ceil(T / 8) for the shared slot, and
// for U routed slots holding 6T pairs in all, sum ceil(n_u / 8) <= (6T + 7U) / 8
// with U <= min(E, 6T).  The item list of every CTA then fits its buffer.
constexpr int DEC_MAX_ROUTED = DEC_T * TOPK < E ? DEC_T * TOPK : E;
constexpr int DEC_MAX_TILES = (DEC_T + 7) / 8 + (DEC_T * TOPK + 7 * DEC_MAX_ROUTED) / 8;
static_assert((DEC_UNITS * DEC_MAX_TILES + DEC_MIN_GRID - 1) / DEC_MIN_GRID <= DEC_MAX_CTA_ITEMS,
              "a CTA's gate/up item list fits its buffer at the smallest grid");

// CTA c's items c, c + G, ... into list[] (all threads of the CTA take part;
// the caller synchronises before reading list).  Returns their count, or -1
// when it exceeds DEC_MAX_CTA_ITEMS (the list is then left empty; with G >=
// DEC_MIN_GRID the static_assert above rules this out).
__device__ __forceinline__ int list_gateup_items(const DecodeTables* tab, int c, int G, int* list) {
    const int n_slots = tab->n_slots, total = DEC_UNITS * tab->slot_tile0[n_slots];
    const int my_items = c < total ? (total - c + G - 1) / G : 0;
    if (my_items > DEC_MAX_CTA_ITEMS) return -1;
    for (int i = threadIdx.x; i < my_items; i += blockDim.x) {
        const int j = c + G * i;
        int lo = 0, hi = n_slots - 1;     // the last slot u with DEC_UNITS * slot_tile0[u] <= j
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (DEC_UNITS * tab->slot_tile0[mid] <= j) lo = mid;
            else hi = mid - 1;
        }
        const int l = j - DEC_UNITS * tab->slot_tile0[lo];
        const int ntu = tab->slot_tile0[lo + 1] - tab->slot_tile0[lo];
        list[i] = (lo << 8) | ((l / ntu) << 2) | (l % ntu);
    }
    return my_items;
}

// Down items: (slot u, column half, tile nt of 8 tokens), packed u << 3 |
// half << 2 | nt; in slot order, each slot's first half before its second
// and the tiles in order within a half: slot u's items start at 2 x
// slot_tile0[u].  At most 2 x (slots + pairs / 8).
constexpr int DEC_MAX_DOWN_ITEMS = 2 * (NEXP + DEC_PAIRS / 8);

// Fills items[] from the tables and returns the count.  One warp.
__device__ __forceinline__ int build_down_items_warp(const DecodeTables* tab, int* items, int lane) {
    const int n_slots = tab->n_slots;
    for (int u = lane; u < n_slots; u += 32) {
        const int t0 = tab->slot_tile0[u], nt = tab->slot_tile0[u + 1] - t0;
        for (int hk = 0; hk < 2; ++hk)
            for (int t = 0; t < nt; ++t) items[2 * t0 + hk * nt + t] = (u << 3) | (hk << 2) | t;
    }
    __syncwarp();
    return 2 * tab->slot_tile0[n_slots];
}

}  // namespace flint
