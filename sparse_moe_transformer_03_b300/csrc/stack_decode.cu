// stack_decode.cu -- cross-layer persistent decode: every layer of a stack
// of MoE layers in ONE kernel launch, for T <= 8 tokens (bf16 experts).
//
// Layer definition: RecursiveSI/flint (vLLM recipe page), "Overview" (256
// experts, top-6 sigmoid routing plus a shared expert).  The recipe page also
// names a low-latency decode path for a handful of requests, and the
// mrchatgpt.org article (section 4) a decode megakernel; this kernel is this
// library's design of that idea for B300.
//
// Why: at decode sizes a layer moves (U + 1) x 6 MiB of expert weights (U =
// distinct routed experts) and little else, so it should run at HBM speed.
// Three kernels per layer leave HBM idle while one kernel drains and the next
// starts, and every launch re-derives the routing.  Here one resident grid
// (one CTA per SM) walks the layers.  Per layer:
//
//   1. x (T rows) -> shared memory; each CTA dots its one or two router rows
//      (prefetched during the previous layer) with every token and publishes
//      the fp32 logits as 64-bit words tagged with the layer's epoch, so the
//      other CTAs read them as soon as they land (no barrier);
//   2. meanwhile the shared expert's gate/up unit of the CTA (prefetched too)
//      is multiplied; every CTA then waits for the 256 tagged logits of each
//      token, takes the top-6 (warp_top6) and builds the (slot, token) tables;
//   3. a producer warp streams the CTA's routed gate/up units and then its
//      down row groups into a ring of 8 KiB slots by cp.async.bulk; eight
//      consumer warps multiply them on the warp-level tensor core
//      (mma.sync m16n8k16, tokens as the M rows, weight rows as the 8 N
//      columns) and write a = silu(g) * u (bf16) to a global buffer;
//   4. grid barrier; the CTA copies every pair's activations into shared
//      memory and applies its down row groups (8 output rows x all slots,
//      the routing weight folded in per token, slots summed in order):
//      y is written once, deterministically;
//   5. grid barrier (layer l + 1 may read y_l), while the producer already
//      streams layer l + 1's router rows and shared-expert unit.
//
// Work split: a gate/up unit is 4 gate rows + the 4 matching up rows x 2048
// columns (32 KiB); an expert has 128.  CTA c owns shared unit c (c < 128)
// and a contiguous range of the routed units chosen so every CTA gets the
// same number of units.  A down row group is 8 rows of Wd x 512 columns
// (8 KiB per slot); CTA c owns row groups c and c + G.  Every output element
// is produced by one CTA, so nothing is reduced across CTAs.  The ring is
// deep (about 200 KiB at T = 1): a CTA requests most of its bytes at once
// and the GPU-wide HBM bandwidth, not the per-CTA split, sets the pace.
#include "flint_common.cuh"
#include "../../include/flint_moe.h"
#include "flint_internal.h"
#include "mma_sync.cuh"
#include "routing.cuh"
#include "tc_ptx.cuh"

#include <cstddef>

namespace flint {

namespace {

constexpr int SK_CW = 8;                          // consumer warps
constexpr int SK_THREADS = (SK_CW + 1) * 32;      // + one producer warp
constexpr int SK_SLOT = 8192;                     // ring slot bytes
constexpr int SK_GU_UNITS = I / 4;                // 128 gate/up units per expert
constexpr int SK_RG = H / 8;                      // 256 down row groups per expert
constexpr int SK_GU_TILES = (2 * I / 128) * (H / 64);  // 256 gate/up tiles of an expert precede its down tiles
constexpr int SK_XSTRIDE = H * 2 + 16;            // padded x row in shared memory
constexpr int SK_MAX_SLOTS = 1 + STACK_MAX_T * TOPK;   // 49
constexpr int SK_NAMED = 1;                       // named barrier of the consumer warps

// Activation rows: pair p's 512 bf16, its 16-byte chunk c stored at c ^ (p % 8)
// (the tokens of one MMA read eight rows through different banks).
__host__ __device__ __forceinline__ int sk_act_index(int p, int j) {
    return p * I + ((((j >> 3) ^ (p & 7))) << 3) + (j & 7);
}

struct SkShared {
    DecodeTables tab;                             // n_slots, n_pairs, slot_expert, slot_pair0 are used
    int slot_of[E];                               // slot of each routed expert of the batch
    float bias[STACK_MAX_LAYERS][2];              // router bias of this CTA's experts, every layer
    int sel_e[STACK_MAX_T * TOPK];
    float sel_w[STACK_MAX_T * TOPK];
    uint32_t tmask[E];
    int pair0[E];
    int tok_pair[SK_MAX_SLOTS][STACK_MAX_T];      // pair of (slot, token), -1: token not routed there
    float tok_w[SK_MAX_SLOTS][STACK_MAX_T];       // its routing weight (0 when not routed)
    alignas(16) float part[SK_CW][128];           // per-warp partial sums (shared unit: [lane][4], read
                                                  // as float4; down: [row group][token][row])
    uint64_t route_bar;                           // consumers -> producer: tables of the layer are built
    // Ring slot i was last handed out for sequence number slot_seq[i] - 1.  A
    // consumer waits for its sequence number here before the slot's full
    // barrier: several warps consume the ring, so one may reach use u of a
    // slot before use u - 1 has landed, and a parity wait for phase u would
    // then succeed on phase u - 1.
    uint32_t slot_seq[32];
    int abort;
};

static_assert(offsetof(SkShared, part) % 16 == 0, "float4 access to the partial sums");
static_assert(offsetof(SkShared, route_bar) % 8 == 0, "mbarrier alignment");

// 128 x 64 tile-copy offsets (repack.cu layout): in-tile row r, 16-byte chunk c
__device__ __forceinline__ uint32_t sw_chunk(int r, int c) { return (uint32_t)(((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Shared memory of a launch: the ring, then the x / activation buffer, the
// ring's full and empty barriers and the tables.
struct SkLayout {
    int nslot;
    uint32_t ubuf_off, bars_off, sh_off, total;
};

__host__ __device__ __forceinline__ uint32_t sk_ubuf_bytes(int T) {
    const uint32_t xb = (uint32_t)T * SK_XSTRIDE, ab = (uint32_t)(T * (TOPK + 1)) * I * 2;
    return ((xb > ab ? xb : ab) + 127u) & ~127u;
}

__host__ __device__ __forceinline__ SkLayout sk_layout(int T, uint32_t max_smem) {
    SkLayout L;
    const uint32_t fixed = sk_ubuf_bytes(T) + (uint32_t)((sizeof(SkShared) + 127) & ~size_t(127));
    int ns = (int)((max_smem - fixed - 64 * 16) / (SK_SLOT + 16));
    if (ns > 32) ns = 32;
    L.nslot = ns;
    L.ubuf_off = (uint32_t)ns * SK_SLOT;
    L.bars_off = L.ubuf_off + sk_ubuf_bytes(T);
    L.sh_off = L.bars_off + (uint32_t)(((2 * ns * 8) + 127) & ~127);
    L.total = L.sh_off + (uint32_t)((sizeof(SkShared) + 127) & ~size_t(127));
    return L;
}

struct SkState {
    const StackParams* p;
    uint8_t* ring;
    uint8_t* ubuf;
    uint64_t* full;
    uint64_t* empty;
    SkShared* sh;
    int nslot, T, c, G;
};

__device__ __forceinline__ void sk_fail(const SkState& s) {
    s.sh->abort = 1;
    atomicExch(s.p->abort_flag, 1u);
    report_status(s.p->status, ST_TIMEOUT);
}

__device__ __forceinline__ bool sk_aborted(const SkState& s) {
    return *reinterpret_cast<volatile int*>(&s.sh->abort) != 0;
}

// Bounded mbarrier wait that gives up early once the CTA is aborting.
__device__ __forceinline__ bool sk_wait(const SkState& s, uint64_t* bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (sk_aborted(s)) return false;
        if (globaltimer_ns() - t0 > s.p->limit_ns) {
            sk_fail(s);
            return false;
        }
    }
}

__device__ __forceinline__ void st_release_shared(uint32_t* p, uint32_t v) {
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_shared(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
    return v;
}

// Wait until ring sequence number q has landed in its slot: first until the
// producer has handed the slot out for q (so the slot's full barrier is at
// q's phase or past it), then on the full barrier.
__device__ __forceinline__ bool sk_wait_full(const SkState& s, uint32_t q) {
    const int slot = (int)(q % (uint32_t)s.nslot);
    const uint32_t* ss = &s.sh->slot_seq[slot];
    if (ld_acquire_shared(ss) != q + 1u) {
        const uint64_t t0 = globaltimer_ns();
        for (;;) {
#pragma unroll 1
            for (int i = 0; i < 64; ++i)
                if (ld_acquire_shared(ss) == q + 1u) goto issued;
            if (sk_aborted(s)) return false;
            if (globaltimer_ns() - t0 > s.p->limit_ns) {
                sk_fail(s);
                return false;
            }
        }
    }
issued:
    return sk_wait(s, &s.full[slot], (q / (uint32_t)s.nslot) & 1);
}

// Grid barrier (one thread, after the consumer warps synchronised): arrive,
// then wait until every CTA of the grid has arrived `target` - base times.
__device__ bool sk_grid_barrier(const SkState& s, unsigned long long target) {
    __threadfence();
    atomicAdd(s.p->bar, 1ull);
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (ld_acquire_u64(s.p->bar) >= target) return true;
        if (*reinterpret_cast<volatile uint32_t*>(s.p->abort_flag)) {
            s.sh->abort = 1;
            return false;
        }
        if (globaltimer_ns() - t0 > s.p->limit_ns) {
            sk_fail(s);
            return false;
        }
    }
}

// ---- per-CTA work of a layer (identical formulas in producer and consumers) ----

__device__ __forceinline__ int sk_router_rows(int c, int G) { return (c < E ? 1 : 0) + (c + G < E ? 1 : 0); }
__device__ __forceinline__ int sk_has_sg(int c) { return c < SK_GU_UNITS ? 1 : 0; }
__device__ __forceinline__ int sk_n_rg(int c, int G) { return (c < SK_RG ? 1 : 0) + (c + G < SK_RG ? 1 : 0); }
__device__ __forceinline__ int sk_rg(int c, int G, int i) { return c + i * G; }

// End of CTA c's range of routed gate/up units (units of slot 1.. in order):
// the cumulative share of all (U + 1) x 128 units minus the shared units the
// CTAs up to c own.
__device__ __forceinline__ int sk_rcum(int c, int G, int U) {
    if (c < 0) return 0;
    const int ntot = SK_GU_UNITS * (U + 1);
    const int tcum = (int)(((long long)(c + 1) * ntot) / G);
    const int scum = c + 1 < SK_GU_UNITS ? c + 1 : SK_GU_UNITS;
    const int r = tcum - scum;
    return r < 0 ? 0 : r;
}

// Slots and pairs of a batch of T <= 8 tokens from their top-6 (one warp):
// slot 0 is the shared expert (pair t = token t), then the routed experts by
// increasing id, each with its tokens in increasing order.  tok_pair[u][t] /
// tok_w[u][t]: the pair and routing weight of token t in slot u (-1 / 0 when
// t is not routed there).  Every lane works on its own experts and pairs.
__device__ void sk_build_tables(int T, SkShared* sh, int lane) {
    DecodeTables* tab = &sh->tab;
#pragma unroll
    for (int k = 0; k < 8; ++k) sh->tmask[lane * 8 + k] = 0u;
    __syncwarp();
    for (int p = lane; p < T * TOPK; p += 32) atomicOr(&sh->tmask[sh->sel_e[p]], 1u << (p / TOPK));
    __syncwarp();
    uint32_t m[8];
    int pres = 0, sum = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        m[k] = sh->tmask[lane * 8 + k];
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
    int slot = 1 + ip - pres, pr = T + is - sum;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int e = lane * 8 + k;
        sh->pair0[e] = pr;
        if (m[k]) {
            tab->slot_expert[slot] = e;
            tab->slot_pair0[slot] = pr;
            sh->slot_of[e] = slot;
            ++slot;
            pr += __popc(m[k]);
        }
    }
    const int ns = __shfl_sync(0xFFFFFFFFu, slot, 31);
    if (lane == 31) {
        tab->n_slots = slot;
        tab->n_pairs = pr;
        tab->slot_pair0[slot] = pr;
        tab->T = T;
        tab->slot_expert[0] = SHARED;
        tab->slot_pair0[0] = 0;
    }
    for (int i = lane; i < ns * STACK_MAX_T; i += 32) {
        sh->tok_pair[i / STACK_MAX_T][i % STACK_MAX_T] = -1;
        sh->tok_w[i / STACK_MAX_T][i % STACK_MAX_T] = 0.f;
    }
    __syncwarp();
    if (lane < T) {
        sh->tok_pair[0][lane] = lane;
        sh->tok_w[0][lane] = 1.f;
    }
    for (int p = lane; p < T * TOPK; p += 32) {
        const int t = p / TOPK, e = sh->sel_e[p], u = sh->slot_of[e];
        sh->tok_pair[u][t] = sh->pair0[e] + __popc(sh->tmask[e] & ((1u << t) - 1u));
        sh->tok_w[u][t] = sh->sel_w[p];
    }
    __syncwarp();
}

// ---------------------------------------------------------------------------
// producer
// ---------------------------------------------------------------------------

struct SkProducer {
    uint32_t seq = 0;   // ring slots handed out so far

    // Take the next slot for a copy of `bytes`; lane 0 only.
    __device__ __forceinline__ bool take(const SkState& s, uint32_t bytes, uint8_t** dst, uint64_t** bar) {
        const int slot = (int)(seq % (uint32_t)s.nslot);
        const uint32_t use = seq / (uint32_t)s.nslot;
        if (use > 0 && !sk_wait(s, &s.empty[slot], (use - 1) & 1)) return false;
        mbar_arrive_expect_tx(&s.full[slot], bytes);
        st_release_shared(&s.sh->slot_seq[slot], seq + 1u);
        *dst = s.ring + (size_t)slot * SK_SLOT;
        *bar = &s.full[slot];
        ++seq;
        return true;
    }
};

// Router rows of CTA c for layer l (one slot, plain bulk copies).  Lane 0 only.
__device__ __forceinline__ bool sk_issue_router(const SkState& s, SkProducer& pr, int l) {
    const int nr = sk_router_rows(s.c, s.G);
    if (nr == 0) return true;
    uint8_t* dst = nullptr;
    uint64_t* bar = nullptr;
    if (!pr.take(s, (uint32_t)nr * H * 2, &dst, &bar)) return false;
    for (int i = 0; i < nr; ++i)
        bulk_g2s(dst + i * H * 2, s.p->layer[l].router + (size_t)(s.c + i * s.G) * H, H * 2, bar);
    return true;
}

// One gate/up unit (4 slots, one 8 KiB tensor box each): gate rows 4q ..
// 4q + 3 over column tiles 0..15 and 16..31, then the matching up rows.
// Lane 0 only.
__device__ __forceinline__ bool sk_issue_gateup(const SkState& s, SkProducer& pr, const CUtensorMap* maps,
                                                int expert, int q) {
    const int r0 = 4 * q, rb = r0 >> 7;
    for (int k = 0; k < 4; ++k) {
        uint8_t* dst = nullptr;
        uint64_t* bar = nullptr;
        if (!pr.take(s, SK_SLOT, &dst, &bar)) return false;
        const int tile = ((k >> 1) * 4 + rb) * (H / 64) + (k & 1) * 16;   // up rows: row blocks 4..7
        tc::tma_load_4d(dst, &maps[0], 0, (r0 & 127) >> 2, tile, expert, bar);
    }
    return true;
}

// One down row group of one expert (one slot, one 8 KiB box: 8 rows x the 8
// column tiles of K = 512).  Lane 0 only.
__device__ __forceinline__ bool sk_issue_down(const SkState& s, SkProducer& pr, const CUtensorMap* maps, int expert,
                                              int rg) {
    uint8_t* dst = nullptr;
    uint64_t* bar = nullptr;
    if (!pr.take(s, SK_SLOT, &dst, &bar)) return false;
    tc::tma_load_4d(dst, &maps[1], 0, (rg & 15) * 2, SK_GU_TILES + (rg >> 4) * (I / 64), expert, bar);
    return true;
}

__device__ void sk_producer(const SkState& s, int lane) {
    if (lane != 0) return;
    SkProducer pr;
    const StackParams& p = *s.p;
    bool ok = sk_issue_router(s, pr, 0);
    if (ok && sk_has_sg(s.c)) ok = sk_issue_gateup(s, pr, p.layer[0].maps, SHARED, s.c);
    for (int l = 0; ok && l < p.n_layers; ++l) {
        // the consumers publish the layer's tables
        if (!sk_wait(s, &s.sh->route_bar, l & 1)) break;
        const DecodeTables& tab = s.sh->tab;
        const int U = tab.n_slots - 1;
        const CUtensorMap* maps = p.layer[l].maps;
        const int k0 = sk_rcum(s.c - 1, s.G, U), k1 = sk_rcum(s.c, s.G, U);
        for (int k = k0; ok && k < k1; ++k)
            ok = sk_issue_gateup(s, pr, maps, tab.slot_expert[1 + k / SK_GU_UNITS], k % SK_GU_UNITS);
        const int nrg = sk_n_rg(s.c, s.G);
        for (int u = 0; ok && u <= U; ++u)
            for (int i = 0; ok && i < nrg; ++i) ok = sk_issue_down(s, pr, maps, tab.slot_expert[u], sk_rg(s.c, s.G, i));
        if (ok && l + 1 < p.n_layers) {
            ok = sk_issue_router(s, pr, l + 1);
            if (ok && sk_has_sg(s.c)) ok = sk_issue_gateup(s, pr, p.layer[l + 1].maps, SHARED, s.c);
        }
    }
    // copies still in flight (only after an abort): wait for them before exiting
    // (a slot whose copies were never issued does not complete: short limit)
    if (sk_aborted(s)) {
        const uint32_t first = pr.seq > (uint32_t)s.nslot ? pr.seq - (uint32_t)s.nslot : 0u;
        for (uint32_t q = first; q < pr.seq; ++q)
            mbar_wait_bounded(&s.full[q % s.nslot], (q / s.nslot) & 1, 10000000ull);
    }
}

// ---------------------------------------------------------------------------
// consumers
// ---------------------------------------------------------------------------

// Gate/up unit q of slot u on the ring slots starting at sequence number sq
// (gate rows over column tiles 0..15, 16..31, then the up rows likewise),
// column tiles [kt0, kt1) only (the shared unit is split over the warps).
// acc receives D[token][n] for weight rows n = (gate r, up r) interleaved.
__device__ __forceinline__ bool sk_gateup_mma(const SkState& s, uint32_t sq, int q, int kt0, int kt1, int lane,
                                              float (&acc)[4]) {
    const int m = lane >> 3, r = lane & 7;
    // A (x rows by token): row r + 8 (m & 1), 16-byte chunk (m >> 1) of the k-step
    const int ta = r + 8 * (m & 1);
    const uint8_t* xa = s.ubuf + (size_t)(ta < s.T ? ta : 0) * SK_XSTRIDE + (m >> 1) * 16;
    // B (weight rows): n = r: gate row 4q + r / 2 (r even) or the up row (r odd)
    const int rr = (4 * q + (r >> 1)) & 127;
    const uint32_t boff = (uint32_t)((r >> 1) * 128);
    float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
    int waited = -1;
    const uint8_t* bslot = nullptr;
    for (int kt = kt0; kt < kt1; ++kt) {
        const int half = kt >> 4;
        if (half != waited) {
            const bool got = sk_wait_full(s, sq + (uint32_t)half) && sk_wait_full(s, sq + 2u + (uint32_t)half);
            if (!__all_sync(0xFFFFFFFFu, got)) return false;
            waited = half;
            bslot = s.ring + (size_t)((sq + (uint32_t)(2 * (r & 1) + half)) % s.nslot) * SK_SLOT + boff;
        }
        const uint8_t* piece = bslot + (kt & 15) * 512;
#pragma unroll
        for (int h = 0; h < 2; ++h) {     // two 32-column halves of the 64-column tile
            uint32_t b[4], a[4], a2[4];
            ldmatrix_x4(b, piece + sw_chunk(rr, 4 * h + m));
            const int k0 = kt * 64 + 32 * h;
            ldmatrix_x4(a, xa + (size_t)k0 * 2);
            ldmatrix_x4(a2, xa + (size_t)(k0 + 16) * 2);
            mma_bf16_16816(a0, a, b[0], b[1]);
            mma_bf16_16816(a1, a2, b[2], b[3]);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[i] = a0[i] + a1[i];
    return true;
}

// a = silu(g) * u of unit q of slot u for the tokens routed to it.
__device__ __forceinline__ void sk_store_act(const SkState& s, int u, int q, int lane, const float (&d)[4]) {
    const int g = lane >> 2, cq = lane & 3;
    if (g < s.T) {
        const int pp = s.sh->tok_pair[u][g];
        if (pp >= 0) s.p->act[sk_act_index(pp, 4 * q + cq)] = __float2bfloat16_rn(silu_f(d[0]) * d[1]);
    }
}

// End of a phase of the consumer warps: a named barrier that also ORs every
// consumer thread's failure flag (and the CTA's abort flag as each thread
// sees it), so all 256 threads take the same branch afterwards.
__device__ __forceinline__ bool sk_phase_end(const SkState& s, bool fail) {
    const uint32_t v = (fail || sk_aborted(s)) ? 1u : 0u;
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(v), "n"(SK_NAMED), "n"(SK_CW * 32)
        : "memory");
    if (r) s.sh->abort = 1;
    return r != 0;
}

__device__ void sk_consumers(const SkState& s, int warp, int lane) {
    const StackParams& p = *s.p;
    const int T = s.T, c = s.c, G = s.G, tid = warp * 32 + lane;
    SkShared* sh = s.sh;
    // router bias of this CTA's experts for every layer (weights: read before
    // the dependency wait)
    for (int i = tid; i < p.n_layers * 2; i += SK_CW * 32) {
        const int l = i >> 1, e = c + (i & 1) * G;
        sh->bias[l][i & 1] = (e < E && p.layer[l].bias) ? __ldg(p.layer[l].bias + e) : 0.f;
    }
    pdl_wait();
    // the barrier counter's value at the launch, rounded down to the grid: every
    // CTA reads it before its own first arrival, when fewer than G have arrived
    unsigned long long base = 0;
    if (lane == 0) base = ld_acquire_u64(p.bar);
    base = __shfl_sync(0xFFFFFFFFu, base, 0);
    base = base / (unsigned long long)G * (unsigned long long)G;
    int nbar = 0;
    uint32_t seq = 0;
    const int m = lane >> 3, r = lane & 7;
    const int g = lane >> 2, cq = lane & 3;
    for (int l = 0; l < p.n_layers; ++l) {
        const StackLayerArgs& Ly = p.layer[l];
        const unsigned int tag = (unsigned int)(base / (unsigned long long)G) + (unsigned int)l + 1u;
        bool fail = false;
        // ---- 1. x rows into shared memory (16-byte loads through L2) ----
        for (int i = tid; i < T * (H / 8); i += SK_CW * 32) {
            const int t = i / (H / 8), k = i % (H / 8);
            const uint4 v = __ldcg(reinterpret_cast<const uint4*>(Ly.x + (size_t)t * H) + k);
            *reinterpret_cast<uint4*>(s.ubuf + (size_t)t * SK_XSTRIDE + k * 16) = v;
        }
        if (sk_phase_end(s, false)) break;
        // ---- 2. this CTA's router rows: tagged fp32 logits (bias included) ----
        const int nr = sk_router_rows(c, G);
        const uint32_t seqR = seq;
        seq += nr ? 1 : 0;
        if (nr) {
            fail = !__all_sync(0xFFFFFFFFu, sk_wait_full(s, seqR));
            const uint8_t* rows = s.ring + (size_t)(seqR % s.nslot) * SK_SLOT;
            for (int pi = warp; !fail && pi < nr * T; pi += SK_CW) {
                const int i = pi / T, t = pi % T, e = c + i * G;
                const uint4* wr = reinterpret_cast<const uint4*>(rows + i * H * 2);
                const uint4* xr = reinterpret_cast<const uint4*>(s.ubuf + (size_t)t * SK_XSTRIDE);
                float acc = 0.f;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint4 w = wr[lane + 32 * k], xv = xr[lane + 32 * k];
                    acc = fmaf(bf_lo(w.x), bf_lo(xv.x), acc);
                    acc = fmaf(bf_hi(w.x), bf_hi(xv.x), acc);
                    acc = fmaf(bf_lo(w.y), bf_lo(xv.y), acc);
                    acc = fmaf(bf_hi(w.y), bf_hi(xv.y), acc);
                    acc = fmaf(bf_lo(w.z), bf_lo(xv.z), acc);
                    acc = fmaf(bf_hi(w.z), bf_hi(xv.z), acc);
                    acc = fmaf(bf_lo(w.w), bf_lo(xv.w), acc);
                    acc = fmaf(bf_hi(w.w), bf_hi(xv.w), acc);
                }
                acc = warp_sum(acc);
                if (lane == 0) {
                    const float v = acc + sh->bias[l][i];
                    st_relaxed_u64(p.logits + (size_t)t * E + e,
                                   ((unsigned long long)tag << 32) | (unsigned long long)__float_as_uint(v));
                }
            }
            if (sk_phase_end(s, fail)) break;
            if (tid == 0) mbar_arrive(&s.empty[seqR % s.nslot]);
        }
        // ---- 3. the shared expert's unit of this CTA, its columns split over the warps ----
        const int has_sg = sk_has_sg(c);
        const uint32_t seqSG = seq;
        seq += has_sg ? 4 : 0;
        if (has_sg) {
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            fail = !__all_sync(0xFFFFFFFFu, sk_gateup_mma(s, seqSG, c, 4 * warp, 4 * warp + 4, lane, d));
            *reinterpret_cast<float4*>(&sh->part[warp][lane * 4]) = make_float4(d[0], d[1], d[2], d[3]);
            if (sk_phase_end(s, fail)) break;
            if (warp == 0) {
                float4 sum = *reinterpret_cast<const float4*>(&sh->part[0][lane * 4]);
                for (int w = 1; w < SK_CW; ++w) {
                    const float4 v = *reinterpret_cast<const float4*>(&sh->part[w][lane * 4]);
                    sum.x += v.x;
                    sum.y += v.y;
                    sum.z += v.z;
                    sum.w += v.w;
                }
                if (g < T)   // the shared slot holds every token: pair = token
                    p.act[sk_act_index(g, 4 * c + cq)] = __float2bfloat16_rn(silu_f(sum.x) * sum.y);
                if (lane < 4) mbar_arrive(&s.empty[(seqSG + lane) % s.nslot]);
            }
        }
        // ---- 4. every token's 256 logits (tagged with this layer's epoch), top-6 ----
        if (warp < T) {
            float v[8];
            const unsigned long long* lg = p.logits + (size_t)warp * E + lane;
            const uint64_t t0 = globaltimer_ns();
            bool got = false;
            for (;;) {
                bool mine = true;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const unsigned long long w = ld_relaxed_u64(lg + 32 * k);
                    mine = mine && (unsigned int)(w >> 32) == tag;
                    v[k] = __uint_as_float((unsigned int)w);
                }
                if (__all_sync(0xFFFFFFFFu, mine)) {
                    got = true;
                    break;
                }
                // warp-uniform decisions: every lane leaves the loop together
                if (__any_sync(0xFFFFFFFFu, sk_aborted(s) || *reinterpret_cast<volatile uint32_t*>(p.abort_flag)))
                    break;
                if (__any_sync(0xFFFFFFFFu, globaltimer_ns() - t0 > p.limit_ns)) {
                    if (lane == 0) sk_fail(s);
                    break;
                }
            }
            fail = !got;
            if (got) {
                int sel[TOPK];
                float wt[TOPK];
                warp_top6(v, lane, sel, wt);
                if (lane < TOPK) {
                    sh->sel_e[warp * TOPK + lane] = pick6(sel, lane);
                    sh->sel_w[warp * TOPK + lane] = pick6(wt, lane);
                }
            }
        }
        if (sk_phase_end(s, fail)) break;
        // ---- 5. tables: slots (shared first, then the routed experts by id), pairs ----
        if (warp == 0) {
            sk_build_tables(T, sh, lane);
            if (lane == 0) mbar_arrive(&sh->route_bar);
        }
        if (sk_phase_end(s, false)) break;
        const int U = sh->tab.n_slots - 1;
        // ---- 6. routed gate/up units: unit j of the CTA's range goes to warp j % 8 ----
        const int k0 = sk_rcum(c - 1, G, U), k1 = sk_rcum(c, G, U);
        const uint32_t seqRG = seq;
        seq += 4u * (uint32_t)(k1 - k0);
        for (int j = warp; j < k1 - k0 && !fail; j += SK_CW) {
            const int k = k0 + j, u = 1 + k / SK_GU_UNITS, q = k % SK_GU_UNITS;
            float d[4];
            if (!__all_sync(0xFFFFFFFFu, sk_gateup_mma(s, seqRG + 4u * j, q, 0, H / 64, lane, d))) {
                fail = true;
                break;
            }
            __syncwarp();
            if (lane < 4) mbar_arrive(&s.empty[(seqRG + 4u * j + lane) % s.nslot]);
            sk_store_act(s, u, q, lane, d);
        }
        // ---- 7. every CTA's activations are written (grid barrier) ----
        if (sk_phase_end(s, fail)) break;
        if (tid == 0) {
            ++nbar;
            if (!sk_grid_barrier(s, base + (unsigned long long)nbar * G)) sh->abort = 1;
        }
        if (sk_phase_end(s, false)) break;
        // ---- 8. all pairs' activations into shared memory (x is no longer read) ----
        const int npairs = sh->tab.n_pairs;
        for (int i = tid; i < npairs * (I / 8); i += SK_CW * 32)
            *reinterpret_cast<uint4*>(s.ubuf + (size_t)i * 16) = __ldcg(reinterpret_cast<const uint4*>(p.act) + i);
        if (sk_phase_end(s, false)) break;
        // ---- 9. down row groups: item (slot u, row group i) -> warp (u * nrg + i) % 8 ----
        const int nrg = sk_n_rg(c, G);
        const uint32_t seqD = seq;
        const int nd = nrg * (U + 1);
        seq += (uint32_t)nd;
        float yacc[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
        for (int it = warp; it < nd && !fail; it += SK_CW) {
            const int u = it / nrg, ri = it % nrg;
            const uint32_t qq = seqD + (uint32_t)it;
            if (!__all_sync(0xFFFFFFFFu, sk_wait_full(s, qq))) {
                fail = true;
                break;
            }
            const uint8_t* wd = s.ring + (size_t)(qq % s.nslot) * SK_SLOT + r * 128;
            // A row: token r (rows 8..15 repeat it; they are never used) -> its pair in slot u
            int pa = r < T ? sh->tok_pair[u][r] : -1;
            pa = pa < 0 ? 0 : pa;
            const uint8_t* ar = s.ubuf + (size_t)pa * (I * 2);
            float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
            for (int kk = 0; kk < I / 32; ++kk) {     // two k-steps of 16 per iteration
                uint32_t b[4], a[4], a2[4];
                const int kt = kk >> 1, h = kk & 1;
                ldmatrix_x4(b, wd + kt * 1024 + sw_chunk(r, 4 * h + m));
                const int ch = 4 * kk + (m >> 1);     // A: 16-byte chunk of the activation row
                ldmatrix_x4(a, ar + ((ch ^ (pa & 7)) << 4));
                ldmatrix_x4(a2, ar + (((ch + 2) ^ (pa & 7)) << 4));
                mma_bf16_16816(d0, a, b[0], b[1]);
                mma_bf16_16816(d1, a2, b[2], b[3]);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&s.empty[qq % s.nslot]);
            // token g's weight for slot u (0 when g is not routed there)
            const float wgt = g < T ? sh->tok_w[u][g] : 0.f;
            yacc[ri][0] = fmaf(wgt, d0[0] + d1[0], yacc[ri][0]);
            yacc[ri][1] = fmaf(wgt, d0[1] + d1[1], yacc[ri][1]);
        }
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) {
            sh->part[warp][ri * 64 + g * 8 + 2 * cq] = yacc[ri][0];
            sh->part[warp][ri * 64 + g * 8 + 2 * cq + 1] = yacc[ri][1];
        }
        if (sk_phase_end(s, fail)) break;
        // ---- 10. y: the warps' partial sums added in warp order ----
        for (int i = tid; i < nrg * T * 8; i += SK_CW * 32) {
            const int ri = i / (T * 8), t = (i / 8) % T, row = i % 8;
            float sum = 0.f;
#pragma unroll
            for (int w = 0; w < SK_CW; ++w) sum += sh->part[w][ri * 64 + t * 8 + row];
            Ly.y[(size_t)t * H + sk_rg(c, G, ri) * 8 + row] = __float2bfloat16_rn(sum);
        }
        // ---- 11. y of this layer is complete everywhere before the next layer reads x ----
        if (l + 1 < p.n_layers) {
            if (sk_phase_end(s, false)) break;
            if (tid == 0) {
                ++nbar;
                if (!sk_grid_barrier(s, base + (unsigned long long)nbar * G)) sh->abort = 1;
            }
            if (sk_phase_end(s, false)) break;
        }
    }
}

__global__ void __launch_bounds__(SK_THREADS, 1) stack_decode_kernel(const __grid_constant__ StackParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const SkLayout Lo = sk_layout(p.T, p.smem_bytes);
    SkState s;
    s.p = &p;
    s.ring = smem;
    s.ubuf = smem + Lo.ubuf_off;
    s.full = reinterpret_cast<uint64_t*>(smem + Lo.bars_off);
    s.empty = s.full + Lo.nslot;
    s.sh = reinterpret_cast<SkShared*>(smem + Lo.sh_off);
    s.nslot = Lo.nslot;
    s.T = p.T;
    s.c = blockIdx.x;
    s.G = gridDim.x;
    if (threadIdx.x == 0) {
        for (int i = 0; i < Lo.nslot; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], 1);
        }
        mbar_init(&s.sh->route_bar, 1);
        for (int i = 0; i < 32; ++i) s.sh->slot_seq[i] = 0u;
        s.sh->abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == SK_CW)
        sk_producer(s, lane);
    else
        sk_consumers(s, warp, lane);
}

}  // namespace

cudaError_t stack_decode_set_attributes(int max_optin) {
    return cudaFuncSetAttribute(stack_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, max_optin);
}

cudaError_t launch_stack_decode(const LaunchCtx& L, StackParams& p, int max_optin) {
    if (p.T < 1 || p.T > STACK_MAX_T || p.n_layers < 1 || p.n_layers > STACK_MAX_LAYERS) return cudaErrorInvalidValue;
    if (L.num_sms < SK_GU_UNITS || L.num_sms > E) return cudaErrorInvalidValue;
    p.smem_bytes = (uint32_t)max_optin;
    const SkLayout Lo = sk_layout(p.T, (uint32_t)max_optin);
    if (Lo.nslot < 8) return cudaErrorInvalidValue;
    return launch_hooked(L, FLINT_KERNEL_GATE_UP, stack_decode_kernel, dim3(L.num_sms), dim3(SK_THREADS), Lo.total, p);
}

}  // namespace flint
