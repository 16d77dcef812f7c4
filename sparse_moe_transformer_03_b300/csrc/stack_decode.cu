// stack_decode.cu -- cross-layer persistent decode: every layer of a stack
// of MoE layers in ONE kernel launch, for T <= 8 tokens (bf16 experts).
//
// Layer definition: RecursiveSI/flint (vLLM recipe page), "Overview" (256
// experts, top-6 sigmoid routing plus a shared expert).  The recipe page also
// names a low-latency decode path for a handful of requests, and the
// mrchatgpt.org article (section 4) a decode megakernel; this kernel is this
// library's design of that idea for B300.
//
// Cross-CTA exchanges cost about half a microsecond one way on B300 and a
// 148-CTA barrier about 1.1 us (a polled counter); an exchange in which every
// CTA polls every other CTA's data measured far slower (about 4 us), so the
// three exchanges of a layer (logits, activations, y) are barriers followed
// by one read.
//
// Why: at decode sizes a layer moves (U + 1) x 6 MiB of expert weights (U =
// distinct routed experts) and little else, so it should run at HBM speed.
// Three kernels per layer leave HBM idle while one kernel drains and the next
// starts, and every launch re-derives the routing.  Here one resident grid
// (one CTA per SM) walks the layers.  Per layer:
//
//   1. x (T rows) -> shared memory; each CTA dots its one or two router rows
//      (prefetched during the previous layer) with every token, writes the
//      fp32 logits and arrives at a grid barrier;
//   2. meanwhile CTAs 0..63 multiply their unit of the shared expert
//      (prefetched too); after the barrier every CTA reads the 256 logits of
//      each token, takes the top-6 (warp_top6) and builds the (slot, token)
//      tables;
//   3. a producer warp streams the CTA's routed gate/up units and then its
//      down row group of every slot into a ring of 16 KiB slots, one TMA
//      tensor box per slot; eight consumer warps multiply them on the
//      warp-level tensor core (mma.sync m16n8k16: 16 weight rows x 16
//      columns against up to 8 tokens), the K dimension split over the
//      warps, and write a = silu(g) * u (bf16) to a scratch buffer;
//   4. grid barrier; each CTA copies every pair's activations into shared
//      memory and applies its 16 down rows to every slot (the routing weight
//      folded in per token, each warp summing its slots in order, then the
//      warps in order): y is written once, deterministically;
//   5. grid barrier (layer l + 1 may read y_l), while the producer already
//      streams layer l + 1's router rows and shared-expert unit.
//
// Work split, in 16 KiB blocks: a gate/up unit is 8 gate rows + the 8
// matching up rows x 2048 columns (4 blocks, 64 units per expert); a down
// item is 16 rows of Wd x 512 columns (1 block, 128 per expert).  CTA c < 64
// owns shared unit c, CTA c < 128 owns down rows 16c .. 16c + 15 of every
// slot, and the routed units are dealt in contiguous ranges so that every CTA
// has the same number of gate/up units (those precede the activation barrier;
// the down items stream while they run and after it).  Every output element
// is produced by one CTA: nothing is reduced across CTAs.
#include "flint_common.cuh"
#include "../../include/flint_moe.h"
#include "flint_internal.h"
#include "mma_sync.cuh"
#include "nvfp4_frag.cuh"
#include "routing.cuh"
#include "tc_ptx.cuh"

#include <cstddef>

namespace flint {

namespace {

constexpr int SK_CW = 8;                          // consumer warps
constexpr int SK_THREADS = (SK_CW + 1) * 32;      // + one producer warp
constexpr int SK_SLOT_BF16 = 16384;               // bf16 ring slot: one tensor box
constexpr int SK_SLOT_NV = NV_CHUNK;              // NVFP4 ring slot: one 4608-byte chunk
constexpr int SK_GU_UNITS = I / 8;                // 64 gate/up units per expert
constexpr int SK_DN_ITEMS = H / 16;               // 128 down row groups per expert
constexpr int SK_GU_TILES = (2 * I / 128) * (H / 64);  // 256 gate/up tiles of an expert precede its down tiles
constexpr int SK_XSTRIDE = H * 2 + 16;            // padded x row in shared memory
constexpr int SK_MAX_SLOTS = 1 + STACK_MAX_T * TOPK;   // 49
constexpr int SK_MAX_RING_BF16 = 16;
constexpr int SK_MAX_RING = 48;                   // NVFP4 (the larger of the two)
constexpr int SK_NAMED = 1;                       // named barrier of the consumer warps

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
    alignas(16) float part[2][2][4][32 * 4];      // gate/up partial sums [quad][unit parity][warp of
                                                  // the quad][lane x 4]; down: [0][0..1] as [warp][lane x 4]
    float xinv[STACK_MAX_T];                      // NVFP4: 2^-e of token t's f16 staging of x
    uint64_t route_bar;                           // consumers -> producer: tables of the layer are built
    // Ring slot i was last handed out for sequence number slot_seq[i] - 1.  A
    // consumer waits for its sequence number here before the slot's full
    // barrier, so a parity wait never mistakes an older phase for its own.
    uint32_t slot_seq[SK_MAX_RING];
    int abort;
};
static_assert(offsetof(SkShared, part) % 16 == 0, "float4 access to the partial sums");
static_assert(offsetof(SkShared, route_bar) % 8 == 0, "mbarrier alignment");

// 128-byte rows of the tiled layout: in-tile row r keeps its 16-byte chunk c at c ^ (r % 8)
__device__ __forceinline__ uint32_t sw_chunk(int r, int c) { return (uint32_t)(((c ^ (r & 7)) << 4)); }

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_release_shared(uint32_t* p, uint32_t v) {
    asm volatile("st.release.cta.shared::cta.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_acquire_shared(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
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

__host__ __device__ __forceinline__ uint32_t sk_slot_bytes(bool nv) { return nv ? SK_SLOT_NV : SK_SLOT_BF16; }

__host__ __device__ __forceinline__ SkLayout sk_layout(int T, uint32_t max_smem, bool nv) {
    SkLayout L;
    const uint32_t bars = 2 * SK_MAX_RING * 8;
    const uint32_t fixed = sk_ubuf_bytes(T) + (uint32_t)((sizeof(SkShared) + 127) & ~size_t(127)) + bars;
    int ns = (int)((max_smem - fixed) / sk_slot_bytes(nv));
    const int cap = nv ? SK_MAX_RING : SK_MAX_RING_BF16;
    if (ns > cap) ns = cap;
    L.nslot = ns;
    L.ubuf_off = (uint32_t)ns * sk_slot_bytes(nv);
    L.ubuf_off = (L.ubuf_off + 127u) & ~127u;
    L.bars_off = L.ubuf_off + sk_ubuf_bytes(T);
    L.sh_off = L.bars_off + bars;
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
    uint32_t slot;                                // ring slot bytes
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

__device__ __forceinline__ uint8_t* sk_slot_ptr(const SkState& s, uint32_t q) {
    return s.ring + (size_t)(q % (uint32_t)s.nslot) * s.slot;
}

// Release ring sequence number q: the warp's share of the slot's SK_CW
// expected arrivals (cnt = SK_CW when it is the slot's only reader).
__device__ __forceinline__ void sk_release(const SkState& s, uint32_t q, int lane, uint32_t cnt) {
    __syncwarp();
    if (lane == 0)
        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(&s.empty[q % (uint32_t)s.nslot])),
                     "r"(cnt)
                     : "memory");
}

// Grid barrier, split so that work can run between arriving and waiting.
// Arrive (one thread, after the consumer warps synchronised, so that the
// CTA's writes are ordered before it by the release): count this CTA in.
__device__ __forceinline__ void sk_grid_arrive(const SkState& s) {
    asm volatile("red.release.gpu.global.add.u64 [%0], 1;" ::"l"(s.p->bar) : "memory");
}

// Wait until every CTA of the grid has arrived `target` - base times.
__device__ bool sk_grid_wait(const SkState& s, unsigned long long target) {
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

__device__ __forceinline__ bool sk_grid_barrier(const SkState& s, unsigned long long target) {
    sk_grid_arrive(s);
    return sk_grid_wait(s, target);
}

// ---- per-CTA work of a layer (identical formulas in producer and consumers) ----

__device__ __forceinline__ int sk_router_rows(int c, int G) { return (c < E ? 1 : 0) + (c + G < E ? 1 : 0); }
__device__ __forceinline__ int sk_has_sg(int c) { return c < SK_GU_UNITS ? 1 : 0; }
__device__ __forceinline__ int sk_has_dn(int c) { return c < SK_DN_ITEMS ? 1 : 0; }

// End of CTA c's range of routed gate/up units (the units of slots 1..U in
// order): every CTA's share of all 64 (U + 1) gate/up units minus the shared
// units the CTAs up to c own.  Only the gate/up units have to be done before
// the activations are complete (the down items are applied after that grid
// barrier), so they alone are balanced.  Non-decreasing in c and equal to
// 64 U at the last CTA (checked on the host for every U).
__host__ __device__ __forceinline__ int sk_rcum(int c, int G, int U) {
    if (c < 0) return 0;
    const int total = SK_GU_UNITS * (U + 1);
    const int ucum = (int)(((long long)(c + 1) * total) / G);
    const int scum = c + 1 < SK_GU_UNITS ? c + 1 : SK_GU_UNITS;
    const int r = ucum - scum;
    return r < 0 ? 0 : (r > SK_GU_UNITS * U ? SK_GU_UNITS * U : r);
}

// Slots and pairs of a batch of T <= 8 tokens from their top-6 (one warp):
// slot 0 is the shared expert (pair t = token t), then the routed experts by
// increasing id, each with its tokens in increasing order.  tok_pair[u][t] /
// tok_w[u][t]: the pair and routing weight of token t in slot u (-1 / 0 when
// t is not routed there).  Every lane works on its own experts and pairs.
// The producer is released (route_bar) as soon as the slots' experts exist.
__device__ void sk_build_tables(int T, SkShared* sh, int lane) {
    DecodeTables* tab = &sh->tab;
    if (T == 1) {
        // one token: its six (distinct) experts are the routed slots 1..6 in
        // increasing id order, expert of rank k in slot and pair 1 + k -- the
        // same tables the general path below builds, from six shuffles
        const int e = lane < TOPK ? sh->sel_e[lane] : E;
        int rank = 0;
#pragma unroll
        for (int j = 0; j < TOPK; ++j) rank += __shfl_sync(0xFFFFFFFFu, e, j) < e ? 1 : 0;
        if (lane < TOPK) {
            tab->slot_expert[1 + rank] = e;
            tab->slot_pair0[1 + rank] = 1 + rank;
            sh->tok_pair[1 + rank][0] = 1 + rank;
            sh->tok_w[1 + rank][0] = sh->sel_w[lane];
        }
        if (lane == 0) {
            tab->n_slots = 1 + TOPK;
            tab->n_pairs = 1 + TOPK;
            tab->slot_pair0[1 + TOPK] = 1 + TOPK;
            tab->T = 1;
            tab->slot_expert[0] = SHARED;
            tab->slot_pair0[0] = 0;
            sh->tok_pair[0][0] = 0;
            sh->tok_w[0][0] = 1.f;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&sh->route_bar);
        __syncwarp();
        return;
    }
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
    __syncwarp();
    // the producer needs only the slots' experts: let it start the routed copies
    if (lane == 0) mbar_arrive(&sh->route_bar);
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
// producer (lanes 0 .. pl - 1 of the producer warp)
// ---------------------------------------------------------------------------
// NVFP4 layers: four lanes run the producer loop together (every loop value
// is the same in each of them) and fill up to four consecutive ring slots at
// once, lane i the slot seq + i: a gate/up unit's four 4608-byte chunks, four
// down items, the router rows.  One lane issuing every small copy in turn
// bounded their streaming (NVFP4 stack at T = 8: 34.9 -> 32.7 us/layer, T = 1:
// 16.9 -> 15.8).  bf16 layers keep one lane: their 16 KiB boxes measured
// slower issued four at a time (T = 8: 39.8 -> 42.9 us/layer).

template <bool NV>
struct SkPl {
    static constexpr int n = NV ? 4 : 1;                     // producer lanes
    static constexpr unsigned mask = (1u << n) - 1u;
};

struct SkProducer {
    uint32_t seq = 0;   // ring slots handed out so far (equal in every producer lane)
    int pl;             // producer lanes
    unsigned mask;

    // Lane i < n takes slot seq + i for a copy of `bytes`, once that slot's
    // previous use is released; every lane then advances seq by n.  Returns
    // the same answer in every lane: false if any lane's wait gave up.
    __device__ __forceinline__ bool take(const SkState& s, int lane, int n, uint32_t bytes, uint8_t** dst,
                                         uint64_t** bar) {
        bool ok = bytes <= s.slot;   // never false: every item fits its slot
        if (ok && lane < n) {
            const uint32_t q = seq + (uint32_t)lane;
            const int slot = (int)(q % (uint32_t)s.nslot);
            const uint32_t use = q / (uint32_t)s.nslot;
            if (use > 0 && !sk_wait(s, &s.empty[slot], (use - 1) & 1)) {
                ok = false;
            } else {
                mbar_arrive_expect_tx(&s.full[slot], bytes);
                st_release_shared(&s.sh->slot_seq[slot], q + 1u);
                *dst = s.ring + (size_t)slot * s.slot;
                *bar = &s.full[slot];
            }
        }
        seq += (uint32_t)n;
        return __all_sync(mask, ok);
    }
};

// Ring slots of CTA c's router rows: both rows in one 16 KiB bf16 slot, one
// row (4 KiB) per 4608-byte NVFP4 slot.
__device__ __forceinline__ int sk_router_slots(const SkState& s) {
    const int nr = sk_router_rows(s.c, s.G);
    return s.slot >= (uint32_t)(2 * H * 2) ? (nr ? 1 : 0) : nr;
}
__device__ __forceinline__ const uint8_t* sk_router_row(const SkState& s, uint32_t seqR, int i) {
    return s.slot >= (uint32_t)(2 * H * 2) ? sk_slot_ptr(s, seqR) + i * H * 2 : sk_slot_ptr(s, seqR + (uint32_t)i);
}

// Router rows of CTA c for layer l (plain bulk copies), lane i slot i0 + i.
__device__ __forceinline__ bool sk_issue_router(const SkState& s, SkProducer& pr, int lane, int l) {
    const int nr = sk_router_rows(s.c, s.G), nrs = sk_router_slots(s);
    if (nrs == 0) return true;
    const int per = nr / nrs;    // rows per slot
    for (int i0 = 0; i0 < nrs; i0 += pr.pl) {
        const int n = min(pr.pl, nrs - i0), i = i0 + lane;
        uint8_t* dst = nullptr;
        uint64_t* bar = nullptr;
        if (!pr.take(s, lane, n, (uint32_t)per * H * 2, &dst, &bar)) return false;
        if (lane < n)
            for (int k = 0; k < per; ++k)
                bulk_g2s(dst + k * H * 2, s.p->layer[l].router + (size_t)(s.c + (i * per + k) * s.G) * H, H * 2, bar);
    }
    return true;
}

// Gate/up unit q of an expert: 4 slots, one box each (lane i slot k0 + i): gate
// rows 8q .. 8q + 7 over column tiles 0..15 and 16..31, then the matching up
// rows likewise.
__device__ __forceinline__ bool sk_issue_gateup(const SkState& s, SkProducer& pr, int lane, const CUtensorMap* maps,
                                                int expert, int q) {
    const int r0 = 8 * q, rb = r0 >> 7;
    for (int k0 = 0; k0 < 4; k0 += pr.pl) {
        const int n = min(pr.pl, 4 - k0), k = k0 + lane;
        uint8_t* dst = nullptr;
        uint64_t* bar = nullptr;
        if (!pr.take(s, lane, n, SK_SLOT_BF16, &dst, &bar)) return false;
        if (lane < n) {
            const int tile = ((k >> 1) * 4 + rb) * (H / 64) + (k & 1) * 16;   // up rows: row blocks 4..7
            tc::tma_load_4d(dst, &maps[0], 0, (r0 & 127) >> 2, tile, expert, bar);
        }
    }
    return true;
}

// Down rows 16 g .. 16 g + 15 of the experts of slots u0 .. u0 + n - 1 (one
// slot each: the 8 column tiles of K = 512), lane i slot u0 + i.
__device__ __forceinline__ bool sk_issue_down(const SkState& s, SkProducer& pr, int lane, const CUtensorMap* maps,
                                              const int* slot_expert, int u0, int n, int g) {
    uint8_t* dst = nullptr;
    uint64_t* bar = nullptr;
    if (!pr.take(s, lane, n, SK_SLOT_BF16, &dst, &bar)) return false;
    if (lane < n)
        tc::tma_load_4d(dst, &maps[1], 0, (g & 7) * 4, SK_GU_TILES + (g >> 3) * (I / 64), slot_expert[u0 + lane],
                        bar);
    return true;
}

// NVFP4 gate/up unit q of an expert: 4 slots, one 4608-byte chunk each (K
// blocks 32 k .. 32 k + 31 of its 8 gate and 8 up rows, in the owned layout),
// lane i chunk k0 + i.
__device__ __forceinline__ bool sk_issue_gateup_nv(const SkState& s, SkProducer& pr, int lane, const uint8_t* nv,
                                                   int expert, int q) {
    for (int k0 = 0; k0 < NV_GU_CHUNKS; k0 += pr.pl) {
        const int n = min(pr.pl, NV_GU_CHUNKS - k0), k = k0 + lane;
        uint8_t* dst = nullptr;
        uint64_t* bar = nullptr;
        if (!pr.take(s, lane, n, NV_CHUNK, &dst, &bar)) return false;
        if (lane < n)
            bulk_g2s(dst, nv + (size_t)expert * NV_EXPERT_BYTES + (size_t)(q * NV_GU_CHUNKS + k) * NV_CHUNK, NV_CHUNK,
                     bar);
    }
    return true;
}

// NVFP4 down rows 16 g .. 16 g + 15 of the experts of slots u0 .. u0 + n - 1
// (one chunk each, K = 512), lane i slot u0 + i.
__device__ __forceinline__ bool sk_issue_down_nv(const SkState& s, SkProducer& pr, int lane, const uint8_t* nv,
                                                 const int* slot_expert, int u0, int n, int g) {
    uint8_t* dst = nullptr;
    uint64_t* bar = nullptr;
    if (!pr.take(s, lane, n, NV_CHUNK, &dst, &bar)) return false;
    if (lane < n)
        bulk_g2s(dst, nv + (size_t)slot_expert[u0 + lane] * NV_EXPERT_BYTES + NV_GU_BYTES + (size_t)g * NV_CHUNK,
                 NV_CHUNK, bar);
    return true;
}

template <bool NV>
__device__ __forceinline__ bool sk_issue_unit(const SkState& s, SkProducer& pr, int lane, const StackLayerArgs& Ly,
                                              int expert, int q) {
    if constexpr (NV)
        return sk_issue_gateup_nv(s, pr, lane, Ly.nv, expert, q);
    else
        return sk_issue_gateup(s, pr, lane, Ly.maps, expert, q);
}

template <bool NV>
__device__ void sk_producer(const SkState& s, int lane) {
    if (lane >= SkPl<NV>::n) return;
    SkProducer pr;
    pr.pl = SkPl<NV>::n;
    pr.mask = SkPl<NV>::mask;
    const StackParams& p = *s.p;
    bool ok = sk_issue_router(s, pr, lane, 0);
    if (ok && sk_has_sg(s.c)) ok = sk_issue_unit<NV>(s, pr, lane, p.layer[0], SHARED, s.c);
    if constexpr (!NV) {
        if (lane == 0) {
            tc::prefetch_tensormap(&p.layer[0].maps[0]);
            tc::prefetch_tensormap(&p.layer[0].maps[1]);
        }
    }
    for (int l = 0; ok && l < p.n_layers; ++l) {
        // the next layer's descriptors, ahead of their first use
        if constexpr (!NV) {
            if (lane == 0 && l + 1 < p.n_layers) {
                tc::prefetch_tensormap(&p.layer[l + 1].maps[0]);
                tc::prefetch_tensormap(&p.layer[l + 1].maps[1]);
            }
        }
        // the consumers publish the layer's tables
        if (!__all_sync(pr.mask, sk_wait(s, &s.sh->route_bar, l & 1))) break;
        const DecodeTables& tab = s.sh->tab;
        const int U = tab.n_slots - 1;
        const StackLayerArgs& Ly = p.layer[l];
        const int k0 = sk_rcum(s.c - 1, s.G, U), k1 = sk_rcum(s.c, s.G, U);
        for (int k = k0; ok && k < k1; ++k)
            ok = sk_issue_unit<NV>(s, pr, lane, Ly, tab.slot_expert[1 + k / SK_GU_UNITS], k % SK_GU_UNITS);
        if (sk_has_dn(s.c))
            for (int u = 0; ok && u <= U; u += pr.pl) {
                const int n = min(pr.pl, U + 1 - u);
                if constexpr (NV)
                    ok = sk_issue_down_nv(s, pr, lane, Ly.nv, tab.slot_expert, u, n, s.c);
                else
                    ok = sk_issue_down(s, pr, lane, Ly.maps, tab.slot_expert, u, n, s.c);
            }
        if (ok && l + 1 < p.n_layers) {
            ok = sk_issue_router(s, pr, lane, l + 1);
            if (ok && sk_has_sg(s.c)) ok = sk_issue_unit<NV>(s, pr, lane, p.layer[l + 1], SHARED, s.c);
        }
    }
    // copies still in flight (only after an abort): wait for them before exiting
    // (a slot whose copies were never issued does not complete: short limit)
    if (lane == 0 && sk_aborted(s)) {
        const uint32_t first = pr.seq > (uint32_t)s.nslot ? pr.seq - (uint32_t)s.nslot : 0u;
        for (uint32_t q = first; q < pr.seq; ++q)
            mbar_wait_bounded(&s.full[q % s.nslot], (q / s.nslot) & 1, 10000000ull);
    }
}

// ---------------------------------------------------------------------------
// consumers
// ---------------------------------------------------------------------------

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

// One gate/up unit (slots sq .. sq + 3: gate tiles 0..15, 16..31, up tiles
// 0..15, 16..31) against the tokens, by a quad of warps: warp wq of the quad
// multiplies column tiles 8 wq .. 8 wq + 7, 16 weight rows (8 gate over 8 up)
// x 512 columns, into d[] (lane (g, cq): gate row g and up row g for tokens
// 2 cq and 2 cq + 1), then releases the two slots it read.  All 32 lanes
// take part; returns false if a wait gave up.
__device__ __forceinline__ bool sk_gateup_part(const SkState& s, uint32_t sq, int wq, int lane, float (&d)[4]) {
    const int half = wq >> 1;
    const bool got = sk_wait_full(s, sq + (uint32_t)half) && sk_wait_full(s, sq + 2u + (uint32_t)half);
    if (!__all_sync(0xFFFFFFFFu, got)) return false;
    const int m = lane >> 3, r = lane & 7;
    // A: matrix m: row r of the gate (m even) or up (m odd) box, chunk (m >> 1) of the k-step
    const uint8_t* arow = sk_slot_ptr(s, sq + (uint32_t)(2 * (m & 1) + half)) + r * 128;
    // B: token rows of x (padding tokens read token 0; their columns are not used)
    const uint8_t* xrow = s.ubuf + (size_t)(r < s.T ? r : 0) * SK_XSTRIDE + m * 16;
    float acc[4][4] = {};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int kt = 8 * wq + i;                        // column tile 0..31
        const uint8_t* tile = arow + (kt & 15) * 1024;
#pragma unroll
        for (int h = 0; h < 2; ++h) {                     // two 32-column halves = two k-step pairs
            uint32_t a[4], a2[4], b[4];
            ldmatrix_x4(a, tile + sw_chunk(r, 4 * h + (m >> 1)));
            ldmatrix_x4(a2, tile + sw_chunk(r, 4 * h + 2 + (m >> 1)));
            ldmatrix_x4(b, xrow + (size_t)(kt * 64 + 32 * h) * 2);
            mma_bf16_16816(acc[2 * h], a, b[0], b[1]);
            mma_bf16_16816(acc[2 * h + 1], a2, b[2], b[3]);
        }
    }
    sk_release(s, sq + (uint32_t)half, lane, 4);
    sk_release(s, sq + 2u + (uint32_t)half, lane, 4);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = (acc[0][i] + acc[1][i]) + (acc[2][i] + acc[3][i]);
    return true;
}

// NVFP4 gate/up unit (slots sq .. sq + 3: its four chunks of K blocks) by a
// quad of warps: warp wq dequantises chunk wq straight into A fragments (16
// rows: 8 gate over 8 up, 512 columns) and multiplies them with x staged as
// f16 (token t scaled by 2^e_t).  Releases the chunk's slot.
__device__ __forceinline__ bool sk_gateup_part_nv(const SkState& s, uint32_t sq, int wq, int lane, float (&d)[4]) {
    if (!__all_sync(0xFFFFFFFFu, sk_wait_full(s, sq + (uint32_t)wq))) return false;
    const uint8_t* buf = sk_slot_ptr(s, sq + (uint32_t)wq);
    const int g = lane >> 2, cq = lane & 3;
    // B: token g's f16 row (padding tokens read token 0), columns 512 wq + 16 kb + 2 cq
    const __half* xb =
        reinterpret_cast<const __half*>(s.ubuf + (size_t)(g < s.T ? g : 0) * SK_XSTRIDE) + 512 * wq + 2 * cq;
    float acc[4][4] = {};
#pragma unroll
    for (int kb = 0; kb < NV_CHUNK_KB; kb += 4) {
        uint32_t a[4][4];
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
            nv_a_frag(*reinterpret_cast<const uint32_t*>(buf + (kb + ch) * 128 + 4 * lane),
                      *reinterpret_cast<const uint16_t*>(buf + NV_CODES + (kb + ch) * 16 + 2 * g), a[ch]);
#pragma unroll
        for (int ch = 0; ch < 4; ++ch)
            mma_f16_16816(acc[ch], a[ch], *reinterpret_cast<const uint32_t*>(xb + (kb + ch) * 16),
                          *reinterpret_cast<const uint32_t*>(xb + (kb + ch) * 16 + 8));
    }
    sk_release(s, sq + (uint32_t)wq, lane, SK_CW);
#pragma unroll
    for (int i = 0; i < 4; ++i) d[i] = (acc[0][i] + acc[1][i]) + (acc[2][i] + acc[3][i]);
    return true;
}

template <bool NV>
__device__ __forceinline__ bool sk_unit_part(const SkState& s, uint32_t sq, int wq, int lane, float (&d)[4]) {
    if constexpr (NV)
        return sk_gateup_part_nv(s, sq, wq, lane, d);
    else
        return sk_gateup_part(s, sq, wq, lane, d);
}

// Activation rows in the scratch buffer: pair p's 512 bf16, its 16-byte
// chunk c stored at c ^ (p % 8), so that the eight token rows of one MMA
// operand read through different banks once copied into shared memory.
__device__ __forceinline__ int sk_act_index(int p, int j) {
    return p * I + ((((j >> 3) ^ (p & 7))) << 3) + (j & 7);
}

// The unit's four partial sums (part[quad][par][w]) added in warp order by
// one warp; a = silu(gate) * up for the tokens routed to slot u (u = 0: the
// shared expert, whose pair of token t is t; it runs before the layer's
// tables exist).  Lane (g, cq) computes column 8q + g of tokens 2 cq and
// 2 cq + 1.
// NVFP4: the sums are scaled by the tensor scale tsg and the token's 2^-e_t
// first.
template <bool NV>
__device__ __forceinline__ void sk_gateup_finish(const SkState& s, int quad, int par, int u, int q, int lane,
                                                 const float* ts) {
    SkShared* sh = s.sh;
    float4 sum = *reinterpret_cast<const float4*>(&sh->part[quad][par][0][lane * 4]);
#pragma unroll
    for (int w = 1; w < 4; ++w) {
        const float4 v = *reinterpret_cast<const float4*>(&sh->part[quad][par][w][lane * 4]);
        sum.x += v.x;
        sum.y += v.y;
        sum.z += v.z;
        sum.w += v.w;
    }
    const int g = lane >> 2, cq = lane & 3, j = 8 * q + g;
    const int t0 = 2 * cq, t1 = 2 * cq + 1;
    if constexpr (NV) {
        const int expert = u == 0 ? SHARED : sh->tab.slot_expert[u];
        const float tsg = __ldg(ts + 2 * expert);
        const float f0 = t0 < s.T ? tsg * sh->xinv[t0] : 0.f, f1 = t1 < s.T ? tsg * sh->xinv[t1] : 0.f;
        sum.x *= f0;
        sum.z *= f0;
        sum.y *= f1;
        sum.w *= f1;
    }
    if (t0 < s.T) {
        const int pp = u == 0 ? t0 : sh->tok_pair[u][t0];
        if (pp >= 0) s.p->act[sk_act_index(pp, j)] = __float2bfloat16_rn(silu_f(sum.x) * sum.z);
    }
    if (t1 < s.T) {
        const int pp = u == 0 ? t1 : sh->tok_pair[u][t1];
        if (pp >= 0) s.p->act[sk_act_index(pp, j)] = __float2bfloat16_rn(silu_f(sum.y) * sum.w);
    }
}

// Named barrier of one quad of consumer warps (ids 2 and 3) that ORs the
// threads' failure flags, like sk_phase_end.
__device__ __forceinline__ bool sk_quad_sync(const SkState& s, int quad, bool fail) {
    const uint32_t v = (fail || sk_aborted(s)) ? 1u : 0u;
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, 128, p;\n selp.u32 %0, 1, 0, q;\n}\n"
        : "=r"(r)
        : "r"(v), "r"(2 + quad)
        : "memory");
    if (r) s.sh->abort = 1;
    return r != 0;
}

template <bool NV>
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
    const int cq = lane & 3;
    for (int l = 0; l < p.n_layers; ++l) {
        const StackLayerArgs& Ly = p.layer[l];
        bool fail = false;
        // ---- 1. x rows into shared memory (16-byte loads through L2) ----
        for (int i0 = tid; i0 < T * (H / 8); i0 += 8 * SK_CW * 32) {   // 8 loads in flight per thread
            uint4 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int i = i0 + k * SK_CW * 32;
                if (i < T * (H / 8)) v[k] = __ldcg(reinterpret_cast<const uint4*>(Ly.x + (size_t)(i / (H / 8)) * H) + i % (H / 8));
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int i = i0 + k * SK_CW * 32;
                if (i < T * (H / 8))
                    *reinterpret_cast<uint4*>(s.ubuf + (size_t)(i / (H / 8)) * SK_XSTRIDE + (i % (H / 8)) * 16) = v[k];
            }
        }
        if (sk_phase_end(s, false)) break;
        // ---- 2. this CTA's router rows: fp32 logits (bias included) ----
        const int nr = sk_router_rows(c, G), nrs = sk_router_slots(s);
        const uint32_t seqR = seq;
        seq += (uint32_t)nrs;
        if (nr) {
            bool got = true;
            for (int k = 0; k < nrs; ++k) got = got && sk_wait_full(s, seqR + (uint32_t)k);
            fail = !__all_sync(0xFFFFFFFFu, got);
            for (int pi = warp; !fail && pi < nr * T; pi += SK_CW) {
                const int i = pi / T, t = pi % T, e = c + i * G;
                const uint4* wr = reinterpret_cast<const uint4*>(sk_router_row(s, seqR, i));
                const uint4* xr = reinterpret_cast<const uint4*>(s.ubuf + (size_t)t * SK_XSTRIDE);
                float ac[4] = {0.f, 0.f, 0.f, 0.f};      // four independent chains
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint4 w = wr[lane + 32 * k], xv = xr[lane + 32 * k];
                    ac[0] = fmaf(bf_lo(w.x), bf_lo(xv.x), ac[0]);
                    ac[1] = fmaf(bf_hi(w.x), bf_hi(xv.x), ac[1]);
                    ac[2] = fmaf(bf_lo(w.y), bf_lo(xv.y), ac[2]);
                    ac[3] = fmaf(bf_hi(w.y), bf_hi(xv.y), ac[3]);
                    ac[0] = fmaf(bf_lo(w.z), bf_lo(xv.z), ac[0]);
                    ac[1] = fmaf(bf_hi(w.z), bf_hi(xv.z), ac[1]);
                    ac[2] = fmaf(bf_lo(w.w), bf_lo(xv.w), ac[2]);
                    ac[3] = fmaf(bf_hi(w.w), bf_hi(xv.w), ac[3]);
                }
                const float acc = warp_sum((ac[0] + ac[1]) + (ac[2] + ac[3]));
                if (lane == 0) p.logits[(size_t)t * E + e] = acc + sh->bias[l][i];
            }
            if (!fail)
                for (int k = 0; k < nrs; ++k) sk_release(s, seqR + (uint32_t)k, lane, 1);
        }
        // the CTA's logits are written: count it in at the logits barrier now,
        // wait for the others after the shared unit
        if (sk_phase_end(s, fail)) break;
        if (tid == 4 * 32) sk_grid_arrive(s);   // warp 4: quad 0 goes on with the shared unit
        if constexpr (NV) {
            // x -> f16 times 2^e_t in place, token t on warp t (the router is done
            // with the bf16 rows): the token's largest |x| lands in [2^14, 2^15),
            // exact for every bf16 value within 28 binades of it
            if (warp < T) {
                uint4* row = reinterpret_cast<uint4*>(s.ubuf + (size_t)warp * SK_XSTRIDE);
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
                if (lane == 0) sh->xinv[warp] = ldexpf(1.f, -e);
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
            if (sk_phase_end(s, false)) break;
        }
        // ---- 3. the shared expert's unit of this CTA (CTAs 0..63) ----
        const int has_sg = sk_has_sg(c);
        const uint32_t seqSG = seq;
        seq += has_sg ? 4 : 0;
        if (has_sg && warp < 4) {   // quad 0 (every warp of it reaches the quad barrier)
            if (!fail) {
                float d[4];
                fail = !sk_unit_part<NV>(s, seqSG, warp, lane, d);
                if (!fail)
                    *reinterpret_cast<float4*>(&sh->part[0][0][warp][lane * 4]) = make_float4(d[0], d[1], d[2], d[3]);
            }
            if (sk_quad_sync(s, 0, fail)) fail = true;
            else if (warp == 0) sk_gateup_finish<NV>(s, 0, 0, 0, c, lane, Ly.nv_ts);
        }
        // ---- 4. every CTA's logits are written (the barrier's wait; the shared
        // unit's multiply above overlapped it); top-6 of token t on warp t ----
        if (sk_phase_end(s, fail)) break;
        if (tid == 0) {
            ++nbar;
            if (!sk_grid_wait(s, base + (unsigned long long)nbar * G)) sh->abort = 1;
        }
        if (sk_phase_end(s, false)) break;
        if (warp < T) {
            float v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = __ldcg(p.logits + (size_t)warp * E + lane + 32 * k);
            int sel[TOPK];
            float wt[TOPK];
            warp_top6(v, lane, sel, wt);
            if (lane < TOPK) {
                sh->sel_e[warp * TOPK + lane] = pick6(sel, lane);
                sh->sel_w[warp * TOPK + lane] = pick6(wt, lane);
            }
        }
        if (sk_phase_end(s, false)) break;
        // ---- 5. tables: slots (shared first, then the routed experts by id), pairs ----
        if (warp == 0) sk_build_tables(T, sh, lane);
        if (sk_phase_end(s, false)) break;
        const int U = sh->tab.n_slots - 1;
        // ---- 6. routed gate/up units of the CTA's range: quad q (warps 4q ..
        // 4q + 3) takes units q, q + 2, ..., K split over its warps; warp
        // (j / 2) % 4 of the quad finishes unit j ----
        const int k0 = sk_rcum(c - 1, G, U), k1 = sk_rcum(c, G, U);
        const uint32_t seqRG = seq;
        seq += 4u * (uint32_t)(k1 - k0);
        {
            const int quad = warp >> 2, wq = warp & 3;
            for (int j = quad; j < k1 - k0; j += 2) {
                float d[4];
                const bool f = !sk_unit_part<NV>(s, seqRG + 4u * j, wq, lane, d);
                const int par = (j >> 1) & 1;
                if (!f)
                    *reinterpret_cast<float4*>(&sh->part[quad][par][wq][lane * 4]) = make_float4(d[0], d[1], d[2], d[3]);
                // the parity buffer is written again two units later, after this
                // quad's next barrier, which the finishing warp reaches after the sum
                if (sk_quad_sync(s, quad, f)) break;
                if (wq == ((j >> 1) & 3)) {
                    const int k = k0 + j;
                    sk_gateup_finish<NV>(s, quad, par, 1 + k / SK_GU_UNITS, k % SK_GU_UNITS, lane, Ly.nv_ts);
                }
            }
        }
        // ---- 7. every CTA's activations are written (grid barrier) ----
        if (sk_phase_end(s, false)) break;
        if (tid == 0) {
            ++nbar;
            if (!sk_grid_barrier(s, base + (unsigned long long)nbar * G)) sh->abort = 1;
        }
        if (sk_phase_end(s, false)) break;
        // ---- 8. all pairs' activations into shared memory (x is no longer read) ----
        {
            const int n16 = sh->tab.n_pairs * (I / 8);
            for (int i0 = tid; i0 < n16; i0 += 8 * SK_CW * 32) {   // 8 loads in flight per thread
                uint4 v[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int i = i0 + k * SK_CW * 32;
                    if (i < n16) v[k] = __ldcg(reinterpret_cast<const uint4*>(p.act) + i);
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int i = i0 + k * SK_CW * 32;
                    if (i < n16) *reinterpret_cast<uint4*>(s.ubuf + (size_t)i * 16) = v[k];
                }
            }
        }
        if (sk_phase_end(s, false)) break;
        // ---- 9. down rows 16c .. 16c + 15 of every slot: warp u % 8 takes slot
        // u's item whole, the routing weights folded in per token ----
        const int has_dn = sk_has_dn(c);
        const uint32_t seqD = seq;
        seq += has_dn ? (uint32_t)(U + 1) : 0u;
        float yacc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int u = warp; has_dn && u <= U && !fail; u += SK_CW) {
            const uint32_t qq = seqD + (uint32_t)u;
            if (!__all_sync(0xFFFFFFFFu, sk_wait_full(s, qq))) {
                fail = true;
                break;
            }
            float acc[4][4] = {};
            if constexpr (NV) {
                // A: the chunk's 32 K blocks dequantised to bf16 fragments; B: token g's
                // pair row in slot u (4-byte reads of the chunk-swizzled activations)
                const uint8_t* buf = sk_slot_ptr(s, qq);
                const int g = lane >> 2;
                int pb = g < T ? sh->tok_pair[u][g] : -1;
                pb = pb < 0 ? 0 : pb;
                const uint8_t* ar = s.ubuf + (size_t)pb * (I * 2) + 4 * cq;
#pragma unroll 8
                for (int kb = 0; kb < NV_CHUNK_KB; ++kb) {
                    uint32_t a[4];
                    nv_a_frag(*reinterpret_cast<const uint32_t*>(buf + kb * 128 + 4 * lane),
                              *reinterpret_cast<const uint16_t*>(buf + NV_CODES + kb * 16 + 2 * g), a);
#pragma unroll
                    for (int q = 0; q < 4; ++q) a[q] = f16x2_to_bf16x2(a[q]);
                    mma_bf16_16816(acc[kb & 3], a, *reinterpret_cast<const uint32_t*>(ar + (((2 * kb) ^ (pb & 7)) << 4)),
                                   *reinterpret_cast<const uint32_t*>(ar + (((2 * kb + 1) ^ (pb & 7)) << 4)));
                }
            } else {
                // A: rows r (m even) or 8 + r (m odd) of the 8 column tiles;
                // B: token rows -> their pairs in slot u (token r: lane's row)
                const uint8_t* wrow = sk_slot_ptr(s, qq) + (r + 8 * (m & 1)) * 128;
                int pb = r < T ? sh->tok_pair[u][r] : -1;
                pb = pb < 0 ? 0 : pb;
                const uint8_t* br = s.ubuf + (size_t)pb * (I * 2);
#pragma unroll
                for (int kt = 0; kt < I / 64; ++kt) {
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t a[4], a2[4], b[4];
                        ldmatrix_x4(a, wrow + kt * 2048 + sw_chunk(r, 4 * h + (m >> 1)));
                        ldmatrix_x4(a2, wrow + kt * 2048 + sw_chunk(r, 4 * h + 2 + (m >> 1)));
                        const int ch = 8 * kt + 4 * h + m;         // 16-byte chunk of the activation row
                        ldmatrix_x4(b, br + ((ch ^ (pb & 7)) << 4));
                        mma_bf16_16816(acc[2 * h], a, b[0], b[1]);
                        mma_bf16_16816(acc[2 * h + 1], a2, b[2], b[3]);
                    }
                }
            }
            sk_release(s, qq, lane, SK_CW);
            // lane (g, cq): rows g and g + 8, tokens 2 cq and 2 cq + 1 (NVFP4: times
            // the down matrix's tensor scale)
            const float tsd = NV ? __ldg(Ly.nv_ts + 2 * sh->tab.slot_expert[u] + 1) : 1.f;
            const float w0 = 2 * cq < T ? sh->tok_w[u][2 * cq] * tsd : 0.f;
            const float w1 = 2 * cq + 1 < T ? sh->tok_w[u][2 * cq + 1] * tsd : 0.f;
            float dd[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) dd[i] = (acc[0][i] + acc[1][i]) + (acc[2][i] + acc[3][i]);
            yacc[0] = fmaf(w0, dd[0], yacc[0]);
            yacc[1] = fmaf(w1, dd[1], yacc[1]);
            yacc[2] = fmaf(w0, dd[2], yacc[2]);
            yacc[3] = fmaf(w1, dd[3], yacc[3]);
        }
        float* ypart = &sh->part[0][0][0][0];
        *reinterpret_cast<float4*>(&ypart[(warp * 32 + lane) * 4]) = make_float4(yacc[0], yacc[1], yacc[2], yacc[3]);
        if (sk_phase_end(s, fail)) break;
        // ---- 10. y: the warps' partial sums added in warp order ----
        if (has_dn) {
            for (int i = tid; i < 16 * T; i += SK_CW * 32) {
                const int row = i & 15, t = i >> 4;
                // the lane holding (row, token t): g = row % 8, cq = t / 2; element 2 (row >= 8) + t % 2
                const int ln = (row & 7) * 4 + (t >> 1), el = (row >> 3) * 2 + (t & 1);
                float sum = 0.f;
#pragma unroll
                for (int w = 0; w < SK_CW; ++w) sum += ypart[(w * 32 + ln) * 4 + el];
                Ly.y[(size_t)t * H + 16 * c + row] = __float2bfloat16_rn(sum);
            }
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

template <bool NV>
__global__ void __launch_bounds__(SK_THREADS, 1) stack_decode_kernel(const __grid_constant__ StackParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const SkLayout Lo = sk_layout(p.T, p.smem_bytes, NV);
    SkState s;
    s.p = &p;
    s.ring = smem;
    s.ubuf = smem + Lo.ubuf_off;
    s.full = reinterpret_cast<uint64_t*>(smem + Lo.bars_off);
    s.empty = s.full + SK_MAX_RING;
    s.sh = reinterpret_cast<SkShared*>(smem + Lo.sh_off);
    s.nslot = Lo.nslot;
    s.T = p.T;
    s.c = blockIdx.x;
    s.G = gridDim.x;
    s.slot = sk_slot_bytes(NV);
    if (threadIdx.x == 0) {
        for (int i = 0; i < Lo.nslot; ++i) {
            mbar_init(&s.full[i], 1);
            mbar_init(&s.empty[i], SK_CW);         // every consumer warp's share of a release
            s.sh->slot_seq[i] = 0u;
        }
        mbar_init(&s.sh->route_bar, 1);
        s.sh->abort = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (warp == SK_CW)
        sk_producer<NV>(s, lane);
    else
        sk_consumers<NV>(s, warp, lane);
}

}  // namespace

cudaError_t stack_decode_set_attributes(int max_optin) {
    const cudaError_t e =
        cudaFuncSetAttribute(stack_decode_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_optin);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(stack_decode_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, max_optin);
}

cudaError_t launch_stack_decode(const LaunchCtx& L, StackParams& p, int max_optin) {
    if (p.T < 1 || p.T > STACK_MAX_T || p.n_layers < 1 || p.n_layers > STACK_MAX_LAYERS) return cudaErrorInvalidValue;
    if (L.num_sms < SK_DN_ITEMS || L.num_sms > E) return cudaErrorInvalidValue;
    p.smem_bytes = (uint32_t)max_optin;
    const bool nv = p.nvfp4 != 0;
    const SkLayout Lo = sk_layout(p.T, (uint32_t)max_optin, nv);
    if (Lo.nslot < (nv ? 16 : 6)) return cudaErrorInvalidValue;
    if (nv)
        return launch_hooked(L, FLINT_KERNEL_GATE_UP, stack_decode_kernel<true>, dim3(L.num_sms), dim3(SK_THREADS),
                             Lo.total, p);
    return launch_hooked(L, FLINT_KERNEL_GATE_UP, stack_decode_kernel<false>, dim3(L.num_sms), dim3(SK_THREADS),
                         Lo.total, p);
}

}  // namespace flint
