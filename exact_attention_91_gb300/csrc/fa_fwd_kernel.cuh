// Attention forward, warp-specialised persistent kernel for sm_103a, for
// equal-length batches [B, H, N, d] and for batches of sequences with their
// own query and key counts (token-major [total, H, d]); the two differ only
// in compile-time branches (VARLEN) on coordinates, masks and the epilogue.
//
// One CTA per SM loops over work items. A unit is one head (of one sequence)
// and a block of 256 query rows, held as two 128-row tiles (t = 0, 1) that
// share every K/V tile the CTA streams through shared memory. The tensor core
// alternates between the two tiles, so the softmax of one tile runs while the
// MMAs of the other are in flight. A work item is a whole unit, or:
//   * (equal length) a half unit: one 128-row tile whose key tiles the two
//     softmax warpgroups share out (even ones to tile 0, odd ones to tile
//     1); their results are merged inside the CTA at the end. The last units
//     of a non-causal launch run this way when a last wave of whole units
//     would leave most SMs idle, and every unit of a causal launch with at
//     most half as many units as SMs. Only the instantiation with HALF set
//     holds this code: carried unused, its branches cost the d = 128 kernel
//     3-5% of its throughput.
//   * (variable length, few units) one share of a unit's key tiles; the
//     shares of a unit run on the CTAs of one thread-block cluster and are
//     merged through distributed shared memory.
// Neither needs memory beyond the kernel's inputs and outputs.
//
// Roles (12 warps):
//   warps 0-3  softmax of tile 0    (one query row per thread, TMEM lanes 0-127)
//   warps 4-7  softmax of tile 1
//   warp  8    issues every S = Q·Kᵀ MMA; TMEM allocation
//   warp  9    TMA loads, the work queue, barrier initialisation
//   warp  10   issues the P·V MMAs of tile 0
//   warp  11   issues the P·V MMAs of tile 1
// (warps 8-11 form the control warpgroup, which gives registers to the
// softmax warpgroups; each control warp runs its loop as a whole warp and one
// elected lane issues each copy or MMA)
// The roles are chosen before anything else runs, so no value is live across
// the register split; each role derives its addresses from the kernel
// parameters and shared memory.
//
// Per key tile j and query tile t ("Mini FlashAttention", §4 "The flash trick:
// online softmax"; "How Did I Write My First FlashAttention Kernel in CUDA?",
// pseudo-algorithm steps 3-5):
//   S_t  = Q_t·K_jᵀ                      tcgen05.mma -> TMEM (fp32)
//   m̃    = rowmax(S_t)·c                  c = scale·log2(e) (base-2 units)
//   if m̃ > m_ref + τ:  α = 2^(m_ref - m̃), m_ref = m̃, O_t ·= α, l ·= α
//   p    = 2^(S_t·c - m_ref),  l += Σp
//   O_t += bf16(p)·V_j                    tcgen05.mma, A = P from TMEM
// and after the last key tile O = O_t / l, LSE = ln2·(m_ref + log2 l). The
// reference max m_ref only moves when the row max rises by more than τ (in
// base-2 units); O_t and l are always relative to the same m_ref, so the
// final O/l is unchanged while O_t·2^τ stays far from fp32 overflow. τ = 0 is
// the rule "rescale whenever the max moves". τ = 32: P is bf16, whose range
// holds 2^32 with the same relative rounding as 1, and O_t, l <= 2^32 · N ·
// max|V| stay far inside fp32, so a row rescales O only when its max jumps by
// 32 (2^32 in p): rarely even for spiky scores. Two partial results over
// disjoint key sets, (m_a, l_a, O_a) and (m_b, l_b, O_b), combine the same
// way: O = (2^(m_a-m) O_a + 2^(m_b-m) O_b) / (2^(m_a-m) l_a + 2^(m_b-m) l_b).
#pragma once

#include "fa_common.cuh"

namespace fa {

// Named barrier with an OR-reduction over a predicate (subset of the CTA).
__device__ __forceinline__ bool named_bar_or(uint32_t id, uint32_t nthreads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "bar.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"(pred ? 1u : 0u), "r"(id), "r"(nthreads)
        : "memory");
    return r != 0;
}

template <int D>
struct WsCfg {
    static constexpr int kThreads = 384;
    static constexpr int kTileBytes = D * kBlockM * 2;       // one 128 x D bf16 tile
    static constexpr int kStages = D == 128 ? 4 : 8;        // K/V ring slots
    static constexpr int kOffQ = 0;                          // Q0, Q1
    static constexpr int kOffRing = kOffQ + 2 * kTileBytes;
    static constexpr int kOffStage = kOffRing + kStages * kTileBytes;  // O staging, one box per tile
    static constexpr int kOffBar = kOffStage + 2 * kBoxBytes;
    static constexpr int kUnitSlots = 4;                     // work items handed from the TMA warp to the others
    // barriers: q_full[2] q_empty[2] kv_full[S] kv_empty[S] s_full[2] p_full[2] o_full[2] fin[3]
    //           u_full[U] u_empty[U] pv_done[2] s_free[2]
    static constexpr int kNumBars = 2 + 2 + 2 * kStages + 2 + 2 + 2 + 3 + 2 * kUnitSlots + 2 + 2;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem slot, abort flag, unit queue, S counts
    static constexpr int kSmemBytes = kOffMisc + 8 + 4 * kUnitSlots + 8 + 1024;  // + base alignment slack
    static constexpr int kTmemCols = 512;
    // TMEM columns. P (bf16 pairs, 64 columns per tile) never overlays S, so
    // no MMA that writes S can race a P·V that is still reading P: tcgen05.mma
    // keeps issue order only between MMAs into the same accumulator.
    //  d = 128: one S buffer shared by the two tiles, used alternately (each
    //           softmax copies S into registers at once); P0, P1, O0, O1.
    //  d = 64:  an S buffer per tile, so S_t(j+1) can be computed as soon as
    //           the softmax has read S_t(j); P0, P1, O0, O1.
    static constexpr bool kSharedS = D == 128;
    // arrivals that free a unit-queue slot: the 3 MMA-issuing warps and the 8 softmax warps
    static constexpr uint32_t kUnitConsumers = 11;
    static constexpr uint32_t kTmemS0 = 0, kTmemS1 = kSharedS ? 0 : 128;
    static constexpr uint32_t kTmemP0 = kSharedS ? 128 : 384, kTmemP1 = kSharedS ? 192 : 448;
    static constexpr uint32_t kTmemO0 = 256, kTmemO1 = 256 + D;
    // Named barriers: 1 + t for softmax warpgroup t; the two softmax
    // warpgroups together (half-item merge, cluster-split hand-over); all 12
    // warps (setup and teardown).
    // kBarSetup: the TMA warp only arrives (it starts its first copies while
    // TMEM is allocated), every other warp waits; a barrier of its own, so
    // that a TMA warp that finishes early cannot count toward it at teardown.
    static constexpr uint32_t kBarPair = 3, kBarPairDone = 4, kBarSetup = 14, kBarAll = 15;
    // The partial results of a cluster split (after the last MMA of the item,
    // when the ring is idle): fp32 O rows [tile][row][D] in the ring, base-2
    // LSE [tile][row] and the CTA's abort flag in the staging area.
    static_assert(2 * kBlockM * D * 4 <= kStages * kTileBytes, "partial O fits the ring");
};

// Shared-memory addresses of one CTA (everything is a fixed offset from the
// 1024-byte aligned base of the dynamic shared memory).
template <int D>
struct WsSmem {
    using Cfg = WsCfg<D>;
    static constexpr int S = Cfg::kStages;
    uint8_t* base;
    uint32_t sbase;
    __device__ __forceinline__ WsSmem() {
        extern __shared__ uint8_t smem_raw[];
        base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
        sbase = ptx::smem_u32(base);
    }
    __device__ __forceinline__ uint32_t bar(int i) const { return sbase + Cfg::kOffBar + 8u * i; }
    __device__ __forceinline__ uint32_t q_full(int t) const { return bar(t); }
    __device__ __forceinline__ uint32_t q_empty(int t) const { return bar(2 + t); }
    __device__ __forceinline__ uint32_t kv_full(int s) const { return bar(4 + s); }
    __device__ __forceinline__ uint32_t kv_empty(int s) const { return bar(4 + S + s); }
    __device__ __forceinline__ uint32_t s_full(int t) const { return bar(4 + 2 * S + t); }
    __device__ __forceinline__ uint32_t p_full(int t) const { return bar(6 + 2 * S + t); }
    __device__ __forceinline__ uint32_t o_full(int t) const { return bar(8 + 2 * S + t); }
    __device__ __forceinline__ uint32_t fin(int m) const { return bar(10 + 2 * S + m); }
    __device__ __forceinline__ uint32_t u_full(int i) const { return bar(13 + 2 * S + i); }
    __device__ __forceinline__ uint32_t u_empty(int i) const { return bar(13 + 2 * S + Cfg::kUnitSlots + i); }
    __device__ __forceinline__ uint32_t pv_done(int t) const { return bar(13 + 2 * S + 2 * Cfg::kUnitSlots + t); }
    __device__ __forceinline__ uint32_t s_free(int t) const { return bar(15 + 2 * S + 2 * Cfg::kUnitSlots + t); }
    __device__ __forceinline__ volatile int* unit_slot(int i) const {
        return reinterpret_cast<volatile int*>(base + Cfg::kOffMisc + 8) + i;
    }
    // per tile: how many S_t MMAs the S warp has issued so far (all items)
    __device__ __forceinline__ volatile uint32_t* s_issued(int t) const {
        return reinterpret_cast<volatile uint32_t*>(base + Cfg::kOffMisc + 8 + 4 * Cfg::kUnitSlots) + t;
    }
    __device__ __forceinline__ uint32_t* tmem_slot() const {
        return reinterpret_cast<uint32_t*>(base + Cfg::kOffMisc);
    }
    __device__ __forceinline__ volatile int* abort_flag() const {
        return reinterpret_cast<volatile int*>(base + Cfg::kOffMisc + 4);
    }
    __device__ __forceinline__ uint32_t q_tile(int t) const { return sbase + Cfg::kOffQ + t * Cfg::kTileBytes; }
    __device__ __forceinline__ uint32_t ring(uint32_t cnt) const {
        return sbase + Cfg::kOffRing + (cnt % S) * Cfg::kTileBytes;
    }
    __device__ __forceinline__ uint8_t* stage(int t) const { return base + Cfg::kOffStage + t * kBoxBytes; }
    // cluster split: this CTA's partial O row (fp32 [D]) and base-2 LSE of (tile, row), its abort flag
    __device__ __forceinline__ float* part_o(int t, int row) const {
        return reinterpret_cast<float*>(base + Cfg::kOffRing) + (t * kBlockM + row) * D;
    }
    __device__ __forceinline__ float* part_lse(int t, int row) const {
        return reinterpret_cast<float*>(base + Cfg::kOffStage) + t * kBlockM + row;
    }
    __device__ __forceinline__ int* part_abort() const {
        return reinterpret_cast<int*>(base + Cfg::kOffStage) + 2 * kBlockM;
    }
};

// Unit u -> (head, 256-row query block). CTAs claim items in increasing
// order from a global counter as they free up. Heads are taken in groups of
// 16 so that the units in flight at any moment share few heads and their K/V
// tiles stay in L2; inside a group the blocks with the most key tiles come
// first, so the lightest units fill the tail.
__device__ __forceinline__ void unit_coords(int u, int nqb, int BH, int& bh, int& qb) {
    constexpr int kGroup = 16;
    const int per_group = kGroup * nqb;
    const int g = u / per_group;
    const int hg = min(kGroup, BH - g * kGroup);
    const int idx = u - g * per_group;
    qb = nqb - 1 - idx / hg;
    bh = g * kGroup + idx % hg;
}

// Key tiles query tile `q_tile` visits in a sequence of nq queries and nk keys
// whose causal mask is aligned at the end (query i sees keys j <= i + nk - nq):
// none when the tile holds no query; every one without the causal mask; else
// up to the last key that its last query sees.
template <bool CAUSAL>
__device__ __forceinline__ int kv_tiles(int q_tile, int nq, int nk) {
    const int i0 = q_tile * kBlockM;
    if (i0 >= nq) return 0;
    const int n_k = (nk + kBlockN - 1) / kBlockN;
    if (!CAUSAL) return n_k;
    const int kmax = min(i0 + kBlockM - 1, nq - 1) + nk - nq;
    return kmax < 0 ? 0 : min(kmax / kBlockN + 1, n_k);
}

// A work item, as every role sees it. Ring step j loads key tile jb + j; tile
// t uses step j when uses(t, j), as the use_index(j)-th of its n_t key tiles.
struct Item {
    int bh;          // b*H + h
    int head;        // h (variable length: the tensor maps' head coordinate)
    int tq0, tk0;    // variable length: first query / key token of the sequence
    int nq, nk;      // queries and keys of the sequence
    int qr0, qr1;    // first query row of tile 0 / tile 1 within the sequence
    int n0, n1;      // key tiles tile 0 / tile 1 visit
    int n_load;      // ring steps
    int jb;          // key tile of ring step 0
    bool half;       // both tiles hold the same queries; tile t takes the steps j with j % 2 == t
    __device__ __forceinline__ int n(int t) const { return t ? n1 : n0; }
    __device__ __forceinline__ int qr(int t) const { return t ? qr1 : qr0; }
    __device__ __forceinline__ bool uses(int t, int j) const { return half ? (j & 1) == t : j < n(t); }
    __device__ __forceinline__ int use_index(int j) const { return half ? j >> 1 : j; }
    __device__ __forceinline__ int key_tile(int t, int i) const { return half ? 2 * i + t : jb + i; }
};

template <bool CAUSAL, bool VARLEN, bool HALF>
__device__ __forceinline__ Item item_coords(int u, const FwdParams& p) {
    Item w;
    w.jb = 0;
    int qb;
    if constexpr (!VARLEN) {
        int unit = u, ht = 0;
        w.half = HALF && u >= p.n_full;
        if (w.half) {
            const int h = u - p.n_full;
            unit = p.n_full + (h >> 1);
            ht = h & 1;
        }
        unit_coords(unit, p.nqb, p.num_heads_total, w.bh, qb);
        w.head = 0;
        w.tq0 = w.tk0 = 0;
        w.nq = w.nk = p.N;
        if (!w.half) {
            w.qr0 = qb * 2 * kBlockM;
            w.qr1 = w.qr0 + kBlockM;
            w.n0 = kv_tiles<CAUSAL>(2 * qb, p.N, p.N);
            w.n1 = kv_tiles<CAUSAL>(2 * qb + 1, p.N, p.N);  // 0: tile 1 lies past the end of the head
            w.n_load = max(w.n0, w.n1);
        } else {
            // the tile's visible key tiles (all of them without the causal mask),
            // the even ones to tile 0's warpgroup and the odd ones to tile 1's
            const int nv = kv_tiles<CAUSAL>(2 * qb + ht, p.N, p.N);
            w.qr0 = w.qr1 = (2 * qb + ht) * kBlockM;
            w.n0 = (nv + 1) >> 1;
            w.n1 = nv >> 1;
            w.n_load = nv;
        }
    } else {
        const int unit = p.nsplit == 1 ? u : u / p.nsplit;
        const int split = u - unit * p.nsplit;
        unit_coords(unit, p.nqb, p.num_heads_total, w.bh, qb);
        const int b = w.bh / p.heads;
        w.head = w.bh - b * p.heads;
        w.half = false;
        w.tq0 = p.cu_q[b];
        w.nq = p.cu_q[b + 1] - w.tq0;
        w.tk0 = p.cu_k[b];
        w.nk = p.cu_k[b + 1] - w.tk0;
        w.qr0 = qb * 2 * kBlockM;
        w.qr1 = w.qr0 + kBlockM;
        w.n0 = kv_tiles<CAUSAL>(2 * qb, w.nq, w.nk);
        w.n1 = kv_tiles<CAUSAL>(2 * qb + 1, w.nq, w.nk);
        w.n_load = max(w.n0, w.n1);
        if (p.nsplit > 1) {
            // split s takes the s-th of nsplit contiguous shares of the key
            // tiles the unit loads; a tile that sees fewer keys takes what of
            // its own range falls there
            const int je = (split + 1) * w.n_load / p.nsplit;
            w.jb = split * w.n_load / p.nsplit;
            w.n0 = max(0, min(je, w.n0) - w.jb);
            w.n1 = max(0, min(je, w.n1) - w.jb);
            w.n_load = max(w.n0, w.n1);
        }
    }
    return w;
}

// Next item of this CTA from the unit queue (consumer side): waits for queue
// slot `it`, reads it, and frees the slot (one arrival per warp, after all
// lanes have read). Returns -1 when the CTA has no more work, and -2 if the
// wait gave up.
template <int D>
__device__ __forceinline__ int next_unit(const WsSmem<D>& sm, int it, int lane, const FwdParams& p) {
    constexpr int U = WsCfg<D>::kUnitSlots;
    const int slot = it % U;
    bool ok = wait_phase(sm.u_full(slot), (it / U) & 1, sm.abort_flag(), kStatusTimeoutOther, p.wait_limit_ns);
    ok = __all_sync(0xffffffffu, ok);
    if (!ok) return -2;
    const int u = *sm.unit_slot(slot);
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(sm.u_empty(slot));
    return u;
}

// Claims the next item (one lane): from the global counter, or, in a cluster
// split, the CTA's own item once. Variable length: a block that starts past
// the end of its sequence is no work and is passed over.
template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ int claim_item(const FwdParams& p, int it) {
    if (p.sched == nullptr) {
        if (it > 0) return -1;
        const int u = static_cast<int>(blockIdx.x);
        if constexpr (VARLEN) {
            const Item c = item_coords<CAUSAL, VARLEN, false>(u, p);
            if (c.qr0 >= c.nq) return -1;
        }
        return u;
    }
    for (;;) {
        const int u = static_cast<int>(atomicAdd(p.sched, 1u));
        if (u >= p.n_items) return -1;
        if constexpr (!VARLEN) return u;
        const Item c = item_coords<CAUSAL, VARLEN, false>(u, p);
        if (c.qr0 < c.nq) return u;
    }
}

// Tensor-map coordinates (y, z) of row `row` of the item's queries / keys.
template <bool VARLEN>
__device__ __forceinline__ void q_coords(const Item& w, int row, int& y, int& z) {
    if constexpr (VARLEN) {
        y = w.head;
        z = w.tq0 + row;
    } else {
        y = row;
        z = w.bh;
    }
}
template <bool VARLEN>
__device__ __forceinline__ void k_coords(const Item& w, int row, int& y, int& z) {
    if constexpr (VARLEN) {
        y = w.head;
        z = w.tk0 + row;
    } else {
        y = row;
        z = w.bh;
    }
}

// ---------------------------------------------------------------- TMA producer
// Run by the whole warp: addresses and coordinates stay warp-uniform and one
// elected lane issues each copy.
template <int D, bool CAUSAL, bool VARLEN, bool HALF>
__device__ __forceinline__ void load_role(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                          const CUtensorMap& tm_v, const FwdParams& p, int lane) {
    using Cfg = WsCfg<D>;
    constexpr int S = Cfg::kStages;
    const WsSmem<D> sm;
    volatile int* abort_flag = sm.abort_flag();
    const unsigned long long lim = p.wait_limit_ns;
    if (lane == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
    }
    const uint64_t keep = ptx::policy_evict_last();
    const uint64_t stream_once = ptx::policy_evict_first();
    constexpr int U = Cfg::kUnitSlots;
    uint32_t kv_cnt = 0;
    bool ok = true;
    for (int it = 0; ok; ++it) {
        // claim the next item and hand it to the other roles
        const int qslot = it % U;
        ok = wait_phase_warp(sm.u_empty(qslot), ((it / U) & 1) ^ 1, abort_flag, kStatusTimeoutOther, lim);
        if (!ok) break;
        int u = 0;
        if (lane == 0) {
            u = claim_item<CAUSAL, VARLEN>(p, it);
            *sm.unit_slot(qslot) = u;
            ptx::mbar_arrive(sm.u_full(qslot));
        }
        u = __shfl_sync(0xffffffffu, u, 0);
        if (u < 0) break;
        const Item w = item_coords<CAUSAL, VARLEN, HALF>(u, p);
        for (int t = 0; t < 2 && ok; ++t) {
            ok = wait_phase_warp(sm.q_empty(t), (it & 1) ^ 1, abort_flag, kStatusTimeoutFree, lim);
            if (!ok) break;
            ptx::mbar_arrive_expect_tx_elect(sm.q_full(t), Cfg::kTileBytes);
            int y, z;
            q_coords<VARLEN>(w, w.qr(t), y, z);
#pragma unroll
            for (int c = 0; c < D / kBoxCols; ++c)
                ptx::tma_load_3d_hint_elect(sm.q_tile(t) + c * kBoxBytes, &tm_q, sm.q_full(t), c * kBoxCols, y, z,
                                            stream_once);
        }
        for (int j = 0; j < w.n_load && ok; ++j) {
            int y, z;
            k_coords<VARLEN>(w, (w.jb + j) * kBlockN, y, z);
            for (int which = 0; which < 2; ++which, ++kv_cnt) {
                const int slot = static_cast<int>(kv_cnt % S);
                ok = wait_phase_warp(sm.kv_empty(slot), ((kv_cnt / S) & 1) ^ 1, abort_flag, kStatusTimeoutFree,
                                     lim);
                if (!ok) break;
                ptx::mbar_arrive_expect_tx_elect(sm.kv_full(slot), Cfg::kTileBytes);
                const CUtensorMap* map = which == 0 ? &tm_k : &tm_v;
#pragma unroll
                for (int c = 0; c < D / kBoxCols; ++c)
                    ptx::tma_load_3d_hint_elect(sm.ring(kv_cnt) + c * kBoxBytes, map, sm.kv_full(slot),
                                                c * kBoxCols, y, z, keep);
            }
        }
    }
}

// ---------------------------------------------------------------- MMA issuers
// Three warps issue the tcgen05.mma work: one issues every S = Q·Kᵀ (both
// tiles, in the order S0(0), S1(0), S0(1), S1(1), ...), and one per tile
// issues that tile's O += P·V. Issuing a tcgen05.mma costs the issuing warp
// tens of cycles, so one warp alone cannot keep the tensor core busy while it
// also waits on the softmax; split three ways, each warp's share of the issue
// and barrier work fits in the time the tensor core spends on its MMAs.
// Every warp runs its loop whole: descriptors stay warp-uniform and one
// elected lane issues each tcgen05.mma / tcgen05.commit.

// S_t = Q_t·K_jᵀ for the tiles that use ring step j, one step after the
// other. An S buffer is rewritten only after the softmax has read (s_free)
// everything written there before; with d = 128 both tiles share one buffer,
// so S1 follows the read of S0 and the next S0 the read of S1. K slots are
// released here.
template <int D, bool CAUSAL, bool VARLEN, bool HALF>
__device__ __forceinline__ void s_role(const FwdParams& p, int lane) {
    using Cfg = WsCfg<D>;
    constexpr int S = Cfg::kStages;
    constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(128, kBlockN, false, false);
    const WsSmem<D> sm;
    volatile int* abort_flag = sm.abort_flag();
    const unsigned long long lim = p.wait_limit_ns;
    const uint32_t tmem = *sm.tmem_slot();
    // S_t over D in steps of 16 (4 steps of 32 bytes per 64-wide box).
    // Descriptors advance by adding the byte offset >> 4 to the start-address field.
    auto issue_s = [&](int t, uint32_t sK) {
        const uint64_t a0 = ptx::sdesc_sw128(sm.q_tile(t), 16, 1024);
        const uint64_t b0 = ptx::sdesc_sw128(sK, 16, 1024);
        const uint32_t tS = tmem + (t == 0 ? Cfg::kTmemS0 : Cfg::kTmemS1);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = static_cast<uint32_t>(((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4);
            ptx::mma_ss_elect(tS, a0 + off, b0 + off, kIdescS, kk > 0 ? 1u : 0u);
        }
    };
    // S MMAs issued / softmax reads seen, per S buffer (one shared buffer with d = 128)
    uint32_t s_cnt0 = 0, s_cnt1 = 0, sf_seen0 = 0, sf_seen1 = 0;
    uint32_t s_iss0 = 0, s_iss1 = 0;  // S_0 / S_1 issued (differ from s_cnt with the shared buffer)
    bool ok = true;
    auto issue_s_safe = [&](int t, uint32_t sK) {
        const int b = Cfg::kSharedS ? 0 : t;
        uint32_t& seen = b == 0 ? sf_seen0 : sf_seen1;
        uint32_t& issued = b == 0 ? s_cnt0 : s_cnt1;
        while (ok && seen < issued) {
            ok = wait_phase_warp(sm.s_free(b), seen & 1, abort_flag, kStatusTimeoutSoftmax, lim);
            ++seen;
        }
        if (!ok) return false;
        ptx::tc_fence_after_sync();
        issue_s(t, sK);
        ++issued;
        ptx::mma_commit_elect(sm.s_full(t));
        uint32_t& n_iss = t == 0 ? s_iss0 : s_iss1;
        ++n_iss;
        if (lane == 0) *sm.s_issued(t) = n_iss;
        return true;
    };
    uint32_t kv_cnt = 0;
    for (int it = 0; ok; ++it) {
        const int u = next_unit(sm, it, lane, p);
        if (u < 0) break;
        const Item w = item_coords<CAUSAL, VARLEN, HALF>(u, p);
        if (!wait_phase_warp(sm.q_full(0), it & 1, abort_flag, kStatusTimeoutLoad, lim)) break;
        if (!wait_phase_warp(sm.q_full(1), it & 1, abort_flag, kStatusTimeoutLoad, lim)) break;
        // a tile that sees no key still hands its Q buffer back
        if (w.n0 == 0) ptx::mma_commit_elect(sm.q_empty(0));
        if (w.n1 == 0) ptx::mma_commit_elect(sm.q_empty(1));
        for (int j = 0; j < w.n_load; ++j) {
            const uint32_t k = kv_cnt + 2u * j;  // ring position of K_j
            ok = wait_phase_warp(sm.kv_full(k % S), (k / S) & 1, abort_flag, kStatusTimeoutLoad, lim);
            if (!ok) break;
            for (int t = 0; t < 2; ++t) {
                if (!w.uses(t, j)) continue;
                if (!issue_s_safe(t, sm.ring(k))) break;
                if (w.use_index(j) == w.n(t) - 1) ptx::mma_commit_elect(sm.q_empty(t));
            }
            if (!ok) break;
            ptx::mma_commit_elect(sm.kv_empty(k % S));
        }
        kv_cnt += 2u * w.n_load;
    }
}

// O_t += P_t·V_j for tile t, once the softmax has written P_t(j); the commit
// after each one (pv_done) tells the softmax when it may overwrite P_t or
// rescale O_t. V slots are released by both P·V warps (two arrivals); the
// ring steps tile t does not use are released without use, after their load,
// so that the arrival lands in the slot's current use.
template <int D, bool CAUSAL, bool VARLEN, bool HALF>
__device__ __forceinline__ void pv_role(const FwdParams& p, int lane, int t) {
    using Cfg = WsCfg<D>;
    constexpr int S = Cfg::kStages;
    constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(128, D, false, true);
    const WsSmem<D> sm;
    volatile int* abort_flag = sm.abort_flag();
    const unsigned long long lim = p.wait_limit_ns;
    const uint32_t tmem = *sm.tmem_slot();
    const uint32_t tP = tmem + (t == 0 ? Cfg::kTmemP0 : Cfg::kTmemP1);
    const uint32_t tO = tmem + (t == 0 ? Cfg::kTmemO0 : Cfg::kTmemO1);
    // 128 keys in steps of 16 (2048 bytes of V each); V is MN-major: 64-wide
    // swizzle atoms 16 KB apart (LBO), 8-key groups 1 KB apart (SBO).
    auto issue_pv = [&](uint32_t sV, bool accumulate) {
        const uint64_t b0 = ptx::sdesc_sw128(sV, kBoxBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk) {
            ptx::mma_ts_elect(tO, tP + kk * 8, b0 + static_cast<uint32_t>(kk * (2048 >> 4)), kIdescPV,
                              (accumulate || kk > 0) ? 1u : 0u);
        }
    };
    uint32_t kv_cnt = 0, p_cnt = 0;
    uint32_t s_base = 0;  // S_t MMAs of earlier items
    volatile uint32_t* s_issued = sm.s_issued(t);
    bool ok = true;
    for (int it = 0; ok; ++it) {
        const int u = next_unit(sm, it, lane, p);
        if (u < 0) break;
        const Item w = item_coords<CAUSAL, VARLEN, HALF>(u, p);
        const int n_t = w.n(t);
        if (n_t == 0) ptx::mma_commit_elect(sm.o_full(t));  // nothing to add: O is all zero
        for (int j = 0; j < w.n_load; ++j) {
            const uint32_t v = kv_cnt + 2u * j + 1u;  // ring position of V_j
            ok = wait_phase_warp(sm.kv_full(v % S), (v / S) & 1, abort_flag, kStatusTimeoutLoad, lim);
            if (!ok) break;
            if (w.uses(t, j)) {
                const int i = w.use_index(j);
                ok = wait_phase_warp(sm.p_full(t), p_cnt & 1, abort_flag, kStatusTimeoutSoftmax, lim);
                ++p_cnt;
                if (!ok) break;
                // The softmax waits for the tile's next S before it needs this
                // P·V, so that S goes to the tensor core first: wait (briefly;
                // this is only an ordering preference) until the S warp has
                // issued it.
                if (i + 1 < n_t) {
                    const uint32_t want = s_base + static_cast<uint32_t>(i) + 2u;
                    for (int spin = 0; spin < 2000 && *s_issued < want; ++spin) __nanosleep(32);
                }
                ptx::tc_fence_after_sync();
                issue_pv(sm.ring(v), i > 0);
                ptx::mma_commit_elect(sm.pv_done(t));
                if (i == n_t - 1) ptx::mma_commit_elect(sm.o_full(t));
                ptx::mma_commit_elect(sm.kv_empty(v % S));
            } else if (lane == 0) {
                ptx::mbar_arrive(sm.kv_empty(v % S));
            }
        }
        kv_cnt += 2u * w.n_load;
        s_base += static_cast<uint32_t>(n_t);
    }
}

// Loads 64 consecutive TMEM columns of this thread's lane into f[0..63].
__device__ __forceinline__ void load_row64(uint32_t taddr, float (&f)[64]) {
    uint32_t ra[32], rb[32];
    ptx::tmem_ld_32x32b_x32(taddr, ra);
    ptx::tmem_ld_32x32b_x32(taddr + 32, rb);
    ptx::tmem_wait_ld(ra);
    ptx::reg_fence(rb);
#pragma unroll
    for (int i = 0; i < 32; ++i) {
        f[i] = __uint_as_float(ra[i]);
        f[32 + i] = __uint_as_float(rb[i]);
    }
}

// 64 fp32 values -> bf16 -> one 16-byte chunk each 8 values, through `store`.
template <class Store>
__device__ __forceinline__ void pack_row64(const float (&f)[64], Store&& store) {
#pragma unroll
    for (int q8 = 0; q8 < 8; ++q8) {
        uint4 v;
        v.x = ptx::pack_bf16x2(f[q8 * 8 + 0], f[q8 * 8 + 1]);
        v.y = ptx::pack_bf16x2(f[q8 * 8 + 2], f[q8 * 8 + 3]);
        v.z = ptx::pack_bf16x2(f[q8 * 8 + 4], f[q8 * 8 + 5]);
        v.w = ptx::pack_bf16x2(f[q8 * 8 + 6], f[q8 * 8 + 7]);
        store(q8, v);
    }
}

// ---------------------------------------------------------------- softmax + epilogue
template <int D, bool CAUSAL, bool VARLEN, bool HALF>
__device__ __forceinline__ void softmax_role(const CUtensorMap& tm_o, const FwdParams& p, int warp, int lane) {
    using Cfg = WsCfg<D>;
    constexpr float kTau = 32.0f;
    const WsSmem<D> sm;
    volatile int* abort_flag = sm.abort_flag();
    const unsigned long long lim = p.wait_limit_ns;
    const uint32_t tmem = *sm.tmem_slot();
    const int t = warp >> 2;                 // query tile of this warpgroup
    const int row = (warp & 3) * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + (t == 0 ? Cfg::kTmemS0 : Cfg::kTmemS1) + lane_base;
    const uint32_t tO = tmem + (t == 0 ? Cfg::kTmemO0 : Cfg::kTmemO1) + lane_base;
    const uint32_t tP = tmem + (t == 0 ? Cfg::kTmemP0 : Cfg::kTmemP1) + lane_base;
    uint8_t* stage = sm.stage(t);
    const uint32_t stage_s = ptx::smem_u32(stage);
    const float c_log2 = p.scale_log2;
    uint32_t s_cnt = 0;
    uint32_t p_made = 0, pv_seen = 0;  // P tiles written / P·V completions observed
    bool failed = false;
    for (int it = 0;; ++it) {
        const int u = next_unit(sm, it, lane, p);
        if (u == -2) failed = true;
        if (named_bar_or(1 + t, 128, u < 0)) break;  // the warpgroup agrees on stopping
        const Item w = item_coords<CAUSAL, VARLEN, HALF>(u, p);
        const int qr = w.qr(t);  // first query row of this tile within its sequence
        const int n_t = w.n(t);
        float m_ref = -INFINITY;  // reference max (base 2) that O and l are relative to
        float l = 0.f;
        for (int i = 0; i < n_t; ++i) {
            bool ok = wait_phase(sm.s_full(t), s_cnt & 1, abort_flag, kStatusTimeoutMma, lim);
            ++s_cnt;
            if (!__all_sync(0xffffffffu, ok)) {
                failed = true;
                break;
            }
            ptx::tc_fence_after_sync();
            // this thread's row of S, all four loads in flight at once; S is free for the next MMA once they land
            float s[kBlockN];
            float mx0, mx1, mx2, mx3;
            const int key0 = w.key_tile(t, i) * kBlockN;  // first key of this tile within the sequence
            // key j is visible to query q when j < nk and (causal) j <= q + nk - nq
            const int nk = VARLEN ? w.nk : p.N, off = VARLEN ? w.nk - w.nq : 0;
            const bool need_mask = key0 + kBlockN > nk || (CAUSAL && key0 + kBlockN - 1 > qr + off);
            int last = nk - 1 - key0;  // last visible column of this tile
            if (CAUSAL && need_mask) last = min(last, qr + row + off - key0);
            {
                uint32_t r0[32], r1[32], r2[32], r3[32];
                ptx::tmem_ld_32x32b_x32(tS + 0, r0);
                ptx::tmem_ld_32x32b_x32(tS + 32, r1);
                ptx::tmem_ld_32x32b_x32(tS + 64, r2);
                ptx::tmem_ld_32x32b_x32(tS + 96, r3);
                ptx::tmem_wait_ld(r0);
                ptx::reg_fence(r1);
                ptx::reg_fence(r2);
                ptx::reg_fence(r3);
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    s[c] = __uint_as_float(r0[c]);
                    s[32 + c] = __uint_as_float(r1[c]);
                    s[64 + c] = __uint_as_float(r2[c]);
                    s[96 + c] = __uint_as_float(r3[c]);
                }
            }
            // S is in registers: the S warp may write the next S into its buffer
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(sm.s_free(Cfg::kSharedS ? 0 : t));
            if (need_mask) {
#pragma unroll
                for (int c = 0; c < kBlockN; ++c) s[c] = (c > last) ? -INFINITY : s[c];
            }
            mx0 = fmaxf(s[0], s[1]), mx1 = fmaxf(s[2], s[3]), mx2 = fmaxf(s[4], s[5]), mx3 = fmaxf(s[6], s[7]);
#pragma unroll
            for (int c = 8; c < kBlockN; c += 8) {
                mx0 = ptx::fmax3(mx0, s[c], s[c + 1]);
                mx1 = ptx::fmax3(mx1, s[c + 2], s[c + 3]);
                mx2 = ptx::fmax3(mx2, s[c + 4], s[c + 5]);
                mx3 = ptx::fmax3(mx3, s[c + 6], s[c + 7]);
            }
            const float m_tile = fmaxf(ptx::fmax3(mx0, mx1, mx2), mx3) * c_log2;
            const bool move = m_tile > m_ref + kTau;
            float alpha = 1.f;
            if (move) {
                alpha = ptx::ex2_approx(m_ref - m_tile);  // 0 on the first visible tile
                m_ref = m_tile;
            }
            {
                // the P·V of every earlier P of this tile must be done before P and O are touched
                bool okp = true;
                while (okp && pv_seen < p_made) {
                    okp = wait_phase(sm.pv_done(t), pv_seen & 1, abort_flag, kStatusTimeoutMma, lim);
                    ++pv_seen;
                }
                if (!__all_sync(0xffffffffu, okp)) {
                    failed = true;
                    break;
                }
                ptx::tc_fence_after_sync();
            }
            // O_t *= alpha (every P·V into O_t so far is done).
            if (i > 0 && __any_sync(0xffffffffu, move)) {
#pragma unroll 1
                for (int c = 0; c < D / 8; ++c) {
                    uint32_t r[8];
                    ptx::tmem_ld_32x32b_x8(tO + c * 8, r);
                    ptx::tmem_wait_ld(r);
#pragma unroll
                    for (int e = 0; e < 8; ++e) r[e] = __float_as_uint(__uint_as_float(r[e]) * alpha);
                    ptx::tmem_st_32x32b_x8(tO + c * 8, r);
                }
            }
            const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;  // fully masked row stays finite
            const float2 cc = make_float2(c_log2, c_log2), mm = make_float2(-m_use, -m_use);
            // p = 2^(S·c - m) over the whole row in three passes (exponent
            // arguments as packed fp32 pairs, the exponentials, then the sums
            // in four packed chains with the bf16 pairs of P, one 32-column
            // store per 64 keys): each pass is 64-128 independent
            // instructions, which keeps the sub-partition issuing while the
            // results of the previous pass land.
#pragma unroll
            for (int c = 0; c < kBlockN; c += 2) {
                const float2 x = ptx::ffma2(make_float2(s[c], s[c + 1]), cc, mm);
                s[c] = x.x;
                s[c + 1] = x.y;
            }
#pragma unroll
            for (int c = 0; c < kBlockN; ++c) s[c] = ptx::ex2_approx(s[c]);
            float2 sa = make_float2(0.f, 0.f), sb = sa, sc = sa, sd = sa;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                uint32_t r[32];
#pragma unroll
                for (int e = 0; e < 32; e += 4) {
                    const int c = h * 64 + 2 * e;
                    sa = ptx::fadd2(sa, make_float2(s[c], s[c + 1]));
                    sb = ptx::fadd2(sb, make_float2(s[c + 2], s[c + 3]));
                    sc = ptx::fadd2(sc, make_float2(s[c + 4], s[c + 5]));
                    sd = ptx::fadd2(sd, make_float2(s[c + 6], s[c + 7]));
                    r[e] = ptx::pack_bf16x2(s[c], s[c + 1]);
                    r[e + 1] = ptx::pack_bf16x2(s[c + 2], s[c + 3]);
                    r[e + 2] = ptx::pack_bf16x2(s[c + 4], s[c + 5]);
                    r[e + 3] = ptx::pack_bf16x2(s[c + 6], s[c + 7]);
                }
                ptx::tmem_st_32x32b_x32(tP + h * 32, r);
            }
            const float2 sum = ptx::fadd2(ptx::fadd2(sa, sb), ptx::fadd2(sc, sd));
            l = l * alpha + (sum.x + sum.y);
            ptx::tmem_wait_st();
            ptx::tc_fence_before_sync();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(sm.p_full(t));
            ++p_made;
        }

        // ---- epilogue of tile t
        bool ok = !failed && wait_phase(sm.o_full(t), it & 1, abort_flag, kStatusTimeoutMma, lim);
        ok = __all_sync(0xffffffffu, ok);
        // (a half item and a cluster split involve both warpgroups: they agree
        // on going on together, so that neither waits at a barrier the other
        // never reaches)
        const bool pair = w.half || (VARLEN && p.nsplit > 1);
        if (w.half && t == 1) {
            // hand this half's running max and sum to tile 0's warpgroup (tile
            // 1's staging box is not used by a half item, once an earlier
            // store from it has been read)
            if (row == 0) ptx::bulk_wait_group_read0();
            ptx::named_bar_sync(1 + t, 128);
            reinterpret_cast<float*>(stage)[2 * row] = m_ref;
            reinterpret_cast<float*>(stage)[2 * row + 1] = l;
        }
        if (pair ? named_bar_or(Cfg::kBarPair, 256, !ok) : named_bar_or(1 + t, 128, !ok)) {
            failed = true;
            break;
        }
        ptx::tc_fence_after_sync();
        // a query that sees no key (variable length, causal, more queries than
        // keys; or a share of a split that holds none of its keys) gets O = 0
        // and LSE = -inf
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        const bool any_key = l > 0.f;
        float lse2 = any_key ? m_use + log2f(l) : -INFINITY;  // base-2 log-sum-exp of the row's scaled scores
        if constexpr (!VARLEN) {
            // one 64-column box of the final O (fp32 row values f[0..63]) -> bf16 -> staging -> TMA store
            // (the store's read of the staging box is waited for only before
            // the box is written again)
            auto store_box = [&](int b, const float (&f)[64]) {
                if (row == 0) ptx::bulk_wait_group_read0();
                ptx::named_bar_sync(1 + t, 128);
                pack_row64(f, [&](int q8, uint4 v) {
                    *reinterpret_cast<uint4*>(stage + sw128_offset(row, q8)) = v;
                });
                ptx::fence_proxy_async_smem();
                ptx::named_bar_sync(1 + t, 128);
                if (row == 0 && qr < p.N) {  // a tile wholly past the end has nothing to store
                    ptx::tma_store_3d(&tm_o, stage_s, b * kBoxCols, qr, w.bh);
                    ptx::bulk_commit_group();
                }
            };
            if (!w.half) {
                const float inv_l = 1.0f / l;
#pragma unroll
                for (int b = 0; b < D / kBoxCols; ++b) {
                    float o[64];
                    load_row64(tO + b * 64, o);
#pragma unroll
                    for (int e = 0; e < 64; ++e) o[e] *= inv_l;
                    store_box(b, o);
                }
            } else if (t == 1) {
                // tile 0's warpgroup merges; O_1 stays untouched until it has read it
                ptx::named_bar_sync(Cfg::kBarPairDone, 256);
                ptx::tc_fence_after_sync();
                continue;
            } else {
                // merge the two halves: weights 2^(m_h - m) / (sum of 2^(m_h - m) l_h)
                // (a half whose tile sees a single key tile leaves tile 1's
                // warpgroup without keys: m1 = -inf, l1 = 0, and O_1 is not read)
                const bool has1 = w.n1 > 0;
                const float m1 = has1 ? reinterpret_cast<const float*>(sm.stage(1))[2 * row] : -INFINITY;
                const float l1 = has1 ? reinterpret_cast<const float*>(sm.stage(1))[2 * row + 1] : 0.f;
                const float mx = fmaxf(m_ref, m1);
                const float mu = (mx == -INFINITY) ? 0.f : mx;
                const float a0 = ptx::ex2_approx(m_ref - mu), a1 = ptx::ex2_approx(m1 - mu);
                const float lsum = a0 * l + a1 * l1;
                const float inv = 1.0f / lsum;
                const float w0 = a0 * inv, w1 = a1 * inv;
                lse2 = mu + log2f(lsum);
                const uint32_t tO1 = tmem + Cfg::kTmemO1 + lane_base;
#pragma unroll 1
                for (int b = 0; b < D / kBoxCols; ++b) {
                    float o[64];
                    load_row64(tO + b * 64, o);
                    if (has1) {
                        float o1[64];
                        load_row64(tO1 + b * 64, o1);
#pragma unroll
                        for (int e = 0; e < 64; ++e) o[e] = fmaf(w0, o[e], w1 * o1[e]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 64; ++e) o[e] *= w0;
                    }
                    if (b == D / kBoxCols - 1) {
                        // every read of O_1 has landed: tile 1's warpgroup may go on
                        ptx::tc_fence_before_sync();
                        ptx::named_bar_arrive(Cfg::kBarPairDone, 256);
                    }
                    store_box(b, o);
                }
            }
            if (p.lse != nullptr && qr + row < p.N)
                p.lse[static_cast<size_t>(w.bh) * p.N + qr + row] = lse2 * 0.69314718055994531f;
        } else {
            const float inv_l = any_key ? 1.0f / l : 0.f;
            const int q = qr + row;  // query index within the sequence
            // (cu_seqlens are the caller's; a row outside [0, total_q) is never written)
            const bool row_in = q < w.nq && w.tq0 + q >= 0 && w.tq0 + q < p.total_q;
            // this row's O (or, in a cluster split, this share's partial O): fp32 f[0..63] of box b
            auto row_box = [&](int b, float (&f)[64]) {
                if (n_t > 0) {
                    load_row64(tO + b * 64, f);
                } else {
#pragma unroll
                    for (int e = 0; e < 64; ++e) f[e] = 0.f;  // O holds nothing of this item
                }
#pragma unroll
                for (int e = 0; e < 64; ++e) f[e] *= inv_l;
            };
            if (p.nsplit == 1 && qr + kBlockM <= w.nq && w.tq0 + qr >= 0 && w.tq0 + qr + kBlockM <= p.total_q) {
                // a tile wholly inside its sequence: staging box and one TMA
                // store per 64-column box (tm_o is the (d, H, total) view of O)
#pragma unroll
                for (int b = 0; b < D / kBoxCols; ++b) {
                    float o[64];
                    row_box(b, o);
                    if (row == 0) ptx::bulk_wait_group_read0();  // the box's previous store has read it
                    ptx::named_bar_sync(1 + t, 128);
                    pack_row64(o, [&](int q8, uint4 v) {
                        *reinterpret_cast<uint4*>(stage + sw128_offset(row, q8)) = v;
                    });
                    ptx::fence_proxy_async_smem();
                    ptx::named_bar_sync(1 + t, 128);
                    if (row == 0) {
                        ptx::tma_store_3d(&tm_o, stage_s, b * kBoxCols, w.head, w.tq0 + qr);
                        ptx::bulk_commit_group();
                    }
                }
                if (p.lse != nullptr && row_in)
                    p.lse[static_cast<size_t>(w.head) * p.total_q + w.tq0 + q] = lse2 * 0.69314718055994531f;
            } else if (p.nsplit == 1) {
                // 16-byte row stores: a TMA box would run into the next sequence
                uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) +
                                                      (static_cast<size_t>(w.tq0 + q) * p.heads + w.head) * D);
#pragma unroll
                for (int b = 0; b < D / kBoxCols; ++b) {
                    float o[64];
                    row_box(b, o);
                    if (row_in) pack_row64(o, [&](int q8, uint4 v) { dst[b * 8 + q8] = v; });
                }
                if (p.lse != nullptr && row_in)
                    p.lse[static_cast<size_t>(w.head) * p.total_q + w.tq0 + q] = lse2 * 0.69314718055994531f;
            } else {
                // A cluster split: both tiles' MMAs are done (the pair barrier
                // above), so the K/V ring is idle and holds this share's
                // normalised partial O; the merge runs after the roles end.
                float* po = sm.part_o(t, row);
#pragma unroll
                for (int b = 0; b < D / kBoxCols; ++b) {
                    float o[64];
                    row_box(b, o);
                    if (q < w.nq) {
#pragma unroll
                        for (int e = 0; e < 64; e += 4)
                            *reinterpret_cast<float4*>(po + b * 64 + e) = make_float4(o[e], o[e + 1], o[e + 2], o[e + 3]);
                    }
                }
                *sm.part_lse(t, row) = lse2;
            }
        }
        ptx::tc_fence_before_sync();
    }
    if (row == 0) ptx::bulk_wait_group0();
}

// Merge of a cluster split (variable length), run by cluster CTA 0's softmax
// threads after every CTA of the cluster has published its share: thread
// (tile t, row) combines the shares of its query row, O = sum_s w_s O_s with
// w_s = 2^(L_s - L) and L = log2 sum_s 2^(L_s) (base-2 LSEs; a share where the
// row sees no key has L_s = -inf and weight 0), and writes O and the LSE.
template <int D, bool CAUSAL>
__device__ __forceinline__ void cluster_merge(const FwdParams& p, int warp, int lane) {
    constexpr int kMaxSplit = 8;
    const WsSmem<D> sm;
    const int t = warp >> 2;
    const int row = (warp & 3) * 32 + lane;
    const int ns = p.nsplit;
    int aborted = 0;
    for (int s = 0; s < ns; ++s) aborted |= ptx::ld_dsmem_s32(ptx::mapa_shared(ptx::smem_u32(sm.part_abort()), s));
    if (aborted) return;  // a share gave up on a wait (the status word says so): no output
    const Item w = item_coords<CAUSAL, true, false>(static_cast<int>(blockIdx.x), p);
    const int q = w.qr(t) + row;
    if (w.qr0 >= w.nq || q >= w.nq || w.tq0 + q < 0 || w.tq0 + q >= p.total_q) return;
    const uint32_t lse_addr = ptx::smem_u32(sm.part_lse(t, row));
    const uint32_t o_addr = ptx::smem_u32(sm.part_o(t, row));
    float wgt[kMaxSplit];
    float mmax = -INFINITY;
#pragma unroll
    for (int s = 0; s < kMaxSplit; ++s) {
        wgt[s] = s < ns ? ptx::ld_dsmem_f32(ptx::mapa_shared(lse_addr, s)) : -INFINITY;
        mmax = fmaxf(mmax, wgt[s]);
    }
    const bool seen = mmax != -INFINITY;  // the row sees some key in some share
    const float m_w = seen ? mmax : 0.f;
    float wsum = 0.f;
#pragma unroll
    for (int s = 0; s < kMaxSplit; ++s) {
        wgt[s] = ptx::ex2_approx(wgt[s] - m_w);
        wsum += wgt[s];
    }
    const float inv_w = seen ? 1.0f / wsum : 0.f;
    uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) +
                                          (static_cast<size_t>(w.tq0 + q) * p.heads + w.head) * D);
#pragma unroll 1
    for (int c = 0; c < D; c += 8) {
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
        for (int s = 0; s < kMaxSplit; ++s) {
            if (s < ns) {
                const uint32_t a = ptx::mapa_shared(o_addr + c * 4, s);
                const float4 v0 = ptx::ld_dsmem_v4(a), v1 = ptx::ld_dsmem_v4(a + 16);
                const float ws = wgt[s] * inv_w;
                acc[0] = fmaf(ws, v0.x, acc[0]);
                acc[1] = fmaf(ws, v0.y, acc[1]);
                acc[2] = fmaf(ws, v0.z, acc[2]);
                acc[3] = fmaf(ws, v0.w, acc[3]);
                acc[4] = fmaf(ws, v1.x, acc[4]);
                acc[5] = fmaf(ws, v1.y, acc[5]);
                acc[6] = fmaf(ws, v1.z, acc[6]);
                acc[7] = fmaf(ws, v1.w, acc[7]);
            }
        }
        uint4 v;
        v.x = ptx::pack_bf16x2(acc[0], acc[1]);
        v.y = ptx::pack_bf16x2(acc[2], acc[3]);
        v.z = ptx::pack_bf16x2(acc[4], acc[5]);
        v.w = ptx::pack_bf16x2(acc[6], acc[7]);
        dst[c / 8] = v;
    }
    if (p.lse != nullptr)
        p.lse[static_cast<size_t>(w.head) * p.total_q + w.tq0 + q] =
            seen ? (mmax + log2f(wsum)) * 0.69314718055994531f : -INFINITY;
}

// The forward kernel. Equal length: tm_q/k/v/o are (d, N, B*H) views of
// [B, H, N, d]. Variable length: tm_q/k/v/o are (d, H, total) views of
// [total, H, d]; a query tile wholly inside its sequence is stored through
// tm_o, a ragged last tile with plain row stores (a box would run into the
// next sequence).
template <int D, bool CAUSAL, bool VARLEN, bool HALF>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdParams p) {
    using Cfg = WsCfg<D>;
    static_assert(D == 64 || D == 128, "head dim");
    // 384 threads launch with 168 registers each (64512); two softmax
    // warpgroups at 200 and one control warpgroup at 104 use 51200 + 13312.
    constexpr uint32_t kRegsSoftmax = 200, kRegsControl = 104;
    static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsControl <= 384 * 168, "register split");
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int lane = static_cast<int>(threadIdx.x & 31);
    // A kernel launched next with programmatic stream serialization may begin
    // on SMs as this grid leaves them (it waits for this grid before reading
    // O or LSE). Issued at entry, this also measured 1-2% faster on the large
    // workloads with no such kernel following.
    if (threadIdx.x == 0) ptx::griddep_launch_dependents();

    if (warp >= 8) {
        ptx::regs_dec<kRegsControl>();  // the whole control warpgroup (warps 8-11)
        const WsSmem<D> sm;
        if (warp == 8) {
            ptx::tmem_alloc(ptx::smem_u32(sm.tmem_slot()), Cfg::kTmemCols);
            ptx::tmem_relinquish();
        }
        if (warp == 9) {
            // lane i initialises barriers i, i + 32, ...
            for (int i = lane; i < Cfg::kNumBars; i += 32) {
                const uint32_t b = sm.bar(i);
                uint32_t count = 1;
                if (b == sm.p_full(0) || b == sm.p_full(1) || b == sm.s_free(0) || b == sm.s_free(1))
                    count = 4;  // one arrival per softmax warp
                for (int q = 0; q < Cfg::kStages; ++q)  // K slots (even): the S warp; V slots: both P·V warps
                    if (b == sm.kv_empty(q)) count = (q & 1) ? 2 : 1;
                for (int q = 0; q < Cfg::kUnitSlots; ++q)
                    if (b == sm.u_empty(q)) count = Cfg::kUnitConsumers;
                ptx::mbar_init(b, count);
            }
            if (lane == 0) {
                *sm.abort_flag() = 0;
                *sm.s_issued(0) = 0u;
                *sm.s_issued(1) = 0u;
            }
            ptx::fence_mbar_init();
        }
        if (warp == 9) {
            // the barriers and flags this warp uses are its own: it hands them
            // over and starts loading at once
            __syncwarp();
            ptx::named_bar_arrive(Cfg::kBarSetup, Cfg::kThreads);
            load_role<D, CAUSAL, VARLEN, HALF>(tm_q, tm_k, tm_v, p, lane);
            __syncwarp();
        } else {
            ptx::tc_fence_before_sync();
            ptx::named_bar_sync(Cfg::kBarSetup, Cfg::kThreads);
            ptx::tc_fence_after_sync();
            // warp 8: every S; warps 10 and 11: P·V of tile 0 and tile 1
            const int m = warp == 8 ? 0 : warp - 9;
            if (warp == 8)
                s_role<D, CAUSAL, VARLEN, HALF>(p, lane);
            else
                pv_role<D, CAUSAL, VARLEN, HALF>(p, lane, warp - 10);
            __syncwarp();
            // every MMA this warp issued is done before TMEM can be freed
            if (lane == 0) {
                ptx::mma_commit(sm.fin(m));
                wait_drain(sm.fin(m), 0, 100000000ull);
            }
            __syncwarp();
        }
        ptx::tc_fence_before_sync();
        ptx::named_bar_sync(Cfg::kBarAll, Cfg::kThreads);
        if (warp == 9 && lane == 0 && p.sched != nullptr) {
            // every CTA has claimed its last item before it counts itself done,
            // so the last one can put the queue slot back to zero for the next launch
            __threadfence();
            if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
                p.sched[0] = 0u;
                p.sched[1] = 0u;
                __threadfence();
            }
        }
        if (warp == 8) {
            ptx::tc_fence_after_sync();
            ptx::tmem_dealloc(*sm.tmem_slot(), Cfg::kTmemCols);
        }
    } else {
        ptx::regs_inc<kRegsSoftmax>();
        ptx::tc_fence_before_sync();
        ptx::named_bar_sync(Cfg::kBarSetup, Cfg::kThreads);
        ptx::tc_fence_after_sync();
        softmax_role<D, CAUSAL, VARLEN, HALF>(tm_o, p, warp, lane);
        ptx::tc_fence_before_sync();
        ptx::named_bar_sync(Cfg::kBarAll, Cfg::kThreads);
        if (VARLEN && p.nsplit > 1 && threadIdx.x == 0) {
            // every role has ended: whether this CTA gave up on a wait is final
            const WsSmem<D> sm;
            *sm.part_abort() = *sm.abort_flag();
        }
    }
    if constexpr (VARLEN) {
        if (p.nsplit > 1) {
            // every CTA of the cluster has published its share (or gave up);
            // CTA 0 merges, and no CTA exits while another may still read its
            // shared memory
            ptx::cluster_sync();
            if (warp < 8 && ptx::cluster_ctarank() == 0) cluster_merge<D, CAUSAL>(p, warp, lane);
            ptx::cluster_sync();
        }
    }
}

}  // namespace fa
