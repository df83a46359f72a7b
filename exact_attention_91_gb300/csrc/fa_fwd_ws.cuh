// Attention forward, warp-specialised persistent kernel for sm_103a.
//
// One CTA per SM loops over work units. A unit is one head and a block of 256
// query rows, held as two 128-row tiles (t = 0, 1) that share every K/V tile
// the CTA streams through shared memory. The tensor core alternates between
// the two tiles, so the softmax of one tile runs while the MMAs of the other
// are in flight.
//
// Roles (12 warps):
//   warps 0-3  softmax of tile 0    (one query row per thread, TMEM lanes 0-127)
//   warps 4-7  softmax of tile 1
//   warp  8    issues every S = Q·Kᵀ MMA; TMEM allocation
//   warp  9    TMA loads and barrier initialisation
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
// 32 (2^32 in p): rarely even for spiky scores.
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
    static constexpr int kUnitSlots = 4;                     // work units handed from the TMA thread to the others
    // barriers: q_full[2] q_empty[2] kv_full[S] kv_empty[S] s_full[2] p_full[2] o_full[2] fin[3]
    //           u_full[U] u_empty[U] pv_done[2] s_free[2]
    static constexpr int kNumBars = 2 + 2 + 2 * kStages + 2 + 2 + 2 + 3 + 2 * kUnitSlots + 2 + 2;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;  // tmem slot, abort flag, unit queue
    static constexpr int kSmemBytes = kOffMisc + 8 + 4 * kUnitSlots + 8 + 8 + 1024;  // + base alignment slack
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
    // CTA-wide rendezvous of all 12 warps (setup and teardown)
    static constexpr uint32_t kBarAll = 15;
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
    // per softmax warpgroup: "this split is the last of its tile" flag
    // per tile: how many S_t MMAs the S warp has issued so far (all units)
    __device__ __forceinline__ volatile uint32_t* s_issued(int t) const {
        return reinterpret_cast<volatile uint32_t*>(base + Cfg::kOffMisc + 16 + 4 * Cfg::kUnitSlots) + t;
    }
    __device__ __forceinline__ volatile int* last_flag(int t) const {
        return reinterpret_cast<volatile int*>(base + Cfg::kOffMisc + 8 + 4 * Cfg::kUnitSlots) + t;
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
};

// Unit u -> (head, 256-row query block). CTAs claim units in increasing u from
// a global counter as they free up. Heads are taken in groups of 16 so that
// the units in flight at any moment share few heads and their K/V tiles stay
// in L2; inside a group the blocks with the most key tiles come first, so the
// lightest units fill the tail.
__device__ __forceinline__ void unit_coords(int u, int nqb, int BH, int& bh, int& qb) {
    constexpr int kGroup = 16;
    const int per_group = kGroup * nqb;
    const int g = u / per_group;
    const int hg = min(kGroup, BH - g * kGroup);
    const int idx = u - g * per_group;
    qb = nqb - 1 - idx / hg;
    bh = g * kGroup + idx % hg;
}

template <bool CAUSAL>
__device__ __forceinline__ int kv_tiles_for(int q_tile, int n_k_tiles) {
    return CAUSAL ? min(q_tile + 1, n_k_tiles) : n_k_tiles;
}

// Next unit of this CTA from the unit queue (consumer side): waits for queue
// slot `it`, reads it, and frees the slot. `mask` names the calling lanes of
// the warp (all 32 for every caller here); the
// lowest of them arrives once after all have read. Returns -1 when the CTA has
// no more work, and -2 if the wait gave up.
template <int D>
__device__ __forceinline__ int next_unit(const WsSmem<D>& sm, int it, int lane, unsigned mask,
                                         const FwdParams& p) {
    constexpr int U = WsCfg<D>::kUnitSlots;
    const int slot = it % U;
    bool ok = wait_phase(sm.u_full(slot), (it / U) & 1, sm.abort_flag(), kStatusTimeoutOther, p.wait_limit_ns);
    ok = __all_sync(mask, ok);
    if (!ok) return -2;
    const int u = *sm.unit_slot(slot);
    __syncwarp(mask);
    if (lane == __ffs(mask) - 1) ptx::mbar_arrive(sm.u_empty(slot));
    return u;
}

struct WsGeometry {
    int BH, n_k_tiles, nqb, n_units, nsplit, n_items;
    __device__ __forceinline__ explicit WsGeometry(const FwdParams& p) {
        BH = p.num_heads_total;
        n_k_tiles = (p.N + kBlockN - 1) / kBlockN;
        nqb = (p.N + 2 * kBlockM - 1) / (2 * kBlockM);
        n_units = nqb * BH;
        nsplit = p.nsplit;
        n_items = n_units * nsplit;
    }
};

// A work item: one unit (head, 256-row block) and, when the key range is
// split, one contiguous share of its key tiles: tiles jb .. jb+n1-1 (tile 0
// of the unit sees n0 of them, n0 <= n1 <= n0 + 1 under the causal mask).
struct WsItem {
    int unit, split, bh, qb, jb, n0, n1;
};

template <bool CAUSAL>
__device__ __forceinline__ WsItem item_coords(int item, const WsGeometry& g) {
    WsItem w;
    w.unit = item / g.nsplit;
    w.split = item - w.unit * g.nsplit;
    unit_coords(w.unit, g.nqb, g.BH, w.bh, w.qb);
    if (CAUSAL || g.nsplit == 1) {
        w.jb = 0;
        w.n0 = kv_tiles_for<CAUSAL>(2 * w.qb, g.n_k_tiles);
        w.n1 = kv_tiles_for<CAUSAL>(2 * w.qb + 1, g.n_k_tiles);
    } else {
        w.jb = w.split * g.n_k_tiles / g.nsplit;
        w.n0 = w.n1 = (w.split + 1) * g.n_k_tiles / g.nsplit - w.jb;
    }
    return w;
}

// ---------------------------------------------------------------- TMA producer
template <int D, bool CAUSAL>
// Run by the whole warp: addresses and coordinates stay warp-uniform and one
// elected lane issues each copy.
__device__ __forceinline__ void ws_load_role(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                             const CUtensorMap& tm_v, const FwdParams& p, int lane) {
    using Cfg = WsCfg<D>;
    constexpr int S = Cfg::kStages;
    const WsSmem<D> sm;
    const WsGeometry g(p);
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
        // claim the next unit and hand it to the other roles
        const int qslot = it % U;
        ok = wait_phase_warp(sm.u_empty(qslot), ((it / U) & 1) ^ 1, abort_flag, kStatusTimeoutOther, lim);
        if (!ok) break;
        int u = 0;
        if (lane == 0) {
            u = static_cast<int>(atomicAdd(p.sched, 1u));
            if (u >= g.n_items) u = -1;
            *sm.unit_slot(qslot) = u;
            ptx::mbar_arrive(sm.u_full(qslot));
        }
        u = __shfl_sync(0xffffffffu, u, 0);
        if (u < 0) break;
        const WsItem w = item_coords<CAUSAL>(u, g);
        const int bh = w.bh, qb = w.qb, n1 = w.n1;
        for (int t = 0; t < 2 && ok; ++t) {
            ok = wait_phase_warp(sm.q_empty(t), (it & 1) ^ 1, abort_flag, kStatusTimeoutFree, lim);
            if (!ok) break;
            ptx::mbar_arrive_expect_tx_elect(sm.q_full(t), Cfg::kTileBytes);
#pragma unroll
            for (int c = 0; c < D / kBoxCols; ++c)
                ptx::tma_load_3d_hint_elect(sm.q_tile(t) + c * kBoxBytes, &tm_q, sm.q_full(t), c * kBoxCols,
                                            qb * 2 * kBlockM + t * kBlockM, bh, stream_once);
        }
        for (int j = 0; j < n1 && ok; ++j) {
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
                                                c * kBoxCols, (w.jb + j) * kBlockN, bh, keep);
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

// S_t = Q_t·K_jᵀ for both tiles, one key tile after the other. An S buffer is
// rewritten only after the softmax has read (s_free) everything written there
// before; with d = 128 both tiles share one buffer, so S1(j) follows the read
// of S0(j) and S0(j+1) the read of S1(j). K slots are released here.
template <int D, bool CAUSAL>
__device__ __forceinline__ void ws_s_role(const FwdParams& p, int lane) {
    using Cfg = WsCfg<D>;
    constexpr int S = Cfg::kStages;
    constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(128, kBlockN, false, false);
    const WsSmem<D> sm;
    const WsGeometry g(p);
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
        const int u = next_unit(sm, it, lane, 0xffffffffu, p);
        if (u < 0) break;
        const WsItem w = item_coords<CAUSAL>(u, g);
        const int n0 = w.n0, n1 = w.n1;  // n0 <= n1 <= n0 + 1
        if (!wait_phase_warp(sm.q_full(0), it & 1, abort_flag, kStatusTimeoutLoad, lim)) break;
        if (!wait_phase_warp(sm.q_full(1), it & 1, abort_flag, kStatusTimeoutLoad, lim)) break;
        for (int j = 0; j < n1; ++j) {
            const uint32_t k = kv_cnt + 2u * j;  // ring position of K_j
            ok = wait_phase_warp(sm.kv_full(k % S), (k / S) & 1, abort_flag, kStatusTimeoutLoad, lim);
            if (!ok) break;
            if (j < n0) {
                if (!issue_s_safe(0, sm.ring(k))) break;
                if (j == n0 - 1) ptx::mma_commit_elect(sm.q_empty(0));
            }
            if (!issue_s_safe(1, sm.ring(k))) break;
            if (j == n1 - 1) ptx::mma_commit_elect(sm.q_empty(1));
            ptx::mma_commit_elect(sm.kv_empty(k % S));
        }
        kv_cnt += 2u * n1;
    }
}

// O_t += P_t·V_j for tile t, once the softmax has written P_t(j); the commit
// after each one (pv_done) tells the softmax when it may overwrite P_t or
// rescale O_t. V slots are released by both P·V warps (two arrivals); the
// key tiles tile 0 does not see under the causal mask are released without
// use, after their load, so that the arrival lands in the slot's current use.
template <int D, bool CAUSAL>
__device__ __forceinline__ void ws_pv_role(const FwdParams& p, int lane, int t) {
    using Cfg = WsCfg<D>;
    constexpr int S = Cfg::kStages;
    constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(128, D, false, true);
    const WsSmem<D> sm;
    const WsGeometry g(p);
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
    uint32_t s_base = 0;  // S_t MMAs of earlier units
    volatile uint32_t* s_issued = sm.s_issued(t);
    bool ok = true;
    for (int it = 0; ok; ++it) {
        const int u = next_unit(sm, it, lane, 0xffffffffu, p);
        if (u < 0) break;
        const WsItem w = item_coords<CAUSAL>(u, g);
        const int n1 = w.n1, n_t = t == 0 ? w.n0 : w.n1;
        for (int j = 0; j < n1; ++j) {
            const uint32_t v = kv_cnt + 2u * j + 1u;  // ring position of V_j
            ok = wait_phase_warp(sm.kv_full(v % S), (v / S) & 1, abort_flag, kStatusTimeoutLoad, lim);
            if (!ok) break;
            if (j < n_t) {
                ok = wait_phase_warp(sm.p_full(t), p_cnt & 1, abort_flag, kStatusTimeoutSoftmax, lim);
                ++p_cnt;
                if (!ok) break;
                // The softmax waits for S_t(j+1) before it needs this P·V, so
                // S_t(j+1) goes to the tensor core first: wait (briefly; this is
                // only an ordering preference) until the S warp has issued it.
                if (j + 1 < n_t) {
                    const uint32_t want = s_base + static_cast<uint32_t>(j) + 2u;
                    for (int spin = 0; spin < 2000 && *s_issued < want; ++spin) __nanosleep(32);
                }
                ptx::tc_fence_after_sync();
                issue_pv(sm.ring(v), j > 0);
                ptx::mma_commit_elect(sm.pv_done(t));
                if (j == n_t - 1) ptx::mma_commit_elect(sm.o_full(t));
                ptx::mma_commit_elect(sm.kv_empty(v % S));
            } else if (lane == 0) {
                ptx::mbar_arrive(sm.kv_empty(v % S));
            }
        }
        kv_cnt += 2u * n1;
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

// ---------------------------------------------------------------- softmax + epilogue
template <int D, bool CAUSAL>
__device__ __forceinline__ void ws_softmax_role(const CUtensorMap& tm_o, const FwdParams& p, int warp, int lane) {
    using Cfg = WsCfg<D>;
    constexpr float kTau = 32.0f;
    const WsSmem<D> sm;
    const WsGeometry g(p);
    volatile int* abort_flag = sm.abort_flag();
    const unsigned long long lim = p.wait_limit_ns;
    const uint32_t tmem = *sm.tmem_slot();
    const int t = warp >> 2;                 // query tile of this warpgroup
    const int row = (warp & 3) * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + (t == 0 ? Cfg::kTmemS0 : Cfg::kTmemS1) + lane_base;
    const uint32_t tO = tmem + (t == 0 ? Cfg::kTmemO0 : Cfg::kTmemO1) + lane_base;
    const uint32_t tP = tmem + (t == 0 ? Cfg::kTmemP0 : Cfg::kTmemP1) + lane_base;
    uint8_t* stage = sm.base + Cfg::kOffStage + t * kBoxBytes;
    const uint32_t stage_s = sm.sbase + Cfg::kOffStage + t * kBoxBytes;
    const float c_log2 = p.scale_log2;
    uint32_t s_cnt = 0;
    uint32_t p_made = 0, pv_seen = 0;  // P tiles written / P·V completions observed
    bool failed = false;
    for (int it = 0;; ++it) {
        const int u = next_unit(sm, it, lane, 0xffffffffu, p);
        if (u == -2) failed = true;
        if (named_bar_or(1 + t, 128, u < 0)) break;  // the warpgroup agrees on stopping
        const WsItem w = item_coords<CAUSAL>(u, g);
        const int bh = w.bh;
        const int q_tile = 2 * w.qb + t;
        const int i0 = q_tile * kBlockM;
        const int n_t = t == 0 ? w.n0 : w.n1;
        float m_ref = -INFINITY;  // reference max (base 2) that O and l are relative to
        float l = 0.f;
        for (int j = 0; j < n_t; ++j) {
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
            const int jt = w.jb + j;  // key tile index within the head
            const int key0 = jt * kBlockN;
            const bool need_mask = key0 + kBlockN > p.N || (CAUSAL && jt == q_tile);
            int last = p.N - 1 - key0;  // last visible column of this tile
            if (CAUSAL && jt == q_tile) last = min(last, row);
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
                for (int i = 0; i < 32; ++i) {
                    s[i] = __uint_as_float(r0[i]);
                    s[32 + i] = __uint_as_float(r1[i]);
                    s[64 + i] = __uint_as_float(r2[i]);
                    s[96 + i] = __uint_as_float(r3[i]);
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
            if (j > 0 && __any_sync(0xffffffffu, move)) {
#pragma unroll 1
                for (int c = 0; c < D / 8; ++c) {
                    uint32_t r[8];
                    ptx::tmem_ld_32x32b_x8(tO + c * 8, r);
                    ptx::tmem_wait_ld(r);
#pragma unroll
                    for (int i = 0; i < 8; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
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
                for (int i = 0; i < 32; i += 4) {
                    const int c = h * 64 + 2 * i;
                    sa = ptx::fadd2(sa, make_float2(s[c], s[c + 1]));
                    sb = ptx::fadd2(sb, make_float2(s[c + 2], s[c + 3]));
                    sc = ptx::fadd2(sc, make_float2(s[c + 4], s[c + 5]));
                    sd = ptx::fadd2(sd, make_float2(s[c + 6], s[c + 7]));
                    r[i] = ptx::pack_bf16x2(s[c], s[c + 1]);
                    r[i + 1] = ptx::pack_bf16x2(s[c + 2], s[c + 3]);
                    r[i + 2] = ptx::pack_bf16x2(s[c + 4], s[c + 5]);
                    r[i + 3] = ptx::pack_bf16x2(s[c + 6], s[c + 7]);
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
        // ---- epilogue of tile t: O_t / l -> bf16 -> staging box -> TMA store; LSE
        bool ok = !failed && wait_phase(sm.o_full(t), it & 1, abort_flag, kStatusTimeoutMma, lim);
        ok = __all_sync(0xffffffffu, ok);
        if (named_bar_or(1 + t, 128, !ok)) {
            failed = true;
            break;
        }
        ptx::tc_fence_after_sync();
        const float inv_l = 1.0f / l;
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        float lse2 = m_use + log2f(l);  // base-2 log-sum-exp of this row's scaled scores
        // one 64-column box of the final O (fp32 row values f[0..63]) -> bf16 -> staging -> TMA store
        auto store_box = [&](int b, const float (&f)[64]) {
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) {
                uint4 v;
                v.x = ptx::pack_bf16x2(f[q8 * 8 + 0], f[q8 * 8 + 1]);
                v.y = ptx::pack_bf16x2(f[q8 * 8 + 2], f[q8 * 8 + 3]);
                v.z = ptx::pack_bf16x2(f[q8 * 8 + 4], f[q8 * 8 + 5]);
                v.w = ptx::pack_bf16x2(f[q8 * 8 + 6], f[q8 * 8 + 7]);
                *reinterpret_cast<uint4*>(stage + sw128_offset(row, q8)) = v;
            }
            ptx::fence_proxy_async_smem();
            ptx::named_bar_sync(1 + t, 128);
            if (row == 0 && i0 < p.N) {  // a tile wholly past the end has nothing to store
                ptx::tma_store_3d(&tm_o, stage_s, b * kBoxCols, i0, bh);
                ptx::bulk_commit_group();
                ptx::bulk_wait_group_read0();
            }
            ptx::named_bar_sync(1 + t, 128);
        };
        bool write_out = true;
        if (g.nsplit > 1) {
            // Split key range: publish this split's normalised O and LSE, take a
            // ticket, and let the last split of the tile merge all of them.
            const size_t slot = static_cast<size_t>(u) * 2 + t;  // (item, tile)
            float* po = p.part_o + slot * (D / 4) * kBlockM * 4;
#pragma unroll
            for (int b = 0; b < D / kBoxCols; ++b) {
                float o[64];
                load_row64(tO + b * 64, o);
#pragma unroll
                for (int cg = 0; cg < 16; ++cg)
                    *reinterpret_cast<float4*>(po + ((b * 16 + cg) * kBlockM + row) * 4) =
                        make_float4(o[cg * 4] * inv_l, o[cg * 4 + 1] * inv_l, o[cg * 4 + 2] * inv_l,
                                    o[cg * 4 + 3] * inv_l);
            }
            p.part_lse[slot * kBlockM + row] = lse2;
            __threadfence();
            ptx::named_bar_sync(1 + t, 128);
            if (row == 0) {
                const unsigned done = atomicAdd(p.tickets + static_cast<size_t>(w.unit) * 2 + t, 1u);
                *sm.last_flag(t) = (done == static_cast<unsigned>(g.nsplit - 1)) ? 1 : 0;
            }
            ptx::named_bar_sync(1 + t, 128);
            write_out = *sm.last_flag(t) != 0;
            if (write_out) {
                __threadfence();
                // merge: O = sum_s 2^(L_s - M) O_s / sum_s 2^(L_s - M), LSE = M + log2(sum)
                const size_t first = static_cast<size_t>(w.unit) * g.nsplit * 2 + t;  // slot of split 0
                float mmax = -INFINITY;
                for (int sp = 0; sp < g.nsplit; ++sp)
                    mmax = fmaxf(mmax, p.part_lse[(first + 2 * sp) * kBlockM + row]);
                float wsum = 0.f;
                for (int sp = 0; sp < g.nsplit; ++sp)
                    wsum += ptx::ex2_approx(p.part_lse[(first + 2 * sp) * kBlockM + row] - mmax);
                const float inv_w = 1.0f / wsum;
#pragma unroll 1
                for (int b = 0; b < D / kBoxCols; ++b) {
                    float acc[64];
#pragma unroll
                    for (int i = 0; i < 64; ++i) acc[i] = 0.f;
                    for (int sp = 0; sp < g.nsplit; ++sp) {
                        const float wgt =
                            ptx::ex2_approx(p.part_lse[(first + 2 * sp) * kBlockM + row] - mmax) * inv_w;
                        const float* ps = p.part_o + (first + 2 * sp) * (D / 4) * kBlockM * 4;
#pragma unroll
                        for (int cg = 0; cg < 16; ++cg) {
                            const float4 v = *reinterpret_cast<const float4*>(ps + ((b * 16 + cg) * kBlockM + row) * 4);
                            acc[cg * 4] = fmaf(wgt, v.x, acc[cg * 4]);
                            acc[cg * 4 + 1] = fmaf(wgt, v.y, acc[cg * 4 + 1]);
                            acc[cg * 4 + 2] = fmaf(wgt, v.z, acc[cg * 4 + 2]);
                            acc[cg * 4 + 3] = fmaf(wgt, v.w, acc[cg * 4 + 3]);
                        }
                    }
                    store_box(b, acc);
                }
                lse2 = mmax + log2f(wsum);
            }
        } else {
#pragma unroll
            for (int b = 0; b < D / kBoxCols; ++b) {
                float o[64];
                load_row64(tO + b * 64, o);
#pragma unroll
                for (int i = 0; i < 64; ++i) o[i] *= inv_l;
                store_box(b, o);
            }
        }
        if (write_out && p.lse != nullptr && i0 + row < p.N)
            p.lse[static_cast<size_t>(bh) * p.N + i0 + row] = lse2 * 0.69314718055994531f;
        ptx::tc_fence_before_sync();
    }
    if (row == 0) ptx::bulk_wait_group0();
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_ws_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
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

    if (warp >= 8) {
        ptx::regs_dec<kRegsControl>();  // the whole control warpgroup (warps 8-11)
        const WsSmem<D> sm;
        if (warp == 8) {
            ptx::tmem_alloc(ptx::smem_u32(sm.tmem_slot()), Cfg::kTmemCols);
            ptx::tmem_relinquish();
        }
        if (warp == 9 && lane == 0) {
            for (int i = 0; i < Cfg::kNumBars; ++i) {
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
            *sm.abort_flag() = 0;
            *sm.s_issued(0) = 0u;
            *sm.s_issued(1) = 0u;
            ptx::fence_mbar_init();
        }
        ptx::tc_fence_before_sync();
        ptx::named_bar_sync(Cfg::kBarAll, Cfg::kThreads);
        ptx::tc_fence_after_sync();
        if (warp == 9) {
            ws_load_role<D, CAUSAL>(tm_q, tm_k, tm_v, p, lane);
            __syncwarp();
        } else {
            // warp 8: every S; warps 10 and 11: P·V of tile 0 and tile 1
            const int m = warp == 8 ? 0 : warp - 9;
            if (warp == 8)
                ws_s_role<D, CAUSAL>(p, lane);
            else
                ws_pv_role<D, CAUSAL>(p, lane, warp - 10);
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
        if (warp == 9 && lane == 0) {
            // every CTA has claimed its last unit before it counts itself done,
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
        ptx::named_bar_sync(Cfg::kBarAll, Cfg::kThreads);
        ptx::tc_fence_after_sync();
        ws_softmax_role<D, CAUSAL>(tm_o, p, warp, lane);
        ptx::tc_fence_before_sync();
        ptx::named_bar_sync(Cfg::kBarAll, Cfg::kThreads);
    }
}

}  // namespace fa
