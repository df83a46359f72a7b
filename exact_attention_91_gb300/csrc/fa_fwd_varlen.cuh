// Attention forward over a batch of sequences of different lengths, each
// with its own number of queries and keys, for sm_103a.
//
// The same warp-specialised persistent design as fa_fwd_ws.cuh (its shared
// memory layout, barriers, TMEM columns and role split are reused), compiled
// as a kernel of its own so that the equal-length kernel keeps its exact code:
//   * tokens are rows of [total, H, d] (a token's H heads side by side); the
//     tensor maps are (d, H, total) and a box is 128 consecutive tokens of one
//     head;
//   * a work unit is (sequence, head, 256-query block); a block that starts
//     past the end of its sequence is skipped when it is claimed;
//   * under the causal mask query i of a sequence with Nq queries and Nk keys
//     sees keys j <= i + Nk - Nq (the mask aligned at the end of the sequence;
//     with Nq = Nk it is the usual one); a query tile whose queries see no key
//     issues no MMA, and such queries get O = 0, LSE = -inf;
//   * O rows are written with 16-byte stores (a TMA box would run into the next
//     sequence), only inside [0, total_q);
//   * when there are few units (decode: a handful of sequences with one query
//     each and long key sets), each unit's key tiles are split among `nsplit`
//     work items; every item writes its normalised partial O and base-2 LSE
//     for the rows that exist, and the last item of a tile to finish merges
//     them (O = sum_s w_s O_s, w_s = 2^(L_s - L) with L the merged LSE).
// ("Mini FlashAttention", §4 "The flash trick: online softmax", checks its
// loop on ragged sequences.)
#pragma once

#include "fa_fwd_ws.cuh"

namespace fa {
namespace vl {

struct VlParams {
    void* o;              // [total_q, H, d] bf16
    float* lse;           // [H, total_q] fp32, or null
    const int* cu_q;      // [B + 1] query-token offsets
    const int* cu_k;      // [B + 1] key-token offsets
    int heads;            // H
    int num_heads_total;  // B*H
    int total_q;
    int max_nq;           // largest query count of the batch
    float scale_log2;     // scale * log2(e)
    unsigned long long wait_limit_ns;
    unsigned* sched;      // work-queue slot {next unit, CTAs finished}
    // Key-range split; nsplit = 1: none, and the four fields below are unused.
    int nsplit;
    int part_tiles;       // query tiles per item that can hold a query: min(2, ceil(max_nq / 128))
    int part_rows;        // rows kept per tile: min(128, max_nq)
    float* part_o;        // [items][part_tiles][d/4][part_rows][4] fp32: normalised partial O
    float* part_lse;      // [items][part_tiles][part_rows] fp32: base-2 LSE of each partial
    unsigned* tickets;    // [units][2], zero at launch: items of a tile finished so far
};

struct Geometry {
    int BH, nqb, nsplit, n_items;
    __device__ __forceinline__ explicit Geometry(const VlParams& p) {
        BH = p.num_heads_total;
        nqb = (p.max_nq + 2 * kBlockM - 1) / (2 * kBlockM);
        nsplit = p.nsplit;
        n_items = nqb * BH * nsplit;
    }
};

// One work item: split `split` of unit `unit` = (sequence b, head h, bh =
// b*H + h, query block qb); its queries are tokens q0 .. q0+nq-1 and its keys
// k0 .. k0+nk-1; query tile t visits key tiles jb .. jb+n_t-1.
struct Item {
    int unit, split, bh, qb, jb, n0, n1;
    int head, q0, nq, k0, nk, off;  // off = nk - nq
    __device__ __forceinline__ int n_load() const { return n0 > n1 ? n0 : n1; }
};

// Key tiles a query tile visits: none when it holds no query of the
// sequence; every one without the causal mask; else up to the last key that
// its last query sees.
template <bool CAUSAL>
__device__ __forceinline__ int kv_tiles(int q_tile, int nq, int nk, int off) {
    const int i0 = q_tile * kBlockM;
    if (i0 >= nq) return 0;
    const int n_k = (nk + kBlockN - 1) / kBlockN;
    if (!CAUSAL) return n_k;
    const int kmax = min(i0 + kBlockM - 1, nq - 1) + off;
    return kmax < 0 ? 0 : min(kmax / kBlockN + 1, n_k);
}

// Item u: unit u / nsplit in the order of the equal-length kernel
// (unit_coords): (sequence, head) pairs in groups of 16 so that the K/V tiles
// in flight stay in L2, and inside a group the latest query blocks first.
// Blocks past the end of a shorter sequence are skipped when claimed. Split s
// takes the s-th of nsplit contiguous shares of the key tiles that the unit
// loads; a tile that sees fewer keys takes what of its own range falls there.
template <bool CAUSAL>
__device__ __forceinline__ Item item_coords(int u, const Geometry& g, const VlParams& p) {
    Item w;
    if (g.nsplit == 1) {
        w.unit = u;
        w.split = 0;
    } else {
        w.unit = u / g.nsplit;
        w.split = u - w.unit * g.nsplit;
    }
    unit_coords(w.unit, g.nqb, g.BH, w.bh, w.qb);
    const int b = w.bh / p.heads;
    w.head = w.bh - b * p.heads;
    w.q0 = p.cu_q[b];
    w.nq = p.cu_q[b + 1] - w.q0;
    w.k0 = p.cu_k[b];
    w.nk = p.cu_k[b + 1] - w.k0;
    w.off = w.nk - w.nq;
    w.jb = 0;
    w.n0 = kv_tiles<CAUSAL>(2 * w.qb, w.nq, w.nk, w.off);
    w.n1 = kv_tiles<CAUSAL>(2 * w.qb + 1, w.nq, w.nk, w.off);
    if (g.nsplit > 1) {
        const int n = w.n_load();
        const int je = (w.split + 1) * n / g.nsplit;
        w.jb = w.split * n / g.nsplit;
        w.n0 = max(0, min(je, w.n0) - w.jb);
        w.n1 = max(0, min(je, w.n1) - w.jb);
    }
    return w;
}

// Next unit of this CTA from the unit queue (consumer side), as fa::next_unit.
template <int D>
__device__ __forceinline__ int next_unit(const WsSmem<D>& sm, int it, int lane, const VlParams& p) {
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

// ---------------------------------------------------------------- TMA producer
template <int D, bool CAUSAL>
// Run by the whole warp: addresses and coordinates stay warp-uniform and one
// elected lane issues each copy.
__device__ __forceinline__ void load_role(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                             const CUtensorMap& tm_v, const VlParams& p, int lane) {
    using Cfg = WsCfg<D>;
    constexpr int S = Cfg::kStages;
    const WsSmem<D> sm;
    const Geometry g(p);
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
            // a block past the end of its sequence is no work
            for (;;) {
                u = static_cast<int>(atomicAdd(p.sched, 1u));
                if (u >= g.n_items) {
                    u = -1;
                    break;
                }
                const Item c = item_coords<CAUSAL>(u, g, p);
                if (2 * kBlockM * c.qb < c.nq) break;
            }
            *sm.unit_slot(qslot) = u;
            ptx::mbar_arrive(sm.u_full(qslot));
        }
        u = __shfl_sync(0xffffffffu, u, 0);
        if (u < 0) break;
        const Item w = item_coords<CAUSAL>(u, g, p);
        const int qb = w.qb, n_load = w.n_load();
        // tensor-map coordinates (head, token) of a row of this sequence
        auto rc_q = [&](int row, int& y, int& z) {
            y = w.head;
            z = w.q0 + row;
        };
        auto rc_k = [&](int row, int& y, int& z) {
            y = w.head;
            z = w.k0 + row;
        };
        for (int t = 0; t < 2 && ok; ++t) {
            ok = wait_phase_warp(sm.q_empty(t), (it & 1) ^ 1, abort_flag, kStatusTimeoutFree, lim);
            if (!ok) break;
            ptx::mbar_arrive_expect_tx_elect(sm.q_full(t), Cfg::kTileBytes);
            int y, z;
            rc_q(qb * 2 * kBlockM + t * kBlockM, y, z);
#pragma unroll
            for (int c = 0; c < D / kBoxCols; ++c)
                ptx::tma_load_3d_hint_elect(sm.q_tile(t) + c * kBoxBytes, &tm_q, sm.q_full(t), c * kBoxCols, y, z,
                                            stream_once);
        }
        for (int j = 0; j < n_load && ok; ++j) {
            for (int which = 0; which < 2; ++which, ++kv_cnt) {
                const int slot = static_cast<int>(kv_cnt % S);
                ok = wait_phase_warp(sm.kv_empty(slot), ((kv_cnt / S) & 1) ^ 1, abort_flag, kStatusTimeoutFree,
                                     lim);
                if (!ok) break;
                ptx::mbar_arrive_expect_tx_elect(sm.kv_full(slot), Cfg::kTileBytes);
                const CUtensorMap* map = which == 0 ? &tm_k : &tm_v;
                int y, z;
                rc_k((w.jb + j) * kBlockN, y, z);
#pragma unroll
                for (int c = 0; c < D / kBoxCols; ++c)
                    ptx::tma_load_3d_hint_elect(sm.ring(kv_cnt) + c * kBoxBytes, map, sm.kv_full(slot),
                                                c * kBoxCols, y, z, keep);
            }
        }
    }
}

// ---------------------------------------------------------------- MMA issuers (as in fa_fwd_ws.cuh)
// S_t = Q_t·K_jᵀ for both tiles, one key tile after the other. An S buffer is
// rewritten only after the softmax has read (s_free) everything written there
// before; with d = 128 both tiles share one buffer, so S1(j) follows the read
// of S0(j) and S0(j+1) the read of S1(j). K slots are released here.
template <int D, bool CAUSAL>
__device__ __forceinline__ void s_role(const VlParams& p, int lane) {
    using Cfg = WsCfg<D>;
    constexpr int S = Cfg::kStages;
    constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(128, kBlockN, false, false);
    const WsSmem<D> sm;
    const Geometry g(p);
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
        const Item w = item_coords<CAUSAL>(u, g, p);
        const int n0 = w.n0, n1 = w.n1, n_load = w.n_load();
        if (!wait_phase_warp(sm.q_full(0), it & 1, abort_flag, kStatusTimeoutLoad, lim)) break;
        if (!wait_phase_warp(sm.q_full(1), it & 1, abort_flag, kStatusTimeoutLoad, lim)) break;
        // a tile that sees no key still hands its Q buffer back
        if (n0 == 0) ptx::mma_commit_elect(sm.q_empty(0));
        if (n1 == 0) ptx::mma_commit_elect(sm.q_empty(1));
        for (int j = 0; j < n_load; ++j) {
            const uint32_t k = kv_cnt + 2u * j;  // ring position of K_j
            ok = wait_phase_warp(sm.kv_full(k % S), (k / S) & 1, abort_flag, kStatusTimeoutLoad, lim);
            if (!ok) break;
            if (j < n0) {
                if (!issue_s_safe(0, sm.ring(k))) break;
                if (j == n0 - 1) ptx::mma_commit_elect(sm.q_empty(0));
            }
            if (j < n1) {
                if (!issue_s_safe(1, sm.ring(k))) break;
                if (j == n1 - 1) ptx::mma_commit_elect(sm.q_empty(1));
            }
            ptx::mma_commit_elect(sm.kv_empty(k % S));
        }
        kv_cnt += 2u * n_load;
    }
}

// O_t += P_t·V_j for tile t, once the softmax has written P_t(j); the commit
// after each one (pv_done) tells the softmax when it may overwrite P_t or
// rescale O_t. V slots are released by both P·V warps (two arrivals); key
// tiles that only the other query tile sees are released without use, after
// their load, so that the arrival lands in the slot's current use.
template <int D, bool CAUSAL>
__device__ __forceinline__ void pv_role(const VlParams& p, int lane, int t) {
    using Cfg = WsCfg<D>;
    constexpr int S = Cfg::kStages;
    constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(128, D, false, true);
    const WsSmem<D> sm;
    const Geometry g(p);
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
        const int u = next_unit(sm, it, lane, p);
        if (u < 0) break;
        const Item w = item_coords<CAUSAL>(u, g, p);
        const int n_load = w.n_load(), n_t = t == 0 ? w.n0 : w.n1;
        if (n_t == 0) ptx::mma_commit_elect(sm.o_full(t));  // nothing to add: O is all zero
        for (int j = 0; j < n_load; ++j) {
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
        kv_cnt += 2u * n_load;
        s_base += static_cast<uint32_t>(n_t);
    }
}

// ---------------------------------------------------------------- softmax + epilogue
template <int D, bool CAUSAL>
__device__ __forceinline__ void softmax_role(const VlParams& p, int warp, int lane) {
    using Cfg = WsCfg<D>;
    constexpr float kTau = 32.0f;  // as in fa_fwd_ws.cuh
    const WsSmem<D> sm;
    const Geometry g(p);
    volatile int* abort_flag = sm.abort_flag();
    const unsigned long long lim = p.wait_limit_ns;
    const uint32_t tmem = *sm.tmem_slot();
    const int t = warp >> 2;                 // query tile of this warpgroup
    const int row = (warp & 3) * 32 + lane;  // row within the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tmem + (t == 0 ? Cfg::kTmemS0 : Cfg::kTmemS1) + lane_base;
    const uint32_t tO = tmem + (t == 0 ? Cfg::kTmemO0 : Cfg::kTmemO1) + lane_base;
    const uint32_t tP = tmem + (t == 0 ? Cfg::kTmemP0 : Cfg::kTmemP1) + lane_base;
    const float c_log2 = p.scale_log2;
    uint32_t s_cnt = 0;
    uint32_t p_made = 0, pv_seen = 0;  // P tiles written / P·V completions observed
    bool failed = false;
    for (int it = 0;; ++it) {
        const int u = next_unit(sm, it, lane, p);
        if (u == -2) failed = true;
        if (named_bar_or(1 + t, 128, u < 0)) break;  // the warpgroup agrees on stopping
        const Item w = item_coords<CAUSAL>(u, g, p);
        const int q_tile = 2 * w.qb + t;
        const int i0 = q_tile * kBlockM;
        const int n_t = t == 0 ? w.n0 : w.n1;
        const int seq_nq = w.nq, seq_nk = w.nk, seq_off = w.off;
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
            const int jt = w.jb + j;  // key tile index within the sequence
            const int key0 = jt * kBlockN;
            const bool need_mask = key0 + kBlockN > seq_nk || (CAUSAL && key0 + kBlockN - 1 > i0 + seq_off);
            int last = seq_nk - 1 - key0;  // last visible column of this tile
            if (CAUSAL) last = min(last, i0 + row + seq_off - key0);
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
            // p = 2^(S·c - m) and P in three passes over the row, as in fa_fwd_ws.cuh
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
        // ---- epilogue of tile t: O_t / l -> bf16 -> global; LSE
        bool ok = !failed && wait_phase(sm.o_full(t), it & 1, abort_flag, kStatusTimeoutMma, lim);
        ok = __all_sync(0xffffffffu, ok);
        if (named_bar_or(1 + t, 128, !ok)) {
            failed = true;
            break;
        }
        ptx::tc_fence_after_sync();
        // a query that sees no key (under the causal mask, when the sequence
        // has more queries than keys) gets O = 0 and LSE = -inf
        const bool any_key = l > 0.f;
        const float inv_l = any_key ? 1.0f / l : 0.f;
        const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
        float lse2 = any_key ? m_use + log2f(l) : -INFINITY;  // base-2 log-sum-exp of the row's scaled scores
        // (cu_seqlens are the caller's; a row outside [0, total_q) is never written)
        const bool row_in = i0 + row < seq_nq && w.q0 + i0 + row >= 0 && w.q0 + i0 + row < p.total_q;
        // element offset of this row of O and index of its LSE
        const size_t o_row = (static_cast<size_t>(w.q0 + i0 + row) * p.heads + w.head) * D;
        const size_t lse_idx = static_cast<size_t>(w.head) * p.total_q + w.q0 + i0 + row;
        // 64 columns (box b) of the final O row, fp32 f[0..63] -> bf16 -> 8 x 16
        // bytes; a TMA box would run into the next sequence
        auto store_cols = [&](int b, const float (&f)[64]) {
            if (!row_in) return;
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) + o_row + b * kBoxCols);
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) {
                uint4 v;
                v.x = ptx::pack_bf16x2(f[q8 * 8 + 0], f[q8 * 8 + 1]);
                v.y = ptx::pack_bf16x2(f[q8 * 8 + 2], f[q8 * 8 + 3]);
                v.z = ptx::pack_bf16x2(f[q8 * 8 + 4], f[q8 * 8 + 5]);
                v.w = ptx::pack_bf16x2(f[q8 * 8 + 6], f[q8 * 8 + 7]);
                dst[q8] = v;
            }
        };
        // this row's final (or, with a split key range, partial) O: fp32 f[0..63] of box b
        auto row_box = [&](int b, float (&f)[64]) {
            if (n_t > 0) {
                load_row64(tO + b * 64, f);
            } else {
#pragma unroll
                for (int i = 0; i < 64; ++i) f[i] = 0.f;  // O holds nothing of this item
            }
#pragma unroll
            for (int i = 0; i < 64; ++i) f[i] *= inv_l;
        };
        bool write_out = true;
        bool lse_ok = row_in;
        if (g.nsplit == 1) {
#pragma unroll
            for (int b = 0; b < D / kBoxCols; ++b) {
                float o[64];
                row_box(b, o);
                store_cols(b, o);
            }
        } else if (i0 < seq_nq && t < p.part_tiles) {  // (the same for every split of the unit and every
                                                       // thread of the tile)
            // Publish this split's O and LSE for the rows that exist, take a
            // ticket, and let the last split of the tile merge all of them.
            // The scratch holds part_tiles x part_rows rows per item, sized by
            // max_seqlen_q; a sequence with more queries than that (which the
            // caller rules out) leaves its extra rows unwritten rather than
            // writing past its slot.
            const int R = p.part_rows;
            const bool row_ok = row_in && row < R;
            lse_ok = row_ok;
            const size_t tile_slot = static_cast<size_t>(u) * p.part_tiles + t;  // (item, tile)
            float* po = p.part_o + tile_slot * R * D;
#pragma unroll
            for (int b = 0; b < D / kBoxCols; ++b) {
                float o[64];
                row_box(b, o);
                if (row_ok) {
#pragma unroll
                    for (int cg = 0; cg < 16; ++cg)
                        __stcg(reinterpret_cast<float4*>(po + (static_cast<size_t>(b * 16 + cg) * R + row) * 4),
                               make_float4(o[cg * 4], o[cg * 4 + 1], o[cg * 4 + 2], o[cg * 4 + 3]));
                }
            }
            if (row_ok) __stcg(p.part_lse + tile_slot * R + row, lse2);
            __threadfence();
            ptx::named_bar_sync(1 + t, 128);
            if (row == 0) {
                const unsigned done = atomicAdd(p.tickets + static_cast<size_t>(w.unit) * 2 + t, 1u);
                *sm.last_flag(t) = (done == static_cast<unsigned>(g.nsplit - 1)) ? 1 : 0;
            }
            ptx::named_bar_sync(1 + t, 128);
            write_out = *sm.last_flag(t) != 0;
            if (write_out && row_ok) {
                __threadfence();
                // O = sum_s 2^(L_s - M) O_s / sum_s 2^(L_s - M), LSE = M + log2(sum);
                // a split where the row sees no key has L_s = -inf and weight 0
                const size_t first = static_cast<size_t>(w.unit) * g.nsplit * p.part_tiles + t;  // split 0
                const size_t step = static_cast<size_t>(p.part_tiles);
                float mmax = -INFINITY;
                for (int sp = 0; sp < g.nsplit; ++sp)
                    mmax = fmaxf(mmax, __ldcg(p.part_lse + (first + sp * step) * R + row));
                const bool seen = mmax != -INFINITY;  // the row sees some key in some split
                const float m_w = seen ? mmax : 0.f;
                float wsum = 0.f;
                for (int sp = 0; sp < g.nsplit; ++sp)
                    wsum += ptx::ex2_approx(__ldcg(p.part_lse + (first + sp * step) * R + row) - m_w);
                const float inv_w = seen ? 1.0f / wsum : 0.f;
#pragma unroll 1
                for (int b = 0; b < D / kBoxCols; ++b) {
                    float acc[64];
#pragma unroll
                    for (int i = 0; i < 64; ++i) acc[i] = 0.f;
                    for (int sp = 0; sp < g.nsplit; ++sp) {
                        const size_t slot = first + sp * step;
                        const float wgt = ptx::ex2_approx(__ldcg(p.part_lse + slot * R + row) - m_w) * inv_w;
                        const float* ps = p.part_o + slot * R * D;
#pragma unroll
                        for (int cg = 0; cg < 16; ++cg) {
                            const float4 v =
                                __ldcg(reinterpret_cast<const float4*>(ps + (static_cast<size_t>(b * 16 + cg) * R + row) * 4));
                            acc[cg * 4] = fmaf(wgt, v.x, acc[cg * 4]);
                            acc[cg * 4 + 1] = fmaf(wgt, v.y, acc[cg * 4 + 1]);
                            acc[cg * 4 + 2] = fmaf(wgt, v.z, acc[cg * 4 + 2]);
                            acc[cg * 4 + 3] = fmaf(wgt, v.w, acc[cg * 4 + 3]);
                        }
                    }
                    store_cols(b, acc);
                }
                lse2 = seen ? mmax + log2f(wsum) : -INFINITY;
            }
        } else {
            write_out = false;  // no query of the sequence in this tile
        }
        if (write_out && p.lse != nullptr && lse_ok) p.lse[lse_idx] = lse2 * 0.69314718055994531f;
        ptx::tc_fence_before_sync();
    }
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_varlen_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const VlParams p) {
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
            load_role<D, CAUSAL>(tm_q, tm_k, tm_v, p, lane);
            __syncwarp();
        } else {
            // warp 8: every S; warps 10 and 11: P·V of tile 0 and tile 1
            const int m = warp == 8 ? 0 : warp - 9;
            if (warp == 8)
                s_role<D, CAUSAL>(p, lane);
            else
                pv_role<D, CAUSAL>(p, lane, warp - 10);
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
        softmax_role<D, CAUSAL>(p, warp, lane);
        ptx::tc_fence_before_sync();
        ptx::named_bar_sync(Cfg::kBarAll, Cfg::kThreads);
    }
}

}  // namespace vl
}  // namespace fa
