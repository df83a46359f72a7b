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
//   warp  8    MMA issue (one thread) and TMEM allocation
//   warp  9    TMA loads (one thread)
//   warps 10-11 idle (they complete the control warpgroup, which gives its
//              registers to the softmax warpgroups)
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
// the rule "rescale whenever the max moves".
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
    // barriers: q_full[2] q_empty[2] kv_full[S] kv_empty[S] s_full[2] p_full[2] o_full[2] fin
    static constexpr int kNumBars = 2 + 2 + 2 * kStages + 2 + 2 + 2 + 1;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + base alignment slack
    static constexpr int kTmemCols = 512;
    static constexpr uint32_t kTmemS0 = 0, kTmemS1 = 128, kTmemO0 = 256, kTmemO1 = 256 + (D == 128 ? 128 : 64);
};

// Unit u -> (head, 256-row query block). Heads are taken in groups of 16 so
// that the CTAs running at any moment share few heads and their K/V tiles
// stay in L2; inside a group the blocks with the most key tiles come first.
__device__ __forceinline__ void unit_coords(int u, int nqb, int BH, int& bh, int& qb) {
    constexpr int kGroup = 16;
    const int per_group = kGroup * nqb;
    const int g = u / per_group;
    const int hg = min(kGroup, BH - g * kGroup);
    const int idx = u - g * per_group;
    qb = nqb - 1 - idx / hg;
    bh = g * kGroup + idx % hg;
}

template <int D, bool CAUSAL>
__device__ __forceinline__ int kv_tiles_for(int q_tile, int n_k_tiles) {
    return CAUSAL ? min(q_tile + 1, n_k_tiles) : n_k_tiles;
}

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(384, 1)
    fa_fwd_ws_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                     const FwdParams p) {
    using Cfg = WsCfg<D>;
    static_assert(D == 64 || D == 128, "head dim");
    constexpr float kTau = 8.0f;
    // 384 threads launch with 168 registers each (64512); two softmax
    // warpgroups at 216 and one control warpgroup at 72 use 55296 + 9216.
    constexpr uint32_t kRegsSoftmax = 216, kRegsControl = 72;
    static_assert(2 * 128 * kRegsSoftmax + 128 * kRegsControl <= 384 * 168, "register split");
    constexpr int S = Cfg::kStages;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t bar0 = sbase + Cfg::kOffBar;
    auto q_full = [&](int t) { return bar0 + 8u * t; };
    auto q_empty = [&](int t) { return bar0 + 16u + 8u * t; };
    auto kv_full = [&](int s) { return bar0 + 32u + 8u * s; };
    auto kv_empty = [&](int s) { return bar0 + 32u + 8u * S + 8u * s; };
    auto s_full = [&](int t) { return bar0 + 32u + 16u * S + 8u * t; };
    auto p_full = [&](int t) { return bar0 + 48u + 16u * S + 8u * t; };
    auto o_full = [&](int t) { return bar0 + 64u + 16u * S + 8u * t; };
    const uint32_t bar_fin = bar0 + 80u + 16u * S;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    if (warp == 8) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), Cfg::kTmemCols);
        ptx::tmem_relinquish();
    }
    if (tid == 9 * 32) {
        for (int t = 0; t < 2; ++t) {
            ptx::mbar_init(q_full(t), 1);
            ptx::mbar_init(q_empty(t), 1);
            ptx::mbar_init(s_full(t), 1);
            ptx::mbar_init(p_full(t), 4);  // one arrival per softmax warp
            ptx::mbar_init(o_full(t), 1);
        }
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(kv_full(s), 1);
            ptx::mbar_init(kv_empty(s), 1);
        }
        ptx::mbar_init(bar_fin, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    const int BH = p.num_heads_total;
    const int n_k_tiles = (p.N + kBlockN - 1) / kBlockN;
    const int nqb = (p.N + 2 * kBlockM - 1) / (2 * kBlockM);
    const int n_units = nqb * BH;
    const unsigned long long lim = p.wait_limit_ns;

    if (warp >= 8) {
      ptx::regs_dec<kRegsControl>();  // the whole control warpgroup (warps 8-11)
      if (warp == 9) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            ptx::prefetch_tensormap(&tm_q);
            ptx::prefetch_tensormap(&tm_k);
            ptx::prefetch_tensormap(&tm_v);
            const uint64_t keep = ptx::policy_evict_last();
            const uint64_t stream_once = ptx::policy_evict_first();
            uint32_t kv_cnt = 0;
            int it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++it) {
                int bh, qb;
                unit_coords(u, nqb, BH, bh, qb);
                const int n1 = kv_tiles_for<D, CAUSAL>(2 * qb + 1, n_k_tiles);
                for (int t = 0; t < 2 && ok; ++t) {
                    ok = wait_phase(q_empty(t), (it & 1) ^ 1, abort_flag, kStatusTimeoutFree, lim);
                    if (!ok) break;
                    ptx::mbar_arrive_expect_tx(q_full(t), Cfg::kTileBytes);
                    const uint32_t dst = sbase + Cfg::kOffQ + t * Cfg::kTileBytes;
                    for (int c = 0; c < D / kBoxCols; ++c)
                        ptx::tma_load_3d_hint(dst + c * kBoxBytes, &tm_q, q_full(t), c * kBoxCols,
                                              qb * 2 * kBlockM + t * kBlockM, bh, stream_once);
                }
                for (int j = 0; j < n1 && ok; ++j) {
                    for (int which = 0; which < 2; ++which, ++kv_cnt) {
                        const int slot = static_cast<int>(kv_cnt % S);
                        const uint32_t round = kv_cnt / S;
                        ok = wait_phase(kv_empty(slot), (round & 1) ^ 1, abort_flag, kStatusTimeoutFree, lim);
                        if (!ok) break;
                        ptx::mbar_arrive_expect_tx(kv_full(slot), Cfg::kTileBytes);
                        const uint32_t dst = sbase + Cfg::kOffRing + slot * Cfg::kTileBytes;
                        const CUtensorMap* map = which == 0 ? &tm_k : &tm_v;
                        for (int c = 0; c < D / kBoxCols; ++c)
                            ptx::tma_load_3d_hint(dst + c * kBoxBytes, map, kv_full(slot), c * kBoxCols,
                                                  j * kBlockN, bh, keep);
                    }
                }
            }
        }
        __syncwarp();
      } else if (warp == 8) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(128, kBlockN, false, false);
            constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(128, D, false, true);
            const uint32_t tS[2] = {tmem + Cfg::kTmemS0, tmem + Cfg::kTmemS1};
            const uint32_t tO[2] = {tmem + Cfg::kTmemO0, tmem + Cfg::kTmemO1};
            const uint32_t sQ[2] = {sbase + Cfg::kOffQ, sbase + Cfg::kOffQ + Cfg::kTileBytes};
            auto slot_addr = [&](uint32_t cnt) { return sbase + Cfg::kOffRing + (cnt % S) * Cfg::kTileBytes; };
            // S_t = Q_t·Kᵀ over D in steps of 16 (4 steps of 32 bytes per 64-wide box).
            // Descriptors advance by adding the byte offset >> 4 to the start-address field.
            auto issue_s = [&](int t, uint32_t sK) {
                const uint64_t a0 = ptx::sdesc_sw128(sQ[t], 16, 1024);
                const uint64_t b0 = ptx::sdesc_sw128(sK, 16, 1024);
#pragma unroll 1
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = ((kk >> 2) * kBoxBytes + (kk & 3) * 32) >> 4;
                    ptx::mma_ss(tS[t], a0 + off, b0 + off, kIdescS, kk > 0 ? 1u : 0u);
                }
            };
            // O_t += P_t·V over 128 keys in steps of 16 (2048 bytes of V each);
            // V is MN-major: 64-wide swizzle atoms 16 KB apart (LBO), 8-key groups 1 KB apart (SBO).
            auto issue_pv = [&](int t, uint32_t sV, bool accumulate) {
                const uint64_t b0 = ptx::sdesc_sw128(sV, kBoxBytes, 1024);
#pragma unroll 1
                for (int kk = 0; kk < kBlockN / 16; ++kk) {
                    ptx::mma_ts(tO[t], tS[t] + kk * 8, b0 + static_cast<uint32_t>(kk * (2048 >> 4)), kIdescPV,
                                (accumulate || kk > 0) ? 1u : 0u);
                }
            };
            uint32_t kv_cnt = 0;
            uint32_t p_cnt[2] = {0, 0};
            int it = 0;
            bool ok = true;
            auto wait_p = [&](int t) {
                ok = ok && wait_phase(p_full(t), p_cnt[t] & 1, abort_flag, kStatusTimeoutSoftmax, lim);
                ++p_cnt[t];
                return ok;
            };
            auto wait_kv = [&](uint32_t cnt) {
                ok = ok && wait_phase(kv_full(cnt % S), (cnt / S) & 1, abort_flag, kStatusTimeoutLoad, lim);
                return ok;
            };
            for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x, ++it) {
                int bh, qb;
                unit_coords(u, nqb, BH, bh, qb);
                const int n0 = kv_tiles_for<D, CAUSAL>(2 * qb, n_k_tiles);
                const int n1 = kv_tiles_for<D, CAUSAL>(2 * qb + 1, n_k_tiles);
                const uint32_t k0 = kv_cnt;  // ring position of K_0; V_j = K_j + 1, K_j = k0 + 2j
                // first key tile: S_0 and S_1
                if (!(wait_phase(q_full(0), it & 1, abort_flag, kStatusTimeoutLoad, lim) && wait_kv(k0))) break;
                ptx::tc_fence_after_sync();
                issue_s(0, slot_addr(k0));
                ptx::mma_commit(s_full(0));
                if (n0 == 1) ptx::mma_commit(q_empty(0));
                if (!wait_phase(q_full(1), it & 1, abort_flag, kStatusTimeoutLoad, lim)) { ok = false; break; }
                ptx::tc_fence_after_sync();
                issue_s(1, slot_addr(k0));
                ptx::mma_commit(s_full(1));
                if (n1 == 1) ptx::mma_commit(q_empty(1));
                ptx::mma_commit(kv_empty(k0 % S));
                for (int j = 1; j < n1; ++j) {
                    const uint32_t kj = k0 + 2 * j, vprev = k0 + 2 * j - 1;
                    // P·V needs only V_{j-1}; K_j may still be in flight. (A second
                    // wait on K_j's slot is immediate: it is not refilled before release.)
                    if (!wait_kv(vprev)) break;
                    if (j <= n0) {
                        if (!wait_p(0)) break;
                        ptx::tc_fence_after_sync();
                        issue_pv(0, slot_addr(vprev), j > 1);
                        if (j < n0) {
                            if (!wait_kv(kj)) break;
                            ptx::tc_fence_after_sync();
                            issue_s(0, slot_addr(kj));
                            ptx::mma_commit(s_full(0));
                            if (j == n0 - 1) ptx::mma_commit(q_empty(0));
                        } else {
                            ptx::mma_commit(o_full(0));
                        }
                    }
                    if (!wait_p(1)) break;
                    ptx::tc_fence_after_sync();
                    issue_pv(1, slot_addr(vprev), j > 1);
                    ptx::mma_commit(kv_empty(vprev % S));
                    if (!wait_kv(kj)) break;
                    ptx::tc_fence_after_sync();
                    issue_s(1, slot_addr(kj));
                    ptx::mma_commit(s_full(1));
                    if (j == n1 - 1) ptx::mma_commit(q_empty(1));
                    ptx::mma_commit(kv_empty(kj % S));
                }
                if (!ok) break;
                // last key tile: P·V of the tiles still open
                const uint32_t vlast = k0 + 2 * n1 - 1;
                if (!wait_kv(vlast)) break;
                if (n0 == n1) {
                    if (!wait_p(0)) break;
                    ptx::tc_fence_after_sync();
                    issue_pv(0, slot_addr(vlast), n1 > 1);
                    ptx::mma_commit(o_full(0));
                }
                if (!wait_p(1)) break;
                ptx::tc_fence_after_sync();
                issue_pv(1, slot_addr(vlast), n1 > 1);
                ptx::mma_commit(o_full(1));
                ptx::mma_commit(kv_empty(vlast % S));
                kv_cnt = k0 + 2 * n1;
            }
        }
        __syncwarp();
      }
    } else {
        ptx::regs_inc<kRegsSoftmax>();
        // ------------------------------------------------------------ softmax (warps 0-7)
        const int t = warp >> 2;                 // query tile of this warpgroup
        const int row = (warp & 3) * 32 + lane;  // row within the tile == TMEM lane
        const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
        const uint32_t tS = tmem + (t == 0 ? Cfg::kTmemS0 : Cfg::kTmemS1) + lane_base;
        const uint32_t tO = tmem + (t == 0 ? Cfg::kTmemO0 : Cfg::kTmemO1) + lane_base;
        uint8_t* stage = smem + Cfg::kOffStage + t * kBoxBytes;
        const uint32_t stage_s = sbase + Cfg::kOffStage + t * kBoxBytes;
        const float c_log2 = p.scale_log2;
        uint32_t s_cnt = 0;
        int it = 0;
        bool failed = false;
        for (int u = blockIdx.x; u < n_units; u += gridDim.x, ++it) {
            int bh, qb;
            unit_coords(u, nqb, BH, bh, qb);
            const int q_tile = 2 * qb + t;
            const int i0 = q_tile * kBlockM;
            const int n_t = kv_tiles_for<D, CAUSAL>(q_tile, n_k_tiles);
            float m_ref = -INFINITY;  // reference max (base 2) that O and l are relative to
            float l = 0.f;
            for (int j = 0; j < n_t; ++j) {
                bool ok = wait_phase(s_full(t), s_cnt & 1, abort_flag, kStatusTimeoutMma, lim);
                ++s_cnt;
                if (!__all_sync(0xffffffffu, ok)) {
                    failed = true;
                    break;
                }
                ptx::tc_fence_after_sync();
                float s[kBlockN];
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
                // keys past the end, and (diagonal tile) keys after this query
                const int key0 = j * kBlockN;
                if (key0 + kBlockN > p.N || (CAUSAL && j == q_tile)) {
                    int last = p.N - 1 - key0;  // last visible column of this tile
                    if (CAUSAL && j == q_tile) last = min(last, row);
#pragma unroll
                    for (int c = 0; c < kBlockN; ++c) s[c] = (c > last) ? -INFINITY : s[c];
                }
                float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
                for (int c = 4; c < kBlockN; c += 4) {
                    mx0 = fmaxf(mx0, s[c]);
                    mx1 = fmaxf(mx1, s[c + 1]);
                    mx2 = fmaxf(mx2, s[c + 2]);
                    mx3 = fmaxf(mx3, s[c + 3]);
                }
                const float m_tile = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * c_log2;
                const bool move = m_tile > m_ref + kTau;
                float alpha = 1.f;
                if (move) {
                    alpha = ptx::ex2_approx(m_ref - m_tile);  // 0 on the first visible tile
                    m_ref = m_tile;
                }
                // O_t *= alpha; the previous P·V of this tile finished before S_t was committed
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
                float sum0 = 0.f, sum1 = 0.f, sum2 = 0.f, sum3 = 0.f;
#pragma unroll
                for (int c = 0; c < kBlockN; c += 4) {
                    s[c] = ptx::ex2_approx(fmaf(s[c], c_log2, -m_use));
                    s[c + 1] = ptx::ex2_approx(fmaf(s[c + 1], c_log2, -m_use));
                    s[c + 2] = ptx::ex2_approx(fmaf(s[c + 2], c_log2, -m_use));
                    s[c + 3] = ptx::ex2_approx(fmaf(s[c + 3], c_log2, -m_use));
                    sum0 += s[c];
                    sum1 += s[c + 1];
                    sum2 += s[c + 2];
                    sum3 += s[c + 3];
                }
                l = l * alpha + ((sum0 + sum1) + (sum2 + sum3));
                // P (bf16 pairs) over the first 64 columns of S_t
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    uint32_t r[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) r[i] = ptx::pack_bf16x2(s[c * 64 + 2 * i], s[c * 64 + 2 * i + 1]);
                    ptx::tmem_st_32x32b_x32(tS + c * 32, r);
                }
                ptx::tmem_wait_st();
                ptx::tc_fence_before_sync();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(p_full(t));
            }
            // ---- epilogue of tile t: O_t / l -> bf16 -> staging box -> TMA store; LSE
            bool ok = !failed && wait_phase(o_full(t), it & 1, abort_flag, kStatusTimeoutMma, lim);
            ok = __all_sync(0xffffffffu, ok);
            if (named_bar_or(1 + t, 128, !ok)) {
                failed = true;
                break;
            }
            ptx::tc_fence_after_sync();
            const float inv_l = 1.0f / l;
#pragma unroll
            for (int b = 0; b < D / kBoxCols; ++b) {
                uint32_t ra[32], rb[32];
                ptx::tmem_ld_32x32b_x32(tO + b * 64, ra);
                ptx::tmem_ld_32x32b_x32(tO + b * 64 + 32, rb);
                ptx::tmem_wait_ld(ra);
                ptx::reg_fence(rb);
#pragma unroll
                for (int q8 = 0; q8 < 8; ++q8) {
                    const uint32_t* r = q8 < 4 ? ra : rb;
                    const int o = (q8 & 3) * 8;
                    uint4 w;
                    w.x = ptx::pack_bf16x2(__uint_as_float(r[o + 0]) * inv_l, __uint_as_float(r[o + 1]) * inv_l);
                    w.y = ptx::pack_bf16x2(__uint_as_float(r[o + 2]) * inv_l, __uint_as_float(r[o + 3]) * inv_l);
                    w.z = ptx::pack_bf16x2(__uint_as_float(r[o + 4]) * inv_l, __uint_as_float(r[o + 5]) * inv_l);
                    w.w = ptx::pack_bf16x2(__uint_as_float(r[o + 6]) * inv_l, __uint_as_float(r[o + 7]) * inv_l);
                    *reinterpret_cast<uint4*>(stage + sw128_offset(row, q8)) = w;
                }
                ptx::fence_proxy_async_smem();
                ptx::named_bar_sync(1 + t, 128);
                if (row == 0 && i0 < p.N) {  // a tile wholly past the end has nothing to store
                    ptx::tma_store_3d(&tm_o, stage_s, b * kBoxCols, i0, bh);
                    ptx::bulk_commit_group();
                    ptx::bulk_wait_group_read0();
                }
                ptx::named_bar_sync(1 + t, 128);
            }
            if (p.lse != nullptr && i0 + row < p.N) {
                const float m_use = (m_ref == -INFINITY) ? 0.f : m_ref;
                p.lse[static_cast<size_t>(bh) * p.N + i0 + row] = (m_use + log2f(l)) * 0.69314718055994531f;
            }
            ptx::tc_fence_before_sync();
        }
        if (row == 0) ptx::bulk_wait_group0();
    }

    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 8) {
        if (lane == 0) {
            ptx::mma_commit(bar_fin);
            wait_drain(bar_fin, 0, 100000000ull);
        }
        __syncwarp();
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

}  // namespace fa
