// Attention forward, first tcgen05 form: one CTA of 4 warps per (head, 128-row
// query tile), single-buffered. It exists to pin the primitives (TMA boxes
// with the 128-byte swizzle, UMMA descriptors, TMEM loads and stores, P as a
// TMEM operand) on the smallest schedule that exercises all of them.
//
// Per key tile j (the loop of "Mini FlashAttention", §4, and steps 2-8 of the
// tiled kernel in "How Did I Write My First FlashAttention Kernel in CUDA?"):
//   S   = Q·K_jᵀ                    tcgen05.mma, fp32 in TMEM
//   m'  = max(m, rowmax(S)·c)       c = scale·log2(e), base-2 units
//   p   = 2^(S·c - m'), l = 2^(m-m')·l + Σp
//   O   = 2^(m-m')·O                in TMEM, only when m moved
//   O  += bf16(p)·V_j               tcgen05.mma, A = P from TMEM (or SMEM)
// then O/l in bf16 and LSE = ln2·(m + log2 l).
#pragma once

#include "fa_common.cuh"

namespace fa {

template <int D, bool P_IN_TMEM>
struct SimpleCfg {
    static constexpr int kTileBytes = D * kBlockM * 2;  // 128 rows x D bf16
    static constexpr int kPBytes = P_IN_TMEM ? 0 : kBlockM * kBlockN * 2;
    static constexpr int kOffQ = 0;
    static constexpr int kOffK = kOffQ + kTileBytes;
    static constexpr int kOffV = kOffK + kTileBytes;
    static constexpr int kOffP = kOffV + kTileBytes;
    static constexpr int kOffBar = kOffP + kPBytes;
    static constexpr int kNumBars = 5;
    static constexpr int kOffMisc = kOffBar + kNumBars * 8;
    static constexpr int kSmemBytes = kOffMisc + 16 + 1024;  // + 1024 for base alignment
    static constexpr int kTmemCols = 256;                     // S: 128 columns, O: D columns
    static constexpr int kThreads = 128;
};

template <int D, bool CAUSAL, bool P_IN_TMEM>
__global__ void __launch_bounds__(128, 1)
    fa_fwd_simple_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                         const FwdParams p) {
    using Cfg = SimpleCfg<D, P_IN_TMEM>;
    static_assert(D == 64 || D == 128, "head dim");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t sQ = sbase + Cfg::kOffQ;
    const uint32_t sK = sbase + Cfg::kOffK;
    const uint32_t sV = sbase + Cfg::kOffV;
    const uint32_t bar_q = sbase + Cfg::kOffBar;
    const uint32_t bar_kv = bar_q + 8;
    const uint32_t bar_s = bar_q + 16;
    const uint32_t bar_o = bar_q + 24;
    const uint32_t bar_fin = bar_q + 32;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Cfg::kOffMisc);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Cfg::kOffMisc + 4);

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    // Work unit = (query tile, head). Blocks are handed out heaviest first:
    // under the causal mask the last query tile has the most key tiles.
    const int bh = static_cast<int>(blockIdx.x % static_cast<unsigned>(p.num_heads_total));
    const int qt = p.num_q_tiles - 1 - static_cast<int>(blockIdx.x / static_cast<unsigned>(p.num_heads_total));
    const int i0 = qt * kBlockM;
    const int row = warp * 32 + lane;  // query row in the tile == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

    if (warp == 0) {
        ptx::tmem_alloc(ptx::smem_u32(tmem_slot), Cfg::kTmemCols);
        ptx::tmem_relinquish();
    }
    if (tid == 32) {
        for (int i = 0; i < Cfg::kNumBars; ++i) ptx::mbar_init(bar_q + 8 * i, 1);
        *abort_flag = 0;
        ptx::fence_mbar_init();
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    ptx::tc_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem;        // S (fp32), later P (bf16x2) in its first 64 columns
    const uint32_t tO = tmem + 128;  // O accumulator (fp32), D columns

    const int n_k_tiles = (p.N + kBlockN - 1) / kBlockN;
    const int n_kv = CAUSAL ? min(qt + 1, n_k_tiles) : n_k_tiles;
    constexpr uint32_t kIdescS = ptx::idesc_bf16_f32(128, kBlockN, false, false);
    constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(128, 64, false, true);

    if (tid == 0) {
        ptx::prefetch_tensormap(&tm_q);
        ptx::prefetch_tensormap(&tm_k);
        ptx::prefetch_tensormap(&tm_v);
        ptx::mbar_arrive_expect_tx(bar_q, Cfg::kTileBytes);
        for (int c = 0; c < D / kBoxCols; ++c)
            ptx::tma_load_3d(sQ + c * kBoxBytes, &tm_q, bar_q, c * kBoxCols, i0, bh);
    }

    float m_run = -INFINITY;  // running max of scale*log2(e)*S (base 2)
    float l_run = 0.f;        // running sum of 2^(S*c - m)
    bool failed = false;

    for (int j = 0; j < n_kv; ++j) {
        const uint32_t ph = static_cast<uint32_t>(j & 1);
        if (tid == 0) {
            ptx::mbar_arrive_expect_tx(bar_kv, 2 * Cfg::kTileBytes);
            for (int c = 0; c < D / kBoxCols; ++c) {
                ptx::tma_load_3d(sK + c * kBoxBytes, &tm_k, bar_kv, c * kBoxCols, j * kBlockN, bh);
                ptx::tma_load_3d(sV + c * kBoxBytes, &tm_v, bar_kv, c * kBoxCols, j * kBlockN, bh);
            }
            bool ok = true;
            if (j == 0) ok = wait_phase(bar_q, 0, abort_flag, kStatusTimeoutLoad, p.wait_limit_ns);
            ok = ok && wait_phase(bar_kv, ph, abort_flag, kStatusTimeoutLoad, p.wait_limit_ns);
            if (ok) {
                ptx::tc_fence_after_sync();
                // S = Q·Kᵀ: K = D in steps of 16; each 64-column box holds 4 steps of 32 bytes.
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                    ptx::mma_ss(tS, ptx::sdesc_sw128(sQ + off, 16, 1024), ptx::sdesc_sw128(sK + off, 16, 1024),
                                kIdescS, kk > 0 ? 1u : 0u);
                }
                ptx::mma_commit(bar_s);
            }
        }
        bool ok = wait_phase(bar_s, ph, abort_flag, kStatusTimeoutMma, p.wait_limit_ns);
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        __syncwarp();  // TMEM loads/stores below are warp-collective
        ptx::tc_fence_after_sync();

        // ---- this thread's row of S
        float s[kBlockN];
        {
            uint32_t r0[32], r1[32], r2[32], r3[32];
            ptx::tmem_ld_32x32b_x32(tS + lane_base + 0, r0);
            ptx::tmem_ld_32x32b_x32(tS + lane_base + 32, r1);
            ptx::tmem_ld_32x32b_x32(tS + lane_base + 64, r2);
            ptx::tmem_ld_32x32b_x32(tS + lane_base + 96, r3);
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

        // ---- mask: keys past the end, and keys after the query under the causal mask
        const int key0 = j * kBlockN;
        if (key0 + kBlockN > p.N || (CAUSAL && j == qt)) {
            const int qi = i0 + row;
#pragma unroll
            for (int c = 0; c < kBlockN; ++c) {
                const int key = key0 + c;
                if (key >= p.N || (CAUSAL && key > qi)) s[c] = -INFINITY;
            }
        }

        // ---- online softmax update (base 2)
        float mx = s[0];
#pragma unroll
        for (int c = 1; c < kBlockN; ++c) mx = fmaxf(mx, s[c]);
        const float m_new = fmaxf(m_run, mx * p.scale_log2);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;  // a fully masked row stays finite
        const float alpha = ptx::ex2_approx(m_run - m_use);
        float sum = 0.f;
#pragma unroll
        for (int c = 0; c < kBlockN; ++c) {
            s[c] = ptx::ex2_approx(fmaf(s[c], p.scale_log2, -m_use));
            sum += s[c];
        }
        l_run = l_run * alpha + sum;
        m_run = m_new;

        // ---- O *= alpha when the max moved (TMEM access is warp-collective)
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(tO + lane_base + c * 32, r);
                ptx::tmem_wait_ld(r);
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha);
                ptx::tmem_st_32x32b_x32(tO + lane_base + c * 32, r);
            }
        }

        // ---- P = bf16(p)
        if constexpr (P_IN_TMEM) {
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t r[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) r[i] = ptx::pack_bf16x2(s[c * 64 + 2 * i], s[c * 64 + 2 * i + 1]);
                ptx::tmem_st_32x32b_x32(tS + lane_base + c * 32, r);
            }
        } else {
            uint8_t* sp = smem + Cfg::kOffP;
#pragma unroll
            for (int c = 0; c < kBlockN; c += 8) {
                uint4 w;
                w.x = ptx::pack_bf16x2(s[c + 0], s[c + 1]);
                w.y = ptx::pack_bf16x2(s[c + 2], s[c + 3]);
                w.z = ptx::pack_bf16x2(s[c + 4], s[c + 5]);
                w.w = ptx::pack_bf16x2(s[c + 6], s[c + 7]);
                *reinterpret_cast<uint4*>(sp + (c / 64) * kBoxBytes + sw128_offset(row, (c % 64) / 8)) = w;
            }
            ptx::fence_proxy_async_smem();
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before_sync();
        __syncthreads();

        if (tid == 0) {
            ptx::tc_fence_after_sync();
            // O += P·V: K = 128 keys in steps of 16 (2048 bytes of V); N = D in 64-wide boxes.
#pragma unroll
            for (int kk = 0; kk < kBlockN / 16; ++kk) {
#pragma unroll
                for (int dc = 0; dc < D / kBoxCols; ++dc) {
                    const uint64_t bdesc = ptx::sdesc_sw128(sV + dc * kBoxBytes + kk * 2048, 1024, 1024);
                    const uint32_t acc = (j > 0 || kk > 0) ? 1u : 0u;
                    if constexpr (P_IN_TMEM) {
                        ptx::mma_ts(tO + dc * 64, tS + kk * 8, bdesc, kIdescPV, acc);
                    } else {
                        const uint32_t off = (kk >> 2) * kBoxBytes + (kk & 3) * 32;
                        ptx::mma_ss(tO + dc * 64, ptx::sdesc_sw128(sbase + Cfg::kOffP + off, 16, 1024), bdesc,
                                    kIdescPV, acc);
                    }
                }
            }
            ptx::mma_commit(bar_o);
        }
        ok = wait_phase(bar_o, ph, abort_flag, kStatusTimeoutMma, p.wait_limit_ns);
        if (__syncthreads_or(!ok)) {
            failed = true;
            break;
        }
        __syncwarp();  // TMEM loads/stores below are warp-collective
        ptx::tc_fence_after_sync();
    }

    if (!failed) {
        // ---- epilogue: O/l -> bf16 -> shared memory (Q's tile is free) -> TMA store
        const float inv_l = 1.0f / l_run;
        uint8_t* so = smem + Cfg::kOffQ;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(tO + lane_base + c * 32, r);
            ptx::tmem_wait_ld(r);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                uint4 w;
                w.x = ptx::pack_bf16x2(__uint_as_float(r[q4 * 8 + 0]) * inv_l, __uint_as_float(r[q4 * 8 + 1]) * inv_l);
                w.y = ptx::pack_bf16x2(__uint_as_float(r[q4 * 8 + 2]) * inv_l, __uint_as_float(r[q4 * 8 + 3]) * inv_l);
                w.z = ptx::pack_bf16x2(__uint_as_float(r[q4 * 8 + 4]) * inv_l, __uint_as_float(r[q4 * 8 + 5]) * inv_l);
                w.w = ptx::pack_bf16x2(__uint_as_float(r[q4 * 8 + 6]) * inv_l, __uint_as_float(r[q4 * 8 + 7]) * inv_l);
                const int col = c * 32 + q4 * 8;
                *reinterpret_cast<uint4*>(so + (col / 64) * kBoxBytes + sw128_offset(row, (col % 64) / 8)) = w;
            }
        }
        ptx::fence_proxy_async_smem();
        if (p.lse != nullptr && i0 + row < p.N) {
            const float m_use = (m_run == -INFINITY) ? 0.f : m_run;
            p.lse[static_cast<size_t>(bh) * p.N + i0 + row] = (m_use + log2f(l_run)) * 0.69314718055994531f;
        }
    }
    __syncthreads();
    if (tid == 0) {
        if (!failed) {
            for (int c = 0; c < D / kBoxCols; ++c)
                ptx::tma_store_3d(&tm_o, sQ + c * kBoxBytes, c * kBoxCols, i0, bh);
            ptx::bulk_commit_group();
            ptx::bulk_wait_group0();
        }
        // drain: every MMA this thread issued has finished before TMEM is freed
        ptx::mma_commit(bar_fin);
        wait_drain(bar_fin, 0, 100000000ull);
    }
    ptx::tc_fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        ptx::tc_fence_after_sync();
        ptx::tmem_dealloc(tmem, Cfg::kTmemCols);
    }
}

}  // namespace fa
