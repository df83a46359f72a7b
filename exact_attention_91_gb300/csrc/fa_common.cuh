// Shared pieces of the attention forward kernels: parameters, the device
// status word, bounded mbarrier waits, and the shared-memory swizzle.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"

namespace fa {

// Query rows per tile (BM) and keys per tile (BN). One query row maps to one
// TMEM lane, so a 128-row tile fills all 128 lanes of an M=128 MMA.
constexpr int kBlockM = 128;
constexpr int kBlockN = 128;
// TMA boxes are 64 bf16 wide (128 bytes, the 128-byte swizzle span) and 128
// rows high: 16 KB each. A tile of head dim d is d/64 such boxes.
constexpr int kBoxCols = 64;
constexpr int kBoxBytes = kBlockM * kBoxCols * 2;

// Status bits the kernels OR into the device status word.
enum : unsigned {
    kStatusTimeoutLoad = 1u << 0,     // a wait for a TMA load gave up
    kStatusTimeoutMma = 1u << 1,      // a wait for a tcgen05.mma commit gave up
    kStatusTimeoutSoftmax = 1u << 2,  // a wait for softmax output (P) gave up
    kStatusTimeoutFree = 1u << 3,     // a wait for a free pipeline slot gave up
    kStatusTimeoutOther = 1u << 4,
};

// Parameters of one launch of the forward kernel. Equal-length batches use
// N and n_full; variable-length batches the last group.
struct FwdParams {
    float* lse;           // equal length: [B*H, N]; variable length: [H, total_q]; fp32, or null
    float scale_log2;     // scale * log2(e): scores are kept in base-2 units
    unsigned long long wait_limit_ns;  // give up on an mbarrier wait after this long
    unsigned* sched;      // work-queue slot (next item, CTAs finished): zero at launch, zero again at
                          // exit. Null: every CTA runs the one item blockIdx.x (a cluster split).
    int num_heads_total;  // B*H
    int nqb;              // 256-row query blocks per head (of the longest sequence, variable length)
    int n_items;          // work items of the launch
    // ---- equal length [B, H, N, d]
    int N;                // sequence length (queries = keys)
    int n_full;           // items [0, n_full) are whole units; every later unit runs as two half items
    // ---- variable length [total, H, d]
    void* o;              // [total_q, H, d] bf16 (plain stores: a TMA box would cross sequences)
    const int* cu_q;      // [B + 1] query-token offsets
    const int* cu_k;      // [B + 1] key-token offsets
    int heads;            // H
    int total_q;
    int nsplit;           // CTAs of a cluster that share out each unit's key tiles (1: none)
};

// Device-wide status word (one per device that loads the library). Zero means
// no kernel has given up on a wait since the host last cleared it.
__device__ unsigned int g_status;

// Slow path of a bounded wait. The polling loop touches only the barrier and
// the clock, so a wait that ends normally costs no memory traffic: the abort
// flag (shared memory) and the device status word (global memory: another CTA
// gave up) are read only once the wait has already lasted kQuietNs. On giving
// up it records `site` and raises the CTA abort flag.
__device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, volatile int* cta_abort,
                                          unsigned site, unsigned long long limit_ns) {
    constexpr unsigned long long kQuietNs = 100000;  // 100 us
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            const uint64_t waited = ptx::globaltimer_ns() - t0;
            if (waited < kQuietNs) continue;
            if (*cta_abort) return false;
            if (*reinterpret_cast<volatile unsigned*>(&g_status) != 0u) {
                *cta_abort = 1;
                return false;
            }
            if (waited > limit_ns) {
                atomicOr(&g_status, site);
                *cta_abort = 1;
                return false;
            }
        }
    }
}

// Waits for phase `parity` of barrier `bar`; false if the wait gave up.
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, volatile int* cta_abort,
                                           unsigned site, unsigned long long limit_ns) {
    if (ptx::mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, cta_abort, site, limit_ns);
}

// wait_phase for a whole converged warp: every lane polls, and the result is
// made warp-uniform (false if any lane gave up).
__device__ __forceinline__ bool wait_phase_warp(uint32_t bar, uint32_t parity, volatile int* cta_abort,
                                                unsigned site, unsigned long long limit_ns) {
    const bool ok = wait_phase(bar, parity, cta_abort, site, limit_ns);
    return __all_sync(0xffffffffu, ok);
}

// Final drain before TMEM is freed: waits for an mbarrier phase with a short
// limit of its own, ignoring the abort flag (the point is to let any MMA still
// in flight finish even after the CTA gave up on something else).
__device__ __forceinline__ bool wait_drain(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
    const uint64_t t0 = ptx::globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0 && ptx::globaltimer_ns() - t0 > limit_ns) {
            atomicOr(&g_status, static_cast<unsigned>(kStatusTimeoutOther));
            return false;
        }
    }
}

// Byte offset of 16-byte chunk `chunk` (0..7) of row `row` inside a box
// written with the 128-byte swizzle: rows are 128 bytes apart and the chunk
// index is XORed with the row index modulo 8.
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk) {
    return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

}  // namespace fa
