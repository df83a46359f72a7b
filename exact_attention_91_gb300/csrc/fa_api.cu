// C ABI of libfa.so: argument checks, TMA tensor maps, kernel selection and
// launch. Declarations and the contract of every entry point are in fa.h.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include "fa.h"
#include "fa_fwd_kernel.cuh"

namespace {

constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;
constexpr int kMaxDevices = 64;

std::mutex g_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
unsigned long long g_wait_limit_ns = kDefaultWaitLimitNs;

// Work-queue slots of the persistent kernel: {next item, CTAs finished},
// one 128-byte line each, in a fixed array of the library (zero when the
// library is loaded; a launch finds its slot zero and leaves it zero).
// Ordinary launches take the next of 64 slots in turn, so that many may be in
// flight on different streams without sharing one. A launch captured into a
// CUDA graph keeps the slot it drew at capture for every replay; it draws
// from 192 further slots that no ordinary launch uses, so a replay never
// shares one with an ordinary launch, nor with another captured launch until
// 192 more have been captured.
constexpr int kSchedSlots = 64;
constexpr int kGraphSlots = 192;
constexpr int kSchedSlotWords = 32;
static __device__ __align__(256) unsigned g_sched_ring[(kSchedSlots + kGraphSlots) * kSchedSlotWords];

// Most CTAs that share out one unit's key tiles (the size of a portable
// thread-block cluster).
constexpr int kMaxClusterSplit = 8;

struct DeviceState {
    bool probed = false;
    int status = FA_OK;  // FA_OK, FA_ERR_UNSUPPORTED_ARCH
    int sm_count = 0;
    unsigned* sched = nullptr;  // device address of g_sched_ring on this device
    std::atomic<unsigned> sched_next{0};
    std::atomic<unsigned> graph_next{0};
    std::atomic<bool> kernels_ready{false};  // shared-memory attributes of every kernel set
};
DeviceState g_devices[kMaxDevices];

// Looks up the device address of the work-queue ring once per device (with
// that device current). In host code the array's name is only a host-side
// stand-in; the kernels must be given this address.
int ensure_sched(DeviceState& st) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (st.sched) return FA_OK;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_sched_ring) != cudaSuccess || ptr == nullptr) {
        cudaGetLastError();
        return FA_ERR_LAUNCH;
    }
    st.sched = static_cast<unsigned*>(ptr);
    return FA_OK;
}

int resolve_encode() {
    if (g_encode) return FA_OK;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr) {
        cudaGetLastError();
        return FA_ERR_LAUNCH;
    }
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return FA_OK;
}

// Checks the current device once: it must be compute capability 10.3.
int probe_device(int* dev_out, DeviceState** st_out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return FA_ERR_NO_DEVICE;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState& st = g_devices[dev];
    if (!st.probed) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return FA_ERR_NO_DEVICE;
        }
        st.status = (major == 10 && minor == 3) ? FA_OK : FA_ERR_UNSUPPORTED_ARCH;
        st.sm_count = sms;
        st.probed = true;
    }
    if (st.status == FA_OK) {
        int rc = resolve_encode();
        if (rc != FA_OK) return rc;
    }
    *dev_out = dev;
    *st_out = &st;
    return st.status;
}

// Work items of an equal-length launch over `units` units of (head, 256
// query rows) on `sms` SMs: every unit whole, except:
//  * a non-causal problem whose last wave of whole units would fill at most
//    half the SMs runs those last units as two half items each (one 128-row
//    tile, its key tiles shared out between the two softmax warpgroups and
//    merged inside the CTA), so that wave takes half as long;
//  * a causal problem with at most half as many units as SMs runs every unit
//    as two half items, so that the longest chain of key tiles (a unit's
//    last tile) is shared by two warpgroups.
// A half item needs at least 4 key tiles (non-causal) or 2 (causal), and the
// units' second tiles must hold rows (so no half item lies wholly past N).
void plan_items(long long units, int N, int sms, bool causal, long long* n_full, long long* n_items) {
    *n_full = units;
    *n_items = units;
    const long long nkt = (static_cast<long long>(N) + fa::kBlockN - 1) / fa::kBlockN;
    const long long nqb = (static_cast<long long>(N) + 2 * fa::kBlockM - 1) / (2 * fa::kBlockM);
    if (sms <= 0 || (2 * nqb - 1) * fa::kBlockM >= N) return;
    if (causal) {
        if (nkt < 2 || 2 * units > sms) return;
        *n_full = 0;
        *n_items = 2 * units;
        return;
    }
    if (nkt < 4) return;
    const long long r = units % sms;
    if (r == 0 || 2 * r > sms) return;
    *n_full = units - r;
    *n_items = units + r;
}

// Number of CTAs that share out each unit's key range in a variable-length
// batch (the cluster size of the launch). Units are (sequence, head,
// 256-query block); with few of them (decode: one query per sequence) most
// SMs would sit idle. One CTA streams K/V at about 60 GB/s (measured on
// GB300, decode at d = 128), so about 0.6 x the SM count of CTAs at work
// reach the HBM limit, and every split beyond that only adds its fixed cost
// (Q load, pipeline fill, merge). The count is the fewest splits that give
// that many items, with at least 4 key tiles (by the mean key count per
// sequence) per split, 8 (a portable cluster) at most.
int choose_nsplit_varlen(long long units, long long B, long long total_k, int sms) {
    const long long kt = (total_k / B + fa::kBlockN - 1) / fa::kBlockN;  // mean key tiles per sequence
    if (sms <= 0 || units <= 0 || kt < 8) return 1;
    const long long target = (6LL * sms + 9) / 10;
    if (units >= target) return 1;
    const long long want = (target + units - 1) / units;
    return static_cast<int>(std::max<long long>(1, std::min<long long>({want, kt / 4, kMaxClusterSplit})));
}

int varlen_splits(long long units, long long B, long long total_k, int sms) {
    return choose_nsplit_varlen(units, B, total_k, sms);
}

// 3-D view [B*H][N][d] of a contiguous bf16 [B,H,N,d] tensor, boxes of
// 128 rows x 64 columns (128 bytes, 128-byte swizzle). Rows past N inside a
// head read as zero and are not written by stores.
int encode_map(CUtensorMap* map, const void* ptr, int BH, int N, int d) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(N) * d * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(fa::kBoxCols), static_cast<cuuint32_t>(fa::kBlockM), 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_LAUNCH;
}

// 3-D view (d, H, total) of a token-major bf16 [total, H, d] tensor: a box is
// 128 consecutive tokens x 64 columns of one head. Tokens past `total` read
// as zero.
int encode_map_tokens(CUtensorMap* map, const void* ptr, int total, int H, int d) {
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(total)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, static_cast<cuuint64_t>(H) * d * 2};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(fa::kBoxCols), 1, static_cast<cuuint32_t>(fa::kBlockM)};
    const cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FA_OK : FA_ERR_LAUNCH;
}

bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

// Warp-specialised kernel: one CTA per SM (its shared memory and all 512
// TMEM columns keep it alone on the SM). With a work-queue slot the grid is
// persistent (min(items, SMs) CTAs loop over the items); without one
// (prm.sched == null: no more items than SMs, or a cluster split) every CTA
// runs the one item blockIdx.x, the CTAs of a unit's shares forming one
// cluster when nsplit > 1.
template <int D, bool CAUSAL, bool VARLEN, bool HALF>
int launch_kernel(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& to,
                  const fa::FwdParams& prm, int sm_count, cudaStream_t stream) {
    using Cfg = fa::WsCfg<D>;
    auto kernel = fa::fa_fwd_kernel<D, CAUSAL, VARLEN, HALF>;
    if (prm.nsplit > 1) {
        cudaLaunchConfig_t cfg{};
        cfg.gridDim = dim3(static_cast<unsigned>(prm.n_items), 1, 1);
        cfg.blockDim = dim3(Cfg::kThreads, 1, 1);
        cfg.dynamicSmemBytes = Cfg::kSmemBytes;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = static_cast<unsigned>(prm.nsplit);
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kernel, tq, tk, tv, to, prm) != cudaSuccess) {
            cudaGetLastError();
            return FA_ERR_LAUNCH;
        }
        return FA_OK;
    }
    const unsigned grid =
        static_cast<unsigned>(prm.sched == nullptr || prm.n_items < sm_count ? prm.n_items : sm_count);
    kernel<<<grid, Cfg::kThreads, Cfg::kSmemBytes, stream>>>(tq, tk, tv, to, prm);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

// HALF: the launch has half items (prm.n_items > prm.n_full; equal length only)
template <bool VARLEN, bool HALF>
int launch_any(int d, bool causal, const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
               const CUtensorMap& to, const fa::FwdParams& prm, int sms, cudaStream_t s) {
    static_assert(!(VARLEN && HALF), "half items are equal-length only");
    if (d == 64)
        return causal ? launch_kernel<64, true, VARLEN, HALF>(tq, tk, tv, to, prm, sms, s)
                      : launch_kernel<64, false, VARLEN, HALF>(tq, tk, tv, to, prm, sms, s);
    return causal ? launch_kernel<128, true, VARLEN, HALF>(tq, tk, tv, to, prm, sms, s)
                  : launch_kernel<128, false, VARLEN, HALF>(tq, tk, tv, to, prm, sms, s);
}

template <typename Kernel>
bool set_smem_attr(Kernel kernel, int bytes) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess) return true;
    cudaGetLastError();
    return false;
}

// The dynamic shared memory size of every kernel, set once per device (with
// that device current) by its first call that is not being captured.
int prepare_kernels(DeviceState& st) {
    if (st.kernels_ready.load(std::memory_order_acquire)) return FA_OK;
    std::lock_guard<std::mutex> lock(g_mu);
    if (st.kernels_ready.load(std::memory_order_relaxed)) return FA_OK;
    const int b64 = fa::WsCfg<64>::kSmemBytes, b128 = fa::WsCfg<128>::kSmemBytes;
    // <D, CAUSAL, VARLEN, HALF>
    const bool ok = set_smem_attr(fa::fa_fwd_kernel<64, false, false, false>, b64) &&
                    set_smem_attr(fa::fa_fwd_kernel<64, true, false, false>, b64) &&
                    set_smem_attr(fa::fa_fwd_kernel<128, false, false, false>, b128) &&
                    set_smem_attr(fa::fa_fwd_kernel<128, true, false, false>, b128) &&
                    set_smem_attr(fa::fa_fwd_kernel<64, false, false, true>, b64) &&
                    set_smem_attr(fa::fa_fwd_kernel<64, true, false, true>, b64) &&
                    set_smem_attr(fa::fa_fwd_kernel<128, false, false, true>, b128) &&
                    set_smem_attr(fa::fa_fwd_kernel<128, true, false, true>, b128) &&
                    set_smem_attr(fa::fa_fwd_kernel<64, false, true, false>, b64) &&
                    set_smem_attr(fa::fa_fwd_kernel<64, true, true, false>, b64) &&
                    set_smem_attr(fa::fa_fwd_kernel<128, false, true, false>, b128) &&
                    set_smem_attr(fa::fa_fwd_kernel<128, true, true, false>, b128);
    if (!ok) return FA_ERR_LAUNCH;
    st.kernels_ready.store(true, std::memory_order_release);
    return FA_OK;
}

// Whether `stream` is being captured into a CUDA graph (-1: the query failed,
// or the capture was already invalidated).
int capturing(cudaStream_t stream) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) {
        cudaGetLastError();
        return -1;
    }
    if (cs == cudaStreamCaptureStatusNone) return 0;
    return cs == cudaStreamCaptureStatusActive ? 1 : -1;
}

// The device's launch setup (kernel attributes, the ring's address), made by
// its first ordinary call; a call made while `stream` is being captured
// needs it made already. *captured tells which of the two it was.
int ready_for_launch(DeviceState& st, cudaStream_t stream, bool* captured) {
    const int cap = capturing(stream);
    if (cap < 0) return FA_ERR_LAUNCH;
    *captured = cap == 1;
    if (cap == 0) return (prepare_kernels(st) == FA_OK && ensure_sched(st) == FA_OK) ? FA_OK : FA_ERR_LAUNCH;
    std::lock_guard<std::mutex> lock(g_mu);
    return (st.kernels_ready.load(std::memory_order_relaxed) && st.sched != nullptr) ? FA_OK : FA_ERR_LAUNCH;
}

// The work-queue slot of a launch (ordinary and captured launches draw from
// separate parts of the ring).
unsigned* take_sched_slot(DeviceState& st, bool captured) {
    if (!captured) return st.sched + (st.sched_next.fetch_add(1) % kSchedSlots) * kSchedSlotWords;
    return st.sched + (kSchedSlots + st.graph_next.fetch_add(1) % kGraphSlots) * kSchedSlotWords;
}

// One warp waits on an mbarrier phase that nothing completes, through the
// same bounded wait the forward kernel uses: after `limit_ns` it records
// kStatusTimeoutOther in the device status word and returns.
__global__ void __launch_bounds__(32, 1) fa_selftest_timeout_kernel(unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        fa::ptx::mbar_init(fa::ptx::smem_u32(&bar), 1);
        fa::ptx::fence_mbar_init();
    }
    __syncwarp();
    fa::wait_phase_warp(fa::ptx::smem_u32(&bar), 0, &abort_flag, fa::kStatusTimeoutOther, limit_ns);
}

// 2^x for n arguments, with the instruction the softmax uses
// (ex2.approx.ftz.f32) and with CUDA's exp2f, so that a test can hold the
// former to its error bound.
__global__ void __launch_bounds__(256) fa_selftest_exp2_kernel(const float* x, float* y_approx, float* y_exp2f,
                                                               int n) {
    const int i = static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x);
    if (i < n) {
        y_approx[i] = fa::ptx::ex2_approx(x[i]);
        y_exp2f[i] = exp2f(x[i]);
    }
}

// Throughput probe of the exponential unit. Each of the block's 1024
// threads runs 8 independent chains of `iters` dependent
// ex2.approx.ftz.f32 (x <- -2^x, which stays in [-1, -0.5]); thread 0 records
// the block's clock64 span between two block barriers. The requested dynamic
// shared memory keeps one block per SM, so ex2 per SM clock = 8192 * iters /
// cycles[b].
constexpr int kEx2RateThreads = 1024, kEx2RateChains = 8, kEx2RateSmem = 120 * 1024;
__global__ void __launch_bounds__(1024) fa_selftest_ex2_rate_kernel(long long* cycles, float* sink, int iters) {
    float x[kEx2RateChains];
#pragma unroll
    for (int c = 0; c < kEx2RateChains; ++c) x[c] = -0.5f - 0.0625f * static_cast<float>(c);
    __syncthreads();
    const long long t0 = clock64();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < kEx2RateChains; ++c) x[c] = -fa::ptx::ex2_approx(x[c]);
    }
    __syncthreads();
    const long long t1 = clock64();
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < kEx2RateChains; ++c) acc += x[c];
    sink[static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x] = acc;
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
}

// Host-side checks shared by the equal-length entry points: FA_OK, or the
// code of the first violated rule. *units receives B*H*ceil(N/256).
int check_dense(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
                float scale, long long* units) {
    if (!q || !k || !v || !o) return FA_ERR_NULL_PTR;
    if (B < 1 || H < 1 || N < 1) return FA_ERR_BAD_SHAPE;
    const long long BH = static_cast<long long>(B) * H;
    const long long nqb = (static_cast<long long>(N) + 2 * fa::kBlockM - 1) / (2 * fa::kBlockM);
    // work items (at most twice the units) plus one over-claim per CTA fit the int counter
    if (BH > 0x7fffffffLL || 2 * BH * nqb > 0x7fffffffLL - 65536) return FA_ERR_BAD_SHAPE;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_HEAD_DIM;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_BAD_SCALE;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                          reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
    if ((mis & 15u) != 0 || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_MISALIGNED;
    const size_t tensor_bytes = static_cast<size_t>(BH) * N * d * 2;
    const size_t lse_bytes = static_cast<size_t>(BH) * N * 4;
    if (overlaps(o, tensor_bytes, q, tensor_bytes) || overlaps(o, tensor_bytes, k, tensor_bytes) ||
        overlaps(o, tensor_bytes, v, tensor_bytes))
        return FA_ERR_ALIAS;
    if (lse && (overlaps(lse, lse_bytes, q, tensor_bytes) || overlaps(lse, lse_bytes, k, tensor_bytes) ||
                overlaps(lse, lse_bytes, v, tensor_bytes) || overlaps(lse, lse_bytes, o, tensor_bytes)))
        return FA_ERR_ALIAS;
    *units = BH * nqb;
    return FA_OK;
}

// Tensor maps, parameters and the launch of an equal-length forward pass
// whose work-queue slot is `sched`.
int run_dense(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d,
              float scale, int causal, long long units, unsigned* sched, int sms, cudaStream_t s) {
    const int bh = B * H;
    CUtensorMap tq, tk, tv, to;
    if (encode_map(&tq, q, bh, N, d) != FA_OK || encode_map(&tk, k, bh, N, d) != FA_OK ||
        encode_map(&tv, v, bh, N, d) != FA_OK || encode_map(&to, o, bh, N, d) != FA_OK)
        return FA_ERR_LAUNCH;
    fa::FwdParams prm{};
    prm.lse = lse;
    prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    {
        std::lock_guard<std::mutex> lock(g_mu);
        prm.wait_limit_ns = g_wait_limit_ns;
    }
    prm.sched = sched;
    prm.num_heads_total = bh;
    prm.nqb = static_cast<int>((static_cast<long long>(N) + 2 * fa::kBlockM - 1) / (2 * fa::kBlockM));
    prm.N = N;
    long long n_full = units, n_items = units;
    plan_items(units, N, sms, causal != 0, &n_full, &n_items);
    prm.n_full = static_cast<int>(n_full);
    prm.n_items = static_cast<int>(n_items);
    prm.nsplit = 1;
    // no more items than SMs: one item per CTA, no work queue to claim from or reset
    if (n_items <= sms) prm.sched = nullptr;
    return n_items > n_full ? launch_any<false, true>(d, causal != 0, tq, tk, tv, to, prm, sms, s)
                            : launch_any<false, false>(d, causal != 0, tq, tk, tv, to, prm, sms, s);
}

}  // namespace

extern "C" {

int fa_abi_version(void) { return FA_ABI_VERSION; }

int fa_selftest_wait_timeout(void* stream, unsigned long long limit_ns) {
    int dev = -1;
    DeviceState* st = nullptr;
    const int rc = probe_device(&dev, &st);
    if (rc != FA_OK) return rc;
    if (limit_ns < 200000ull || limit_ns > 1000000000ull) return FA_ERR_BAD_SHAPE;
    fa_selftest_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_selftest_exp2(const float* x, float* y_approx, float* y_exp2f, int n, void* stream) {
    if (n < 0) return FA_ERR_BAD_SHAPE;
    if (n == 0) return FA_OK;
    if (!x || !y_approx || !y_exp2f) return FA_ERR_NULL_PTR;
    if (((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y_approx) |
          reinterpret_cast<uintptr_t>(y_exp2f)) & 3u) != 0)
        return FA_ERR_MISALIGNED;
    int dev = -1;
    DeviceState* st = nullptr;
    const int rc = probe_device(&dev, &st);
    if (rc != FA_OK) return rc;
    const unsigned blocks = static_cast<unsigned>((static_cast<long long>(n) + 255) / 256);
    fa_selftest_exp2_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(x, y_approx, y_exp2f, n);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_selftest_ex2_rate(long long* cycles, float* sink, int blocks, int iters, void* stream) {
    if (blocks < 1 || blocks > 4096 || iters < 1 || iters > (1 << 20)) return FA_ERR_BAD_SHAPE;
    if (!cycles || !sink) return FA_ERR_NULL_PTR;
    if ((reinterpret_cast<uintptr_t>(cycles) & 7u) != 0 || (reinterpret_cast<uintptr_t>(sink) & 3u) != 0)
        return FA_ERR_MISALIGNED;
    int dev = -1;
    DeviceState* st = nullptr;
    const int rc = probe_device(&dev, &st);
    if (rc != FA_OK) return rc;
    if (cudaFuncSetAttribute(fa_selftest_ex2_rate_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kEx2RateSmem) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_LAUNCH;
    }
    fa_selftest_ex2_rate_kernel<<<static_cast<unsigned>(blocks), kEx2RateThreads, kEx2RateSmem,
                                  static_cast<cudaStream_t>(stream)>>>(cycles, sink, iters);
    return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

const char* fa_strerror(int status) {
    switch (status) {
        case FA_OK: return "ok";
        case FA_ERR_NULL_PTR: return "q, k, v or o is a null pointer";
        case FA_ERR_BAD_SHAPE: return "B, H and N must be >= 1 and within the size limits";
        case FA_ERR_UNSUPPORTED_HEAD_DIM: return "head dimension d must be 64 or 128";
        case FA_ERR_MISALIGNED: return "q, k, v, o must be 16-byte aligned and lse 4-byte aligned";
        case FA_ERR_NO_DEVICE: return "no usable CUDA device";
        case FA_ERR_UNSUPPORTED_ARCH: return "the current device is not compute capability 10.3 (sm_103a)";
        case FA_ERR_LAUNCH: return "tensor-map encoding or kernel launch failed";
        case FA_ERR_DEVICE_TIMEOUT: return "a kernel gave up waiting on an mbarrier";
        case FA_ERR_BAD_SCALE: return "scale must be finite and > 0";
        case FA_ERR_ALIAS: return "an output buffer overlaps an input buffer or the other output";
        default: return "unknown fa status";
    }
}

void fa_set_wait_limit_ns(unsigned long long ns) {
    std::lock_guard<std::mutex> lock(g_mu);
    g_wait_limit_ns = ns ? ns : kDefaultWaitLimitNs;
}

int fa_device_status(void* stream, unsigned* bits) {
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_NO_DEVICE;
    }
    unsigned word = 0;
    const unsigned zero = 0;
    if (cudaMemcpyFromSymbol(&word, fa::g_status, sizeof(word)) != cudaSuccess ||
        cudaMemcpyToSymbol(fa::g_status, &zero, sizeof(zero)) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_LAUNCH;
    }
    if (bits) *bits = word;
    return word ? FA_ERR_DEVICE_TIMEOUT : FA_OK;
}

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int N, int d, float scale,
           int causal, void* stream) {
    long long units = 0;
    int rc = check_dense(q, k, v, o, lse, B, H, N, d, scale, &units);
    if (rc != FA_OK) return rc;
    int dev = -1;
    DeviceState* st = nullptr;
    rc = probe_device(&dev, &st);
    if (rc != FA_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool captured = false;
    if (ready_for_launch(*st, s, &captured) != FA_OK) return FA_ERR_LAUNCH;
    return run_dense(q, k, v, o, lse, B, H, N, d, scale, causal, units, take_sched_slot(*st, captured),
                     st->sm_count, s);
}

int fa_varlen_num_splits(int B, int H, int total_k, int max_seqlen_q, int sm_count) {
    if (B < 1 || H < 1 || total_k < 0 || max_seqlen_q < 0 || sm_count < 1) return FA_ERR_BAD_SHAPE;
    const long long BH = static_cast<long long>(B) * H;
    const long long nqb = (static_cast<long long>(max_seqlen_q) + 2 * fa::kBlockM - 1) / (2 * fa::kBlockM);
    if (BH > 0x7fffffffLL || BH * nqb > 0x7fffffffLL - 65536) return FA_ERR_BAD_SHAPE;
    return varlen_splits(BH * nqb, B, total_k, sm_count);
}

int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse, const int* cu_seqlens_q,
                  const int* cu_seqlens_k, int B, int H, int total_q, int total_k, int max_seqlen_q, int d,
                  float scale, int causal, void* stream) {
    if (B < 1 || H < 1 || total_q < 0 || total_k < 0 || max_seqlen_q < 0 || max_seqlen_q > total_q)
        return FA_ERR_BAD_SHAPE;
    // (an empty tensor may come with a null pointer)
    if (!cu_seqlens_q || !cu_seqlens_k || (total_q > 0 && (!q || !o)) || (total_k > 0 && (!k || !v)))
        return FA_ERR_NULL_PTR;
    if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_HEAD_DIM;
    if (!std::isfinite(scale) || !(scale > 0.f)) return FA_ERR_BAD_SCALE;
    const long long BH = static_cast<long long>(B) * H;
    const long long nqb = (static_cast<long long>(max_seqlen_q) + 2 * fa::kBlockM - 1) / (2 * fa::kBlockM);
    // (element offsets are 64-bit; token indices and the unit count, plus one
    // over-claim per CTA, must fit in int)
    if (BH > 0x7fffffffLL || BH * nqb > 0x7fffffffLL - 65536) return FA_ERR_BAD_SHAPE;
    const uintptr_t mis = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
                          reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(o);
    if ((mis & 15u) != 0 || (reinterpret_cast<uintptr_t>(lse) & 3u) != 0 ||
        ((reinterpret_cast<uintptr_t>(cu_seqlens_q) | reinterpret_cast<uintptr_t>(cu_seqlens_k)) & 3u) != 0)
        return FA_ERR_MISALIGNED;
    const size_t q_bytes = static_cast<size_t>(total_q) * H * d * 2, k_bytes = static_cast<size_t>(total_k) * H * d * 2;
    const size_t lse_bytes = static_cast<size_t>(total_q) * H * 4;
    if (overlaps(o, q_bytes, q, q_bytes) || overlaps(o, q_bytes, k, k_bytes) || overlaps(o, q_bytes, v, k_bytes))
        return FA_ERR_ALIAS;
    if (lse && (overlaps(lse, lse_bytes, q, q_bytes) || overlaps(lse, lse_bytes, k, k_bytes) ||
                overlaps(lse, lse_bytes, v, k_bytes) || overlaps(lse, lse_bytes, o, q_bytes)))
        return FA_ERR_ALIAS;

    int dev = -1;
    DeviceState* st = nullptr;
    int rc = probe_device(&dev, &st);
    if (rc != FA_OK) return rc;
    if (total_q == 0 || max_seqlen_q == 0) return FA_OK;  // no query: nothing to write

    CUtensorMap tq, tk, tv, to;
    // a map needs at least one row: an empty key set is read through a one-row view of q
    if (encode_map_tokens(&tq, q, total_q, H, d) != FA_OK ||
        encode_map_tokens(&tk, total_k ? k : q, total_k ? total_k : 1, H, d) != FA_OK ||
        encode_map_tokens(&tv, total_k ? v : q, total_k ? total_k : 1, H, d) != FA_OK ||
        encode_map_tokens(&to, o, total_q, H, d) != FA_OK)
        return FA_ERR_LAUNCH;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool captured = false;
    if (ready_for_launch(*st, s, &captured) != FA_OK) return FA_ERR_LAUNCH;
    const int sms = st->sm_count;
    const long long units = BH * nqb;
    fa::FwdParams prm{};
    prm.lse = lse;
    prm.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634074);
    {
        std::lock_guard<std::mutex> lock(g_mu);
        prm.wait_limit_ns = g_wait_limit_ns;
    }
    prm.num_heads_total = static_cast<int>(BH);
    prm.nqb = static_cast<int>(nqb);
    prm.o = o;
    prm.cu_q = cu_seqlens_q;
    prm.cu_k = cu_seqlens_k;
    prm.heads = H;
    prm.total_q = total_q;
    prm.nsplit = varlen_splits(units, B, total_k, sms);
    prm.n_items = static_cast<int>(units * prm.nsplit);
    prm.n_full = prm.n_items;
    // a cluster split, or no more items than SMs: one item per CTA, no work queue
    prm.sched = (prm.nsplit > 1 || prm.n_items <= sms) ? nullptr : take_sched_slot(*st, captured);
    return launch_any<true, false>(d, causal != 0, tq, tk, tv, to, prm, sms, s);
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Allocation-free entry point.
//
// Some callers cannot have a library call allocate device memory: code that
// runs inside a custom allocator or memory-pool callback (where cudaMalloc
// would re-enter the allocator or synchronise the device at the wrong
// moment), a caller-side memory budget that must account for every byte, or
// a runtime that plans all device memory before it starts. fa_fwd_noalloc is
// the entry point with that promise in its contract: it runs the same kernel
// as fa_fwd with its work-queue counters in the fixed array below, which
// every GPU that loads the library holds until the process exits. It never
// calls cudaMalloc, cudaFree or any allocating routine.
namespace {

// One work-queue slot {next item, CTAs finished}, padded to a 128-byte line.
constexpr int kNoAllocScratchWords = 32;
static __device__ __align__(256) unsigned g_noalloc_scratch[kNoAllocScratchWords];

// Device address of g_noalloc_scratch, per device. In host code the array's
// name is only a host-side stand-in, so the kernel must be given this
// address, looked up once per device with that device current.
unsigned* g_noalloc_ptr[kMaxDevices] = {};

int noalloc_scratch(int dev, unsigned** out) {
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_noalloc_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
            cudaGetLastError();
            return FA_ERR_LAUNCH;
        }
        g_noalloc_ptr[dev] = static_cast<unsigned*>(ptr);
    }
    *out = g_noalloc_ptr[dev];
    return FA_OK;
}

}  // namespace

extern "C" int fa_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                              int N, int d, float scale, int causal, void* stream) {
    // The scratch is one fixed work-queue slot whatever the shape; the shape
    // limits are fa_fwd's.
    long long units = 0;
    int rc = check_dense(q, k, v, o, lse, B, H, N, d, scale, &units);
    if (rc != FA_OK) return rc;
    int dev = -1;
    DeviceState* st = nullptr;
    rc = probe_device(&dev, &st);
    if (rc != FA_OK) return rc;
    unsigned* scratch = nullptr;
    if (noalloc_scratch(dev, &scratch) != FA_OK) return FA_ERR_LAUNCH;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    {
        // kernel attributes are set by an ordinary call, never during a capture
        const int cap = capturing(s);
        if (cap < 0) return FA_ERR_LAUNCH;
        if (cap == 0 ? prepare_kernels(*st) != FA_OK : !st->kernels_ready.load(std::memory_order_acquire))
            return FA_ERR_LAUNCH;
    }
    // the two counters must start at zero (the kernel also leaves them zero)
    if (cudaMemsetAsync(scratch, 0, 2 * sizeof(unsigned), s) != cudaSuccess) {
        cudaGetLastError();
        return FA_ERR_LAUNCH;
    }
    return run_dense(q, k, v, o, lse, B, H, N, d, scale, causal, units, scratch, st->sm_count, s);
}
