/*
 * fa.h — C ABI of the GB300 (sm_103a) exact-attention forward library
 * (libfa.so).
 *
 * The operation is exact softmax attention computed tile by tile with the
 * online softmax, never writing the N×N score matrix to memory:
 *
 *   S = scale · Q Kᵀ,   causal: S[i, j] = -inf for j > i
 *   P = softmax(S) by rows
 *   O = P V,            LSE_i = ln Σ_j exp(S[i, j])
 *
 * Definition: "Mini FlashAttention", §1 "What attention is" (the three-line
 * math and the causal-mask sentence). Streaming form: "Mini FlashAttention",
 * §4 "The flash trick: online softmax" (running max, running sum, rescale of
 * the running output, O = acc / l after the last chunk); "How Did I Write My
 * First FlashAttention Kernel in CUDA?", the pseudo-algorithm steps 1-5 and the
 * surrogate running-output paragraph. Initialisation and final normalisation:
 * the grasp.study lesson on the complete forward pass, "1. Initialization" and
 * "3. Finalization".
 *
 * Plain C types only: device pointers are `const void*` / `void*`, the CUDA
 * stream is passed as `void*` (a cudaStream_t; NULL is the legacy default
 * stream).
 *
 * Every forward kernel allows programmatic dependent launch: a kernel that the
 * caller launches next on the same stream with programmatic stream
 * serialization may start before the forward kernel has finished, and must
 * call cudaGridDependencySynchronize (griddepcontrol.wait) before it reads O
 * or LSE. Launches without that attribute keep plain stream order.
 */
#ifndef FA_H_
#define FA_H_

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. 0 is success; every error is negative. */
typedef enum fa_status {
    FA_OK = 0,
    FA_ERR_NULL_PTR = -1,             /* q, k, v or o is NULL */
    FA_ERR_BAD_SHAPE = -2,            /* B, H or N < 1, or a size past the limits below */
    FA_ERR_UNSUPPORTED_HEAD_DIM = -3, /* d is not 64 or 128 */
    FA_ERR_MISALIGNED = -4,           /* q, k, v, o not 16-byte aligned, or lse not 4-byte aligned */
    FA_ERR_NO_DEVICE = -5,            /* no CUDA device, or the current device cannot be queried */
    FA_ERR_UNSUPPORTED_ARCH = -6,     /* the current device is not compute capability 10.3 */
    FA_ERR_LAUNCH = -7,               /* tensor-map encoding or the kernel launch failed, or a call was
                                         captured into a CUDA graph before the device's first ordinary call */
    FA_ERR_DEVICE_TIMEOUT = -8,       /* a kernel gave up waiting on an mbarrier (see fa_device_status) */
    FA_ERR_BAD_SCALE = -9,            /* scale is not finite, or not > 0 */
    FA_ERR_ALIAS = -10                /* o or lse overlaps q, k or v, or lse overlaps o */
} fa_status;

/*
 * fa_fwd — attention forward pass on the current CUDA device.
 *
 * q, k, v  device, bf16, contiguous [B, H, N, d] (row-major: d fastest).
 *          Read only.
 * o        device, bf16, contiguous [B, H, N, d]. Written: O = P V.
 * lse      device, fp32, contiguous [B, H, N], or NULL to skip it. Written:
 *          the natural-log log-sum-exp of each query row's scaled scores
 *          over the keys the row may see.
 * B, H, N  batch, heads, sequence length (queries = keys = N), each >= 1;
 *          B*H <= 2^31-1 and 2*B*H*ceil(N/256) <= 2^31-1 - 65536 (work
 *          items and one over-claim per CTA fit the int counter).
 * d        head dimension: 64 or 128.
 * scale    score scale (the pages use 1/sqrt(d)); finite and > 0.
 * causal   nonzero: key j is hidden from query i when j > i (top-left
 *          aligned; every row keeps at least its own key).
 * stream   cudaStream_t to run on, as void*; NULL = legacy default stream.
 *
 * Ownership: the caller allocates and owns every buffer; the library keeps
 * no pointer after the call returns and allocates no device memory, neither
 * per call nor once: its only device state is a fixed 32 KB array inside the
 * library (work-queue counters: 256 slots of 128 bytes) and the device status
 * word, which every GPU that loads the library holds until the process exits.
 * Per device it caches the SM count, the kernels' shared-memory attributes
 * and that array's device address, all set by the first ordinary call of any
 * forward entry point on that device (with the device current). Each launch
 * uses one of 64 counter slots in turn and leaves it zeroed, so up to 64
 * launches may be in flight at once on different streams. A non-causal
 * problem whose last wave of work units would leave most SMs idle runs those
 * units as half units (one 128-row query tile whose key tiles the CTA's two
 * softmax warpgroups share out, merged inside the CTA), and so does every
 * unit of a causal problem with at most half as many units as SMs: no
 * scratch memory.
 * The call is asynchronous: argument errors are returned before anything is
 * queued; faults inside the kernel appear at the caller's next
 * synchronisation, and a kernel that gave up on a wait leaves its O/LSE rows
 * unwritten and reports through fa_device_status(). The current device must
 * be compute capability 10.3 (sm_103a).
 *
 * CUDA graphs: fa_fwd, fa_fwd_varlen and fa_fwd_noalloc may be called while
 * `stream` is being captured (cudaStreamBeginCapture, torch.cuda.graph),
 * once the device has had one ordinary call of a forward entry point: that
 * call sets what a capture may not (the kernels' shared-memory sizes, the
 * counter array's address). A call captured before then returns
 * FA_ERR_LAUNCH and enqueues nothing. The tensor maps are encoded from the
 * pointers given at capture, so a replay reads and writes those buffers,
 * which must stay allocated while the graph may be replayed (a replay after
 * one was freed reads or writes unmapped or reused memory; torch.cuda.graph
 * returns the allocator's free blocks to the driver when a capture begins). A
 * captured call keeps the counter slot it drew for every replay, from 192
 * slots that ordinary calls never use, so replays may overlap ordinary
 * launches and replays of other graphs on other streams (until 192 calls have
 * been captured on the device, when the slots wrap). fa_fwd_noalloc's one
 * shared slot stays shared when captured.
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * fa_fwd_noalloc — the same attention forward pass as fa_fwd, for callers
 * that cannot let a library call allocate device memory: code running inside
 * an allocator or memory-pool callback, under a memory budget that must
 * account for every byte, or in a runtime that plans all device memory
 * before it starts. (The pages describe no such entry point; it is part of
 * this library's interface only.)
 *
 * Arguments, layouts, ownership, limits and errors are those of fa_fwd,
 * and it gives fa_fwd's results bit for bit. It never calls cudaMalloc,
 * cudaFree or any allocating routine (fa_fwd does not either; this entry
 * point states it as its contract and keeps its own counters): its scratch
 * (one 128-byte work-queue slot) is a fixed array inside the library that
 * every GPU which loads the library keeps until the process exits. The
 * first call on a device looks up that array's device address (with that
 * device current); make the first call before any stream capture. Each call
 * clears the slot's counters on `stream` before its kernel, and every call
 * shares the one slot: calls whose kernels overlap on the GPU (different
 * streams, no ordering between them) race on it and must not be issued. The
 * scratch does not grow with the problem.
 */
int fa_fwd_noalloc(const void* q, const void* k, const void* v, void* o, float* lse,
                   int B, int H, int N, int d, float scale, int causal, void* stream);

/*
 * fa_fwd_varlen — the same forward pass over a batch of B sequences of
 * different lengths, each with its own number of queries and keys ("Mini
 * FlashAttention", §4 "The flash trick: online softmax", checks the loop on
 * ragged sequences).
 *
 *   q, o   bf16 [total_q, H, d], token-major (a token's H heads side by side),
 *          device, contiguous, 16-byte aligned
 *   k, v   bf16 [total_k, H, d], likewise
 *   lse    fp32 [H, total_q], device, or NULL; natural-log log-sum-exp
 *   cu_seqlens_q, cu_seqlens_k
 *          int32 [B + 1], device: sequence b holds query tokens
 *          cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and key tokens
 *          cu_seqlens_k[b] .. cu_seqlens_k[b+1]-1. The caller guarantees
 *          cu[0] = 0, non-decreasing offsets, cu_seqlens_q[B] = total_q,
 *          cu_seqlens_k[B] = total_k and every query count <= max_seqlen_q;
 *          the library reads them only on the GPU. Offsets that break this
 *          give undefined values but no write outside o[0, total_q) and
 *          lse's rows (reads past total_k see zeros).
 *   max_seqlen_q
 *          the largest query count of the batch (it sizes the launch)
 *   causal non-zero: the mask is aligned at the end of each sequence, so
 *          query i (0-based within its sequence) sees keys j <= i + Nk - Nq;
 *          with Nq = Nk this is fa_fwd's mask, and a single query (decode)
 *          sees every key. A query that sees no key gets O = 0, LSE = -inf.
 *
 * Same return codes as fa_fwd (FA_ERR_BAD_SHAPE for negative totals,
 * max_seqlen_q > total_q, or B*H*ceil(max_seqlen_q/256) >= 2^31 - 65536; q/o
 * and k/v may be NULL when total_q, resp. total_k, is 0); a batch with no
 * query returns FA_OK at once.
 *
 * Work is split into units of (sequence, head, 256 queries). When there are
 * few units for the GPU's SMs (decode: a few sequences of one query against
 * long key sets), each unit's key tiles are shared out among the CTAs of a
 * thread-block cluster (2-8 of them; fa_varlen_num_splits gives how many).
 * Each CTA keeps its partial O, normalised, and its LSE in its own shared
 * memory, and the cluster's first CTA merges them through distributed
 * shared memory: O = sum_s 2^(L_s - L) O_s with L = log2 sum_s 2^L_s (base-2
 * LSEs), the online-softmax rescaling applied across the shares. No device
 * memory is allocated (fa_fwd's ownership rules apply).
 */
int fa_fwd_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                  const int* cu_seqlens_q, const int* cu_seqlens_k, int B, int H, int total_q,
                  int total_k, int max_seqlen_q, int d, float scale, int causal, void* stream);

/*
 * fa_varlen_num_splits — host-only, no device call: among how many CTAs
 * (a cluster) fa_fwd_varlen shares out each unit's key range for these sizes
 * on a GPU with `sm_count` SMs (1 = no split, at most 8). Returns
 * FA_ERR_BAD_SHAPE under the same shape rules as fa_fwd_varlen, or when
 * sm_count < 1.
 */
int fa_varlen_num_splits(int B, int H, int total_k, int max_seqlen_q, int sm_count);

/* Static English text for a return code (never NULL). */
const char* fa_strerror(int status);

/*
 * fa_device_status — synchronises `stream` (a cudaStream_t as void*, NULL =
 * legacy default), then reads and clears the current device's status word.
 * Returns FA_OK if no kernel gave up on a wait since the last call,
 * FA_ERR_DEVICE_TIMEOUT if one did (then *bits, if not NULL, receives the
 * word: which kind of wait gave up), or FA_ERR_NO_DEVICE / FA_ERR_LAUNCH if
 * the synchronisation or the read failed.
 */
int fa_device_status(void* stream, unsigned* bits);

/*
 * fa_set_wait_limit_ns — how long a kernel waits on one mbarrier phase before
 * giving up (default 2e9 ns). Applies to launches made after the call, on
 * every device. 0 restores the default.
 */
void fa_set_wait_limit_ns(unsigned long long ns);

/*
 * fa_selftest_wait_timeout — failure-detection self-test. Launches, on
 * `stream`, one warp that waits on an mbarrier phase nothing completes, using
 * the forward kernel's bounded wait with a limit of `limit_ns` (200 µs to 1 s,
 * else FA_ERR_BAD_SHAPE). The wait gives up, records "other wait" (bit 4) in
 * the device status word and the kernel returns; nothing faults or hangs, and
 * the context stays usable. fa_device_status() then reports
 * FA_ERR_DEVICE_TIMEOUT. Returns FA_OK once launched, FA_ERR_NO_DEVICE /
 * FA_ERR_UNSUPPORTED_ARCH / FA_ERR_LAUNCH otherwise. The pages have no
 * counterpart (they have no failure handling).
 */
int fa_selftest_wait_timeout(void* stream, unsigned long long limit_ns);

/*
 * fa_selftest_exp2 — numerics self-test of the exponential. For i < n, writes
 * y_approx[i] = 2^x[i] computed by the instruction the softmax uses
 * (ex2.approx.ftz.f32: subnormal arguments and results flush to zero, 2^-inf
 * = +0) and y_exp2f[i] = CUDA's exp2f(x[i]). x, y_approx, y_exp2f are device
 * fp32 arrays of n elements, 4-byte aligned, owned by the caller; the call is
 * asynchronous on `stream`. Returns FA_OK (also for n = 0), FA_ERR_BAD_SHAPE
 * for n < 0, FA_ERR_NULL_PTR / FA_ERR_MISALIGNED for bad pointers, else the
 * device and launch codes of fa_fwd. The pages have no counterpart (they call
 * exp / expf without stating its accuracy).
 */
int fa_selftest_exp2(const float* x, float* y_approx, float* y_exp2f, int n, void* stream);

/*
 * fa_selftest_ex2_rate — throughput probe of the exponential unit, the
 * softmax's second ceiling beside the tensor cores (one ex2 per query and
 * visible key). Launches `blocks` blocks of 1024 threads, one per SM (each
 * asks for 120 KB of shared memory); every thread runs 8 independent chains
 * of `iters` dependent ex2.approx.ftz.f32. cycles (device, int64 [blocks],
 * 8-byte aligned) receives each block's span in SM clocks; sink (device,
 * fp32 [blocks * 1024], 4-byte aligned) receives the chains' final values so
 * that no work is elided. The rate is 8192 * iters / cycles[b] ex2 per clock
 * of block b's SM. Asynchronous on `stream`. Returns FA_OK once launched,
 * FA_ERR_BAD_SHAPE unless 1 <= blocks <= 4096 and 1 <= iters <= 2^20,
 * FA_ERR_NULL_PTR / FA_ERR_MISALIGNED for bad pointers, else the device and
 * launch codes of fa_fwd. The pages have no counterpart.
 */
int fa_selftest_ex2_rate(long long* cycles, float* sink, int blocks, int iters, void* stream);

/* ABI version of this header (bumped on any incompatible change). */
int fa_abi_version(void);

#define FA_ABI_VERSION 1

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
