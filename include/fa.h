/*
 * fa.h -- C ABI of libfa: exact IO-aware scaled-dot-product attention on one
 * NVIDIA GB300 (sm_103a), forward and backward.
 *
 * What it computes.  For each sequence b and query head h, with kv head
 * g = h / (Hq / Hkv) and positions i (query) and j (key) local to the
 * sequence:
 *     S = scale * Q K^T + B_h,   P = softmax(S) row-wise,   O = P V,
 *     LSE_i = log sum_j exp(S_ij)                         (natural log)
 * ("FlashAttention: Faster Attention Without Dropping a Single Interaction",
 * Key design 1, the S/P/O definition; Key design 2, the saved statistic
 * L = m + log l).  B_h[i,j] = -slope_h * (i - j) when ALiBi slopes are given,
 * else 0; with causal != 0, S_ij = -inf for j > i, and with a sliding window
 * w >= 0 also for j < i - w (the causal band i - w <= j <= i; the sliding
 * window is named among the mask variants in the Usage contract table of
 * "FlashAttention: Faster Attention Without Dropping a Single Interaction").
 * The bias is added after scaling and is not scaled.
 * The backward recomputes P from LSE tile by tile (Key design 3):
 *     dV = P^T dO,  dP = dO V^T,  D_i = dO_i . O_i,  dS = P o (dP - D),
 *     dQ = scale * dS K,  dK = scale * dS^T Q,
 * with dK and dV of kv head g summed over the query heads of its group.
 * S and P are never written to device memory.
 *
 * Layouts (all row-major and contiguous; q, k, v, dO, dq, dk, dv have the
 * element type `dtype`, o has `o_dtype`):
 *     q, o, dO, dq : [T, Hq,  d]
 *     k, v, dk, dv : [T, Hkv, d]
 *     lse          : float32 [Hq, T]
 * where T is the total token count.  Dense batches: cu_seqlens == NULL, the
 * B sequences of length N are stored back to back, T = B * N.  Packed
 * ("varlen") batches ("FlashAttention: The Algorithm That Beat the Memory
 * Wall", "Varlen Is the Quiet Superpower"): cu_seqlens is a device int32
 * array [B + 1] with cu_seqlens[0] = 0, non-decreasing, cu_seqlens[B] = T;
 * sequence b occupies tokens [cu_seqlens[b], cu_seqlens[b+1]); N is the
 * maximum sequence length (it sizes the grid; a longer sequence is an
 * error).  Query and key lengths are equal per sequence.
 *
 * Pointers: q..dv, lse, cu_seqlens, alibi_slopes and workspace are DEVICE
 * pointers owned by the caller; the library allocates no device memory and
 * keeps no per-call state: only a per-device status word and a host-side
 * cache of TMA descriptors per tensor shape and address
 * (fa_host_cache_stats).  bf16 tensors must start on a 16-byte boundary.
 * `stream` is a cudaStream_t (NULL = legacy default stream).  Every call is
 * asynchronous on `stream`; calls are not thread-safe on one stream.
 *
 * Errors.  Argument checks run on the host before any launch; a failing
 * check returns its status and launches nothing.  Launch failures return
 * FA_ERR_CUDA.  Faults found on the device (malformed cu_seqlens, a sequence
 * longer than N, a pipeline wait that ran out of its time limit) set a
 * per-device status word and make the affected blocks return early;
 * fa_check_device_error() reads and clears it.  No C++ exception crosses
 * this interface.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_NULL = 1,            /* a required pointer is NULL */
  FA_ERR_SHAPE = 2,           /* negative / inconsistent sizes */
  FA_ERR_UNSUPPORTED = 3,     /* valid but not implemented (d, dtype, scale) */
  FA_ERR_ALIGN = 4,           /* a bf16 tensor not 16-byte aligned */
  FA_ERR_WORKSPACE = 5,       /* workspace NULL or smaller than required */
  FA_ERR_CUDA = 6,            /* a CUDA runtime / launch error */
  FA_ERR_DEVICE_TIMEOUT = 7,  /* device: a pipeline wait exceeded its limit */
  FA_ERR_CU_SEQLENS = 8       /* device: cu_seqlens malformed or length > N */
} fa_status;

typedef enum { FA_BF16 = 0, FA_FP32 = 1 } fa_dtype;

/*
 * Forward: writes o ([T, Hq, d], o_dtype) and lse ([Hq, T], float32).
 *   B            number of sequences (>= 0)
 *   Hq, Hkv      query / key-value heads, Hq % Hkv == 0 (GQA/MQA groups are
 *                contiguous: kv head g serves query heads g*Hq/Hkv ...)
 *   N            sequence length (dense) or maximum length (packed)
 *   d            head dimension: bf16 d in {64, 128}; fp32 1 <= d <= 128
 *   scale        softmax scale (> 0, finite), usually 1/sqrt(d)
 *   causal       0 or 1
 *   window       sliding window w: key j visible to query i iff
 *                i - w <= j <= i.  < 0: no window.  w >= 0 requires
 *                causal == 1 (else FA_ERR_UNSUPPORTED); w = 0 lets each
 *                query see only its own key; w >= N - 1 equals plain causal.
 *   cu_seqlens   device int32 [B+1] or NULL (dense)
 *   total_tokens T; for dense batches 0 or B*N
 *   alibi_slopes device float32 [Hq] or NULL
 *   dtype        element type of q, k, v
 *   o_dtype      element type of o: FA_FP32 always allowed; FA_BF16 only
 *                with dtype == FA_BF16.  bf16 storage alone rounds O by up
 *                to 2^-9 |O| (1.6e-2 at |O| >= 4); FA_FP32 keeps the
 *                kernel's fp32 result.
 * FA_FP32 runs the fp32 SIMT kernel (forward only); FA_BF16 the tensor-core
 * kernel (bf16 operands, fp32 accumulation and softmax).
 */
fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int Hq, int Hkv, int N, int d, float scale, int causal, int window,
                 const int32_t* cu_seqlens, long long total_tokens,
                 const float* alibi_slopes, fa_dtype dtype, fa_dtype o_dtype,
                 void* stream);

/*
 * Bytes of device workspace fa_bwd needs: D (float32 [Hq, T]; the row-dot
 * D_i = dO_i . O_i of "FlashAttention: Faster Attention Without Dropping a
 * Single Interaction", Key design 3), the dQ accumulator (float32
 * [Hq, T, d]; the same design's dQ += dS K summed over key tiles) and 256
 * bytes for the dK/dV kernel's work-item counter, each part 256-byte
 * aligned.  T is total_tokens when
 * > 0, else B*N.  Returns 0 for invalid sizes.  The deterministic backward
 * does not use the accumulator; this size serves both.
 */
size_t fa_bwd_workspace_size(int B, int Hq, int N, int d, long long total_tokens);

/*
 * A larger workspace for grouped-query problems (Hq / Hkv even and >= 2):
 * fa_bwd_workspace_size plus room for two per-part sums of dK and dV
 * (float32 [2][2][T, Hkv, d]).  Given at least this many bytes, fa_bwd may
 * split the dK/dV work of each (key tile, kv head, sequence) of a dense
 * batch between two blocks, each taking half of the group's query heads;
 * the parts are added in a fixed order by the last stage, so results stay
 * reproducible.
 * This evens out the work per SM when the items are few and large (e.g.
 * B=2, Hq=32, Hkv=4, N=8192: 512 items of up to 1024 steps on 152 SMs).
 * Whether to split is decided per shape on the host from a simulation of
 * the kernel's largest-first schedule, against the cost of adding the
 * parts.  When work is split, FA_BWD_DKDV leaves the parts in the workspace
 * and FA_BWD_DQ_CONVERT writes dk and dv.  With a smaller workspace, or for
 * packed batches, the work is not split.  Returns fa_bwd_workspace_size's
 * value when the problem is never split (Hq / Hkv odd or 1), 0 for invalid
 * sizes.
 */
size_t fa_bwd_workspace_size_gqa(int B, int Hq, int Hkv, int N, int d, long long total_tokens);

/*
 * The number of parts (1 or 2) fa_bwd splits each dK/dV work item into
 * for these sizes, mask, packed layout (cu_seqlens NULL or not; it is not
 * read) and workspace size on the current device; 1 for arguments fa_bwd
 * would reject.  Diagnostic: callers need not call it.
 */
int fa_bwd_dkdv_split(int B, int Hq, int Hkv, int N, int d, int causal, int window,
                      const int32_t* cu_seqlens, size_t workspace_bytes);

/*
 * Backward: from q, k, v, the forward's o (element type o_dtype) and lse,
 * and dO, writes dq ([T, Hq, d]), dk and dv ([T, Hkv, d]), all bf16.  Same
 * size, mask and window arguments as fa_fwd.  `workspace` (device,
 * >= fa_bwd_workspace_size bytes, 256-byte aligned, contents irrelevant on
 * entry) is scratch owned by the caller; it must not be used by anything
 * else until the call completes on `stream`.
 *   deterministic  0: dQ is accumulated with float32 reductions in an order
 *                  that is not fixed, so dq may differ in the last bits from
 *                  run to run.  1: a separate kernel computes dQ per query
 *                  tile without atomics (two more MMAs per attended pair);
 *                  dq, dk and dv are then bit-identical from run to run
 *                  (the same page, Limitations, "Numerical exactness, low
 *                  precision, and reproducibility": a deterministic backward
 *                  is an option and is slower).  Other values:
 *                  FA_ERR_UNSUPPORTED.
 * Only FA_BF16.
 */
fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o,
                 const void* dO, const float* lse, void* dq, void* dk, void* dv,
                 int B, int Hq, int Hkv, int N, int d, float scale, int causal, int window,
                 const int32_t* cu_seqlens, long long total_tokens,
                 const float* alibi_slopes, fa_dtype dtype, fa_dtype o_dtype,
                 int deterministic, void* workspace, size_t workspace_bytes, void* stream);

/*
 * One stage of fa_bwd, with fa_bwd's arguments, so a caller can time or
 * schedule the stages separately.  fa_bwd == the three stages in order on
 * one stream:
 *   FA_BWD_PREPROCESS  D = rowsum(dO o O) and the dQ accumulator zeroed
 *                      (both in the workspace; deterministic: D only)
 *   FA_BWD_DKDV        dk, dv, and dQ accumulated in the workspace
 *                      (deterministic: dk and dv only; with split GQA
 *                      work, see fa_bwd_workspace_size_gqa, the dK / dV
 *                      parts in the workspace instead of dk and dv)
 *   FA_BWD_DQ_CONVERT  dq = scale * accumulator, as bf16 (deterministic:
 *                      dq computed by its own kernel from q, k, v, dO, lse
 *                      and D, one query tile per block); with split GQA
 *                      work also dk and dv from their parts
 * The same checks as fa_bwd run first; an unknown stage is
 * FA_ERR_UNSUPPORTED.
 * FA_BWD_DKDV hands out its work items from a counter in the workspace that
 * must read zero when it starts: FA_BWD_PREPROCESS zeroes it, and each
 * FA_BWD_DKDV that completes sets it back to zero.  So on a fresh workspace
 * (or after a call that ended in FA_ERR_DEVICE_TIMEOUT) run
 * FA_BWD_PREPROCESS before FA_BWD_DKDV; repeating FA_BWD_DKDV alone on a
 * workspace is otherwise allowed.  A negative counter found on the device
 * ends the stage's work and sets FA_ERR_WORKSPACE in the status word.
 */
typedef enum { FA_BWD_PREPROCESS = 0, FA_BWD_DKDV = 1, FA_BWD_DQ_CONVERT = 2 } fa_bwd_stage_id;

fa_status fa_bwd_stage(int stage, const void* q, const void* k, const void* v, const void* o,
                       const void* dO, const float* lse, void* dq, void* dk, void* dv,
                       int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                       int window, const int32_t* cu_seqlens, long long total_tokens,
                       const float* alibi_slopes, fa_dtype dtype, fa_dtype o_dtype,
                       int deterministic, void* workspace, size_t workspace_bytes,
                       void* stream);

/*
 * fa_bwd for callers that cannot allocate device memory.  (The pages have no
 * counterpart: this is an interface convenience of this library.)
 *
 * Some callers cannot hand fa_bwd a workspace: a plugin or custom-op hook
 * in another framework that gets no workspace and cannot reach that
 * framework's allocator, a runtime that fixes its device memory at start-up
 * and allows no allocation later, or code that must not call cudaMalloc
 * because it would synchronise the device or disturb a stream capture.
 * This entry point takes the same arguments as fa_bwd minus the workspace,
 * runs the same kernels, and keeps D and the dQ accumulator in a fixed
 * array of FA_BWD_STATIC_SCRATCH_BYTES inside the library's device memory.
 * It calls no cudaMalloc, cudaFree or other allocating routine.
 *
 * - Limit: fa_bwd's argument checks run first (same status codes); then a
 *   problem needing more than FA_BWD_STATIC_SCRATCH_BYTES of workspace
 *   (fa_bwd_workspace_size) is refused with FA_ERR_WORKSPACE before
 *   anything is launched.  64 MiB holds about 130,000 (token,
 *   query head) rows at d = 128 and 258,000 at d = 64, e.g. B = 8, H = 16,
 *   N = 1024, d = 64 (34 MB).
 * - Memory: the array, once reserved on a GPU, stays until the process
 *   exits.  With CUDA's lazy module loading (CUDA_MODULE_LOADING=LAZY, the
 *   default since CUDA 12.2) it is reserved only when the first call on that
 *   device looks it up, so that first call may itself take 64 MiB of device
 *   memory; with eager loading it is reserved when the library's module is
 *   loaded, whether or not this entry point is used.
 * - Set-up: the first call with a given device current looks up the
 *   array's device address (cudaGetSymbolAddress) and caches it.  Make that
 *   first call at start-up: before the caller's runtime fixes its device
 *   memory, and before any stream capture on that device.  A call with no
 *   tokens to process returns FA_OK without this set-up.
 * - Sharing: all calls on a device use the same array and it keeps the last
 *   call's contents.  Each call rewrites everything it reads (D, and a
 *   zeroed dQ accumulator), but calls that overlap on the GPU (different
 *   streams, or host threads, without ordering between them) race on it:
 *   order them on one stream or synchronise between them.
 * - Other errors: as fa_bwd.
 */
#define FA_BWD_STATIC_SCRATCH_BYTES (64ull << 20)

fa_status fa_bwd_static_scratch(const void* q, const void* k, const void* v, const void* o,
                                const void* dO, const float* lse, void* dq, void* dk, void* dv,
                                int B, int Hq, int Hkv, int N, int d, float scale, int causal,
                                int window, const int32_t* cu_seqlens, long long total_tokens,
                                const float* alibi_slopes, fa_dtype dtype, fa_dtype o_dtype,
                                int deterministic, void* stream);

/*
 * Decode over a KV cache: the q_len newest tokens of each sequence attend to
 * that sequence's cached keys and values ("FlashAttention: Faster Attention
 * Without Dropping a Single Interaction", Long context and inference: a tiny
 * query scanning a growing cache).  Sequence b holds L_b = cache_seqlens[b]
 * tokens, the q_len new ones included; query row i of b is the token at
 * position L_b - q_len + i and sees keys j <= L_b - q_len + i (causal), with
 * the ALiBi bias and sliding window of fa_fwd.  The result equals the last
 * q_len rows of fa_fwd's causal attention over the whole sequence.  The keys
 * are split into chunks processed in parallel and merged with the pages'
 * (m, l, O) merge rule (Key design 2), so this call launches two kernels.
 *   q             bf16 [B * q_len, Hq, d]: rows b*q_len .. b*q_len+q_len-1
 *                 are sequence b's new tokens
 *   k_cache,
 *   v_cache       bf16 [B, S_max, Hkv, d]; slots at or past L_b are not read
 *   cache_seqlens device int32 [B] with q_len <= L_b <= S_max, or NULL (every
 *                 cache holds S_max tokens); a value out of range is reported
 *                 on the device as FA_ERR_CU_SEQLENS
 *   o             [B * q_len, Hq, d], o_dtype FA_FP32 or FA_BF16
 *   lse           float32 [Hq, B * q_len] (natural log)
 *   d             64 or 128; (Hq / Hkv) * q_len <= 16, else FA_ERR_UNSUPPORTED
 *   window        as fa_fwd (< 0: none)
 *   workspace     device, >= fa_decode_workspace_size bytes, 256-byte
 *                 aligned; holds the per-chunk partial states
 * All pointers are device pointers owned by the caller; bf16 tensors and o
 * 16-byte aligned.  Errors as fa_fwd.
 */
size_t fa_decode_workspace_size(int B, int Hq, int Hkv, int S_max, int q_len, int d);

fa_status fa_decode(const void* q, const void* k_cache, const void* v_cache,
                    const int32_t* cache_seqlens, void* o, float* lse, int B, int Hq, int Hkv,
                    int S_max, int q_len, int d, float scale, int window,
                    const float* alibi_slopes, fa_dtype o_dtype, void* workspace,
                    size_t workspace_bytes, void* stream);

/*
 * FP8 forward ("FlashAttention: Faster Attention Without Dropping a Single
 * Interaction", FA3: per-block quantization and the same random orthogonal
 * Hadamard transform on Q and K, so that (QM)(KM)^T = QK^T before
 * quantization; the result is not exact).  Two calls:
 *   fa_fp8_quantize  Q' = (Q D) H and K' = (K D) H with D = diag(signs) and
 *                    H the unnormalised d x d Sylvester Hadamard matrix (the
 *                    butterfly in float32); then Q', K' and V are quantized
 *                    to e4m3 per block of 128 rows of one head of one
 *                    sequence, scale = amax / 448 (1 for an all-zero block),
 *                    code = e4m3(x * (448 / amax)) (the reciprocal once per
 *                    block, in float32), round to nearest even, saturated.
 *   fa_fwd_fp8       attention from those codes: S = scale * s_q * s_k
 *                    * (Q8 K8^T) / d, the online softmax of fa_fwd, P rounded
 *                    to e4m3 for the P V product (tensor cores, kind f8f6f4,
 *                    fp32 accumulation); o and lse as fa_fwd.
 * Only d = 128.  The codes and scales live in one caller-owned device buffer
 * laid out as below (byte offsets from its start, each 256-byte aligned);
 * nblk = ceil(N / 128); block i of sequence b has index b * nblk + i.
 */
typedef struct {
  size_t q8;           /* uint8 [T, Hq, 128]: codes of Q' */
  size_t k8;           /* uint8 [T, Hkv, 128]: codes of K' */
  size_t v8t;          /* uint8 [Hkv, 128, B * nblk * 128]: codes of V transposed; key r
                          of block (b, i) at column (b * nblk + i) * 128 + r; padding 0 */
  size_t q_scale;      /* float32 [Hq, B * nblk] (1 where a block is empty) */
  size_t k_scale;      /* float32 [Hkv, B * nblk] */
  size_t v_scale;      /* float32 [Hkv, B * nblk] */
  size_t v_scale_max;  /* float32 [Hkv]: the largest v_scale of each kv head */
  size_t total;        /* bytes of the whole buffer */
  int nblk;
} fa_fp8_layout;

/* Fills *out for a problem (sizes as fa_fwd; d must be 128). */
fa_status fa_fp8_layout_get(int B, int Hq, int Hkv, int N, int d, long long total_tokens,
                            fa_fp8_layout* out);

/* q, k, v: bf16 as fa_fwd; signs: device float32 [d], each +1 or -1 (the
 * random diagonal D, drawn by the caller); fp8_buf: device, >= total bytes,
 * 256-byte aligned.  Launches one kernel on `stream` (after a memset of the
 * per-head maximum V scale). */
fa_status fa_fp8_quantize(const void* q, const void* k, const void* v, const float* signs,
                          int B, int Hq, int Hkv, int N, int d, const int32_t* cu_seqlens,
                          long long total_tokens, void* fp8_buf, size_t fp8_bytes, void* stream);

/* Attention from the buffer fa_fp8_quantize filled (same sizes, cu_seqlens
 * and d); other arguments as fa_fwd. */
fa_status fa_fwd_fp8(const void* fp8_buf, size_t fp8_bytes, void* o, float* lse, int B, int Hq,
                     int Hkv, int N, int d, float scale, int causal, int window,
                     const int32_t* cu_seqlens, long long total_tokens,
                     const float* alibi_slopes, fa_dtype o_dtype, void* stream);

/*
 * Error reporting of this library (the pages have no counterpart; their
 * usage contract only names the inputs a call takes).
 * Synchronises `stream`, then reads and clears the current device's status
 * word.  Returns FA_OK, FA_ERR_DEVICE_TIMEOUT, FA_ERR_CU_SEQLENS, or
 * FA_ERR_CUDA if the synchronisation itself failed.
 */
fa_status fa_check_device_error(void* stream);

/*
 * Diagnostic: launches (asynchronously, on `stream`) one block whose bounded
 * pipeline wait can never be satisfied, with a limit of `limit_ns`
 * nanoseconds (1 ns .. 10 s).  The block records FA_ERR_DEVICE_TIMEOUT in
 * the device status word and returns; nothing hangs and nothing faults.  It
 * exercises the same wait the attention kernels use, so a caller can check
 * that a stalled pipeline surfaces through fa_check_device_error() on its
 * device, and that the context is usable afterwards.
 */
fa_status fa_selftest_wait_timeout(unsigned long long limit_ns, void* stream);

/*
 * Host-side set-up counters since the library was loaded (diagnostic; the
 * pages have no counterpart).  Each launch needs TMA descriptors for its
 * tensors and a shared-memory limit for its kernel.  The library keeps the
 * descriptors in a per-shape cache keyed on (base address, sizes, strides,
 * box, element type): a call whose tensors match an earlier call's reuses
 * its descriptors instead of encoding them again, so repeated calls on the
 * same buffers encode nothing.  The shared-memory limit is set once per
 * (device, kernel).  Any pointer may be NULL.
 *   tmaps_encoded   descriptors encoded
 *   tmaps_reused    descriptors served from the cache
 *   smem_attrs_set  kernel shared-memory limits set
 */
void fa_host_cache_stats(unsigned long long* tmaps_encoded, unsigned long long* tmaps_reused,
                         unsigned long long* smem_attrs_set);

/* Static description of a status code (never NULL); part of this library's
 * error reporting, with no counterpart on the pages. */
const char* fa_status_string(fa_status status);

/* Library version, major * 10000 + minor * 100 + patch. */
int fa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
