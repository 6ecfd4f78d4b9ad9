/*
 * fa_gb300.h -- C ABI of the GB300 (sm_103a) fused attention forward library.
 *
 * Exact scaled-dot-product attention, O = softmax(scale * Q K^T) V, computed
 * with the online-softmax recurrence so that the score matrix never reaches
 * device memory.
 *
 * Sources (page title, section):
 *   "Kernel visualization: Flash Attention 1": "Derivation" and "The tiled
 *       version" (the per-row recurrence for the running max, sum and output).
 *   "Softmax and FlashAttention": "Concept" (the problem: S = QK^T, P =
 *       softmax(S), O = PV; FlashAttention-2 loop order) and "Maths"
 *       (exactness of the online softmax).
 *   "Attention kernel chains: tiling, the online softmax, merges and masks":
 *       "The log-sum-exp merge", "How many splits for decode", "The causal
 *       mask for a decode step", "What the backward pass saves" (one fp32 LSE
 *       per query row), "GQA loads KV once per group", "The block-table cost
 *       of paged attention".
 *
 * Conventions shared by every call
 *   - Every tensor argument is a DEVICE pointer owned by the caller, dense
 *     row-major, 16-byte aligned. The library never frees or keeps them.
 *   - Layouts: q, o are [B][Hq][T][d]; k, v are [B][Hkv][S][d]; lse is
 *     [B][Hq][T] fp32 (natural log of the sum of exp of the scaled scores).
 *   - GQA: Hq % Hkv == 0; query head h reads KV head h / (Hq / Hkv).
 *   - causal != 0 applies the bottom-right-aligned mask: query row i (of T)
 *     sees key j iff j <= i + (S - T). A row that sees no key (T > S) gets
 *     O = 0 and lse = -inf.
 *   - scale must be finite and > 0 (the pages use 1/sqrt(d)).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *     default stream). Argument errors are returned synchronously, before
 *     anything is launched; FA_ERR_CUDA reports a failed launch.
 *   - The prefill, decode and backward kernels launch as programmatic
 *     dependents of the launch before them on `stream` and may start while
 *     it finishes; each waits (griddepcontrol.wait) before its first access
 *     to global memory, so stream order holds for every input and output.
 *     The unsplit prefill, the decode kernel, the LSE merge and the backward's
 *     main grid also let the next launch on the stream start early; a kernel of
 *     the caller's launched that way after them must likewise wait before
 *     reading their outputs.
 *   - Kernels never trap. Every wait inside a kernel is bounded; a wait that
 *     runs out, or a bounds check that fails (paged block-table entries),
 *     records a code in a device-side error word and the kernel returns.
 *     fa_get_last_device_error() reads and clears that word.
 *   - The library allocates no device memory. Scratch space (split-KV
 *     partials, the backward's per-row values, the running state of the
 *     FlashAttention-1 order) is passed in by the caller as `workspace`.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = 1, /* null pointer, bad size, Hq % Hkv != 0, misaligned pointer, ... */
  FA_ERR_UNSUPPORTED = 2, /* valid but not implemented (e.g. head dim not in {64, 128}) */
  FA_ERR_CUDA = 3,        /* a CUDA runtime/driver call failed; see fa_last_cuda_error_string() */
  FA_ERR_TIMEOUT = 4,     /* device side: a bounded wait ran out */
  FA_ERR_BOUNDS = 5       /* device side: a block-table entry outside [0, num_pages) */
} fa_status;

/* Library version, major*10000 + minor*100 + patch. */
FA_API int fa_version(void);

/* Human-readable name of a status code (static storage). */
FA_API const char* fa_status_string(int status);

/* Text of the last CUDA error seen by this library in this thread (static storage). */
FA_API const char* fa_last_cuda_error_string(void);

/*
 * fa_fwd -- prefill / general forward, BF16 in, BF16 O, FP32 LSE.
 * ("Softmax and FlashAttention", "Concept": FlashAttention-2 order; "Attention
 *  kernel chains", "What the backward pass saves": one FP32 LSE per row;
 *  "GQA loads KV once per group": a group's query heads share each K/V tile.)
 *   q   [B][Hq][Tq][d]  bf16      k, v [B][Hkv][Skv][d] bf16
 *   o   [B][Hq][Tq][d]  bf16 out  lse  [B][Hq][Tq] fp32 out, may be NULL
 *   d in {64, 128}; Hq / Hkv in {1, 2, 4, 8, 16}; Tq, Skv >= 1; B*Hq*Tq < 2^31.
 * Runs the tcgen05 tensor-core kernel (TMA ring, TMEM accumulators).
 */
FA_API fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
                 int B, int Hq, int Hkv, int Tq, int Skv, int d, float scale, int causal,
                 void* stream);

/*
 * fa_fwd_f32 -- the same operation in FP32 throughout (inputs, accumulation,
 * output) on the CUDA cores; for checking at 1e-5 against the fp64 oracle.
 *   q, o [B][Hq][Tq][d] fp32; k, v [B][Hkv][Skv][d] fp32; lse as fa_fwd.
 *   1 <= d <= 128.
 */
FA_API fa_status fa_fwd_f32(const float* q, const float* k, const float* v, float* o, float* lse,
                     int B, int Hq, int Hkv, int Tq, int Skv, int d, float scale, int causal,
                     void* stream);

/*
 * fa_bwd -- gradients of the forward for an upstream gradient dO.
 * ("Attention kernel chains", "What the backward pass saves": the forward keeps
 *  Q, K, V, O and the fp32 log-sum-exp per query row; the backward rebuilds
 *  each probability tile as P = exp(S - LSE) and needs D = rowsum(dO * O),
 *  formed once before the main loops.) With S = scale * Q K^T:
 *  dV = P^T dO, dP = dO V^T, dS = P * (dP - D), dQ = scale * dS K,
 *  dK = scale * dS^T Q; a KV head's dK and dV sum over its group's query heads.
 *   q, o, d_o [B][Hq][Tq][d] bf16; k, v [B][Hkv][Skv][d] bf16 (as fa_fwd);
 *   lse [B][Hq][Tq] fp32, the forward's (natural log, -inf for keyless rows);
 *   dq [B][Hq][Tq][d], dk, dv [B][Hkv][Skv][d] bf16 out (overwritten).
 *   causal: the same bottom-right mask as fa_fwd. d in {64, 128}; Hq / Hkv in
 *   {1, 2, 4, 8, 16}.
 *   workspace: device scratch of at least fa_bwd_workspace_bytes(B, Hq, Tq)
 *   bytes, 16-byte aligned, for two fp32 values per query row: -D and the LSE in
 *   base 2, negated. Two launches on `stream`: those row values, then one grid
 *   whose first CTAs compute dK/dV (one per 128-key tile) and whose others
 *   compute dQ (one per 128-row query tile).
 */
FA_API fa_status fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                        const void* d_o, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int Tq,
                        int Skv, int d, float scale, int causal, void* workspace, size_t ws_bytes,
                        void* stream);

/* fa_bwd_workspace_bytes -- 8 * B * Hq * Tq', Tq' = Tq rounded up to a multiple of 4
 * (two fp32 values per query row, rows padded to 16 bytes); 0 for invalid sizes. */
FA_API size_t fa_bwd_workspace_bytes(int B, int Hq, int Tq);

/*
 * fa_fwd_kv_outer -- the operation of fa_fwd computed in the FlashAttention-1
 * loop order, kept as a measured contrast to fa_fwd's order.
 * ("Kernel visualization: Flash Attention 1", "The tiled version", "Kernel
 *  implementation", "Counting trips across HBM": the key/value tiles form the
 *  outer loop and the query tiles the inner one. Each (key tile, query tile) step
 *  reads the query tile's running max m, sum l and normalised output O' from HBM,
 *  folds the key tile in, and writes them back. Only the last key tile's step
 *  leaves the final O. "Softmax and FlashAttention", "Concept": the
 *  FlashAttention-2 order of fa_fwd reads each query tile and writes each output
 *  tile once.)
 *   q, k, v, o, lse, scale, causal: as fa_fwd. The same bottom-right mask applies.
 *   row_bands: CTAs per (batch, query head), each running the loop nest over a
 *   contiguous band of 128-row query tiles and loading every key tile once per
 *   band. 1 gives the pages' grid, one CTA per (batch, head). Values above the
 *   number of query tiles are clamped to it.
 *   workspace: device scratch of at least fa_fwd_kv_outer_workspace_bytes(B, Hq,
 *   Tq, d) bytes, 16-byte aligned. It holds the running O', m and l in fp32. The
 *   first key tile of a query tile starts from m = -inf, l = 0, O' = 0 without
 *   reading it, so it needs no initialisation.
 *   d in {64, 128}; Hq / Hkv in {1, 2, 4, 8, 16}. Each query head's CTA loads its
 *   KV head's tiles, without GQA stacking.
 *   Errors: FA_ERR_INVALID_ARG for null or misaligned pointers, bad sizes, a
 *   non-positive scale, row_bands < 1 or a workspace that is too small.
 *   FA_ERR_UNSUPPORTED for other d or group sizes, or too many CTAs.
 */
FA_API fa_status fa_fwd_kv_outer(const void* q, const void* k, const void* v, void* o, float* lse,
                                 int B, int Hq, int Hkv, int Tq, int Skv, int d, float scale, int causal,
                                 int row_bands, void* workspace, size_t ws_bytes, void* stream);

/* fa_fwd_kv_outer_workspace_bytes -- O' (4 * B*Hq*Tq*d bytes, rounded up to 256)
 * plus m and l (4 * B*Hq*Tq bytes each); 0 for invalid sizes. */
FA_API size_t fa_fwd_kv_outer_workspace_bytes(int B, int Hq, int Tq, int d);

/*
 * fa_num_splits_heuristic -- how many key ranges a decode step should use.
 * ("Attention kernel chains", "How many splits for decode": split so that
 *  batch x KV heads x splits fills at most one wave of SMs; no split once
 *  batch x KV heads already fills the GPU.)
 * Returns max(1, min(num_sms / (B*Hkv), ceil(S / 256))); 1 when B*Hkv >= num_sms.
 * Pure host arithmetic. Returns 1 for non-positive arguments.
 */
FA_API int fa_num_splits_heuristic(int B, int Hkv, int S, int num_sms);

/*
 * fa_num_splits_prefill -- key ranges for a call with more than 16 query rows
 * per KV head (a prefill-shaped problem) whose query tiles alone do not fill
 * the GPU, e.g. one head of a long sequence. The same one-wave rule as the
 * decode heuristic ("How many splits for decode"), counted in the prefill
 * kernel's work items: units = ceil(ceil(T / (128 / g)) / 2) * B * Hkv pairs
 * of 128-row query tiles (g = Hq / Hkv). Returns 1 when units >= num_sms,
 * else max(1, min(num_sms / units, ceil(S / 512), 64)).
 * Pure host arithmetic. Returns 1 for invalid arguments.
 */
FA_API int fa_num_splits_prefill(int B, int Hq, int Hkv, int T, int S, int num_sms);

/*
 * fa_decode_num_splits -- the key ranges fa_decode_splitkv (paged = 0) or
 * fa_decode_paged (paged = 1, S = max_pages * page_size) take for
 * num_splits == 0 when the workspace holds them: with (Hq / Hkv) * T <= 16,
 * fa_num_splits_heuristic(B, Hkv, S, num_sms); with more rows,
 * fa_num_splits_prefill(B, Hq, Hkv, T, S, num_sms) for contiguous K/V and 1
 * for paged K/V. The one place this choice is made: a binding that sizes the
 * workspace calls it and passes num_splits == 0 through. Pure host
 * arithmetic. Returns 1 for invalid arguments.
 */
FA_API int fa_decode_num_splits(int B, int Hq, int Hkv, int T, int S, int paged, int num_sms);

/*
 * fa_decode_workspace_bytes -- bytes of `workspace` a split decode needs:
 * FP32 partial outputs [num_splits][B*Hq*T][d] followed (256-byte aligned) by
 * FP32 partial lse [num_splits][B*Hq*T]. 0 when num_splits <= 1.
 */
FA_API size_t fa_decode_workspace_bytes(int B, int Hq, int T, int d, int num_splits);

/*
 * fa_decode_splitkv -- attention of T new queries over S contiguous cached
 * keys, split into num_splits contiguous key ranges of ceil(S / num_splits)
 * keys, each processed by its own CTAs, then merged by fa_lse_merge on the
 * same stream. ("Attention kernel chains", "The log-sum-exp merge" and "How
 * many splits for decode".)
 *   q [B][Hq][T][d] bf16; k, v [B][Hkv][S][d] bf16; o [B][Hq][T][d] bf16 out;
 *   lse [B][Hq][T] fp32 out (may be NULL).
 *   d in {64, 128}.
 *   With more than 16 query rows per KV head ((Hq / Hkv) * T > 16: a chunked
 *   prefill, a multi-token step, or a whole prefill) the call runs the
 *   tensor-core prefill kernel, which tiles the queries itself; Hq / Hkv must
 *   be one of 1, 2, 4, 8, 16 (else FA_ERR_UNSUPPORTED). num_splits > 1 cuts
 *   the keys into that many ranges of whole 128-key tiles for shapes whose
 *   query tiles do not fill the GPU, with the workspace and merge as above;
 *   num_splits == 0 takes fa_decode_num_splits (fa_num_splits_prefill here),
 *   lowered to what `workspace` holds (no workspace: no split). The result is
 *   the same attention.
 *   num_splits: 0 = fa_decode_num_splits(B, Hq, Hkv, T, S, 0, SM count), here
 *   fa_num_splits_heuristic(B, Hkv, S, SM count); else 1..1024.
 *   workspace: device scratch of at least fa_decode_workspace_bytes(...)
 *   bytes, 256-byte aligned (may be NULL when the split count is 1).
 *   Returns FA_ERR_INVALID_ARG if ws_bytes is too small.
 */
FA_API fa_status fa_decode_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                            int B, int Hq, int Hkv, int T, int S, int d, float scale, int causal,
                            int num_splits, void* workspace, size_t ws_bytes, void* stream);

/*
 * fa_decode_splitkv_static -- fa_decode_splitkv without a workspace argument.
 * The pages have no counterpart: this serves callers that cannot allocate
 * device memory for the split partials (work recorded into a CUDA graph
 * while it is being captured, engines whose device memory is carved up once
 * by their host, latency-critical paths that must not risk an allocation).
 * The partials go to a fixed 4 MiB array inside the library's device image
 * (every device that loads the library holds one until the process exits);
 * the call allocates nothing.
 *   Arguments and results as fa_decode_splitkv, except that (Hq / Hkv) * T
 *   must be <= 16 (FA_ERR_UNSUPPORTED otherwise); B * Hq * T and
 *   B * Hkv * S must be below 2^31 and B * Hkv at most 65535 (the same
 *   limits, FA_ERR_UNSUPPORTED).
 *   Returns FA_ERR_UNSUPPORTED when the partials would need more than 4 MiB,
 *   i.e. fa_decode_workspace_bytes(B, Hq, T, d, splits) > 4194304.
 *   The first call on a device looks up the array's device address (with
 *   that device current); make that first call before any stream capture.
 *   The address is kept for the life of the process: resetting the device
 *   (cudaDeviceReset) after that first call is not supported.
 *   All calls on a device share the array and it keeps the last call's
 *   contents (every call rewrites what it reads). Calls that overlap on the
 *   GPU -- other streams, other host threads -- race on it: serialise them.
 *   If a kernel of the call records FA_ERR_TIMEOUT or FA_ERR_BOUNDS (see
 *   fa_get_last_device_error), o and lse are undefined: the merge may have
 *   read partials an earlier call left in the array.
 */
FA_API fa_status fa_decode_splitkv_static(const void* q, const void* k, const void* v, void* o, float* lse,
                                          int B, int Hq, int Hkv, int T, int S, int d, float scale, int causal,
                                          int num_splits, void* stream);

/*
 * fa_lse_merge -- merge normalised partial results of `num_splits` key ranges.
 * ("Attention kernel chains", "The log-sum-exp merge": lse = ln sum_s e^{lse_s},
 *  O = sum_s e^{lse_s - lse} O_s.)
 *   o_part   [num_splits][rows][d] fp32   lse_part [num_splits][rows] fp32
 *   o        [rows][d] bf16 out           lse      [rows] fp32 out (may be NULL)
 *   A split with lse_s = -inf has weight 0; a row whose splits are all -inf
 *   gets O = 0 and lse = -inf. 1 <= d <= 256, num_splits >= 1.
 */
FA_API fa_status fa_lse_merge(const float* o_part, const float* lse_part, void* o, float* lse,
                       int num_splits, int rows, int d, void* stream);

/*
 * fa_decode_paged -- decode over a paged K/V cache.
 * ("Attention kernel chains", "The block-table cost of paged attention":
 *  token t of sequence b lives in slot t % page_size of pool page
 *  block_table[b][t / page_size]; K and V share the table.)
 *   q           [B][Hq][T][d] bf16
 *   k_pages,
 *   v_pages     [num_pages][page_size][Hkv][d] bf16
 *   block_table [B][max_pages] int32 (device)
 *   seqlens     [B] int32 (device): keys of each sequence, each in [0, max_pages*page_size]
 *   o, lse      as fa_decode_splitkv
 *   page_size == 16; d in {64, 128}.
 *   Each sequence's keys are split into num_splits ranges (0 = heuristic on
 *   max_pages*page_size); workspace as fa_decode_splitkv.
 *   With (Hq / Hkv) * T > 16 (chunked prefill over the cache: T new tokens at
 *   positions seqlens[b] - T .. seqlens[b] - 1 under the bottom-right mask)
 *   the tensor-core prefill kernel gathers each 128-key tile from eight pages;
 *   num_splits must then be 0 or 1 (no key split, no workspace) and Hq / Hkv
 *   one of 1, 2, 4, 8, 16. Pool rows past a sequence's end are never used,
 *   whatever they hold.
 *   A table entry outside [0, num_pages) is not dereferenced: the kernel
 *   records FA_ERR_BOUNDS (read it with fa_get_last_device_error) and that
 *   sequence's output is undefined.
 */
FA_API fa_status fa_decode_paged(const void* q, const void* k_pages, const void* v_pages,
                          const int* block_table, const int* seqlens, void* o, float* lse,
                          int B, int Hq, int Hkv, int T, int max_pages, int page_size,
                          int num_pages, int d, float scale, int causal, int num_splits,
                          void* workspace, size_t ws_bytes, void* stream);

/*
 * fa_get_last_device_error -- synchronise `stream`, read and clear the
 * device-side error word. Returns FA_OK, FA_ERR_TIMEOUT or FA_ERR_BOUNDS
 * (or FA_ERR_CUDA if the read itself fails). *detail (may be NULL) receives
 * the raw word: code | site << 8.
 */
FA_API fa_status fa_get_last_device_error(void* stream, int* detail);

/*
 * fa_set_wait_timeout_ns -- bound, in nanoseconds of %globaltimer, for every
 * wait of one role of a CTA on another inside the kernels launched after this
 * call (default 4e9 = 4 s). Values below 1e6 (1 ms) are raised to 1e6. The
 * waits a CTA makes before it exits or frees its tensor memory (its own bulk
 * copies landing, its own MMAs draining) are bounded by max(this, 1e9): a
 * short setting never lets a CTA leave with copies or MMAs still running.
 */
FA_API void fa_set_wait_timeout_ns(unsigned long long ns);

/*
 * fa_get_wait_timeouts -- the bounds in force, in nanoseconds: *wait_ns the
 * bound of fa_set_wait_timeout_ns as clamped, *unwind_ns the bound of the
 * waits before a CTA exits (max(*wait_ns, 1e9)). Either pointer may be NULL.
 */
FA_API void fa_get_wait_timeouts(unsigned long long* wait_ns, unsigned long long* unwind_ns);

/*
 * fa_selftest_wait_timeout -- failure-detection self test (no counterpart on
 * the pages). Launches one CTA that waits, through the same bounded wait the
 * attention kernels use, on an mbarrier that nothing ever arrives on, with a
 * limit of `timeout_ns`. The wait must run out: the kernel records
 * FA_ERR_TIMEOUT in the device error word and returns, leaving the context
 * usable. Read the outcome with fa_get_last_device_error().
 */
FA_API fa_status fa_selftest_wait_timeout(unsigned long long timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
