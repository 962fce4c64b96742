/*
 * swa.h - sliding-window split-KV verify attention for GB300 (sm_103a).
 *
 * One call computes, for a block of q_len query rows per sequence (one
 * committed token plus the drafted tokens of a speculative-decoding step),
 * grouped-query attention over a bf16 KV cache in which the query at
 * absolute position p sees only the keys at positions (p - W, p]:
 *
 *   "The Fast Gemma Challenge: our verified-SOTA recipe, in full",
 *   manifest keys SLIDING_WINDOW=188 / FA_SLIDING=1 (attend to the most
 *   recent W tokens, section "What each piece does, and why"),
 *   SPECULATIVE_CONFIG num_speculative_tokens=7 (q_len = 1 + 7 = 8),
 *   SPLITKV_VERIFY=1 and SPLITKV_VERIFY_MAX_Q=64 (split-KV verify kernel,
 *   at most 64 query rows per verify call); MAX_NUM_BATCHED_TOKENS=512 (the
 *   same windowed attention over prefill chunks of up to 512 tokens).
 *
 * Definition (per sequence b, query head h, draft row i, p = q_pos[b] + i,
 * KV head g = floor(h / (Hq / Hkv))):
 *   K(p) = { j : max(0, p - W + 1) <= j <= p, j < seq_len[b], j < max_len }
 *   s_j  = scale * <q[b,i,h,:], k_cache[b,g,j,:]>
 *   lse  = ln sum_{j in K(p)} exp(s_j)
 *   out  = sum_{j in K(p)} exp(s_j - lse) * v_cache[b,g,j,:]
 * A row with an empty K(p) gets out = 0 and lse = -inf.
 *
 * All entry points are plain C: device pointers and host structs, no
 * framework types.  Nothing here synchronises the device unless stated.
 */
#ifndef SWA_H
#define SWA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream; NULL is the legacy default stream. */
typedef struct CUstream_st *swa_stream_t;

typedef enum {
    SWA_OK = 0,
    SWA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad shape or size      */
    SWA_ERR_UNSUPPORTED = 2,  /* well-formed but outside what the kernels cover  */
    SWA_ERR_WORKSPACE = 3,    /* split partials need more workspace than is set  */
                              /* and it cannot be grown (stream capture active)  */
    SWA_ERR_CUDA = 4          /* a CUDA runtime call failed; see swa_last_error  */
} swa_status;

/* Shapes of one call.  The pages give no shapes; these name the tensors'
 * dimensions.  All tensors are contiguous row-major. */
typedef struct {
    int32_t batch;         /* B, number of sequences, 1..65535                  */
    int32_t q_len;         /* query rows per sequence, 1..512: verify blocks of up to
                              64 rows (SPLITKV_VERIFY_MAX_Q) and sliding-window
                              prefill chunks of up to 512 (MAX_NUM_BATCHED_TOKENS) */
    int32_t num_q_heads;   /* Hq                                                */
    int32_t num_kv_heads;  /* Hkv, Hq % Hkv == 0; G = Hq / Hkv query heads per KV head */
    int32_t head_dim;      /* D, one of 64, 128, 256                            */
    int32_t max_len;       /* L, cache rows per (sequence, KV head), >= 1       */
    int32_t num_splits;    /* 0: the library picks the split count; n >= 1 forces n
                              chunks per (sequence, KV head) (clamped to 1..64)   */
} swa_dims;

/* Windowed verify attention ("split-KV verify kernel", SPLITKV_VERIFY).
 *
 *   q        bf16 [B, q_len, Hq, D]   device, 16-byte aligned
 *   k_cache  bf16 [B, Hkv, L, D]      device, 16-byte aligned
 *   v_cache  bf16 [B, Hkv, L, D]      device, 16-byte aligned
 *   seq_lens int32 [B]                device: valid cache rows per sequence
 *   q_pos    int32 [B]                device: absolute position of query row 0;
 *                                      row i sits at q_pos + i
 *   window   W >= 1                   keys (p - W, p] are visible to row p
 *   scale    finite                   multiplies q.k (1/sqrt(D) for plain attention)
 *   out      bf16 [B, q_len, Hq, D]   device, 16-byte aligned, written
 *   lse      fp32 [B, q_len, Hq]      device or NULL; natural-log log-sum-exp
 *   dims     host struct, read during the call only
 *   stream   work is enqueued on this stream; the call returns without waiting
 *
 * Device-side preconditions (not checked on the host because the values
 * live on the device): 0 <= q_pos, q_pos + q_len <= seq_len <= L, and the
 * caller has written the q_len new K/V rows before the call.  If they do not
 * hold the kernels still never read a cache row outside [0, L) of the
 * sequence's own slab, and rows without a visible key get out = 0,
 * lse = -inf.
 *
 * Ownership: every pointer stays owned by the caller; nothing is retained
 * after the call except through the workspace described below.
 *
 * Workspace: when the chosen split count needs split partials in global
 * memory, they go to the workspace set with swa_set_workspace() for the
 * current device, or else to a library-owned buffer grown on demand with
 * cudaMalloc (never while `stream` is capturing: then SWA_ERR_WORKSPACE).
 * All calls on one device share that buffer, so calls that may run at the
 * same time on different streams race on it; order them on one stream or
 * give each its own device.
 *
 * Errors: SWA_ERR_INVALID_ARG / SWA_ERR_UNSUPPORTED are returned before any
 * CUDA call and leave the outputs untouched.  SWA_ERR_INVALID_ARG: a NULL or
 * misaligned pointer, a non-finite scale, or dims outside the ranges above
 * (also num_kv_heads > 65535).  SWA_ERR_UNSUPPORTED: head_dim not in {64,
 * 128, 256}; more than 4096 packed rows q_len * (Hq / Hkv) per KV head; or
 * num_kv_heads * ceil(q_len * (Hq / Hkv) / 32) > 65535.  SWA_ERR_CUDA
 * reports a failed launch or allocation.  swa_last_error() gives the
 * message. */
swa_status swa_verify_attn(const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *seq_lens, const int32_t *q_pos, int32_t window,
                           float scale, void *out, float *lse, const swa_dims *dims,
                           swa_stream_t stream);

/* Paged KV cache (vLLM-style block tables): the cache is a pool of pages,
 * each holding page_size consecutive key positions of one sequence for
 * every KV head, and a sequence's block table lists its pages in position
 * order.  The pages mention a reduced KV cache and the window as its reason
 * ("What each piece does, and why"); a pool lets a server hold only the
 * pages a window still needs.  A window-sized ring per sequence (position
 * j kept in slot j mod R) is the same map with a cyclic table: R a multiple
 * of page_size and at least window + q_len - 1, the ring's R / page_size
 * pages listed over and over (block k -> ring page k mod (R / page_size)).
 * Keys outside a row's window are never weighted, so ring slots that newer
 * positions overwrote do not matter. */
typedef struct {
    const int32_t *block_table;  /* device int32 [batch, max_blocks], 4-byte aligned: block k of
                                    sequence b (positions k*page_size ..) is page block_table[b][k] */
    int32_t max_blocks;          /* row length of block_table; dims->max_len must equal
                                    max_blocks * page_size (a sequence's logical capacity) */
    int32_t page_size;           /* key positions per page, a positive multiple of 8 */
    int32_t num_pages;           /* pages in the pool */
} swa_paged;

/* swa_verify_attn on a paged cache:
 *   k_pages, v_pages  bf16 [num_pages, Hkv, page_size, D], device, 16-byte aligned
 * and everything else as for swa_verify_attn.  Results equal the contiguous
 * call on the cache the block tables describe, up to fp32 summation order.
 * Device preconditions (not checked): for every sequence, block_table[b][k]
 * is a valid page (0 <= page < num_pages) for each block holding positions
 * below seq_lens[b]; entries past that are never read.  Returns
 * SWA_ERR_INVALID_ARG for a NULL or misaligned table, a page size that is not
 * a positive multiple of 8, or dims->max_len != max_blocks * page_size;
 * SWA_ERR_UNSUPPORTED if the pool holds 2^31 or more rows. */
swa_status swa_verify_attn_paged(const void *q, const void *k_pages, const void *v_pages,
                                 const swa_paged *paged, const int32_t *seq_lens,
                                 const int32_t *q_pos, int32_t window, float scale, void *out,
                                 float *lse, const swa_dims *dims, swa_stream_t stream);

/* Fused KV append + verify: the step before the verify (writing the draft
 * block's freshly projected K/V rows into the cache) done inside the
 * attention kernels, so one launch both stores the rows and attends over
 * them.  The pages name no such kernel; it serves the launch trimming they
 * credit to the single-graph step (ONEGRAPH, "What each piece does, and
 * why"): one launch fewer per verify step.
 *   k_new, v_new  bf16 [B, q_len, Hkv, D], device, 16-byte aligned: row i of
 *                 sequence b is key position q_pos[b] + i
 *   k_cache, v_cache  writable caches: contiguous [B, Hkv, max_len, D]
 *                 (paged == NULL) or page pools [num_pages, Hkv, page_size, D]
 *                 described by *paged (as for swa_verify_attn_paged)
 * Afterwards every cache row at position q_pos[b] + i < min(seq_lens[b],
 * max_len) holds row i of k_new / v_new (bit copies); no other cache byte
 * changes.  out / lse are those of swa_verify_attn on the updated cache.
 * The same device preconditions hold (q_pos + q_len <= seq_len <= max_len;
 * with a paged cache the blocks holding the new positions are valid pages);
 * rows outside [0, min(seq_len, max_len)) are never written.  k_new / v_new
 * must not overlap the caches, q or out.  Errors as for swa_verify_attn,
 * plus SWA_ERR_INVALID_ARG for a NULL or misaligned k_new / v_new. */
swa_status swa_append_verify_attn(const void *q, const void *k_new, const void *v_new,
                                  void *k_cache, void *v_cache, const swa_paged *paged,
                                  const int32_t *seq_lens, const int32_t *q_pos, int32_t window,
                                  float scale, void *out, float *lse, const swa_dims *dims,
                                  swa_stream_t stream);

/* Upper bound, in bytes, of the split-partial workspace any call with these
 * dims and window may need on any device (pure host arithmetic; 0 if the
 * arguments are invalid).  Layout: fp32 acc [B, Hkv, splits, R, D] followed
 * by fp32 (m, l) pairs [B, Hkv, splits, R, 2], R = q_len * Hq / Hkv. */
size_t swa_workspace_bytes(const swa_dims *dims, int32_t window);

/* Use caller-owned device memory [dev_ptr, dev_ptr + bytes) as the
 * workspace of the current device (16-byte aligned).  The library frees any
 * buffer it grew itself.  dev_ptr = NULL, bytes = 0 returns to the
 * library-owned buffer.  The memory must stay valid until replaced. */
swa_status swa_set_workspace(void *dev_ptr, size_t bytes);

/* Release the library-owned workspace of the current device (synchronises
 * the device through cudaFree). */
swa_status swa_release_workspace(void);

/* What the library would launch for these dims on a GPU with `num_sms`
 * SMs (pure host arithmetic, no CUDA call). */
typedef struct {
    int32_t kernel;        /* 1 = CUDA-core (SIMT) chunk kernel, 2 = key-major tensor-core
                              (tcgen05) kernel, 3 = rows-major tensor-core kernel, 4 = the
                              rows-major kernel on CTA pairs (clusters of two CTAs, 2 x 128
                              packed rows per item; swa_verify_attn only: a paged or fused-
                              append call with these dims takes kernel 3 instead) */
    int32_t num_splits;    /* chunks per (sequence, KV head)                    */
    int32_t chunk_keys;    /* keys per chunk                                    */
    int32_t row_tiles;     /* work items along the packed rows R = q_len * G    */
    int32_t rows_per_tile; /* packed rows per work item (kernel 4: two CTAs')   */
    int32_t grid_ctas;     /* CTAs of the attention kernel                      */
    int32_t merge;         /* 0 none, 1 separate log-sum-exp merge kernel       */
    int64_t workspace_bytes; /* global scratch this plan uses                   */
} swa_plan_info;

swa_status swa_plan(const swa_dims *dims, int32_t window, int32_t num_sms,
                    swa_plan_info *plan);

/* Thread-local message of the last failing call on this thread ("" if none). */
const char *swa_last_error(void);

/* Device-side fault word of the current device: every bounded wait inside
 * the kernels that gives up sets a bit here instead of hanging.  Reading it
 * synchronises the device; the word is cleared after the read.
 * Bit 0: a K/V tile copy did not complete within the wait limit. */
swa_status swa_read_device_errors(uint32_t *flags);

/* Out-of-range index attempts counted since the last read by a library built
 * with SWA_DEBUG_CHECKS (libswa_debug.so): indices that come from device-side
 * inputs, which the header states as preconditions and the kernels otherwise
 * do not check: a block-table page outside [0, num_pages) (the kernel reads
 * page 0 instead, and a fused append drops the store) and a sequence length
 * outside [0, max_len] (clamped, as in every build).  Nothing traps.  Reading
 * synchronises the device and clears the count.  A library built without the
 * checks sets *count to 0 and returns SWA_ERR_UNSUPPORTED; NULL count:
 * SWA_ERR_INVALID_ARG. */
swa_status swa_read_debug_checks(uint32_t *count);

/* Library version, e.g. "swa 0.1.0 sm_103a" ("... debug-checks" for the
 * build with SWA_DEBUG_CHECKS). */
const char *swa_version(void);

/* Test and sweep controls.  Not for serving: every call uses the defaults
 * unless a test or a benchmark sweep changes them; a change applies to all
 * later calls in the process (every thread and device).  The library reads
 * no environment variable. */
typedef struct {
    int32_t force_kernel;      /* 0 (default): the plan's kernel; 1 CUDA-core, 2 key-major
                                  tensor-core, 3 rows-major tensor-core, 4 rows-major on CTA
                                  pairs (a shape the forced kernel does not take runs the
                                  plan's kernel; 4 falls back to 3 off head_dim 256, on a
                                  paged cache and under a fused append) */
    int32_t pdl;               /* 1 (default): launches with programmatic dependent launch;
                                  0: plain stream-ordered launches */
    int64_t wait_limit_cycles; /* 0 (default): every bounded wait inside the kernels gives up
                                  after 2e9 SM cycles (about 1 s); n > 0: after n cycles */
    int32_t withhold_fill;     /* -1 (default); n >= 0: the first CTA's copy producer posts
                                  its n-th K/V fill but never issues the copies, so every wait
                                  on that fill runs out and the call reports bit 0 through
                                  swa_read_device_errors (the test of the bounded waits) */
    int32_t rows_per_item;     /* 0 (default): the plan's packed rows per tensor-core work
                                  item; n > 0: n capped at the kernel's maximum (64
                                  key-major, 128 rows-major) and at q_len * Hq / Hkv,
                                  then rounded down to a multiple of Hq / Hkv (at least
                                  one); no effect on CUDA-core plans or when num_splits
                                  is forced */
    int32_t fail_launch;       /* 0 (default); n > 0: the n-th kernel launch the library
                                  makes from now on is not made and reports
                                  cudaErrorLaunchOutOfResources to its call, which returns
                                  SWA_ERR_CUDA (the test of the host's launch-error path);
                                  the field then returns to 0 */
    int32_t reserved;          /* must be 0 */
} swa_debug_options;

/* Set the controls above (NULL restores the defaults).  Returns
 * SWA_ERR_INVALID_ARG for a field outside its range. */
swa_status swa_set_debug_options(const swa_debug_options *opt);

/* The controls in effect. */
swa_status swa_get_debug_options(swa_debug_options *opt);

/* Greedy verification of a draft block: the argmax of every verify row's
 * logits (FUSED_SPARSE_ARGMAX, with the keep set of a pruned LM head) and
 * the number of drafted tokens accepted (SPECULATIVE_CONFIG's drafts), in
 * one launch ("The Fast Gemma Challenge: our verified-SOTA recipe, in full",
 * manifest entries FUSED_SPARSE_ARGMAX / FUSED_SPARSE_ARGMAX_BLOCK and
 * SPECULATIVE_CONFIG; section "What each piece does, and why": the fused
 * sparse argmax removes sampling overhead).
 *
 *   logits     bf16 [batch, q_len, vocab]  device, 2-byte aligned; row i of a
 *              sequence scores the token after its position q_pos + i
 *   keep_ids   int32 [vocab]  device or NULL: column j scores token keep_ids[j]
 *              (NULL: token j)
 *   draft      int32 [batch, q_len - 1]  device (may be NULL when q_len == 1):
 *              the drafted tokens that were fed as rows 1 .. q_len - 1
 *   argmax_out int32 [batch, q_len]  device, written: per row the token of the
 *              largest logit; among equal maxima the first column; a NaN is
 *              never the largest; a row with nothing above -inf gives column 0
 *   accepted   int32 [batch]  device, written: n = the largest n <= q_len - 1
 *              with argmax_out[b][i] == draft[b][i] for every i < n; the step
 *              emits draft[b][0 .. n) and then argmax_out[b][n]
 *   batch 1..65535, q_len 1..64, vocab >= 1.
 *
 * Asynchronous on `stream`; returns SWA_ERR_INVALID_ARG on bad arguments
 * before any CUDA call.  The library keeps a small per-device scratch
 * (8 bytes per row and 4 per sequence, zero between calls): the first call
 * with a larger batch * q_len allocates and zeroes it, which is refused
 * with SWA_ERR_WORKSPACE while the stream is capturing (make one call of
 * the largest size before capture).  Calls that overlap on one device race
 * on that scratch; order them (one stream, or events). */
swa_status swa_greedy_accept(const void *logits, const int32_t *keep_ids, const int32_t *draft,
                             int32_t *argmax_out, int32_t *accepted, int32_t batch,
                             int32_t q_len, int32_t vocab, swa_stream_t stream);

/* Bytes of the fixed device scratch used by swa_verify_attn_noalloc. */
#define SWA_NOALLOC_SCRATCH_BYTES ((size_t)16 << 20)

/* Allocation-free variant of swa_verify_attn (no counterpart on the pages:
 * it serves callers, not the method).
 *
 * Some callers must not allocate device memory at call time: an engine that
 * reserves (nearly) all GPU memory for its own pool at start-up, a plugin
 * that is only handed pointers by a host framework owning every allocation,
 * or a latency-critical path that cannot afford cudaMalloc's implicit device
 * synchronisation.  This entry point never calls cudaMalloc, cudaFree or any
 * allocating routine.  When the plan splits the keys into several chunks,
 * the split partials go to a fixed scratch array of
 * SWA_NOALLOC_SCRATCH_BYTES (16 MiB) that the library declares statically;
 * every GPU on which the library's kernels are loaded holds that array until
 * the process exits.
 *
 * Arguments, layouts, preconditions and results are those of
 * swa_verify_attn; the caller still owns and passes every input and output.
 * Differences:
 *  - If the chosen plan needs more scratch than SWA_NOALLOC_SCRATCH_BYTES
 *    (see swa_plan(): workspace_bytes), the call returns SWA_ERR_WORKSPACE
 *    with a message naming both sizes and launches nothing; a smaller
 *    dims->num_splits (1 needs no scratch) brings it under the limit.
 *  - The first call on a device resolves the scratch array's device address
 *    with cudaGetSymbolAddress (with that device current) and caches it; make
 *    that first call before any stream capture.
 *  - All calls on one device share the one array, and it keeps the last
 *    call's contents (nothing in it needs to start at zero: every partial is
 *    written before it is read within a call).  Calls that may overlap on the
 *    GPU, e.g. on different streams without ordering, race on it. */
swa_status swa_verify_attn_noalloc(const void *q, const void *k_cache, const void *v_cache,
                                   const int32_t *seq_lens, const int32_t *q_pos,
                                   int32_t window, float scale, void *out, float *lse,
                                   const swa_dims *dims, swa_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* SWA_H */
