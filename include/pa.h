/*
 * pa.h -- paged-attention decode on GB300 (sm_103a): the C ABI of libpa103.so.
 *
 * The operation.  A decode step gives each sequence b a few new query tokens
 * (q_lens[b] <= max_q_len rows per query head) that attend over that
 * sequence's cached keys and values.  The cache is a pool of fixed-size
 * physical pages; sequence b reaches its logical page p at physical block
 * block_tables[b][p] ("HSTU Paged Attention", RecSDK issue 1281, background:
 * historical K/V are read page by page from the paged KV cache).  For query
 * head h (KV head g = h / (Hq / Hkv)) and new-token row i < q_lens[b]:
 *
 *     n   = context_lens[b]          (counts the q_lens[b] new tokens, which are
 *                                     the last q_lens[b] positions)
 *     L   = causal ? n - q_lens[b] + i + 1 : n     visible keys 0 .. L-1
 *     s_j = sm_scale * <q[b,i,h,:], k_j>           k_j = K[block_tables[b][j/bs], j%bs, g, :]
 *     out[b,i,h,:] = sum_j softmax(s)_j v_j ,  lse[b,i,h] = log sum_j exp(s_j)
 *
 * Rows i >= q_lens[b] are padding: out = 0, lse = -inf.
 *
 * The work is split as in "Optimize paged-attention metadata decode" (FlyDSL
 * PR #910, Summary and Changes): a planner emits a work list for a persistent
 * grid of one CTA per SM (times a grid multiplier, default 1); a persistent
 * decode kernel processes it, writing whole results directly and per-range
 * partials (o_s, lse_s) otherwise; a reducer merges the partials by
 *     m* = max_s lse_s,  w_s = exp(lse_s - m*),  out = sum_s w_s o_s / sum_s w_s.
 * fp8 caches hold OCP E4M3 codes with one fp32 scale per tensor or one per
 * (block, slot, kv-head) row (FlyDSL PR #910, per_token_kv scale mode).
 *
 * Calling convention.  The caller owns all memory.  pa_plan, pa_decode and
 * pa_reduce allocate nothing, never synchronise the host and never abort: each
 * validates its arguments on the host, enqueues its kernel on `stream` and
 * returns a status.  They are stream-ordered, so the three calls on one stream
 * with one workspace form one decode step and can be captured in a CUDA graph.
 * Problems in the device-resident lengths or block tables cannot be seen by the
 * host.  The planner flags bad lengths and empties the work list (the output is
 * then all zeros with lse = -inf); the decode kernel checks every block id before
 * it loads the page, skips a page outside the pool and flags it (the rows of that
 * sequence are then unspecified).  Either way no kernel touches memory outside the
 * inputs.  pa_read_flags (the one synchronising call) returns the flags.
 *
 * Device pointers: q, k_cache, v_cache, k_scale, v_scale, block_tables,
 * context_lens, q_lens, out, lse and ws.  q, k_cache, v_cache and out must be
 * 16-byte aligned; ws 256-byte aligned.
 *
 * Besides the step, pa_append_kv writes a step's new K/V rows into their pages
 * (quantising them to fp8 where the cache is fp8), and pa_gather_kv copies a batch's
 * cached K and V rows out of the pages into contiguous buffers (the workspace copy of
 * the HSTU paged attention), with the same calling convention.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Entry points are the only symbols the library exports. */
#if defined(__GNUC__)
#define PA_API __attribute__((visibility("default")))
#else
#define PA_API
#endif

/* The same type as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st *pa_stream;

typedef enum {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = 1, /* null pointer, misalignment, negative size, bad enum value */
  PA_ERR_UNSUPPORTED = 2, /* head_dim, block_size or dtype combination not supported */
  PA_ERR_WORKSPACE = 3,   /* ws_bytes below pa_workspace_size() */
  PA_ERR_CUDA = 4,        /* a CUDA runtime call or a kernel launch failed */
  PA_ERR_DEVICE = 5       /* pa_read_flags: the device recorded an input problem */
} pa_status;

typedef enum { PA_BF16 = 0, PA_FP16 = 1, PA_FP8_E4M3 = 2 } pa_dtype;

typedef enum {
  PA_SCALE_NONE = 0,       /* 16-bit cache, or fp8 codes used as they are */
  PA_SCALE_PER_TENSOR = 1, /* k_scale, v_scale: one fp32 each */
  PA_SCALE_PER_TOKEN = 2   /* k_scale, v_scale: fp32 [num_blocks, block_size, num_kv_heads] */
} pa_scale_mode;

/* Where the log-sum-exp merge of split units runs.  A unit cut into ns pieces can be merged
 * by the last CTA to finish one of its pieces, inside pa_decode (an atomic arrival counter
 * per unit; no CTA ever waits for another), or by pa_reduce's own kernel, which spreads the
 * rows of the unit over many CTAs.  The first costs no launch but runs on one SM, so it
 * suits units of a few pieces; the second suits units cut into many.
 *   PA_MERGE_AUTO (0, the default): the library's choice, currently that of
 *     PA_MERGE_IN_REDUCE (measured fastest: a merge inside the decode runs after the merging
 *     CTA's own work and lengthens the decode's tail).
 *   PA_MERGE_IN_DECODE: pa_decode merges every unit and pa_reduce launches nothing.
 *   PA_MERGE_IN_REDUCE: pa_decode only writes partials and pa_reduce merges them all.
 * The choice changes the order of no sum inside a merge: outputs agree to rounding. */
typedef enum { PA_MERGE_AUTO = 0, PA_MERGE_IN_DECODE = 1, PA_MERGE_IN_REDUCE = 2 } pa_split_merge;

/* Device-side input problems, OR-ed into the flags word. */
enum {
  PA_FLAG_BAD_LENGTHS = 1,   /* q_lens[b] outside [0, max_q_len], context_lens[b] < q_lens[b],
                                or context_lens[b] > max_blocks_per_seq * block_size */
  PA_FLAG_BAD_BLOCK_ID = 2,  /* a block_tables entry in use lies outside [0, num_blocks) */
  PA_FLAG_WAIT_TIMEOUT = 4,  /* a kernel gave up a bounded wait on its own copies */
  PA_FLAG_STALE_PLAN = 8     /* pa_decode read lengths other than those pa_plan planned for
                                (they changed between the two calls); outputs unspecified */
};

typedef struct {
  int32_t batch;              /* B >= 1 */
  int32_t max_q_len;          /* Sq >= 1: query rows per sequence in q and out */
  int32_t num_q_heads;        /* Hq */
  int32_t num_kv_heads;       /* Hkv, divides Hq */
  int32_t head_dim;           /* D: 64, 128 or 256 */
  int32_t block_size;         /* tokens per page: a power of two in [16, 1024] */
  int32_t max_blocks_per_seq; /* columns of block_tables */
  int32_t num_blocks;         /* physical pages in the pool */
  int32_t q_dtype;            /* pa_dtype of q and out: PA_BF16 or PA_FP16 */
  int32_t kv_dtype;           /* pa_dtype of the cache: q_dtype or PA_FP8_E4M3 */
  int32_t kv_scale_mode;      /* pa_scale_mode; PA_SCALE_NONE unless kv_dtype is fp8 */
  int32_t causal;             /* 1: new token i sees keys up to its own position */
  float sm_scale;             /* logit scale, usually 1/sqrt(D) */
  int32_t num_ctas;           /* persistent grid size; 0: (SMs of the current device x grid_mult)
                                 x the decode CTAs that fit on one SM */
  int32_t grid_mult;          /* grid multiplier when num_ctas is 0; 0 means 1 */
  int32_t split_merge;        /* pa_split_merge: where units cut into several pieces are merged */
} pa_config;

/* Bytes of workspace a pa_plan/pa_decode/pa_reduce sequence needs for cfg:
 * the work list for (C + units) items and fp32 partials for as many splits,
 * where C is the persistent grid size and units = B * Hkv * row blocks.
 * May query the current device (num_ctas == 0).  Writes *bytes. */
PA_API pa_status pa_workspace_size(const pa_config *cfg, size_t *bytes);

/* Plan one decode step (device work, no host sync).  Reads context_lens[B] and
 * q_lens[B]; checks the lengths; writes the work list into ws.  Cuts the
 * concatenated token ranges of all (sequence, kv-head, row-block) units into C
 * contiguous tile-aligned pieces of equal size, one per CTA, so every CTA of the
 * persistent grid reads the same number of pages.  block_tables is not read here
 * (pa_decode checks every block id it uses) but must not be NULL. */
PA_API pa_status pa_plan(const pa_config *cfg, const int32_t *block_tables, const int32_t *context_lens,
                  const int32_t *q_lens, void *ws, size_t ws_bytes, pa_stream stream);

/* Run the persistent decode over the work list pa_plan left in ws.
 *   q        [B, Sq, Hq, D]            q_dtype
 *   k_cache  [num_blocks, block_size, Hkv, D]   kv_dtype (uint8 codes for fp8)
 *   v_cache  same layout as k_cache
 *   k_scale, v_scale  NULL unless fp8 with a scale mode (see pa_scale_mode)
 *   out      [B, Sq, Hq, D]            q_dtype; written for every unit done in one piece,
 *            with no keys, or merged here (see pa_split_merge)
 *   lse      [B, Sq, Hq] fp32 natural-log LSE, or NULL
 * The tables and lengths must be the ones given to pa_plan, with the same contents.  A CTA
 * of the tcgen05 decode (33 or more query rows per kv head; head dim 128 or 256, 128 for an
 * fp8 cache) derives its first work item from the lengths (the planner's rules) and starts
 * on it while the planner may still be running; it waits for the planner before the rest of
 * its list and before writing anything, and raises PA_FLAG_STALE_PLAN if the planner's first
 * item differs.  The other decode kernels wait for the planner first.
 * The kernels launch with programmatic dependent launch, so pa_decode reads q, the caches,
 * the tables and the lengths once the launch before it in the stream has let its dependents
 * start (a pa_plan call does so after its own wait on the launch before it): a kernel between
 * pa_plan and pa_decode that writes any of them must not let its dependents start early.
 * A decode that completed leaves the merge counters as pa_plan set them, so pa_decode may
 * run again on the same plan. */
PA_API pa_status pa_decode(const pa_config *cfg, const void *q, const void *k_cache, const void *v_cache,
                    const float *k_scale, const float *v_scale, const int32_t *block_tables,
                    const int32_t *context_lens, const int32_t *q_lens, void *out, float *lse,
                    void *ws, size_t ws_bytes, pa_stream stream);

/* Completes the step: merges the split partials pa_decode left in ws into out (and lse) for
 * every unit pa_decode did not merge itself (see pa_split_merge).  With PA_MERGE_IN_DECODE
 * there is none, and this call only validates its arguments and launches nothing. */
PA_API pa_status pa_reduce(const pa_config *cfg, void *out, float *lse, void *ws, size_t ws_bytes,
                    pa_stream stream);

/* Synchronise `stream` and return the device flags of the last plan/decode in ws
 * (PA_FLAG_* bits; 0 when the step was clean) in *flags.  Returns PA_ERR_DEVICE
 * when any flag is set, PA_OK otherwise. */
PA_API pa_status pa_read_flags(const void *ws, size_t ws_bytes, int32_t *flags, pa_stream stream);

/* Size of the device scratch array behind pa_decode_step_static (16 MiB). */
#define PA_STATIC_SCRATCH_BYTES ((size_t)16 << 20)

/* One whole decode step (plan, decode, reduce) that allocates nothing and needs no
 * workspace from the caller.  The pages have no counterpart: it exists for callers that
 * cannot allocate device memory -- code running under a framework or plugin interface that
 * hands out no allocator, loops that must not call cudaMalloc once serving has started
 * (cudaMalloc can synchronise the device and is not allowed during stream capture), and
 * deployments that forbid allocation after start-up.  Arguments are those of pa_decode
 * without ws/ws_bytes; the caller still provides q, the caches, scales, tables, lengths,
 * out and lse.
 *
 * The scratch is one file-scope __device__ array of PA_STATIC_SCRATCH_BYTES, reserved on
 * every GPU where the library's device code is loaded and held until the process exits.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 * with that device current and caches it; make that first call before any stream capture.
 * The cached address belongs to the device's primary context: after cudaDeviceReset (or any
 * other teardown of that context) it names freed memory, so a process that resets a device
 * must not call this entry point on that device again.
 * A problem whose pa_workspace_size() exceeds PA_STATIC_SCRATCH_BYTES is rejected with
 * PA_ERR_WORKSPACE before anything is launched.  All calls on a device share the one array
 * and each call overwrites what the previous one left there: calls whose kernels overlap on
 * the GPU (different streams, or different host threads without ordering) race and corrupt
 * each other's results.  Calls on one stream are ordered and safe.  pa_read_flags is not
 * available for this scratch (its address is private); device-side input problems leave
 * out unspecified. */
PA_API pa_status pa_decode_step_static(const pa_config *cfg, const void *q, const void *k_cache,
                                       const void *v_cache, const float *k_scale,
                                       const float *v_scale, const int32_t *block_tables,
                                       const int32_t *context_lens, const int32_t *q_lens,
                                       void *out, float *lse, pa_stream stream);

/* Paged -> contiguous copy of a batch's cached K and V (the copy the HSTU paged attention
 * makes from its paged cache into its workspace before attending: "HSTU Paged Attention"
 * K/V double-buffering issue, background and optimisation plan).
 *
 * Sequence b's tokens 0 .. context_lens[b] - 1 are copied, in token order, to rows
 * row_off[b] .. row_off[b] + context_lens[b] - 1 of k_out and of v_out, where
 * row_off[b] = context_lens[0] + ... + context_lens[b - 1]; a row is one token's
 * [num_kv_heads, head_dim] values exactly as the cache stores them (bf16, fp16 or E4M3
 * codes; per-token fp8 scales are not copied).  Reads cfg's batch, num_kv_heads, head_dim,
 * block_size, max_blocks_per_seq, num_blocks and kv_dtype; the other fields are ignored.
 *
 *   k_cache, v_cache  device, [num_blocks, block_size, num_kv_heads, head_dim], 16-byte aligned
 *   block_tables      device int32 [batch, max_blocks_per_seq]
 *   context_lens      device int32 [batch]
 *   k_out, v_out      device, room for max_rows rows of num_kv_heads * head_dim elements,
 *                     16-byte aligned
 *   row_offsets       NULL, or device int32 [batch + 1] that receives row_off[0 .. batch]
 *                     (row_off[batch] = rows copied)
 *   flags             NULL, or a device int32 the call ORs PA_FLAG_* bits into:
 *                     PA_FLAG_BAD_LENGTHS when a length is negative or exceeds
 *                     max_blocks_per_seq * block_size (that sequence counts as empty) or the
 *                     rows exceed max_rows (nothing is copied), PA_FLAG_BAD_BLOCK_ID for a
 *                     page whose block id lies outside [0, num_blocks) (its rows are not
 *                     written)
 *
 * Stream-ordered, allocates nothing.  PA_ERR_UNSUPPORTED for batch > 8192, head_dim or
 * block_size outside the decode's sets, or problems whose row or copy counts exceed int32. */
PA_API pa_status pa_gather_kv(const pa_config *cfg, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, const int32_t *context_lens,
                              void *k_out, void *v_out, int64_t max_rows, int32_t *row_offsets,
                              int32_t *flags, pa_stream stream);

/* Quantise-on-write KV append: write a decode step's new K/V rows into their pages.
 *
 * New row i < q_lens[b] of sequence b is cache position pos = context_lens[b] - q_lens[b] + i
 * (the new tokens are the last q_lens[b] of the context_lens[b] tokens, the positions the
 * decode's causal mask gives them), i.e. slot pos % block_size of physical block
 * block_tables[b][pos / block_size] ("HSTU Paged Attention", RecSDK issue 1281, background:
 * the paged KV cache).  Call it before pa_plan / pa_decode with the same tables and lengths.
 *   16-bit cache (kv_dtype == q_dtype): the row's bits are copied unchanged.
 *   fp8 cache: OCP E4M3 codes of row / scale, rounded to nearest (ties to even), magnitudes
 *   past 448 saturating to 448; scale modes of "Optimize paged-attention metadata decode"
 *   (FlyDSL PR #910, Breaking Changes: per_token_kv):
 *     PA_SCALE_PER_TOKEN   scale = amax(|row|) / 448 (1 for an all-zero row), computed in fp32
 *                          and WRITTEN to k_scale / v_scale [num_blocks, block_size, Hkv];
 *     PA_SCALE_PER_TENSOR  scale = k_scale[0] / v_scale[0], READ (one fp32 each);
 *     PA_SCALE_NONE        scale 1; k_scale / v_scale may be NULL.
 *   Quotients are IEEE fp32 divisions.  A NaN element gives a NaN code (0x7f or 0xff).
 * Reads cfg's batch, max_q_len, num_kv_heads, head_dim, block_size, max_blocks_per_seq,
 * num_blocks, q_dtype, kv_dtype and kv_scale_mode.
 *
 *   k_new, v_new   device, [batch, max_q_len, num_kv_heads, head_dim] in q_dtype, 16-byte
 *                  aligned; rows i >= q_lens[b] are ignored
 *   block_tables, context_lens, q_lens   device int32, as for pa_plan
 *   k_cache, v_cache   device, [num_blocks, block_size, num_kv_heads, head_dim] in kv_dtype,
 *                  16-byte aligned; only the new rows' slots are written
 *   k_scale, v_scale   device fp32 (see the scale modes)
 *   flags          NULL, or a device int32 the call ORs PA_FLAG_* bits into:
 *                  PA_FLAG_BAD_LENGTHS for a sequence whose lengths break the rules of
 *                  pa_plan (none of its rows is written), PA_FLAG_BAD_BLOCK_ID for a new row
 *                  whose page lies outside [0, num_blocks) (that row is not written)
 *
 * Stream-ordered, allocates nothing, never synchronises.  PA_ERR_INVALID_ARG for NULL or
 * misaligned pointers (scales NULL with a scale mode), PA_ERR_UNSUPPORTED for head_dim,
 * block_size or dtype combinations the decode does not take. */
PA_API pa_status pa_append_kv(const pa_config *cfg, const void *k_new, const void *v_new,
                              const int32_t *block_tables, const int32_t *context_lens,
                              const int32_t *q_lens, void *k_cache, void *v_cache,
                              float *k_scale, float *v_scale, int32_t *flags, pa_stream stream);

/* A static, human-readable name of a status. */
PA_API const char *pa_status_string(pa_status status);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
