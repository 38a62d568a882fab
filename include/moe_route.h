/*
 * moe_route.h -- C ABI of the GB300 (sm_103a) MoE token-routing library
 * (libmoe_route.so): route top-k, dispatch count, dispatch pack, combine.
 *
 * The routing problem follows "Enabling trillion-parameter models on AWS
 * EFA", section "Send and receive buffers": N ranks, T tokens per rank, each
 * token routed to R of E experts, hidden size H; one rank receives at most
 * N*T*max(R, E/N) rows.  Here all N ranks are partitions of one GPU's memory:
 * rank d owns experts [d*E/N, (d+1)*E/N) and a receive region of cap_rows
 * rows; a "send" is a store into another rank's region.
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers owned by the caller; the library
 *     allocates nothing and keeps no pointer after the call returns.
 *   - Arrays are dense and row-major; token g = s*T + t is token t of source
 *     rank s.  Rows of x, packed_x, y and out must start on 16-byte
 *     boundaries (H as required below guarantees it when the base is).
 *   - Work is enqueued on `stream` (a cudaStream_t passed as void*; NULL is
 *     the legacy default stream).  No call synchronises the host except
 *     moe_read_status.  Grids depend only on the dimensions, never on
 *     routing results, so a call sequence can be captured in a CUDA graph.
 *   - Return value: MOE_OK, or a negative MOE_ERR_* code.  Argument errors
 *     are detected on the host before anything is enqueued; the message is
 *     available from moe_last_error() in the calling thread.
 *   - Device-side problems (a rank over capacity, invalid expert ids) never
 *     trap: moe_dispatch_count writes a status word on the device, pos
 *     entries of affected pairs become -1, and later steps skip them.
 *   - Kernels are launched with programmatic stream serialization and let
 *     the next kernel in the stream be scheduled early (before their own
 *     results are complete).  This only matters to a caller whose own next
 *     kernel is also launched with that attribute: such a kernel must wait
 *     (griddepcontrol.wait / cudaGridDependencySynchronize) before it reads
 *     anything the library writes.  Kernels launched without it, copies and
 *     events are ordered as usual.
 *
 * Points where this interface departs from the plain problem statement's
 * naming, so that a reader can map one onto the other:
 *   - moe_dispatch_count takes no workspace: it runs in one thread-block
 *     cluster whose blocks exchange histograms through distributed shared
 *     memory, so it needs no global scratch.
 *   - MoeSizes has one field per caller allocation: topk_idx_bytes and
 *     topk_w_bytes rather than one top-k size; five count-array sizes rather
 *     than one; total_pairs (N*T*R routed pairs, not rows of a buffer);
 *     fused_workspace_bytes, the only scratch any call takes.
 *   - MoeDims.reserved makes the padding before the 64-bit cap_rows explicit
 *     (the same layout under every compiler and binding); it must be 0.
 *   - The device status word also reports invalid expert ids
 *     (MOE_ERR_INVALID_ARG).  MOE_ERR_TIMEOUT, reserved in the problem
 *     statement, reports a bounded wait that gave up (the bulk pack's
 *     shared-memory barriers, through moe_take_device_error; the wait
 *     self-test, through its status word).
 */
#ifndef MOE_ROUTE_H
#define MOE_ROUTE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
#define MOE_OK 0
#define MOE_ERR_INVALID_ARG (-1) /* bad dims/pointers; also device status for invalid expert ids */
#define MOE_ERR_UNSUPPORTED (-2) /* valid request this build does not implement */
#define MOE_ERR_CUDA (-3)        /* a CUDA runtime call or kernel launch failed */
#define MOE_ERR_CAPACITY (-4)    /* device status: a rank received more than cap_rows rows */
#define MOE_ERR_TIMEOUT (-5)     /* device status: a bounded wait gave up */

/* ---- element types ------------------------------------------------------ */
#define MOE_BF16 0           /* bfloat16 */
#define MOE_F32 1            /* IEEE binary32 */
#define MOE_FP8E4M3_BLK128 2 /* fp8 e4m3 codes + one f32 scale per 128 elements (x only) */

/* ---- router score functions --------------------------------------------- */
#define MOE_SOFTMAX 0 /* softmax over all E experts, then top-R */
#define MOE_SIGMOID 1 /* logistic sigmoid per expert */
/* Flag OR'ed into score_fn: the bias takes part in the selection only (the
 * DeepSeek-V3 router convention): scores s_e = score(logit_e), selection
 * key fl32(s_e + bias_e), weights s_e of the selected experts. */
#define MOE_BIAS_SELECT_ONLY 0x10

/* Problem dimensions.  Limits: N >= 1, T >= 0, 1 <= E <= 1024, E % N == 0,
 * 1 <= R <= min(E, 32), 8 <= H <= 2^24 and H % 8 == 0 (H % 128 == 0 for
 * fp8 x), N*T*R < 2^31, N*cap_rows < 2^31. */
typedef struct MoeDims {
    int32_t N;        /* ranks (partitions of one GPU's memory) */
    int32_t T;        /* tokens per rank */
    int32_t E;        /* experts; expert e lives on rank e / (E/N) */
    int32_t R;        /* experts per token */
    int32_t H;        /* hidden size (elements per token row); H % 8 == 0,
                         H % 128 == 0 for fp8 rows, H <= 2^24 */
    int32_t x_dtype;  /* MOE_BF16, MOE_F32 or MOE_FP8E4M3_BLK128: dispatched rows */
    int32_t y_dtype;  /* MOE_BF16 or MOE_F32: expert outputs read by combine and its output */
    int32_t reserved; /* must be 0 */
    int64_t cap_rows; /* rows per rank receive region; 0 selects N*T*max(R, E/N) */
} MoeDims;

/* Sizes of every buffer the caller allocates, in bytes (moe_buffer_sizes). */
typedef struct MoeSizes {
    int64_t bound_rows;          /* N*T*max(R, E/N): the pages' worst case per rank */
    int64_t cap_rows;            /* effective per-rank capacity */
    int64_t total_pairs;         /* N*T*R routed (token, expert) pairs */
    int64_t logits_bytes;        /* f32 [N*T][E] */
    int64_t topk_idx_bytes;      /* i32 [N*T][R] */
    int64_t topk_w_bytes;        /* f32 [N*T][R] */
    int64_t pos_bytes;           /* i32 [N*T][R] */
    int64_t expert_counts_bytes; /* i32 [E] */
    int64_t expert_offsets_bytes;/* i32 [E+1] */
    int64_t rank_counts_bytes;   /* i32 [N] */
    int64_t rank_offsets_bytes;  /* i32 [N+1] */
    int64_t send_counts_bytes;   /* i32 [N][N] */
    int64_t x_bytes;             /* [N*T][H] of x_dtype */
    int64_t x_scales_bytes;      /* f32 [N*T][H/128] (fp8 only, else 0) */
    int64_t packed_x_bytes;      /* [N*cap][H] of x_dtype */
    int64_t packed_scales_bytes; /* f32 [N*cap][H/128] (fp8 only, else 0) */
    int64_t packed_src_bytes;    /* i32 [N*cap] */
    int64_t y_bytes;             /* [N*cap][H] of y_dtype */
    int64_t out_bytes;           /* [N*T][H] of y_dtype */
    int64_t status_bytes;        /* i32 [1] */
    int64_t partial_slots;       /* P = min(R, N): partial rows per token */
    int64_t partial_bytes;       /* [N*T][P][H] of y_dtype (moe_combine_partials) */
    int64_t slot_rank_bytes;     /* i32 [N*T][P] */
    int64_t fused_workspace_bytes; /* workspace of moe_dispatch_fused (zero-fill once before first use;
                                      0 when no fused form that uses one takes the batch) */
} MoeSizes;

/* Fill *out with the buffer sizes for dims (host only, no CUDA call).
 * Returns MOE_OK or MOE_ERR_INVALID_ARG / MOE_ERR_UNSUPPORTED. */
int moe_buffer_sizes(const MoeDims *dims, MoeSizes *out);

/* Route top-k.  Source: "Efficient and portable mixture-of-experts
 * communication", section "Introduction" (a small linear router yields a
 * probability distribution; the top-K experts are chosen and weighted by
 * it); "Lower latency and higher throughput with multi-node DeepSeek
 * deployment", section "MoE Router" (top-k with index tracking; one router
 * serves DeepSeek- and Mixtral-style models).
 *   logits   f32 [N*T][E]            router logits
 *   bias     f32 [E] or NULL         per-expert bias added to every logit
 *   score_fn MOE_SOFTMAX | MOE_SIGMOID, optionally | MOE_BIAS_SELECT_ONLY
 *   renormalize  nonzero: divide the selected scores by their sum
 *   topk_idx i32 [N*T][R] (out)      experts by key descending; equal keys
 *                                    -> lower index.  Key z = fl32(logit +
 *                                    bias); with MOE_BIAS_SELECT_ONLY the key
 *                                    is fl32(s + bias), s = f32 score of the
 *                                    raw logit
 *   topk_w   f32 [N*T][R] (out)      score of each selected expert
 * Scores are computed in f32 (softmax over all E) from z, or from the raw
 * logits with MOE_BIAS_SELECT_ONLY.  The pages do not say where the bias
 * enters; adding it to the logit is the default reading.  With the flag,
 * the selection is decided on f32 scores: keys within a few units in the
 * last place of each other may order differently from an exact-arithmetic
 * reference.  Non-finite logits give unspecified, but always in-range,
 * selections. */
int moe_route_topk(const MoeDims *dims, const float *logits, const float *bias, int score_fn,
                   int renormalize, int32_t *topk_idx, float *topk_w, void *stream);

/* Dispatch count.  Source: "Enabling trillion-parameter models on AWS EFA",
 * section "Dispatch and combine" (per-expert token counts from
 * shared-memory atomics, then a cumulative sum gives the offsets for
 * packing tokens contiguously per destination); "Efficient and portable
 * mixture-of-experts communication", section "Dispatch" (tokens grouped per
 * expert for the grouped GEMM).
 *   topk_idx       i32 [N*T][R] (in)
 *   expert_counts  i32 [E]   (out) pairs routed to each expert
 *   expert_offsets i32 [E+1] (out) exclusive prefix sum of expert_counts
 *   rank_counts    i32 [N]   (out) rows each rank receives (may exceed cap)
 *   rank_offsets   i32 [N+1] (out) exclusive prefix sum of rank_counts
 *   send_counts    i32 [N][N](out) [s][d]: rows source rank s sends to rank d
 *   pos            i32 [N*T][R] (out) receive row of pair (g,k):
 *                  d*cap + (expert_offsets[e] - rank_offsets[d]) + (number of
 *                  earlier tokens routed to e); -1 for a dropped pair
 *   status         i32 [1]   (out, device) MOE_OK, MOE_ERR_CAPACITY (some
 *                  rank over cap; its last rows get pos = -1) or
 *                  MOE_ERR_INVALID_ARG (an expert id outside [0,E) or a
 *                  repeated expert within a token; those pairs get pos = -1
 *                  and are not counted)
 * Within a rank region rows are grouped by expert (ascending) and ordered
 * by token (ascending) inside an expert: deterministic, independent of
 * scheduling.  Read status with moe_read_status. */
int moe_dispatch_count(const MoeDims *dims, const int32_t *topk_idx, int32_t *expert_counts,
                       int32_t *expert_offsets, int32_t *rank_counts, int32_t *rank_offsets,
                       int32_t *send_counts, int32_t *pos, int32_t *status, void *stream);

/* Dispatch pack.  Source: "Efficient and portable mixture-of-experts
 * communication", section "Dispatch" (the message of a token is its
 * activations, their block scales and its index on the source rank);
 * "Enabling trillion-parameter models on AWS EFA", section "Dispatch and
 * combine" (tokens packed contiguously per destination).
 *   x             [N*T][H] of x_dtype (in)
 *   x_scales      f32 [N*T][H/128] (in, fp8 only; else NULL)
 *   pos           i32 [N*T][R] from moe_dispatch_count
 *   packed_x      [N*cap][H] of x_dtype (out): row pos[g][k] = x[g]
 *   packed_scales f32 [N*cap][H/128] (out, fp8 only; else NULL)
 *   packed_src    i32 [N*cap] (out): row pos[g][k] = g*R + k
 * Only rows [d*cap, d*cap + min(rank_counts[d], cap)) of each region are
 * written; pairs with pos < 0 (or outside [0, N*cap)) are skipped.
 * Ordering: like every kernel here, pack reads its inputs only after the
 * previous kernel in the stream has completed.  Before that it may issue L2
 * prefetches of x (hints only, which never return stale data) so that the
 * rows are on chip by the time count finishes. */
int moe_dispatch_pack(const MoeDims *dims, const void *x, const float *x_scales,
                      const int32_t *pos, void *packed_x, float *packed_scales,
                      int32_t *packed_src, void *stream);

/* Decode-fused dispatch: moe_route_topk, moe_dispatch_count and
 * moe_dispatch_pack in one call, with the same arguments and identical
 * outputs.  Source: "Hosting Qwen on Blackwell", section "Expert parallel"
 * (for decode the whole dispatch kernel is fused into one).
 *   workspace  device scratch of MoeSizes.fused_workspace_bytes bytes,
 *              16-byte aligned, owned by the caller, ZERO-FILLED BEFORE ITS
 *              FIRST USE (cudaMemset once after allocating it).  Every call
 *              leaves it ready for the next one, so it is set up once and
 *              reused; calls that may run at the same time need separate
 *              workspaces.
 * Decode batches only, in one of two forms (else MOE_ERR_UNSUPPORTED before
 * anything is enqueued: use the three calls):
 *   - N*T <= 512, E <= 256 and at most 256 KB of rows read and written per
 *     32 tokens (32 * (1 + R) * row bytes), any T and R: one thread-block
 *     cluster whose blocks own 32 tokens each and exchange only per-expert
 *     counts through distributed shared memory (no grid barrier; the
 *     workspace is not touched);
 *   - otherwise N*T <= 4096 and E <= 512, any T and R: two kernels.  The
 *     first routes the tokens in blocks of at most 32 (never across a
 *     source rank), records each pair's rank among its block's pairs of the
 *     same expert and publishes the block's per-expert counts to the
 *     workspace; the block that finishes last scans them into prefixes per
 *     chunk of 8 blocks and the count outputs.  No block waits for
 *     another.  The second is the pack kernel, which derives each pair's
 *     row from those and writes pos as it packs.
 * On GB300 both forms beat the three separate calls: 256 tokens with R = 2
 * and 2 KB rows 12.5 vs 15.5 us; the DeepSeek-V3-shaped decode batch (4096
 * tokens, 14 KB rows) 85.0 vs 85.9 us; the Kimi-K2-shaped one 87.1 vs
 * 88.9 us.
 * An empty batch (N*T == 0) is always accepted: like moe_dispatch_count it
 * writes zero counts and offsets and MOE_OK (the workspace is not touched
 * and may be NULL). */
int moe_dispatch_fused(const MoeDims *dims, const float *logits, const float *bias, int score_fn,
                       int renormalize, const void *x, const float *x_scales, int32_t *topk_idx,
                       float *topk_w, int32_t *expert_counts, int32_t *expert_offsets,
                       int32_t *rank_counts, int32_t *rank_offsets, int32_t *send_counts, int32_t *pos,
                       int32_t *status, void *packed_x, float *packed_scales, int32_t *packed_src,
                       void *workspace, void *stream);

/* Decode-fused dispatch with fp8 quantisation: moe_route_topk,
 * moe_dispatch_count and moe_dispatch_pack_quant in one call, with the same
 * arguments and identical outputs (bf16 rows in; e4m3 codes and one f32
 * scale per 128 elements out, as moe_dispatch_pack_quant writes them).
 * Sources: "Hosting Qwen on Blackwell", section "Expert parallel" (the
 * decode dispatch fused into one); "Lower latency and higher throughput
 * with multi-node DeepSeek deployment", section "Quantization" (activations
 * quantised on the fly, one scaling factor per 128-element vector).
 *   dims       describe the bf16 rows (x_dtype MOE_BF16, H % 128 == 0)
 *   x          bf16 [N*T][H] (in)
 *   packed_q   e4m3 [N*cap][H] (out), packed_scales f32 [N*cap][H/128] (out),
 *              packed_src i32 [N*cap] (out): sized as for
 *              moe_dispatch_pack_quant (MoeSizes of the same dims with
 *              x_dtype MOE_FP8E4M3_BLK128)
 *   workspace  as for moe_dispatch_fused (MoeSizes.fused_workspace_bytes,
 *              zero-filled before its first use, ready again after every
 *              call); NULL allowed for an empty batch
 * Always the two-kernel form: N*T <= 4096, E <= 512, any T and R (else
 * MOE_ERR_UNSUPPORTED before anything is enqueued: use the three calls).
 * On GB300, DeepSeek-V3-shaped decode batch: 55.0 us against 58.3 us for
 * the three separate calls. */
int moe_dispatch_fused_quant(const MoeDims *dims, const float *logits, const float *bias, int score_fn,
                             int renormalize, const void *x, int32_t *topk_idx, float *topk_w,
                             int32_t *expert_counts, int32_t *expert_offsets, int32_t *rank_counts,
                             int32_t *rank_offsets, int32_t *send_counts, int32_t *pos, int32_t *status,
                             void *packed_q, float *packed_scales, int32_t *packed_src, void *workspace,
                             void *stream);

/* moe_dispatch_fused without a workspace argument: for callers that cannot
 * allocate device memory when they dispatch (a plug-in inside another
 * framework's execution loop that has no allocator of its own, or serving
 * code whose memory is fixed at start-up and must not call cudaMalloc on
 * its hot path, where it would synchronise the device and could fail under
 * memory pressure).  The pages have no counterpart: this is a deployment
 * convenience of this library.
 *   Scratch: a fixed array of 256 KiB in the library's device memory,
 *   reserved on every GPU that loads the library until the process exits
 *   (enough for every batch moe_dispatch_fused accepts: N*T <= 4096 and
 *   E <= 512 need at most 216,064 bytes; larger needs are rejected with
 *   MOE_ERR_UNSUPPORTED).  It starts zero-filled and every call leaves it
 *   ready for the next.
 *   The first call on a device looks up the array's device address (with
 *   that device current); make that first call before any stream capture.
 *   The address is cached per device and CUDA context: after
 *   cudaDeviceReset the next call looks it up again, so after a reset, too,
 *   make one call before capturing.  The call itself allocates nothing.
 *   Every call shares the one array, which keeps the last call's contents.
 *   Calls that overlap on the GPU (other streams, other host threads) race
 *   on the array and must be ordered by the caller.
 * Other arguments, outputs and limits as moe_dispatch_fused. */
int moe_dispatch_fused_static(const MoeDims *dims, const float *logits, const float *bias, int score_fn,
                              int renormalize, const void *x, const float *x_scales, int32_t *topk_idx,
                              float *topk_w, int32_t *expert_counts, int32_t *expert_offsets,
                              int32_t *rank_counts, int32_t *rank_offsets, int32_t *send_counts,
                              int32_t *pos, int32_t *status, void *packed_x, float *packed_scales,
                              int32_t *packed_src, void *stream);

/* Dispatch pack with fp8 block quantisation fused in.  Source: "Lower
 * latency and higher throughput with multi-node DeepSeek deployment",
 * section "Quantization" (activations quantised on the fly, one scaling
 * factor per 128-element vector); "Efficient and portable mixture-of-experts
 * communication", section "Dispatch" (the message carries the activations
 * and their block scales).
 *   dims          x_dtype must be MOE_BF16 (the rows read); H % 128 == 0
 *   x             bf16 [N*T][H] (in)
 *   pos           i32 [N*T][R] from moe_dispatch_count
 *   packed_q      u8 [N*cap][H] (out): e4m3 codes of x[g] at row pos[g][k]
 *   packed_scales f32 [N*cap][H/128] (out): the block scales of that row
 *   packed_src    i32 [N*cap] (out): row pos[g][k] = g*R + k
 * Per 128-element block of a row: amax = max |x|; scale = fl32(amax/448);
 * code = e4m3 (sign, 4-bit exponent with bias 7, 3-bit mantissa; no
 * infinities; largest value 448) of fl32(x/scale), rounded to nearest with
 * ties to even and saturated at +-448; amax == 0 gives scale 0 and codes 0.
 * The packed buffers have the sizes moe_buffer_sizes reports for the same
 * dims with x_dtype = MOE_FP8E4M3_BLK128.  NaN or infinite inputs give
 * unspecified codes.  Rows are skipped like in moe_dispatch_pack. */
int moe_dispatch_pack_quant(const MoeDims *dims, const void *x, const int32_t *pos, void *packed_q,
                            float *packed_scales, int32_t *packed_src, void *stream);

/* Combine.  Source: "Efficient and portable mixture-of-experts
 * communication", section "Combine" (each token reads its experts' outputs
 * through the routing table and forms their router-weighted average);
 * "Enabling trillion-parameter models on AWS EFA", sections "Dispatch and
 * combine" and "Evaluation" (accumulation on the receiving side only).
 *   y      [N*cap][H] of y_dtype (in): expert output of each received row
 *   pos    i32 [N*T][R], topk_w f32 [N*T][R] (in)
 *   out    [N*T][H] of y_dtype (out): out[g] = sum_k topk_w[g][k] * y[pos[g][k]],
 *          accumulated in f32 in k order, rounded once (bf16: to nearest even).
 * Pairs with pos < 0 (or outside [0, N*cap)) contribute nothing. */
int moe_combine(const MoeDims *dims, const void *y, const int32_t *pos, const float *topk_w,
                void *out, void *stream);

/* Dispatch pack restricted to one rank (expert-parallel prefill with
 * replicated inputs: a rank selects only the tokens routed to its own
 * experts).  Source: "Hosting Qwen on Blackwell", section "Expert parallel".
 * Same arguments and layout as moe_dispatch_pack; only pairs whose row lies
 * in rank `rank`'s region [rank*cap, (rank+1)*cap) are written.
 * 0 <= rank < N. */
int moe_dispatch_pack_rank(const MoeDims *dims, int rank, const void *x, const float *x_scales,
                           const int32_t *pos, void *packed_x, float *packed_scales,
                           int32_t *packed_src, void *stream);

/* Local accumulation of one rank (expert-parallel prefill: each rank sums
 * its own experts' outputs for every token; an all-reduce over ranks, not
 * part of this library, completes the combine).  Source: "Hosting Qwen on
 * Blackwell", section "Expert parallel".
 *   out [N*T][H] of y_dtype (out): out[g] = sum over the pairs of g on rank
 *       `rank` of topk_w * y[pos], f32 accumulation in k order (0 for
 *       tokens with no pair there).  Summed over all ranks this is
 *       moe_combine's result up to rounding.  0 <= rank < N. */
int moe_combine_rank(const MoeDims *dims, int rank, const void *y, const int32_t *pos,
                     const float *topk_w, void *out, void *stream);

/* Combine with send-side accumulation, first half: one partial row per
 * (token, destination rank).  Source: "Enabling trillion-parameter models on
 * AWS EFA", section "Evaluation" (accumulating on the send side moves less
 * data back, with some accuracy cost).
 *   partial   [N*T][P][H] of y_dtype (out), P = min(R, N): slot j of token g
 *             is the j-th distinct rank of g's pairs in k order; it holds the
 *             sum over g's pairs on that rank of topk_w * y[pos] (f32,
 *             rounded once to y_dtype).  Unused slots are zero rows.
 *   slot_rank i32 [N*T][P] (out): the rank of each slot, -1 if unused. */
int moe_combine_partials(const MoeDims *dims, const void *y, const int32_t *pos,
                         const float *topk_w, void *partial, int32_t *slot_rank, void *stream);

/* Combine with send-side accumulation, second half: out[g] = sum of token
 * g's used partial rows (f32 accumulation, rounded once to y_dtype). */
int moe_combine_reduce_partials(const MoeDims *dims, const void *partial, const int32_t *slot_rank,
                                void *out, void *stream);

/* Wait for `stream`, then read the device status word written by
 * moe_dispatch_count.  Returns that status (MOE_OK or a MOE_ERR_* code), or
 * MOE_ERR_CUDA if the wait or the copy failed. */
int moe_read_status(const int32_t *status, void *stream);

/* Self-test of a bounded wait (the pages have no counterpart: this is a
 * diagnostic of this implementation).  Enqueues one thread that waits, with
 * a bounded poll (a sleep of 32 ns doubling to 128 ns between polls), for
 * status[1] to become nonzero, at most `polls` times (1 <= polls <= 2^20,
 * well under a second at the upper end).  status[0] then becomes MOE_OK if
 * the word changed and MOE_ERR_TIMEOUT if the wait gave up.  Nothing in the
 * library writes status[1]: left at zero, the wait runs out, which shows
 * that a wait that is never satisfied ends with a status the host can read
 * and leaves the context usable.
 *   status  i32 [2] (device; [1] is read, [0] written)
 * Returns MOE_OK once enqueued (read status[0] after synchronising),
 * MOE_ERR_INVALID_ARG or MOE_ERR_CUDA. */
int moe_selftest_bounded_wait(int32_t *status, int64_t polls, void *stream);

/* Wait for `stream`, then return and clear the library's device error word:
 * MOE_OK, or MOE_ERR_TIMEOUT if a bounded wait inside one of the library's
 * kernels gave up since the last call (that kernel's output is then
 * incomplete).  MOE_ERR_CUDA if the wait or the copy failed.  The word is
 * shared by every stream and thread of the process. */
int moe_take_device_error(void *stream);

/* Message for the last error returned in the calling thread ("" if none). */
const char *moe_last_error(void);

/* Library ABI version (major*10000 + minor*100 + patch).  1.1: the
 * MOE_BIAS_SELECT_ONLY flag, moe_dispatch_fused_static,
 * moe_selftest_bounded_wait, the single-cluster fused path and H <= 2^24.
 * 1.2: moe_dispatch_fused_quant; the fused dispatch's workspace is
 * zero-filled once by the caller (no clearing inside the call) and may be
 * NULL for an empty batch; R up to 32 in the fused dispatch.
 * A caller can compare MOE_VERSION (the header it was built against) with
 * moe_version() (the library it loaded). */
#define MOE_VERSION 10200
int moe_version(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ROUTE_H */
