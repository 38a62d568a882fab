// Internal declarations shared by the translation units of libmoe_route.so.
// Not part of the public ABI (that is include/moe_route.h).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "moe_route.h"

namespace moe {

// Sets the calling thread's message for moe_last_error(); returns `code`.
int set_error(int code, const char *fmt, ...);

// Unique key of the calling thread's current CUDA context (0 if there is
// none yet or the driver cannot say).  Host-side caches of per-context state
// (kernel attributes, symbol addresses) key on it as well as on the device,
// because cudaDeviceReset ends the context and the next call gets a new one.
unsigned long long context_key();

// Multiprocessor count of the current device (cached per device).
int sm_count();
int64_t l2_bytes();  // L2 cache size of the current device (0 if unknown)

// ---- launchers (arguments already validated by the C entry points) -------

cudaError_t launch_route_topk(const float *logits, const float *bias, int64_t NT, int E, int R,
                              int score_fn, int renormalize, int32_t *topk_idx, float *topk_w,
                              cudaStream_t stream);

cudaError_t launch_dispatch_count(const int32_t *topk_idx, int N, int T, int E, int R,
                                  int64_t cap, int32_t *expert_counts, int32_t *expert_offsets,
                                  int32_t *rank_counts, int32_t *rank_offsets,
                                  int32_t *send_counts, int32_t *pos, int32_t *status,
                                  cudaStream_t stream);

// Pairs whose row lies outside [row_lo, row_hi) are skipped.
cudaError_t launch_dispatch_pack(const void *x, const float *x_scales, const int32_t *pos,
                                 int64_t NT, int R, int64_t row_bytes, int scales_per_row,
                                 int64_t rows_total, void *packed_x, float *packed_scales,
                                 int32_t *packed_src, cudaStream_t stream);

// Pack whose positions are derived from per-block ranks (the second kernel
// of the decode-fused dispatch).  Token g lies in block b of the fused
// route kernel: b = g / (ranks_per_block * T) when blocks hold whole source
// ranks (ranks_per_block > 0), else (g / T) * blocks_per_rank + (g % T) / 32.
// On entry pos[g][k] holds the pair's rank among block b's pairs of its
// expert e = topk_idx[g][k]; the kernel replaces it with the row
//   local = expert_offsets[e] - expert_offsets[d*L] + chunk_prefix[(b/8)*Ep + e]
//           + sum over b' in [8*(b/8), b) of block_hist[b'*Ep + e] + rank,
//   pos   = local < cap ? d*cap + local : -1          (d = e / L)
// and packs as launch_dispatch_pack does.  When source ranks are split over
// several blocks (blocks_per_rank > 0), block s < N of the pack kernel also
// writes row s of send_counts, the sum of the per-block counts block_send.
struct PackDerive {
    const int32_t *topk_idx;
    const int32_t *expert_offsets;
    const uint16_t *chunk_prefix;  // [blocks/8][Ep]: pairs of expert e in chunks of 8 blocks before
    const unsigned char *block_hist;  // [blocks][Ep]: pairs of expert e in block b
    const uint16_t *block_send;    // [blocks][N]: pairs of block b sent to rank d
    int32_t *send_counts;
    int N, T, ranks_per_block, blocks_per_rank, L, Ep, cap;
    int route_blocks;  // blocks of the fused route kernel (each fills an SM)
};
cudaError_t launch_dispatch_pack_derive(const void *x, const float *x_scales, int32_t *pos, int64_t NT,
                                        int R, int64_t row_bytes, int scales_per_row, int64_t rows_total,
                                        const PackDerive &D, void *packed_x, float *packed_scales,
                                        int32_t *packed_src, cudaStream_t stream);
// The fp8-quantising pack in the same deriving form (bf16 rows in).
cudaError_t launch_dispatch_pack_quant_derive(const void *x, int32_t *pos, int64_t NT, int R, int H,
                                              int64_t rows_total, const PackDerive &D, void *packed_q,
                                              float *packed_scales, int32_t *packed_src, cudaStream_t stream);
// Rows of x the pack prefetches into L2 (at most half the L2; 0 for rows
// wider than one bulk prefetch).
int64_t pack_prefetch_rows(int64_t NT, int64_t row_bytes);

// Bulk-copy pack (whole rows through shared memory); rows of more than
// 48 KB are not supported (pack_bulk_stages returns 0).
int pack_bulk_stages(int64_t row_bytes);
cudaError_t launch_dispatch_pack_bulk(const void *x, const float *x_scales, const int32_t *pos,
                                      int64_t NT, int R, int64_t row_bytes, int scales_per_row,
                                      int64_t rows_total, void *packed_x, float *packed_scales,
                                      int32_t *packed_src, cudaStream_t stream);

// Reads and clears the library's device error word (set when a bounded
// wait inside a kernel gives up).
cudaError_t take_device_error(int *err, cudaStream_t stream);

// Decode-fused route + count + pack.  Workspace bytes for a batch (0 when
// no fused form that uses a workspace takes it).
int64_t fused_workspace_bytes(int N, int T, int E);
const char *fused_unsupported(int N, int T, int E, int R, int64_t row_bytes);  // "" when supported
cudaError_t launch_dispatch_fused(const float *logits, const float *bias, int score_fn, int renormalize,
                                  const void *x, const float *x_scales, int N, int T, int E, int R,
                                  int64_t row_bytes, int spr, int64_t cap, int32_t *topk_idx,
                                  float *topk_w, int32_t *expert_counts, int32_t *expert_offsets,
                                  int32_t *rank_counts, int32_t *rank_offsets, int32_t *send_counts,
                                  int32_t *pos, int32_t *status, void *packed_x, float *packed_scales,
                                  int32_t *packed_src, void *workspace, cudaStream_t stream);

// Decode-fused route + count + fp8-quantising pack (bf16 rows in; always the
// two-kernel form).  "" when the batch is within its limits.
const char *fused_quant_unsupported(int N, int T, int E, int R);
cudaError_t launch_dispatch_fused_quant(const float *logits, const float *bias, int score_fn, int renormalize,
                                        const void *x, int N, int T, int E, int R, int H, int64_t cap,
                                        int32_t *topk_idx, float *topk_w, int32_t *expert_counts,
                                        int32_t *expert_offsets, int32_t *rank_counts, int32_t *rank_offsets,
                                        int32_t *send_counts, int32_t *pos, int32_t *status, void *packed_q,
                                        float *packed_scales, int32_t *packed_src, void *workspace,
                                        cudaStream_t stream);

// Small decode batches: route + count + pack in one thread-block cluster.
bool dispatch_small_eligible(int64_t NT, int E, int R, int64_t row_bytes);
cudaError_t launch_dispatch_small(const float *logits, const float *bias, int score_fn, int renormalize,
                                  const void *x, const float *x_scales, int N, int T, int E, int R,
                                  int64_t row_bytes, int spr, int64_t cap, int32_t *topk_idx,
                                  float *topk_w, int32_t *expert_counts, int32_t *expert_offsets,
                                  int32_t *rank_counts, int32_t *rank_offsets, int32_t *send_counts,
                                  int32_t *pos, int32_t *status, void *packed_x, float *packed_scales,
                                  int32_t *packed_src, cudaStream_t stream);

// Bounded-wait self-test: status[0] <- MOE_OK / MOE_ERR_TIMEOUT after waiting
// (at most `polls` polls) for status[1] to become nonzero.
cudaError_t launch_selftest_wait(int32_t *status, long long polls, cudaStream_t stream);

// Scratch for the allocation-free fused dispatch: a fixed device array of
// the library (size in bytes; address on the current device).
int64_t fused_static_scratch_bytes();
cudaError_t fused_static_scratch(void **out);

cudaError_t launch_dispatch_pack_quant(const void *x, const int32_t *pos, int64_t NT, int R, int H,
                                       int64_t rows_total, void *packed_q, float *packed_scales,
                                       int32_t *packed_src, cudaStream_t stream);

// Pairs whose row lies outside [row_lo, row_hi) contribute nothing.
cudaError_t launch_combine(const void *y, int y_dtype, const int32_t *pos, const float *topk_w,
                           int64_t NT, int R, int H, int64_t rows_total, void *out,
                           cudaStream_t stream);

// Expert-parallel local path of one rank (rows [row_lo, row_hi) only).
cudaError_t launch_pack_rank(const void *x, const float *x_scales, const int32_t *pos, int64_t NT,
                             int R, int64_t row_bytes, int scales_per_row, int64_t row_lo,
                             int64_t row_hi, void *packed_x, float *packed_scales,
                             int32_t *packed_src, cudaStream_t stream);
cudaError_t launch_combine_rank(const void *y, int y_dtype, const int32_t *pos, const float *topk_w,
                                int64_t NT, int R, int H, int64_t row_lo, int64_t row_hi, void *out,
                                cudaStream_t stream);

cudaError_t launch_combine_partials(const void *y, int y_dtype, const int32_t *pos,
                                    const float *topk_w, int64_t NT, int R, int H, int64_t cap,
                                    int64_t rows_total, int P, void *partial, int32_t *slot_rank,
                                    cudaStream_t stream);

cudaError_t launch_reduce_partials(const void *partial, int y_dtype, const int32_t *slot_rank,
                                   int64_t NT, int P, int H, void *out, cudaStream_t stream);

}  // namespace moe
