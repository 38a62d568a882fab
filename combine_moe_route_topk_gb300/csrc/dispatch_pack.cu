// Dispatch pack: copy every token row to the R receive rows chosen by the
// count step.
//
// "Efficient and portable mixture-of-experts communication", section
// "Dispatch": a token's message is its activations, their block scaling
// factors and its index on the source rank.  "Enabling trillion-parameter
// models on AWS EFA", section "Dispatch and combine": tokens are packed
// contiguously per destination.  Here the destination regions are
// partitions of one allocation, so the "send" is the packing store itself.
//
// Pairs whose row is negative (dropped by count) or outside the N*cap rows
// of the receive buffer are skipped.
//
// The kernel is a pure HBM stream: each x row is read once and written R
// times.  One block handles one token at a time and is sized to the row:
// each thread moves two 16-byte vectors of it (every row starts on a
// 16-byte boundary because H*elem % 16 == 0), loads first, then the R
// stores.  Wide blocks with few vectors per thread kept the store stream
// closest to the write bandwidth (448 threads for a 14 KB row: about 7 %
// faster than 128 threads moving 7 vectors each).
//
// Reads and writes are separated in time: the kernel is scheduled while
// route and count (latency-bound, HBM nearly idle) still run, and its first
// blocks use that time to pull the x rows into L2 with bulk prefetches
// (evict-last) before they wait for count; the R-fold row stores carry an
// evict-first hint so that they do not push those rows out again.  The
// prefetch covers at most half of the L2.
//
// The decode-fused dispatch launches the same kernel in a second form that
// computes each pair's row itself from the per-block ranks and prefixes of
// the fused route kernel (PackDerive) and writes it to pos.
#include "fused_rows.cuh"
#include "mem_ops.cuh"
#include "moe_internal.cuh"
#include "pdl.cuh"

namespace moe {
namespace {

constexpr int kPackVecs = 2;          // 16-byte vectors of a row per thread
constexpr int kPackMaxThreads = 1024;

// Copies token g's row (and its fp8 scales) to the rows sp[0..R) (< 0:
// dropped); the block's threads each move two 16-byte vectors at a time,
// loads first, then the R stores.
__device__ __forceinline__ void copy_token(const uint4 *__restrict__ x, const float *__restrict__ x_scales,
                                           int64_t g, const int *sp, int R, int nvec, int spr,
                                           uint4 *__restrict__ packed_x, float *__restrict__ packed_scales,
                                           uint64_t stream_out) {
    const int tid = threadIdx.x, nthr = blockDim.x;
    bool any = false;  // a token whose pairs were all dropped is not read
    for (int k = 0; k < R; ++k) any |= sp[k] >= 0;
    const uint4 *src = x + g * nvec;
    for (int c0 = tid; any && c0 < nvec; c0 += nthr * kPackVecs) {
        uint4 v[kPackVecs];
#pragma unroll
        for (int u = 0; u < kPackVecs; ++u) {
            const int c = c0 + u * nthr;
            if (c < nvec) v[u] = ld_stream(src + c);
        }
        for (int k = 0; k < R; ++k) {
            const int p = sp[k];
            if (p < 0) continue;
            uint4 *dst = packed_x + (int64_t)p * nvec;
#pragma unroll
            for (int u = 0; u < kPackVecs; ++u) {
                const int c = c0 + u * nthr;
                if (c < nvec) st_evict_first(dst + c, v[u], stream_out);
            }
        }
    }
    if (spr > 0) {
        for (int i = tid; i < R * spr; i += nthr) {
            const int k = i / spr, j = i - k * spr;
            const int p = sp[k];
            if (p >= 0) packed_scales[(int64_t)p * spr + j] = __ldg(x_scales + g * spr + j);
        }
    }
}

// The pack kernel: pos[g][k] is the row of pair (g, k), written by the
// count kernel.  One token per block step.
__global__ void __launch_bounds__(kPackMaxThreads)
dispatch_pack_kernel(const uint4 *__restrict__ x, const float *__restrict__ x_scales,
                     const int32_t *__restrict__ pos, int64_t NT, int R, int nvec, int spr,
                     int64_t rows_total, int64_t pf_rows, int pf_blocks,
                     uint4 *__restrict__ packed_x, float *__restrict__ packed_scales,
                     int32_t *__restrict__ packed_src) {
    __shared__ int s_pos[32];
    const int tid = threadIdx.x;  // blockDim.x >= 32 >= R
    prefetch_rows_l2(x, (int64_t)nvec * 16, pf_rows, pf_blocks);  // before the wait: hints only
    grid_dependency_wait();  // pos comes from the count kernel (x may come from earlier ones)
    grid_launch_dependents();
    const uint64_t stream_out = l2_policy_evict_first();
    for (int64_t g = blockIdx.x; g < NT; g += gridDim.x) {
        if (tid < R) {
            const int p = __ldg(pos + g * R + tid);
            const bool ok = p >= 0 && (int64_t)p < rows_total;
            s_pos[tid] = ok ? p : -1;
            if (ok) packed_src[p] = (int32_t)(g * R + tid);
        }
        __syncthreads();
        copy_token(x, x_scales, g, s_pos, R, nvec, spr, packed_x, packed_scales, stream_out);
        __syncthreads();  // s_pos is rewritten for the next token
    }
}

// The deriving form (the decode-fused dispatch, see PackDerive): each pair's
// row is computed here and written to pos.  It takes two tokens per block
// step and derives the rows of both before copying either, so its extra
// dependent round trip to L2 is paid once per two tokens; held to 32
// registers, like the plain form, so that as many blocks share an SM.
__global__ void __launch_bounds__(kPackMaxThreads, 2)
dispatch_pack_derive_kernel(const uint4 *__restrict__ x, const float *__restrict__ x_scales,
                            int32_t *pos, int64_t NT, int R, int nvec, int spr,
                            int64_t rows_total, int64_t pf_rows, int pf_blocks, PackDerive D,
                            uint4 *__restrict__ packed_x, float *__restrict__ packed_scales,
                            int32_t *__restrict__ packed_src) {
    constexpr int kTok = 2;
    __shared__ int s_pos[kTok * 32];
    const int tid = threadIdx.x, nthr = blockDim.x;
    prefetch_rows_l2(x, (int64_t)nvec * 16, pf_rows, pf_blocks);  // before the wait: hints only
    grid_dependency_wait();  // ranks and prefixes come from the fused route kernel
    grid_launch_dependents();
    fused_send_counts(D);
    const uint64_t stream_out = l2_policy_evict_first();
    for (int64_t g0 = (int64_t)blockIdx.x * kTok; g0 < NT; g0 += (int64_t)gridDim.x * kTok) {
        for (int i = tid; i < kTok * R; i += nthr) {
            const int u = i / R, k = i - u * R;
            const int64_t g = g0 + u;
            int p = -1;
            if (g < NT) {
                p = fused_row(D, g, __ldg(D.topk_idx + g * R + k), pos[g * R + k]);
                pos[g * R + k] = p;
                if (p >= 0 && (int64_t)p < rows_total) packed_src[p] = (int32_t)(g * R + k);
                else p = -1;
            }
            s_pos[i] = p;
        }
        __syncthreads();
        for (int u = 0; u < kTok && g0 + u < NT; ++u)
            copy_token(x, x_scales, g0 + u, s_pos + u * R, R, nvec, spr, packed_x, packed_scales, stream_out);
        __syncthreads();  // s_pos is rewritten for the next tokens
    }
}

// Grid, block and prefetch shape shared by both forms.
template <bool kDerive>
cudaError_t launch_pack(const void *x, const float *x_scales, int32_t *pos, int64_t NT, int R,
                        int64_t row_bytes, int scales_per_row, int64_t rows_total, bool prefetch,
                        const PackDerive &D, void *packed_x, float *packed_scales,
                        int32_t *packed_src, cudaStream_t stream) {
    if (NT == 0) return cudaSuccess;
    const int nvec = (int)(row_bytes / 16);
    const int64_t steps = kDerive ? (NT + 1) / 2 : NT;  // the deriving form takes two tokens per step
    const int64_t grid = steps < (int64_t)0x7fffffff ? steps : (int64_t)0x7fffffff;
    // threads: two vectors of the row each, a whole number of warps (>= 32,
    // which also covers the R <= 32 position loads), at most 1024
    int64_t threads = ((nvec + kPackVecs - 1) / kPackVecs + 31) / 32 * 32;
    if (threads < 32) threads = 32;
    if (threads > kPackMaxThreads) threads = kPackMaxThreads;
    // prefetch: rows filling at most half the L2, issued by one block per SM
    // or, in the deriving form, by the blocks that fit beside the fused
    // route kernel (its blocks of 1024 threads fill the SMs they run on)
    int64_t pf_rows = prefetch ? pack_prefetch_rows(NT, row_bytes) : 0;
    int64_t pf_blocks = sm_count();
    if (kDerive && D.route_blocks < pf_blocks) {
        int64_t per_sm = 2048 / threads;
        if (per_sm > 32) per_sm = 32;
        pf_blocks = (pf_blocks - D.route_blocks) * per_sm;
    }
    if (pf_blocks > grid) pf_blocks = grid;
    if (pf_rows <= 0 || pf_blocks <= 0) pf_rows = pf_blocks = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if constexpr (kDerive)
        return cudaLaunchKernelEx(&cfg, dispatch_pack_derive_kernel, reinterpret_cast<const uint4 *>(x),
                                  x_scales, pos, NT, R, nvec, scales_per_row, rows_total, pf_rows,
                                  (int)pf_blocks, D, reinterpret_cast<uint4 *>(packed_x), packed_scales,
                                  packed_src);
    else
        return cudaLaunchKernelEx(&cfg, dispatch_pack_kernel, reinterpret_cast<const uint4 *>(x), x_scales,
                                  static_cast<const int32_t *>(pos), NT, R, nvec, scales_per_row, rows_total,
                                  pf_rows, (int)pf_blocks, reinterpret_cast<uint4 *>(packed_x),
                                  packed_scales, packed_src);
}

}  // namespace

int64_t pack_prefetch_rows(int64_t NT, int64_t row_bytes) {
    int64_t rows = row_bytes <= 65536 ? (l2_bytes() / 2) / row_bytes : 0;
    return rows < NT ? rows : NT;
}

cudaError_t launch_dispatch_pack(const void *x, const float *x_scales, const int32_t *pos,
                                 int64_t NT, int R, int64_t row_bytes, int scales_per_row,
                                 int64_t rows_total, void *packed_x,
                                 float *packed_scales, int32_t *packed_src, cudaStream_t stream) {
    // pos is only read in this form
    return launch_pack<false>(x, x_scales, const_cast<int32_t *>(pos), NT, R, row_bytes, scales_per_row,
                              rows_total, true, PackDerive{}, packed_x, packed_scales, packed_src, stream);
}

cudaError_t launch_dispatch_pack_derive(const void *x, const float *x_scales, int32_t *pos, int64_t NT,
                                        int R, int64_t row_bytes, int scales_per_row, int64_t rows_total,
                                        const PackDerive &D, void *packed_x, float *packed_scales,
                                        int32_t *packed_src, cudaStream_t stream) {
    return launch_pack<true>(x, x_scales, pos, NT, R, row_bytes, scales_per_row, rows_total, true, D,
                             packed_x, packed_scales, packed_src, stream);
}

}  // namespace moe
