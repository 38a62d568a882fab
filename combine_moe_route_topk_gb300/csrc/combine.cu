// Combine: out[g] = sum_k topk_w[g][k] * y[pos[g][k]], f32 accumulation;
// and its expert-parallel local form, the same sum over only the pairs whose
// row lies in one rank's receive region.
//
// "Efficient and portable mixture-of-experts communication", section
// "Combine": each token reads its experts' outputs through the routing table
// (which buffer, which weight) and forms their router-weighted average.
// "Enabling trillion-parameter models on AWS EFA", section "Evaluation":
// accumulation happens on the receiving side only, R rows per token.
// "Hosting Qwen on Blackwell", section "Expert parallel": with replicated
// inputs a rank accumulates its own experts' outputs for every token before
// an all-reduce (out_d[g] = 0 for a token with no pair on rank d).
//
// Both are one kernel over a row window [row_lo, row_hi): the whole receive
// buffer [0, N*cap) for the combine (which also drops pairs whose row is
// negative, i.e. dropped by count, or out of range), rank d's region
// [d*cap, (d+1)*cap) for the local sum.  Summed over all ranks the local
// sums give the combine up to rounding.
//
// HBM stream: a token's rows gathered, one row written.  One block of 128
// threads per token (grid = N*T, the hardware schedules them): warp 0 loads
// the R positions and weights, keeps the pairs inside the window in k order
// (ballot compaction into shared memory); then every thread owns two
// 16-byte output vectors per pass and loads up to four of the token's rows
// for both at once before the FMAs, accumulating in f32 in k order.  The
// kernel is held to 64 registers so that 8 blocks (1024 threads) share an
// SM: each SM keeps the rows of 8 tokens in flight, which a gather of a
// variable number of rows per token needs in order to stream at HBM rate
// when a token has few rows in the window.  Measured on GB300 (events, L2
// flushed first), against the previous kernels (8 tokens per block with a
// flattened (token, vector) split for the local sum; 16 loads in flight per
// thread at 103 registers for the combine): local sum of rank 0 on the
// Qwen3-235B-shaped prefill batch (32,602 rows of 16,384 tokens) 71.6 ->
// 63.9 us, on the skewed batch (74,454 rows) 232 -> 189 us, on the
// DeepSeek-V3 decode batch 19.1 -> 17.2 us; whole combine 173.6 -> 170.9 us
// (Qwen3), 77.8 -> 77.2 us (DeepSeek-V3), 305.7 -> 302.6 us (skewed).
// Variants that were slower: rows staged in shared memory by bulk copies
// from one producer warp per SM (Qwen3 local sum 124 us), a persistent grid
// prefetching the next token's positions (64-74 us), 256-thread blocks,
// four output vectors per thread, 10 or 12 blocks per SM at fewer
// registers (spills).
#include "mem_ops.cuh"
#include "moe_internal.cuh"
#include "pdl.cuh"
#include "vec_traits.cuh"

namespace moe {
namespace {

constexpr int kCombThreads = 128;
constexpr int kCombU = 2;        // output vectors per thread per pass
constexpr int kCombKB = 4;       // rows loaded together
constexpr int kCombMinBlocks = 8;  // blocks per SM: caps the kernel at 64 registers

template <int kBf16>
__global__ void __launch_bounds__(kCombThreads, kCombMinBlocks)
combine_window_kernel(const uint4 *__restrict__ y, const int32_t *__restrict__ pos,
                      const float *__restrict__ topk_w, int64_t NT, int R, int nvec, int64_t row_lo,
                      int64_t row_hi, uint4 *__restrict__ out) {
    using VT = Vec<kBf16>;
    constexpr int EL = VT::kElems;
    __shared__ int s_p[32];    // rows of the token's pairs inside the window, in k order
    __shared__ float s_w[32];  // their weights
    __shared__ int s_n;
    const int tid = threadIdx.x;
    grid_dependency_wait();  // y, pos and topk_w come from earlier kernels
    grid_launch_dependents();
    for (int64_t g = blockIdx.x; g < NT; g += gridDim.x) {
        if (tid < 32) {
            const int p = tid < R ? __ldg(pos + g * R + tid) : -1;
            const float w = tid < R ? __ldg(topk_w + g * R + tid) : 0.f;
            const bool in = tid < R && (int64_t)p >= row_lo && (int64_t)p < row_hi;
            const unsigned m = __ballot_sync(0xffffffffu, in);
            if (in) {
                const int j = __popc(m & ((1u << tid) - 1u));
                s_p[j] = p;
                s_w[j] = w;
            }
            if (tid == 0) s_n = __popc(m);
        }
        __syncthreads();
        const int n = s_n;
        for (int c0 = tid; c0 < nvec; c0 += kCombThreads * kCombU) {
            float acc[kCombU][EL];
#pragma unroll
            for (int u = 0; u < kCombU; ++u)
#pragma unroll
                for (int i = 0; i < EL; ++i) acc[u][i] = 0.f;
            for (int j0 = 0; j0 < n; j0 += kCombKB) {
                uint4 v[kCombKB][kCombU];
#pragma unroll
                for (int jj = 0; jj < kCombKB; ++jj)
#pragma unroll
                    for (int u = 0; u < kCombU; ++u) {
                        const int c = c0 + u * kCombThreads;
                        v[jj][u] = (j0 + jj < n && c < nvec) ? ld_stream(y + (int64_t)s_p[j0 + jj] * nvec + c)
                                                             : make_uint4(0u, 0u, 0u, 0u);
                    }
#pragma unroll
                for (int jj = 0; jj < kCombKB; ++jj) {
                    if (j0 + jj < n) {
                        const float w = s_w[j0 + jj];
#pragma unroll
                        for (int u = 0; u < kCombU; ++u) VT::fma(acc[u], w, v[jj][u]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kCombU; ++u) {
                const int c = c0 + u * kCombThreads;
                if (c < nvec) out[g * nvec + c] = VT::pack(acc[u]);
            }
        }
        __syncthreads();  // s_p, s_w and s_n are rewritten for the next token
    }
}

cudaError_t launch_window(const void *y, int y_dtype, const int32_t *pos, const float *topk_w,
                          int64_t NT, int R, int H, int64_t row_lo, int64_t row_hi, void *out,
                          cudaStream_t stream) {
    if (NT == 0) return cudaSuccess;
    const int elem = (y_dtype == MOE_BF16) ? 2 : 4;
    const int nvec = (int)((int64_t)H * elem / 16);
    const int64_t grid = NT < (int64_t)0x7fffffff ? NT : (int64_t)0x7fffffff;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kCombThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    auto kern = (y_dtype == MOE_BF16) ? combine_window_kernel<1> : combine_window_kernel<0>;
    return cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const uint4 *>(y), pos, topk_w, NT, R,
                              nvec, row_lo, row_hi, reinterpret_cast<uint4 *>(out));
}

}  // namespace

cudaError_t launch_combine(const void *y, int y_dtype, const int32_t *pos, const float *topk_w,
                           int64_t NT, int R, int H, int64_t rows_total, void *out,
                           cudaStream_t stream) {
    return launch_window(y, y_dtype, pos, topk_w, NT, R, H, 0, rows_total, out, stream);
}

cudaError_t launch_combine_rank(const void *y, int y_dtype, const int32_t *pos, const float *topk_w,
                                int64_t NT, int R, int H, int64_t row_lo, int64_t row_hi, void *out,
                                cudaStream_t stream) {
    return launch_window(y, y_dtype, pos, topk_w, NT, R, H, row_lo, row_hi, out, stream);
}

}  // namespace moe
