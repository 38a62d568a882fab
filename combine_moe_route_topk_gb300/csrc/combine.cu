// Combine: out[g] = sum_k topk_w[g][k] * y[pos[g][k]], f32 accumulation.
//
// "Efficient and portable mixture-of-experts communication", section
// "Combine": each token reads its experts' outputs through the routing table
// (which buffer, which weight) and forms their router-weighted average.
// "Enabling trillion-parameter models on AWS EFA", section "Evaluation":
// accumulation happens on the receiving side only, R rows per token.
//
// Pairs whose row is negative (dropped by count) or outside the N*cap rows
// of the receive buffer contribute nothing.
//
// HBM stream: R rows gathered per token, one row written.  One block per
// token at a time; every thread owns 16-byte output vectors and issues the
// loads of all R source rows (up to 8 at once) before accumulating them in
// k order, so each thread keeps 8 x 2 x 16 bytes in flight.
#include "mem_ops.cuh"
#include "moe_internal.cuh"
#include "pdl.cuh"
#include "vec_traits.cuh"

namespace moe {
namespace {

constexpr int kCombThreads = 128;
constexpr int kCombU = 2;   // output vectors per thread per pass
constexpr int kCombKB = 8;  // source rows loaded together

template <int kBf16>
__global__ void __launch_bounds__(kCombThreads)
combine_kernel(const uint4 *__restrict__ y, const int32_t *__restrict__ pos,
               const float *__restrict__ topk_w, int64_t NT, int R, int nvec, int64_t rows_total,
               uint4 *__restrict__ out) {
    using VT = Vec<kBf16>;
    constexpr int EL = VT::kElems;
    __shared__ int s_pos[32];
    __shared__ float s_w[32];
    const int tid = threadIdx.x;
    grid_dependency_wait();  // y, pos and topk_w come from earlier kernels
    grid_launch_dependents();
    for (int64_t g = blockIdx.x; g < NT; g += gridDim.x) {
        if (tid < R) {
            const int p = __ldg(pos + g * R + tid);
            s_pos[tid] = (p >= 0 && (int64_t)p < rows_total) ? p : -1;
            s_w[tid] = __ldg(topk_w + g * R + tid);
        }
        __syncthreads();
        for (int c0 = tid; c0 < nvec; c0 += kCombThreads * kCombU) {
            float acc[kCombU][EL];
#pragma unroll
            for (int u = 0; u < kCombU; ++u)
#pragma unroll
                for (int i = 0; i < EL; ++i) acc[u][i] = 0.f;
            for (int k0 = 0; k0 < R; k0 += kCombKB) {
                uint4 v[kCombKB][kCombU];
#pragma unroll
                for (int kk = 0; kk < kCombKB; ++kk) {
                    const int k = k0 + kk;
                    const int p = (k < R) ? s_pos[k] : -1;
#pragma unroll
                    for (int u = 0; u < kCombU; ++u) {
                        const int c = c0 + u * kCombThreads;
                        if (p >= 0 && c < nvec) v[kk][u] = ld_stream(y + (int64_t)p * nvec + c);
                        else v[kk][u] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
#pragma unroll
                for (int kk = 0; kk < kCombKB; ++kk) {
                    const int k = k0 + kk;
                    if (k < R && s_pos[k] >= 0) {
                        const float w = s_w[k];
#pragma unroll
                        for (int u = 0; u < kCombU; ++u) VT::fma(acc[u], w, v[kk][u]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kCombU; ++u) {
                const int c = c0 + u * kCombThreads;
                if (c < nvec) out[g * nvec + c] = VT::pack(acc[u]);
            }
        }
        __syncthreads();
    }
}

}  // namespace

cudaError_t launch_combine(const void *y, int y_dtype, const int32_t *pos, const float *topk_w,
                           int64_t NT, int R, int H, int64_t rows_total, void *out,
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
    auto kern = (y_dtype == MOE_BF16) ? combine_kernel<1> : combine_kernel<0>;
    return cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const uint4 *>(y), pos, topk_w, NT, R,
                              nvec, rows_total, reinterpret_cast<uint4 *>(out));
}

}  // namespace moe
