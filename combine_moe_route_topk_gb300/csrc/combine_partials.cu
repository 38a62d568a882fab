// Combine with send-side accumulation: the rows a token sent to one rank
// are first reduced into one partial row (what that rank sends back), and
// the token's output is the sum of its at most min(R, N) partial rows.
//
// "Enabling trillion-parameter models on AWS EFA", section "Evaluation":
// accumulating on the send side (as DeepEP does) reduces the data moved
// back, at some cost in accuracy, compared with accumulating every expert
// row on the receiving side.  Here every "rank" is a region of one GPU, so
// the partial rows are the data a rank would send back; they are stored in
// y's 16-bit type (rounded once from the f32 sum), which is the accuracy
// cost the pages mention.
//
// Partial slots: the distinct ranks of token g, in the order of their first
// pair k, get slots 0, 1, ...; partial[g][j] holds slot j's row and
// slot_rank[g][j] its rank (-1 and a zero row for unused slots).  The values
// equal those of a rank-side pass over each rank's received rows grouped by
// source token; computing them per token keeps all R row loads of a token
// in flight at once, as in the plain combine.
#include <cuda_bf16.h>

#include "mem_ops.cuh"
#include "moe_internal.cuh"
#include "pdl.cuh"

namespace moe {
namespace {

constexpr int kThreads = 128;
constexpr int kU = 1;   // output vectors per thread per pass
constexpr int kKB = 8;  // source rows loaded together

template <int kBf16>
struct Vec;

template <>
struct Vec<1> {  // 8 x bf16
    static constexpr int kElems = 8;
    __device__ static void fma(float (&a)[8], float w, const uint4 &v) {
        const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            a[2 * i] = fmaf(w, __uint_as_float(u[i] << 16), a[2 * i]);
            a[2 * i + 1] = fmaf(w, __uint_as_float(u[i] & 0xffff0000u), a[2 * i + 1]);
        }
    }
    __device__ static void add(float (&a)[8], const uint4 &v) { fma(a, 1.0f, v); }
    __device__ static uint4 pack(const float (&a)[8]) {
        uint32_t u[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(a[2 * i], a[2 * i + 1]);
            u[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
        return make_uint4(u[0], u[1], u[2], u[3]);
    }
};

template <>
struct Vec<0> {  // 4 x f32
    static constexpr int kElems = 4;
    __device__ static void fma(float (&a)[4], float w, const uint4 &v) {
        a[0] = fmaf(w, __uint_as_float(v.x), a[0]);
        a[1] = fmaf(w, __uint_as_float(v.y), a[1]);
        a[2] = fmaf(w, __uint_as_float(v.z), a[2]);
        a[3] = fmaf(w, __uint_as_float(v.w), a[3]);
    }
    __device__ static void add(float (&a)[4], const uint4 &v) {
        a[0] += __uint_as_float(v.x);
        a[1] += __uint_as_float(v.y);
        a[2] += __uint_as_float(v.z);
        a[3] += __uint_as_float(v.w);
    }
    __device__ static uint4 pack(const float (&a)[4]) {
        return make_uint4(__float_as_uint(a[0]), __float_as_uint(a[1]), __float_as_uint(a[2]),
                          __float_as_uint(a[3]));
    }
};

template <int kBf16>
__global__ void __launch_bounds__(kThreads)
combine_partials_kernel(const uint4 *__restrict__ y, const int32_t *__restrict__ pos,
                        const float *__restrict__ topk_w, int64_t NT, int R, int nvec, int64_t cap,
                        int64_t rows_total, int P, uint4 *__restrict__ partial,
                        int32_t *__restrict__ slot_rank) {
    using V = Vec<kBf16>;
    constexpr int EL = V::kElems;
    __shared__ int s_pos[32], s_slot[32];
    __shared__ float s_w[32];
    __shared__ int s_nslot;
    const int tid = threadIdx.x;
    grid_dependency_wait();  // y, pos and topk_w come from earlier kernels
    grid_launch_dependents();
    for (int64_t g = blockIdx.x; g < NT; g += gridDim.x) {
        if (tid < R) {
            int p = __ldg(pos + g * R + tid);
            s_pos[tid] = (p >= 0 && (int64_t)p < rows_total) ? p : -1;
            s_w[tid] = __ldg(topk_w + g * R + tid);
        }
        __syncthreads();
        if (tid == 0) {
            // slots: the token's distinct ranks in the order of their first pair
            int ranks[32];
            int nslot = 0;
            for (int k = 0; k < R; ++k) {
                const int p = s_pos[k];
                if (p < 0) {
                    s_slot[k] = -1;
                    continue;
                }
                const int d = (int)((int64_t)p / cap);
                int j = 0;
                while (j < nslot && ranks[j] != d) ++j;
                if (j == nslot && nslot < P) ranks[nslot++] = d;
                s_slot[k] = (j < nslot) ? j : -1;
            }
            for (int j = 0; j < P; ++j) slot_rank[g * P + j] = (j < nslot) ? ranks[j] : -1;
            s_nslot = nslot;
        }
        __syncthreads();
        const int nslot = s_nslot;
        for (int c0 = tid; c0 < nvec; c0 += kThreads * kU) {
            // R <= 8: every row of the token is loaded once, up front
            uint4 v[kKB][kU];
            if (R <= kKB) {
#pragma unroll
                for (int kk = 0; kk < kKB; ++kk) {
                    const int p = (kk < R) ? s_pos[kk] : -1;
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const int c = c0 + u * kThreads;
                        v[kk][u] = (p >= 0 && c < nvec) ? ld_stream(y + (int64_t)p * nvec + c)
                                                        : make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            for (int j = 0; j < P; ++j) {
                float acc[kU][EL];
#pragma unroll
                for (int u = 0; u < kU; ++u)
#pragma unroll
                    for (int i = 0; i < EL; ++i) acc[u][i] = 0.f;
                if (j < nslot) {
                    if (R <= kKB) {
#pragma unroll
                        for (int kk = 0; kk < kKB; ++kk) {
                            if (kk < R && s_slot[kk] == j) {
                                const float w = s_w[kk];
#pragma unroll
                                for (int u = 0; u < kU; ++u) V::fma(acc[u], w, v[kk][u]);
                            }
                        }
                    } else {
                        // R > 8: the rows of one slot at a time
                        for (int k = 0; k < R; ++k) {
                            if (s_slot[k] != j) continue;
                            const int p = s_pos[k];
                            const float w = s_w[k];
#pragma unroll
                            for (int u = 0; u < kU; ++u) {
                                const int c = c0 + u * kThreads;
                                if (c < nvec) V::fma(acc[u], w, ld_stream(y + (int64_t)p * nvec + c));
                            }
                        }
                    }
                }
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int c = c0 + u * kThreads;
                    if (c < nvec) partial[(g * P + j) * nvec + c] = V::pack(acc[u]);
                }
            }
        }
        __syncthreads();
    }
}

template <int kBf16>
__global__ void __launch_bounds__(kThreads)
reduce_partials_kernel(const uint4 *__restrict__ partial, const int32_t *__restrict__ slot_rank,
                       int64_t NT, int P, int nvec, uint4 *__restrict__ out) {
    using V = Vec<kBf16>;
    constexpr int EL = V::kElems;
    __shared__ int s_used[32];
    const int tid = threadIdx.x;
    grid_dependency_wait();  // partial rows come from the previous kernel
    grid_launch_dependents();
    for (int64_t g = blockIdx.x; g < NT; g += gridDim.x) {
        if (tid < P) s_used[tid] = __ldg(slot_rank + g * P + tid) >= 0;
        __syncthreads();
        for (int c0 = tid; c0 < nvec; c0 += kThreads * kU) {
            float acc[kU][EL];
#pragma unroll
            for (int u = 0; u < kU; ++u)
#pragma unroll
                for (int i = 0; i < EL; ++i) acc[u][i] = 0.f;
            for (int j = 0; j < P; ++j) {
                if (!s_used[j]) continue;
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int c = c0 + u * kThreads;
                    if (c < nvec) V::add(acc[u], ld_stream(partial + (g * P + j) * nvec + c));
                }
            }
#pragma unroll
            for (int u = 0; u < kU; ++u) {
                const int c = c0 + u * kThreads;
                if (c < nvec) out[g * nvec + c] = V::pack(acc[u]);
            }
        }
        __syncthreads();
    }
}

cudaLaunchConfig_t grid_cfg(int64_t NT, cudaStream_t stream, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(NT < (int64_t)0x7fffffff ? NT : (int64_t)0x7fffffff));
    cfg.blockDim = dim3(kThreads);
    cfg.stream = stream;
    attr[0] = pdl_attribute();
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

}  // namespace

cudaError_t launch_combine_partials(const void *y, int y_dtype, const int32_t *pos,
                                    const float *topk_w, int64_t NT, int R, int H, int64_t cap,
                                    int64_t rows_total, int P, void *partial, int32_t *slot_rank,
                                    cudaStream_t stream) {
    if (NT == 0) return cudaSuccess;
    const int nvec = (int)((int64_t)H * (y_dtype == MOE_BF16 ? 2 : 4) / 16);
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = grid_cfg(NT, stream, attr);
    auto kern = (y_dtype == MOE_BF16) ? combine_partials_kernel<1> : combine_partials_kernel<0>;
    return cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const uint4 *>(y), pos, topk_w, NT, R,
                              nvec, cap, rows_total, P, reinterpret_cast<uint4 *>(partial),
                              slot_rank);
}

cudaError_t launch_reduce_partials(const void *partial, int y_dtype, const int32_t *slot_rank,
                                   int64_t NT, int P, int H, void *out, cudaStream_t stream) {
    if (NT == 0) return cudaSuccess;
    const int nvec = (int)((int64_t)H * (y_dtype == MOE_BF16 ? 2 : 4) / 16);
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = grid_cfg(NT, stream, attr);
    auto kern = (y_dtype == MOE_BF16) ? reduce_partials_kernel<1> : reduce_partials_kernel<0>;
    return cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const uint4 *>(partial), slot_rank, NT,
                              P, nvec, reinterpret_cast<uint4 *>(out));
}

}  // namespace moe
