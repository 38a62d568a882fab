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
// Only pairs whose row lies in [row_lo, row_hi) are copied: all rank
// regions for the dispatch, one rank's region when a rank selects the
// tokens routed to its own experts from replicated inputs ("Hosting Qwen on
// Blackwell", section "Expert parallel").
//
// The kernel is a pure HBM stream: each x row is read once and written R
// times.  One block handles one token at a time; its threads move 16-byte
// vectors (every row starts on a 16-byte boundary because H*elem % 16 == 0),
// keeping all of their loads of a row in flight before issuing the R stores.
#include "moe_internal.cuh"
#include "pdl.cuh"

namespace moe {
namespace {

constexpr int kPackThreads = 128;
constexpr int kPackVecs = 8;  // 16-byte vectors per thread in flight

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__global__ void __launch_bounds__(kPackThreads)
dispatch_pack_kernel(const uint4 *__restrict__ x, const float *__restrict__ x_scales,
                     const int32_t *__restrict__ pos, int64_t NT, int R, int nvec, int spr,
                     int64_t row_lo, int64_t row_hi, uint4 *__restrict__ packed_x,
                     float *__restrict__ packed_scales, int32_t *__restrict__ packed_src) {
    __shared__ int s_pos[32];
    const int tid = threadIdx.x;
    // The first token's row is loaded before waiting for the previous kernel:
    // x is not produced by the count kernel (only pos is), and every kernel
    // of this library lets its dependents start only after its own inputs
    // are final, so the row is complete here.  This overlaps the row load
    // with the tail of the count kernel.
    const int64_t g_first = blockIdx.x;
    const bool preload = g_first < NT && nvec <= kPackThreads * kPackVecs;
    uint4 pre[kPackVecs];
    if (preload) {
#pragma unroll
        for (int u = 0; u < kPackVecs; ++u) {
            const int c = tid + u * kPackThreads;
            if (c < nvec) pre[u] = ld_stream(x + g_first * nvec + c);
        }
    }
    grid_dependency_wait();  // pos comes from the count kernel
    grid_launch_dependents();
    for (int64_t g = blockIdx.x; g < NT; g += gridDim.x) {
        if (tid < R) {
            const int p = __ldg(pos + g * R + tid);
            const bool ok = (int64_t)p >= row_lo && (int64_t)p < row_hi;
            s_pos[tid] = ok ? p : -1;
            if (ok) packed_src[p] = (int32_t)(g * R + tid);
        }
        __syncthreads();
        bool any = false;  // a token with no pair in the window is not read
        for (int k = 0; k < R; ++k) any |= s_pos[k] >= 0;
        const uint4 *src = x + g * nvec;
        for (int c0 = tid; any && c0 < nvec; c0 += kPackThreads * kPackVecs) {
            uint4 v[kPackVecs];
            if (preload && g == g_first) {
#pragma unroll
                for (int u = 0; u < kPackVecs; ++u) v[u] = pre[u];
            } else {
#pragma unroll
                for (int u = 0; u < kPackVecs; ++u) {
                    const int c = c0 + u * kPackThreads;
                    if (c < nvec) v[u] = ld_stream(src + c);
                }
            }
            for (int k = 0; k < R; ++k) {
                const int p = s_pos[k];
                if (p < 0) continue;
                uint4 *dst = packed_x + (int64_t)p * nvec;
#pragma unroll
                for (int u = 0; u < kPackVecs; ++u) {
                    const int c = c0 + u * kPackThreads;
                    if (c < nvec) dst[c] = v[u];
                }
            }
        }
        if (spr > 0) {
            for (int i = tid; i < R * spr; i += kPackThreads) {
                const int k = i / spr, j = i - k * spr;
                const int p = s_pos[k];
                if (p >= 0) packed_scales[(int64_t)p * spr + j] = __ldg(x_scales + g * spr + j);
            }
        }
        __syncthreads();  // s_pos is rewritten for the next token
    }
}

}  // namespace

cudaError_t launch_dispatch_pack(const void *x, const float *x_scales, const int32_t *pos,
                                 int64_t NT, int R, int64_t row_bytes, int scales_per_row,
                                 int64_t row_lo, int64_t row_hi, void *packed_x,
                                 float *packed_scales, int32_t *packed_src, cudaStream_t stream) {
    if (NT == 0) return cudaSuccess;
    const int nvec = (int)(row_bytes / 16);
    const int64_t grid = NT < (int64_t)0x7fffffff ? NT : (int64_t)0x7fffffff;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kPackThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dispatch_pack_kernel, reinterpret_cast<const uint4 *>(x),
                              x_scales, pos, NT, R, nvec, scales_per_row, row_lo, row_hi,
                              reinterpret_cast<uint4 *>(packed_x), packed_scales, packed_src);
}

}  // namespace moe
