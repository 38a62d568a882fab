// Dispatch pack with on-the-fly fp8 quantisation: bf16 token rows are
// quantised to e4m3 with one f32 scale per 128 elements while they are
// copied to their R receive rows.
//
// "Lower latency and higher throughput with multi-node DeepSeek
// deployment", section "Quantization": activations are quantised on the fly
// with one scaling factor per 128-element vector (the pages' kernel takes
// the per-128 maximum with cross-warp max reductions).  "Efficient and
// portable mixture-of-experts communication", section "Dispatch": the
// dispatched message carries the activations and their block scales.
//
// Per 128-element block: amax = max |x|, scale = fl32(amax / 448), code =
// e4m3 round-to-nearest-even saturating of fl32(x / scale) (all codes 0 and
// scale 0 when amax == 0).  A thread owns 8 consecutive elements (one
// 16-byte bf16 load), so 16 consecutive lanes own one block and reduce its
// amax with four butterfly shuffles.  Reading 2H bytes and writing
// R*(H + H/32) bytes instead of R*2H halves the write traffic of the bf16
// pack at R = 8.
#include <cuda_fp8.h>

#include "moe_internal.cuh"
#include "pdl.cuh"

namespace moe {
namespace {

constexpr int kQThreads = 128;
constexpr int kQVecs = 8;  // 16-byte bf16 vectors per thread in flight

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Two values -> two e4m3 codes (first value in the low byte).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

__global__ void __launch_bounds__(kQThreads)
dispatch_pack_quant_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ pos, int64_t NT,
                           int R, int nvec, int spr, int64_t rows_total,
                           uint2 *__restrict__ packed_q, float *__restrict__ packed_scales,
                           int32_t *__restrict__ packed_src) {
    __shared__ int s_pos[32];
    const int tid = threadIdx.x;
    grid_dependency_wait();  // pos comes from the count kernel
    grid_launch_dependents();
    for (int64_t g = blockIdx.x; g < NT; g += gridDim.x) {
        if (tid < R) {
            const int p = __ldg(pos + g * R + tid);
            const bool ok = p >= 0 && (int64_t)p < rows_total;
            s_pos[tid] = ok ? p : -1;
            if (ok) packed_src[p] = (int32_t)(g * R + tid);
        }
        __syncthreads();
        const uint4 *src = x + g * nvec;
        // The loop test uses the warp's first vector (c0 - lane), so every
        // lane of a warp runs the same iterations and takes part in the
        // full-warp shuffles below; lanes past the row contribute zeros.
        const int lane = tid & 31;
        for (int c0 = tid; c0 - lane < nvec; c0 += kQThreads * kQVecs) {
            uint4 v[kQVecs];
#pragma unroll
            for (int u = 0; u < kQVecs; ++u) {
                const int c = c0 + u * kQThreads;
                v[u] = (c < nvec) ? ld_stream(src + c) : make_uint4(0u, 0u, 0u, 0u);
            }
            uint2 q[kQVecs];
            float sc[kQVecs];
#pragma unroll
            for (int u = 0; u < kQVecs; ++u) {
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                float f[8];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    f[2 * i] = bf16_lo(w[i]);
                    f[2 * i + 1] = bf16_hi(w[i]);
                }
                float m = 0.f;
#pragma unroll
                for (int i = 0; i < 8; ++i) m = fmaxf(m, fabsf(f[i]));
                // the 16 lanes of this lane's half-warp hold one 128-element
                // block (nvec % 16 == 0, so all of them are in or out together)
#pragma unroll
                for (int off = 8; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                const float scale = __fdiv_rn(m, 448.0f);
                sc[u] = scale;
                uint32_t lo = 0u, hi = 0u;
                if (m != 0.f) {
                    lo = e4m3x2(__fdiv_rn(f[0], scale), __fdiv_rn(f[1], scale)) |
                         (e4m3x2(__fdiv_rn(f[2], scale), __fdiv_rn(f[3], scale)) << 16);
                    hi = e4m3x2(__fdiv_rn(f[4], scale), __fdiv_rn(f[5], scale)) |
                         (e4m3x2(__fdiv_rn(f[6], scale), __fdiv_rn(f[7], scale)) << 16);
                }
                q[u] = make_uint2(lo, hi);
            }
            for (int k = 0; k < R; ++k) {
                const int p = s_pos[k];
                if (p < 0) continue;
                uint2 *dst = packed_q + (int64_t)p * nvec;
                float *dsc = packed_scales + (int64_t)p * spr;
#pragma unroll
                for (int u = 0; u < kQVecs; ++u) {
                    const int c = c0 + u * kQThreads;
                    if (c < nvec) {
                        dst[c] = q[u];
                        if ((c & 15) == 0) dsc[c >> 4] = sc[u];
                    }
                }
            }
        }
        __syncthreads();  // s_pos is rewritten for the next token
    }
}

}  // namespace

cudaError_t launch_dispatch_pack_quant(const void *x, const int32_t *pos, int64_t NT, int R, int H,
                                       int64_t rows_total, void *packed_q, float *packed_scales,
                                       int32_t *packed_src, cudaStream_t stream) {
    if (NT == 0) return cudaSuccess;
    const int nvec = H / 8;  // 8 elements per 16-byte bf16 vector
    const int64_t grid = NT < (int64_t)0x7fffffff ? NT : (int64_t)0x7fffffff;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kQThreads);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dispatch_pack_quant_kernel, reinterpret_cast<const uint4 *>(x),
                              pos, NT, R, nvec, H / 128, rows_total,
                              reinterpret_cast<uint2 *>(packed_q), packed_scales, packed_src);
}

}  // namespace moe
