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
// scale 0 when amax == 0).  A thread owns 16 consecutive elements (two
// 16-byte bf16 loads, one 16-byte store of codes per receive row), so 8
// consecutive lanes own one block and reduce its amax with three butterfly
// shuffles; each thread takes two such chunks per pass.  Reading 2H bytes and writing R*(H + H/32) bytes instead of
// R*2H halves the write traffic of the bf16 pack at R = 8.
//
// Memory schedule as in the bf16 pack: blocks sized to the row (two
// 16-element chunks per thread: 224 threads for H = 7168, which measured
// faster than one chunk per thread or than 8-byte code stores), the x rows
// prefetched into L2 while route and count run, the receive-row stores
// marked evict-first.
#include <cuda_fp8.h>

#include "fused_rows.cuh"
#include "mem_ops.cuh"
#include "moe_internal.cuh"
#include "pdl.cuh"

namespace moe {
namespace {

constexpr int kQMaxThreads = 1024;
constexpr int kQChunks = 2;  // 16-element chunks per thread per pass

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

// Two values -> two e4m3 codes (first value in the low byte).
__device__ __forceinline__ uint32_t e4m3x2(float a, float b) {
    return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
}

// Quantises token g's row and stores its codes and scales to the rows
// sp[0..R) (< 0: dropped).  The loop test uses the warp's first chunk
// (c - lane), so every lane of a warp runs the same iterations and takes
// part in the full-warp shuffles; lanes past the row contribute zeros.
__device__ __forceinline__ void quant_token(const uint4 *__restrict__ x, int64_t g, const int *sp, int R,
                                            int nchunk, int spr, uint4 *__restrict__ packed_q,
                                            float *__restrict__ packed_scales, uint64_t stream_out) {
    const int tid = threadIdx.x, nthr = blockDim.x, lane = tid & 31;
    const uint4 *src = x + g * (int64_t)nchunk * 2;
    for (int c0 = tid; c0 - lane < nchunk; c0 += nthr * kQChunks) {
        uint4 a[kQChunks], b[kQChunks];
#pragma unroll
        for (int u = 0; u < kQChunks; ++u) {
            const int c = c0 + u * nthr;
            const bool in = c < nchunk;
            a[u] = in ? ld_stream(src + 2 * c) : make_uint4(0u, 0u, 0u, 0u);
            b[u] = in ? ld_stream(src + 2 * c + 1) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kQChunks; ++u) {
            const int c = c0 + u * nthr;
            const uint32_t w[8] = {a[u].x, a[u].y, a[u].z, a[u].w, b[u].x, b[u].y, b[u].z, b[u].w};
            float f[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                f[2 * i] = bf16_lo(w[i]);
                f[2 * i + 1] = bf16_hi(w[i]);
            }
            float m = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(f[i]));
            // the 8 lanes of this lane's group hold one 128-element block
            // (nchunk % 8 == 0 and nthr % 32 == 0, so groups never straddle)
#pragma unroll
            for (int off = 4; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
            const float scale = __fdiv_rn(m, 448.0f);
            uint32_t q[4] = {0u, 0u, 0u, 0u};
            if (m != 0.f) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    q[i] = e4m3x2(__fdiv_rn(f[4 * i], scale), __fdiv_rn(f[4 * i + 1], scale)) |
                           (e4m3x2(__fdiv_rn(f[4 * i + 2], scale), __fdiv_rn(f[4 * i + 3], scale)) << 16);
            }
            const uint4 codes = make_uint4(q[0], q[1], q[2], q[3]);
            if (c < nchunk) {
                for (int k = 0; k < R; ++k) {
                    const int p = sp[k];
                    if (p < 0) continue;
                    st_evict_first(packed_q + (int64_t)p * nchunk + c, codes, stream_out);
                    if ((c & 7) == 0) packed_scales[(int64_t)p * spr + (c >> 3)] = scale;
                }
            }
        }
    }
}

// pos[g][k] = the row of pair (g, k), written by the count kernel.
__global__ void __launch_bounds__(kQMaxThreads)
dispatch_pack_quant_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ pos, int64_t NT,
                           int R, int nchunk, int spr, int64_t rows_total, int64_t pf_rows,
                           int pf_blocks, uint4 *__restrict__ packed_q,
                           float *__restrict__ packed_scales, int32_t *__restrict__ packed_src) {
    __shared__ int s_pos[32];
    const int tid = threadIdx.x;  // blockDim.x: whole warps, >= 32 >= R
    prefetch_rows_l2(x, (int64_t)nchunk * 32, pf_rows, pf_blocks);  // before the wait: hints only
    grid_dependency_wait();  // pos comes from the count kernel
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
        quant_token(x, g, s_pos, R, nchunk, spr, packed_q, packed_scales, stream_out);
        __syncthreads();  // s_pos is rewritten for the next token
    }
}

// The decode-fused dispatch's form: each pair's row is derived here from the
// fused route kernel's ranks and prefixes (fused_rows.cuh) and written to
// pos, then the token is quantised and stored as above.
__global__ void __launch_bounds__(kQMaxThreads)
dispatch_pack_quant_derive_kernel(const uint4 *__restrict__ x, int32_t *pos, int64_t NT, int R,
                                  int nchunk, int spr, int64_t rows_total, int64_t pf_rows,
                                  int pf_blocks, PackDerive D, uint4 *__restrict__ packed_q,
                                  float *__restrict__ packed_scales, int32_t *__restrict__ packed_src) {
    __shared__ int s_pos[32];
    const int tid = threadIdx.x;  // blockDim.x: whole warps, >= 32 >= R
    prefetch_rows_l2(x, (int64_t)nchunk * 32, pf_rows, pf_blocks);  // before the wait: hints only
    grid_dependency_wait();  // ranks and prefixes come from the fused route kernel
    grid_launch_dependents();
    fused_send_counts(D);
    const uint64_t stream_out = l2_policy_evict_first();
    for (int64_t g = blockIdx.x; g < NT; g += gridDim.x) {
        if (tid < R) {
            int p = fused_row(D, g, __ldg(D.topk_idx + g * R + tid), pos[g * R + tid]);
            pos[g * R + tid] = p;
            if (p >= 0 && (int64_t)p < rows_total) packed_src[p] = (int32_t)(g * R + tid);
            else p = -1;
            s_pos[tid] = p;
        }
        __syncthreads();
        quant_token(x, g, s_pos, R, nchunk, spr, packed_q, packed_scales, stream_out);
        __syncthreads();  // s_pos is rewritten for the next token
    }
}

}  // namespace

namespace {
template <bool kDerive>
cudaError_t launch_quant(const void *x, int32_t *pos, int64_t NT, int R, int H, int64_t rows_total,
                         const PackDerive &D, void *packed_q, float *packed_scales, int32_t *packed_src,
                         cudaStream_t stream) {
    if (NT == 0) return cudaSuccess;
    const int nchunk = H / 16;  // 16 elements: 32 bytes of bf16 in, 16 codes out
    const int64_t grid = NT < (int64_t)0x7fffffff ? NT : (int64_t)0x7fffffff;
    int64_t threads = ((nchunk + kQChunks - 1) / kQChunks + 31) / 32 * 32;
    if (threads > kQMaxThreads) threads = kQMaxThreads;
    // x rows prefetched into L2 (at most half of it), one issuing block per
    // SM or, in the fused form, by the blocks that fit beside the fused
    // route kernel (its blocks of 1024 threads fill the SMs they run on)
    const int64_t row_bytes = (int64_t)H * 2;
    int64_t pf_rows = row_bytes <= 65536 ? (l2_bytes() / 2) / row_bytes : 0;
    if (pf_rows > NT) pf_rows = NT;
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
        return cudaLaunchKernelEx(&cfg, dispatch_pack_quant_derive_kernel, reinterpret_cast<const uint4 *>(x),
                                  pos, NT, R, nchunk, H / 128, rows_total, pf_rows, (int)pf_blocks, D,
                                  reinterpret_cast<uint4 *>(packed_q), packed_scales, packed_src);
    else
        return cudaLaunchKernelEx(&cfg, dispatch_pack_quant_kernel, reinterpret_cast<const uint4 *>(x),
                                  static_cast<const int32_t *>(pos), NT, R, nchunk, H / 128, rows_total,
                                  pf_rows, (int)pf_blocks, reinterpret_cast<uint4 *>(packed_q),
                                  packed_scales, packed_src);
}
}  // namespace

cudaError_t launch_dispatch_pack_quant(const void *x, const int32_t *pos, int64_t NT, int R, int H,
                                       int64_t rows_total, void *packed_q, float *packed_scales,
                                       int32_t *packed_src, cudaStream_t stream) {
    // pos is only read in this form
    return launch_quant<false>(x, const_cast<int32_t *>(pos), NT, R, H, rows_total, PackDerive{}, packed_q,
                               packed_scales, packed_src, stream);
}

cudaError_t launch_dispatch_pack_quant_derive(const void *x, int32_t *pos, int64_t NT, int R, int H,
                                              int64_t rows_total, const PackDerive &D, void *packed_q,
                                              float *packed_scales, int32_t *packed_src, cudaStream_t stream) {
    return launch_quant<true>(x, pos, NT, R, H, rows_total, D, packed_q, packed_scales, packed_src, stream);
}

}  // namespace moe
