// Expert-parallel local path of one rank: with replicated inputs, a rank
// selects the tokens routed to its own experts, runs them, and accumulates
// their outputs locally before an all-reduce ("Hosting Qwen on Blackwell",
// section "Expert parallel").  Here:
//   pack_rank    copies x[g] to every receive row pos[g][k] inside rank d's
//                region [d*cap, (d+1)*cap) (and sets packed_src there);
//   combine_rank out[g] = sum, in k order, of w[g][k] * y[pos[g][k]] over
//                the pairs of g inside that region; 0 for the other tokens.
//
// Only some tokens have a pair on a given rank (DeepSeek-V3 decode: about a
// quarter), so a block takes 8 tokens at once: lanes of warp 0 read their
// positions, one lane per token and eight positions per batch of loads,
// and list the pairs that fall in the region; the block then works through
// the listed rows only.  Every thread owns vectors of the flattened (row,
// vector) space and keeps several of them in flight.  One block per token,
// as in the whole-batch kernels, would leave most blocks with nothing to do
// but a position load.
#include "mem_ops.cuh"
#include "moe_internal.cuh"
#include "pdl.cuh"
#include "vec_traits.cuh"

namespace moe {
namespace {

constexpr int kLThreads = 256;
constexpr int kLTok = 8;   // tokens per block (one lane of warp 0 each)
constexpr int kLU = 8;     // vectors per thread in flight (pack)
constexpr int kLCU = 4;    // output vectors per thread in flight (combine)
constexpr int kLKB = 2;    // rows of one token loaded together (combine)
constexpr int kLPB = 8;    // positions of one token loaded together

__device__ __forceinline__ bool in_window(int p, int64_t lo, int64_t hi) {
    return (int64_t)p >= lo && (int64_t)p < hi;
}

// The pairs of token g that fall in [lo, hi): f(k, p) for each, in k order.
// Positions are loaded kLPB at a time, so their latencies overlap.
template <typename F>
__device__ __forceinline__ void for_pairs_in_window(const int32_t *__restrict__ pos, int64_t g, int R,
                                                    int64_t lo, int64_t hi, F &&f) {
    for (int k0 = 0; k0 < R; k0 += kLPB) {
        int pv[kLPB];
#pragma unroll
        for (int j = 0; j < kLPB; ++j) pv[j] = (k0 + j < R) ? __ldg(pos + g * R + k0 + j) : -1;
#pragma unroll
        for (int j = 0; j < kLPB; ++j)
            if (k0 + j < R && in_window(pv[j], lo, hi)) f(k0 + j, pv[j]);
    }
}

__device__ __forceinline__ int warp_exclusive_scan(int x, int lane) {
    int incl = x;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += t;
    }
    return incl - x;
}

__global__ void __launch_bounds__(kLThreads)
pack_rank_kernel(const uint4 *__restrict__ x, const float *__restrict__ x_scales,
                 const int32_t *__restrict__ pos, int64_t NT, int R, int nvec, int spr,
                 FastDiv div_nvec, int64_t row_lo, int64_t row_hi, uint4 *__restrict__ packed_x,
                 float *__restrict__ packed_scales, int32_t *__restrict__ packed_src) {
    __shared__ int s_g[kLTok * 32], s_p[kLTok * 32];  // listed pairs (R <= 32)
    __shared__ int s_n;
    const int tid = threadIdx.x, lane = tid & 31;
    const int64_t g0 = (int64_t)blockIdx.x * kLTok;
    grid_dependency_wait();  // pos comes from the count kernel
    grid_launch_dependents();
    if (tid < 32) {
        const int64_t g = g0 + lane;
        const bool mine = lane < kLTok && g < NT;
        int cnt = 0;
        if (mine) for_pairs_in_window(pos, g, R, row_lo, row_hi, [&](int, int) { ++cnt; });
        int at = warp_exclusive_scan(cnt, lane);
        if (lane == 31) s_n = at + cnt;
        if (mine)
            for_pairs_in_window(pos, g, R, row_lo, row_hi, [&](int k, int p) {
                s_g[at] = (int)g;
                s_p[at] = p;
                packed_src[p] = (int32_t)(g * R + k);
                ++at;
            });
    }
    __syncthreads();
    const int n = s_n;
    const int total = n * nvec;  // < 2^31: checked by the launcher
    for (int i0 = tid; i0 < total; i0 += kLThreads * kLU) {
        uint4 v[kLU];
        int64_t dst[kLU];
#pragma unroll
        for (int u = 0; u < kLU; ++u) {
            const int i = i0 + u * kLThreads;
            dst[u] = -1;
            if (i < total) {
                const int e = (int)fast_div((uint32_t)i, div_nvec);
                const int c = i - e * nvec;
                v[u] = ld_stream(x + (int64_t)s_g[e] * nvec + c);
                dst[u] = (int64_t)s_p[e] * nvec + c;
            }
        }
#pragma unroll
        for (int u = 0; u < kLU; ++u)
            if (dst[u] >= 0) packed_x[dst[u]] = v[u];
    }
    if (spr > 0)
        for (int i = tid; i < n * spr; i += kLThreads) {
            const int e = i / spr, j = i - (i / spr) * spr;
            packed_scales[(int64_t)s_p[e] * spr + j] = __ldg(x_scales + (int64_t)s_g[e] * spr + j);
        }
}

template <int kBf16>
__global__ void __launch_bounds__(kLThreads)
combine_rank_kernel(const uint4 *__restrict__ y, const int32_t *__restrict__ pos,
                    const float *__restrict__ topk_w, int64_t NT, int R, int nvec,
                    FastDiv div_nvec, int64_t row_lo, int64_t row_hi, uint4 *__restrict__ out) {
    using V = Vec<kBf16>;
    constexpr int EL = V::kElems;
    __shared__ int s_p[kLTok][32];  // per token: its pairs in the region, in k order
    __shared__ float s_w[kLTok][32];
    __shared__ int s_cnt[kLTok];
    __shared__ int s_tok[kLTok];    // tokens with pairs first, then the others
    __shared__ int s_nnz;
    const int tid = threadIdx.x, lane = tid & 31;
    const int64_t g0 = (int64_t)blockIdx.x * kLTok;
    grid_dependency_wait();  // y, pos and topk_w come from earlier kernels
    grid_launch_dependents();
    if (tid < kLTok) {
        const int64_t g = g0 + lane;
        int cnt = 0;
        if (g < NT)
            for_pairs_in_window(pos, g, R, row_lo, row_hi, [&](int k, int p) {
                s_p[lane][cnt] = p;
                s_w[lane][cnt] = __ldg(topk_w + g * R + k);
                ++cnt;
            });
        s_cnt[lane] = cnt;
        const unsigned nz = __ballot_sync((1u << kLTok) - 1u, cnt > 0 && g < NT);
        const unsigned z = __ballot_sync((1u << kLTok) - 1u, cnt == 0 && g < NT);
        const unsigned below = (1u << lane) - 1u;
        if (g < NT) s_tok[cnt > 0 ? __popc(nz & below) : __popc(nz) + __popc(z & below)] = lane;
        if (lane == 0) s_nnz = __popc(nz);
    }
    __syncthreads();
    const int ntok = (int)((NT - g0) < kLTok ? (NT - g0) : kLTok);
    const int nnz = s_nnz;
    // tokens without a pair on the rank: zero rows, plain stores
    for (int zt = nnz; zt < ntok; ++zt) {
        uint4 *row = out + (g0 + s_tok[zt]) * nvec;
        for (int c = tid; c < nvec; c += kLThreads) row[c] = make_uint4(0u, 0u, 0u, 0u);
    }
    // tokens with pairs: flattened (token, vector) work
    const int total = nnz * nvec;  // < 2^31: checked by the launcher
    for (int i0 = tid; i0 < total; i0 += kLThreads * kLCU) {
        int t[kLCU], c[kLCU], n[kLCU];
        float acc[kLCU][EL];
        int nmax = 0;
#pragma unroll
        for (int u = 0; u < kLCU; ++u) {
            const int i = i0 + u * kLThreads;
            t[u] = -1;
            c[u] = 0;
            n[u] = 0;
            if (i < total) {
                const int q = (int)fast_div((uint32_t)i, div_nvec);
                t[u] = s_tok[q];
                c[u] = i - q * nvec;
                n[u] = s_cnt[t[u]];
            }
            nmax = n[u] > nmax ? n[u] : nmax;
#pragma unroll
            for (int e = 0; e < EL; ++e) acc[u][e] = 0.f;
        }
        for (int j0 = 0; j0 < nmax; j0 += kLKB) {
            uint4 v[kLCU][kLKB];
#pragma unroll
            for (int u = 0; u < kLCU; ++u)
#pragma unroll
                for (int jj = 0; jj < kLKB; ++jj)
                    v[u][jj] = (j0 + jj < n[u]) ? ld_stream(y + (int64_t)s_p[t[u]][j0 + jj] * nvec + c[u])
                                                : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int u = 0; u < kLCU; ++u)
#pragma unroll
                for (int jj = 0; jj < kLKB; ++jj)
                    if (j0 + jj < n[u]) V::fma(acc[u], s_w[t[u]][j0 + jj], v[u][jj]);
        }
#pragma unroll
        for (int u = 0; u < kLCU; ++u)
            if (t[u] >= 0) out[(g0 + t[u]) * nvec + c[u]] = V::pack(acc[u]);
    }
}

cudaLaunchConfig_t local_cfg(int64_t NT, cudaStream_t stream, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((NT + kLTok - 1) / kLTok));
    cfg.blockDim = dim3(kLThreads);
    cfg.stream = stream;
    attr[0] = pdl_attribute();
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

}  // namespace

cudaError_t launch_pack_rank(const void *x, const float *x_scales, const int32_t *pos, int64_t NT,
                             int R, int64_t row_bytes, int scales_per_row, int64_t row_lo,
                             int64_t row_hi, void *packed_x, float *packed_scales,
                             int32_t *packed_src, cudaStream_t stream) {
    if (NT == 0) return cudaSuccess;
    const int64_t nvec = row_bytes / 16;
    if (nvec * kLTok * 32 >= (int64_t)1 << 31) return cudaErrorInvalidValue;  // flattened index
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = local_cfg(NT, stream, attr);
    return cudaLaunchKernelEx(&cfg, pack_rank_kernel, reinterpret_cast<const uint4 *>(x), x_scales,
                              pos, NT, R, (int)nvec, scales_per_row, make_fast_div((uint32_t)nvec),
                              row_lo, row_hi,
                              reinterpret_cast<uint4 *>(packed_x), packed_scales, packed_src);
}

cudaError_t launch_combine_rank(const void *y, int y_dtype, const int32_t *pos, const float *topk_w,
                                int64_t NT, int R, int H, int64_t row_lo, int64_t row_hi, void *out,
                                cudaStream_t stream) {
    if (NT == 0) return cudaSuccess;
    const int64_t nvec = (int64_t)H * (y_dtype == MOE_BF16 ? 2 : 4) / 16;
    if (nvec * kLTok >= (int64_t)1 << 31) return cudaErrorInvalidValue;  // flattened index
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = local_cfg(NT, stream, attr);
    auto kern = (y_dtype == MOE_BF16) ? combine_rank_kernel<1> : combine_rank_kernel<0>;
    return cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const uint4 *>(y), pos, topk_w, NT, R, (int)nvec,
                              make_fast_div((uint32_t)nvec), row_lo, row_hi,
                              reinterpret_cast<uint4 *>(out));
}

}  // namespace moe
