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
// and list the pairs that fall in the region; the block then works only on
// the tokens that have some.  Every thread owns vectors of the flattened
// (token, vector) space of those tokens and keeps several in flight.  One
// block per token, as in the whole-batch kernels, would leave most blocks
// with nothing to do but a position load.
//
// pack_rank loads each vector of x[g] once and stores it to every row of g
// in the region.  combine_rank loads the first kLKB rows of its kLCU output
// vectors at once, then finishes one vector at a time (its f32 sum, any
// further rows, the store), so that only one vector's accumulator is live:
// 64 registers and four blocks per SM instead of 96 and two; its positions
// and weights are loaded together rather than the weights after the
// positions.  Measured on GB300 (rank 0, L2 flushed first), before -> after:
// Qwen3-235B-shaped prefill (16384 tokens, 90 % with pairs on the rank)
// pack 90 -> 65 us (one load per row copy before), combine 94 -> 78 us;
// DeepSeek-V3 decode pack 18.7 -> 14.7 us, combine 24.6 -> 22.5 us.
#include "mem_ops.cuh"
#include "moe_internal.cuh"
#include "pdl.cuh"
#include "vec_traits.cuh"

namespace moe {
namespace {

constexpr int kLThreads = 256;  // combine_rank
constexpr int kPThreads = 512;  // pack_rank
constexpr int kLTok = 8;   // tokens per block (one lane of warp 0 each)
constexpr int kLU = 4;     // vectors per thread in flight (pack)
constexpr int kLCU = 4;    // output vectors per thread in flight (combine)
constexpr int kLKB = 2;    // rows per output vector loaded together (combine)
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

// kScales: fp8 rows carry block scales.  A separate instance for the rows
// without them: a scales loop after the row copy, even skipped, made the
// copy about 20 % slower (GB300, Qwen3-235B-shaped prefill, rank 0: 78 vs
// 65 us).  With scales, they are copied before the rows, one load per
// (token, scale) stored to each of the token's rows: on the skewed fp8
// batch (rank 0: 74,454 rows) 106.5 us, against 124.4 us with the scales
// loop after the rows and 101 us for the rows alone.
template <bool kScales>
__global__ void __launch_bounds__(kPThreads)
pack_rank_kernel(const uint4 *__restrict__ x, const float *__restrict__ x_scales,
                 const int32_t *__restrict__ pos, int64_t NT, int R, int nvec, int spr,
                 FastDiv div_nvec, int64_t row_lo, int64_t row_hi, uint4 *__restrict__ packed_x,
                 float *__restrict__ packed_scales, int32_t *__restrict__ packed_src) {
    __shared__ int s_p[kLTok][32];  // per token: its rows in the region, in k order
    __shared__ int s_cnt[kLTok];
    __shared__ int s_tok[kLTok];    // the tokens with rows in the region
    __shared__ int s_nnz;
    const int tid = threadIdx.x, lane = tid & 31;
    const int64_t g0 = (int64_t)blockIdx.x * kLTok;
    grid_dependency_wait();  // pos comes from the count kernel
    grid_launch_dependents();
    if (tid < kLTok) {
        const int64_t g = g0 + lane;
        int cnt = 0;
        if (g < NT)
            for_pairs_in_window(pos, g, R, row_lo, row_hi, [&](int k, int p) {
                s_p[lane][cnt++] = p;
                packed_src[p] = (int32_t)(g * R + k);
            });
        s_cnt[lane] = cnt;
        const unsigned nz = __ballot_sync((1u << kLTok) - 1u, cnt > 0);
        if (cnt > 0) s_tok[__popc(nz & ((1u << lane) - 1u))] = lane;
        if (lane == 0) s_nnz = __popc(nz);
    }
    __syncthreads();
    const int nnz = s_nnz;
    if (kScales)
        for (int i = tid; i < nnz * spr; i += kPThreads) {
            const int q = i / spr, k = i - q * spr;
            const int t = s_tok[q], n = s_cnt[t];
            const float sv = __ldg(x_scales + (g0 + t) * spr + k);
            for (int j = 0; j < n; ++j) packed_scales[(int64_t)s_p[t][j] * spr + k] = sv;
        }
    const int total = nnz * nvec;  // < 2^31: checked by the launcher
    for (int i0 = tid; i0 < total; i0 += kPThreads * kLU) {
        uint4 v[kLU];
        int t[kLU], c[kLU];
#pragma unroll
        for (int u = 0; u < kLU; ++u) {
            const int i = i0 + u * kPThreads;
            t[u] = -1;
            c[u] = 0;
            if (i < total) {
                const int q = (int)fast_div((uint32_t)i, div_nvec);
                t[u] = s_tok[q];
                c[u] = i - q * nvec;
                v[u] = ld_stream(x + (g0 + t[u]) * nvec + c[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < kLU; ++u) {
            if (t[u] < 0) continue;
            const int n = s_cnt[t[u]];
            for (int j = 0; j < n; ++j) packed_x[(int64_t)s_p[t[u]][j] * nvec + c[u]] = v[u];
        }
    }
}

template <int kBf16>
__global__ void __launch_bounds__(kLThreads, 4)
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
            for (int k0 = 0; k0 < R; k0 += kLPB) {  // positions and weights in one batch
                int pv[kLPB];
                float wv[kLPB];
#pragma unroll
                for (int j = 0; j < kLPB; ++j) {
                    pv[j] = (k0 + j < R) ? __ldg(pos + g * R + k0 + j) : -1;
                    wv[j] = (k0 + j < R) ? __ldg(topk_w + g * R + k0 + j) : 0.f;
                }
#pragma unroll
                for (int j = 0; j < kLPB; ++j)
                    if (k0 + j < R && in_window(pv[j], row_lo, row_hi)) {
                        s_p[lane][cnt] = pv[j];
                        s_w[lane][cnt] = wv[j];
                        ++cnt;
                    }
            }
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
        }
        // the first kLKB rows of every vector in flight together
        uint4 v[kLCU][kLKB];
#pragma unroll
        for (int u = 0; u < kLCU; ++u)
#pragma unroll
            for (int jj = 0; jj < kLKB; ++jj)
                v[u][jj] = (jj < n[u]) ? ld_stream(y + (int64_t)s_p[t[u]][jj] * nvec + c[u])
                                       : make_uint4(0u, 0u, 0u, 0u);
        // then one vector at a time: its sum in k order, its later rows, its store
#pragma unroll
        for (int u = 0; u < kLCU; ++u) {
            if (t[u] < 0) continue;
            float acc[EL];
#pragma unroll
            for (int e = 0; e < EL; ++e) acc[e] = 0.f;
#pragma unroll
            for (int jj = 0; jj < kLKB; ++jj)
                if (jj < n[u]) V::fma(acc, s_w[t[u]][jj], v[u][jj]);
            for (int j0 = kLKB; j0 < n[u]; j0 += kLKB) {
                uint4 v2[kLKB];
#pragma unroll
                for (int jj = 0; jj < kLKB; ++jj)
                    v2[jj] = (j0 + jj < n[u]) ? ld_stream(y + (int64_t)s_p[t[u]][j0 + jj] * nvec + c[u])
                                              : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int jj = 0; jj < kLKB; ++jj)
                    if (j0 + jj < n[u]) V::fma(acc, s_w[t[u]][j0 + jj], v2[jj]);
            }
            out[(g0 + t[u]) * nvec + c[u]] = V::pack(acc);
        }
    }
}

cudaLaunchConfig_t local_cfg(int64_t NT, int threads, cudaStream_t stream, cudaLaunchAttribute *attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((NT + kLTok - 1) / kLTok));
    cfg.blockDim = dim3(threads);
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
    if (nvec * kLTok >= (int64_t)1 << 31) return cudaErrorInvalidValue;  // flattened index
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = local_cfg(NT, kPThreads, stream, attr);
    auto kern = scales_per_row > 0 ? pack_rank_kernel<true> : pack_rank_kernel<false>;
    return cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const uint4 *>(x), x_scales,
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
    cudaLaunchConfig_t cfg = local_cfg(NT, kLThreads, stream, attr);
    auto kern = (y_dtype == MOE_BF16) ? combine_rank_kernel<1> : combine_rank_kernel<0>;
    return cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const uint4 *>(y), pos, topk_w, NT, R, (int)nvec,
                              make_fast_div((uint32_t)nvec), row_lo, row_hi,
                              reinterpret_cast<uint4 *>(out));
}

}  // namespace moe
