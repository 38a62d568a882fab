// Expert-parallel local path of one rank, the dispatch side: with
// replicated inputs, a rank selects the tokens routed to its own experts
// ("Hosting Qwen on Blackwell", section "Expert parallel").  pack_rank
// copies x[g] to every receive row pos[g][k] inside rank d's region
// [d*cap, (d+1)*cap) (and sets packed_src there).  The local accumulation
// that follows the experts is the combine kernel restricted to the same
// region (combine.cu).
//
// Only some tokens have a pair on a given rank (DeepSeek-V3 decode: about a
// quarter), so a block takes 8 tokens at once: lanes of warp 0 read their
// positions, one lane per token and eight positions per batch of loads,
// and list the pairs that fall in the region; the block then works only on
// the tokens that have some.  Every thread owns vectors of the flattened
// (token, vector) space of those tokens and keeps several in flight: it
// loads each vector of x[g] once and stores it to every row of g in the
// region.  Measured on GB300 (rank 0, L2 flushed first), against one load
// per row copy: Qwen3-235B-shaped prefill (16384 tokens, 90 % with pairs on
// the rank) 90 -> 65 us; DeepSeek-V3 decode 18.7 -> 14.7 us.
#include "mem_ops.cuh"
#include "moe_internal.cuh"
#include "pdl.cuh"

namespace moe {
namespace {

constexpr int kPThreads = 512;  // pack_rank
constexpr int kLTok = 8;   // tokens per block (one lane of warp 0 each)
constexpr int kLU = 4;     // vectors per thread in flight (pack)
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

}  // namespace moe
