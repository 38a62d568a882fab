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
#include "mem_ops.cuh"
#include "moe_internal.cuh"
#include "pdl.cuh"
#include "vec_traits.cuh"

namespace moe {
namespace {

constexpr int kThreads = 128;
constexpr int kU = 1;     // output vectors per thread per pass (partials)
constexpr int kRedU = 2;  // output vectors per thread per pass (reduction)
constexpr int kKB = 8;  // source rows loaded together

// kFew: R <= 8 (every row of a token loaded at once); else the rows of one
// slot at a time.  Separate instances keep the rare path from perturbing
// the register allocation of the common one.
template <int kBf16, bool kFew>
__global__ void __launch_bounds__(kThreads)
combine_partials_kernel(const uint4 *__restrict__ y, const int32_t *__restrict__ pos,
                        const float *__restrict__ topk_w, int64_t NT, int R, int nvec, int64_t cap,
                        int64_t rows_total, int P, uint4 *__restrict__ partial,
                        int32_t *__restrict__ slot_rank) {
    using V = Vec<kBf16>;
    constexpr int EL = V::kElems;
    __shared__ int s_pos[32], s_slot[32];
    __shared__ float s_w[32];
    // the same pairs stably ordered by slot (invalid pairs last)
    __shared__ int o_pos[32], o_slot[32];
    __shared__ float o_w[32];
    __shared__ int s_nslot;
    const int tid = threadIdx.x;
    grid_dependency_wait();  // y, pos and topk_w come from earlier kernels
    grid_launch_dependents();
    for (int64_t g = blockIdx.x; g < NT; g += gridDim.x) {
        if (tid < 32) {
            // Warp 0, lane k = pair k: slots are the token's distinct ranks in
            // the order of their first pair.  A lane's rank d = p / cap (32-bit:
            // N * cap < 2^31 is checked on the host); lanes that share d form
            // one match group whose lowest lane is its first pair, and the
            // slot is the number of first pairs before that one.
            const unsigned lane_bit = 1u << tid;
            int p = -1;
            float wk = 0.f;
            if (tid < R) {
                p = __ldg(pos + g * R + tid);
                if (p < 0 || (int64_t)p >= rows_total) p = -1;
                wk = __ldg(topk_w + g * R + tid);
            }
            const bool valid = p >= 0;
            // invalid lanes get a key of their own, so they match nobody
            const int d = valid ? (int)((unsigned)p / (unsigned)cap) : -1 - tid;
            const unsigned same = __match_any_sync(0xffffffffu, d);
            const int first = __ffs(same) - 1;
            const unsigned firsts = __ballot_sync(0xffffffffu, valid && first == tid);
            const int slot = valid ? __popc(firsts & ((1u << first) - 1u)) : -1;
            const int nslot = __popc(firsts);  // <= min(R, N) = P
            // Position of pair k in the by-slot order: the pairs of earlier
            // slots (group sizes summed over the first pairs below this
            // pair's first pair, by an exclusive warp scan) plus the pairs of
            // its own slot below it; invalid pairs go after all valid ones.
            const unsigned below = lane_bit - 1u;
            const int gsize = (valid && first == tid) ? __popc(same) : 0;
            int incl = gsize;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int t = __shfl_up_sync(0xffffffffu, incl, off);
                if (tid >= off) incl += t;
            }
            const int before_first = __shfl_sync(0xffffffffu, incl - gsize, first);
            const unsigned valid_mask = __ballot_sync(0xffffffffu, valid);
            const unsigned invalid_mask = __ballot_sync(0xffffffffu, tid < R && !valid);
            const int order = valid ? before_first + __popc(same & below)
                                    : __popc(valid_mask) + __popc(invalid_mask & below);
            if (tid < R) {
                s_pos[tid] = p;
                s_w[tid] = wk;
                s_slot[tid] = slot;
                o_pos[order] = p;
                o_w[order] = wk;
                o_slot[order] = slot;
            }
            if (valid && (firsts & lane_bit)) slot_rank[g * P + slot] = d;
            if (tid >= nslot && tid < P) slot_rank[g * P + tid] = -1;
            if (tid == 0) s_nslot = nslot;
        }
        __syncthreads();
        const int nslot = s_nslot;
        for (int c0 = tid; c0 < nvec; c0 += kThreads * kU) {
            if constexpr (kFew) {
                // R <= 8: the token's rows are loaded once, up front, in slot
                // order; one pass sums each slot's run of pairs (in k order)
                // and stores its partial row where the run ends.
                uint4 v[kKB][kU];
#pragma unroll
                for (int i = 0; i < kKB; ++i) {
                    const int p = (i < R) ? o_pos[i] : -1;
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const int c = c0 + u * kThreads;
                        v[i][u] = (p >= 0 && c < nvec) ? ld_stream(y + (int64_t)p * nvec + c)
                                                       : make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                float acc[kU][EL];
#pragma unroll
                for (int u = 0; u < kU; ++u)
#pragma unroll
                    for (int e = 0; e < EL; ++e) acc[u][e] = 0.f;
#pragma unroll
                for (int i = 0; i < kKB; ++i) {
                    const int sl = (i < R) ? o_slot[i] : -1;  // invalid pairs sit at the end
                    if (sl >= 0) {
#pragma unroll
                        for (int u = 0; u < kU; ++u) V::fma(acc[u], o_w[i], v[i][u]);
                        const int next = (i + 1 < R) ? o_slot[i + 1] : -1;
                        if (next != sl) {
#pragma unroll
                            for (int u = 0; u < kU; ++u) {
                                const int c = c0 + u * kThreads;
                                if (c < nvec) partial[(g * P + sl) * nvec + c] = V::pack(acc[u]);
#pragma unroll
                                for (int e = 0; e < EL; ++e) acc[u][e] = 0.f;
                            }
                        }
                    }
                }
                for (int j = nslot; j < P; ++j) {
#pragma unroll
                    for (int u = 0; u < kU; ++u) {
                        const int c = c0 + u * kThreads;
                        if (c < nvec) partial[(g * P + j) * nvec + c] = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            } else {
            // R > 8: the rows of one slot at a time
            for (int j = 0; j < P; ++j) {
                float acc[kU][EL];
#pragma unroll
                for (int u = 0; u < kU; ++u)
#pragma unroll
                    for (int e = 0; e < EL; ++e) acc[u][e] = 0.f;
                if (j < nslot) {
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
#pragma unroll
                for (int u = 0; u < kU; ++u) {
                    const int c = c0 + u * kThreads;
                    if (c < nvec) partial[(g * P + j) * nvec + c] = V::pack(acc[u]);
                }
            }
            }
        }
        __syncthreads();
    }
}

// kFew: P <= 8 (all partial rows of a token loaded at once)
template <int kBf16, bool kFew>
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
        for (int c0 = tid; c0 < nvec; c0 += kThreads * kRedU) {
            float acc[kRedU][EL];
#pragma unroll
            for (int u = 0; u < kRedU; ++u)
#pragma unroll
                for (int i = 0; i < EL; ++i) acc[u][i] = 0.f;
            if constexpr (kFew) {
                // all used partial rows loaded first, then summed in slot order
                uint4 v[kKB][kRedU];
#pragma unroll
                for (int j = 0; j < kKB; ++j)
#pragma unroll
                    for (int u = 0; u < kRedU; ++u) {
                        const int c = c0 + u * kThreads;
                        v[j][u] = (j < P && s_used[j] && c < nvec)
                                      ? ld_stream(partial + (g * P + j) * nvec + c)
                                      : make_uint4(0u, 0u, 0u, 0u);
                    }
#pragma unroll
                for (int j = 0; j < kKB; ++j)
                    if (j < P && s_used[j])
#pragma unroll
                        for (int u = 0; u < kRedU; ++u) V::add(acc[u], v[j][u]);
            } else {
                for (int j = 0; j < P; ++j) {
                    if (!s_used[j]) continue;
#pragma unroll
                    for (int u = 0; u < kRedU; ++u) {
                        const int c = c0 + u * kThreads;
                        if (c < nvec) V::add(acc[u], ld_stream(partial + (g * P + j) * nvec + c));
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < kRedU; ++u) {
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
    const bool few = R <= kKB;
    auto kern = (y_dtype == MOE_BF16) ? (few ? combine_partials_kernel<1, true> : combine_partials_kernel<1, false>)
                                      : (few ? combine_partials_kernel<0, true> : combine_partials_kernel<0, false>);
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
    const bool few = P <= kKB;
    auto kern = (y_dtype == MOE_BF16) ? (few ? reduce_partials_kernel<1, true> : reduce_partials_kernel<1, false>)
                                      : (few ? reduce_partials_kernel<0, true> : reduce_partials_kernel<0, false>);
    return cudaLaunchKernelEx(&cfg, kern, reinterpret_cast<const uint4 *>(partial), slot_rank, NT,
                              P, nvec, reinterpret_cast<uint4 *>(out));
}

}  // namespace moe
