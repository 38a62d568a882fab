// Decode-fused dispatch for small batches: route, count and pack in one
// launch of ONE thread-block cluster, with no grid-wide barrier.
//
// "Hosting Qwen on Blackwell", section "Expert parallel": decode runs the
// whole dispatch as one kernel; "Lower latency and higher throughput with
// multi-node DeepSeek deployment", section "CUDA Graph": launch and latency
// costs dominate small decode batches.
//
// Block b of the cluster (C <= 16 blocks) owns the 32 consecutive tokens
// [32b, 32b + 32).  What a block needs from the others is only their
// per-expert pair counts, read through distributed shared memory:
//   route    warp w routes token 32b + w (the route kernel's per-token body)
//            and keeps the token's R experts in shared memory;
//   count    lane l of warp 0 is token 32b + l: it counts its experts and
//            sets bit l of each one's mask (shared-memory atomics); its rank
//            among the block's earlier tokens with that expert is the
//            number of mask bits below l;
//   --- cluster barrier: every block's counts are final ---
//   offsets  each block sums the counts of the blocks before it (its base
//            per expert) and of all blocks (the totals), and scans the
//            totals over experts; send counts are added with atomics;
//   pos      d*cap + (start of expert e within rank d) + base + rank, or -1
//            past cap (reported as MOE_ERR_CAPACITY);
//   pack     the block copies its own tokens' rows to their positions.
// Counts, offsets and send counts are integer sums, so every output equals
// that of the separate route, count and pack kernels bit for bit.
// Used for N*T <= 512 tokens (16 blocks of 32), E <= 256 and at most 256 KB of
// rows read and written per block (more would be copied by too few SMs).
#include <cooperative_groups.h>

#include "mem_ops.cuh"
#include "moe_internal.cuh"
#include "pdl.cuh"
#include "route_impl.cuh"

namespace cg = cooperative_groups;

namespace moe {
namespace {

constexpr int kSThreads = 1024;  // 32 warps: one token per warp while routing
constexpr int kSTok = 32;        // tokens per block
constexpr int kSMaxBlocks = 16;  // non-portable cluster size limit
constexpr int kSPackU = 4;       // row vectors per thread in flight while packing
constexpr int kSMaxE = 256;  // 8 experts per lane: the route body fits 64 registers
// Rows read and written per block (32 tokens x (1 + R) rows).  The pack
// runs on at most 16 SMs; up to about this much per block it beats the
// two-kernel form of dispatch_fused.cu, which packs on every SM (measured
// on GB300, 512-token batches, cluster vs two kernels: 48-160 KB per block
// 12.3-18.4 vs 14.4-20.5 us, 190-320 KB about equal, 384-640 KB 16.4-24.6
// vs 14.3-20.5 us).
constexpr int64_t kSMaxBlockPackBytes = 256 << 10;

struct SmallParams {
    const float *logits;
    const float *bias;
    int score_fn, renormalize;
    const uint4 *x;
    const float *x_scales;
    int nvec, spr;
    int N, T, E, R, cap;
    int64_t NT;
    FastDiv div_nvec;
    int32_t *topk_idx;
    float *topk_w;
    int32_t *expert_counts, *expert_offsets, *rank_counts, *rank_offsets, *send_counts, *pos,
        *status;
    uint4 *packed_x;
    float *packed_scales;
    int32_t *packed_src;
};

size_t small_smem_bytes(int E) { return (size_t)(4 * E + 1) * sizeof(int); }

template <int J, bool kVec4>
__global__ void __launch_bounds__(kSThreads, 1) dispatch_small_kernel(SmallParams P) {
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int b = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int E = P.E, R = P.R, N = P.N, L = P.E / P.N;
    const int64_t lo = (int64_t)b * kSTok;
    const int ntok = (int)(P.NT - lo < kSTok ? P.NT - lo : kSTok);  // >= 1: C = ceil(NT / 32)

    extern __shared__ __align__(16) int sm[];
    int *hist = sm;                                        // [E] this block's pairs per expert
    unsigned *gmask = reinterpret_cast<unsigned *>(sm + E);  // [E] bit l: token l chose e
    int *sbase = sm + 2 * E;                               // [E] pairs of earlier blocks
    int *eoff = sm + 3 * E;                                // [E + 1] totals, then their scan
    __shared__ int s_idx[kSTok][32];  // expert of pair k of token l
    __shared__ int s_pos[kSTok][32];  // its rank in the block, then its receive row
    __shared__ int s_wsum[32];

    for (int i = tid; i < E; i += kSThreads) {
        hist[i] = 0;
        gmask[i] = 0u;
    }
    grid_dependency_wait();  // logits and every output are shared with earlier kernels
    grid_launch_dependents();
    if (b == 0)
        for (int i = tid; i < N * N; i += kSThreads) P.send_counts[i] = 0;

    // ---- route: warp w routes token lo + w
    if (warp < ntok) {
        const int e = route_impl::route_token<J, kVec4>(P.logits, P.bias, lo + warp, E, R, P.score_fn,
                                                        P.renormalize, P.topk_idx, P.topk_w, lane);
        if (lane < R) s_idx[warp][lane] = e;
    }
    __syncthreads();

    // ---- count within the block: lane l of warp 0 is token lo + l
    if (warp == 0) {
        if (lane < ntok)
            for (int k = 0; k < R; ++k) {
                const int e = s_idx[lane][k];
                atomicOr(&gmask[e], 1u << lane);
                atomicAdd(&hist[e], 1);
            }
        __syncwarp();
        const unsigned below = (1u << lane) - 1u;
        if (lane < ntok)
            for (int k = 0; k < R; ++k) s_pos[lane][k] = __popc(gmask[s_idx[lane][k]] & below);
    }
    cluster.sync();  // every block's counts final; send_counts cleared by block 0

    // send counts: pairs of source rank s (token g = s*T + t) to rank d
    if (warp == 0 && lane < ntok) {
        const int s = (int)((lo + lane) / P.T);
        for (int k = 0; k < R; ++k) atomicAdd(P.send_counts + s * N + s_idx[lane][k] / L, 1);
    }
    // bases and totals through distributed shared memory (all loads first)
    for (int e = tid; e < E; e += kSThreads) {
        int v[kSMaxBlocks];
#pragma unroll
        for (int bb = 0; bb < kSMaxBlocks; ++bb) v[bb] = (bb < C) ? *cluster.map_shared_rank(hist + e, bb) : 0;
        int base = 0, tot = 0;
#pragma unroll
        for (int bb = 0; bb < kSMaxBlocks; ++bb) {
            tot += v[bb];
            if (bb < b) base += v[bb];
        }
        sbase[e] = base;
        eoff[e] = tot;
    }
    // no remote shared memory is read after this point; the wait before
    // exiting keeps this block's memory alive for the others
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
    __syncthreads();

    // exclusive scan of the totals over experts (E <= 256 < 1024: one each)
    {
        const int v = (tid < E) ? eoff[tid] : 0;
        int x = v;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) s_wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = s_wsum[lane];
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w += y;
            }
            s_wsum[lane] = w;
        }
        __syncthreads();
        const int excl = x - v + (warp > 0 ? s_wsum[warp - 1] : 0);
        if (tid < E) eoff[tid] = excl;  // each thread rewrites only the entry it read
        if (tid == E - 1) eoff[E] = excl + v;
    }
    __syncthreads();

    int over = 0;
    for (int d = tid; d < N; d += kSThreads)
        if (eoff[(d + 1) * L] - eoff[d * L] > P.cap) over = 1;
    over = __syncthreads_or(over);
    if (b == 0) {
        for (int e = tid; e < E; e += kSThreads) {
            P.expert_counts[e] = eoff[e + 1] - eoff[e];
            P.expert_offsets[e] = eoff[e];
        }
        for (int d = tid; d < N; d += kSThreads) {
            P.rank_counts[d] = eoff[(d + 1) * L] - eoff[d * L];
            P.rank_offsets[d] = eoff[d * L];
        }
        if (tid == 0) {
            P.expert_offsets[E] = eoff[E];
            P.rank_offsets[N] = eoff[E];
            *P.status = over ? MOE_ERR_CAPACITY : MOE_OK;
        }
    }

    // ---- receive rows of this block's pairs
    if (warp == 0 && lane < ntok) {
        const int64_t g = lo + lane;
        for (int k = 0; k < R; ++k) {
            const int e = s_idx[lane][k], d = e / L;
            const int local = eoff[e] - eoff[d * L] + sbase[e] + s_pos[lane][k];
            const int p = (local < P.cap) ? d * P.cap + local : -1;
            s_pos[lane][k] = p;
            P.pos[g * R + k] = p;
            if (p >= 0) P.packed_src[p] = (int32_t)(g * R + k);
        }
    }
    __syncthreads();

    // ---- pack: the block's rows, flattened (token, vector), loads first
    const int total = ntok * P.nvec;
    for (int i0 = tid; i0 < total; i0 += kSThreads * kSPackU) {
        uint4 v[kSPackU];
        int t[kSPackU], c[kSPackU];
#pragma unroll
        for (int u = 0; u < kSPackU; ++u) {
            const int i = i0 + u * kSThreads;
            t[u] = -1;
            c[u] = 0;
            if (i < total) {
                t[u] = (int)fast_div((uint32_t)i, P.div_nvec);
                c[u] = i - t[u] * P.nvec;
                v[u] = ld_stream(P.x + (lo + t[u]) * P.nvec + c[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < kSPackU; ++u) {
            if (t[u] < 0) continue;
            for (int k = 0; k < R; ++k) {
                const int p = s_pos[t[u]][k];
                if (p >= 0) P.packed_x[(int64_t)p * P.nvec + c[u]] = v[u];
            }
        }
    }
    if (P.spr > 0)
        for (int i = tid; i < ntok * R * P.spr; i += kSThreads) {
            const int t = i / (R * P.spr), rem = i - t * (R * P.spr), k = rem / P.spr, j = rem - k * P.spr;
            const int p = s_pos[t][k];
            if (p >= 0) P.packed_scales[(int64_t)p * P.spr + j] = __ldg(P.x_scales + (lo + t) * P.spr + j);
        }
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

template <int J, bool kVec4>
cudaError_t launch_small_jv(const SmallParams &P, int C, cudaStream_t stream) {
    auto kern = dispatch_small_kernel<J, kVec4>;
    const size_t smem = small_smem_bytes(P.E);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    // the cluster must fit the device: checked once per host thread, device,
    // context and cluster size reached so far
    static thread_local int ok_dev = -1, ok_c = 0;
    static thread_local unsigned long long ok_ctx = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long ctx = context_key();
    if (dev != ok_dev || ctx == 0 || ctx != ok_ctx || C > ok_c) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
        int n = 0;
        cfg.numAttrs = 1;  // occupancy query: cluster shape only
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n < 1) {
            cudaGetLastError();
            return cudaErrorNotSupported;
        }
        cfg.numAttrs = 2;
        if (dev != ok_dev || ctx != ok_ctx) ok_c = 0;
        ok_dev = dev;
        ok_ctx = context_key();
        ok_c = C > ok_c ? C : ok_c;
    }
    return cudaLaunchKernelEx(&cfg, kern, P);
}

template <int J>
cudaError_t launch_small_j(const SmallParams &P, int C, cudaStream_t stream) {
    if constexpr (J % 4 == 0) {
        if (P.E % 4 == 0 && (reinterpret_cast<uintptr_t>(P.logits) & 15) == 0)
            return launch_small_jv<J, true>(P, C, stream);
    }
    return launch_small_jv<J, false>(P, C, stream);
}

}  // namespace

bool dispatch_small_eligible(int64_t NT, int E, int R, int64_t row_bytes) {
    const int64_t per_block = NT < kSTok ? NT : kSTok;
    return NT >= 1 && NT <= (int64_t)kSTok * kSMaxBlocks && E <= kSMaxE && R <= 32 &&
           per_block * (R + 1) * row_bytes <= kSMaxBlockPackBytes;
}

cudaError_t launch_dispatch_small(const float *logits, const float *bias, int score_fn, int renormalize,
                                  const void *x, const float *x_scales, int N, int T, int E, int R,
                                  int64_t row_bytes, int spr, int64_t cap, int32_t *topk_idx,
                                  float *topk_w, int32_t *expert_counts, int32_t *expert_offsets,
                                  int32_t *rank_counts, int32_t *rank_offsets, int32_t *send_counts,
                                  int32_t *pos, int32_t *status, void *packed_x, float *packed_scales,
                                  int32_t *packed_src, cudaStream_t stream) {
    SmallParams P;
    P.logits = logits;
    P.bias = bias;
    P.score_fn = score_fn;
    P.renormalize = renormalize;
    P.x = reinterpret_cast<const uint4 *>(x);
    P.x_scales = x_scales;
    P.nvec = (int)(row_bytes / 16);
    P.spr = spr;
    P.N = N;
    P.T = T;
    P.E = E;
    P.R = R;
    P.cap = (int)cap;
    P.NT = (int64_t)N * T;
    P.div_nvec = make_fast_div((uint32_t)P.nvec);
    P.topk_idx = topk_idx;
    P.topk_w = topk_w;
    P.expert_counts = expert_counts;
    P.expert_offsets = expert_offsets;
    P.rank_counts = rank_counts;
    P.rank_offsets = rank_offsets;
    P.send_counts = send_counts;
    P.pos = pos;
    P.status = status;
    P.packed_x = reinterpret_cast<uint4 *>(packed_x);
    P.packed_scales = packed_scales;
    P.packed_src = packed_src;
    const int C = (int)((P.NT + kSTok - 1) / kSTok);
    // the same experts per lane as the route kernel, so that the softmax
    // denominator is summed in the same order and the weights agree bit for bit
    const int need = (E + 31) / 32;
    if (need <= 1) return launch_small_j<1>(P, C, stream);
    if (need <= 2) return launch_small_j<2>(P, C, stream);
    if (need <= 4) return launch_small_j<4>(P, C, stream);
    return launch_small_j<8>(P, C, stream);
}

}  // namespace moe
