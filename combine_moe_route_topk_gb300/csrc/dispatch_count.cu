// Dispatch count: per-expert counts, prefix sums, per-rank totals, the
// source->destination count matrix and the receive row of every routed pair,
// in ONE launch of one thread-block cluster.
//
// "Enabling trillion-parameter models on AWS EFA", section "Dispatch and
// combine": token counts per expert come from shared-memory atomics inside
// one block, and a cumulative sum of the counts gives the offsets at which
// tokens are packed contiguously per destination.  "Efficient and portable
// mixture-of-experts communication", section "Dispatch": the receiver lays
// tokens out in one contiguous buffer per expert.
//
// One block is not enough parallelism for the larger batches, so the work
// is split over the C blocks of a cluster (C <= 16) and the blocks exchange
// their per-expert histograms through distributed shared memory.  The
// cluster barrier is a hardware barrier, so nothing here spins on memory.
//
// Ordering (deterministic): rows of rank d are grouped by expert ascending
// and, inside an expert, by token g ascending.  Token ranges are contiguous
// per block (block b owns tokens [b*per, (b+1)*per)), so the row of pair
// (g, k) routed to expert e is
//     d*cap + (expert_offsets[e] - rank_offsets[d])          expert start
//           + sum over blocks b' < b of hist_b'[e]            earlier blocks
//           + sum over earlier 32-token groups of this block  earlier groups
//           + popc(group_mask[e] & lanes below this one)      inside the group
// where group_mask[e] has bit l set when lane l's token chose e.
#include <cooperative_groups.h>

#include "moe_internal.cuh"

namespace cg = cooperative_groups;

namespace moe {
namespace {

constexpr int kSendSmem = 4096;  // ints of per-block send matrix staging

struct CountSmem {
    // byte offsets inside dynamic shared memory
    int gmask, run, base, tot, eoff, send, flags, bytes;
};

// kWarps 32-token groups per tile (one token per thread).
__host__ __device__ inline CountSmem count_smem_layout(int E, int kWarps) {
    CountSmem s;
    int o = 0;
    s.gmask = o; o += kWarps * E * 4;    // u32 [kWarps][E]: group masks, then group prefix
    s.run = o;   o += E * 4;             // running count of this block per expert
    s.base = o;  o += E * 4;             // sum over earlier blocks
    s.tot = o;   o += E * 4;             // sum over all blocks
    s.eoff = o;  o += (E + 1) * 4 + 12;  // exclusive scan of tot (+ pad to 16 B)
    s.send = o;  o += kSendSmem * 4;     // staged send_counts rows of this block
    s.flags = o; o += 64 + 32 * 4;       // [0]: invalid pair seen; [16..48): scan partials
    s.bytes = o;
    return s;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

template <int kCountThreads, int kMaxR>
__global__ void __launch_bounds__(kCountThreads, 1)
dispatch_count_kernel(const int32_t *__restrict__ topk_idx, int N, int T, int E, int R,
                      int64_t cap, int32_t *__restrict__ expert_counts,
                      int32_t *__restrict__ expert_offsets, int32_t *__restrict__ rank_counts,
                      int32_t *__restrict__ rank_offsets, int32_t *__restrict__ send_counts,
                      int32_t *__restrict__ pos, int32_t *__restrict__ status) {
    constexpr int kWarps = kCountThreads / 32;
    extern __shared__ __align__(16) unsigned char smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int b = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const CountSmem lay = count_smem_layout(E, kWarps);
    uint32_t *gmask = reinterpret_cast<uint32_t *>(smem + lay.gmask);
    int *run = reinterpret_cast<int *>(smem + lay.run);
    int *sbase = reinterpret_cast<int *>(smem + lay.base);
    int *stot = reinterpret_cast<int *>(smem + lay.tot);
    int *eoff = reinterpret_cast<int *>(smem + lay.eoff);
    int *ssend = reinterpret_cast<int *>(smem + lay.send);
    int *flags = reinterpret_cast<int *>(smem + lay.flags);
    int *wsum = flags + 16;

    const int L = E / N;
    const int64_t NT = (int64_t)N * T;
    const int64_t per = (NT + C - 1) / C;
    const int64_t lo = min(NT, (int64_t)b * per);
    const int64_t hi = min(NT, lo + per);
    const int s_first = (hi > lo) ? (int)(lo / T) : 0;
    const int span = (hi > lo) ? (int)((hi - 1) / T) - s_first + 1 : 0;
    const bool send_in_smem = (int64_t)span * N <= kSendSmem;

    // ---- phase 0: clear; send_counts is accumulated with atomics below ----
    for (int i = tid; i < E; i += kCountThreads) run[i] = 0;
    for (int i = tid; i < kSendSmem; i += kCountThreads) ssend[i] = 0;
    if (tid == 0) flags[0] = 0;
    for (int64_t i = (int64_t)b * kCountThreads + tid; i < (int64_t)N * N; i += (int64_t)C * kCountThreads)
        send_counts[i] = 0;
    cluster.sync();  // zeroed send_counts visible to every block; all blocks running

    // ---- phase 1: group masks, in-block ranks, histograms ------------------
    bool bad = false;
    for (int64_t t0 = lo; t0 < hi; t0 += kCountThreads) {
        for (int i = tid; i < kWarps * E; i += kCountThreads) gmask[i] = 0u;
        __syncthreads();
        const int64_t g = t0 + tid;
        const bool active = g < hi;
        int ek[kMaxR];
        int rk[kMaxR];
        const unsigned bit = 1u << lane;
        uint32_t *mymask = gmask + warp * E;
#pragma unroll
        for (int k = 0; k < kMaxR; ++k) {
            ek[k] = -1;
            rk[k] = 0;
            if (k < R && active) {
                int e = __ldg(topk_idx + g * R + k);
                bool ok = (e >= 0 && e < E);
                if (ok) {
                    unsigned old = atomicOr(mymask + e, bit);
                    ok = (old & bit) == 0u;  // a repeat of an earlier k of this token
                }
                if (ok) {
                    ek[k] = e;
                    const int s = (int)(g / T), d = e / L;
                    if (send_in_smem) atomicAdd(ssend + (s - s_first) * N + d, 1);
                    else atomicAdd(send_counts + (int64_t)s * N + d, 1);
                } else {
                    bad = true;
                }
            }
        }
        __syncwarp();
        const unsigned lt = lanemask_lt();
#pragma unroll
        for (int k = 0; k < kMaxR; ++k)
            if (k < R && ek[k] >= 0) rk[k] = __popc(mymask[ek[k]] & lt);
        __syncthreads();
        // per expert: prefix over the 32 groups of this tile, then advance run
        for (int e = tid; e < E; e += kCountThreads) {
            int r = run[e];
#pragma unroll 8
            for (int w = 0; w < kWarps; ++w) {
                const uint32_t m = gmask[w * E + e];
                gmask[w * E + e] = (uint32_t)r;
                r += __popc(m);
            }
            run[e] = r;
        }
        __syncthreads();
        if (active) {
#pragma unroll
            for (int k = 0; k < kMaxR; ++k)
                if (k < R) pos[g * R + k] = (ek[k] >= 0) ? (int)mymask[ek[k]] + rk[k] : -1;
        }
        __syncthreads();  // gmask is cleared again by the next tile
    }
    if (bad) atomicOr(flags, 1);
    if (send_in_smem) {
        for (int i = tid; i < span * N; i += kCountThreads) {
            const int v = ssend[i];
            if (v != 0) atomicAdd(send_counts + (int64_t)(s_first + i / N) * N + (i % N), v);
        }
    }

    cluster.sync();  // every block's run[] and flags final

    // ---- phase 2: exchange histograms through distributed shared memory ----
    int any_bad = 0;
    for (int e = tid; e < E; e += kCountThreads) {
        int base = 0, tot = 0;
        for (int bb = 0; bb < C; ++bb) {
            const int v = *cluster.map_shared_rank(run + e, bb);
            tot += v;
            if (bb < b) base += v;
        }
        sbase[e] = base;
        stot[e] = tot;
    }
    if (tid < C) any_bad = *cluster.map_shared_rank(flags, tid);
    any_bad = __syncthreads_or(any_bad);
    cluster.sync();  // no remote shared memory access after this point

    // exclusive scan of stot over experts: thread t sums the kIpt
    // consecutive experts [t*kIpt, t*kIpt + kIpt), then a two-level warp scan
    {
        constexpr int kIpt = (1024 + kCountThreads - 1) / kCountThreads;  // E <= 1024
        int v[kIpt];
        int local = 0;
#pragma unroll
        for (int i = 0; i < kIpt; ++i) {
            const int e = tid * kIpt + i;
            v[i] = (e < E) ? stot[e] : 0;
            local += v[i];
        }
        int x = local;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) wsum[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int s = (lane < kWarps) ? wsum[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, s, off);
                if (lane >= off) s += y;
            }
            if (lane < kWarps) wsum[lane] = s;  // inclusive over warps
        }
        __syncthreads();
        int run_e = x - local + (warp > 0 ? wsum[warp - 1] : 0);  // exclusive start
#pragma unroll
        for (int i = 0; i < kIpt; ++i) {
            const int e = tid * kIpt + i;
            if (e < E) eoff[e] = run_e;
            run_e += v[i];
            if (e == E - 1) eoff[E] = run_e;
        }
        __syncthreads();
    }

    if (b == 0) {
        int over = 0;
        for (int e = tid; e < E; e += kCountThreads) {
            expert_counts[e] = stot[e];
            expert_offsets[e] = eoff[e];
        }
        if (tid == 0) expert_offsets[E] = eoff[E];
        for (int d = tid; d < N; d += kCountThreads) {
            const int rc = eoff[(d + 1) * L] - eoff[d * L];
            rank_counts[d] = rc;
            rank_offsets[d] = eoff[d * L];
            if ((int64_t)rc > cap) over = 1;
        }
        if (tid == 0) rank_offsets[N] = eoff[E];
        over = __syncthreads_or(over);
        if (tid == 0) *status = any_bad ? MOE_ERR_INVALID_ARG : (over ? MOE_ERR_CAPACITY : MOE_OK);
    }

    // ---- phase 3: final rows --------------------------------------------------
    for (int64_t t0 = lo; t0 < hi; t0 += kCountThreads) {
        const int64_t g = t0 + tid;
        if (g >= hi) continue;
        for (int k = 0; k < R; ++k) {
            const int part = pos[g * R + k];  // written by this thread in phase 1
            if (part < 0) continue;
            const int e = __ldg(topk_idx + g * R + k);
            const int d = e / L;
            const int64_t local = (int64_t)(eoff[e] - eoff[d * L]) + sbase[e] + part;
            pos[g * R + k] = (local < cap) ? (int)((int64_t)d * cap + local) : -1;
        }
    }
}

// Largest cluster (<= 16 blocks) of this kernel with this much shared memory
// that the current device can co-schedule; 0 if none.  Cached per host thread
// and device for the largest shared-memory request seen.
template <int kThreads, int kMaxR>
int max_cluster_blocks(size_t smem_bytes) {
    static thread_local int cached_dev = -1;
    static thread_local size_t cached_smem = 0;
    static thread_local int cached_c = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev == cached_dev && smem_bytes <= cached_smem) return cached_c;
    auto kern = dispatch_count_kernel<kThreads, kMaxR>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes) !=
        cudaSuccess)
        return 0;
    cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    cudaGetLastError();
    int best = 0;
    for (int c : {16, 8, 4, 2, 1}) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(c);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem_bytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = c;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) {
            best = c;
            break;
        }
        cudaGetLastError();
    }
    cached_dev = dev;
    cached_smem = smem_bytes;
    cached_c = best;
    return best;
}

template <int kThreads, int kMaxR>
cudaError_t launch_count(const int32_t *topk_idx, int N, int T, int E, int R, int64_t cap,
                         int32_t *expert_counts, int32_t *expert_offsets, int32_t *rank_counts,
                         int32_t *rank_offsets, int32_t *send_counts, int32_t *pos,
                         int32_t *status, cudaStream_t stream) {
    const CountSmem lay = count_smem_layout(E, kThreads / 32);
    const size_t smem = (size_t)lay.bytes;
    const int cmax = max_cluster_blocks<kThreads, kMaxR>(smem);
    if (cmax <= 0) return cudaErrorNotSupported;
    const int64_t NT = (int64_t)N * T;
    // one tile (one token per thread) per block when possible
    const int64_t want = (NT + kThreads - 1) / kThreads;
    const int c = (int)(want < 1 ? 1 : (want > cmax ? cmax : want));

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dispatch_count_kernel<kThreads, kMaxR>, topk_idx, N, T, E, R,
                              cap, expert_counts, expert_offsets, rank_counts, rank_offsets,
                              send_counts, pos, status);
}

}  // namespace

cudaError_t launch_dispatch_count(const int32_t *topk_idx, int N, int T, int E, int R,
                                  int64_t cap, int32_t *expert_counts, int32_t *expert_offsets,
                                  int32_t *rank_counts, int32_t *rank_offsets,
                                  int32_t *send_counts, int32_t *pos, int32_t *status,
                                  cudaStream_t stream) {
    // R <= 8 keeps the per-pair state of a thread in registers at 1024
    // threads per block; larger R uses 512-thread blocks.
    if (R <= 8)
        return launch_count<1024, 8>(topk_idx, N, T, E, R, cap, expert_counts, expert_offsets,
                                     rank_counts, rank_offsets, send_counts, pos, status, stream);
    return launch_count<512, 32>(topk_idx, N, T, E, R, cap, expert_counts, expert_offsets,
                                 rank_counts, rank_offsets, send_counts, pos, status, stream);
}

}  // namespace moe
