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
// their per-expert histograms and per-destination send counts through
// distributed shared memory.  The cluster barrier is a hardware barrier, so
// nothing here spins on memory.
//
// Ordering (deterministic): rows of rank d are grouped by expert ascending
// and, inside an expert, by token g ascending.  Token ranges are contiguous
// per block (block b owns tokens [b*per, (b+1)*per), per a multiple of 32),
// so the row of pair (g, k) routed to expert e is
//     d*cap + (expert_offsets[e] - rank_offsets[d])          expert start
//           + sum over blocks b' < b of hist_b'[e]            earlier blocks
//           + sum over earlier 32-token groups of this block  earlier groups
//           + popc(group_mask[e] & lanes below this one)      inside the group
// where group_mask[e] has bit l set when lane l's token chose e.
//
// send_counts[s][d] needs no per-pair atomics when T % 32 == 0: source-rank
// boundaries then fall on group boundaries, and the pairs rank s sends to
// rank d are differences of the group prefixes summed over d's experts.
#include <cooperative_groups.h>

#include "moe_internal.cuh"
#include "pdl.cuh"

namespace cg = cooperative_groups;

namespace moe {
namespace {

constexpr int kSendSmem = 4096;  // ints of per-block send-count staging
constexpr int kMaxCluster = 16;

enum SendMode { kSendFromPrefix = 0, kSendSmemAtomics = 1, kSendGlobalAtomics = 2 };

struct CountSmem {
    // byte offsets inside dynamic shared memory
    int gmask, subsum, run, base, tot, eoff, fin, send, flags, bytes;
};

__host__ __device__ inline int count_ksub(int threads, int E) {
    const int warps = threads / 32;
    int k = threads / E;
    return k >= warps ? warps : (k >= 16 ? 16 : k >= 8 ? 8 : k >= 4 ? 4 : k >= 2 ? 2 : 1);
}

// kWarps 32-token groups per tile (one token per thread); kSub parts of the
// group prefix per expert.
// Every section starts on a 16-byte boundary (fin is read as int2, and E
// may be odd).
__host__ __device__ inline CountSmem count_smem_layout(int E, int kWarps, int kSub) {
    CountSmem s;
    int o = 0;
    auto take = [&o](int bytes) {
        const int at = o;
        o += (bytes + 15) & ~15;
        return at;
    };
    s.gmask = take(kWarps * E * 4);   // u32 [kWarps][E]: group masks, then group prefixes
    s.subsum = take(kSub * E * 4);    // group-prefix partial sums
    s.run = take(2 * E * 4);          // pairs of this block so far (double buffered)
    s.base = take(E * 4);             // pairs in earlier blocks
    s.tot = take(E * 4);              // pairs in all blocks
    s.eoff = take((E + 1) * 4);       // exclusive scan of tot
    s.fin = take(E * 8);              // int2 per expert: first row, rows left before cap
    s.send = take(kSendSmem * 4);     // this block's send counts, rows s_first..
    s.flags = take(64 + 32 * 4);      // [0]: invalid pair seen; [16..48): scan partials
    s.bytes = o;
    return s;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

template <int kThreads, int kMaxR>
__global__ void __launch_bounds__(kThreads, 1)
dispatch_count_kernel(const int32_t *__restrict__ topk_idx, int N, int T, int E, int R, int cap,
                      int32_t *__restrict__ expert_counts, int32_t *__restrict__ expert_offsets,
                      int32_t *__restrict__ rank_counts, int32_t *__restrict__ rank_offsets,
                      int32_t *__restrict__ send_counts, int32_t *__restrict__ pos,
                      int32_t *__restrict__ status) {
    constexpr int kWarps = kThreads / 32;
    extern __shared__ __align__(16) unsigned char smem[];
    cg::cluster_group cluster = cg::this_cluster();
    const int C = (int)cluster.num_blocks();
    const int b = (int)cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kSub = count_ksub(kThreads, E);
    const int wps = kWarps / kSub;  // groups per part
    const CountSmem lay = count_smem_layout(E, kWarps, kSub);
    uint32_t *gmask = reinterpret_cast<uint32_t *>(smem + lay.gmask);
    int *subsum = reinterpret_cast<int *>(smem + lay.subsum);
    int *run = reinterpret_cast<int *>(smem + lay.run);
    int *sbase = reinterpret_cast<int *>(smem + lay.base);
    int *stot = reinterpret_cast<int *>(smem + lay.tot);
    int *eoff = reinterpret_cast<int *>(smem + lay.eoff);
    int2 *fin = reinterpret_cast<int2 *>(smem + lay.fin);
    int *ssend = reinterpret_cast<int *>(smem + lay.send);
    int *flags = reinterpret_cast<int *>(smem + lay.flags);
    int *wsum = flags + 16;
    __shared__ int sfirst_tab[kMaxCluster];  // first source rank of each block

    // N*T*R < 2^31 and N*cap < 2^31 are checked on the host: 32-bit math.
    const int L = E / N;
    const int NT = N * T;
    const int per = (((NT + C - 1) / C) + 31) & ~31;  // tokens per block, multiple of 32
    const int lo = min(NT, b * per);
    const int hi = min(NT, lo + per);
    const int s_first = (hi > lo) ? lo / T : 0;
    const int span = (hi > lo) ? (hi - 1) / T - s_first + 1 : 0;
    const int max_span = (T > 0) ? (per + T - 1) / T + 1 : 0;  // bound for every block
    const int mode = (max_span * N > kSendSmem) ? kSendGlobalAtomics
                     : (T % 32 == 0)            ? kSendFromPrefix
                                                : kSendSmemAtomics;
    const bool one_tile = per <= kThreads;

    // Dependents may be scheduled at once: the library's kernels that follow
    // count read nothing before their own wait except L2 prefetch hints,
    // which cannot return stale data, so pack can start pulling x into L2
    // while route and count are still running.
    grid_launch_dependents();

    // ---- phase 0: clear shared state (overlaps the previous kernel's tail)
    if (tid < kMaxCluster) sfirst_tab[tid] = (T > 0) ? min(NT, tid * per) / T : 0;
    for (int i = tid; i < 2 * E; i += kThreads) run[i] = 0;
    if (mode != kSendGlobalAtomics)
        for (int i = tid; i < span * N; i += kThreads) ssend[i] = 0;
    if (tid == 0) flags[0] = 0;
    for (int i = tid; i < kWarps * E; i += kThreads) gmask[i] = 0u;

    grid_dependency_wait();  // topk_idx comes from the previous kernel
    if (mode == kSendGlobalAtomics) {
        for (int i = b * kThreads + tid; i < N * N; i += C * kThreads) send_counts[i] = 0;
        cluster.sync();
    }
    __syncthreads();

    // ---- phase 1: group masks, in-block ranks, histograms -----------------
    bool bad = false;
    int ek[kMaxR];    // expert of pair k (-1: invalid), kept for phase 3
    int part[kMaxR];  // rank of pair k among earlier pairs of this block with that expert
    int cur = 0;      // run[] buffer holding the counts before this tile
    for (int t0 = lo; t0 < hi; t0 += kThreads) {
        const int g = t0 + tid;
        const bool active = g < hi;
#pragma unroll
        for (int k = 0; k < kMaxR; ++k) ek[k] = -1;
        if (active) {
            const int32_t *row = topk_idx + (int64_t)g * R;
            if ((R & 3) == 0 && (reinterpret_cast<uintptr_t>(topk_idx) & 15) == 0) {
#pragma unroll
                for (int k = 0; k < kMaxR; k += 4) {
                    if (k < R) {
                        const int4 v = __ldg(reinterpret_cast<const int4 *>(row + k));
                        ek[k] = v.x;
                        ek[k + 1] = v.y;
                        ek[k + 2] = v.z;
                        ek[k + 3] = v.w;
                    }
                }
            } else {
#pragma unroll
                for (int k = 0; k < kMaxR; ++k)
                    if (k < R) ek[k] = __ldg(row + k);
            }
        }
        if (t0 != lo) {
            for (int i = tid; i < kWarps * E; i += kThreads) gmask[i] = 0u;
            __syncthreads();
        }
        // validity: in range and not a repeat of an earlier expert of the token
#pragma unroll
        for (int k = 0; k < kMaxR; ++k) {
            if (k < R && active) {
                const int e = ek[k];
                bool ok = (e >= 0 && e < E);
#pragma unroll
                for (int k2 = 0; k2 < k; ++k2) ok = ok && (ek[k2] != e);
                if (!ok) {
                    ek[k] = -1;
                    bad = true;
                }
            }
        }
        const unsigned bit = 1u << lane;
        uint32_t *mymask = gmask + warp * E;
        const int s_rel = active ? g / T - s_first : 0;
#pragma unroll
        for (int k = 0; k < kMaxR; ++k) {
            if (k < R && ek[k] >= 0) {
                atomicOr(mymask + ek[k], bit);
                if (mode == kSendSmemAtomics) atomicAdd(ssend + s_rel * N + ek[k] / L, 1);
                else if (mode == kSendGlobalAtomics)
                    atomicAdd(send_counts + (s_rel + s_first) * N + ek[k] / L, 1);
            }
        }
        __syncwarp();
        const unsigned lt = lanemask_lt();
#pragma unroll
        for (int k = 0; k < kMaxR; ++k)
            part[k] = (k < R && ek[k] >= 0) ? __popc(mymask[ek[k]] & lt) : 0;
        __syncthreads();
        // group prefix per expert, split into kSub parts of wps groups each.
        // Pass A turns the masks of a part into prefixes inside the part (all
        // loads first) and, when source ranks start on group boundaries,
        // adds each group's pairs to the send count of the group's rank.
        // With kSub > 1, pass B adds the sums of earlier parts.
        const int nxt = cur ^ 1;
        for (int i = tid; i < E * kSub; i += kThreads) {
            const int sub = i / E, e = i - sub * E;
            const int wb = sub * wps;
            int r = (kSub == 1) ? run[cur * E + e] : 0;
            // send-count walk state: source rank of the current group, tokens
            // of that rank seen so far in this part, pairs not yet flushed
            const int g0 = t0 + 32 * wb;
            int s_cur = g0 / T, rem = g0 - s_cur * T, acc = 0;
            const int d = e / L;
            auto flush = [&]() {  // pending pairs of (s_cur, d)
                if (acc) atomicAdd(ssend + (s_cur - s_first) * N + d, acc);
                acc = 0;
            };
            for (int j0 = 0; j0 < wps; j0 += 8) {  // 8 groups at a time: loads first
                int c[8];
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    c[j] = (j0 + j < wps) ? __popc(gmask[(wb + j0 + j) * E + e]) : 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    if (j0 + j < wps) {
                        gmask[(wb + j0 + j) * E + e] = (uint32_t)r;
                        r += c[j];
                        if (mode == kSendFromPrefix && g0 + 32 * (j0 + j) < hi) {
                            if (rem == T) {  // this group starts the next source rank
                                flush();
                                ++s_cur;
                                rem = 0;
                            }
                            acc += c[j];
                            rem += 32;
                        }
                    }
                }
            }
            if (mode == kSendFromPrefix) flush();
            if (kSub == 1) run[nxt * E + e] = r;
            else subsum[sub * E + e] = r;
        }
        if (kSub > 1) {
            __syncthreads();
            for (int i = tid; i < E * kSub; i += kThreads) {
                const int sub = i / E, e = i - sub * E;
                const int wb = sub * wps;
                int add = run[cur * E + e];
                for (int s2 = 0; s2 < sub; ++s2) add += subsum[s2 * E + e];
#pragma unroll
                for (int j = 0; j < kWarps; ++j)
                    if (j < wps) gmask[(wb + j) * E + e] += (uint32_t)add;
                if (sub == kSub - 1) run[nxt * E + e] = add + subsum[sub * E + e];
            }
        }
        __syncthreads();
        if (!one_tile) {
#pragma unroll
            for (int k = 0; k < kMaxR; ++k)
                if (k < R && ek[k] >= 0) part[k] += (int)mymask[ek[k]];
        }
        if (!one_tile && active) {
            // several tiles: park the partial rank in pos until phase 3
#pragma unroll
            for (int k = 0; k < kMaxR; ++k)
                if (k < R) pos[(int64_t)g * R + k] = (ek[k] >= 0) ? part[k] : -1;
        }
        cur = nxt;
        __syncthreads();  // gmask is cleared again by the next tile
    }
    if (bad) atomicOr(flags, 1);
    if (cur != 0) {  // leave this block's histogram in run[0..E) for the other blocks
        for (int e = tid; e < E; e += kThreads) run[e] = run[E + e];
    }

    cluster.sync();  // every block's histogram, send counts and flags final

    // ---- phase 2: exchange through distributed shared memory ----------------
    // Every remote load of one item is issued before any of them is used.
    // Small blocks handle an expert and a send_counts entry per iteration so
    // that both sets of remote loads overlap; 1024-thread blocks (64
    // registers per thread) handle them in two loops.
    if constexpr (kThreads <= 256) {
        const bool smem_send = mode != kSendGlobalAtomics;
        const int n_e = (E + kThreads - 1) / kThreads;
        const int n_p = smem_send ? (N * N + C * kThreads - 1) / (C * kThreads) : 0;
        const int iters = max(n_e, n_p);
        for (int it = 0; it < iters; ++it) {
            const int e = tid + it * kThreads;
            const int i = b * kThreads + tid + it * C * kThreads;
            const bool do_e = e < E;
            const bool do_p = smem_send && i < N * N;
            int s = 0, d = 0, b_lo = 0, b_hi = -1;
            if (do_p && T > 0) {  // T == 0: no tokens, the count is 0
                s = i / N;
                d = i - s * N;
                b_lo = (s * T) / per;
                b_hi = min(C - 1, ((s + 1) * T - 1) / per);
            }
            int ve[kMaxCluster], vp[kMaxCluster];
#pragma unroll
            for (int bb = 0; bb < kMaxCluster; ++bb) {
                ve[bb] = (do_e && bb < C) ? *cluster.map_shared_rank(run + e, bb) : 0;
                const int blk = b_lo + bb;
                vp[bb] = (blk <= b_hi) ? *cluster.map_shared_rank(ssend + (s - sfirst_tab[blk]) * N + d, blk) : 0;
            }
            if (do_e) {
                int base = 0, tot = 0;
#pragma unroll
                for (int bb = 0; bb < kMaxCluster; ++bb) {
                    tot += ve[bb];
                    if (bb < b) base += ve[bb];
                }
                sbase[e] = base;
                stot[e] = tot;
            }
            if (do_p) {
                int sum = 0;
#pragma unroll
                for (int bb = 0; bb < kMaxCluster; ++bb) sum += vp[bb];
                send_counts[i] = sum;
            }
        }
    } else {
        for (int e = tid; e < E; e += kThreads) {
            int v[kMaxCluster];
#pragma unroll
            for (int bb = 0; bb < kMaxCluster; ++bb)
                v[bb] = (bb < C) ? *cluster.map_shared_rank(run + e, bb) : 0;
            int base = 0, tot = 0;
#pragma unroll
            for (int bb = 0; bb < kMaxCluster; ++bb) {
                tot += v[bb];
                if (bb < b) base += v[bb];
            }
            sbase[e] = base;
            stot[e] = tot;
        }
        if (mode != kSendGlobalAtomics) {
            // send_counts[s][d]: add the staged counts of every block whose
            // token range meets source rank s
            for (int i = b * kThreads + tid; i < N * N; i += C * kThreads) {
                const int s = i / N, d = i - (i / N) * N;
                int b_lo = 0, b_hi = -1;  // T == 0: no tokens, the count is 0
                if (T > 0) {
                    b_lo = (s * T) / per;
                    b_hi = min(C - 1, ((s + 1) * T - 1) / per);
                }
                int v[kMaxCluster];
#pragma unroll
                for (int bb = 0; bb < kMaxCluster; ++bb) {
                    const int blk = b_lo + bb;
                    v[bb] = (blk <= b_hi) ? *cluster.map_shared_rank(ssend + (s - sfirst_tab[blk]) * N + d, blk) : 0;
                }
                int sum = 0;
#pragma unroll
                for (int bb = 0; bb < kMaxCluster; ++bb) sum += v[bb];
                send_counts[i] = sum;
            }
        }
    }
    int any_bad = 0;
    if (tid < C) any_bad = *cluster.map_shared_rank(flags, tid);
    any_bad = __syncthreads_or(any_bad);
    // this block reads no remote shared memory after this point; it waits for
    // the others to say the same only before exiting
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");

    // exclusive scan of stot over experts: thread t sums the ipt consecutive
    // experts [t*ipt, t*ipt + ipt), then a two-level warp scan
    {
        constexpr int kIptMax = (1024 + kThreads - 1) / kThreads;  // E <= 1024
        const int ipt = (E + kThreads - 1) / kThreads;
        int v[kIptMax];
        int local = 0;
#pragma unroll
        for (int i = 0; i < kIptMax; ++i) {
            const int e = tid * ipt + i;
            v[i] = (i < ipt && e < E) ? stot[e] : 0;
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
        for (int i = 0; i < kIptMax; ++i) {
            const int e = tid * ipt + i;
            if (i < ipt && e < E) {
                eoff[e] = run_e;
                run_e += v[i];
                if (e == E - 1) eoff[E] = run_e;
            }
        }
        __syncthreads();
    }

    // does some rank receive more rows than its region holds?
    int over = 0;
    for (int d = tid; d < N; d += kThreads)
        if (eoff[(d + 1) * L] - eoff[d * L] > cap) over = 1;
    over = __syncthreads_or(over);
    // first row of this block's pairs of expert e and the rows its rank's
    // region has left from there; without overflow the first row is folded
    // into the group prefixes so that phase 3 reads one word per pair
    for (int e = tid; e < E; e += kThreads) {
        const int d = e / L;
        const int local = eoff[e] - eoff[d * L] + sbase[e];
        fin[e] = make_int2(d * cap + local, cap - local);
        if (!over && one_tile) {
#pragma unroll
            for (int w = 0; w < kWarps; ++w) gmask[w * E + e] += (uint32_t)(d * cap + local);
        }
    }
    __syncthreads();

    if (b == 0) {
        for (int e = tid; e < E; e += kThreads) {
            expert_counts[e] = stot[e];
            expert_offsets[e] = eoff[e];
        }
        if (tid == 0) expert_offsets[E] = eoff[E];
        for (int d = tid; d < N; d += kThreads) {
            rank_counts[d] = eoff[(d + 1) * L] - eoff[d * L];
            rank_offsets[d] = eoff[d * L];
        }
        if (tid == 0) {
            rank_offsets[N] = eoff[E];
            *status = any_bad ? MOE_ERR_INVALID_ARG : (over ? MOE_ERR_CAPACITY : MOE_OK);
        }
    }

    // ---- phase 3: final rows --------------------------------------------------
    if (one_tile) {
        const int g = lo + tid;
        const bool active = g < hi;
        uint32_t *mymask = gmask + warp * E;  // group prefixes of this warp's group
        if (active) {
            int out[kMaxR];
#pragma unroll
            for (int k = 0; k < kMaxR; ++k) {
                out[k] = -1;
                if (k < R && ek[k] >= 0) {
                    if (!over) {
                        out[k] = (int)mymask[ek[k]] + part[k];
                    } else {
                        const int2 f = fin[ek[k]];
                        const int pr = (int)mymask[ek[k]] + part[k];
                        out[k] = (pr < f.y) ? f.x + pr : -1;
                    }
                }
            }
            int32_t *prow = pos + (int64_t)g * R;
            if ((R & 3) == 0 && (reinterpret_cast<uintptr_t>(pos) & 15) == 0) {
#pragma unroll
                for (int k = 0; k < kMaxR; k += 4)
                    if (k < R)
                        *reinterpret_cast<int4 *>(prow + k) = make_int4(out[k], out[k + 1], out[k + 2], out[k + 3]);
            } else {
#pragma unroll
                for (int k = 0; k < kMaxR; ++k)
                    if (k < R) prow[k] = out[k];
            }
        }
    } else {
        for (int t0 = lo; t0 < hi; t0 += kThreads) {
            const int g = t0 + tid;
            if (g >= hi) continue;
            for (int k = 0; k < R; ++k) {
                const int pr = pos[(int64_t)g * R + k];  // parked by this thread in phase 1
                if (pr < 0) continue;
                const int2 f = fin[__ldg(topk_idx + (int64_t)g * R + k)];
                pos[(int64_t)g * R + k] = (pr < f.y) ? f.x + pr : -1;
            }
        }
    }
    // keep this block's shared memory alive until every block has finished
    // reading it
    asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}

// Largest cluster (<= 16 blocks) of this kernel with this much shared memory
// that the current device can co-schedule; 0 if none.  Cached per host
// thread, device and context for the largest shared-memory request seen.
template <int kThreads, int kMaxR>
int max_cluster_blocks(size_t smem_bytes) {
    static thread_local int cached_dev = -1;
    static thread_local unsigned long long cached_ctx = 0;
    static thread_local size_t cached_smem = 0;
    static thread_local int cached_c = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const unsigned long long ctx = context_key();
    if (dev == cached_dev && ctx != 0 && ctx == cached_ctx && smem_bytes <= cached_smem) return cached_c;
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
    cached_ctx = context_key();  // the attribute calls above created the context if needed
    cached_smem = smem_bytes;
    cached_c = best;
    return best;
}

template <int kThreads, int kMaxR>
cudaError_t launch_count(const int32_t *topk_idx, int N, int T, int E, int R, int cap,
                         int32_t *expert_counts, int32_t *expert_offsets, int32_t *rank_counts,
                         int32_t *rank_offsets, int32_t *send_counts, int32_t *pos,
                         int32_t *status, cudaStream_t stream) {
    const CountSmem lay = count_smem_layout(E, kThreads / 32, count_ksub(kThreads, E));
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
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = c;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1] = pdl_attribute();
    cfg.attrs = attr;
    cfg.numAttrs = 2;
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
    // cap < 2^31 / N is checked by the caller
    const int icap = (int)cap;
    const int64_t NT = (int64_t)N * T;
    // R <= 8 keeps the per-pair state of a thread in registers.  Batches that
    // fit one token per thread in a 16-block cluster of 256-thread blocks use
    // that shape (less serial work per SM); larger ones use 1024-thread
    // blocks; R > 8 uses 512-thread blocks.
    if (R <= 8) {
        if (NT <= 16 * 256) {
            const CountSmem lay = count_smem_layout(E, 256 / 32, count_ksub(256, E));
            if (max_cluster_blocks<256, 8>((size_t)lay.bytes) * 256 >= NT)
                return launch_count<256, 8>(topk_idx, N, T, E, R, icap, expert_counts, expert_offsets,
                                            rank_counts, rank_offsets, send_counts, pos, status, stream);
        }
        return launch_count<1024, 8>(topk_idx, N, T, E, R, icap, expert_counts, expert_offsets,
                                     rank_counts, rank_offsets, send_counts, pos, status, stream);
    }
    return launch_count<512, 32>(topk_idx, N, T, E, R, icap, expert_counts, expert_offsets,
                                 rank_counts, rank_offsets, send_counts, pos, status, stream);
}

}  // namespace moe
