// Decode-fused dispatch: route top-k, dispatch count and dispatch pack in
// ONE cooperative launch.
//
// "Hosting Qwen on Blackwell", section "Expert parallel": for decode the
// whole dispatch kernel is fused into one, while prefill splits it into
// several kernels because routing needs fewer blocks than the rest.
// "Lower latency and higher throughput with multi-node DeepSeek
// deployment", section "CUDA Graph": a fixed number of kernels splits the
// dynamically routed work.  The method of each phase is that of the
// separate kernels (route_topk.cu, dispatch_count.cu, dispatch_pack.cu) and
// the outputs are identical to theirs.
//
// Phases, separated by grid-wide barriers (all blocks are co-resident: the
// kernel is launched cooperatively):
//   1. route: every warp routes tokens (grid-stride), writing topk_idx/w;
//   2. count: the first CB = ceil(N*T/256) <= 16 blocks each own 256
//      consecutive tokens (one per thread), build their histograms in shared
//      memory as the count kernel does, publish them to the workspace, meet
//      at a barrier of their own, then each derives offsets, send counts and
//      the rows of its tokens;
//   3. pack: every block copies token rows (grid-stride) to their rows.
// x is an input, not written here: while the count blocks work, the other
// blocks (idle until the second barrier) ask for the x rows to be brought
// into L2 (bulk prefetch, evict-last, at most half of the L2), so that
// pack reads them from L2, and the packed rows are stored with an
// evict-first hint so that they do not push those rows out.  Measured on
// the DeepSeek-V3 decode batch (GB300, L2 flushed before each launch):
// pack phase 65 -> 56 us, count phase 12 -> 18 us (its L2 accesses queue
// behind the prefetch), whole kernel 118 -> 115 us; issued before routing
// instead, the prefetches slowed routing from 5.5 to 14 us.  Every barrier
// wait is bounded: a wait that gives up makes the status word
// MOE_ERR_TIMEOUT and the kernel returns.
//
// Scope: decode batches (N*T <= 4096), T % 32 == 0, R <= 8, E <= 512; the
// host rejects anything else with MOE_ERR_UNSUPPORTED (use the three
// separate calls).
#include <mutex>

#include <cuda.h>  // CUcontext and CUresult only: the two driver calls are fetched at run time

#include "mem_ops.cuh"
#include "moe_internal.cuh"
#include "route_impl.cuh"

namespace moe {
namespace {

constexpr int kFThreads = 256;  // 8 warps; one token per thread in the count
constexpr int kFWarps = kFThreads / 32;
constexpr int kMaxCountBlocks = 16;
constexpr int kFMaxR = 8;
constexpr int kSendStage = 2048;               // ints of send staging per count block
constexpr long long kSpinLimit = 1ll << 20;    // polls per barrier wait (about a second)

// workspace words; the grid barrier, the count barrier and the error word
// sit in different 128-byte lines so that blocks polling one do not slow the
// atomics of another
constexpr int kWsGridArrive = 0, kWsGridGen = 1, kWsCntArrive = 32, kWsCntGen = 33, kWsError = 64;
constexpr int kWsHeader = 96;

struct FusedParams {
    const float *logits;
    const float *bias;
    int score_fn, renormalize;
    const uint4 *x;
    const float *x_scales;
    int nvec, spr;
    int N, T, E, R, cap, CB;
    int64_t rows_total;
    int64_t pf_rows;  // x rows [0, pf_rows) are prefetched into L2 (0: none)
    int32_t *topk_idx;
    float *topk_w;
    int32_t *expert_counts, *expert_offsets, *rank_counts, *rank_offsets, *send_counts, *pos,
        *status;
    uint4 *packed_x;
    float *packed_scales;
    int32_t *packed_src;
    int *ws;
};

__device__ __forceinline__ int ld_acquire(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Barrier of `nblocks` blocks on (arrive, gen) words of the workspace.
// Returns false when the wait gave up or another block recorded an error.
// Polls *word until it differs from `value`, at most `limit` times with a
// growing sleep between polls (32 ns doubling to 512 ns); false if it gave up.
__device__ bool wait_while_equal(const int *word, int value, long long limit) {
    long long it = 0;
    unsigned ns = 32;
    while (ld_acquire(word) == value) {
        if (++it > limit) return false;
        __nanosleep(ns);
        if (ns < 512) ns <<= 1;  // back off: hundreds of blocks poll one word
    }
    return true;
}

__device__ bool bounded_barrier(int *arrive, int *gen, int nblocks, int *err) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        const int g0 = ld_acquire(gen);
        __threadfence();  // this block's writes before its arrival
        if (atomicAdd(arrive, 1) == nblocks - 1) {
            atomicExch(arrive, 0);
            __threadfence();
            atomicAdd(gen, 1);  // release the others
        } else if (!wait_while_equal(gen, g0, kSpinLimit)) {
            atomicCAS(err, 0, MOE_ERR_TIMEOUT);
            ok = 0;
        }
        __threadfence();
        s_ok = ok && ld_acquire(err) == 0;
    }
    __syncthreads();
    return s_ok != 0;
}

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

struct FusedSmem {
    int gmask, run, base, tot, eoff, fin, send, misc, bytes;
};

// Every section starts on a 16-byte boundary (fin is read as int2).
__host__ __device__ inline FusedSmem fused_smem_layout(int E) {
    FusedSmem s;
    int o = 0;
    auto take = [&o](int bytes) {
        const int at = o;
        o += (bytes + 15) & ~15;
        return at;
    };
    s.gmask = take(kFWarps * E * 4);  // group masks, then group prefixes
    s.run = take(E * 4);              // this block's histogram
    s.base = take(E * 4);             // pairs in earlier count blocks
    s.tot = take(E * 4);              // pairs in all count blocks
    s.eoff = take((E + 1) * 4);       // exclusive scan of tot
    s.fin = take(E * 8);              // first row / rows left per expert
    s.send = take(kSendStage * 4);    // send counts of this block's source ranks
    s.misc = take(64 * 4);            // flags and scan partials
    s.bytes = o;
    return s;
}

constexpr int kPackU = 4;  // 16-byte vectors of a row per thread in flight (pack)

// 3 co-resident blocks per SM.  4 (64 registers per thread, no spills for
// up to 8 experts per lane) routes a 4096-token batch in one pass, but the
// whole kernel took longer on the DeepSeek-V3 decode batch (123 vs 115 us).
template <int J, bool kVec4>
__global__ void __launch_bounds__(kFThreads, 3)
dispatch_fused_kernel(FusedParams P) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_pos[kFMaxR];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int NT = P.N * P.T;
    int *err = P.ws + kWsError;

    // ---- phase 1: route ------------------------------------------------------
    for (int64_t g = (int64_t)blockIdx.x * kFWarps + warp; g < NT; g += (int64_t)gridDim.x * kFWarps)
        route_impl::route_token<J, kVec4>(P.logits, P.bias, g, P.E, P.R, P.score_fn,
                                          P.renormalize, P.topk_idx, P.topk_w, lane);
    bool alive = bounded_barrier(P.ws + kWsGridArrive, P.ws + kWsGridGen, gridDim.x, err);

    // ---- phase 2: count (blocks 0 .. CB-1) -------------------------------------
    const int b = blockIdx.x;
    // meanwhile the other blocks prefetch x, one row per lane of warp 0
    const int nb = (int)gridDim.x - P.CB;
    if (alive && b >= P.CB && warp == 0) {
        const uint64_t keep = l2_policy_evict_last();
        for (int64_t r = (b - P.CB) + (int64_t)lane * nb; r < P.pf_rows; r += 32ll * nb)
            prefetch_l2(P.x + r * P.nvec, (uint32_t)P.nvec * 16u, keep);
    }
    if (alive && b < P.CB) {
        const int E = P.E, N = P.N, T = P.T, R = P.R, L = E / N, CB = P.CB;
        const FusedSmem lay = fused_smem_layout(E);
        uint32_t *gmask = reinterpret_cast<uint32_t *>(smem + lay.gmask);
        int *run = reinterpret_cast<int *>(smem + lay.run);
        int *sbase = reinterpret_cast<int *>(smem + lay.base);
        int *stot = reinterpret_cast<int *>(smem + lay.tot);
        int *eoff = reinterpret_cast<int *>(smem + lay.eoff);
        int2 *fin = reinterpret_cast<int2 *>(smem + lay.fin);
        int *ssend = reinterpret_cast<int *>(smem + lay.send);
        int *misc = reinterpret_cast<int *>(smem + lay.misc);  // [0] bad, [1] over, [16..48) scan
        int *ws_hist = P.ws + kWsHeader;                            // [CB][E]
        int *ws_send = ws_hist + kMaxCountBlocks * E;               // [CB][kSendStage]
        int *ws_bad = ws_send + kMaxCountBlocks * kSendStage;       // [CB]

        const int lo = b * kFThreads, hi = min(NT, lo + kFThreads);
        const int s_first = lo / T;
        const int span = (hi - 1) / T - s_first + 1;
        for (int i = tid; i < kFWarps * E; i += kFThreads) gmask[i] = 0u;
        for (int i = tid; i < E; i += kFThreads) run[i] = 0;
        for (int i = tid; i < span * N; i += kFThreads) ssend[i] = 0;
        if (tid == 0) misc[0] = 0;
        __syncthreads();

        const int g = lo + tid;
        const bool active = g < hi;
        int ek[kFMaxR], part[kFMaxR];
#pragma unroll
        for (int k = 0; k < kFMaxR; ++k) {
            ek[k] = -1;
            part[k] = 0;
            if (k < R && active) ek[k] = __ldcg(P.topk_idx + (int64_t)g * R + k);  // written in phase 1
        }
        bool bad = false;
#pragma unroll
        for (int k = 0; k < kFMaxR; ++k) {
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
        uint32_t *mymask = gmask + warp * E;
#pragma unroll
        for (int k = 0; k < kFMaxR; ++k)
            if (k < R && ek[k] >= 0) atomicOr(mymask + ek[k], 1u << lane);
        __syncwarp();
        const unsigned lt = lanemask_lt();
#pragma unroll
        for (int k = 0; k < kFMaxR; ++k)
            if (k < R && ek[k] >= 0) part[k] = __popc(mymask[ek[k]] & lt);
        if (bad) atomicOr(misc, 1);
        __syncthreads();
        // group prefixes, histogram and send counts (groups never straddle
        // source ranks: T % 32 == 0)
        for (int e = tid; e < E; e += kFThreads) {
            int c[kFWarps];
#pragma unroll
            for (int w = 0; w < kFWarps; ++w) c[w] = __popc(gmask[w * E + e]);
            int r = 0, acc = 0, s_cur = s_first;
            const int d = e / L;
#pragma unroll
            for (int w = 0; w < kFWarps; ++w) {
                gmask[w * E + e] = (uint32_t)r;
                r += c[w];
                const int gw = lo + 32 * w;
                if (gw < hi) {
                    if (gw / T != s_cur) {
                        if (acc) atomicAdd(ssend + (s_cur - s_first) * N + d, acc);
                        acc = 0;
                        s_cur = gw / T;
                    }
                    acc += c[w];
                }
            }
            if (acc) atomicAdd(ssend + (s_cur - s_first) * N + d, acc);
            run[e] = r;
        }
        __syncthreads();
        int any_bad = 0;
        if (CB == 1) {
            // a single count block: its own histogram and send counts are final
            for (int e = tid; e < E; e += kFThreads) {
                sbase[e] = 0;
                stot[e] = run[e];
            }
            for (int i = tid; i < N * N; i += kFThreads) {
                const int s = i / N, d = i - (i / N) * N;
                P.send_counts[i] = (s >= s_first && s < s_first + span) ? ssend[(s - s_first) * N + d] : 0;
            }
            any_bad = __syncthreads_or(misc[0]);
        } else {
            // publish this block's histogram, send counts and flag
            for (int e = tid; e < E; e += kFThreads) ws_hist[b * E + e] = run[e];
            for (int i = tid; i < span * N; i += kFThreads) ws_send[b * kSendStage + i] = ssend[i];
            if (tid == 0) ws_bad[b] = misc[0];
            alive = bounded_barrier(P.ws + kWsCntArrive, P.ws + kWsCntGen, CB, err);
            if (alive) {
                // every workspace load of an item is issued before any is used
                for (int e = tid; e < E; e += kFThreads) {
                    int v[kMaxCountBlocks];
#pragma unroll
                    for (int bb = 0; bb < kMaxCountBlocks; ++bb)
                        v[bb] = (bb < CB) ? __ldcg(ws_hist + bb * E + e) : 0;
                    int base = 0, tot = 0;
#pragma unroll
                    for (int bb = 0; bb < kMaxCountBlocks; ++bb) {
                        tot += v[bb];
                        if (bb < b) base += v[bb];
                    }
                    sbase[e] = base;
                    stot[e] = tot;
                }
                // send_counts rows, split over the count blocks
                for (int i = b * kFThreads + tid; i < N * N; i += CB * kFThreads) {
                    const int s = i / N, d = i - (i / N) * N;
                    const int b_lo = (s * T) / kFThreads;
                    const int b_hi = min(CB - 1, ((s + 1) * T - 1) / kFThreads);
                    int v[kMaxCountBlocks];
#pragma unroll
                    for (int j = 0; j < kMaxCountBlocks; ++j) {
                        const int bb = b_lo + j;
                        v[j] = (bb <= b_hi)
                                   ? __ldcg(ws_send + bb * kSendStage + (s - (bb * kFThreads) / T) * N + d)
                                   : 0;
                    }
                    int sum = 0;
#pragma unroll
                    for (int j = 0; j < kMaxCountBlocks; ++j) sum += v[j];
                    P.send_counts[i] = sum;
                }
                for (int bb = tid; bb < CB; bb += kFThreads) any_bad |= __ldcg(ws_bad + bb);
            }
            any_bad = __syncthreads_or(any_bad);
        }
        if (alive) {
            // exclusive scan of stot over experts (E <= 512: 2 per thread)
            {
                const int ipt = (E + kFThreads - 1) / kFThreads;
                int v0 = 0, v1 = 0;
                if (tid * ipt < E) v0 = stot[tid * ipt];
                if (ipt > 1 && tid * ipt + 1 < E) v1 = stot[tid * ipt + 1];
                const int local = v0 + v1;
                int x = local;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, x, off);
                    if (lane >= off) x += y;
                }
                int *wsum = misc + 16;
                if (lane == 31) wsum[warp] = x;
                __syncthreads();
                if (warp == 0) {
                    int sv = (lane < kFWarps) ? wsum[lane] : 0;
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const int y = __shfl_up_sync(0xffffffffu, sv, off);
                        if (lane >= off) sv += y;
                    }
                    if (lane < kFWarps) wsum[lane] = sv;
                }
                __syncthreads();
                int start = x - local + (warp > 0 ? wsum[warp - 1] : 0);
                if (tid * ipt < E) {
                    eoff[tid * ipt] = start;
                    start += v0;
                    if (tid * ipt == E - 1) eoff[E] = start;
                }
                if (ipt > 1 && tid * ipt + 1 < E) {
                    eoff[tid * ipt + 1] = start;
                    start += v1;
                    if (tid * ipt + 1 == E - 1) eoff[E] = start;
                }
                __syncthreads();
            }
            int over = 0;
            for (int d = tid; d < N; d += kFThreads)
                if (eoff[(d + 1) * L] - eoff[d * L] > P.cap) over = 1;
            over = __syncthreads_or(over);
            for (int e = tid; e < E; e += kFThreads) {
                const int d = e / L;
                const int local = eoff[e] - eoff[d * L] + sbase[e];
                fin[e] = make_int2(d * P.cap + local, P.cap - local);
                if (!over) {
#pragma unroll
                    for (int w = 0; w < kFWarps; ++w) gmask[w * E + e] += (uint32_t)(d * P.cap + local);
                }
            }
            __syncthreads();
            if (b == 0) {
                for (int e = tid; e < E; e += kFThreads) {
                    P.expert_counts[e] = stot[e];
                    P.expert_offsets[e] = eoff[e];
                }
                for (int d = tid; d < N; d += kFThreads) {
                    P.rank_counts[d] = eoff[(d + 1) * L] - eoff[d * L];
                    P.rank_offsets[d] = eoff[d * L];
                }
                if (tid == 0) {
                    P.expert_offsets[E] = eoff[E];
                    P.rank_offsets[N] = eoff[E];
                    *P.status = any_bad ? MOE_ERR_INVALID_ARG : (over ? MOE_ERR_CAPACITY : MOE_OK);
                }
            }
            if (active) {
#pragma unroll
                for (int k = 0; k < kFMaxR; ++k) {
                    if (k < R) {
                        int out = -1;
                        if (ek[k] >= 0) {
                            const int pr = (int)mymask[ek[k]] + part[k];
                            if (!over) out = pr;
                            else {
                                const int2 f = fin[ek[k]];
                                const int rel = pr;  // prefix without the expert start
                                out = (rel < f.y) ? f.x + rel : -1;
                            }
                        }
                        P.pos[(int64_t)g * R + k] = out;
                    }
                }
            }
        }
    }
    alive = bounded_barrier(P.ws + kWsGridArrive, P.ws + kWsGridGen, gridDim.x, err) && alive;

    // ---- phase 3: pack --------------------------------------------------------
    if (alive) {
        const uint64_t stream_out = l2_policy_evict_first();
        for (int64_t g = blockIdx.x; g < NT; g += gridDim.x) {
            if (tid < P.R) {
                const int p = __ldcg(P.pos + g * P.R + tid);  // written in phase 2
                const bool ok = p >= 0 && (int64_t)p < P.rows_total;
                s_pos[tid] = ok ? p : -1;
                if (ok) P.packed_src[p] = (int32_t)(g * P.R + tid);
            }
            __syncthreads();
            for (int c0 = tid; c0 < P.nvec; c0 += kFThreads * kPackU) {
                uint4 v[kPackU];
#pragma unroll
                for (int u = 0; u < kPackU; ++u) {
                    const int c = c0 + u * kFThreads;
                    if (c < P.nvec) v[u] = ld_stream(P.x + g * P.nvec + c);
                }
                for (int k = 0; k < P.R; ++k) {
                    const int p = s_pos[k];
                    if (p < 0) continue;
                    uint4 *dst = P.packed_x + (int64_t)p * P.nvec;
#pragma unroll
                    for (int u = 0; u < kPackU; ++u) {
                        const int c = c0 + u * kFThreads;
                        if (c < P.nvec) st_evict_first(dst + c, v[u], stream_out);
                    }
                }
            }
            if (P.spr > 0) {
                for (int i = tid; i < P.R * P.spr; i += kFThreads) {
                    const int k = i / P.spr, j = i - k * P.spr;
                    const int p = s_pos[k];
                    if (p >= 0) P.packed_scales[(int64_t)p * P.spr + j] = __ldg(P.x_scales + g * P.spr + j);
                }
            }
            __syncthreads();
        }
    }
    if (!alive && blockIdx.x == 0 && tid == 0) *P.status = MOE_ERR_TIMEOUT;
}

template <int J, bool kVec4>
cudaError_t launch_fused_jv(FusedParams P, cudaStream_t stream) {
    auto kern = dispatch_fused_kernel<J, kVec4>;
    const size_t smem = (size_t)fused_smem_layout(P.E).bytes;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kFThreads, smem);
    if (e != cudaSuccess) return e;
    const int sms = sm_count();
    if (per_sm < 1 || sms < 1) return cudaErrorNotSupported;
    int grid = sms * per_sm;
    const int NT = P.N * P.T;
    const int need = (NT + kFWarps - 1) / kFWarps;  // one routing warp per token is plenty
    if (grid > need) grid = need;
    if (grid < P.CB) return cudaErrorNotSupported;
    // L2 prefetch of x: rows of at most 64 KB filling at most half the L2
    const int64_t row_bytes = (int64_t)P.nvec * 16;
    P.pf_rows = row_bytes <= 65536 ? (l2_bytes() / 2) / row_bytes : 0;
    if (P.pf_rows > NT) P.pf_rows = NT;
    if (P.pf_rows < 0) P.pf_rows = 0;
    e = cudaMemsetAsync(P.ws, 0, kWsHeader * sizeof(int), stream);  // barrier words
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kFThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, P);
}

template <int J>
cudaError_t launch_fused_j(FusedParams P, cudaStream_t stream) {
    if constexpr (J % 4 == 0) {
        if (P.E % 4 == 0 && (reinterpret_cast<uintptr_t>(P.logits) & 15) == 0)
            return launch_fused_jv<J, true>(P, stream);
    }
    return launch_fused_jv<J, false>(P, stream);
}

}  // namespace

int64_t fused_workspace_bytes(int E) {
    return (int64_t)(kWsHeader + kMaxCountBlocks * E + kMaxCountBlocks * kSendStage + kMaxCountBlocks) *
           (int64_t)sizeof(int);
}

// Empty string when the fused kernel handles these dimensions, else why not.
namespace {
// Limits of the cooperative kernel ("" when it can run the batch).
const char *cooperative_unsupported(int N, int T, int E, int R) {
    const int64_t NT = (int64_t)N * T;
    if (R > kFMaxR) return "R > 8";
    if (E > 512) return "E > 512";
    if (T % 32 != 0) return "T is not a multiple of 32";
    if (NT > (int64_t)kMaxCountBlocks * kFThreads) return "N*T > 4096 (not a decode batch)";
    if (NT > 0 && (int64_t)(kFThreads / T + 2) * N > kSendStage) return "too many ranks per count block";
    return "";
}
}  // namespace

// A batch runs fused if the single-cluster kernel takes it (no limit on T
// or R beyond the interface's) or else the cooperative kernel does.
const char *fused_unsupported(int N, int T, int E, int R, int64_t row_bytes) {
    if ((int64_t)N * T == 0) return "";  // empty batch: only the (zero) counts are written
    if (dispatch_small_eligible((int64_t)N * T, E, R, row_bytes)) return "";
    return cooperative_unsupported(N, T, E, R);
}

cudaError_t launch_dispatch_fused(const float *logits, const float *bias, int score_fn, int renormalize,
                                  const void *x, const float *x_scales, int N, int T, int E, int R,
                                  int64_t row_bytes, int spr, int64_t cap, int32_t *topk_idx,
                                  float *topk_w, int32_t *expert_counts, int32_t *expert_offsets,
                                  int32_t *rank_counts, int32_t *rank_offsets, int32_t *send_counts,
                                  int32_t *pos, int32_t *status, void *packed_x, float *packed_scales,
                                  int32_t *packed_src, void *workspace, cudaStream_t stream) {
    // An empty batch has nothing to route or pack: the count step alone
    // writes its zero counts and offsets and MOE_OK, as the separate calls do.
    if ((int64_t)N * T == 0)
        return launch_dispatch_count(topk_idx, N, T, E, R, cap, expert_counts, expert_offsets, rank_counts,
                                     rank_offsets, send_counts, pos, status, stream);
    // Small batches: one thread-block cluster, no grid barriers and no
    // workspace (the cooperative kernel below handles everything else, and
    // takes over if the device cannot schedule the cluster).
    if (dispatch_small_eligible((int64_t)N * T, E, R, row_bytes)) {
        cudaError_t e = launch_dispatch_small(logits, bias, score_fn, renormalize, x, x_scales, N, T, E, R,
                                              row_bytes, spr, cap, topk_idx, topk_w, expert_counts,
                                              expert_offsets, rank_counts, rank_offsets, send_counts, pos,
                                              status, packed_x, packed_scales, packed_src, stream);
        if (e != cudaErrorNotSupported) return e;
        // the device cannot schedule the cluster: the cooperative kernel, if
        // the batch is within its limits
        if (cooperative_unsupported(N, T, E, R)[0] != '\0') return cudaErrorNotSupported;
    }
    FusedParams P;
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
    P.CB = (int)(((int64_t)N * T + kFThreads - 1) / kFThreads);
    if (P.CB < 1) P.CB = 1;
    P.rows_total = (int64_t)N * cap;
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
    P.ws = reinterpret_cast<int *>(workspace);
    const int need = (E + 31) / 32;
    // the same experts per lane as the route kernel, so that the softmax
    // denominator is summed in the same order and the weights agree bit for bit
    if (need <= 1) return launch_fused_j<1>(P, stream);
    if (need <= 2) return launch_fused_j<2>(P, stream);
    if (need <= 4) return launch_fused_j<4>(P, stream);
    if (need <= 8) return launch_fused_j<8>(P, stream);
    if (need <= 12) return launch_fused_j<12>(P, stream);
    return launch_fused_j<16>(P, stream);
}

}  // namespace moe

// ---- self-test of the bounded wait -----------------------------------------
//
// One thread waits, through the same bounded poll as the grid barriers, for
// status[1] to become nonzero; status[0] gets MOE_OK if it did and
// MOE_ERR_TIMEOUT if the wait gave up.  Nothing in the library writes
// status[1], so unless the caller set it beforehand the wait runs out: this
// shows on a given GPU that a wait which is never satisfied ends with a
// status the host can read, and leaves the context usable.
namespace moe {
namespace {
__global__ void selftest_wait_kernel(int *status, long long polls) {
    if (threadIdx.x == 0 && blockIdx.x == 0)
        status[0] = wait_while_equal(status + 1, 0, polls) ? MOE_OK : MOE_ERR_TIMEOUT;
}
}  // namespace

cudaError_t launch_selftest_wait(int32_t *status, long long polls, cudaStream_t stream) {
    selftest_wait_kernel<<<1, 32, 0, stream>>>(status, polls);
    return cudaGetLastError();
}
}  // namespace moe

// ---- allocation-free variant -------------------------------------------------
//
// Some callers cannot allocate device memory at the point where they
// dispatch: a plug-in running inside another framework's execution loop has
// no allocator of its own, and serving code whose memory is fixed at
// start-up must not call cudaMalloc on its hot path (it synchronises the
// device and can fail under memory pressure).  For them the fused dispatch
// can use scratch that lives in the library itself: a fixed array in device
// memory, reserved on every GPU that loads the library for as long as the
// process runs.  Its size covers the workspace of every batch the fused
// kernel accepts (E <= 512 needs at most 164,288 bytes).
namespace moe {

constexpr int64_t kStaticScratchBytes = 192 * 1024;
static __device__ __align__(256) unsigned char g_fused_static_scratch[kStaticScratchBytes];

namespace {
constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mutex;

// The array's address belongs to the CUDA context the library's module was
// loaded into.  After cudaDeviceReset (or any other end of the primary
// context) the module is loaded again into a new context, possibly at
// another address, so the cached address is keyed on the context's unique
// id as well as on the device.
struct ScratchEntry {
    void *addr;
    unsigned long long ctx_id;
};
ScratchEntry g_scratch[kMaxScratchDevices] = {};

// Driver functions fetched through the runtime (no link against libcuda).
typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;
bool g_driver_fns_looked_up = false;

// Unique id of the calling thread's current context; false if there is
// none yet or the driver cannot say.
bool current_context_id(unsigned long long *id) {
    if (!g_driver_fns_looked_up) {
        g_driver_fns_looked_up = true;
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f);
        cudaGetLastError();
    }
    if (g_ctx_get_current == nullptr || g_ctx_get_id == nullptr) return false;
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return false;
    return g_ctx_get_id(ctx, id) == CUDA_SUCCESS;
}
}  // namespace

int64_t fused_static_scratch_bytes() { return kStaticScratchBytes; }

// Device address of the scratch array in the current device's context.  In
// host code the array's name only stands in for it, so the address is
// looked up with the device current, once per context, and cached.  Where
// the driver cannot identify the context the lookup is simply repeated on
// every call.
cudaError_t fused_static_scratch(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxScratchDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    if (have_id && g_scratch[dev].addr != nullptr && g_scratch[dev].ctx_id == id) {
        *out = g_scratch[dev].addr;
        return cudaSuccess;
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_fused_static_scratch);  // creates the context if needed
    if (e != cudaSuccess) return e;
    if (current_context_id(&id)) g_scratch[dev] = ScratchEntry{p, id};
    *out = p;
    return cudaSuccess;
}

}  // namespace moe
