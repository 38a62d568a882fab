// Dispatch pack through the tensor memory accelerator's bulk copies: each
// token row is brought into shared memory by one cp.async.bulk load and
// written to its R receive rows by R cp.async.bulk stores.
//
// Same contract as the vector kernel in dispatch_pack.cu ("Efficient and
// portable mixture-of-experts communication", section "Dispatch"; "Enabling
// trillion-parameter models on AWS EFA", section "Dispatch and combine").
// The vector kernel moves every byte through registers with 16-byte loads
// and stores, and at R = 8 its store stream saturates the load/store unit
// queues before HBM; here the copy engine moves whole rows, so one thread
// issues a 14 KB store with a single instruction.
//
// Pipeline (one warp per block, several blocks per SM): the block's tokens
// g = blockIdx.x + i * gridDim.x cycle through S shared-memory stages.  The
// row of token i is loaded into stage i % S (completion tracked by that
// stage's mbarrier, phase (i / S) & 1); once it has landed, lanes k < R
// issue the stores to pos[g][k] and commit one bulk group each; the stage
// of token i-1 is refilled with token i-1+S as soon as the stores of token
// i-1 have finished reading it (bulk wait_group.read 1).  Every mbarrier wait
// is bounded; a wait that gives up records MOE_ERR_TIMEOUT in the library's
// device error word, lets its own copies finish and leaves the kernel.
#include "moe_internal.cuh"
#include "pdl.cuh"

namespace moe {

__device__ int g_device_error = 0;  // sticky: first error recorded by a kernel

namespace {

constexpr int kBulkThreads = 32;
constexpr int kMaxStages = 4;
constexpr long long kWaitLimit = 1ll << 22;  // try_wait polls (each may suspend briefly)

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.b32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void bulk_store(void *dst, uint32_t src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(src),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__global__ void __launch_bounds__(kBulkThreads)
dispatch_pack_bulk_kernel(const unsigned char *__restrict__ x, const float *__restrict__ x_scales,
                          const int32_t *__restrict__ pos, int64_t NT, int R, int row_bytes,
                          int spr, int stages, int64_t rows_total, unsigned char *__restrict__ packed_x,
                          float *__restrict__ packed_scales, int32_t *__restrict__ packed_src) {
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ __align__(8) unsigned long long bars[kMaxStages];
    const int lane = threadIdx.x;
    const int64_t first = blockIdx.x, stride = gridDim.x;
    const int64_t n = (first < NT) ? (NT - 1 - first) / stride + 1 : 0;  // tokens of this block

    if (lane == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(smem_addr(&bars[s]), 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();
    grid_dependency_wait();  // pos comes from the count kernel
    grid_launch_dependents();

    auto stage_ptr = [&](int s) { return smem + (size_t)s * row_bytes; };
    auto load_token = [&](int64_t i) {  // lane 0 only
        const int s = (int)(i % stages);
        const uint32_t bar = smem_addr(&bars[s]);
        mbar_expect_tx(bar, (uint32_t)row_bytes);
        bulk_load(smem_addr(stage_ptr(s)), x + (first + i * stride) * (int64_t)row_bytes,
                  (uint32_t)row_bytes, bar);
    };
    if (lane == 0)
        for (int64_t i = 0; i < n && i < stages; ++i) load_token(i);

    bool failed = false;
    int64_t fail_at = 0;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t g = first + i * stride;
        const int s = (int)(i % stages);
        const uint32_t parity = (uint32_t)((i / stages) & 1);
        int p = -1;
        if (lane < R) {
            p = __ldg(pos + g * R + lane);
            if (p < 0 || (int64_t)p >= rows_total) p = -1;
        }
        // bounded wait for the row (every lane polls the same barrier)
        bool ok = false;
        for (long long it = 0; it < kWaitLimit && !ok; ++it) ok = mbar_try_wait(smem_addr(&bars[s]), parity);
        if (!__all_sync(0xffffffffu, ok)) {
            failed = true;
            fail_at = i;
            break;
        }
        if (p >= 0) {
            bulk_store(packed_x + (int64_t)p * row_bytes, smem_addr(stage_ptr(s)), (uint32_t)row_bytes);
            packed_src[p] = (int32_t)(g * R + lane);
        }
        bulk_commit();  // one group per lane and token (empty when nothing was stored)
        if (spr > 0) {
            // block scales: a few dozen floats per row, plain copies
            for (int k = 0; k < R; ++k) {
                const int pk = __shfl_sync(0xffffffffu, p, k);
                if (pk < 0) continue;
                for (int j = lane; j < spr; j += 32)
                    packed_scales[(int64_t)pk * spr + j] = __ldg(x_scales + g * spr + j);
            }
        }
        // refill the stage of token i-1 once its stores have read it
        if (i >= 1 && i - 1 + stages < n) {
            bulk_wait_read1();
            __syncwarp();
            if (lane == 0) load_token(i - 1 + stages);
        }
    }
    if (failed) {
        if (lane == 0) atomicCAS(&g_device_error, 0, MOE_ERR_TIMEOUT);
        // let the loads already issued land before the shared memory goes
        // away (again with a bound): tokens fail_at .. fail_at + stages - 2
        for (int64_t t = fail_at; t < n && t < fail_at + stages - 1; ++t) {
            bool ok = false;
            for (long long it = 0; it < kWaitLimit && !ok; ++it)
                ok = mbar_try_wait(smem_addr(&bars[t % stages]), (uint32_t)((t / stages) & 1));
        }
    }
    bulk_wait_all();  // stores complete before the block (and its shared memory) goes away
}

}  // namespace

// Read the device error word (MOE_OK if no kernel recorded one) and clear it.
cudaError_t take_device_error(int *err, cudaStream_t stream) {
    cudaError_t e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(err, g_device_error, sizeof(int));
    if (e != cudaSuccess) return e;
    const int zero = 0;
    return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int));
}

// Shared-memory stages for a row size (0: rows too large for this kernel).
int pack_bulk_stages(int64_t row_bytes) {
    if (row_bytes % 16 != 0 || row_bytes > 48 * 1024) return 0;
    int s = (int)((96 * 1024) / row_bytes);
    return s < 2 ? 0 : (s > kMaxStages ? kMaxStages : s);
}

cudaError_t launch_dispatch_pack_bulk(const void *x, const float *x_scales, const int32_t *pos,
                                      int64_t NT, int R, int64_t row_bytes, int scales_per_row,
                                      int64_t rows_total, void *packed_x, float *packed_scales,
                                      int32_t *packed_src, cudaStream_t stream) {
    if (NT == 0) return cudaSuccess;
    const int stages = pack_bulk_stages(row_bytes);
    if (stages == 0) return cudaErrorInvalidValue;
    const size_t smem = (size_t)stages * (size_t)row_bytes;
    // the attribute belongs to the current device's context: cached per
    // host thread, device and context
    static thread_local int configured_dev = -1;
    static thread_local unsigned long long configured_ctx = 0;
    static thread_local size_t configured = 0;
    int dev = 0;
    cudaError_t de = cudaGetDevice(&dev);
    if (de != cudaSuccess) return de;
    const unsigned long long ctx = context_key();
    if (dev != configured_dev || ctx == 0 || ctx != configured_ctx || smem > configured) {
        cudaError_t e = cudaFuncSetAttribute(dispatch_pack_bulk_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured_dev = dev;
        configured_ctx = context_key();
        configured = smem;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, dispatch_pack_bulk_kernel,
                                                                  kBulkThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) per_sm = 1;
    int64_t grid = (int64_t)sm_count() * per_sm;
    if (grid > NT) grid = NT;
    if (grid < 1) grid = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kBulkThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1] = {pdl_attribute()};
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, dispatch_pack_bulk_kernel, reinterpret_cast<const unsigned char *>(x),
                              x_scales, pos, NT, R, (int)row_bytes, scales_per_row, stages, rows_total,
                              reinterpret_cast<unsigned char *>(packed_x), packed_scales, packed_src);
}

}  // namespace moe
