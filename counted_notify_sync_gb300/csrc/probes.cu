// probes.cu -- latency and throughput probes that give the barrier its
// roofline: the round trip of one L2 atomic (and of one load, and of the
// arrive/poll pair) from a single thread, and the rate at which the L2 can
// apply same-address reductions.
#include <cooperative_groups.h>
#include <cuda_runtime.h>

#include <chrono>
#include <cstdint>

#include "cns.h"
#include "cns_device.cuh"
#include "cns_host.h"

namespace cns {

// A chain of `iters` operations where each address depends on the previous
// result (the count stays below 2^31, so the offset is always 0): nothing
// can overlap, each link costs one round trip.
__global__ void probe_rtt_kernel(int kind, int probe_cta, int iters, uint32_t *line, uint64_t *out)
{
    if (static_cast<int>(blockIdx.x) != probe_cta || threadIdx.x != 0)
        return;
    uint32_t x = 0;
    // one untimed link brings the line into L2
    x = atom_add_relaxed_gpu(line, 0u);
    const uint64_t t0 = globaltimer_ns();
    for (int i = 0; i < iters; ++i) {
        uint32_t *p = line + (x >> 31);
        if (kind == 0) {
            x = atom_add_relaxed_gpu(p, 1u);
        } else if (kind == 1) {
            x = ld_relaxed_gpu(p);
        } else {
            x = atom_add_release_gpu(p, 1u);
            x = ld_acquire_gpu(line + (x >> 31));
        }
    }
    const uint64_t t1 = globaltimer_ns();
    out[0] = t1 - t0;
    out[1] = smid() | (static_cast<uint64_t>(x & 0u) << 32);
}

// The ring-rotate rounds of CNS_WL_RING_ROTATE (one uint4 per CTA), separated
// by the CUDA runtime's own grid barrier (cooperative groups), for comparison.
__global__ void probe_grid_sync_kernel(uint4 *buf0, uint4 *buf1, int64_t rounds)
{
    cooperative_groups::grid_group grid = cooperative_groups::this_grid();
    const uint32_t P = gridDim.x, p = blockIdx.x;
    for (int64_t r = 0; r < rounds; ++r) {
        const uint4 *src = (r & 1) ? buf1 : buf0;
        uint4 *dst = (r & 1) ? buf0 : buf1;
        if (threadIdx.x == 0)
            dst[p] = src[(p + 1u == P) ? 0u : p + 1u];
        grid.sync();
    }
}

// Two CTAs hand a counted-notify signal back and forth `iters` times with the
// library's record and wait rules at scope S: CTA 0 records ADD 1 on count a
// and waits for count b to reach i + 1; CTA 1 waits for a to reach i + 1 and
// records ADD 1 on b.  out[0] = CTA 0's time for all iterations (two
// hand-offs each), out[1] = 0 or the first wait's failure (each wait is
// bounded by timeout_ns), out[2] / out[3] = the SMs of CTA 0 / CTA 1.
template <int S>
__global__ void probe_pingpong_kernel(int iters, uint32_t *a, uint32_t *b, uint64_t timeout_ns, uint64_t *out)
{
    if (threadIdx.x != 0 || blockIdx.x > 1)
        return;
    const bool first = blockIdx.x == 0;
    uint32_t *mine = first ? a : b;
    uint32_t *theirs = first ? b : a;
    int rc = CNS_SUCCESS;
    const uint64_t t0 = globaltimer_ns();
    for (int i = 0; i < iters && rc == CNS_SUCCESS; ++i) {
        const uint32_t want = static_cast<uint32_t>(i) + 1u;
        if (first) {
            cnt_record_scoped<S>(mine, CNS_REC_ADD, 1u);
            rc = cnt_wait_scoped<S>(theirs, CNS_WAIT_BIGGER_OR_EQUAL, want, false, timeout_ns, nullptr);
        } else {
            rc = cnt_wait_scoped<S>(theirs, CNS_WAIT_BIGGER_OR_EQUAL, want, false, timeout_ns, nullptr);
            if (rc == CNS_SUCCESS)
                cnt_record_scoped<S>(mine, CNS_REC_ADD, 1u);
        }
    }
    const uint64_t t1 = globaltimer_ns();
    if (first)
        out[0] = t1 - t0;
    if (rc != CNS_SUCCESS)
        out[1] = static_cast<uint64_t>(rc);
    out[2 + blockIdx.x] = smid();
}

// The cost of one fence.release.gpu by one thread, by what the thread did
// since its previous fence: out[0] nothing, out[1] a store to a line of the
// block homed on its own die, out[2] a store to a line of the other block
// (the two 4 KB blocks of `region` differ only in address bit 12, so they sit
// on different dies).  Each sample follows a quiet spell and a fence; the
// mean of `iters` samples, in ns, from %globaltimer around the fence alone.
__device__ __forceinline__ void spin_for_ns(uint64_t ns)
{
    const uint64_t s = globaltimer_ns();
    while (globaltimer_ns() - s < ns) {
    }
}

__global__ void probe_fence_kernel(uint32_t *region, int iters, uint64_t *out)
{
    if (threadIdx.x != 0 || blockIdx.x != 0)
        return;
    uint32_t *blk0 = region, *blk1 = region + 1024;
    uint32_t *nearb = copy_is_farther(blk0 + 1020, blk1 + 1020) ? blk1 : blk0;
    uint32_t *farb = (nearb == blk0) ? blk1 : blk0;
    for (int kind = 0; kind < 3; ++kind) {
        uint64_t sum = 0;
        for (int i = 0; i < iters; ++i) {
            spin_for_ns(2000);
            fence_release_gpu();
            spin_for_ns(500);
            if (kind == 1)
                st_relaxed_gpu(nearb + 32, static_cast<uint32_t>(i));
            else if (kind == 2)
                st_relaxed_gpu(farb + 32, static_cast<uint32_t>(i));
            const uint64_t a = globaltimer_ns();
            fence_release_gpu();
            const uint64_t b = globaltimer_ns();
            sum += b - a;
        }
        out[kind] = sum / static_cast<uint64_t>(iters);
    }
}

__global__ void probe_empty_kernel() {}

__global__ void probe_red_kernel(int iters, uint32_t *word)
{
    for (int i = 0; i < iters; ++i)
        red_add_relaxed_gpu(word, 1u);
}

}  // namespace cns

using namespace cns;

extern "C" int cns_probe_atomic_rtt(int kind, int32_t grid, int32_t probe_cta, int32_t iters, uint32_t *line_dev,
                                    uint64_t *out_dev, cns_stream_t stream)
{
    if (!line_dev || !out_dev)
        return CNS_ERR_NULL_PTR;
    if (kind < 0 || kind > 2 || grid < 1 || grid > (1 << 20) || probe_cta < 0 || probe_cta >= grid || iters < 1 ||
        iters > (1 << 24))
        return CNS_ERR_INVALID_VALUE;
    if (reinterpret_cast<uintptr_t>(line_dev) & (CNS_SYNCALL_LINE_BYTES - 1))
        return CNS_ERR_INVALID_VALUE;
    DeviceInfo dev;
    if (int rc = current_device(&dev))
        return rc;
    cudaStream_t s = to_stream(stream);
    CNS_CUDA(cudaMemsetAsync(line_dev, 0, CNS_SYNCALL_LINE_BYTES, s));
    probe_rtt_kernel<<<grid, 32, 0, s>>>(kind, probe_cta, iters, line_dev, out_dev);
    CNS_CUDA(cudaGetLastError());
    return CNS_SUCCESS;
}

extern "C" int cns_probe_same_address_throughput(int32_t grid, int32_t threads, int32_t iters, uint32_t *word_dev,
                                                 cns_stream_t stream)
{
    if (!word_dev)
        return CNS_ERR_NULL_PTR;
    if (grid < 1 || grid > (1 << 20) || threads < 32 || threads > 1024 || threads % 32 || iters < 1)
        return CNS_ERR_INVALID_VALUE;
    DeviceInfo dev;
    if (int rc = current_device(&dev))
        return rc;
    probe_red_kernel<<<grid, threads, 0, to_stream(stream)>>>(iters, word_dev);
    CNS_CUDA(cudaGetLastError());
    return CNS_SUCCESS;
}

extern "C" int cns_probe_grid_sync(int32_t ctas, int32_t threads, int64_t rounds, void *buf0_dev, void *buf1_dev,
                                   cns_stream_t stream)
{
    if (!buf0_dev || !buf1_dev)
        return CNS_ERR_NULL_PTR;
    if (ctas < 1 || threads < 32 || threads > 1024 || threads % 32 || rounds < 0)
        return CNS_ERR_INVALID_VALUE;
    if ((reinterpret_cast<uintptr_t>(buf0_dev) & 15) || (reinterpret_cast<uintptr_t>(buf1_dev) & 15))
        return CNS_ERR_INVALID_VALUE;
    DeviceInfo dev;
    if (int rc = current_device(&dev))
        return rc;
    uint4 *b0 = static_cast<uint4 *>(buf0_dev);
    uint4 *b1 = static_cast<uint4 *>(buf1_dev);
    void *args[] = {&b0, &b1, &rounds};
    cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(probe_grid_sync_kernel), dim3(ctas),
                                                dim3(threads), args, 0, to_stream(stream));
    if (e == cudaErrorCooperativeLaunchTooLarge) {
        (void)cudaGetLastError();
        return CNS_ERR_NOT_RESIDENT;
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "grid-sync probe launch");
    return CNS_SUCCESS;
}

extern "C" int cns_probe_notify_pingpong(int scope, int32_t iters, uint32_t *lines_dev, uint64_t *out_dev,
                                         cns_stream_t stream)
{
    if (!lines_dev || !out_dev)
        return CNS_ERR_NULL_PTR;
    if ((scope != 0 && scope != 1) || iters < 1 || iters > (1 << 24))
        return CNS_ERR_INVALID_VALUE;
    if (reinterpret_cast<uintptr_t>(lines_dev) & (CNS_SYNCALL_LINE_BYTES - 1))
        return CNS_ERR_INVALID_VALUE;
    DeviceInfo dev;
    if (int rc = current_device(&dev))
        return rc;
    cudaStream_t s = to_stream(stream);
    CNS_CUDA(cudaMemsetAsync(lines_dev, 0, 2 * CNS_SYNCALL_LINE_BYTES, s));
    CNS_CUDA(cudaMemsetAsync(out_dev, 0, 4 * sizeof(uint64_t), s));
    uint32_t *a = lines_dev;
    uint32_t *b = lines_dev + CNS_SYNCALL_LINE_BYTES / 4;
    uint64_t timeout_ns = 1000000000ull;
    void *args[] = {&iters, &a, &b, &timeout_ns, &out_dev};
    // both CTAs must run at once: a cooperative launch guarantees it or refuses
    const void *k = scope == 1 ? reinterpret_cast<const void *>(probe_pingpong_kernel<kScopeSys>)
                               : reinterpret_cast<const void *>(probe_pingpong_kernel<kScopeGpu>);
    CNS_CUDA(cudaLaunchCooperativeKernel(k, dim3(2), dim3(32), args, 0, s));
    return CNS_SUCCESS;
}

extern "C" int cns_probe_release_fence(uint32_t *region_dev, int32_t iters, uint64_t *out_dev, cns_stream_t stream)
{
    if (!region_dev || !out_dev)
        return CNS_ERR_NULL_PTR;
    if (iters < 1 || iters > 100000)
        return CNS_ERR_INVALID_VALUE;
    if (reinterpret_cast<uintptr_t>(region_dev) % CNS_SYNCALL_DIE_LOCAL_ALIGN != 0)
        return CNS_ERR_INVALID_VALUE;
    DeviceInfo dev;
    if (int rc = current_device(&dev))
        return rc;
    probe_fence_kernel<<<1, 32, 0, to_stream(stream)>>>(region_dev, iters, out_dev);
    CNS_CUDA(cudaGetLastError());
    return CNS_SUCCESS;
}

extern "C" int cns_probe_launch_cost(int32_t launches, int32_t early, double *us_per_launch, cns_stream_t stream)
{
    if (!us_per_launch)
        return CNS_ERR_NULL_PTR;
    if (launches < 1 || launches > 1000000 || (early != 0 && early != 1))
        return CNS_ERR_INVALID_VALUE;
    DeviceInfo dev;
    if (int rc = current_device(&dev))
        return rc;
    cudaStream_t s = to_stream(stream);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(32);
    cfg.stream = s;
    cfg.attrs = early ? attr : nullptr;
    cfg.numAttrs = early ? 1 : 0;
    CNS_CUDA(cudaLaunchKernelEx(&cfg, probe_empty_kernel));   // loaded and warm before the clock starts
    CNS_CUDA(cudaStreamSynchronize(s));
    const auto t0 = std::chrono::steady_clock::now();
    for (int32_t i = 0; i < launches; ++i)
        CNS_CUDA(cudaLaunchKernelEx(&cfg, probe_empty_kernel));
    const auto t1 = std::chrono::steady_clock::now();
    CNS_CUDA(cudaStreamSynchronize(s));
    *us_per_launch = std::chrono::duration<double, std::micro>(t1 - t0).count() / launches;
    return CNS_SUCCESS;
}
