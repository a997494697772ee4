// Test-only user kernels built on include/cns_device.h: the ring-rotate rounds
// separated by cns_syncall_soft, records with cns_cnt_record_dev, and waits
// with cns_cnt_wait_dev, each behind a plain C launcher.  Compiled by the GPU
// tests into a shared library of their own.
#include <cstdint>
#include <cuda_runtime.h>

#include "cns_device.h"

namespace {

// CTAs below `participants` run `rounds` ring rounds (dst[p] = src[(p + 1) % P],
// buffers swapping each round), each followed by the soft barrier; CTA
// `short_cta` (if below participants) takes one barrier fewer.  Other CTAs
// return at once.  status[p] = the first non-zero barrier result, or 0.
__global__ void ring_kernel(uint4 *b0, uint4 *b1, uint32_t participants, int64_t rounds, void *ws,
                            uint64_t timeout_ns, uint32_t short_cta, int *status)
{
    const uint32_t p = blockIdx.x;
    if (p >= participants)
        return;
    const int64_t mine = (p == short_cta) ? rounds - 1 : rounds;
    int st = 0;
    for (int64_t r = 0; r < rounds; ++r) {
        const uint4 *src = (r & 1) ? b1 : b0;
        uint4 *dst = (r & 1) ? b0 : b1;
        if (threadIdx.x == 0)
            dst[p] = src[(p + 1 == participants) ? 0 : p + 1];
        if (r >= mine)
            break;
        st = cns_syncall_soft(ws, participants, timeout_ns);
        if (st != CNS_SUCCESS)
            break;
    }
    if (threadIdx.x == 0)
        status[p] = st;
}

// The same rounds with the die-local barrier: the CTA's state lives in shared
// memory, set before the first barrier.
__global__ void ring_kernel_die_local(uint4 *b0, uint4 *b1, uint32_t participants, int64_t rounds, void *ws,
                                      uint64_t timeout_ns, uint32_t short_cta, int *status)
{
    __shared__ cns_soft_state_t st;
    const uint32_t p = blockIdx.x;
    if (p >= participants)
        return;
    if (threadIdx.x == 0)
        st = cns_soft_state_t CNS_SOFT_STATE_INIT;
    __syncthreads();
    const int64_t mine = (p == short_cta) ? rounds - 1 : rounds;
    int rc = 0;
    for (int64_t r = 0; r < rounds; ++r) {
        const uint4 *src = (r & 1) ? b1 : b0;
        uint4 *dst = (r & 1) ? b0 : b1;
        if (threadIdx.x == 0)
            dst[p] = src[(p + 1 == participants) ? 0 : p + 1];
        if (r >= mine)
            break;
        rc = cns_syncall_soft_die_local(ws, participants, timeout_ns, &st);
        if (rc != CNS_SUCCESS)
            break;
    }
    if (threadIdx.x == 0)
        status[p] = rc;
}

__global__ void record_kernel(uint32_t *count, int mode, uint32_t v, int per_thread)
{
    for (int i = 0; i < per_thread; ++i)
        cns_cnt_record_dev(count, mode, v);
}

__global__ void wait_kernel(uint32_t *count, int mode, uint32_t v, int is_clear, uint64_t timeout_ns, int *rc,
                            uint32_t *observed)
{
    if (threadIdx.x == 0)
        *rc = cns_cnt_wait_dev(count, mode, v, is_clear, timeout_ns, observed);
}

}  // namespace

extern "C" int user_ring(int32_t ctas, int32_t threads, uint32_t participants, int64_t rounds, void *b0, void *b1,
                         void *ws, uint64_t timeout_ns, uint32_t short_cta, int *status)
{
    void *args[] = {&b0, &b1, &participants, &rounds, &ws, &timeout_ns, &short_cta, &status};
    cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(ring_kernel), dim3(ctas),
                                                dim3(threads), args, 0, 0);
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    return static_cast<int>(e);
}

extern "C" int user_ring_die_local(int32_t ctas, int32_t threads, uint32_t participants, int64_t rounds, void *b0,
                                   void *b1, void *ws, uint64_t timeout_ns, uint32_t short_cta, int *status)
{
    void *args[] = {&b0, &b1, &participants, &rounds, &ws, &timeout_ns, &short_cta, &status};
    cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(ring_kernel_die_local), dim3(ctas),
                                                dim3(threads), args, 0, 0);
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    return static_cast<int>(e);
}

extern "C" int user_record(uint32_t *count, int mode, uint32_t v, int32_t ctas, int32_t threads, int per_thread)
{
    record_kernel<<<ctas, threads>>>(count, mode, v, per_thread);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    return static_cast<int>(e);
}

extern "C" int user_wait(uint32_t *count, int mode, uint32_t v, int is_clear, uint64_t timeout_ns, int *rc,
                         uint32_t *observed)
{
    wait_kernel<<<1, 32>>>(count, mode, v, is_clear, timeout_ns, rc, observed);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    return static_cast<int>(e);
}
