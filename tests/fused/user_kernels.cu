// Test-only user kernels built on include/cns_device.h: the ring-rotate rounds
// separated by cns_syncall_soft (or its system-scope form), records with
// cns_cnt_record_dev, waits with
// cns_cnt_wait_dev, and a grid-wide consumer on cns_cnt_wait_grid_dev, each
// behind a plain C launcher.  Compiled by the GPU
// tests into a shared library of their own.
#include <cstdint>
#include <cuda_runtime.h>

#include "cns_device.h"

namespace {

// CTAs below `participants` run `rounds` ring rounds (dst[p] = src[(p + 1) % P],
// buffers swapping each round), each followed by the soft barrier; CTA
// `short_cta` (if below participants) takes one barrier fewer.  Other CTAs
// return at once.  status[p] = the first non-zero barrier result, or 0.
// kSys: the barrier at system scope (cns_syncall_soft_sys).
template <bool kSys>
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
        st = kSys ? cns_syncall_soft_sys(ws, participants, timeout_ns) : cns_syncall_soft(ws, participants, timeout_ns);
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

// The same at system scope (a count word that peer GPUs also use).
__global__ void record_sys_kernel(uint32_t *count, int mode, uint32_t v, int per_thread)
{
    for (int i = 0; i < per_thread; ++i)
        cns_cnt_record_sys_dev(count, mode, v);
}

__global__ void wait_sys_kernel(uint32_t *count, int mode, uint32_t v, int is_clear, uint64_t timeout_ns, int *rc,
                                uint32_t *observed)
{
    if (threadIdx.x == 0)
        *rc = cns_cnt_wait_sys_dev(count, mode, v, is_clear, timeout_ns, observed);
}

// A grid-wide consumer: CTAs 0 .. G-1 take cns_cnt_wait_grid_dev (count >=
// k, clear) as call r of `rounds`, then each sums the `words` words of area
// r % 2 into sums[r * G + cta] and records ADD 1 on ack.  CTA G produces:
// for round r it waits until the consumers of round r - 2 have all recorded
// on ack, writes word w of area r % 2 as w * 2654435761 + r, waits until
// call r - 1 is published on go (its clear is done), and records ADD 1 k
// times.  rcs[r * G + cta] = the wait's result.
__global__ void grid_wait_kernel(uint32_t *count, uint32_t *go, uint32_t *ack, uint32_t *area, int words,
                                 uint32_t k, int rounds, uint64_t timeout_ns, uint32_t *sums, int *rcs,
                                 uint32_t *observed)
{
    const uint32_t G = gridDim.x - 1;
    __shared__ uint32_t part[32];
    for (int r = 0; r < rounds; ++r) {
        uint32_t *a = area + (r & 1) * words;
        if (blockIdx.x == G) {
            int ok = 1;
            if (threadIdx.x == 0 && r >= 2)
                ok = cns_cnt_wait_dev(ack, CNS_WAIT_BIGGER_OR_EQUAL, static_cast<uint32_t>(r - 1) * G, 0,
                                      timeout_ns, nullptr) == CNS_SUCCESS;
            if (!__syncthreads_and(ok))
                return;
            for (int w = threadIdx.x; w < words; w += blockDim.x)
                a[w] = static_cast<uint32_t>(w) * 2654435761u + static_cast<uint32_t>(r);
            __syncthreads();
            if (threadIdx.x == 0) {
                ok = cns_cnt_wait_dev(go, CNS_WAIT_BIGGER_OR_EQUAL, static_cast<uint32_t>(r), 0, timeout_ns,
                                      nullptr) == CNS_SUCCESS;
                for (uint32_t i = 0; ok && i < k; ++i)
                    cns_cnt_record_dev(count, CNS_REC_ADD, 1u);
            }
            if (!__syncthreads_and(ok))
                return;
            continue;
        }
        const int rc = cns_cnt_wait_grid_dev(count, go, static_cast<uint32_t>(r), CNS_WAIT_BIGGER_OR_EQUAL, k, 1,
                                             timeout_ns, observed + r);
        uint32_t s = 0;
        if (rc == CNS_SUCCESS)
            for (int w = threadIdx.x; w < words; w += blockDim.x)
                s += a[w];
        for (int o = 16; o > 0; o >>= 1)
            s += __shfl_xor_sync(0xffffffffu, s, o);
        if ((threadIdx.x & 31) == 0)
            part[threadIdx.x >> 5] = s;
        __syncthreads();
        if (threadIdx.x == 0) {
            uint32_t t = 0;
            for (int i = 0; i < static_cast<int>(blockDim.x >> 5); ++i)
                t += part[i];
            sums[r * G + blockIdx.x] = t;
            rcs[r * G + blockIdx.x] = rc;
            cns_cnt_record_dev(ack, CNS_REC_ADD, 1u);
        }
        __syncthreads();
        if (rc != CNS_SUCCESS)
            return;
    }
}

// Every CTA takes call `call` of a grid-wide wait with (mode, v); rcs[cta] = its result.
__global__ void grid_wait_only_kernel(uint32_t *count, uint32_t *go, uint32_t call, int mode, uint32_t v,
                                      uint64_t timeout_ns, int *rcs)
{
    const int rc = cns_cnt_wait_grid_dev(count, go, call, mode, v, 1, timeout_ns, nullptr);
    if (threadIdx.x == 0)
        rcs[blockIdx.x] = rc;
}

}  // namespace

extern "C" int user_grid_wait(int32_t consumers, int32_t threads, uint32_t *count, uint32_t *go, uint32_t *ack,
                              uint32_t *area, int words, uint32_t k, int rounds, uint64_t timeout_ns, uint32_t *sums,
                              int *rcs, uint32_t *observed)
{
    void *args[] = {&count, &go, &ack, &area, &words, &k, &rounds, &timeout_ns, &sums, &rcs, &observed};
    cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(grid_wait_kernel),
                                                dim3(consumers + 1), dim3(threads), args, 0, 0);
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    return static_cast<int>(e);
}

extern "C" int user_grid_wait_only(int32_t ctas, uint32_t *count, uint32_t *go, uint32_t call, int mode, uint32_t v,
                                   uint64_t timeout_ns, int *rcs)
{
    void *args[] = {&count, &go, &call, &mode, &v, &timeout_ns, &rcs};
    cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(grid_wait_only_kernel), dim3(ctas),
                                                dim3(128), args, 0, 0);
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    return static_cast<int>(e);
}

extern "C" int user_ring(int32_t ctas, int32_t threads, uint32_t participants, int64_t rounds, void *b0, void *b1,
                         void *ws, uint64_t timeout_ns, uint32_t short_cta, int *status)
{
    void *args[] = {&b0, &b1, &participants, &rounds, &ws, &timeout_ns, &short_cta, &status};
    cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(ring_kernel<false>), dim3(ctas),
                                                dim3(threads), args, 0, 0);
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    return static_cast<int>(e);
}

extern "C" int user_ring_sys(int32_t ctas, int32_t threads, uint32_t participants, int64_t rounds, void *b0,
                             void *b1, void *ws, uint64_t timeout_ns, uint32_t short_cta, int *status)
{
    void *args[] = {&b0, &b1, &participants, &rounds, &ws, &timeout_ns, &short_cta, &status};
    cudaError_t e = cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(ring_kernel<true>), dim3(ctas),
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

extern "C" int user_record_sys(uint32_t *count, int mode, uint32_t v, int32_t ctas, int32_t threads, int per_thread)
{
    record_sys_kernel<<<ctas, threads>>>(count, mode, v, per_thread);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    return static_cast<int>(e);
}

extern "C" int user_wait_sys(uint32_t *count, int mode, uint32_t v, int is_clear, uint64_t timeout_ns, int *rc,
                             uint32_t *observed)
{
    wait_sys_kernel<<<1, 32>>>(count, mode, v, is_clear, timeout_ns, rc, observed);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess)
        e = cudaDeviceSynchronize();
    return static_cast<int>(e);
}
