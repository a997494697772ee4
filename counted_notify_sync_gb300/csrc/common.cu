// common.cu -- device checks, timeouts, version and error strings.
#include <cuda_runtime.h>

#include <cstdlib>
#include <mutex>

#include "cns.h"
#include "cns_host.h"

namespace cns {

int current_device(DeviceInfo *out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return cuda_fail(e, "cudaGetDevice");
    }
    // properties are fixed per device: cache them
    static std::mutex mu;
    static DeviceInfo cache[64];
    std::lock_guard<std::mutex> lk(mu);
    if (dev < 0 || dev >= 64)
        return CNS_ERR_CUDA;
    DeviceInfo &c = cache[dev];
    if (c.device != dev) {
        DeviceInfo d;
        d.device = dev;
        CNS_CUDA(cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev));
        CNS_CUDA(cudaDeviceGetAttribute(&d.max_threads_per_sm, cudaDevAttrMaxThreadsPerMultiProcessor, dev));
        CNS_CUDA(cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev));
        CNS_CUDA(cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev));
        c = d;
    }
    *out = c;
    if (c.cc_major != 10 || c.cc_minor != 3) {
        CNS_LOG(1, "device %d is compute capability %d.%d; this library is built for 10.3", dev, c.cc_major,
                c.cc_minor);
        return CNS_ERR_ARCH;
    }
    return CNS_SUCCESS;
}

static uint64_t env_ms(const char *name, uint64_t dflt)
{
    const char *e = std::getenv(name);
    if (!e || !*e)
        return dflt;
    char *end = nullptr;
    unsigned long long v = std::strtoull(e, &end, 10);
    return (end && *end == 0 && v > 0) ? v : dflt;
}

uint64_t barrier_timeout_ns(uint32_t timeout_ms)
{
    const uint64_t ms = timeout_ms ? timeout_ms : env_ms("CNS_TIMEOUT_MS", 2000);
    return ms * 1000000ull;
}

uint64_t notify_timeout_cap_ns() { return env_ms("CNS_TIMEOUT_MS", 30000) * 1000000ull; }

}  // namespace cns

extern "C" int cns_version(int32_t *version, int32_t *built_sm)
{
    if (!version || !built_sm)
        return CNS_ERR_NULL_PTR;
    *version = 100;   // 0.1.0
    *built_sm = 103;
    return CNS_SUCCESS;
}

extern "C" const char *cns_error_string(int code)
{
    switch (code) {
    case CNS_SUCCESS: return "success";
    case CNS_ERR_INVALID_VALUE: return "invalid value";
    case CNS_ERR_NULL_PTR: return "null pointer";
    case CNS_ERR_INVALID_HANDLE: return "invalid handle";
    case CNS_ERR_RESOURCE: return "resource exhausted";
    case CNS_ERR_TIMEOUT: return "timeout";
    case CNS_ERR_NOT_RESIDENT: return "grid cannot be co-resident";
    case CNS_ERR_CUDA: return "CUDA error";
    case CNS_ERR_ARCH: return "unsupported device architecture";
    default: return "unknown error";
    }
}
