// cns_host.h -- host-side helpers shared by the library's translation units:
// error mapping, device checks, environment settings, logging.
#pragma once

#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>

#include "cns.h"

namespace cns {

inline cudaStream_t to_stream(cns_stream_t s) { return reinterpret_cast<cudaStream_t>(s); }

inline int log_level()
{
    static int lvl = [] {
        const char *e = std::getenv("CNS_LOG");
        return e ? std::atoi(e) : 0;
    }();
    return lvl;
}

#define CNS_LOG(lvl, ...)                                   \
    do {                                                    \
        if (::cns::log_level() >= (lvl)) {                  \
            std::fprintf(stderr, "[cns] " __VA_ARGS__);     \
            std::fputc('\n', stderr);                       \
        }                                                   \
    } while (0)

// An NVTX range around a host entry point (shown by Nsight tools; the
// header-only NVTX costs a null check when no tool is attached).  `id` rides
// along as the range's payload: the notify id for the counted-notify calls.
class TraceRange {
public:
    explicit TraceRange(const char *name, uint64_t id = 0)
    {
        nvtxEventAttributes_t a = {};
        a.version = NVTX_VERSION;
        a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
        a.messageType = NVTX_MESSAGE_TYPE_ASCII;
        a.message.ascii = name;
        a.payloadType = NVTX_PAYLOAD_TYPE_UNSIGNED_INT64;
        a.payload.ullValue = id;
        nvtxRangePushEx(&a);
    }
    ~TraceRange() { nvtxRangePop(); }
    TraceRange(const TraceRange &) = delete;
    TraceRange &operator=(const TraceRange &) = delete;
};

// A CUDA call failed: log it and map to CNS_ERR_CUDA.
inline int cuda_fail(cudaError_t e, const char *what)
{
    CNS_LOG(1, "%s: %s", what, cudaGetErrorString(e));
    return CNS_ERR_CUDA;
}

#define CNS_CUDA(call)                                      \
    do {                                                    \
        cudaError_t e_ = (call);                            \
        if (e_ != cudaSuccess)                              \
            return ::cns::cuda_fail(e_, #call);             \
    } while (0)

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int max_threads_per_sm = 0;
    int cc_major = 0, cc_minor = 0;
};

// Current device and its properties; CNS_ERR_ARCH unless compute
// capability 10.3, CNS_ERR_CUDA if there is no usable device.
int current_device(DeviceInfo *out);

// Bound on one barrier wait: the argument if non-zero, else CNS_TIMEOUT_MS,
// else 2000 ms.  In nanoseconds.
uint64_t barrier_timeout_ns(uint32_t timeout_ms);

// Cap on one notify wait (CNS_TIMEOUT_MS if set, else 30 s), in nanoseconds.
uint64_t notify_timeout_cap_ns();

// Largest multiple of P not above 2^32, minus one (the atom.inc bound).
inline uint32_t counter_bound(uint32_t P)
{
    const uint64_t M = static_cast<uint64_t>(P) * ((1ull << 32) / P);
    return static_cast<uint32_t>(M - 1u);
}

}  // namespace cns
