// syncall.cu -- the host entry points of SYNCALL (syncall_workspace_init,
// syncall_run, syncall_read_workspace) and the headline round's phase probe.
//
// One launch runs R rounds of { data phase; barrier } (syncall_kernels.cuh).
// The barrier is the soft-mode epoch barrier of the "PTO-ISA SYNCALL
// cross-core barrier guide" (§5.2) or its hard counterpart built on
// thread-block clusters (§5.1's two-level shape: the group synchronises
// locally, one member takes part in the device-wide step, then releases the
// group).  Participants are CTAs; see cns.h for the role classes (§3.1) and
// the participant count (§4.2).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>

#include "cns.h"
#include "cns_host.h"
#include "syncall_kernels.cuh"

namespace cns {
// ---------------------------------------------------------------------------
// Where the headline round's time goes (a probe)
// ---------------------------------------------------------------------------
//
// The round of syncall_kernel<SOFT, RING_ROTATE, die-local> as syncall_run
// runs it for rows of one uint4 (thread 0 alone, through the per-die payload
// copies when the workspace has room for them), step for step, with
// %globaltimer stamps at the phase boundaries.  A stamp that follows a load
// or an atomic is taken only once its value has arrived.  The stamps of the
// last `stamp_rounds` rounds stay in shared memory until the run ends, so the
// probe adds no memory operation to the chain it measures (only the timer
// reads).  Per round and CTA:
//   [0] round start (taken afresh each round, after the previous round's
//       stamps were saved, so the probe's own bookkeeping falls between
//       rounds and in no phase)
//   [1] the neighbour's row has arrived
//   [2] the new row's stores are issued
//   [3] the release fence is done (the stores performed)
//   [4] the near copy's returning increment has arrived (the far one issued)
//   [5] the count that releases the round has arrived (= [4] for the round's
//       last arrival on the copy)
//   [6] the acquire fence is done
//   [7] the cursor is advanced
constexpr int kPhaseStamps = 8;

// The global timer, read only once `dep` (a loaded value) is known.
__device__ __forceinline__ uint64_t globaltimer_after(uint32_t dep)
{
    uint64_t t;
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0x9E3779B9;\n\tmov.u64 %0, 0;\n\t"
                 "@p mov.u64 %0, %%globaltimer;\n\t@!p mov.u64 %0, %%globaltimer;\n\t}"
                 : "=l"(t)
                 : "r"(dep));
    return t;
}

__global__ void __launch_bounds__(1024) round_phase_probe_kernel(const SyncallParams p, uint64_t *stamps,
                                                                 int32_t stamp_rounds)
{
    extern __shared__ uint64_t s_stamp[];   // stamp_rounds * kPhaseStamps
    if (threadIdx.x != 0)
        return;
    const uint32_t b = blockIdx.x;
    Barrier bar = p.bar;
    choose_near_copy(bar);
    const uint32_t q = (b + 1u == p.P) ? 0u : b + 1u;
    MirrorRow w{};   // one-uint4 rows through the copies, as the headline kernel moves them
    if (p.mirror) {
        const uint32_t q_slot = mirror_slot(p, q, 1u);
        w = mirror_row(p, mirror_setup(p, q_slot), q, b, 1u, q_slot, mirror_slot(p, b, 1u));
    }
    EpochCursor cursor{0u, 0u, false};
    const int64_t first = p.rounds - stamp_rounds;
    uint64_t t[kPhaseStamps];
    bool stop = false;
    for (int64_t r = 0; r < p.rounds && !stop; ++r) {
        const uint32_t k = static_cast<uint32_t>(r) & 1u;   // reads region k (buffer k), writes the other
        const bool odd = k != 0u;
        t[0] = globaltimer_ns();
        const uint4 *from = p.mirror ? (r == 0 ? w.first : (odd ? w.src1 : w.src0))
                                     : static_cast<const uint4 *>(k ? p.buf1 : p.buf0) + q;
        const uint4 v = ld_relaxed_gpu_v4(from);   // ring rotate: the row as it is
        t[1] = globaltimer_after(v.x ^ v.w);
        if (p.mirror) {
            uint4 *dst = odd ? w.dst0 : w.dst1;
            st_relaxed_gpu_v4(dst, v);
            st_relaxed_gpu_v4(dst + kMirrorBlock4, v);
            if (r + 2 >= p.rounds)
                st_relaxed_gpu_v4(odd ? w.last0 : w.last1, v);
        } else {
            st_relaxed_gpu_v4(static_cast<uint4 *>(k ? p.buf0 : p.buf1) + b, v);
        }
        t[2] = globaltimer_ns();
        fence_release_gpu();
        t[3] = globaltimer_ns();
        uint32_t target;
        const uint32_t before = copies_arrive<false>(bar.ctr, bar.ctr2, bar.e, cursor, &target);
        t[4] = globaltimer_after(before);
        const uint32_t mine = (before == bar.e.Mm1) ? 0u : before + 1u;
        if (epoch_reached(mine, target, bar.e)) {
            t[5] = t[4];
        } else {
            uint32_t seen = 0;
            stop = poll_until(bar.ctr,
                              [&](uint32_t cur) {
                                  seen = cur;
                                  return epoch_reached(cur, target, bar.e);
                              },
                              bar.status_line, bar.timeout_ns, static_cast<uint32_t>(r), b, true, 0, false);
            t[5] = globaltimer_after(seen);
        }
        fence_acquire_gpu();
        t[6] = globaltimer_ns();
        epoch_advance(cursor, target, bar.e);
        t[7] = globaltimer_ns();
        if (r >= first) {
            uint64_t *row = s_stamp + (r - first) * kPhaseStamps;
            for (int k = 0; k < kPhaseStamps; ++k)
                row[k] = t[k];
        }
    }
    if (!stop) {
        for (int32_t k = 0; k < stamp_rounds; ++k)
            for (int i = 0; i < kPhaseStamps; ++i)
                stamps[(static_cast<int64_t>(k) * gridDim.x + b) * kPhaseStamps + i] = s_stamp[k * kPhaseStamps + i];
    }
}

// Word offsets of the second copies of the counters (die-local variant).
constexpr uint32_t kSoftCopyWord = CNS_SYNCALL_REPLICA_OFFSET / 4;
constexpr uint32_t kHardCopyWord = (CNS_SYNCALL_REPLICA_OFFSET + 2 * CNS_SYNCALL_LINE_BYTES) / 4;

// The per-die payload copies' layout for P rows of `elems` uint32 (see
// mirror_slot): rows per 4 KB block and 8 KB pairs per region.  False when
// the rows cannot be copied: not a whole number of 16-byte units, or longer
// than a block less its timing slot (4080 bytes).
static bool mirror_layout(uint32_t P, int64_t elems, uint32_t *rows, uint32_t *pairs)
{
    if (P == 0 || elems < 4 || (elems & 3) != 0 || elems / 4 > kMirrorTiming4)
        return false;
    const uint32_t row4 = static_cast<uint32_t>(elems / 4);
    *rows = kMirrorTiming4 / row4;
    *pairs = (P + *rows - 1) / *rows;
    return true;
}

// Workspace bytes for the die-local counters and `pairs` pairs per region.
static uint64_t mirror_workspace_bytes(uint32_t pairs)
{
    return CNS_SYNCALL_WORKSPACE_DIE_LOCAL_BYTES + 2ull * pairs * kMirrorPair4 * 16u;
}

__global__ void workspace_init_kernel(uint32_t *ws, uint32_t n_words, uint32_t start, int with_copies)
{
    for (uint32_t i = threadIdx.x; i < n_words; i += blockDim.x)
        ws[i] = 0u;
    if (with_copies) {
        for (uint32_t i = threadIdx.x; i < 3 * CNS_SYNCALL_LINE_BYTES / 4; i += blockDim.x)
            ws[kSoftCopyWord + i] = 0u;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t *status_line = ws + CNS_SYNCALL_LINE_BYTES / 4;
        status_line[kBaseWordSoft] = start;
        status_line[kBaseWordHard] = start;
        status_line[kTagWord] = CNS_SYNCALL_WORKSPACE_TAG;
        ws[0] = start;                                  // soft counter
        ws[2 * CNS_SYNCALL_LINE_BYTES / 4] = start;     // hard counter
        ws[3 * CNS_SYNCALL_LINE_BYTES / 4] = start;     // soft release word
        ws[3 * CNS_SYNCALL_LINE_BYTES / 4 + 16] = start;  // hard release word
        if (with_copies) {
            ws[kSoftCopyWord] = start;
            ws[kHardCopyWord] = start;
        }
    }
}

// Can `grid` CTAs (in clusters of C when C > 0) be resident at once?
static int fits(KernelFn k, int grid, int threads, int C, size_t smem, cudaStream_t s, const DeviceInfo &dev, bool *ok)
{
    if (C <= 0) {
        int per_sm = 0;
        CNS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, reinterpret_cast<const void *>(k), threads, smem));
        *ok = static_cast<int64_t>(per_sm) * dev.sm_count >= grid;
        return CNS_SUCCESS;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = C;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    cudaError_t e = cudaOccupancyMaxActiveClusters(&n, reinterpret_cast<const void *>(k), &cfg);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        *ok = false;
        return CNS_SUCCESS;
    }
    *ok = static_cast<int64_t>(n) * C >= grid;
    return CNS_SUCCESS;
}

static bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Two timing events, destroyed on every exit path.
struct EventPair {
    cudaEvent_t a = nullptr, b = nullptr;
    ~EventPair()
    {
        if (a)
            cudaEventDestroy(a);
        if (b)
            cudaEventDestroy(b);
    }
};

}  // namespace cns

using namespace cns;

extern "C" int syncall_workspace_init(void *ws_dev, size_t bytes, uint32_t start_value, cns_stream_t stream)
{
    if (!ws_dev)
        return CNS_ERR_NULL_PTR;
    if (bytes < CNS_SYNCALL_WORKSPACE_BYTES || !aligned(ws_dev, CNS_SYNCALL_LINE_BYTES))
        return CNS_ERR_INVALID_VALUE;
    DeviceInfo dev;
    if (int rc = current_device(&dev))
        return rc;
    const int with_copies = bytes >= CNS_SYNCALL_WORKSPACE_DIE_LOCAL_BYTES ? 1 : 0;
    workspace_init_kernel<<<1, 128, 0, to_stream(stream)>>>(static_cast<uint32_t *>(ws_dev),
                                                             CNS_SYNCALL_WORKSPACE_BYTES / 4, start_value,
                                                             with_copies);
    CNS_CUDA(cudaGetLastError());
    return CNS_SUCCESS;
}

extern "C" int syncall_read_workspace(const void *ws_dev, cns_stream_t stream, uint32_t *soft_counter,
                                      uint32_t *hard_counter, int32_t *status)
{
    if (!ws_dev)
        return CNS_ERR_NULL_PTR;
    uint32_t w[CNS_SYNCALL_WORKSPACE_BYTES / 4];
    CNS_CUDA(cudaStreamSynchronize(to_stream(stream)));
    CNS_CUDA(cudaMemcpy(w, ws_dev, sizeof(w), cudaMemcpyDeviceToHost));
    if (soft_counter)
        *soft_counter = w[0];
    if (status)
        *status = static_cast<int32_t>(w[CNS_SYNCALL_LINE_BYTES / 4]);
    if (hard_counter)
        *hard_counter = w[2 * CNS_SYNCALL_LINE_BYTES / 4];
    return CNS_SUCCESS;
}

extern "C" int syncall_workspace_bytes(int32_t participants, int64_t elems, size_t *bytes)
{
    if (!bytes)
        return CNS_ERR_NULL_PTR;
    if (participants < 1 || elems < 0)
        return CNS_ERR_INVALID_VALUE;
    uint32_t rows = 0, pairs = 0;
    *bytes = mirror_layout(static_cast<uint32_t>(participants), elems, &rows, &pairs)
                 ? static_cast<size_t>(mirror_workspace_bytes(pairs))
                 : static_cast<size_t>(CNS_SYNCALL_WORKSPACE_DIE_LOCAL_BYTES);
    return CNS_SUCCESS;
}

extern "C" int syncall_run(int mode, int core_type, int32_t used_cores, int32_t aiv_ratio, int64_t rounds,
                           cns_syncall_data_t *d)
{
    TraceRange tr("syncall_run", static_cast<uint64_t>(rounds));
    // ---- argument checks (no CUDA call before these) ----
    if (!d)
        return CNS_ERR_NULL_PTR;
    if (mode != CNS_SYNCALL_SOFT && mode != CNS_SYNCALL_HARD)
        return CNS_ERR_INVALID_VALUE;
    if (core_type < CNS_AIV_ONLY || core_type > CNS_MIX)
        return CNS_ERR_INVALID_VALUE;
    if (d->workload < CNS_WL_EMPTY || d->workload > CNS_WL_JACOBI)
        return CNS_ERR_INVALID_VALUE;
    if (d->barrier_variant < 0 || d->barrier_variant > CNS_BARRIER_ARRIVAL_ONLY_DIE_LOCAL)
        return CNS_ERR_INVALID_VALUE;
    // arrival only orders no data: refuse it where rounds exchange data
    const bool arrival_only = d->barrier_variant == CNS_BARRIER_ARRIVAL_ONLY ||
                              d->barrier_variant == CNS_BARRIER_ARRIVAL_ONLY_DIE_LOCAL;
    if (arrival_only && d->workload != CNS_WL_EMPTY)
        return CNS_ERR_INVALID_VALUE;
    if (d->workspace_bytes != 0 && d->workspace_bytes < CNS_SYNCALL_WORKSPACE_BYTES)
        return CNS_ERR_INVALID_VALUE;
    if (d->launch_flags & ~(CNS_LAUNCH_NO_CLUSTER_ATTR | CNS_LAUNCH_NO_COOPERATIVE_ATTR))
        return CNS_ERR_INVALID_VALUE;
    if (d->hard_step != CNS_HARD_STEP_CLUSTER_BARRIER &&
        !(mode == CNS_SYNCALL_HARD && d->hard_step == CNS_HARD_STEP_PAIRED_MBARRIER))
        return CNS_ERR_INVALID_VALUE;
    if ((d->barrier_variant == CNS_BARRIER_DIE_LOCAL || d->barrier_variant == CNS_BARRIER_ARRIVAL_ONLY_DIE_LOCAL) &&
        d->workspace_bytes < CNS_SYNCALL_WORKSPACE_DIE_LOCAL_BYTES)
        return CNS_ERR_INVALID_VALUE;
    if ((d->barrier_variant == CNS_BARRIER_DIE_LOCAL || d->barrier_variant == CNS_BARRIER_ARRIVAL_ONLY_DIE_LOCAL) &&
        reinterpret_cast<uintptr_t>(d->workspace_dev) % CNS_SYNCALL_DIE_LOCAL_ALIGN != 0)
        CNS_LOG(2, "die-local workspace %p is not %d-byte aligned: its counter copies may share a die (slower, "
                   "same results)", d->workspace_dev, CNS_SYNCALL_DIE_LOCAL_ALIGN);
    if (rounds < 0 || used_cores < 0 || aiv_ratio < 0 || d->launch_ctas <= 0 || d->elems < 0)
        return CNS_ERR_INVALID_VALUE;
    const int threads = d->threads ? d->threads : 256;
    if (threads < 32 || threads > 1024 || threads % 32 != 0)
        return CNS_ERR_INVALID_VALUE;
    const int ratio = core_type == CNS_MIX ? (aiv_ratio ? aiv_ratio : 1) : 0;
    const int64_t group = core_type == CNS_MIX ? 1 + ratio : 1;
    const int64_t grid64 = static_cast<int64_t>(d->launch_ctas) * group;
    if (grid64 > (1 << 24))
        return CNS_ERR_INVALID_VALUE;
    const int grid = static_cast<int>(grid64);
    if (used_cores > grid)
        return CNS_ERR_INVALID_VALUE;   // [SYNCALL] §6.3: the set must match the launch
    const uint32_t P = (mode == CNS_SYNCALL_HARD) ? grid : (used_cores ? used_cores : grid);
    if (!d->workspace_dev)
        return CNS_ERR_NULL_PTR;
    if (!aligned(d->workspace_dev, CNS_SYNCALL_LINE_BYTES))
        return CNS_ERR_INVALID_VALUE;
    const bool has_payload = d->workload != CNS_WL_EMPTY && d->elems > 0;
    if (has_payload && (!d->buf0_dev || !d->buf1_dev))
        return CNS_ERR_NULL_PTR;
    if (has_payload && (!aligned(d->buf0_dev, 16) || !aligned(d->buf1_dev, 16)))
        return CNS_ERR_INVALID_VALUE;
    int C = 1;
    if (mode == CNS_SYNCALL_HARD) {
        if (core_type == CNS_MIX) {
            if (group > 8)
                return CNS_ERR_INVALID_VALUE;
            C = static_cast<int>(group);
        } else if (d->cluster_dim != 0) {
            if (d->cluster_dim < 1 || d->cluster_dim > 8 || grid % d->cluster_dim != 0)
                return CNS_ERR_INVALID_VALUE;
            C = d->cluster_dim;
        } else {
            C = 0;   // choose below
        }
    }
    const int64_t payload_bytes = !has_payload ? 0
                                  : d->workload == CNS_WL_JACOBI ? d->elems * 4
                                                                 : static_cast<int64_t>(P) * d->elems * 4;
    if ((d->host_in || d->host_out) && !has_payload)
        return CNS_ERR_INVALID_VALUE;

    // ---- device ----
    DeviceInfo dev;
    if (int rc = current_device(&dev))
        return rc;
    cudaStream_t s = to_stream(d->stream);
    KernelFn k = mode == CNS_SYNCALL_SOFT                             ? pick_soft_kernel(d->workload, d->barrier_variant)
                 : d->hard_step == CNS_HARD_STEP_PAIRED_MBARRIER ? pick_paired_kernel(d->workload, d->barrier_variant)
                                                                 : pick_hard_kernel(d->workload, d->barrier_variant);
    const size_t smem = d->workload == CNS_WL_JACOBI ? kJacSmemBytes : 0;
    // thread 0 alone touches memory: no payload, or rows of one uint4 or one word
    const bool ring = d->workload == CNS_WL_RING_AFFINE || d->workload == CNS_WL_RING_ROTATE ||
                      d->workload == CNS_WL_XORSHIFT;
    const bool solo = mode == CNS_SYNCALL_SOFT &&
                      (d->workload == CNS_WL_EMPTY || (ring && (d->elems == 4 || d->elems <= 1)));
    bool ok = false;
    if (solo && threads <= 256) {
        // the solo kernel when its grid can be resident, else syncall_kernel's own solo branch
        KernelFn ks = pick_solo_kernel(d->workload, d->barrier_variant);
        if (int rc = fits(ks, grid, threads, 0, 0, s, dev, &ok))
            return rc;
        if (ok)
            k = ks;
    }
    if (ok) {
        // the solo kernel fits
    } else if (mode == CNS_SYNCALL_HARD && C == 0) {
        // clusters of 2 first: measured 1634-1663 ns/round on the 148-CTA ring
        // against 1786-1819 for clusters of 4 (a cluster barrier waits for its
        // slowest member's payload) and 1616-1648 for clusters of 1, which
        // however costs ~80 ns more without a payload
        for (int c : {2, 4, 1}) {
            if (grid % c != 0)
                continue;
            if (int rc = fits(k, grid, threads, c, smem, s, dev, &ok))
                return rc;
            if (ok) {
                C = c;
                break;
            }
        }
        if (!ok)
            return CNS_ERR_NOT_RESIDENT;
    } else {
        if (int rc = fits(k, grid, threads, mode == CNS_SYNCALL_HARD ? C : 0, smem, s, dev, &ok))
            return rc;
        if (!ok)
            return CNS_ERR_NOT_RESIDENT;
    }

    SyncallParams prm;
    std::memset(&prm, 0, sizeof(prm));
    prm.buf0 = d->buf0_dev;
    prm.buf1 = d->buf1_dev;
    prm.elems = d->elems;
    prm.rounds = rounds;
    uint32_t *ws = static_cast<uint32_t *>(d->workspace_dev);
    prm.bar.status_line = ws + CNS_SYNCALL_LINE_BYTES / 4;
    prm.bar.timeout_ns = barrier_timeout_ns(d->timeout_ms);
    prm.bar.variant = d->barrier_variant;
    prm.cta_status = d->cta_status_dev;
    prm.P = P;
    prm.group = static_cast<uint32_t>(group);
    prm.core_type = core_type;
    prm.solo = solo ? 1 : 0;
    // the per-die payload copies: die-local variant, a ring whose rows can be copied (P rows; on the hard
    // path every CTA is a participant), room for them in the workspace
    uint32_t mrows = 0, mpairs = 0;
    const bool copies = ring && d->barrier_variant == CNS_BARRIER_DIE_LOCAL &&
                        mirror_layout(P, d->elems, &mrows, &mpairs) &&
                        d->workspace_bytes >= mirror_workspace_bytes(mpairs);
    prm.mirror = copies ? ws + CNS_SYNCALL_WORKSPACE_DIE_LOCAL_BYTES / 4 : nullptr;
    prm.mirror_rows = copies ? mrows : 0u;
    prm.mirror_region4 = copies ? mpairs * kMirrorPair4 : 0u;
    if (mode == CNS_SYNCALL_SOFT) {
        prm.bar.ctr = ws;
        prm.bar.ctr2 = ws + kSoftCopyWord;
        prm.bar.flag = ws + 3 * CNS_SYNCALL_LINE_BYTES / 4;
        prm.bar.e.P = P;
    } else {
        prm.bar.ctr = ws + 2 * CNS_SYNCALL_LINE_BYTES / 4;
        prm.bar.ctr2 = ws + kHardCopyWord;
        prm.bar.flag = ws + 3 * CNS_SYNCALL_LINE_BYTES / 4 + 16;
        prm.bar.e.P = static_cast<uint32_t>(grid / C);
    }
    prm.bar.e.Mm1 = counter_bound(prm.bar.e.P);

    d->grid_ctas = grid;
    d->participants = static_cast<int32_t>(P);
    d->cluster_used = mode == CNS_SYNCALL_HARD ? C : 1;

    EventPair ev;
    if (d->sync) {
        CNS_CUDA(cudaEventCreate(&ev.a));
        CNS_CUDA(cudaEventCreate(&ev.b));
        CNS_CUDA(cudaEventRecord(ev.a, s));
    }
    if (d->host_in)
        CNS_CUDA(cudaMemcpyAsync(d->buf0_dev, d->host_in, payload_bytes, cudaMemcpyHostToDevice, s));

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attrs[2];
    int na = 0;
    const bool cooperative = !(d->launch_flags & CNS_LAUNCH_NO_COOPERATIVE_ATTR);
    if (cooperative) {
        attrs[na].id = cudaLaunchAttributeCooperative;
        attrs[na].val.cooperative = 1;
        ++na;
    }
    if (mode == CNS_SYNCALL_HARD && !(d->launch_flags & CNS_LAUNCH_NO_CLUSTER_ATTR)) {
        attrs[na].id = cudaLaunchAttributeClusterDimension;
        attrs[na].val.clusterDim.x = C;
        attrs[na].val.clusterDim.y = 1;
        attrs[na].val.clusterDim.z = 1;
        ++na;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = na;
    void *args[] = {&prm};
    cudaError_t le = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(k), args);
    if (le == cudaErrorCooperativeLaunchTooLarge) {
        (void)cudaGetLastError();
        return CNS_ERR_NOT_RESIDENT;
    }
    if (le != cudaSuccess && mode == CNS_SYNCALL_HARD && cooperative && na == 2) {
        // the cooperative attribute together with clusters may be refused;
        // residency was checked above, so launch without it
        CNS_LOG(1, "cooperative cluster launch refused (%s); launching without it", cudaGetErrorString(le));
        (void)cudaGetLastError();
        cfg.attrs = attrs + 1;
        cfg.numAttrs = 1;
        le = cudaLaunchKernelExC(&cfg, reinterpret_cast<const void *>(k), args);
    }
    if (le != cudaSuccess)
        return cuda_fail(le, "syncall launch");

    if (d->host_out) {
        void *fin = (rounds & 1) ? d->buf1_dev : d->buf0_dev;
        CNS_CUDA(cudaMemcpyAsync(d->host_out, fin, payload_bytes, cudaMemcpyDeviceToHost, s));
    }
    if (!d->sync)
        return CNS_SUCCESS;

    CNS_CUDA(cudaEventRecord(ev.b, s));
    CNS_CUDA(cudaEventSynchronize(ev.b));
    float ms = 0.f;
    CNS_CUDA(cudaEventElapsedTime(&ms, ev.a, ev.b));
    d->elapsed_ms = ms;
    uint32_t sc = 0, hc = 0;
    int32_t st = 0;
    if (int rc = syncall_read_workspace(d->workspace_dev, d->stream, &sc, &hc, &st))
        return rc;
    d->final_counter = mode == CNS_SYNCALL_SOFT ? sc : hc;
    d->device_status = st;
    if (mode == CNS_SYNCALL_HARD) {
        uint32_t seen = 0;
        CNS_CUDA(cudaMemcpy(&seen, ws + CNS_SYNCALL_LINE_BYTES / 4 + 4, sizeof(seen), cudaMemcpyDeviceToHost));
        if (seen >= 1 && seen <= 16)
            d->cluster_used = static_cast<int32_t>(seen);
    }
    return (st == CNS_ERR_TIMEOUT || st == CNS_ERR_INVALID_VALUE) ? st : CNS_SUCCESS;
}

extern "C" int cns_probe_round_phases(int32_t ctas, int32_t threads, int64_t rounds, int32_t stamp_rounds,
                                      void *buf0_dev, void *buf1_dev, void *workspace_dev, size_t workspace_bytes,
                                      uint64_t *stamps_dev, cns_stream_t stream)
{
    TraceRange tr("cns_probe_round_phases", static_cast<uint64_t>(rounds));
    if (!buf0_dev || !buf1_dev || !workspace_dev || !stamps_dev)
        return CNS_ERR_NULL_PTR;
    if (ctas < 1 || threads < 32 || threads > 1024 || threads % 32 != 0 || stamp_rounds < 1 ||
        stamp_rounds > 1024 || rounds < stamp_rounds)
        return CNS_ERR_INVALID_VALUE;
    if (!aligned(workspace_dev, CNS_SYNCALL_LINE_BYTES) || !aligned(buf0_dev, 16) || !aligned(buf1_dev, 16) ||
        !aligned(stamps_dev, 8) || workspace_bytes < CNS_SYNCALL_WORKSPACE_DIE_LOCAL_BYTES)
        return CNS_ERR_INVALID_VALUE;
    DeviceInfo dev;
    if (int rc = current_device(&dev))
        return rc;
    cudaStream_t s = to_stream(stream);
    const size_t smem = static_cast<size_t>(stamp_rounds) * kPhaseStamps * sizeof(uint64_t);
    const void *k = reinterpret_cast<const void *>(round_phase_probe_kernel);
    if (smem > 48 * 1024)
        CNS_CUDA(cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)));
    int per_sm = 0;
    CNS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, threads, smem));
    if (static_cast<int64_t>(per_sm) * dev.sm_count < ctas)
        return CNS_ERR_NOT_RESIDENT;
    workspace_init_kernel<<<1, 128, 0, s>>>(static_cast<uint32_t *>(workspace_dev), CNS_SYNCALL_WORKSPACE_BYTES / 4,
                                            0u, 1);
    CNS_CUDA(cudaGetLastError());
    SyncallParams prm;
    std::memset(&prm, 0, sizeof(prm));
    uint32_t *ws = static_cast<uint32_t *>(workspace_dev);
    prm.buf0 = buf0_dev;
    prm.buf1 = buf1_dev;
    prm.elems = 4;
    prm.rounds = rounds;
    prm.bar.ctr = ws;
    prm.bar.ctr2 = ws + kSoftCopyWord;
    prm.bar.status_line = ws + CNS_SYNCALL_LINE_BYTES / 4;
    prm.bar.timeout_ns = barrier_timeout_ns(0);
    prm.bar.variant = CNS_BARRIER_DIE_LOCAL;
    prm.bar.e.P = static_cast<uint32_t>(ctas);
    prm.bar.e.Mm1 = counter_bound(prm.bar.e.P);
    prm.P = static_cast<uint32_t>(ctas);
    prm.group = 1;
    prm.solo = 1;
    uint32_t mrows = 0, mpairs = 0;
    const bool copies = mirror_layout(static_cast<uint32_t>(ctas), 4, &mrows, &mpairs) &&
                        workspace_bytes >= mirror_workspace_bytes(mpairs);
    prm.mirror = copies ? ws + CNS_SYNCALL_WORKSPACE_DIE_LOCAL_BYTES / 4 : nullptr;
    prm.mirror_rows = copies ? mrows : 0u;
    prm.mirror_region4 = copies ? mpairs * kMirrorPair4 : 0u;
    void *args[] = {&prm, &stamps_dev, &stamp_rounds};
    CNS_CUDA(cudaLaunchCooperativeKernel(k, dim3(ctas), dim3(threads), args, smem, s));
    return CNS_SUCCESS;
}
