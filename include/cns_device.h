/*
 * cns_device.h -- the device side of counted_notify_sync for code that runs
 * inside the caller's own CUDA kernels (nvcc, sm_103a): record on a counted
 * notify, wait on one, and take the soft SYNCALL barrier, with no library
 * call and no kernel boundary.  Header only; include it from .cu files
 * compiled with -gencode arch=compute_103a,code=sm_103a, with the directory
 * of cns.h on the include path.
 *
 *   cns_cnt_record_dev   one record ("CANN Runtime CntNotify management API"
 *                        §3.1: SET, ADD, BIT_OR, BIT_AND) as one release
 *                        atomic on the notify's count word
 *                        (cntnotify_get_device_ptr gives its address)
 *   cns_cnt_wait_dev     a bounded wait on that word (§3.2: LESS, EQUAL,
 *                        BIGGER, BIGGER_OR_EQUAL, EQUAL_WITH_BITMASK, with
 *                        isClear) from one thread
 *   cns_cnt_wait_grid_dev  the same wait taken by several CTAs of a grid
 *                        together, call after call: CTA 0 waits and clears,
 *                        the others follow a `go` word it publishes
 *   cns_syncall_soft     the soft SYNCALL barrier ("PTO-ISA SYNCALL
 *                        cross-core barrier guide" §5.2) among the first P
 *                        CTAs of a grid, on a workspace that
 *                        syncall_workspace_init prepared, called by every
 *                        thread of each of those CTAs
 *   cns_syncall_soft_die_local  the same on the two counter copies of a
 *                        die-local workspace, one on each of GB300's dies
 *                        (faster; the caller keeps a small per-CTA state)
 *   cns_syncall_soft_sys  the soft barrier at system scope, for participants
 *                        on several GPUs arriving on one workspace through
 *                        peer mappings
 *   cns_cnt_record_sys_dev, cns_cnt_wait_sys_dev  record and wait at system
 *                        scope, for a count word that GPUs other than its
 *                        own also record on or wait on (§1: CntNotify between
 *                        devices), through a peer mapping
 *
 * Every wait is bounded and reports CNS_ERR_TIMEOUT instead of trapping.  The
 * caller makes the participating CTAs co-resident (a cooperative launch, or a
 * grid no larger than the GPU holds at once): a barrier or grid-wide wait
 * whose participants are not all running at the same time ends in that
 * timeout.
 *
 * The library's own kernels are built on the same primitives (namespace cns).
 */
#ifndef CNS_DEVICE_H
#define CNS_DEVICE_H

#include <stdint.h>

#include "cns.h"

#if defined(__CUDACC__)

namespace cns {

// ---------------------------------------------------------------------------
// Scoped memory operations (PTX ISA memory consistency model, .gpu scope)
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t atom_inc_release_gpu(uint32_t *p, uint32_t bound)
{
    // old = *p; *p = (old >= bound) ? 0 : old + 1
    uint32_t old;
    asm volatile("atom.release.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(bound) : "memory");
    return old;
}

__device__ __forceinline__ uint32_t atom_add_relaxed_gpu(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint32_t atom_add_release_gpu(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.release.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint32_t atom_exch_release_gpu(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.release.gpu.global.exch.b32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint32_t atom_exch_relaxed_gpu(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.relaxed.gpu.global.exch.b32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint32_t atom_cas_relaxed_gpu(uint32_t *p, uint32_t cmp, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.relaxed.gpu.global.cas.b32 %0, [%1], %2, %3;" : "=r"(old) : "l"(p), "r"(cmp), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void red_add_release_gpu(uint32_t *p, uint32_t v)
{
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_inc_relaxed_gpu(uint32_t *p, uint32_t bound)
{
    uint32_t old;
    asm volatile("atom.relaxed.gpu.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(bound) : "memory");
    return old;
}

__device__ __forceinline__ void red_inc_relaxed_gpu(uint32_t *p, uint32_t bound)
{
    asm volatile("red.relaxed.gpu.global.inc.u32 [%0], %1;" ::"l"(p), "r"(bound) : "memory");
}

__device__ __forceinline__ void red_inc_release_gpu(uint32_t *p, uint32_t bound)
{
    asm volatile("red.release.gpu.global.inc.u32 [%0], %1;" ::"l"(p), "r"(bound) : "memory");
}

__device__ __forceinline__ void fence_release_gpu()
{
    asm volatile("fence.release.gpu;" ::: "memory");
}

// After a strong read (here: the read half of an atomic), makes the reading
// thread see what the writers it read from released.
__device__ __forceinline__ void fence_acquire_gpu()
{
    asm volatile("fence.acquire.gpu;" ::: "memory");
}

__device__ __forceinline__ void red_add_relaxed_gpu(uint32_t *p, uint32_t v)
{
    asm volatile("red.relaxed.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_or_release_gpu(uint32_t *p, uint32_t v)
{
    asm volatile("red.release.gpu.global.or.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_and_release_gpu(uint32_t *p, uint32_t v)
{
    asm volatile("red.release.gpu.global.and.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t ld_relaxed_gpu(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_gpu(uint32_t *p, uint32_t v)
{
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// 16-byte relaxed gpu-scope load and store: served by L2, past the SM's L1
// (data that other SMs write every round gains nothing from L1).
__device__ __forceinline__ uint4 ld_relaxed_gpu_v4(const uint4 *p)
{
    uint4 v;
    asm volatile("ld.relaxed.gpu.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p)
                 : "memory");
    return v;
}

__device__ __forceinline__ void st_relaxed_gpu_v4(uint4 *p, const uint4 &v)
{
    asm volatile("st.relaxed.gpu.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ uint64_t ld_acquire_gpu_u64(const uint64_t *p)
{
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release_gpu_u64(uint64_t *p, uint64_t v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void st_release_gpu(uint32_t *p, uint32_t v)
{
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ uint32_t smid()
{
    uint32_t s;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(s));
    return s;
}

// System scope (.sys): the same operations, ordered with threads of other
// GPUs too.  A count word that a peer GPU records on through a peer mapping
// (or waits on) is accessed with these on both sides; a gpu-scope acquire
// does not synchronise with a release performed on another GPU.
__device__ __forceinline__ uint32_t ld_relaxed_sys(const uint32_t *p)
{
    uint32_t v;
    asm volatile("ld.relaxed.sys.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t atom_exch_release_sys(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.release.sys.global.exch.b32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ uint32_t atom_exch_relaxed_sys(uint32_t *p, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.relaxed.sys.global.exch.b32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void red_add_release_sys(uint32_t *p, uint32_t v)
{
    asm volatile("red.release.sys.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_or_release_sys(uint32_t *p, uint32_t v)
{
    asm volatile("red.release.sys.global.or.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_and_release_sys(uint32_t *p, uint32_t v)
{
    asm volatile("red.release.sys.global.and.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t atom_inc_release_sys(uint32_t *p, uint32_t bound)
{
    uint32_t old;
    asm volatile("atom.release.sys.global.inc.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(bound) : "memory");
    return old;
}

__device__ __forceinline__ uint32_t atom_cas_relaxed_sys(uint32_t *p, uint32_t cmp, uint32_t v)
{
    uint32_t old;
    asm volatile("atom.relaxed.sys.global.cas.b32 %0, [%1], %2, %3;" : "=r"(old) : "l"(p), "r"(cmp), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void st_relaxed_sys(uint32_t *p, uint32_t v)
{
    asm volatile("st.relaxed.sys.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void fence_acquire_sys()
{
    asm volatile("fence.acquire.sys;" ::: "memory");
}

// The scope of a counted notify's operations: kScopeGpu for a count that only
// its own GPU touches, kScopeSys once other GPUs record on or wait on it.
enum : int { kScopeGpu = 0, kScopeSys = 1 };

template <int S>
__device__ __forceinline__ uint32_t ld_relaxed_scoped(const uint32_t *p)
{
    if constexpr (S == kScopeSys)
        return ld_relaxed_sys(p);
    else
        return ld_relaxed_gpu(p);
}

template <int S>
__device__ __forceinline__ void fence_acquire_scoped()
{
    if constexpr (S == kScopeSys)
        fence_acquire_sys();
    else
        fence_acquire_gpu();
}

template <int S>
__device__ __forceinline__ uint32_t atom_exch_relaxed_scoped(uint32_t *p, uint32_t v)
{
    if constexpr (S == kScopeSys)
        return atom_exch_relaxed_sys(p, v);
    else
        return atom_exch_relaxed_gpu(p, v);
}

// ---------------------------------------------------------------------------
// Epoch arithmetic of the soft barrier ("PTO-ISA SYNCALL cross-core barrier
// guide", §5.2).  The counter lives in Z_M with M = P * floor(2^32 / P): the
// arrival is atom.inc with bound M - 1, the target is ((before / P) + 1) * P
// taken mod M, and the count has reached the target when (cur - target) mod M
// is below P -- a waiter sees counts in [before + 1, target + P - 1] only.
// For a power-of-two P, M = 2^32 and this is the plain wrapping add.
// ---------------------------------------------------------------------------

struct Epoch {
    uint32_t P;     // participants arriving on this counter
    uint32_t Mm1;   // M - 1 (the atom.inc bound)
};

__device__ __forceinline__ uint32_t epoch_target(uint32_t before, const Epoch &e)
{
    const uint64_t M = static_cast<uint64_t>(e.Mm1) + 1u;
    uint64_t t = (static_cast<uint64_t>(before / e.P) + 1u) * e.P;   // <= M since before < M
    return t == M ? 0u : static_cast<uint32_t>(t);
}

// (cur - target) mod M < P in 32-bit arithmetic: the wrapping difference is
// the distance in Z_M unless it wrapped, in which case it exceeds that
// distance by 2^32 - M (= ~Mm1; zero when M = 2^32).
__device__ __forceinline__ bool epoch_reached(uint32_t cur, uint32_t target, const Epoch &e)
{
    uint32_t d = cur - target;
    if (cur < target)
        d -= ~e.Mm1;
    return d < e.P;
}

// The epoch of P participants: M - 1 = P * floor(2^32 / P) - 1.
__device__ __forceinline__ Epoch epoch_of(uint32_t P)
{
    const uint64_t M = static_cast<uint64_t>(P) * ((static_cast<uint64_t>(1) << 32) / P);
    return Epoch{P, static_cast<uint32_t>(M - 1u)};
}

// The epoch that the caller's previous barrier closed: [start, start + P) in
// Z_M, start a multiple of P.  In a well-formed round an arrival's `before`
// lies in that epoch, so ((before / P) + 1) * P mod M is just `end`; the
// cursor gives the same target as the formula without the division, and the
// formula is still evaluated whenever `before` falls outside (first round, or
// a counter that someone else moved).
struct EpochCursor {
    uint32_t start;
    uint32_t end;     // start + P in Z_M
    bool valid;
};

__device__ __forceinline__ uint32_t epoch_target(uint32_t before, const Epoch &e, const EpochCursor &c)
{
    if (c.valid && before - c.start < e.P)   // wraps to >= P when before < start (start <= M - P)
        return c.end;
    return epoch_target(before, e);
}

__device__ __forceinline__ void epoch_advance(EpochCursor &c, uint32_t target, const Epoch &e)
{
    c.start = target;
    c.end = (target == e.Mm1 + 1u - e.P) ? 0u : target + e.P;   // M - P wraps to 0
    c.valid = true;
}

// Two copies of a counter (die-local arrivals) --------------------------------
//
// GB300 homes each 4 KB block on one of its two dies, by the parity of the
// block number's bits; an atomic is performed by the L2 of the home die,
// ~150 ns from that die's SMs and ~350 ns from the other's.  A counter kept
// twice, in two blocks that differ only in address bit 12, has one copy on
// each die: every arrival increments both, each participant polls the copy
// on its own die.

// Whether copy `a` answers this SM more slowly than copy `b` (a dependent
// chain of adds of 0 on each: the counts do not change, whoever else is
// arriving; (x >> 31) picks word 0 or 1 of the copy's line).
__device__ __forceinline__ bool copy_is_farther(uint32_t *a, uint32_t *b)
{
    uint32_t x = 0;
    const uint64_t t0 = globaltimer_ns();
    for (int i = 0; i < 8; ++i)
        x = atom_add_relaxed_gpu(a + (x >> 31), 0u);
    const uint64_t t1 = globaltimer_ns();
    for (int i = 0; i < 8; ++i)
        x = atom_add_relaxed_gpu(b + (x >> 31), 0u);
    const uint64_t t2 = globaltimer_ns();
    return t2 - t1 < t1 - t0;
}

// One arrival on both copies; returns the near copy's old value and sets
// *target.  kRelease: one release fence first (the arrival carries the
// caller's writes).  The far increment is issued with the near one, so the
// two may land in either order, and another participant's next-round
// increment may reach the near copy before this one does: the returned value
// can then lie one epoch ahead.  So from the second barrier on the target is
// the cursor's (the last target plus P), whatever the returned value; in the
// first barrier, whose target comes from the returned value, the far
// increment is a release that lands after the near one, so no participant
// can leave the first barrier before every first-round increment is on every
// copy.  (An all-interleavings model of both copies shows the returned
// value's target failing without these two rules and holding with them.)
template <bool kRelease>
__device__ __forceinline__ uint32_t copies_arrive(uint32_t *near, uint32_t *far, const Epoch &e,
                                                  const EpochCursor &c, uint32_t *target)
{
    if (kRelease)
        fence_release_gpu();
    uint32_t before;
    if (c.valid) {
        red_inc_relaxed_gpu(far, e.Mm1);
        before = atom_inc_relaxed_gpu(near, e.Mm1);
        *target = c.end;
    } else {
        before = atom_inc_relaxed_gpu(near, e.Mm1);
        red_inc_release_gpu(far, e.Mm1);
        *target = epoch_target(before, e);
    }
    return before;
}

// ---------------------------------------------------------------------------
// Counted-notify record and wait rules ("CANN Runtime CntNotify management
// API", §3.1 and §3.2)
// ---------------------------------------------------------------------------

// Whether a wait with this mode/value is released at count c (mode checked
// by the caller, <= 4).
__device__ __forceinline__ bool cnt_wait_released(uint32_t c, uint32_t mode, uint32_t v)
{
    const bool lt = c < v, eq = c == v, gt = c > v, mask = (c & v) == v;
    return (mode == CNS_WAIT_LESS) ? lt
         : (mode == CNS_WAIT_EQUAL) ? eq
         : (mode == CNS_WAIT_BIGGER) ? gt
         : (mode == CNS_WAIT_BIGGER_OR_EQUAL) ? (gt || eq)
                                              : mask;   // CNS_WAIT_EQUAL_WITH_BITMASK
}

// A record as one device atomic with release semantics, at scope S.  Usable
// from inside any kernel (one thread per record).
template <int S>
__device__ __forceinline__ void cnt_record_scoped(uint32_t *count, uint32_t mode, uint32_t v)
{
    if constexpr (S == kScopeSys) {
        switch (mode) {
        case CNS_REC_SET: atom_exch_release_sys(count, v); break;
        case CNS_REC_ADD: red_add_release_sys(count, v); break;
        case CNS_REC_BIT_OR: red_or_release_sys(count, v); break;
        case CNS_REC_BIT_AND: red_and_release_sys(count, v); break;
        default: break;
        }
    } else {
        switch (mode) {
        case CNS_REC_SET: atom_exch_release_gpu(count, v); break;
        case CNS_REC_ADD: red_add_release_gpu(count, v); break;
        case CNS_REC_BIT_OR: red_or_release_gpu(count, v); break;
        case CNS_REC_BIT_AND: red_and_release_gpu(count, v); break;
        default: break;
        }
    }
}

__device__ __forceinline__ void cnt_record_device(uint32_t *count, uint32_t mode, uint32_t v)
{
    cnt_record_scoped<kScopeGpu>(count, mode, v);
}

// A bounded wait on a count word from the calling thread, at scope S: relaxed
// polls, one acquire fence once released, then the optional clear.  Returns
// CNS_SUCCESS or CNS_ERR_TIMEOUT.
template <int S>
__device__ __forceinline__ int cnt_wait_scoped(uint32_t *count, uint32_t mode, uint32_t v, bool is_clear,
                                               uint64_t limit, uint32_t *observed)
{
    uint32_t spins = 0;
    uint64_t deadline = 0;
    for (;;) {
        const uint32_t c = ld_relaxed_scoped<S>(count);
        if (cnt_wait_released(c, mode, v)) {
            fence_acquire_scoped<S>();
            if (observed)
                *observed = c;
            if (is_clear)
                atom_exch_relaxed_scoped<S>(count, 0u);
            return CNS_SUCCESS;
        }
        if ((++spins & 63u) == 0u) {
            const uint64_t now = globaltimer_ns();
            if (deadline == 0)
                deadline = now + limit;
            else if (now > deadline)
                return CNS_ERR_TIMEOUT;
        }
    }
}

}  // namespace cns

/* One record on a counted notify's count word: SET, ADD, BIT_OR or BIT_AND
 * with value v, one release atomic (the caller's earlier writes are visible
 * to whoever is released by it).  Any thread may call it; each call is one
 * record.  Other modes do nothing (the host API refuses them). */
__device__ __forceinline__ void cns_cnt_record_dev(uint32_t *count, int mode, uint32_t v)
{
    cns::cnt_record_device(count, static_cast<uint32_t>(mode), v);
}

/* Wait, from the calling thread only, until the count word satisfies
 * (mode, v); then, with is_clear, set it to 0 (an exchange right after the
 * release was seen).  Polls with relaxed loads and takes one acquire fence
 * once released, so the records' earlier writes are visible afterwards.
 * timeout_ns = 0 means 2 s.  Returns CNS_SUCCESS, CNS_ERR_TIMEOUT, or
 * CNS_ERR_INVALID_VALUE for a mode outside 0..4; *observed (if not NULL)
 * gets the count that released the wait. */
__device__ __forceinline__ int cns_cnt_wait_dev(uint32_t *count, int mode, uint32_t v, int is_clear,
                                                uint64_t timeout_ns, uint32_t *observed)
{
    if (mode < 0 || mode > 4)
        return CNS_ERR_INVALID_VALUE;
    return cns::cnt_wait_scoped<cns::kScopeGpu>(count, static_cast<uint32_t>(mode), v, is_clear != 0,
                                                timeout_ns ? timeout_ns : 2000000000ull, observed);
}

/* cns_cnt_record_dev at system scope: for a count word that threads of other
 * GPUs also record on or wait on (a notify prepared by cntnotify_enable_peer,
 * recorded from a peer GPU through the same address).  The caller's earlier
 * writes, to any GPU's memory, are visible to whoever is released by it. */
__device__ __forceinline__ void cns_cnt_record_sys_dev(uint32_t *count, int mode, uint32_t v)
{
    cns::cnt_record_scoped<cns::kScopeSys>(count, static_cast<uint32_t>(mode), v);
}

/* cns_cnt_wait_dev at system scope: released by records made at system scope
 * on any GPU (cntnotify_record on a notify prepared by cntnotify_enable_peer,
 * or cns_cnt_record_sys_dev); the count word may live on another GPU, reached
 * through a peer mapping.  Same arguments and results as cns_cnt_wait_dev. */
__device__ __forceinline__ int cns_cnt_wait_sys_dev(uint32_t *count, int mode, uint32_t v, int is_clear,
                                                    uint64_t timeout_ns, uint32_t *observed)
{
    if (mode < 0 || mode > 4)
        return CNS_ERR_INVALID_VALUE;
    return cns::cnt_wait_scoped<cns::kScopeSys>(count, static_cast<uint32_t>(mode), v, is_clear != 0,
                                                timeout_ns ? timeout_ns : 2000000000ull, observed);
}

namespace cns {

// The bounded poll of cns_cnt_wait_grid_dev: on word w until ok(value), or
// until go[1] is raised or the time runs out (then it raises go[1] itself if
// it is still 0).  The value that passed goes to *seen if given.
template <class Ok>
__device__ __forceinline__ int grid_wait_poll(const uint32_t *w, Ok ok, uint32_t *go, uint64_t limit,
                                              uint32_t *seen)
{
    uint32_t spins = 0;
    uint64_t deadline = 0;
    for (;;) {
        const uint32_t c = ld_relaxed_gpu(w);
        if (ok(c)) {
            fence_acquire_gpu();
            if (seen)
                *seen = c;
            return CNS_SUCCESS;
        }
        if ((++spins & 63u) == 0u) {
            if (ld_relaxed_gpu(go + 1) != 0u)
                return CNS_ERR_TIMEOUT;
            const uint64_t now = globaltimer_ns();
            if (deadline == 0) {
                deadline = now + limit;
            } else if (now > deadline) {
                atom_cas_relaxed_gpu(go + 1, 0u, static_cast<uint32_t>(CNS_ERR_TIMEOUT));
                return CNS_ERR_TIMEOUT;
            }
        }
    }
}

}  // namespace cns

/* A counted-notify wait taken by several CTAs of a grid together, call after
 * call (CntNotify §3.2 with isClear, for a consumer that is a whole grid).
 * They cannot all poll the count: once one of them had cleared it, a CTA
 * that had not yet looked would wait until its timeout.  So thread 0 of CTA
 * 0 waits on the count (mode, v), clears it if is_clear, and then publishes
 * the call on go[0] (release); thread 0 of every other calling CTA waits
 * until go[0] shows the call.  CTA 0 first waits for go[0] to show the
 * previous call, so when grids that follow one another overlap, the count it
 * then looks at was cleared by the call before.  Writes released by the
 * records are visible to every thread of the calling CTAs afterwards.
 *   count       the notify's count word (cntnotify_get_device_ptr)
 *   go          two words on a line of their own, zeroed before the first
 *               call and shared by no other grid-wide wait: go[0] counts the
 *               calls published, go[1] holds the first failure's code
 *   call        the call's index, 0, 1, 2, ..., the same in every CTA (a grid
 *               that follows another continues its count)
 *   timeout_ns  per wait; 0 = 2 s.  A wait that runs out stores
 *               CNS_ERR_TIMEOUT in go[1] (if it is still 0), and the other
 *               CTAs' waits then give up too
 *   observed    if not NULL, CTA 0 stores the count that released its wait
 * All threads of every calling CTA call it, and CTA 0 must be among them.
 * With is_clear, the records meant for call r must land after call r - 1 has
 * cleared the count, or that clear wipes them and call r waits until its
 * timeout.  A producer that may run ahead of the consumer therefore records
 * for call r only once it has seen go[0] >= r (call r - 1 published after its
 * clear), or after some other event ordered after that clear.  With
 * is_clear = 0 there is no such rule: nothing is wiped.
 * The CTAs other than 0 wait up to twice the limit for go[0]: CTA 0 may take
 * one limit for the previous call's go and one for the count.
 * Returns, in every thread, CNS_SUCCESS, CNS_ERR_TIMEOUT (this or an earlier
 * call failed: go[1] stays set until the caller zeroes it, and every later
 * call fails at once until then), or CNS_ERR_INVALID_VALUE for a mode outside
 * 0..4 (no wait taken). */
__device__ __forceinline__ int cns_cnt_wait_grid_dev(uint32_t *count, uint32_t *go, uint32_t call, int mode,
                                                     uint32_t v, int is_clear, uint64_t timeout_ns,
                                                     uint32_t *observed)
{
    if (mode < 0 || mode > 4)
        return CNS_ERR_INVALID_VALUE;
    int rc = CNS_SUCCESS;
    if (threadIdx.x == 0) {
        const uint64_t limit = timeout_ns ? timeout_ns : 2000000000ull;
        const uint32_t m = static_cast<uint32_t>(mode);
        if (cns::ld_relaxed_gpu(go + 1) != 0u) {
            rc = CNS_ERR_TIMEOUT;
        } else if (blockIdx.x == 0) {
            uint32_t seen = 0;
            rc = cns::grid_wait_poll(go, [=](uint32_t g) { return static_cast<int32_t>(g - call) >= 0; }, go, limit,
                                     nullptr);
            if (rc == CNS_SUCCESS)
                rc = cns::grid_wait_poll(count, [=](uint32_t c) { return cns::cnt_wait_released(c, m, v); }, go,
                                         limit, &seen);
            if (rc == CNS_SUCCESS) {
                if (observed)
                    *observed = seen;
                if (is_clear)
                    cns::atom_exch_relaxed_gpu(count, 0u);   // the clear comes after the release ...
                cns::st_release_gpu(go, call + 1u);          // ... and before the call is published
            }
        } else {
            // CTA 0 may spend one limit on the previous call's go and one on
            // the count before it publishes: wait for both
            const uint32_t next = call + 1u;
            rc = cns::grid_wait_poll(go, [=](uint32_t g) { return static_cast<int32_t>(g - next) >= 0; }, go,
                                     2u * limit, nullptr);
        }
    }
    return __syncthreads_or(rc != CNS_SUCCESS) ? CNS_ERR_TIMEOUT : CNS_SUCCESS;
}

namespace cns {

// The soft barrier of cns_syncall_soft at scope S (kScopeSys: participants on
// several GPUs, the workspace reached through peer mappings).
template <int S>
__device__ __forceinline__ int syncall_soft_scoped(void *workspace, uint32_t participants, uint64_t timeout_ns)
{
    if (participants == 0u)
        return CNS_ERR_INVALID_VALUE;
    uint32_t *ctr = static_cast<uint32_t *>(workspace);
    uint32_t *status = ctr + CNS_SYNCALL_LINE_BYTES / 4;
    int stop = 0;
    __syncthreads();
    if (threadIdx.x == 0 && threadIdx.y == 0 && threadIdx.z == 0) {
        const Epoch e = epoch_of(participants);
        const uint32_t before = (S == kScopeSys) ? atom_inc_release_sys(ctr, e.Mm1) : atom_inc_release_gpu(ctr, e.Mm1);
        const uint32_t target = epoch_target(before, e);
        const uint32_t mine = (before == e.Mm1) ? 0u : before + 1u;
        if (epoch_reached(mine, target, e)) {
            fence_acquire_scoped<S>();   // the last arrival: its increment read every other one's
        } else {
            const uint64_t limit = timeout_ns ? timeout_ns : 2000000000ull;
            uint32_t spins = 0;
            uint64_t deadline = 0;
            for (;;) {
                if (epoch_reached(ld_relaxed_scoped<S>(ctr), target, e)) {
                    fence_acquire_scoped<S>();
                    break;
                }
                if ((++spins & 63u) == 0u) {
                    if (ld_relaxed_scoped<S>(status + 1) != 0u) {
                        stop = 1;
                        break;
                    }
                    const uint64_t now = globaltimer_ns();
                    if (deadline == 0) {
                        deadline = now + limit;
                    } else if (now > deadline) {
                        const uint32_t code = static_cast<uint32_t>(CNS_ERR_TIMEOUT);
                        if constexpr (S == kScopeSys) {
                            if (atom_cas_relaxed_sys(status, 0u, code) == 0u)
                                st_relaxed_sys(status + 3, blockIdx.x);
                            atom_exch_release_sys(status + 1, 1u);
                        } else {
                            if (atom_cas_relaxed_gpu(status, 0u, code) == 0u)
                                st_relaxed_gpu(status + 3, blockIdx.x);
                            atom_exch_release_gpu(status + 1, 1u);
                        }
                        stop = 1;
                        break;
                    }
                }
            }
        }
    }
    return __syncthreads_or(stop) ? CNS_ERR_TIMEOUT : CNS_SUCCESS;
}

}  // namespace cns

/* The soft SYNCALL barrier among CTAs 0 .. participants - 1 of the grid.
 * Every thread of each participating CTA calls it, the same number of times
 * in each CTA; CTAs with blockIdx.x >= participants must not call it.  The
 * CTA's threads first finish what they were doing (a block barrier), one
 * thread arrives with an increment of the workspace's soft counter (line 0,
 * word 0; release), takes target = (before / P + 1) * P in the wrap-safe
 * counter arithmetic of syncall_run, and polls until the count reaches it
 * (the last arrival of a round skips the poll); a second block barrier
 * releases the CTA.  Writes made by any participant before its call are
 * visible to every participant after the barrier.
 *   workspace    CNS_SYNCALL_WORKSPACE_BYTES, 128-byte aligned, prepared by
 *                syncall_workspace_init (start 0 or a multiple of P; again
 *                whenever P changes) and used by no other barrier at the
 *                same time
 *   timeout_ns   per wait; 0 = 2 s.  A wait that runs out records
 *                CNS_ERR_TIMEOUT in the workspace status line (line 1, with
 *                the CTA that gave up) and raises its abort flag; the other
 *                participants' waits then give up too.
 * Returns CNS_SUCCESS, or CNS_ERR_TIMEOUT in every thread of the CTA once
 * the barrier failed (the caller should then leave its kernel);
 * CNS_ERR_INVALID_VALUE without arriving when participants is 0. */
__device__ __forceinline__ int cns_syncall_soft(void *workspace, uint32_t participants, uint64_t timeout_ns)
{
    return cns::syncall_soft_scoped<cns::kScopeGpu>(workspace, participants, timeout_ns);
}

/* cns_syncall_soft at system scope, for participants on several GPUs (the
 * SYNCALL barrier across devices): every participating CTA of every GPU
 * calls it with the same workspace -- one syncall_workspace_init prepared on
 * one GPU, reached from the others through a peer mapping (the caller
 * enables peer access, cudaDeviceEnablePeerAccess, from each other GPU to
 * the workspace's) -- and `participants` = the participating CTAs of all
 * GPUs together.  Arrivals are system-scope release increments and the wait
 * acquires at system scope, so each GPU's writes before the barrier are
 * visible to every participant after it.  The caller makes every
 * participating CTA of every GPU co-resident for the whole run, as for
 * cns_syncall_soft; a participant that never arrives ends the others' wait
 * in CNS_ERR_TIMEOUT.  Same results and status line as cns_syncall_soft. */
__device__ __forceinline__ int cns_syncall_soft_sys(void *workspace, uint32_t participants, uint64_t timeout_ns)
{
    return cns::syncall_soft_scoped<cns::kScopeSys>(workspace, participants, timeout_ns);
}

/* Per-CTA state of cns_syncall_soft_die_local, held by the caller (shared
 * memory, one per CTA) and set to CNS_SOFT_STATE_INIT before the CTA's first
 * barrier: which copy is near, and the epoch the last barrier closed. */
typedef struct {
    uint32_t start, end;   /* the last barrier's target and the next one */
    int32_t valid;         /* 0 before the first barrier */
    int32_t near;          /* -1 until the first barrier has timed both copies; then 0 or 1 */
} cns_soft_state_t;
#define CNS_SOFT_STATE_INIT {0u, 0u, 0, -1}

/* cns_syncall_soft on the two counter copies of a die-local workspace
 * (CNS_SYNCALL_WORKSPACE_DIE_LOCAL_BYTES, 8 KB-aligned: see
 * CNS_SYNCALL_DIE_LOCAL_ALIGN), as syncall_run's CNS_BARRIER_DIE_LOCAL does:
 * each CTA arrives on both copies and polls the one on its own die.  Same
 * contract as cns_syncall_soft, plus `state`: one cns_soft_state_t per CTA
 * (in shared memory), CNS_SOFT_STATE_INIT before the first call, passed to
 * every call by every thread of the CTA, and not touched by the caller in
 * between.  The first call times both copies (~16 atomics). */
__device__ __forceinline__ int cns_syncall_soft_die_local(void *workspace, uint32_t participants,
                                                          uint64_t timeout_ns, cns_soft_state_t *state)
{
    if (participants == 0u)
        return CNS_ERR_INVALID_VALUE;
    uint32_t *w = static_cast<uint32_t *>(workspace);
    uint32_t *status = w + CNS_SYNCALL_LINE_BYTES / 4;
    int stop = 0;
    __syncthreads();
    if (threadIdx.x == 0 && threadIdx.y == 0 && threadIdx.z == 0) {
        uint32_t *c0 = w, *c1 = w + CNS_SYNCALL_REPLICA_OFFSET / 4;
        if (state->near < 0)
            state->near = cns::copy_is_farther(c0, c1) ? 1 : 0;
        uint32_t *nr = state->near ? c1 : c0, *fr = state->near ? c0 : c1;
        const cns::Epoch e = cns::epoch_of(participants);
        cns::EpochCursor cur{state->start, state->end, state->valid != 0};
        uint32_t target;
        const uint32_t before = cns::copies_arrive<true>(nr, fr, e, cur, &target);
        const uint32_t mine = (before == e.Mm1) ? 0u : before + 1u;
        if (cns::epoch_reached(mine, target, e)) {
            cns::fence_acquire_gpu();   // the round's last arrival on this copy
        } else {
            const uint64_t limit = timeout_ns ? timeout_ns : 2000000000ull;
            uint32_t spins = 0;
            uint64_t deadline = 0;
            for (;;) {
                if (cns::epoch_reached(cns::ld_relaxed_gpu(nr), target, e)) {
                    cns::fence_acquire_gpu();
                    break;
                }
                if ((++spins & 63u) == 0u) {
                    if (cns::ld_relaxed_gpu(status + 1) != 0u) {
                        stop = 1;
                        break;
                    }
                    const uint64_t now = cns::globaltimer_ns();
                    if (deadline == 0) {
                        deadline = now + limit;
                    } else if (now > deadline) {
                        if (cns::atom_cas_relaxed_gpu(status, 0u, static_cast<uint32_t>(CNS_ERR_TIMEOUT)) == 0u)
                            cns::st_relaxed_gpu(status + 3, blockIdx.x);
                        cns::atom_exch_release_gpu(status + 1, 1u);
                        stop = 1;
                        break;
                    }
                }
            }
        }
        cns::epoch_advance(cur, target, e);
        state->start = cur.start;
        state->end = cur.end;
        state->valid = 1;
    }
    return __syncthreads_or(stop) ? CNS_ERR_TIMEOUT : CNS_SUCCESS;
}

#endif /* __CUDACC__ */

#endif /* CNS_DEVICE_H */
