// syncall_kernels.cuh -- the device side of SYNCALL: the persistent
// multi-round kernel (data phase, then barrier, R times), its data phases and
// its solo form, shared by the translation units that instantiate its kernel
// tables (syncall_soft_kernels.cu, syncall_hard_kernels.cu,
// syncall_paired_kernels.cu; compiled in parallel) and by syncall.cu, which
// holds the host entry points.
//
// The barrier is the soft-mode epoch barrier of the "PTO-ISA SYNCALL
// cross-core barrier guide" (§5.2: arrive with an atomic increment that
// returns `before`, target = (before / P + 1) * P, poll until reached) or its
// hard counterpart built on thread-block clusters (§5.1's two-level shape).
#pragma once

#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

#include "cns.h"
#include "cns_device.cuh"

namespace cns {

struct SyncallParams {
    void *buf0;
    void *buf1;
    int64_t elems;          // ring: slots per participant; Jacobi: field length
    int64_t rounds;
    Barrier bar;            // counter, release word, status line, epoch, timeout, variant
    int32_t *cta_status;    // optional per-CTA marks
    uint32_t P;             // participants (ring length / Jacobi chunks)
    uint32_t group;         // MIX group size, else 1
    int32_t core_type;
    int32_t solo;           // soft path, thread 0 alone touches memory: the other threads leave at once
    uint32_t *mirror;       // die-local rings: the per-die payload copies (see mirror_row), else null
    uint32_t mirror_rows;   // rows per 4 KB block of the copies
    uint32_t mirror_region4;// uint4 per region (the copies of one round parity)
};

// ---------------------------------------------------------------------------
// Data phases
// ---------------------------------------------------------------------------

template <int WL>
__device__ __forceinline__ uint32_t ring_op(uint32_t x, uint32_t r)
{
    if (WL == CNS_WL_RING_AFFINE)
        return x * 3u + r;
    if (WL == CNS_WL_XORSHIFT) {
        // Marsaglia's xorshift32 step, shifts (13, 17, 5), then the round index
        x ^= x << 13;
        x ^= x >> 17;
        x ^= x << 5;
        return x ^ r;
    }
    return x;   // ring rotate
}

// Participant p writes its own row of dst from row (p + 1) mod P of src.
// The rows are exchanged between SMs every round, so they are read and
// written with relaxed gpu-scope accesses, which L2 serves directly: with
// 1 KB rows (P = 8 ring-affine, the xorshift rings) a round took 70-170 ns
// less than with plain accesses through L1; the 16-byte rows of the
// 148-CTA ring-rotate did not change.
template <int WL>
__device__ __forceinline__ void ring_phase(const uint32_t *src, uint32_t *dst, uint32_t p, uint32_t P,
                                           int64_t elems, uint32_t r)
{
    const uint32_t q = (p + 1u == P) ? 0u : p + 1u;
    const uint32_t *s = src + static_cast<int64_t>(q) * elems;
    uint32_t *d = dst + static_cast<int64_t>(p) * elems;
    if ((elems & 3) == 0) {
        const uint4 *s4 = reinterpret_cast<const uint4 *>(s);
        uint4 *d4 = reinterpret_cast<uint4 *>(d);
        const int64_t n4 = elems >> 2;
        for (int64_t i = threadIdx.x; i < n4; i += blockDim.x) {
            uint4 v = ld_relaxed_gpu_v4(s4 + i);
            v.x = ring_op<WL>(v.x, r);
            v.y = ring_op<WL>(v.y, r);
            v.z = ring_op<WL>(v.z, r);
            v.w = ring_op<WL>(v.w, r);
            st_relaxed_gpu_v4(d4 + i, v);
        }
    } else {
        for (int64_t i = threadIdx.x; i < elems; i += blockDim.x)
            st_relaxed_gpu(d + i, ring_op<WL>(ld_relaxed_gpu(s + i), r));
    }
}

// One Jacobi sweep over participant p's chunk of the field:
// u'[i] = (u[i-1] + u[i+1]) * 0.5f for interior points, ends copied.
// The field is cut into N/4 float4 columns shared out as evenly as possible.
// The chunk is streamed through shared memory in tiles of kJacTile float4:
// thread 0 arms an mbarrier and starts one bulk copy (TMA engine) of the
// tile plus one float4 of halo on each side; every thread then waits for it,
// computes its outputs from shared memory and stores them with plain float4
// stores.  One tile in flight per CTA and four CTAs per SM measured fastest
// on GB300 (deeper pipelines and register-only streaming were slower).  The
// scalar tail (N mod 4 points) belongs to the last participant.
constexpr int kJacTile = 1024;
constexpr uint32_t kJacSmemBytes = (kJacTile + 2) * 16;

struct JacState {
    float4 *stage;     // kJacTile + 2 float4 of shared memory
    uint64_t *bar;     // its mbarrier
    uint32_t parity;   // phase to wait for next
    int *flag;         // shared: a wait in this sweep gave up
};

// One output float4 column j of a sweep from its input v, the last float of
// the column on its left (lw) and the first float on its right (rx).
__device__ __forceinline__ float4 jacobi_column(const float4 v, float lw, float rx, int64_t j, int64_t N)
{
    float4 o;
    o.x = (j == 0) ? v.x : (lw + v.y) * 0.5f;
    o.y = (v.x + v.z) * 0.5f;
    o.z = (v.y + v.w) * 0.5f;
    o.w = (4 * j + 3 == N - 1) ? v.w : (v.z + rx) * 0.5f;
    return o;
}

// Participant p's float4 columns [j0, j1): N/4 columns shared out as evenly as possible.
__device__ __forceinline__ void jacobi_chunk(int64_t N4, uint32_t p, uint32_t P, int64_t *j0, int64_t *j1)
{
    const int64_t base = N4 / P, rem = N4 % P;
    *j0 = static_cast<int64_t>(p) * base + (p < rem ? p : rem);
    *j1 = *j0 + base + (p < rem ? 1 : 0);
}

// Sweep of columns [c0, c1) through shared memory.  The bulk copies read
// columns clipped to [r0, r1): the whole field for a full sweep; only the
// participant's own chunk for the interior of a split-phase sweep, which
// then needs nothing another participant wrote.  Returns after the columns;
// a bulk copy that never completes within the barrier timeout is recorded as
// CNS_ERR_TIMEOUT (the round's barrier then stops every participant).
__device__ __forceinline__ void jacobi_tiles(const float *src, float *dst, int64_t N, int64_t c0, int64_t c1,
                                             int64_t r0, int64_t r1, JacState &js, uint32_t *status_line,
                                             uint64_t timeout_ns, uint32_t round)
{
    const int64_t N4 = N >> 2;
    const int64_t nT = (c1 > c0) ? (c1 - c0 + kJacTile - 1) / kJacTile : 0;
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
    float4 *d4 = reinterpret_cast<float4 *>(dst);
    for (int64_t k = 0; k < nT; ++k) {
        const int64_t o0 = c0 + k * kJacTile;
        const int64_t o1 = (o0 + kJacTile < c1) ? o0 + kJacTile : c1;
        if (threadIdx.x == 0) {
            // the stage was read by everyone (barrier below / previous round)
            // and src was written by generic stores: order both before the copy
            if (k == 0)
                fence_proxy_async_global();
            fence_proxy_async_shared();
            const int64_t lo = (o0 - 1 < r0) ? r0 : o0 - 1;
            const int64_t hi = (o1 + 1 > r1) ? r1 : o1 + 1;
            const uint32_t bytes = static_cast<uint32_t>((hi - lo) * 16);
            mbar_arrive_expect_tx(js.bar, bytes);
            bulk_copy_g2s(js.stage + (lo - (o0 - 1)), s4 + lo, bytes, js.bar);
        }
        // bounded wait for the tile: every thread observes the completion
        uint32_t spins = 0;
        uint64_t deadline = 0;
        bool ok = true;
        while (!mbar_try_wait(js.bar, js.parity)) {
            if ((++spins & 63u) == 0u) {
                const uint64_t now = globaltimer_ns();
                if (deadline == 0) {
                    deadline = now + timeout_ns;
                } else if (now > deadline) {
                    ok = false;
                    break;
                }
            }
        }
        if (!ok)
            *js.flag = 1;
        js.parity ^= 1u;
        const float4 *t = js.stage;   // t[i] holds column o0 - 1 + i
        for (int64_t j = o0 + threadIdx.x; j < o1 && ok; j += blockDim.x) {
            const int i = static_cast<int>(j - o0) + 1;
            const float lw = (j > 0) ? t[i - 1].w : 0.f;
            const float rx = (j + 1 < N4) ? t[i + 1].x : ((4 * j + 4 < N) ? src[4 * j + 4] : 0.f);
            d4[j] = jacobi_column(t[i], lw, rx, j, N);
        }
        __syncthreads();   // everyone is done with the stage (and sees the flag)
        if (*js.flag) {
            if (threadIdx.x == 0)
                raise_timeout(status_line, round, blockIdx.x);
            return;
        }
    }
}

// The scalar tail (N mod 4 points) belongs to the last participant.
__device__ __forceinline__ void jacobi_tail(const float *src, float *dst, int64_t N, uint32_t p, uint32_t P)
{
    if (p == P - 1) {
        for (int64_t i = 4 * (N >> 2) + threadIdx.x; i < N; i += blockDim.x)
            dst[i] = (i == 0 || i == N - 1) ? src[i] : (src[i - 1] + src[i + 1]) * 0.5f;
    }
}

// One Jacobi sweep over participant p's chunk (fused barrier form).
__device__ __forceinline__ void jacobi_phase(const float *src, float *dst, int64_t N, uint32_t p, uint32_t P,
                                             JacState &js, uint32_t *status_line, uint64_t timeout_ns,
                                             uint32_t round)
{
    int64_t j0, j1;
    jacobi_chunk(N >> 2, p, P, &j0, &j1);
    jacobi_tiles(src, dst, N, j0, j1, 0, N >> 2, js, status_line, timeout_ns, round);
    if (*js.flag)
        return;
    jacobi_tail(src, dst, N, p, P);
}

// The part of a split-phase sweep that waits for the previous round's
// barrier: the chunk's first and last column (they read the neighbours'
// columns), straight from global memory, and the tail.
__device__ __forceinline__ void jacobi_edges(const float *src, float *dst, int64_t N, uint32_t p, uint32_t P)
{
    const int64_t N4 = N >> 2;
    int64_t j0, j1;
    jacobi_chunk(N4, p, P, &j0, &j1);
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
    float4 *d4 = reinterpret_cast<float4 *>(dst);
    if (threadIdx.x < 2 && j1 > j0) {
        const int64_t j = (threadIdx.x == 0) ? j0 : j1 - 1;
        if (threadIdx.x == 0 || j > j0) {
            const float lw = (j > 0) ? s4[j - 1].w : 0.f;
            const float rx = (j + 1 < N4) ? s4[j + 1].x : ((4 * j + 4 < N) ? src[4 * j + 4] : 0.f);
            d4[j] = jacobi_column(s4[j], lw, rx, j, N);
        }
    }
    jacobi_tail(src, dst, N, p, P);
}

template <int WL>
__device__ __forceinline__ void data_phase(const SyncallParams &p, int64_t r, uint32_t part, JacState &js)
{
    if (WL == CNS_WL_EMPTY)
        return;
    const bool odd = (r & 1) != 0;
    void *src = odd ? p.buf1 : p.buf0;
    void *dst = odd ? p.buf0 : p.buf1;
    if (WL == CNS_WL_JACOBI)
        jacobi_phase(static_cast<const float *>(src), static_cast<float *>(dst), p.elems, part, p.P, js,
                     p.bar.status_line, p.bar.timeout_ns, static_cast<uint32_t>(r));
    else
        ring_phase<WL>(static_cast<const uint32_t *>(src), static_cast<uint32_t *>(dst), part, p.P, p.elems,
                       static_cast<uint32_t>(r));
}

// ---------------------------------------------------------------------------
// The persistent kernel
// ---------------------------------------------------------------------------

// Words of the workspace's status line (line 1) beyond the status itself.
constexpr uint32_t kBaseWordSoft = 5;   // base count of the soft counter
constexpr uint32_t kBaseWordHard = 6;   // base count of the hard counter
constexpr uint32_t kTagWord = 7;        // CNS_SYNCALL_WORKSPACE_TAG, _TAG_FLIP or 0

// Whether the workspace check refuses a run: a tag the library did not write
// (0 is accepted with a base of 0: a zeroed workspace), or, for the variants
// on the pages' arithmetic, a base count that is not a multiple of P below M
// (it would put the participants in different epochs).  The sense-flip
// variant checks its own count at every arrival.
template <int V>
__device__ __forceinline__ bool workspace_refused(uint32_t tag, uint32_t base, const Epoch &e)
{
    if constexpr (V == kBvSenseFlip) {
        return !(tag == CNS_SYNCALL_WORKSPACE_TAG || tag == CNS_SYNCALL_WORKSPACE_TAG_FLIP || tag == 0u);
    } else {
        const bool tag_ok = tag == CNS_SYNCALL_WORKSPACE_TAG || (tag == 0u && base == 0u);
        return !tag_ok || base > e.Mm1 || base % e.P != 0u;
    }
}

__device__ __forceinline__ uint32_t cta_role(const SyncallParams &p, uint32_t b)
{
    if (p.core_type == CNS_MIX)
        return (b % p.group == 0) ? 1u : 0u;   // group rank 0 plays the AIC part
    return p.core_type == CNS_AIC_ONLY ? 1u : 0u;
}

// The workspace check's decision for the calling thread (see
// workspace_refused), reading the status, abort, tag and base words.
template <int V>
__device__ __forceinline__ bool workspace_check_refuses(const Barrier &bar, const uint32_t *base_word, uint32_t *base)
{
    const uint32_t tag = ld_relaxed_gpu(bar.status_line + kTagWord);
    *base = ld_relaxed_gpu(base_word);
    // a status or abort flag left by an earlier run that failed
    const bool failed = (ld_relaxed_gpu(bar.status_line) | ld_relaxed_gpu(bar.status_line + 1)) != 0u;
    return failed || workspace_refused<V>(tag, *base, bar.e);
}

// A refused run: CTA 0 reports it (keeping an earlier failure's code;
// anything else in the status word, garbage, becomes INVALID_VALUE).
__device__ __forceinline__ void report_refusal(const Barrier &bar, uint32_t b)
{
    if (b != 0)
        return;
    const uint32_t cur = ld_relaxed_gpu(bar.status_line);
    if (cur != static_cast<uint32_t>(CNS_ERR_TIMEOUT) && cur != static_cast<uint32_t>(CNS_ERR_INVALID_VALUE)) {
        st_relaxed_gpu(bar.status_line + 2, 0u);
        st_relaxed_gpu(bar.status_line + 3, 0u);
        st_relaxed_gpu(bar.status_line, static_cast<uint32_t>(CNS_ERR_INVALID_VALUE));
    }
    atom_exch_release_gpu(bar.status_line + 1, 1u);
}

// After a run that CTA 0 finished without a failure: every arrival of the run
// has landed once CTA 0 is past its last barrier, so the counter stands at
// base + rounds * P (mod M); that becomes the base count.
template <int V>
__device__ __forceinline__ void record_base(const SyncallParams &p, const Barrier &bar, uint32_t *base_word,
                                            uint32_t base)
{
    if constexpr (V == kBvSenseFlip) {
        st_relaxed_gpu(bar.status_line + kTagWord, CNS_SYNCALL_WORKSPACE_TAG_FLIP);
    } else {
        const uint64_t M = static_cast<uint64_t>(bar.e.Mm1) + 1u;
        const uint64_t steps = static_cast<uint64_t>(p.rounds) % (M / bar.e.P);
        st_relaxed_gpu(base_word, static_cast<uint32_t>((base + steps * bar.e.P) % M));
        st_relaxed_gpu(bar.status_line + kTagWord, CNS_SYNCALL_WORKSPACE_TAG);
    }
}

// The per-die payload copies of a ring (die-local variant, rows of a multiple
// of 16 bytes up to 4080, on a workspace of syncall_workspace_bytes(P, elems)).
// After the die-local counters come two regions, one per round parity: region
// k holds the state that rounds of parity k read.  A region is a run of 8 KB
// pairs of 4 KB blocks; row p sits in pair p / rows at slot p % rows of BOTH
// blocks (rows = floor(4080 / row bytes); the last 16 bytes of every block
// are never a row: they are the word each CTA times to find its near block).
// The two blocks of a pair differ in address bit 12, so they sit on different
// dies.  A participant writes its new row into both blocks of its pair and
// reads its neighbour's row from the block of the neighbour's pair that is
// on its own die, so every payload load stays on its die.  Round 0 reads the
// caller's buffer 0, and the last two rounds also write the caller's buffers,
// which then end exactly as without copies.
constexpr uint32_t kMirrorPair4 = 512;       // uint4 per 8 KB pair
constexpr uint32_t kMirrorBlock4 = 256;      // uint4 per 4 KB block
constexpr uint32_t kMirrorTiming4 = kMirrorBlock4 - 1;   // the timing slot of a block: never a row

// A row's place in a region: uint4 offset of its slot in block 0 of its pair
// (block 1 is kMirrorBlock4 further on).
__device__ __forceinline__ uint32_t mirror_slot(const SyncallParams &p, uint32_t row, uint32_t row4)
{
    const uint32_t pair = row / p.mirror_rows;
    return pair * kMirrorPair4 + (row - pair * p.mirror_rows) * row4;
}

// Which block of the neighbour's pair is on this SM's die, in each region, as
// one word (bit k: block 1 in region k).  The rows' addresses are worked out
// from it each round with a few integer operations, so the state stays one
// register: kept as an array of pointers indexed by the round's parity it
// went to local memory (every payload load then first waited for a local load
// of its address, ~90 ns a round), and as six pointers it made the hard
// kernel, held to 64 registers by its 1024-thread bound, spill.
struct MirrorState {
    uint32_t near_bits;
};

// q_slot: mirror_slot of the neighbour's row.
__device__ __forceinline__ MirrorState mirror_setup(const SyncallParams &p, uint32_t q_slot)
{
    MirrorState m{0u};
    const uint32_t pair0 = q_slot - q_slot % kMirrorPair4;
    for (uint32_t k = 0; k < 2; ++k) {
        uint4 *b0 = reinterpret_cast<uint4 *>(p.mirror) + k * p.mirror_region4 + pair0;
        uint4 *b1 = b0 + kMirrorBlock4;
        // time both blocks on their timing slot (adds of 0: nothing changes)
        if (copy_is_farther(reinterpret_cast<uint32_t *>(b0 + kMirrorTiming4),
                            reinterpret_cast<uint32_t *>(b1 + kMirrorTiming4)))
            m.near_bits |= 1u << k;
    }
    return m;
}

// The addresses one participant's rows use through the copies, fixed for the
// whole run: round r reads the neighbour's row from region r & 1, in the block
// of its pair on this SM's die (from buffer 0 in round 0), and writes its own
// row into both blocks of region (r & 1) ^ 1 (and, in the last two rounds,
// into the caller's buffer: buffer 1 after an even round, 0 after an odd one).
// Worked out from the round number in every round instead, the addresses cost
// ~25 ns a round of the headline on the chain from the acquire to the stores.
struct MirrorRow {
    const uint4 *src0, *src1;   // the neighbour's row, region 0 / 1, near block
    uint4 *dst0, *dst1;         // this row, region 0 / 1, first block (the other is kMirrorBlock4 on)
    const uint4 *first;         // the neighbour's row in buffer 0 (round 0)
    uint4 *last0, *last1;       // this row in buffer 0 / 1
};

// q / b the neighbour's and this participant's index, row4 uint4 per row,
// q_slot / b_slot from mirror_slot, m from mirror_setup.
__device__ __forceinline__ MirrorRow mirror_row(const SyncallParams &p, MirrorState m, uint32_t q, uint32_t b,
                                                uint32_t row4, uint32_t q_slot, uint32_t b_slot)
{
    uint4 *base = reinterpret_cast<uint4 *>(p.mirror);
    MirrorRow w;
    w.src0 = base + q_slot + (m.near_bits & 1u) * kMirrorBlock4;
    w.src1 = base + p.mirror_region4 + q_slot + ((m.near_bits >> 1) & 1u) * kMirrorBlock4;
    w.dst0 = base + b_slot;
    w.dst1 = base + p.mirror_region4 + b_slot;
    w.first = static_cast<const uint4 *>(p.buf0) + static_cast<int64_t>(q) * row4;
    w.last0 = static_cast<uint4 *>(p.buf0) + static_cast<int64_t>(b) * row4;
    w.last1 = static_cast<uint4 *>(p.buf1) + static_cast<int64_t>(b) * row4;
    return w;
}

// Uint4 i of round r (of R) through the copies.
template <int WL>
__device__ __forceinline__ void mirror_move(const MirrorRow &w, int64_t r, int64_t R, uint32_t i)
{
    const bool odd = (r & 1) != 0;
    uint4 v = ld_relaxed_gpu_v4((r == 0 ? w.first : (odd ? w.src1 : w.src0)) + i);
    const uint32_t rr = static_cast<uint32_t>(r);
    v.x = ring_op<WL>(v.x, rr);
    v.y = ring_op<WL>(v.y, rr);
    v.z = ring_op<WL>(v.z, rr);
    v.w = ring_op<WL>(v.w, rr);
    uint4 *dst = (odd ? w.dst0 : w.dst1) + i;
    st_relaxed_gpu_v4(dst, v);
    st_relaxed_gpu_v4(dst + kMirrorBlock4, v);
    if (r + 2 >= R)
        st_relaxed_gpu_v4((odd ? w.last0 : w.last1) + i, v);
}

// The soft rounds when thread 0 alone touches memory (no payload, or a row of
// one uint4 or one word): the other threads of the CTA have left, and the
// barrier needs no drain and no closing block barrier -- thread 0 arrives
// and waits itself.  Same arithmetic, same memory operations otherwise.
template <int WL, int V>
__device__ __forceinline__ void solo_rounds(const SyncallParams &p, uint32_t b, uint32_t role)
{
    Barrier bar = p.bar;
    uint32_t *base_word = bar.status_line + kBaseWordSoft;
    uint32_t base = 0;
    if (workspace_check_refuses<V>(bar, base_word, &base)) {
        report_refusal(bar, b);
        if (p.cta_status)
            p.cta_status[b] = static_cast<int32_t>(CNS_CTA_ABORTED | (role << 8));
        return;
    }
    if constexpr (V == kBvDieLocal || V == kBvArrivalDieLocal)
        choose_near_copy(bar);
    MirrorState m{};
    const bool mirrored = (V == kBvDieLocal) && p.mirror != nullptr;
    const uint32_t q = (b + 1u == p.P) ? 0u : b + 1u;
    uint32_t q_slot = 0, b_slot = 0;   // one-uint4 rows
    if (mirrored) {
        q_slot = mirror_slot(p, q, 1u);
        b_slot = mirror_slot(p, b, 1u);
        m = mirror_setup(p, q_slot);
    }
    EpochCursor cursor{0u, 0u, false};
    bool stop = false;
    if (WL != CNS_WL_EMPTY && mirrored) {
        const MirrorRow w = mirror_row(p, m, q, b, 1u, q_slot, b_slot);
        const int64_t R = p.rounds;
        for (int64_t r = 0; r < R && !stop; ++r) {
            mirror_move<WL>(w, r, R, 0u);
            stop = arrive_and_wait<V>(bar, cursor, static_cast<uint32_t>(r), b);
        }
    } else {
        for (int64_t r = 0; r < p.rounds; ++r) {
            if (WL != CNS_WL_EMPTY) {
                const bool odd = (r & 1) != 0;
                ring_phase<WL>(static_cast<const uint32_t *>(odd ? p.buf1 : p.buf0),
                               static_cast<uint32_t *>(odd ? p.buf0 : p.buf1), b, p.P, p.elems,
                               static_cast<uint32_t>(r));
            }
            stop = arrive_and_wait<V>(bar, cursor, static_cast<uint32_t>(r), b);
            if (stop)
                break;
        }
    }
    if (b == 0 && !stop)
        record_base<V>(p, bar, base_word, base);
    if (p.cta_status)
        p.cta_status[b] = static_cast<int32_t>((stop ? CNS_CTA_ABORTED : CNS_CTA_DONE) | (role << 8));
}

// The same solo rounds in a kernel of their own, for CTAs of up to 256
// threads.  Within syncall_kernel they are held to the 64 registers a thread
// that its 1024-thread bound allows, and the headline round spilled there;
// here thread 0 has the registers it needs.  Same rounds, same memory
// operations.
template <int WL, int V>
__global__ void __launch_bounds__(256) syncall_solo_kernel(const SyncallParams p)
{
    if (threadIdx.x != 0)
        return;
    const uint32_t b = blockIdx.x;
    const uint32_t role = cta_role(p, b);
    if (b >= p.P) {
        // not a participant: never touches the counter ([SYNCALL] §4.2, §7.2)
        if (p.cta_status)
            p.cta_status[b] = static_cast<int32_t>(CNS_CTA_IDLE | (role << 8));
        return;
    }
    solo_rounds<WL, V>(p, b, role);
}

// STEP (hard path): kHardStepClusterBarrier or kHardStepPairedMbarrier, the
// intra-cluster step of each barrier.
template <int MODE, int WL, int V, int STEP = kHardStepClusterBarrier>
__global__ void __launch_bounds__(1024) syncall_kernel(const SyncallParams p)
{
    __shared__ int s_flag;
    __shared__ uint32_t s_epoch;   // hard path: the epoch the cluster leader hands on
    __shared__ __align__(8) uint64_t s_pair[2];   // paired step: gather and release mbarriers
    __shared__ uint32_t s_near_bits;              // payload copies: thread 0's timing, for every thread
    constexpr bool kPaired = MODE == CNS_SYNCALL_HARD && STEP == kHardStepPairedMbarrier;
    PairedBars pb{&s_pair[0], &s_pair[1], 0u, 0u};
    __shared__ __align__(8) uint64_t s_jac_bar;
    __shared__ int s_jac_flag;
    extern __shared__ float4 s_jac_stage[];   // JACOBI only: kJacSmemBytes
    const uint32_t b = blockIdx.x;
    const uint32_t role = cta_role(p, b);
    if (MODE == CNS_SYNCALL_SOFT && b >= p.P) {
        // not a participant: never touches the counter ([SYNCALL] §4.2, §7.2)
        if (threadIdx.x == 0 && p.cta_status)
            p.cta_status[b] = static_cast<int32_t>(CNS_CTA_IDLE | (role << 8));
        return;
    }
    if constexpr (MODE == CNS_SYNCALL_SOFT && WL != CNS_WL_JACOBI) {
        if (p.solo) {
            if (threadIdx.x == 0)
                solo_rounds<WL, V>(p, b, role);
            return;
        }
    }
    JacState js{s_jac_stage, &s_jac_bar, 0u, &s_jac_flag};
    if (threadIdx.x == 0) {
        s_flag = 0;
        if (kPaired)
            paired_bars_init(pb);
        if (WL == CNS_WL_JACOBI) {
            s_jac_flag = 0;
            mbar_init(&s_jac_bar, 1);
            mbar_init_fence();
        }
    }
    if (MODE == CNS_SYNCALL_HARD) {
        __syncwarp();
        cluster_sync_all();   // every CTA's flag is initialised before anyone may write it
    } else {
        __syncthreads();
    }

    // the elected thread's copy of the barrier description (variant 5 turns
    // its counter pair into near / far for this SM)
    Barrier bar = p.bar;
    if constexpr (MODE == CNS_SYNCALL_HARD) {
        // The hard path's participants are the clusters the launch really
        // has, and each cluster's members are the CTAs it really holds: both
        // come from the launch, not from the cluster size the host asked for
        // (a tool or a replay may launch the kernel without the cluster
        // attribute, and every CTA is then a cluster leader of its own).  The
        // observed size goes to the status line for the host to report.
        bar.e = epoch_of(nclusters_x());
        if (b == 0 && threadIdx.x == 0)
            st_relaxed_gpu(bar.status_line + 4, cluster_nctarank());
    }
    // The workspace check, before anyone arrives: every participant reads the
    // same words and takes the same decision, so a refused run leaves no CTA
    // behind at a barrier (see CNS_SYNCALL_WORKSPACE_TAG in cns.h).
    uint32_t *base_word = bar.status_line + (MODE == CNS_SYNCALL_SOFT ? kBaseWordSoft : kBaseWordHard);
    uint32_t base = 0;
    {
        int refuse = 0;
        if (threadIdx.x == 0)
            refuse = workspace_check_refuses<V>(bar, base_word, &base) ? 1 : 0;
        if (__syncthreads_or(refuse)) {
            if (threadIdx.x == 0) {
                report_refusal(bar, b);
                if (p.cta_status)
                    p.cta_status[b] = static_cast<int32_t>(CNS_CTA_ABORTED | (role << 8));
            }
            return;
        }
    }
    if ((V == kBvDieLocal || V == kBvArrivalDieLocal) && threadIdx.x == 0)
        choose_near_copy(bar);   // every CTA polls its own near copy (hard path: the leader arrives on both)
    EpochCursor cursor{0u, 0u, false};
    bool stop = false;
    if constexpr (MODE == CNS_SYNCALL_SOFT && WL == CNS_WL_JACOBI) {
        // Split phase: a sweep's interior columns read only this chunk's own
        // columns and overwrite only columns no neighbour reads, so they run
        // between this CTA's arrival at the previous round's barrier and its
        // wait; the chunk's first and last column (and the tail) follow the
        // wait.  Same barriers, same arithmetic; the wait overlaps the sweep.
        int64_t j0, j1;
        jacobi_chunk(p.elems >> 2, b, p.P, &j0, &j1);
        Pending pd{0u, true, false};
        for (int64_t r = 0; r < p.rounds; ++r) {
            const bool odd = (r & 1) != 0;
            const float *src = static_cast<const float *>(odd ? p.buf1 : p.buf0);
            float *dst = static_cast<float *>(odd ? p.buf0 : p.buf1);
            if (r == 0) {
                jacobi_phase(src, dst, p.elems, b, p.P, js, bar.status_line, bar.timeout_ns, 0u);
            } else {
                jacobi_tiles(src, dst, p.elems, j0 + 1, j1 - 1, j0, j1, js, bar.status_line, bar.timeout_ns,
                             static_cast<uint32_t>(r));
                stop = soft_wait<V>(bar, pd, static_cast<uint32_t>(r - 1));
                if (stop)
                    break;
                jacobi_edges(src, dst, p.elems, b, p.P);
            }
            soft_arrive<V>(bar, cursor, static_cast<uint32_t>(r), pd);
        }
        if (!stop && p.rounds > 0)
            stop = soft_wait<V>(bar, pd, static_cast<uint32_t>(p.rounds - 1));
    } else {
        // The rounds, in one of two forms fixed at compile time, so that the
        // form without payload copies carries none of their state (a run-time
        // branch inside one loop kept it live and made the 1 KB-row rings of
        // this kernel spill).  With copies (one-uint4 rings of the die-local
        // variant, on a workspace with room for them) thread 0 moves the row.
        auto rounds = [&](auto with_copies) {
            constexpr bool kCopies = decltype(with_copies)::value;
            uint32_t row4 = 0;
            MirrorRow w{};
            if constexpr (kCopies) {
                const uint32_t q = (b + 1u == p.P) ? 0u : b + 1u;
                row4 = static_cast<uint32_t>(p.elems >> 2);
                const uint32_t q_slot = mirror_slot(p, q, row4);
                if (threadIdx.x == 0)
                    s_near_bits = mirror_setup(p, q_slot).near_bits;
                __syncthreads();
                w = mirror_row(p, MirrorState{s_near_bits}, q, b, row4, q_slot, mirror_slot(p, b, row4));
            }
            bool halt = false;
            for (int64_t r = 0; r < p.rounds; ++r) {
                if constexpr (kCopies) {
                    for (uint32_t i = threadIdx.x; i < row4; i += blockDim.x)
                        mirror_move<WL>(w, r, p.rounds, i);
                } else {
                    data_phase<WL>(p, r, b, js);
                }
                if constexpr (MODE == CNS_SYNCALL_SOFT)
                    halt = soft_barrier<V>(bar, cursor, static_cast<uint32_t>(r));
                else if constexpr (kPaired)
                    halt = paired_barrier<V>(bar, cursor, static_cast<uint32_t>(r), &s_flag, pb);
                else
                    halt = hard_barrier<V>(bar, cursor, static_cast<uint32_t>(r), r == 0, &s_flag, &s_epoch);
                if (halt)
                    break;
            }
            return halt;
        };
        constexpr bool kRing = WL == CNS_WL_RING_AFFINE || WL == CNS_WL_RING_ROTATE || WL == CNS_WL_XORSHIFT;
        if constexpr (kRing && V == kBvDieLocal) {
            if (p.mirror != nullptr)
                stop = rounds(std::true_type{});
            else
                stop = rounds(std::false_type{});
        } else {
            stop = rounds(std::false_type{});
        }
        if constexpr (MODE == CNS_SYNCALL_HARD)
            stop = hard_barrier_finish(&s_flag);
    }
    if (threadIdx.x == 0 && b == 0 && !stop)
        record_base<V>(p, bar, base_word, base);
    if (threadIdx.x == 0 && p.cta_status)
        p.cta_status[b] = static_cast<int32_t>((stop ? CNS_CTA_ABORTED : CNS_CTA_DONE) | (role << 8));
}

// One kernel per (mode, workload, barrier variant[, hard step]), chosen on the
// host from tables that the kernel translation units build.
using KernelFn = void (*)(const SyncallParams);

KernelFn pick_soft_kernel(int wl, int variant);   // syncall_kernel<SOFT, wl, variant>
KernelFn pick_solo_kernel(int wl, int variant);   // syncall_solo_kernel<wl, variant>, wl < CNS_WL_JACOBI
KernelFn pick_hard_kernel(int wl, int variant);   // syncall_kernel<HARD, wl, variant>, cluster-barrier step
KernelFn pick_paired_kernel(int wl, int variant); // the hard path with the paired-mbarrier step

}  // namespace cns
