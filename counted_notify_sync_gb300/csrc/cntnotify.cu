// cntnotify.cu -- the counted notify ("CANN Runtime CntNotify management
// API"): a device-resident pool of counters, handle registry, stream-ordered
// record / wait / reset kernels, the op-stream state machine and the
// two-stream counting pipeline.
//
// Each notify owns one 128-byte line of the pool: word 0 is the count,
// word 1 a sticky status that a timed-out wait sets to CNS_ERR_TIMEOUT,
// word 2 an abort word used by the pipeline.  A record is one device atomic
// (release); a wait is one thread polling the count with acquire loads under
// a time bound, so the *stream* is blocked, not the host (§4.3).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>
#include <unordered_map>
#include <unordered_set>
#include <vector>

#include "cns.h"
#include "cns_device.cuh"
#include "cns_host.h"

struct cns_cnt_notify_s {
    uint32_t magic;
    int device;
    uint32_t slot;
    uint32_t *line;   // device: [0] count, [1] sticky status, [2] abort word
    // cntnotify_enable_peer: the devices (bit d) whose streams may record on
    // and wait on this notify besides its own, and whether its stream-ordered
    // operations run at system scope (set by the first enable)
    std::atomic<uint64_t> peers{0};
    std::atomic<int> sys{0};
};

namespace cns {

constexpr uint32_t kMagic = 0x434E5446u;   // "CNTF"
constexpr uint32_t kWordsPerSlot = 32;     // 128 B

struct Pool {
    uint32_t *base = nullptr;
    uint32_t cap = 0;
    std::vector<uint32_t> free_slots;   // LIFO
};

static std::mutex g_mu;
static std::unordered_map<int, Pool> g_pools;
static std::unordered_set<cns_cnt_notify_s *> g_live;

static uint32_t pool_cap()
{
    const char *e = std::getenv("CNS_POOL_CAP");
    if (e && *e) {
        long v = std::atol(e);
        if (v > 0 && v <= (1 << 20))
            return static_cast<uint32_t>(v);
    }
    return 1024;
}

// A live handle, or nullptr.  The handle pointer is only dereferenced once it
// is known to be live, so stale or foreign pointers give an error instead of
// a crash ([CNTN] §6.1: handles are validated and unwrapped).
static cns_cnt_notify_s *lookup(cns_cnt_notify_t h)
{
    if (!h)
        return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_live.find(h) == g_live.end() || h->magic != kMagic)
        return nullptr;
    return h;
}

// Makes the handle's device current for the call, restoring the caller's.
struct DeviceGuard {
    int prev = -1;
    bool switched = false;
    int set(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            (void)cudaGetLastError();
            return CNS_ERR_CUDA;
        }
        if (prev != dev) {
            if (cudaSetDevice(dev) != cudaSuccess) {
                (void)cudaGetLastError();
                return CNS_ERR_CUDA;
            }
            switched = true;
        }
        return CNS_SUCCESS;
    }
    ~DeviceGuard()
    {
        if (switched)
            cudaSetDevice(prev);
    }
};

// The device a stream-ordered operation on notify n runs on: the stream's own
// device.  A NULL stream (and the special handles cudaStreamLegacy and
// cudaStreamPerThread) means the default stream of the notify's device.  A
// device other than the notify's must have been given access by
// cntnotify_enable_peer.
static int launch_device(const cns_cnt_notify_s *n, cudaStream_t s, int *dev)
{
    if (s == nullptr || s == cudaStreamLegacy || s == cudaStreamPerThread) {
        *dev = n->device;
        return CNS_SUCCESS;
    }
    int d = -1;
    const cudaError_t e = cudaStreamGetDevice(s, &d);
    if (e != cudaSuccess)
        return cuda_fail(e, "cudaStreamGetDevice");
    if (d != n->device && (d < 0 || d >= 64 || ((n->peers.load(std::memory_order_acquire) >> d) & 1u) == 0))
        return CNS_ERR_NO_PEER_ACCESS;
    *dev = d;
    return CNS_SUCCESS;
}

// ---------------------------------------------------------------------------
// Record / wait kernels
// ---------------------------------------------------------------------------

template <int S>
__global__ void cnt_record_kernel(uint32_t *count, uint32_t mode, uint32_t v)
{
    if (threadIdx.x == 0)
        cnt_record_scoped<S>(count, mode, v);
}

// One thread polls the count until the predicate holds; then the optional
// clear.  On timeout the sticky status is set and the kernel returns.  With
// an `abort` word (used by the pipeline), a wait that finds it raised returns
// at once and a wait that times out raises it, so one lost signal costs one
// timeout rather than one per remaining round.  kEarlyNext (the pipeline's
// own waits) lets the stream's next kernel, launched with programmatic
// stream serialization, be scheduled while this one polls; that kernel waits
// on the device for this one to end (grid_dependency_wait).  kAfterPrev (the
// two-area pipeline, whose waits are themselves launched that way behind the
// previous consumer): before it ends, the kernel waits on the device for
// that consumer to complete, so the kernels of the stream still complete in
// stream order.
// S: kScopeGpu, or kScopeSys for a notify that other GPUs record on or wait
// on (cntnotify_enable_peer); then the line may also be another GPU's,
// reached through a peer mapping.
template <bool kEarlyNext, bool kAfterPrev, int S = kScopeGpu>
__global__ void cnt_wait_kernel(uint32_t *line, uint32_t mode, uint32_t v, uint32_t clear, uint64_t timeout_ns,
                                uint32_t *observed, uint32_t *abort, uint64_t *released_at)
{
    if (kEarlyNext)
        grid_launch_dependents();
    if (threadIdx.x == 0 && !(abort && ld_relaxed_scoped<S>(abort) != 0u)) {
        uint32_t spins = 0;
        uint64_t deadline = 0;
        for (;;) {
            // relaxed polls; the fence after the one that releases makes it an
            // acquire of the records it read from (they are release operations)
            const uint32_t c = ld_relaxed_scoped<S>(line);
            if (cnt_wait_released(c, mode, v)) {
                fence_acquire_scoped<S>();
                if (released_at)
                    *released_at = globaltimer_ns();
                if (observed)
                    *observed = c;
                if (clear)
                    atom_exch_relaxed_scoped<S>(line, 0u);   // the clear comes after the release
                break;
            }
            if ((++spins & 63u) == 0u) {
                if (abort && ld_relaxed_scoped<S>(abort) != 0u)
                    break;
                const uint64_t now = globaltimer_ns();
                if (deadline == 0)
                    deadline = now + timeout_ns;
                else if (now > deadline) {
                    atom_exch_relaxed_scoped<S>(line + 1, static_cast<uint32_t>(CNS_ERR_TIMEOUT));
                    if (abort)
                        atom_exch_relaxed_scoped<S>(abort, 1u);
                    break;
                }
            }
        }
    }
    if (kAfterPrev)
        grid_dependency_wait();
}

// Zero the count, the sticky status, the abort word and the spare word of a
// notify line.
__global__ void cnt_clear_line_kernel(uint32_t *line)
{
    if (threadIdx.x < 4)
        line[threadIdx.x] = 0u;
}

static uint64_t wait_timeout_ns(uint32_t timeout_s)
{
    const uint64_t cap = notify_timeout_cap_ns();
    if (timeout_s == 0)
        return cap;
    return std::min<uint64_t>(static_cast<uint64_t>(timeout_s) * 1000000000ull, cap);
}

static bool record_mode_ok(int32_t m)
{
    return m == CNS_REC_SET || m == CNS_REC_ADD || m == CNS_REC_BIT_OR || m == CNS_REC_BIT_AND;
}

static int enqueue_wait(cns_cnt_notify_s *n, cudaStream_t s, const cns_wait_info_t *info, uint32_t *observed,
                        uint32_t *abort = nullptr, bool early_next = false, uint64_t *released_at = nullptr)
{
    const bool sys = n->sys.load(std::memory_order_acquire) != 0;
    auto k = sys ? (early_next ? cnt_wait_kernel<true, false, kScopeSys> : cnt_wait_kernel<false, false, kScopeSys>)
                 : (early_next ? cnt_wait_kernel<true, false> : cnt_wait_kernel<false, false>);
    k<<<1, 32, 0, s>>>(n->line, static_cast<uint32_t>(info->mode), info->value, info->is_clear ? 1u : 0u,
                       wait_timeout_ns(info->timeout), observed, abort, released_at);
    CNS_CUDA(cudaGetLastError());
    return CNS_SUCCESS;
}

// ---------------------------------------------------------------------------
// Op-stream state machine.  A SET record gives a count that does not depend
// on what came before, so the stream can be cut at SETs: from a SET on, the
// trace can be computed without knowing the earlier count.  Other ops can fix
// the count too: an AND with few bits set leaves few unknown bits, an OR sets
// them, an add with a known carry keeps them known, a clearing wait whose
// test does not depend on the unknown bits releases to 0.  So where a tile's
// SETs leave a long stretch, each chunk's thread follows which bits of the
// count are known (known zeros and known ones, starting from nothing known at
// the chunk's first op) and marks the first op of its chunk after which every
// bit is known, together with that op's outcome: a "fixing" op, which then
// starts a stretch as a SET does.  The marking is exact (a bit is only called
// known when every count the earlier ops could have left gives it the same
// value), so the trace is the same as the sequential one; it only shortens
// the stretches.
//
// One persistent cooperative launch.  The stream is cut into tiles of up to
// 4096 ops; CTA b takes tiles b, b + grid, b + 2 grid, ...  Within a tile, 512
// threads each own a chunk of 8 ops:
//   F  if a stretch between SETs is long (or the tile holds no SET), every
//      thread marks its chunk's first fixing op, if any, and turns it into a
//      SET of the count it fixes (same outcome);
//   A  the thread of every chunk with a start (its first SET, or the fixing
//      op F marked) walks from it up to the tile's next start after the
//      chunk (or the tile's end, in which case it publishes the tile's end
//      count, tagged with this call's tag, for the next tile) -- one
//      contiguous stretch of ops per thread;
//   C  the last thread takes the previous tile's end count (init for tile 0),
//      waiting on the device until it is published, and replays the ops in
//      front of the tile's first start -- all of them if the tile has none,
//      in which case it publishes the tile's end count itself.
// Every op is applied exactly once, in stream order along its stretch.  A
// tile with a start publishes before it waits, so a wait lasts only as long
// as a run of tiles without one in front of it (a stream of adds alone, for
// instance, has none: it is one dependent chain).  Every CTA is resident
// (cooperative launch) and takes its tiles in increasing order, so the tile a
// CTA waits for is always held by a running CTA (or done).  The tag makes the
// link words need no initial content: a word holds (tag << 32) | count, and a
// word from an earlier call carries an earlier tag.  A replay of a CUDA graph
// that captured the call repeats the call's tag, so the thread that takes a
// word sets it to 0 (no call has tag 0): the only word a launch leaves behind
// is its last tile's, which no tile of a launch of the same size reads.  The
// wait is bounded; if it runs out (only a stalled GPU can make it), the tile's
// leading entries get count 0 and outcome CNS_OUT_INVALID.
// ---------------------------------------------------------------------------

// The link words between tiles, one to a 128-byte line: a tile's word is
// written once and polled by the next tile's CTA, and words that shared lines
// (16 to a line) made every call ~1.4 us slower (1e6 ops, an A/B on one box).
// A tile holds 16 to 4096 ops, and the kernel has at most kMaxSmCtas CTAs, so
// a call has at most min(ceil(n / 16), max(ceil(n / 4096), kMaxSmCtas)) tiles.
constexpr int kLinkStride = 16;   // uint64 words from one tile's link word to the next
constexpr int64_t kMaxSmCtas = 4096;
constexpr int64_t sm_max_tiles(int64_t n)
{
    return n <= 0 ? 0
                  : ((n + 15) / 16 < ((n + 4095) / 4096 > kMaxSmCtas ? (n + 4095) / 4096 : kMaxSmCtas)
                         ? (n + 15) / 16
                         : ((n + 4095) / 4096 > kMaxSmCtas ? (n + 4095) / 4096 : kMaxSmCtas));
}
constexpr size_t sm_scratch_bytes(int64_t n)
{
    return static_cast<size_t>(sm_max_tiles(n)) * kLinkStride * sizeof(uint64_t);
}

// An op turned into a micro-op that one short branch-free sequence applies
// (neighbouring lanes of a warp apply different kinds and modes):
//   record  x = AND mask a, y = OR value o, z = addend d: the count becomes
//           ((c & a) | o) + d.  SET v is (0, v, 0), ADD v (~0, 0, v), OR v
//           (~0, v, 0), AND v (v, 0, 0).
//   wait    x = compare mask, y = lo, z = span: released when
//           (c & mask) - lo <= span, unsigned -- every wait mode is a range of
//           (c & mask): LESS v is [0, v - 1], EQUAL v [v, v], BIGGER v
//           [v + 1, 2^32 - 1], BIGGER_OR_EQUAL v [v, 2^32 - 1], and
//           EQUAL_WITH_BITMASK v is c & v in [v, v].  An empty range (LESS 0,
//           BIGGER 2^32 - 1) is mask 0, lo 1, span 0: 0 - 1 is never <= 0.
//   w       flags: bit 8 wait, bit 12 the wait clears once released, bits
//           9-10 the outcome of anything else (CNS_OUT_RECORD or
//           CNS_OUT_INVALID, or, for a fixing op turned into a SET, the
//           op's own outcome), bit 11 SET.
// An op of no valid kind and mode is the record (~0, 0, 0) with outcome
// CNS_OUT_INVALID.
constexpr uint32_t kMicroWait = 1u << 8;
constexpr uint32_t kMicroSet = 1u << 11;
constexpr uint32_t kMicroClear = 1u << 12;

// Built with selects, not branches: the lanes of a warp stage ops of every
// kind and mode at once.
__device__ __forceinline__ uint4 sm_micro(const uint4 &op)
{
    const uint32_t kind = op.x, mode = op.y, v = op.z;
    const bool rec = kind == 0u && (mode <= 2u || mode == 4u);   // SET, ADD, BIT_OR, BIT_AND
    const bool wait = kind == 1u && mode <= 4u;
    // record: ((c & a) | o) + d
    const uint32_t a = mode == CNS_REC_SET ? 0u : (mode == CNS_REC_BIT_AND ? v : ~0u);
    const uint32_t o = (mode == CNS_REC_SET || mode == CNS_REC_BIT_OR) ? v : 0u;
    const uint32_t d = mode == CNS_REC_ADD ? v : 0u;
    // wait: the range of (c & mask) that releases it
    const bool never = (mode == CNS_WAIT_LESS && v == 0u) || (mode == CNS_WAIT_BIGGER && v == ~0u);
    const uint32_t mask = never ? 0u : (mode == CNS_WAIT_EQUAL_WITH_BITMASK ? v : ~0u);
    const uint32_t lo = never ? 1u
                        : mode == CNS_WAIT_LESS ? 0u
                        : mode == CNS_WAIT_BIGGER ? v + 1u
                                                  : v;   // EQUAL, BIGGER_OR_EQUAL, EQUAL_WITH_BITMASK
    const uint32_t span = never ? 0u
                          : mode == CNS_WAIT_LESS ? v - 1u
                          : (mode == CNS_WAIT_BIGGER || mode == CNS_WAIT_BIGGER_OR_EQUAL) ? ~0u - lo
                                                                                          : 0u;
    const uint32_t wflags = kMicroWait | (op.w != 0u ? kMicroClear : 0u);
    const uint32_t rflags = (static_cast<uint32_t>(CNS_OUT_RECORD) << 9) | (mode == CNS_REC_SET ? kMicroSet : 0u);
    return make_uint4(rec ? a : (wait ? mask : ~0u), rec ? o : (wait ? lo : 0u), rec ? d : (wait ? span : 0u),
                      rec ? rflags : (wait ? wflags : static_cast<uint32_t>(CNS_OUT_INVALID) << 9));
}

// One micro-op applied to count c; *outcome gets the op's CNS_OUT_* code.
// The chain from one count to the next is four dependent instructions: the
// AND, the subtraction, the range compare (with the clear flag folded in)
// and the final select; the record's update and the outcome are computed
// beside it.
__device__ __forceinline__ uint32_t sm_apply_micro(uint32_t c, const uint4 m, uint32_t *outcome)
{
    const bool wait = (m.w & kMicroWait) != 0u;
    const uint32_t x = c & m.x;
    const bool in_range = x - m.y <= m.z;                         // a wait's release test
    const uint32_t keep = wait ? c : (x | m.y) + m.z;              // a record's update, or the count as it is
    *outcome = wait ? (in_range ? 1u : 0u) : ((m.w >> 9) & 3u);   // a wait: RELEASED (1) or HELD (0)
    return (in_range && (m.w & kMicroClear) != 0u) ? 0u : keep;
}

// What one micro-op does to the known bits of a count: kz the bits known to
// be 0, ko those known to be 1 (a count consistent with them is any value
// that has them).  A record's AND and OR fix bits outright.  Its add keeps a
// sum bit known when the addend bit's partner in the count is known and the
// carry into that bit is: the carry into bit i rises monotonically with the
// count's low i bits, so it is known when the smallest and the largest
// consistent counts (unknown bits 0, unknown bits 1) give the same carry.  A
// wait is decided when every bit under its compare mask is known; a decided
// clearing wait that releases leaves 0, an undecided one leaves 0 or the
// count (so only the known zeros stay).  Returns whether the op's outcome is
// known, and writes it to *outcome.
__device__ __forceinline__ bool sm_known_step(uint32_t &kz, uint32_t &ko, const uint4 m, uint32_t *outcome)
{
    const bool wait = (m.w & kMicroWait) != 0u;
    const bool clears = (m.w & kMicroClear) != 0u;
    // record ((c & a) | o) + d
    const uint32_t z = (kz | ~m.x) & ~m.y;
    const uint32_t o = (ko & m.x) | m.y;
    const uint32_t cmin = (o + m.z) ^ o ^ m.z;      // carries with every unknown bit 0
    const uint32_t cmax = (~z + m.z) ^ ~z ^ m.z;    // and with every unknown bit 1
    const uint32_t known = (z | o) & ~(cmin ^ cmax);
    const uint32_t rko = (o ^ m.z ^ cmin) & known;
    // wait on the range of (c & mask)
    const bool decided = ((kz | ko) & m.x) == m.x;
    const bool in_range = (ko & m.x) - m.y <= m.z;
    if (!wait) {
        kz = known & ~rko;
        ko = rko;
        *outcome = (m.w >> 9) & 3u;
        return true;
    }
    if (clears) {
        if (decided && in_range) {
            kz = ~0u;
            ko = 0u;
        } else if (!decided) {
            ko = 0u;
        }
    }
    *outcome = in_range ? 1u : 0u;
    return decided;
}

// A tile looks for fixing ops only when this many words of its start bits in a
// row (32 ops each) hold no SET -- a stretch between SETs, or in front of the
// first, of at least kFixWords * 32 ops -- or when it holds no SET at all (its
// count would otherwise wait for the tiles before it).  Shorter stretches are
// walked sooner than the search would run.
constexpr int kFixWords = 3;

constexpr uint64_t kSmLinkTimeoutNs = 10ull * 1000000000ull;

__device__ __forceinline__ void sm_publish(uint64_t *link, uint32_t tag, uint32_t c)
{
    st_release_gpu_u64(link, (static_cast<uint64_t>(tag) << 32) | c);
}

// Returns false if the wait ran out.
__device__ __forceinline__ bool sm_take(const uint64_t *link, uint32_t tag, uint32_t *c)
{
    uint32_t spins = 0;
    uint64_t deadline = 0;
    for (;;) {
        const uint64_t v = ld_acquire_gpu_u64(link);
        if (static_cast<uint32_t>(v >> 32) == tag) {
            *c = static_cast<uint32_t>(v);
            return true;
        }
        if ((++spins & 63u) == 0u) {
            const uint64_t now = globaltimer_ns();
            if (deadline == 0)
                deadline = now + kSmLinkTimeoutNs;
            else if (now > deadline)
                return false;
        }
    }
}

// Tile shape: 512 threads x chunks of 8 ops, micro-ops in shared memory with
// a one-entry pad per chunk (conflict-free per-thread walks), and a bit per op
// telling whether it is a SET, gathered by warp ballots while staging: 32
// consecutive ops per word, byte j of word w covering chunk 4w + j.
constexpr int kFChunk = 8;
constexpr int kFThreads = 512;
constexpr int kTileOps = kFChunk * kFThreads;
constexpr int kFPad = kFChunk + 1;
constexpr size_t kFSmemBytes = static_cast<size_t>(kFThreads) * kFPad * (sizeof(uint4) + sizeof(uint2)) +
                               kTileOps / 32 * sizeof(uint32_t);

__device__ __forceinline__ int f_slot(int i) { return (i / kFChunk) * kFPad + (i % kFChunk); }

// Length classes of the stretches: floor(log2(length)) for lengths 1 .. 4096,
// longest first, and a last class for chunks without a stretch.
constexpr int kJobClasses = 14;

// Position of the tile's first SET at or after `from` (cnt if none) from the
// tile's SET bits; positions at or past cnt carry no SET bit.
__device__ __forceinline__ int f_next_set(const uint32_t *s_setm, int from, int cnt)
{
    if (from >= cnt)
        return cnt;
    int w = from >> 5;
    uint32_t bits = s_setm[w] & (~0u << (from & 31));
    while (bits == 0u && ++w < kTileOps / 32)
        bits = s_setm[w];
    return bits ? (w << 5) + __ffs(bits) - 1 : cnt;
}

// The stretch of the chunk at chunk0, if the chunk has a start: from its first
// start to the tile's next start after the chunk (or the tile's end).
__device__ __forceinline__ void f_stretch(const uint32_t *s_setm, int chunk0, int cnt, int *start, int *end)
{
    const uint32_t own = reinterpret_cast<const uint8_t *>(s_setm)[chunk0 / kFChunk];   // no bits at or past cnt
    if (own != 0u) {
        *start = chunk0 + __ffs(own) - 1;
        *end = f_next_set(s_setm, chunk0 + kFChunk, cnt);
    }
}

// Apply ops [p, end) of the tile to count c, writing their trace entries.
// The next op is loaded while the current one is applied.
__device__ __forceinline__ uint32_t f_walk(const uint4 *s_ops, uint2 *s_tr, int p, int end, uint32_t c)
{
    if (p >= end)
        return c;
    int slot = f_slot(p);
    uint4 m = s_ops[slot];
    for (;;) {
        const int next = slot + ((p & (kFChunk - 1)) == kFChunk - 1 ? 2 : 1);   // over the chunk's pad entry
        const bool more = p + 1 < end;
        const uint4 mn = more ? s_ops[next] : m;
        uint32_t o;
        c = sm_apply_micro(c, m, &o);
        s_tr[slot] = make_uint2(c, o);
        if (!more)
            return c;
        m = mn;
        slot = next;
        ++p;
    }
}

__global__ void __launch_bounds__(kFThreads, 2) sm_onepass_kernel(const uint4 *ops, int64_t n, int tile_ops,
                                                                  uint32_t init, uint2 *trace, uint64_t *link,
                                                                  uint32_t tag, uint32_t *final_count)
{
    extern __shared__ uint4 f_smem[];
    uint4 *s_ops = f_smem;
    uint2 *s_tr = reinterpret_cast<uint2 *>(f_smem + kFThreads * kFPad);
    uint32_t *s_setm = reinterpret_cast<uint32_t *>(s_tr + kFThreads * kFPad);
    __shared__ uint32_t s_job[kFThreads];   // stretch handed to thread i: (start << 16) | end
    __shared__ int s_cls[kJobClasses];       // per length class: its stretches' count
    const int64_t tiles = (n + tile_ops - 1) / tile_ops;
    const int k = threadIdx.x;
    const int lane = k & 31;
    for (int64_t t = blockIdx.x; t < tiles; t += gridDim.x) {
        const int64_t base = t * tile_ops;
        const int cnt = (n - base < tile_ops) ? static_cast<int>(n - base) : tile_ops;
        if (k < kJobClasses)
            s_cls[k] = 0;
        {   // stage: the 8 loads of a thread in flight four at a time, turned into micro-ops on the way in
            const uint4 *src = ops + base;
#pragma unroll
            for (int h = 0; h < kFChunk; h += 4) {
                uint4 v[4];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int i = k + (h + j) * kFThreads;
                    v[j] = i < cnt ? __ldg(src + i) : make_uint4(2u, 0u, 0u, 0u);   // past the end: no SET
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int i = k + (h + j) * kFThreads;
                    const uint4 m = sm_micro(v[j]);
                    if (i < cnt)
                        s_ops[f_slot(i)] = m;
                    const uint32_t sets = __ballot_sync(0xffffffffu, (m.w & kMicroSet) != 0u);
                    if (lane == 0)
                        s_setm[i >> 5] = sets;
                }
            }
        }
        __syncthreads();
        const bool last_tile = base + cnt == n;
        const int chunk0 = k * kFChunk;
        // words k .. k + kFixWords - 1 of the start bits (4 chunks each) hold no SET, or the tile
        // holds none at all
        const int words = (cnt + 32 - 1) / 32;
        bool gap = false;
        if (k < words) {
            const int upto = min(words, k + kFixWords);
            uint32_t any = 0u;
            for (int j = k; j < upto; ++j)
                any |= s_setm[j];
            gap = any == 0u && (upto - k == kFixWords || (k == 0 && upto == words));
        }
        if (__syncthreads_or(gap)) {
            // F: a stretch between SETs (or in front of the first) is long enough that the
            // fixing ops are worth finding: this chunk's first one (byte k of the start bits
            // covers chunk k) becomes a SET of the count it fixes, with the op's outcome
            const int stop = min(cnt, chunk0 + kFChunk);
            uint32_t kz = 0u, ko = 0u, fixed_at = 0u, out = 0u;
            int fix = -1;
            for (int i = chunk0; i < stop; ++i) {
                uint32_t o;
                const bool known_out = sm_known_step(kz, ko, s_ops[f_slot(i)], &o);
                if (known_out && (kz | ko) == ~0u) {
                    fix = i;
                    fixed_at = ko;
                    out = o;
                    break;
                }
            }
            reinterpret_cast<uint8_t *>(s_setm)[k] = fix >= 0 ? static_cast<uint8_t>(1u << (fix - chunk0)) : 0u;
            __syncthreads();   // every start bit in place
            if (fix >= 0)
                s_ops[f_slot(fix)] = make_uint4(0u, fixed_at, 0u, (out << 9) | kMicroSet);
        }
        int start = cnt, end = cnt;   // this chunk's stretch, if it has a start
        f_stretch(s_setm, chunk0, cnt, &start, &end);
        {   // A
            // The stretches are handed to threads longest class first (class = floor(log2(length)),
            // counted per warp; each thread then adds up the counts of the longer classes for its
            // place), so that a warp's lanes walk stretches of similar length instead of waiting for
            // one long stretch among short ones.
            const int len = end - start;   // 0: none
            const int cls = len > 0 ? kJobClasses - 2 - min(31 - __clz(len), kJobClasses - 2) : kJobClasses - 1;
            const uint32_t same = __match_any_sync(0xffffffffu, cls);
            const int leader = __ffs(same) - 1;
            int wbase = 0;
            if (lane == leader)
                wbase = atomicAdd(&s_cls[cls], __popc(same));
            wbase = __shfl_sync(0xffffffffu, wbase, leader) + __popc(same & ((1u << lane) - 1u));
            __syncthreads();   // every class's count in
            int place = wbase, jobs = 0;   // the jobs of the longer classes come first
#pragma unroll
            for (int q = 0; q < kJobClasses - 1; ++q) {
                const int n_q = s_cls[q];
                place += q < cls ? n_q : 0;
                jobs += n_q;
            }
            if (len > 0)
                s_job[place] = (static_cast<uint32_t>(start) << 16) | static_cast<uint32_t>(end);
            __syncthreads();
            if (k < jobs) {
                const int js = static_cast<int>(s_job[k] >> 16), je = static_cast<int>(s_job[k] & 0xFFFFu);
                const uint32_t c = f_walk(s_ops, s_tr, js, je, 0u);   // starts with a SET: any count will do
                if (je >= cnt) {
                    sm_publish(link + t * kLinkStride, tag, c);
                    if (last_tile)
                        *final_count = c;
                }
            }
        }
        if (k == kFThreads - 1) {   // C, on the thread handed the shortest stretch (or none)
            const int lead = f_next_set(s_setm, 0, cnt);
            uint32_t cp = init;
            if (t == 0 || sm_take(link + (t - 1) * kLinkStride, tag, &cp)) {
                if (t > 0)   // taken: tag 0 is no call's, so no later launch can take this word again
                    *reinterpret_cast<volatile uint64_t *>(link + (t - 1) * kLinkStride) = 0ull;
                cp = f_walk(s_ops, s_tr, 0, lead, cp);
            } else {
                for (int i = 0; i < lead; ++i)
                    s_tr[f_slot(i)] = make_uint2(0u, CNS_OUT_INVALID);
                cp = 0u;
            }
            if (lead >= cnt) {
                sm_publish(link + t * kLinkStride, tag, cp);
                if (last_tile)
                    *final_count = cp;
            }
        }
        __syncthreads();
        for (int i = k; i < cnt; i += kFThreads)   // every entry was written once
            trace[base + i] = s_tr[f_slot(i)];
        __syncthreads();   // the shared tile is free for the next one
    }
}

// The kernel's co-resident CTAs per device (set by sm_prepare) and the call
// tags of this process.
static int64_t g_sm_max_ctas[64];
static std::atomic<uint32_t> g_sm_tag{0};

// Shared-memory opt-in and the co-residency limit, once per device.
static int sm_prepare(int device)
{
    static std::mutex mu;
    static bool done[64];
    std::lock_guard<std::mutex> lk(mu);
    if (device < 0 || device >= 64)
        return CNS_ERR_CUDA;
    if (!done[device]) {
        CNS_CUDA(cudaFuncSetAttribute(sm_onepass_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                      static_cast<int>(kFSmemBytes)));
        int per_sm = 0;
        CNS_CUDA(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, sm_onepass_kernel, kFThreads, kFSmemBytes));
        int sms = 0;
        CNS_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device));
        if (per_sm < 1)
            return CNS_ERR_CUDA;
        g_sm_max_ctas[device] = std::min<int64_t>(static_cast<int64_t>(per_sm) * sms, kMaxSmCtas);
        done[device] = true;
    }
    return CNS_SUCCESS;
}

// One state-machine run (n > 0): one cooperative launch of at most as many
// CTAs as fit at once.  A tile holds up to 4096 ops; when the GPU holds more
// CTAs than that needs, the ops are spread evenly over all of them instead
// (tiles of ceil(n / CTAs) ops rounded up to a multiple of 8, at least 16), so
// that every SM gets the same share.  `link` needs one 128-byte line per tile
// (sm_scratch_bytes(n) bytes).
static int sm_launch(const uint4 *ops, int64_t n, uint32_t init, uint2 *trace, uint64_t *link, uint32_t *final_dev,
                     int device, cudaStream_t s)
{
    if (int rc = sm_prepare(device))
        return rc;
    const int64_t max_ctas = g_sm_max_ctas[device];
    int64_t tile_ops = (n + max_ctas - 1) / max_ctas;
    tile_ops = (tile_ops + kFChunk - 1) / kFChunk * kFChunk;
    tile_ops = std::min<int64_t>(std::max<int64_t>(tile_ops, 16), kTileOps);
    const int64_t tiles = (n + tile_ops - 1) / tile_ops;
    const int64_t grid = tiles < max_ctas ? tiles : max_ctas;
    uint32_t tag = ++g_sm_tag;
    if (tag == 0)
        tag = ++g_sm_tag;
    const uint4 *a0 = ops;
    int64_t a1 = n;
    int a2 = static_cast<int>(tile_ops);
    uint32_t a3 = init;
    uint2 *a4 = trace;
    uint64_t *a5 = link;
    uint32_t a6 = tag;
    uint32_t *a7 = final_dev;
    void *args[] = {&a0, &a1, &a2, &a3, &a4, &a5, &a6, &a7};
    CNS_CUDA(cudaLaunchCooperativeKernel(reinterpret_cast<const void *>(sm_onepass_kernel),
                                         dim3(static_cast<unsigned>(grid)), dim3(kFThreads), args, kFSmemBytes, s));
    return CNS_SUCCESS;
}

__global__ void write_word_kernel(uint32_t *w, uint32_t v) { *w = v; }

// The dependent chain of the state machine's rule on its own: one thread
// applies 16 micro-ops held in registers, over and over, with the walks' own
// sm_apply_micro (a stream without SETs is one such chain).
__global__ void sm_chain_probe_kernel(const uint4 *ops, int32_t iters, uint64_t *out)
{
    if (threadIdx.x != 0 || blockIdx.x != 0)
        return;
    uint4 m[16];
#pragma unroll
    for (int i = 0; i < 16; ++i)
        m[i] = sm_micro(ops[i]);
    uint32_t c = 0u, acc = 0u;
    const uint64_t t0 = globaltimer_ns();
    for (int32_t it = 0; it < iters; ++it) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            uint32_t o;
            c = sm_apply_micro(c, m[i], &o);
            acc += o;
        }
    }
    const uint64_t t1 = globaltimer_ns();
    out[0] = t1 - t0;
    out[1] = (static_cast<uint64_t>(acc) << 32) | c;
}

// ---------------------------------------------------------------------------
// Two-stream pipeline kernels
// ---------------------------------------------------------------------------

// The pipeline's device-side waits: thread 0 polls *word (relaxed) until
// `ok(value)`, then an acquire fence; the value that passed goes to *seen if
// given.  Returns true if the caller must skip the round: the pipeline's abort
// word is raised, or the wait ran out, in which case it records
// CNS_ERR_TIMEOUT in status_word and raises the abort.
template <class Ok>
__device__ __forceinline__ bool pipe_wait(const uint32_t *word, Ok ok, uint64_t timeout_ns, uint32_t *abort,
                                          uint32_t *status_word, uint32_t *seen = nullptr)
{
    uint32_t spins = 0;
    uint64_t deadline = 0;
    for (;;) {
        const uint32_t v = ld_relaxed_gpu(word);
        if (ok(v)) {
            fence_acquire_gpu();
            if (seen)
                *seen = v;
            return false;
        }
        if ((++spins & 63u) == 0u) {
            if (ld_relaxed_gpu(abort) != 0u)
                return true;
            const uint64_t now = globaltimer_ns();
            if (deadline == 0) {
                deadline = now + timeout_ns;
            } else if (now > deadline) {
                atom_exch_relaxed_gpu(status_word, static_cast<uint32_t>(CNS_ERR_TIMEOUT));
                atom_exch_relaxed_gpu(abort, 1u);
                return true;
            }
        }
    }
}

// Producer of one round, writing the tile area `area`.
// CTA b owns tiles b, b + grid, b + 2 grid, ...; all of its threads store
// them, then, after the block barrier, lane j of warp 0 adds 1 to `done` for
// the CTA's tile j (j < 32, then the next 32, ...).  Each of those is one
// release ADD 1 record of the counted notify; the lanes of one instruction
// reach the same word, and the memory system combines them into one L2
// operation, so a CTA with k <= 32 tiles costs the count line one operation,
// not k.  (Same-address operations are served one at a time by the L2 slice
// that homes the line, about 1.25 ns each on GB300: one record per tile from
// 4096 CTAs costs 5 us per round on that line alone.)
//   Before storing, every CTA waits on the device (if wait_ack) until
// ack >= ack_target: every consumer CTA that read this area last has
// finished.
//   kTwoAreas: rounds alternate between two areas, so this round's stores
// overlap the previous round's reads.  Its records must still come after the
// consumer-side wait has cleared the previous round's count (a record that
// landed before that clear would be wiped by it), so after storing, the CTA
// waits for the previous producer grid to complete (it is launched behind it
// with programmatic stream serialization) and then for done < tiles, which
// holds from the clear on: the previous round left exactly `tiles` on done,
// and this round's own records total `tiles`, the last of them added after
// the CTA that makes it has looked.  Only then does the CTA let the next
// producer grid be scheduled, so at most two producer grids are resident.
constexpr int kPipeProducerThreads = 256;

template <bool kTwoAreas>
__global__ void __launch_bounds__(kPipeProducerThreads, 8)
    pipeline_producer_kernel(uint32_t *area, int64_t n_tiles, int tile_words, uint32_t round, bool wait_ack,
                             uint32_t ack_target, uint32_t *done, uint32_t *ack, uint64_t timeout_ns, uint32_t *abort,
                             uint64_t *started_at)
{
    __shared__ int s_skip, s_skip_rec;
    if (threadIdx.x == 0) {
        // ack counts consumer CTAs (mod 2^32); it never runs more than one
        // round's worth past the target, so the signed difference decides
        const bool skip = wait_ack && pipe_wait(ack, [&](uint32_t a) {
            return static_cast<int32_t>(a - ack_target) >= 0;
        }, timeout_ns, abort, ack + 1);
        s_skip = skip ? 1 : 0;
        if (!kTwoAreas && started_at && blockIdx.x == 0)
            *started_at = globaltimer_ns();   // CTA 0 released: the round's recording phase begins
    }
    __syncthreads();
    if (s_skip)
        return;
    const int64_t grid = gridDim.x;
    const int64_t mine = (n_tiles - blockIdx.x + grid - 1) / grid;   // tiles of this CTA (blockIdx.x < n_tiles)
    const uint32_t q = static_cast<uint32_t>(tile_words) >> 2;      // uint4 per tile
    const uint32_t total = static_cast<uint32_t>(mine) * q;          // <= 2^30: tiles * tile_words <= 2^32
    for (uint32_t e = threadIdx.x; e < total; e += blockDim.x) {
        const uint32_t j = e / q;
        const uint32_t i = e - j * q;
        const int64_t t = blockIdx.x + static_cast<int64_t>(j) * grid;
        uint4 *d = reinterpret_cast<uint4 *>(area + t * tile_words);
        const uint32_t w = static_cast<uint32_t>(t * tile_words) + 4u * static_cast<uint32_t>(i);
        d[i] = make_uint4(w * 2654435761u + round, (w + 1u) * 2654435761u + round, (w + 2u) * 2654435761u + round,
                          (w + 3u) * 2654435761u + round);
    }
    if constexpr (kTwoAreas) {
        grid_dependency_wait();   // the previous round's producer has completed
        if (threadIdx.x == 0) {
            const uint32_t k = static_cast<uint32_t>(n_tiles);
            s_skip_rec = pipe_wait(done, [&](uint32_t c) { return c < k; }, timeout_ns, abort, done + 1) ? 1 : 0;
            if (started_at && blockIdx.x == 0)
                *started_at = globaltimer_ns();   // CTA 0 may record: the round's recording phase begins
        }
        grid_launch_dependents();
    }
    __syncthreads();   // every tile of the CTA is stored ...
    if (kTwoAreas && s_skip_rec)
        return;
    if (threadIdx.x < 32) {
        for (int64_t j0 = 0; j0 < mine; j0 += 32)
            if (j0 + threadIdx.x < mine)
                cnt_record_device(done, CNS_REC_ADD, 1u);   // ... before any of them is counted (release)
    }
}

// Consumer of one round: sums the tile area mod 2^32 into *checksum; each
// CTA, once its reads are done, records ADD 1 on `ack` (release), and the
// producer that next writes this area waits for all of them.  One record per
// CTA, no returning atomic: nobody has to find out which CTA finished last.
// The record comes before the checksum's atomic add, so that its release
// waits for the reads only.
// It is launched with programmatic stream serialization behind the wait, so
// its CTAs may be scheduled while the wait still polls: they first wait on the
// device until the wait kernel has ended.  Each thread issues four
// independent loads at a time.
//   kTwoAreas: the next round's wait is launched the same way behind this
// kernel; once the CTA is past its own dependency wait (the wait before it,
// and its clear, are complete), it lets that wait be scheduled.
//   kInKernelWait: there is no wait kernel; the consumer itself takes the
// counted-notify wait (BIGGER_OR_EQUAL tiles, isClear) at its start.  CTA 0
// waits on `done`, clears it, and publishes the round on a `go` word of its
// own line (release); the other CTAs wait for that word.  (They may not all
// poll `done`: once CTA 0 has cleared it, a CTA that had not yet looked
// would wait for ever.)  CTA 0 first waits for the previous round's `go`,
// which its CTA 0 published after clearing, so the count it then sees holds
// this round's records only.  With two areas the grid is launched behind the
// previous consumer with programmatic stream serialization and takes its wait
// while that one still reads; only then does it wait for the previous grid to
// complete (so at most two consumer grids are resident) and let the next be
// scheduled.
constexpr int kPipeConsumerThreads = 256;

struct PipeConsumerWait {   // kInKernelWait only
    uint32_t *done;         // the notify line: [0] count, [1] status
    uint32_t *go;           // round + 1 once round's wait has released and cleared
    uint32_t *abort;
    uint32_t *observed;     // optional: count seen at release
    uint64_t *released_at;  // optional: device time of the release
    uint64_t timeout_ns;
    uint32_t tiles;
    uint32_t round;
};

template <bool kTwoAreas, bool kInKernelWait>
__global__ void __launch_bounds__(kPipeConsumerThreads, 8)
    pipeline_consumer_kernel(const uint32_t *tiles, int64_t n_words, uint32_t *checksum, uint32_t *ack,
                             PipeConsumerWait w)
{
    if constexpr (kInKernelWait) {
        if (threadIdx.x == 0) {
            if (blockIdx.x == 0) {
                uint32_t seen = 0;
                const bool stop =
                    pipe_wait(w.go, [&](uint32_t g) { return static_cast<int32_t>(g - w.round) >= 0; }, w.timeout_ns,
                              w.abort, w.done + 1) ||
                    pipe_wait(w.done, [&](uint32_t c) { return c >= w.tiles; }, w.timeout_ns, w.abort, w.done + 1,
                              &seen);
                if (!stop) {
                    if (w.released_at)
                        *w.released_at = globaltimer_ns();
                    if (w.observed)
                        *w.observed = seen;
                    atom_exch_relaxed_gpu(w.done, 0u);   // the clear comes after the release ...
                    st_release_gpu(w.go, w.round + 1u);  // ... and before the round is published
                }
            } else {
                pipe_wait(w.go, [&](uint32_t g) { return static_cast<int32_t>(g - (w.round + 1u)) >= 0; },
                          w.timeout_ns, w.abort, w.done + 1);
            }
        }
        __syncthreads();
    }
    grid_dependency_wait();
    if (kTwoAreas)
        grid_launch_dependents();
    const uint4 *t4 = reinterpret_cast<const uint4 *>(tiles);
    uint32_t s = 0;
    const int64_t n4 = n_words >> 2;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
#pragma unroll 1
    for (; i + 3 * stride < n4; i += 4 * stride) {
        const uint4 a = t4[i], b = t4[i + stride], c = t4[i + 2 * stride], d = t4[i + 3 * stride];
        s += (a.x + a.y + a.z + a.w) + (b.x + b.y + b.z + b.w) + (c.x + c.y + c.z + c.w) + (d.x + d.y + d.z + d.w);
    }
#pragma unroll 1
    for (; i < n4; i += stride) {
        const uint4 v = t4[i];
        s += v.x + v.y + v.z + v.w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        s += __shfl_xor_sync(0xffffffffu, s, o);
    // one add per CTA, not per warp: same-address atomics serialise in L2
    __shared__ uint32_t warp_sum[32];
    if ((threadIdx.x & 31u) == 0u)
        warp_sum[threadIdx.x >> 5] = s;
    __syncthreads();   // every read of this CTA is done ...
    if (threadIdx.x < 32) {
        uint32_t w = (threadIdx.x < (blockDim.x >> 5)) ? warp_sum[threadIdx.x] : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            w += __shfl_xor_sync(0xffffffffu, w, o);
        if (threadIdx.x == 0) {
            cnt_record_device(ack, CNS_REC_ADD, 1u);   // ... before the CTA counts itself done (release)
            atomicAdd(checksum, w);
        }
    }
}

}  // namespace cns

using namespace cns;

// ---------------------------------------------------------------------------
// Handle lifecycle
// ---------------------------------------------------------------------------

// Load every kernel that the notify calls and the pipeline launch, on the
// current device.  Under CUDA's lazy loading (the default) a kernel's code is
// loaded at its first launch, and that load can wait for kernels already
// running: a record launched for the first time on one stream while a wait
// kernel polls on another is then held back until the wait times out (a
// test measured exactly that: a 1 s timeout on the first wait of a process,
// 49 us for the same calls once both kernels had been loaded).  Getting a
// kernel's attributes loads it; done once per device, when its notify pool is
// made.
static int preload_notify_kernels()
{
    const void *kernels[] = {
        reinterpret_cast<const void *>(cnt_record_kernel<kScopeGpu>),
        reinterpret_cast<const void *>(cnt_record_kernel<kScopeSys>),
        reinterpret_cast<const void *>(cnt_wait_kernel<false, false, kScopeSys>),
        reinterpret_cast<const void *>(cnt_wait_kernel<true, false, kScopeSys>),
        reinterpret_cast<const void *>(cnt_wait_kernel<false, false>),
        reinterpret_cast<const void *>(cnt_wait_kernel<true, false>),
        reinterpret_cast<const void *>(cnt_wait_kernel<true, true>),
        reinterpret_cast<const void *>(cnt_clear_line_kernel),
        reinterpret_cast<const void *>(write_word_kernel),
        reinterpret_cast<const void *>(sm_onepass_kernel),
        reinterpret_cast<const void *>(pipeline_producer_kernel<true>),
        reinterpret_cast<const void *>(pipeline_producer_kernel<false>),
        reinterpret_cast<const void *>(pipeline_consumer_kernel<true, true>),
        reinterpret_cast<const void *>(pipeline_consumer_kernel<false, true>),
        reinterpret_cast<const void *>(pipeline_consumer_kernel<true, false>),
        reinterpret_cast<const void *>(pipeline_consumer_kernel<false, false>),
    };
    for (const void *k : kernels) {
        cudaFuncAttributes a;
        CNS_CUDA(cudaFuncGetAttributes(&a, k));
    }
    return CNS_SUCCESS;
}

extern "C" int cntnotify_create(cns_cnt_notify_t *out, uint64_t flag)
{
    if (!out)
        return CNS_ERR_NULL_PTR;
    if (flag != 0)
        return CNS_ERR_INVALID_VALUE;   // [CNTN] §4.1: flag is reserved and must be 0
    DeviceInfo dev;
    if (int rc = current_device(&dev))
        return rc;
    std::lock_guard<std::mutex> lk(g_mu);
    Pool &pool = g_pools[dev.device];
    if (!pool.base) {
        if (int rc = preload_notify_kernels())
            return rc;
        const uint32_t cap = pool_cap();
        void *p = nullptr;
        CNS_CUDA(cudaMalloc(&p, static_cast<size_t>(cap) * kWordsPerSlot * 4));
        CNS_CUDA(cudaMemset(p, 0, static_cast<size_t>(cap) * kWordsPerSlot * 4));
        pool.base = static_cast<uint32_t *>(p);
        pool.cap = cap;
        pool.free_slots.reserve(cap);
        for (uint32_t i = cap; i-- > 0;)
            pool.free_slots.push_back(i);
    }
    if (pool.free_slots.empty()) {
        CNS_LOG(1, "too many counted notifies (pool of %u)", pool.cap);
        return CNS_ERR_RESOURCE;
    }
    const uint32_t slot = pool.free_slots.back();
    uint32_t *line = pool.base + static_cast<size_t>(slot) * kWordsPerSlot;
    // a fresh notify starts at count 0 with a clear status
    CNS_CUDA(cudaMemset(line, 0, kWordsPerSlot * 4));
    pool.free_slots.pop_back();
    auto *h = new cns_cnt_notify_s;
    h->magic = kMagic;
    h->device = dev.device;
    h->slot = slot;
    h->line = line;
    g_live.insert(h);
    *out = h;
    return CNS_SUCCESS;
}

extern "C" int cntnotify_destroy(cns_cnt_notify_t h)
{
    std::lock_guard<std::mutex> lk(g_mu);
    auto it = h ? g_live.find(h) : g_live.end();
    if (it == g_live.end())
        return CNS_ERR_INVALID_HANDLE;
    g_live.erase(it);
    g_pools[h->device].free_slots.push_back(h->slot);
    h->magic = 0;
    delete h;
    return CNS_SUCCESS;
}

extern "C" int cntnotify_get_id(cns_cnt_notify_t h, uint32_t *id)
{
    cns_cnt_notify_s *n = lookup(h);
    if (!n)
        return CNS_ERR_INVALID_HANDLE;
    if (!id)
        return CNS_ERR_NULL_PTR;
    *id = (static_cast<uint32_t>(n->device) << 24) | n->slot;
    return CNS_SUCCESS;
}

extern "C" int cntnotify_get_device_ptr(cns_cnt_notify_t h, uint32_t **count_dev)
{
    cns_cnt_notify_s *n = lookup(h);
    if (!n)
        return CNS_ERR_INVALID_HANDLE;
    if (!count_dev)
        return CNS_ERR_NULL_PTR;
    *count_dev = n->line;
    return CNS_SUCCESS;
}

// ---------------------------------------------------------------------------
// Stream-ordered operations
// ---------------------------------------------------------------------------

// One record (mode, v) on stream s, launched on the stream's device, at
// system scope once the notify has peers.
static int enqueue_record(cns_cnt_notify_s *n, cudaStream_t s, uint32_t mode, uint32_t v)
{
    int dev = -1;
    if (int rc = launch_device(n, s, &dev))
        return rc;
    DeviceGuard g;
    if (int rc = g.set(dev))
        return rc;
    if (n->sys.load(std::memory_order_acquire))
        cnt_record_kernel<kScopeSys><<<1, 32, 0, s>>>(n->line, mode, v);
    else
        cnt_record_kernel<kScopeGpu><<<1, 32, 0, s>>>(n->line, mode, v);
    CNS_CUDA(cudaGetLastError());
    return CNS_SUCCESS;
}

extern "C" int cntnotify_enable_peer(cns_cnt_notify_t h, int peer_device)
{
    cns_cnt_notify_s *n = lookup(h);
    if (!n)
        return CNS_ERR_INVALID_HANDLE;
    TraceRange tr("cntnotify_enable_peer", n->slot);
    if (peer_device < 0 || peer_device >= 64)
        return CNS_ERR_INVALID_VALUE;
    int count = 0;
    CNS_CUDA(cudaGetDeviceCount(&count));
    if (peer_device >= count)
        return CNS_ERR_INVALID_VALUE;
    if (peer_device != n->device) {
        int can = 0;
        CNS_CUDA(cudaDeviceCanAccessPeer(&can, peer_device, n->device));
        if (!can)
            return CNS_ERR_NO_PEER_ACCESS;
        DeviceGuard g;
        if (int rc = g.set(peer_device))
            return rc;
        DeviceInfo dev;   // the peer runs the library's kernels too: same architecture check
        if (int rc = current_device(&dev))
            return rc;
        const cudaError_t e = cudaDeviceEnablePeerAccess(n->device, 0);
        if (e == cudaErrorPeerAccessAlreadyEnabled)
            (void)cudaGetLastError();
        else if (e != cudaSuccess)
            return cuda_fail(e, "cudaDeviceEnablePeerAccess");
        // the peer's streams will launch the notify kernels: load them there now
        // (see preload_notify_kernels)
        if (int rc = preload_notify_kernels())
            return rc;
    }
    n->sys.store(1, std::memory_order_release);
    n->peers.fetch_or(1ull << peer_device, std::memory_order_acq_rel);
    return CNS_SUCCESS;
}

extern "C" int cntnotify_record(cns_cnt_notify_t h, cns_stream_t stream, const cns_record_info_t *info)
{
    cns_cnt_notify_s *n = lookup(h);
    if (!n)
        return CNS_ERR_INVALID_HANDLE;
    TraceRange tr("cntnotify_record", n->slot);
    if (!info)
        return CNS_ERR_NULL_PTR;
    if (!record_mode_ok(info->mode))
        return CNS_ERR_INVALID_VALUE;
    return enqueue_record(n, to_stream(stream), static_cast<uint32_t>(info->mode), info->value);
}

extern "C" int cntnotify_wait_with_timeout(cns_cnt_notify_t h, cns_stream_t stream, const cns_wait_info_t *info)
{
    cns_cnt_notify_s *n = lookup(h);
    if (!n)
        return CNS_ERR_INVALID_HANDLE;
    TraceRange tr("cntnotify_wait_with_timeout", n->slot);
    if (!info)
        return CNS_ERR_NULL_PTR;
    if (info->mode < CNS_WAIT_LESS || info->mode > CNS_WAIT_EQUAL_WITH_BITMASK)
        return CNS_ERR_INVALID_VALUE;
    int dev = -1;
    if (int rc = launch_device(n, to_stream(stream), &dev))
        return rc;
    DeviceGuard g;
    if (int rc = g.set(dev))
        return rc;
    return enqueue_wait(n, to_stream(stream), info, nullptr);
}

extern "C" int cntnotify_reset(cns_cnt_notify_t h, cns_stream_t stream)
{
    cns_cnt_notify_s *n = lookup(h);
    if (!n)
        return CNS_ERR_INVALID_HANDLE;
    TraceRange tr("cntnotify_reset", n->slot);
    return enqueue_record(n, to_stream(stream), CNS_REC_SET, 0u);
}

extern "C" int cntnotify_query_status(cns_cnt_notify_t h, int32_t *status, uint32_t *count)
{
    cns_cnt_notify_s *n = lookup(h);
    if (!n)
        return CNS_ERR_INVALID_HANDLE;
    if (!status)
        return CNS_ERR_NULL_PTR;
    DeviceGuard g;
    if (int rc = g.set(n->device))
        return rc;
    // a private non-blocking stream: reads the words as they are now, without
    // waiting for work on other streams
    cudaStream_t s;
    CNS_CUDA(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
    uint32_t w[2] = {0, 0};
    cudaError_t e = cudaMemcpyAsync(w, n->line, sizeof(w), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess)
        e = cudaStreamSynchronize(s);
    cudaStreamDestroy(s);
    if (e != cudaSuccess)
        return cuda_fail(e, "cntnotify_query_status");
    *status = static_cast<int32_t>(w[1]);
    if (count)
        *count = w[0];
    return CNS_SUCCESS;
}

// ---------------------------------------------------------------------------
// State machine
// ---------------------------------------------------------------------------

extern "C" size_t cns_statemachine_scratch_bytes(int64_t n)
{
    return sm_scratch_bytes(n);
}

extern "C" int cns_statemachine_run(const uint32_t *ops_dev, int64_t n, uint32_t init, uint32_t *trace_dev,
                                    uint32_t *final_dev, void *scratch_dev, size_t scratch_bytes,
                                    cns_stream_t stream)
{
    TraceRange tr("cns_statemachine_run");
    if (n < 0)
        return CNS_ERR_INVALID_VALUE;
    if (!final_dev)
        return CNS_ERR_NULL_PTR;
    if (n > 0 && (!ops_dev || !trace_dev || !scratch_dev))
        return CNS_ERR_NULL_PTR;
    if ((reinterpret_cast<uintptr_t>(ops_dev) & 15) || (reinterpret_cast<uintptr_t>(trace_dev) & 7) ||
        (reinterpret_cast<uintptr_t>(scratch_dev) & 7))
        return CNS_ERR_INVALID_VALUE;
    if (scratch_bytes < cns_statemachine_scratch_bytes(n))
        return CNS_ERR_INVALID_VALUE;
    DeviceInfo dev;
    if (int rc = current_device(&dev))
        return rc;
    cudaStream_t s = to_stream(stream);
    if (n == 0) {
        write_word_kernel<<<1, 1, 0, s>>>(final_dev, init);
        CNS_CUDA(cudaGetLastError());
        return CNS_SUCCESS;
    }
    return sm_launch(reinterpret_cast<const uint4 *>(ops_dev), n, init, reinterpret_cast<uint2 *>(trace_dev),
                     static_cast<uint64_t *>(scratch_dev), final_dev, dev.device, s);
}

// ---------------------------------------------------------------------------
// State machine for callers that cannot allocate device memory
// ---------------------------------------------------------------------------

// The chunk summaries of cns_statemachine_run_noalloc live in this fixed
// 1 MiB array, part of the library's own device image: every GPU that loads
// the library holds it until the process exits.  On the host the name is
// only a stand-in for the symbol, not a device address; the address comes
// from cudaGetSymbolAddress, looked up once per device on first use, and
// again after a device reset (cudaDeviceReset destroys the context; the next
// one loads the library's device image anew, and the array may move).
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
static_assert(sm_scratch_bytes(CNS_STATEMACHINE_NOALLOC_MAX_OPS) <= kNoAllocScratchBytes,
              "the op limit must fit the scratch array");
static __device__ __align__(256) uint2 g_sm_noalloc_scratch[kNoAllocScratchBytes / sizeof(uint2)];

struct NoAllocScratch {
    uint2 *addr = nullptr;          // device address of the array in the context below
    unsigned long long ctx_id = 0;  // unique id of that context (0: unknown)
};
static std::mutex g_noalloc_mu;
static NoAllocScratch g_noalloc_scratch[64];   // per device

// Unique id of the calling thread's current context (the driver's cuCtxGetId,
// reached through the runtime without linking the driver library): ids are
// never reused within a process, so a context made after a device reset
// gets a new one.  False when there is no current context or the driver
// cannot tell.
static bool current_context_id(unsigned long long *id)
{
    using GetCurrentFn = CUresult (*)(CUcontext *);
    using GetIdFn = CUresult (*)(CUcontext, unsigned long long *);
    static GetCurrentFn get_current = nullptr;
    static GetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<GetCurrentFn>(f);
        f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<GetIdFn>(f);
        (void)cudaGetLastError();
    });
    CUcontext c = nullptr;
    if (!get_current || !get_id || get_current(&c) != CUDA_SUCCESS || !c)
        return false;
    return get_id(c, id) == CUDA_SUCCESS;
}

extern "C" int cns_statemachine_run_noalloc(const uint32_t *ops_dev, int64_t n, uint32_t init, uint32_t *trace_dev,
                                            uint32_t *final_dev, cns_stream_t stream)
{
    TraceRange tr("cns_statemachine_run_noalloc");
    if (n < 0 || n > CNS_STATEMACHINE_NOALLOC_MAX_OPS)
        return CNS_ERR_INVALID_VALUE;
    if (!final_dev)
        return CNS_ERR_NULL_PTR;
    if (n > 0 && (!ops_dev || !trace_dev))
        return CNS_ERR_NULL_PTR;
    if ((reinterpret_cast<uintptr_t>(ops_dev) & 15) || (reinterpret_cast<uintptr_t>(trace_dev) & 7))
        return CNS_ERR_INVALID_VALUE;
    DeviceInfo dev;
    if (int rc = current_device(&dev))
        return rc;
    uint2 *summ = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_noalloc_mu);
        if (dev.device < 0 || dev.device >= 64)
            return CNS_ERR_CUDA;
        NoAllocScratch &cache = g_noalloc_scratch[dev.device];
        unsigned long long ctx = 0;
        const bool known = current_context_id(&ctx);
        if (!cache.addr || !known || cache.ctx_id != ctx) {
            // first call on this device, or its context changed (a device
            // reset): look the array up in the current context
            void *p = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&p, g_sm_noalloc_scratch);
            if (e != cudaSuccess || !p) {
                (void)cudaGetLastError();
                cache = NoAllocScratch{};
                return cuda_fail(e, "cudaGetSymbolAddress(state-machine scratch)");
            }
            // the lookup made the context current if nothing had yet
            unsigned long long now = 0;
            cache.addr = static_cast<uint2 *>(p);
            cache.ctx_id = current_context_id(&now) ? now : 0;
        }
        summ = cache.addr;
    }
    cudaStream_t s = to_stream(stream);
    if (n == 0) {
        write_word_kernel<<<1, 1, 0, s>>>(final_dev, init);
        CNS_CUDA(cudaGetLastError());
        return CNS_SUCCESS;
    }
    // Whatever an earlier call left in the array never matters: the link
    // words carry the tag of their call.
    return sm_launch(reinterpret_cast<const uint4 *>(ops_dev), n, init, reinterpret_cast<uint2 *>(trace_dev),
                     reinterpret_cast<uint64_t *>(summ), final_dev, dev.device, s);
}

// ---------------------------------------------------------------------------
// Two-stream pipeline
// ---------------------------------------------------------------------------

extern "C" int cns_pipeline_run(cns_pipeline_t *cfg)
{
    TraceRange tr("cns_pipeline_run");
    if (!cfg)
        return CNS_ERR_NULL_PTR;
    cns_cnt_notify_s *done = lookup(cfg->done);
    cns_cnt_notify_s *ack = lookup(cfg->ack);
    if (!done || !ack || done == ack)
        return CNS_ERR_INVALID_HANDLE;
    if (!cfg->tiles_dev || !cfg->checksums_dev)
        return CNS_ERR_NULL_PTR;
    if (cfg->tiles < 1 || cfg->rounds < 0 || cfg->tile_words < 4 || cfg->tile_words > 8192 ||
        cfg->tile_words % 4 != 0 || cfg->producer_ctas < 0 || cfg->tiles > (int64_t(1) << 32) / cfg->tile_words ||
        cfg->areas < 0 || cfg->areas > 2 || cfg->consumer_wait < CNS_PIPE_WAIT_STREAM ||
        cfg->consumer_wait > CNS_PIPE_WAIT_IN_KERNEL)
        return CNS_ERR_INVALID_VALUE;
    if (reinterpret_cast<uintptr_t>(cfg->tiles_dev) & 15)
        return CNS_ERR_INVALID_VALUE;
    if (done->device != ack->device)
        return CNS_ERR_INVALID_VALUE;
    DeviceInfo dev;
    if (int rc = current_device(&dev))
        return rc;
    if (dev.device != done->device)
        return CNS_ERR_INVALID_VALUE;
    cudaStream_t sp = to_stream(cfg->producer_stream), sc = to_stream(cfg->consumer_stream);
    // Residency.  Producer CTAs wait on the device for the consumer's release
    // (ack), and the consumer's CTAs, scheduled early behind the stream wait,
    // wait on the device for that wait to end; neither group may keep the
    // other from being placed.  One area: the producer grid holds at most half
    // of the GPU's thread slots, the consumer grid a quarter.  Two areas: a
    // grid is scheduled early only once every CTA of the grid before it in its
    // stream is past its own dependency wait, and every kernel of the pipeline
    // waits for its predecessor before it ends, so at most two producer grids
    // (an eighth each), two consumer grids (a quarter each) and one wait
    // kernel are resident.  All CTAs run at <= 32 registers a thread (launch
    // bounds), so registers run in step with thread slots.  A CTA (256
    // threads) that found no SM with room would need every SM to have more
    // than (slots - 256) threads in use, i.e. more than 7/8 of the GPU, while
    // everything here holds at most 3/4 plus two one-warp wait kernels.  With
    // the wait inside the consumer there are no wait kernels, and a consumer
    // grid is scheduled early only once every CTA of the one before it is past
    // its dependency wait, so the same two consumer grids at most.  (Work
    // of other streams running at the same time can still starve a round; the
    // bounded waits then end it with CNS_ERR_TIMEOUT.)
    const bool two = cfg->areas == 2;
    const int per_sm = dev.max_threads_per_sm > 0 ? dev.max_threads_per_sm : 2048;
    const int pshare = two ? 8 : 2;   // a producer grid holds at most 1/pshare of the slots
    const int64_t pcap = static_cast<int64_t>(dev.sm_count) * std::max(1, per_sm / pshare / kPipeProducerThreads);
    const int64_t pwant = cfg->producer_ctas ? cfg->producer_ctas : cfg->tiles;
    const int pgrid = static_cast<int>(std::max<int64_t>(1, std::min(std::min(pwant, pcap), cfg->tiles)));
    const int64_t n_words = cfg->tiles * cfg->tile_words;
    const int64_t ccap = static_cast<int64_t>(dev.sm_count) * std::max(1, per_sm / 4 / kPipeConsumerThreads);
    const int cgrid = static_cast<int>(
        std::max<int64_t>(1, std::min<int64_t>(ccap, (n_words / 4 + kPipeConsumerThreads - 1) / kPipeConsumerThreads)));
    cudaLaunchAttribute early[1];
    early[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    early[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t ccfg = {};
    ccfg.gridDim = dim3(cgrid);
    ccfg.blockDim = dim3(kPipeConsumerThreads);
    ccfg.stream = sc;
    ccfg.attrs = early;
    ccfg.numAttrs = 1;
    cudaLaunchConfig_t wcfg = {};   // two areas: each wait behind the last consumer, scheduled early
    wcfg.gridDim = dim3(1);
    wcfg.blockDim = dim3(32);
    wcfg.stream = sc;
    wcfg.attrs = early;
    wcfg.numAttrs = 1;
    cudaLaunchConfig_t pcfg = {};   // two areas: each producer behind the last, scheduled early
    pcfg.gridDim = dim3(pgrid);
    pcfg.blockDim = dim3(kPipeProducerThreads);
    pcfg.stream = sp;
    pcfg.attrs = early;
    pcfg.numAttrs = 1;
    cfg->consumer_ctas = cgrid;   // ack grows by this much per round

    std::vector<cudaEvent_t> ev;
    auto cleanup = [&] {
        for (cudaEvent_t e : ev)
            cudaEventDestroy(e);
    };
    cudaEvent_t join;
    CNS_CUDA(cudaEventCreateWithFlags(&join, cudaEventDisableTiming));
    ev.push_back(join);
    // Timing (sync=1): two events around the whole run, and per round two
    // device timestamps -- CTA 0 of the producer passing its release, the
    // stream wait releasing -- whose differences sum to producer_ms.  (An
    // event pair per round would sit between the producer launches and slow
    // the round trip it measures.)
    const bool timed = cfg->sync != 0;
    const int64_t n_ev = timed ? 2 : 0;
    for (int64_t i = 0; i < n_ev; ++i) {
        cudaEvent_t e;
        if (cudaEventCreate(&e) != cudaSuccess) {
            cleanup();
            return CNS_ERR_CUDA;
        }
        ev.push_back(e);
    }
    auto T = [&](int64_t i) { return ev[1 + i]; };   // timing events
    int rc = CNS_SUCCESS;
    auto check = [&](cudaError_t e, const char *what) {
        if (e != cudaSuccess && rc == CNS_SUCCESS)
            rc = cuda_fail(e, what);
        return e == cudaSuccess;
    };

    // start state: both counts and statuses 0, checksums 0, then let the
    // consumer stream follow.  Word 2 of `done` is the pipeline's abort word.
    uint32_t *abort = done->line + 2;
    cnt_clear_line_kernel<<<1, 32, 0, sp>>>(done->line);
    cnt_clear_line_kernel<<<1, 32, 0, sp>>>(ack->line);
    check(cudaMemsetAsync(cfg->checksums_dev, 0, cfg->rounds * sizeof(uint32_t), sp), "memset checksums");
    if (cfg->released_dev)
        check(cudaMemsetAsync(cfg->released_dev, 0, cfg->rounds * sizeof(uint32_t), sp), "memset released");
    uint64_t *stamps = nullptr;   // [2][rounds]: producer started, wait released
    if (timed && cfg->rounds > 0) {
        if (check(cudaMallocAsync(reinterpret_cast<void **>(&stamps), 2 * cfg->rounds * sizeof(uint64_t), sp),
                  "stamp buffer"))
            check(cudaMemsetAsync(stamps, 0, 2 * cfg->rounds * sizeof(uint64_t), sp), "memset stamps");
    }
    const bool in_kernel = cfg->consumer_wait == CNS_PIPE_WAIT_IN_KERNEL;
    uint32_t *go = nullptr;   // in-kernel waits: the last round released, on a line of its own
    if (in_kernel && cfg->rounds > 0) {
        if (check(cudaMallocAsync(reinterpret_cast<void **>(&go), 128, sp), "go word"))
            check(cudaMemsetAsync(go, 0, 128, sp), "memset go word");
    }
    check(cudaEventRecord(join, sp), "event");
    check(cudaStreamWaitEvent(sc, join, 0), "stream wait");
    if (timed)
        check(cudaEventRecord(T(0), sp), "event");

    cns_wait_info_t w_done = {CNS_WAIT_BIGGER_OR_EQUAL, static_cast<uint32_t>(cfg->tiles), cfg->timeout_s, 1, {0, 0, 0}};
    const uint64_t ack_timeout = wait_timeout_ns(cfg->timeout_s);
    for (int64_t r = 0; r < cfg->rounds && rc == CNS_SUCCESS; ++r) {
        // Submission order is a valid serial schedule: every wait (the
        // producer's device-side wait on ack, the stream wait on done) comes
        // after the work that releases it.  CUDA may feed both streams through
        // one hardware queue in submission order, and a wait ahead of its
        // record would then hold that record back until it timed out.
        const uint32_t r32 = static_cast<uint32_t>(r);
        uint32_t *area = cfg->tiles_dev + (two ? (r & 1) * n_words : 0);
        uint64_t *started = stamps ? stamps + r : nullptr;
        if (two) {
            // the area was last read in round r - 2
            check(cudaLaunchKernelEx(&pcfg, pipeline_producer_kernel<true>, area, cfg->tiles, cfg->tile_words, r32,
                                     r >= 2, (r32 - 1u) * static_cast<uint32_t>(cgrid), done->line, ack->line,
                                     ack_timeout, abort, started),
                  "producer launch");
        } else {
            pipeline_producer_kernel<false><<<pgrid, kPipeProducerThreads, 0, sp>>>(
                area, cfg->tiles, cfg->tile_words, r32, r >= 1, r32 * static_cast<uint32_t>(cgrid), done->line,
                ack->line, ack_timeout, abort, started);
            check(cudaGetLastError(), "producer launch");
        }
        uint32_t *observed = cfg->released_dev ? cfg->released_dev + r : nullptr;
        uint64_t *released = stamps ? stamps + cfg->rounds + r : nullptr;
        if (in_kernel) {
            const PipeConsumerWait cw = {done->line, go,    abort,           observed, released,
                                         ack_timeout, static_cast<uint32_t>(cfg->tiles), r32};
            check(cudaLaunchKernelEx(&ccfg, two ? pipeline_consumer_kernel<true, true>
                                                : pipeline_consumer_kernel<false, true>,
                                     static_cast<const uint32_t *>(area), n_words, cfg->checksums_dev + r, ack->line,
                                     cw),
                  "consumer launch");
        } else if (two) {
            check(cudaLaunchKernelEx(&wcfg, cnt_wait_kernel<true, true>, done->line,
                                     static_cast<uint32_t>(w_done.mode), w_done.value, 1u,
                                     wait_timeout_ns(w_done.timeout), observed, abort, released),
                  "wait launch");
            check(cudaLaunchKernelEx(&ccfg, pipeline_consumer_kernel<true, false>,
                                     static_cast<const uint32_t *>(area), n_words, cfg->checksums_dev + r, ack->line,
                                     PipeConsumerWait{}),
                  "consumer launch");
        } else {
            if (int e = enqueue_wait(done, sc, &w_done, observed, abort, true, released))
                rc = e;
            check(cudaLaunchKernelEx(&ccfg, pipeline_consumer_kernel<false, false>,
                                     static_cast<const uint32_t *>(area), n_words, cfg->checksums_dev + r, ack->line,
                                     PipeConsumerWait{}),
                  "consumer launch");
        }
    }
    check(cudaEventRecord(join, sc), "event");
    check(cudaStreamWaitEvent(sp, join, 0), "stream wait");
    if (timed)
        check(cudaEventRecord(T(1), sp), "event");
    if (go)
        check(cudaFreeAsync(go, sp), "free go word");
    std::vector<uint64_t> host_stamps;
    if (stamps) {
        host_stamps.resize(2 * cfg->rounds);
        check(cudaMemcpyAsync(host_stamps.data(), stamps, 2 * cfg->rounds * sizeof(uint64_t), cudaMemcpyDeviceToHost,
                              sp),
              "read stamps");
        check(cudaFreeAsync(stamps, sp), "free stamps");
    }
    if (rc != CNS_SUCCESS || !timed) {
        cleanup();
        return rc;
    }
    if (!check(cudaStreamSynchronize(sp), "sync")) {
        cleanup();
        return rc;
    }
    float total = 0.f;
    check(cudaEventElapsedTime(&total, T(0), T(1)), "elapsed");
    cleanup();
    double prod_ns = 0.0;
    for (int64_t r = 0; r < cfg->rounds; ++r) {
        const uint64_t a = host_stamps[r], b = host_stamps[cfg->rounds + r];
        if (a && b > a)
            prod_ns += static_cast<double>(b - a);
    }
    const float prod = static_cast<float>(prod_ns * 1e-6);
    cfg->elapsed_ms = total;
    cfg->producer_ms = prod;
    int32_t st_done = 0, st_ack = 0;
    if (int e = cntnotify_query_status(cfg->done, &st_done, nullptr))
        return e;
    if (int e = cntnotify_query_status(cfg->ack, &st_ack, nullptr))
        return e;
    cfg->device_status = (st_done || st_ack) ? CNS_ERR_TIMEOUT : 0;
    return rc != CNS_SUCCESS ? rc : (cfg->device_status ? CNS_ERR_TIMEOUT : CNS_SUCCESS);
}

extern "C" int cns_probe_op_chain(const uint32_t *ops_dev, int32_t iters, uint64_t *out_dev, cns_stream_t stream)
{
    if (!ops_dev || !out_dev)
        return CNS_ERR_NULL_PTR;
    if (iters < 1 || (reinterpret_cast<uintptr_t>(ops_dev) & 15) || (reinterpret_cast<uintptr_t>(out_dev) & 7))
        return CNS_ERR_INVALID_VALUE;
    DeviceInfo dev;
    if (int rc = current_device(&dev))
        return rc;
    sm_chain_probe_kernel<<<1, 32, 0, to_stream(stream)>>>(reinterpret_cast<const uint4 *>(ops_dev), iters, out_dev);
    CNS_CUDA(cudaGetLastError());
    return CNS_SUCCESS;
}
