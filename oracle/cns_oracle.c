/*
 * cns_oracle.c -- plain, sequential CPU oracle for the counted-notify / SYNCALL
 * hot path.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this file's library.  The CUDA library
 * never includes, links or calls anything here, and nothing here comes from
 * the CUDA side: the two are written independently and meet only in the
 * parity tests, on the same seeded inputs.
 *
 * Sources (web pages; section numbers are the pages' own):
 *   [SYNCALL] "PTO-ISA 跨核同步屏障 SYNCALL 实战指南" (PTO-ISA SYNCALL cross-core
 *             barrier guide), lmnt.cn/news/269652.
 *   [CNTN]    "CANN Runtime CntNotify（计数型通知）管理接口详解" (CANN Runtime
 *             CntNotify management API), bjdmk.com.cn/news/4842886.
 *
 * Readings taken where the pages are silent or garbled (each is repeated in
 * the design notes):
 *   - the target formula lost its '=' and '+' in extraction; it is read as
 *     target = (before / P + 1) * P with floor division   ([SYNCALL] §5.2)
 *   - "poll until the count reaches target" is read as cur >= target, taken
 *     modulo the counter's cycle length (below), not cur == target
 *   - the counter is unsigned 32-bit.  The wrap-safe form keeps it in Z_M with
 *     M = P * floor(2^32 / P), a multiple of P, so the epoch arithmetic never
 *     breaks at the wrap; for a power-of-two P, M = 2^32 and this is the plain
 *     wrapping u32 add.
 *   - record and wait values are uint32 and compare unsigned ([CNTN] §3.3)
 *   - a wait inside the op-stream state machine is a try-wait: it tests the
 *     predicate once, applies the clear only if satisfied, never blocks.
 *
 * Every floating-point step is single precision, as the Jacobi workload is
 * defined in fp32; build with -ffp-contract=off.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_DEADLOCK 1
#define ORC_BAD_ARG 2

/* ------------------------------------------------------------------------- */
/* SYNCALL soft-mode epoch barrier arithmetic  ([SYNCALL] §5.2, §4.1, §4.2)    */
/* ------------------------------------------------------------------------- */

/* Literal target of the soft barrier: the count at which the last of the P
 * participants of the current round has arrived.  u32 arithmetic. */
uint32_t oracle_epoch_target(uint32_t before, uint32_t P)
{
    return (before / P + 1u) * P;
}

/* Cycle length M of the wrap-safe counter: the largest multiple of P that is
 * <= 2^32.  Returned as 64-bit because M = 2^32 for every power-of-two P. */
uint64_t oracle_counter_modulus(uint32_t P)
{
    return (uint64_t)P * ((UINT64_C(1) << 32) / (uint64_t)P);
}

/* One arrival on the wrap-safe counter: c -> (c + 1) mod M. */
uint32_t oracle_arrive_mod(uint32_t c, uint64_t M)
{
    return (uint32_t)(((uint64_t)c + 1u) % M);
}

/* Target in Z_M: ((before div P) + 1) * P mod M. */
uint32_t oracle_target_mod(uint32_t before, uint32_t P, uint64_t M)
{
    uint64_t t = ((uint64_t)before / P + 1u) * (uint64_t)P;
    return (uint32_t)(t % M);
}

/* "The count has reached target" in Z_M.  While a participant polls, the
 * counter lies in [before+1, target+P-1] (the fastest peers can be at most one
 * round ahead), so cur has reached target exactly when (cur - target) mod M
 * is below P.  Needs M >= 2P, true for every P <= 2^31. */
int oracle_reached_mod(uint32_t cur, uint32_t target, uint32_t P, uint64_t M)
{
    uint64_t d = ((uint64_t)cur + M - (uint64_t)target) % M;
    return d < (uint64_t)P;
}

/* ------------------------------------------------------------------------- */
/* Round payloads.  Each round every participant p reads its ring neighbour  */
/* (p+1) mod P from the previous round's buffer and writes its own slots of  */
/* the next buffer; the barrier separates the rounds.  The pages' multi-round */
/* soft test checks cross-core visibility of values written before a barrier */
/* ([SYNCALL] §6.1, §8); these payloads make every round depend on another   */
/* participant's previous round, so a missed barrier changes the result.     */
/* ------------------------------------------------------------------------- */

enum { ORC_WL_EMPTY = 0, ORC_WL_RING_AFFINE = 1, ORC_WL_RING_ROTATE = 2, ORC_WL_XORSHIFT = 3, ORC_WL_JACOBI = 4 };

/* Marsaglia's xorshift32 step with shifts (13, 17, 5) ("Xorshift RNGs",
 * Journal of Statistical Software 8(14), 2003). */
uint32_t oracle_xorshift32(uint32_t x)
{
    x ^= x << 13;
    x ^= x >> 17;
    x ^= x << 5;
    return x;
}

/* One payload round r for participant p on the u32 ring workloads.
 * old and nw are [P][slots] row-major. */
static void ring_round(int wl, const uint32_t *old, uint32_t *nw, uint32_t P, int64_t slots, uint64_t r)
{
    for (uint32_t p = 0; p < P; ++p) {
        const uint32_t *src = old + (int64_t)((p + 1u) % P) * slots;
        uint32_t *dst = nw + (int64_t)p * slots;
        for (int64_t i = 0; i < slots; ++i) {
            uint32_t x = src[i];
            if (wl == ORC_WL_RING_AFFINE)
                x = x * 3u + (uint32_t)r;
            else if (wl == ORC_WL_XORSHIFT)
                x = oracle_xorshift32(x) ^ (uint32_t)r;
            /* ORC_WL_RING_ROTATE: plain copy */
            dst[i] = x;
        }
    }
}

/* 3-point Jacobi sweep on a 1-D field with fixed ends:
 * u'[i] = (u[i-1] + u[i+1]) * 0.5 for 0 < i < N-1, u'[0] = u[0], u'[N-1] = u[N-1]. */
static void jacobi_sweep(const float *u, float *un, int64_t N)
{
    if (N <= 0)
        return;
    un[0] = u[0];
    for (int64_t i = 1; i < N - 1; ++i)
        un[i] = (u[i - 1] + u[i + 1]) * 0.5f;
    if (N > 1)
        un[N - 1] = u[N - 1];
}

/* One soft barrier among P participants, arriving in index order, on the
 * wrap-safe counter *c.  Every participant computes its target from the
 * value it got back; the barrier opens only if all of them have reached their
 * target once everyone has arrived.  Returns ORC_DEADLOCK otherwise. */
static int barrier_round(uint32_t *c, uint32_t P, uint64_t M, uint32_t *targets)
{
    for (uint32_t p = 0; p < P; ++p) {
        uint32_t before = *c;
        *c = oracle_arrive_mod(*c, M);
        targets[p] = oracle_target_mod(before, P, M);
    }
    for (uint32_t p = 0; p < P; ++p)
        if (!oracle_reached_mod(*c, targets[p], P, M))
            return ORC_DEADLOCK;
    return ORC_OK;
}

/*
 * Sequential definition of a SYNCALL soft run: `rounds` times { payload round
 * r for every participant; one soft barrier }.
 *   wl        ORC_WL_* workload
 *   P         participant count (>= 1)
 *   rounds    number of rounds R
 *   start     counter value before the first arrival (the workspace must be
 *             zeroed before first use, [SYNCALL] §4.1; other multiples of P
 *             model a reused workspace)
 *   u32       [P][slots] ring state (ring workloads), in: round 0, out: round R
 *   f32, n    Jacobi field of n points (Jacobi workload), in/out
 *   final_counter  out: counter after the last barrier
 * Returns ORC_OK, ORC_DEADLOCK (a barrier could not open) or ORC_BAD_ARG.
 */
int oracle_syncall_run(int wl, uint32_t P, uint64_t rounds, uint32_t start,
                       uint32_t *u32, int64_t slots, float *f32, int64_t n,
                       uint32_t *final_counter)
{
    if (P == 0)
        return ORC_BAD_ARG;
    uint64_t M = oracle_counter_modulus(P);
    uint32_t *targets = (uint32_t *)malloc(sizeof(uint32_t) * P);
    void *tmp = NULL;
    if (wl == ORC_WL_RING_AFFINE || wl == ORC_WL_RING_ROTATE || wl == ORC_WL_XORSHIFT) {
        if (slots < 0 || (slots > 0 && u32 == NULL)) { free(targets); return ORC_BAD_ARG; }
        tmp = malloc(sizeof(uint32_t) * (size_t)(P * (slots > 0 ? slots : 1)));
    } else if (wl == ORC_WL_JACOBI) {
        if (n < 0 || (n > 0 && f32 == NULL)) { free(targets); return ORC_BAD_ARG; }
        tmp = malloc(sizeof(float) * (size_t)(n > 0 ? n : 1));
    } else if (wl != ORC_WL_EMPTY) {
        free(targets);
        return ORC_BAD_ARG;
    }
    uint32_t c = start;
    int status = ORC_OK;
    for (uint64_t r = 0; r < rounds && status == ORC_OK; ++r) {
        if (wl == ORC_WL_JACOBI) {
            jacobi_sweep(f32, (float *)tmp, n);
            memcpy(f32, tmp, sizeof(float) * (size_t)n);
        } else if (wl != ORC_WL_EMPTY) {
            ring_round(wl, u32, (uint32_t *)tmp, P, slots, r);
            memcpy(u32, tmp, sizeof(uint32_t) * (size_t)(P * slots));
        }
        status = barrier_round(&c, P, M, targets);
    }
    if (final_counter)
        *final_counter = c;
    free(tmp);
    free(targets);
    return status;
}

/* Jacobi values of selected points after `sweeps` sweeps, one point at a
 * time.  A point after S sweeps depends only on the S points either side of
 * it, so each point is computed from that window of u0 with the same sweep
 * rule; a window edge that is not an end of the field loses one valid point
 * per sweep.  Gives the same single-precision value as the full run. */
int oracle_jacobi_points(const float *u0, int64_t N, int64_t sweeps,
                         const int64_t *idx, int64_t k, float *out)
{
    if (N <= 0 || sweeps < 0)
        return ORC_BAD_ARG;
    float *w = (float *)malloc(sizeof(float) * (size_t)(2 * sweeps + 1));
    float *wn = (float *)malloc(sizeof(float) * (size_t)(2 * sweeps + 1));
    for (int64_t q = 0; q < k; ++q) {
        int64_t i = idx[q];
        if (i < 0 || i >= N) { free(w); free(wn); return ORC_BAD_ARG; }
        int64_t a = i - sweeps < 0 ? 0 : i - sweeps;
        int64_t b = i + sweeps > N - 1 ? N - 1 : i + sweeps;
        int64_t L = b - a + 1;
        memcpy(w, u0 + a, sizeof(float) * (size_t)L);
        int64_t lo = 0, hi = L - 1;               /* valid window positions */
        for (int64_t s = 0; s < sweeps; ++s) {
            int64_t nlo = (a + lo == 0) ? lo : lo + 1;
            int64_t nhi = (a + hi == N - 1) ? hi : hi - 1;
            for (int64_t j = nlo; j <= nhi; ++j) {
                int64_t g = a + j;
                if (g == 0 || g == N - 1)
                    wn[j] = w[j];
                else
                    wn[j] = (w[j - 1] + w[j + 1]) * 0.5f;
            }
            for (int64_t j = nlo; j <= nhi; ++j)
                w[j] = wn[j];
            lo = nlo;
            hi = nhi;
        }
        out[q] = w[i - a];
    }
    free(w);
    free(wn);
    return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* CntNotify counter state machine  ([CNTN] §3.1, §3.2, §3.3)                 */
/* ------------------------------------------------------------------------- */

enum { ORC_REC_SET = 0, ORC_REC_ADD = 1, ORC_REC_OR = 2, ORC_REC_AND = 4 };
enum { ORC_WAIT_LESS = 0, ORC_WAIT_EQUAL = 1, ORC_WAIT_BIGGER = 2, ORC_WAIT_BGE = 3, ORC_WAIT_MASK = 4 };

/* Record: the new count for each record mode.  SET: value; ADD: count + value
 * (mod 2^32); BIT_OR: count | value; BIT_AND: count & value.  Mode 3 is not
 * defined.  Returns 0, or -1 for an undefined mode (count unchanged). */
int oracle_cnt_record(uint32_t c, uint32_t mode, uint32_t v, uint32_t *out)
{
    switch (mode) {
    case ORC_REC_SET: *out = v; return 0;
    case ORC_REC_ADD: *out = c + v; return 0;
    case ORC_REC_OR:  *out = c | v; return 0;
    case ORC_REC_AND: *out = c & v; return 0;
    default: *out = c; return -1;
    }
}

/* Wait predicate: when the wait is released.  LESS: count < value; EQUAL:
 * count == value; BIGGER: count > value; BIGGER_OR_EQUAL: count >= value;
 * EQUAL_WITH_BITMASK: (count & value) == value.  Unsigned compares.
 * Returns 1 (released), 0 (keeps waiting) or -1 (undefined mode). */
int oracle_cnt_wait_satisfied(uint32_t c, uint32_t mode, uint32_t v)
{
    switch (mode) {
    case ORC_WAIT_LESS:   return c < v;
    case ORC_WAIT_EQUAL:  return c == v;
    case ORC_WAIT_BIGGER: return c > v;
    case ORC_WAIT_BGE:    return c >= v;
    case ORC_WAIT_MASK:   return (c & v) == v;
    default: return -1;
    }
}

/* Outcome codes written to the trace. */
#define ORC_OUT_WAIT_HELD 0u
#define ORC_OUT_WAIT_RELEASED 1u
#define ORC_OUT_RECORD 2u
#define ORC_OUT_INVALID 3u

/*
 * Apply an op stream to one counter, in order.
 *   ops    [n][4] uint32: kind (0 record, 1 try-wait), mode, value, is_clear
 *   init   counter before the first op
 *   trace  out [n][2] uint32: counter after the op, outcome code
 *   final  out: counter after the last op
 * A try-wait that is released and has is_clear != 0 sets the counter to 0
 * afterwards ("clear after the wait is released", [CNTN] §3.3, §7 item 4).
 */
void oracle_cnt_statemachine(const uint32_t *ops, int64_t n, uint32_t init,
                             uint32_t *trace, uint32_t *final)
{
    uint32_t c = init;
    for (int64_t i = 0; i < n; ++i) {
        uint32_t kind = ops[4 * i + 0], mode = ops[4 * i + 1];
        uint32_t v = ops[4 * i + 2], clr = ops[4 * i + 3];
        uint32_t outcome;
        if (kind == 0) {
            uint32_t nc;
            if (oracle_cnt_record(c, mode, v, &nc) == 0) {
                c = nc;
                outcome = ORC_OUT_RECORD;
            } else {
                outcome = ORC_OUT_INVALID;
            }
        } else if (kind == 1) {
            int s = oracle_cnt_wait_satisfied(c, mode, v);
            if (s < 0) {
                outcome = ORC_OUT_INVALID;
            } else if (s) {
                outcome = ORC_OUT_WAIT_RELEASED;
                if (clr)
                    c = 0;
            } else {
                outcome = ORC_OUT_WAIT_HELD;
            }
        } else {
            outcome = ORC_OUT_INVALID;
        }
        trace[2 * i + 0] = c;
        trace[2 * i + 1] = outcome;
    }
    if (final)
        *final = c;
}

/* ------------------------------------------------------------------------- */
/* Two-stream counting pipeline ([CNTN] §5: producer records ADD, waiter     */
/* uses BIGGER_OR_EQUAL N with isClear)                                       */
/* ------------------------------------------------------------------------- */

/* Word w of the tile area in round r, as the producer writes it. */
uint32_t oracle_pipeline_word(int64_t w, uint64_t r)
{
    return (uint32_t)((uint64_t)w * 2654435761u) + (uint32_t)r;
}

/*
 * Per-round result of the producer/consumer pipeline: each round the producer
 * fills `tiles` tiles of `tile_words` words (oracle_pipeline_word) and adds 1
 * to the "done" notify per tile; the consumer, released once done >= tiles
 * (and clearing it), sums all words mod 2^32.  checksums[r] is that sum;
 * counts[r] is the done count the consumer was released at (tiles, since
 * exactly that many adds happen per round).
 */
void oracle_pipeline(int64_t tiles, int64_t tile_words, int64_t rounds,
                     uint32_t *checksums, uint32_t *counts)
{
    int64_t W = tiles * tile_words;
    for (int64_t r = 0; r < rounds; ++r) {
        uint32_t done = 0, sum = 0;
        for (int64_t w = 0; w < W; ++w)
            sum += oracle_pipeline_word(w, (uint64_t)r);
        for (int64_t t = 0; t < tiles; ++t) {
            uint32_t nd;
            oracle_cnt_record(done, ORC_REC_ADD, 1u, &nd);
            done = nd;
        }
        checksums[r] = sum;
        counts[r] = done;   /* released: done >= tiles; then cleared */
    }
}
