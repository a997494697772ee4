/*
 * Multithreaded CPU timing twin of the SYNCALL data rounds and of the
 * counted-notify pipeline.
 *
 * TEST AND BASELINE INFRASTRUCTURE ONLY.  This is not the correctness oracle
 * (cns_oracle.c is): it exists to put a parallel CPU figure beside the GPU's
 * in the benchmark, and its results are checked against the oracle in the
 * CPU tests.
 *
 * The soft barrier follows "PTO-ISA SYNCALL cross-core barrier guide" §5.2
 * among T host threads: each arrival is one atomic add that returns `before`,
 * the target is (before / T + 1) * T, and the thread spins on acquire loads
 * until the count has reached the target.  The runs here start the count at 0
 * and stay far below 2^31 arrivals, so the literal u32 arithmetic with a
 * signed-difference "reached" test is exact (the wrap-safe form is the
 * oracle's and the GPU's business).  P participants are shared out over T
 * threads in contiguous blocks; a thread runs the data phase of each of its
 * participants and then arrives once.
 *
 * The pipeline follows "CANN Runtime CntNotify management API" §5: a
 * producer thread stores each tile and records ADD 1 per tile on `done`
 * (release); a consumer thread waits until done >= tiles (acquire), clears
 * it, sums the tile area mod 2^32 and records ack = round + 1 (release);
 * the producer of round r first waits for ack >= r.
 *
 * Build: gcc -O2 -std=c11 -pthread -ffp-contract=off -fPIC -shared.
 */
#define _POSIX_C_SOURCE 200809L
#include <pthread.h>
#include <stdatomic.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <time.h>

enum { TW_OK = 0, TW_BAD_ARG = 2, TW_NO_THREAD = 3 };
enum { TW_RING_AFFINE = 1, TW_RING_ROTATE = 2, TW_XORSHIFT = 3 };

static double now_s(void)
{
    struct timespec t;
    clock_gettime(CLOCK_MONOTONIC, &t);
    return (double)t.tv_sec + 1e-9 * (double)t.tv_nsec;
}

/* ---- the epoch barrier among T threads ---------------------------------- */

typedef struct {
    _Alignas(128) atomic_uint count;
    _Alignas(128) uint32_t T;
} twin_barrier_t;

static void twin_barrier_wait(twin_barrier_t *b)
{
    const uint32_t before = atomic_fetch_add_explicit(&b->count, 1u, memory_order_acq_rel);
    const uint32_t target = (before / b->T + 1u) * b->T;
    while ((int32_t)(atomic_load_explicit(&b->count, memory_order_acquire) - target) < 0) {
    }
}

/* ---- ring workloads ----------------------------------------------------- */

typedef struct {
    int wl;
    uint32_t P;
    int64_t rounds, slots;
    uint32_t *buf[2];
    twin_barrier_t *bar;
    atomic_int *ready;
    int threads;
    uint32_t p0, p1;          /* this thread's participants */
    double t0, t1;            /* thread 0: timed span */
} ring_job_t;

static uint32_t xs32(uint32_t x)
{
    x ^= x << 13;
    x ^= x >> 17;
    x ^= x << 5;
    return x;
}

static void *ring_thread(void *arg)
{
    ring_job_t *j = (ring_job_t *)arg;
    /* start line: every thread is running before the clock starts */
    atomic_fetch_add_explicit(j->ready, 1, memory_order_acq_rel);
    while (atomic_load_explicit(j->ready, memory_order_acquire) < j->threads) {
    }
    if (j->p0 == 0)
        j->t0 = now_s();
    for (int64_t r = 0; r < j->rounds; ++r) {
        const uint32_t *src = j->buf[r & 1];
        uint32_t *dst = j->buf[(r + 1) & 1];
        for (uint32_t p = j->p0; p < j->p1; ++p) {
            const uint32_t q = (p + 1u == j->P) ? 0u : p + 1u;
            const uint32_t *s = src + (int64_t)q * j->slots;
            uint32_t *d = dst + (int64_t)p * j->slots;
            for (int64_t i = 0; i < j->slots; ++i) {
                const uint32_t x = s[i];
                if (j->wl == TW_RING_AFFINE)
                    d[i] = x * 3u + (uint32_t)r;
                else if (j->wl == TW_RING_ROTATE)
                    d[i] = x;
                else
                    d[i] = xs32(x) ^ (uint32_t)r;
            }
        }
        twin_barrier_wait(j->bar);
    }
    if (j->p0 == 0)
        j->t1 = now_s();
    return NULL;
}

/* R rounds of a ring workload over P participants (slots uint32 each) on
 * `threads` host threads.  buf0 holds the input; the result is in buf[R & 1].
 * Out: seconds of the timed span (thread 0, from the start line to its last
 * barrier), the final barrier count (R * T). */
int twin_syncall_ring(int wl, uint32_t P, int64_t rounds, int threads, uint32_t *buf0, uint32_t *buf1,
                      int64_t slots, double *seconds, uint32_t *final_count)
{
    if (P < 1 || rounds < 0 || slots < 0 || threads < 1 || !buf0 || !buf1 || !seconds || !final_count)
        return TW_BAD_ARG;
    if (wl != TW_RING_AFFINE && wl != TW_RING_ROTATE && wl != TW_XORSHIFT)
        return TW_BAD_ARG;
    const uint32_t T = (uint32_t)threads < P ? (uint32_t)threads : P;
    twin_barrier_t bar;
    atomic_init(&bar.count, 0u);
    bar.T = T;
    atomic_int ready;
    atomic_init(&ready, 0);
    ring_job_t *jobs = calloc(T, sizeof(ring_job_t));
    pthread_t *tid = calloc(T, sizeof(pthread_t));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return TW_NO_THREAD;
    }
    for (uint32_t k = 0; k < T; ++k) {
        ring_job_t *j = &jobs[k];
        j->wl = wl;
        j->P = P;
        j->rounds = rounds;
        j->slots = slots;
        j->buf[0] = buf0;
        j->buf[1] = buf1;
        j->bar = &bar;
        j->ready = &ready;
        j->threads = (int)T;
        j->p0 = (uint32_t)(((uint64_t)P * k) / T);
        j->p1 = (uint32_t)(((uint64_t)P * (k + 1)) / T);
    }
    uint32_t started = 0;
    int rc = TW_OK;
    for (; started < T; ++started) {
        if (pthread_create(&tid[started], NULL, ring_thread, &jobs[started]) != 0) {
            rc = TW_NO_THREAD;
            break;
        }
    }
    if (rc != TW_OK) {
        /* the started threads wait at the start line for the missing ones: let
           them through with no rounds to run */
        for (uint32_t k = 0; k < started; ++k)
            jobs[k].rounds = 0;
        atomic_fetch_add_explicit(&ready, (int)(T - started), memory_order_acq_rel);
    }
    for (uint32_t k = 0; k < started; ++k)
        pthread_join(tid[k], NULL);
    *seconds = jobs[0].t1 - jobs[0].t0;
    *final_count = atomic_load(&bar.count);
    free(jobs);
    free(tid);
    return rc;
}

/* ---- Jacobi ------------------------------------------------------------- */

typedef struct {
    float *buf[2];
    int64_t n, sweeps, i0, i1;
    twin_barrier_t *bar;
    atomic_int *ready;
    int threads, first;
    double t0, t1;
} jac_job_t;

static void *jac_thread(void *arg)
{
    jac_job_t *j = (jac_job_t *)arg;
    atomic_fetch_add_explicit(j->ready, 1, memory_order_acq_rel);
    while (atomic_load_explicit(j->ready, memory_order_acquire) < j->threads) {
    }
    if (j->first)
        j->t0 = now_s();
    for (int64_t s = 0; s < j->sweeps; ++s) {
        const float *u = j->buf[s & 1];
        float *v = j->buf[(s + 1) & 1];
        for (int64_t i = j->i0; i < j->i1; ++i)
            v[i] = (i == 0 || i == j->n - 1) ? u[i] : (u[i - 1] + u[i + 1]) * 0.5f;
        twin_barrier_wait(j->bar);
    }
    if (j->first)
        j->t1 = now_s();
    return NULL;
}

/* `sweeps` Jacobi sweeps of the 3-point Laplacian (fixed ends) over n points
 * on `threads` host threads, contiguous chunks, one barrier per sweep.  The
 * result is in buf[sweeps & 1].  Out: seconds of the timed span. */
int twin_jacobi(float *buf0, float *buf1, int64_t n, int64_t sweeps, int threads, double *seconds)
{
    if (!buf0 || !buf1 || n < 1 || sweeps < 0 || threads < 1 || !seconds)
        return TW_BAD_ARG;
    const int64_t T = threads < n ? threads : n;
    twin_barrier_t bar;
    atomic_init(&bar.count, 0u);
    bar.T = (uint32_t)T;
    atomic_int ready;
    atomic_init(&ready, 0);
    jac_job_t *jobs = calloc((size_t)T, sizeof(jac_job_t));
    pthread_t *tid = calloc((size_t)T, sizeof(pthread_t));
    if (!jobs || !tid) {
        free(jobs);
        free(tid);
        return TW_NO_THREAD;
    }
    for (int64_t k = 0; k < T; ++k) {
        jac_job_t *j = &jobs[k];
        j->buf[0] = buf0;
        j->buf[1] = buf1;
        j->n = n;
        j->sweeps = sweeps;
        j->i0 = n * k / T;
        j->i1 = n * (k + 1) / T;
        j->bar = &bar;
        j->ready = &ready;
        j->threads = (int)T;
        j->first = (k == 0);
    }
    int64_t started = 0;
    int rc = TW_OK;
    for (; started < T; ++started) {
        if (pthread_create(&tid[started], NULL, jac_thread, &jobs[started]) != 0) {
            rc = TW_NO_THREAD;
            break;
        }
    }
    if (rc != TW_OK) {
        for (int64_t k = 0; k < started; ++k)
            jobs[k].sweeps = 0;
        atomic_fetch_add_explicit(&ready, (int)(T - started), memory_order_acq_rel);
    }
    for (int64_t k = 0; k < started; ++k)
        pthread_join(tid[k], NULL);
    *seconds = jobs[0].t1 - jobs[0].t0;
    free(jobs);
    free(tid);
    return rc;
}

/* ---- counted-notify pipeline -------------------------------------------- */

typedef struct {
    _Alignas(128) atomic_uint done;
    _Alignas(128) atomic_uint ack;
    uint32_t *tiles;
    int64_t n_tiles, rounds;
    int tile_words, areas;
    uint32_t *checksums;
} pipe_t;

/* Round r writes area r % areas.  With one area the producer waits until the
 * consumer has read round r - 1; with two, until it has read round r - 2 (the
 * area's last use) and has cleared round r - 1's count, which every record of
 * round r must follow. */
static void *pipe_producer(void *arg)
{
    pipe_t *p = (pipe_t *)arg;
    const int64_t n = p->n_tiles * p->tile_words;
    for (int64_t r = 0; r < p->rounds; ++r) {
        const uint32_t need = p->areas == 2 ? (r >= 1 ? (uint32_t)(r - 1) : 0u) : (uint32_t)r;
        while (atomic_load_explicit(&p->ack, memory_order_acquire) < need) {
        }
        if (p->areas == 2) {
            while (atomic_load_explicit(&p->done, memory_order_acquire) >= (uint32_t)p->n_tiles) {
            }
        }
        uint32_t *area = p->tiles + (p->areas == 2 ? (r & 1) * n : 0);
        for (int64_t t = 0; t < p->n_tiles; ++t) {
            uint32_t *d = area + t * p->tile_words;
            const uint32_t w0 = (uint32_t)(t * p->tile_words);
            for (int i = 0; i < p->tile_words; ++i)
                d[i] = (w0 + (uint32_t)i) * 2654435761u + (uint32_t)r;
            atomic_fetch_add_explicit(&p->done, 1u, memory_order_release);   /* record ADD 1 */
        }
    }
    return NULL;
}

static void pipe_consume(pipe_t *p)
{
    const int64_t n = p->n_tiles * p->tile_words;
    for (int64_t r = 0; r < p->rounds; ++r) {
        while (atomic_load_explicit(&p->done, memory_order_acquire) < (uint32_t)p->n_tiles) {
        }
        atomic_store_explicit(&p->done, 0u, memory_order_relaxed);              /* isClear */
        const uint32_t *area = p->tiles + (p->areas == 2 ? (r & 1) * n : 0);
        uint32_t s = 0;
        for (int64_t i = 0; i < n; ++i)
            s += area[i];
        p->checksums[r] = s;
        atomic_store_explicit(&p->ack, (uint32_t)(r + 1), memory_order_release);   /* record SET r + 1 */
    }
}

/* `rounds` rounds of the two-thread pipeline over tiles x tile_words words in
 * `areas` (1 or 2) tile areas.  Out: checksums[rounds], seconds of the whole run. */
int twin_pipeline(int64_t n_tiles, int tile_words, int64_t rounds, int areas, uint32_t *checksums, double *seconds)
{
    if (n_tiles < 1 || tile_words < 1 || rounds < 0 || !checksums || !seconds || areas < 1 || areas > 2)
        return TW_BAD_ARG;
    if (n_tiles > ((int64_t)1 << 32) / tile_words)
        return TW_BAD_ARG;
    pipe_t p;
    atomic_init(&p.done, 0u);
    atomic_init(&p.ack, 0u);
    p.tiles = malloc((size_t)(areas * n_tiles * tile_words) * sizeof(uint32_t));
    if (!p.tiles)
        return TW_NO_THREAD;
    p.n_tiles = n_tiles;
    p.tile_words = tile_words;
    p.areas = areas;
    p.rounds = rounds;
    p.checksums = checksums;
    pthread_t prod;
    const double t0 = now_s();
    if (pthread_create(&prod, NULL, pipe_producer, &p) != 0) {
        free(p.tiles);
        return TW_NO_THREAD;
    }
    pipe_consume(&p);
    pthread_join(prod, NULL);
    *seconds = now_s() - t0;
    free(p.tiles);
    return TW_OK;
}
