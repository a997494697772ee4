/* A plain C program that uses libcns.so through include/cns.h only (no Python):
 * a die-local soft SYNCALL ring of 148 CTAs on an 8 KB-aligned workspace, the
 * same through the hard path (with the cluster barrier and with the paired
 * step), each also on a workspace sized by syncall_workspace_bytes for the
 * per-die payload copies, and a counted notify recorded on one stream and
 * waited on another, at gpu scope and after cntnotify_enable_peer (system
 * scope, the peer being this device).  Expected values are closed forms: after R ring-rotate
 * rounds participant p holds participant (p + R) mod P's starting row; the soft
 * counter ends at R * P.  Prints "ok" and exits 0, or names the first failure
 * and exits 1.  Built and run by the GPU tests. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime.h>

#include "cns.h"

#define P 148
#define ROUNDS 1001

static int fail(const char *what, int code)
{
    printf("FAIL %s: %d (%s)\n", what, code, cns_error_string(code));
    return 1;
}

static int ring(int mode, int copies, int hard_step)
{
    uint32_t host0[P * 4], host_out[P * 4];
    for (int i = 0; i < P * 4; ++i)
        host0[i] = (uint32_t)i * 2654435761u + 12345u;
    size_t ws_bytes = CNS_SYNCALL_WORKSPACE_DIE_LOCAL_BYTES;
    int rc;
    if (copies && (rc = syncall_workspace_bytes(P, 4, &ws_bytes)))
        return fail("syncall_workspace_bytes", rc);
    void *b0, *b1, *raw;
    if (cudaMalloc(&b0, sizeof host0) || cudaMalloc(&b1, sizeof host0) ||
        cudaMalloc(&raw, ws_bytes + CNS_SYNCALL_DIE_LOCAL_ALIGN))
        return fail("cudaMalloc", 0);
    void *ws = (void *)(((uintptr_t)raw + CNS_SYNCALL_DIE_LOCAL_ALIGN - 1) &
                        ~(uintptr_t)(CNS_SYNCALL_DIE_LOCAL_ALIGN - 1));
    rc = syncall_workspace_init(ws, ws_bytes, 0, NULL);
    if (rc)
        return fail("syncall_workspace_init", rc);
    cns_syncall_data_t d;
    memset(&d, 0, sizeof d);
    d.workload = CNS_WL_RING_ROTATE;
    d.launch_ctas = P;
    d.threads = 256;
    d.buf0_dev = b0;
    d.buf1_dev = b1;
    d.elems = 4;
    d.workspace_dev = ws;
    d.workspace_bytes = (uint32_t)ws_bytes;
    d.barrier_variant = CNS_BARRIER_DIE_LOCAL;
    d.hard_step = hard_step;
    d.sync = 1;
    d.host_in = host0;
    d.host_out = host_out;
    rc = syncall_run(mode, CNS_AIV_ONLY, 0, 0, ROUNDS, &d);
    if (rc)
        return fail(mode == CNS_SYNCALL_SOFT ? "syncall_run soft" : "syncall_run hard", rc);
    for (int p = 0; p < P; ++p)
        for (int j = 0; j < 4; ++j)
            if (host_out[p * 4 + j] != host0[((p + ROUNDS) % P) * 4 + j])
                return fail("ring payload", p);
    const uint32_t groups = mode == CNS_SYNCALL_SOFT ? P : P / (uint32_t)d.cluster_used;
    if (d.device_status != 0 || d.final_counter != (uint32_t)ROUNDS * groups)
        return fail("final counter", (int)d.final_counter);
    cudaFree(b0);
    cudaFree(b1);
    cudaFree(raw);
    return 0;
}

static int notify(int peer)
{
    cudaStream_t s1, s2;
    if (cudaStreamCreate(&s1) || cudaStreamCreate(&s2))
        return fail("cudaStreamCreate", 0);
    cns_cnt_notify_t n;
    int rc = cntnotify_create(&n, 0);
    if (rc)
        return fail("cntnotify_create", rc);
    int dev = 0;
    if (peer && (cudaGetDevice(&dev) || (rc = cntnotify_enable_peer(n, dev))))
        return fail("cntnotify_enable_peer", rc);
    const cns_record_info_t add = {CNS_REC_ADD, 1};
    const cns_wait_info_t wait = {CNS_WAIT_BIGGER_OR_EQUAL, 3, 10, 1, {0, 0, 0}};
    for (int i = 0; i < 3; ++i)
        if ((rc = cntnotify_record(n, s1, &add)))
            return fail("cntnotify_record", rc);
    if ((rc = cntnotify_wait_with_timeout(n, s2, &wait)))
        return fail("cntnotify_wait_with_timeout", rc);
    cudaStreamSynchronize(s2);
    int32_t st = -1;
    uint32_t count = 99;
    if ((rc = cntnotify_query_status(n, &st, &count)) || st != 0 || count != 0)
        return fail("cntnotify_query_status", rc ? rc : (int)count);
    if ((rc = cntnotify_destroy(n)))
        return fail("cntnotify_destroy", rc);
    cudaStreamDestroy(s1);
    cudaStreamDestroy(s2);
    return 0;
}

int main(void)
{
    int32_t version = 0, sm = 0;
    if (cns_version(&version, &sm) || sm != 103)
        return fail("cns_version", sm);
    for (int copies = 0; copies < 2; ++copies)
        if (ring(CNS_SYNCALL_SOFT, copies, CNS_HARD_STEP_CLUSTER_BARRIER) ||
            ring(CNS_SYNCALL_HARD, copies, CNS_HARD_STEP_CLUSTER_BARRIER) ||
            ring(CNS_SYNCALL_HARD, copies, CNS_HARD_STEP_PAIRED_MBARRIER))
            return 1;
    if (notify(0) || notify(1))
        return 1;
    printf("ok\n");
    return 0;
}
