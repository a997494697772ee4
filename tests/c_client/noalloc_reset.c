/* cns_statemachine_run_noalloc across a device reset, from a plain C program.
 * The entry point finds its built-in scratch array's device address once per
 * device; cudaDeviceReset destroys the context, and the next context loads
 * the library's device image anew, so the address must be looked up again.
 * The program runs one op stream through cns_statemachine_run (caller
 * scratch) for the expected trace, then through the allocation-free entry
 * point, resets the device, and runs it once more with fresh buffers.  It
 * calls the allocation-free entry point after the reset only when the
 * driver reports a new context id (the library keys its lookup on that id);
 * otherwise it prints "skip".  Prints "ok" and exits 0, or names the first
 * failure and exits 1.  Built and run by the GPU tests. */
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda.h>
#include <cuda_runtime.h>

#include "cns.h"

#define N 200003

static int fail(const char *what, int code)
{
    printf("FAIL %s: %d\n", what, code);
    return 1;
}

/* The current context's unique id from the driver (cuCtxGetCurrent,
 * cuCtxGetId, reached through the runtime), 0 if unknown. */
static unsigned long long context_id(void)
{
    CUresult (*get_current)(CUcontext *) = NULL;
    CUresult (*get_id)(CUcontext, unsigned long long *) = NULL;
    enum cudaDriverEntryPointQueryResult q;
    void *f = NULL;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) ||
        q != cudaDriverEntryPointSuccess)
        return 0;
    get_current = (CUresult(*)(CUcontext *))f;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &f, 12000, cudaEnableDefault, &q) ||
        q != cudaDriverEntryPointSuccess)
        return 0;
    get_id = (CUresult(*)(CUcontext, unsigned long long *))f;
    CUcontext c = NULL;
    unsigned long long id = 0;
    if (get_current(&c) != CUDA_SUCCESS || !c || get_id(c, &id) != CUDA_SUCCESS)
        return 0;
    return id;
}

/* One run of the allocation-free entry point on fresh device buffers; the
 * trace and final count come back into trace_h / final_h. */
static int run_noalloc(const uint32_t *ops_h, uint32_t *trace_h, uint32_t *final_h)
{
    void *ops_d, *trace_d, *final_d;
    if (cudaMalloc(&ops_d, (size_t)N * 16) || cudaMalloc(&trace_d, (size_t)N * 8) || cudaMalloc(&final_d, 4))
        return fail("cudaMalloc", 0);
    if (cudaMemcpy(ops_d, ops_h, (size_t)N * 16, cudaMemcpyHostToDevice))
        return fail("cudaMemcpy", 0);
    int rc = cns_statemachine_run_noalloc((const uint32_t *)ops_d, N, 7u, (uint32_t *)trace_d, (uint32_t *)final_d,
                                          NULL);
    if (rc)
        return fail("cns_statemachine_run_noalloc", rc);
    if (cudaMemcpy(trace_h, trace_d, (size_t)N * 8, cudaMemcpyDeviceToHost) ||
        cudaMemcpy(final_h, final_d, 4, cudaMemcpyDeviceToHost))
        return fail("cudaMemcpy back", 0);
    cudaFree(ops_d);
    cudaFree(trace_d);
    cudaFree(final_d);
    return 0;
}

int main(void)
{
    uint32_t *ops = malloc((size_t)N * 16), *want = malloc((size_t)N * 8), *got = malloc((size_t)N * 8);
    if (!ops || !want || !got)
        return fail("malloc", 0);
    /* ops: record or try-wait, a valid mode, small values so that waits go both ways */
    uint64_t x = 0x9E3779B97F4A7C15ull;
    for (int i = 0; i < N; ++i) {
        x = x * 6364136223846793005ull + 1442695040888963407ull;
        const uint32_t r = (uint32_t)(x >> 33);
        const uint32_t kind = r & 1u;
        const uint32_t rec_modes[4] = {CNS_REC_SET, CNS_REC_ADD, CNS_REC_BIT_OR, CNS_REC_BIT_AND};
        ops[4 * i + 0] = kind;
        ops[4 * i + 1] = kind ? (r >> 1) % 5u : rec_modes[(r >> 1) & 3u];
        ops[4 * i + 2] = (r >> 4) & 15u;
        ops[4 * i + 3] = ((r >> 12) & 7u) == 0u;
    }
    /* expected: the entry point with caller scratch */
    void *ops_d, *trace_d, *final_d, *scratch_d;
    const size_t sb = cns_statemachine_scratch_bytes(N);
    if (cudaMalloc(&ops_d, (size_t)N * 16) || cudaMalloc(&trace_d, (size_t)N * 8) || cudaMalloc(&final_d, 4) ||
        cudaMalloc(&scratch_d, sb))
        return fail("cudaMalloc", 0);
    if (cudaMemcpy(ops_d, ops, (size_t)N * 16, cudaMemcpyHostToDevice))
        return fail("cudaMemcpy", 0);
    int rc = cns_statemachine_run((const uint32_t *)ops_d, N, 7u, (uint32_t *)trace_d, (uint32_t *)final_d, scratch_d,
                                  sb, NULL);
    if (rc)
        return fail("cns_statemachine_run", rc);
    uint32_t want_final = 0, got_final = 0;
    if (cudaMemcpy(want, trace_d, (size_t)N * 8, cudaMemcpyDeviceToHost) ||
        cudaMemcpy(&want_final, final_d, 4, cudaMemcpyDeviceToHost))
        return fail("cudaMemcpy back", 0);
    cudaFree(ops_d);
    cudaFree(trace_d);
    cudaFree(final_d);
    cudaFree(scratch_d);

    if (run_noalloc(ops, got, &got_final))
        return 1;
    if (memcmp(got, want, (size_t)N * 8) || got_final != want_final)
        return fail("trace before the reset", 0);

    const unsigned long long before = context_id();
    if (cudaDeviceReset())
        return fail("cudaDeviceReset", 0);
    if (cudaSetDevice(0))   /* makes the new primary context */
        return fail("cudaSetDevice", 0);
    void *probe = NULL;
    if (cudaMalloc(&probe, 16))   /* any runtime call that needs the context brings it up */
        return fail("cudaMalloc after reset", 0);
    cudaFree(probe);
    const unsigned long long after = context_id();
    if (before == 0 || after == 0 || after == before) {
        printf("skip\n");
        return 0;
    }
    memset(got, 0xFF, (size_t)N * 8);
    got_final = 0xFFFFFFFFu;
    if (run_noalloc(ops, got, &got_final))
        return 1;
    if (memcmp(got, want, (size_t)N * 8) || got_final != want_final)
        return fail("trace after the reset", 0);
    printf("ok\n");
    return 0;
}
