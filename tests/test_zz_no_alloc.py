"""cns_statemachine_run_noalloc: the op-stream state machine for callers that
may not allocate device memory (for instance a plug-in whose host framework
owns the whole GPU through its own pool, or a loop that cannot afford the
device-wide stalls cudaMalloc can cause).  Its results must be exactly those
of cns_statemachine_run, which takes caller-provided scratch, and of the
oracle, on two calls in a row -- the second sees whatever the first left in
the library's built-in scratch array.  This file is collected last on
purpose."""
import os
import subprocess

import numpy as np
import pytest

import cns_inputs as ci
import oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_noalloc_state_machine_matches_scratch_entry_point_twice():
    import torch
    import counted_notify_sync_gb300 as cns

    cns.build()
    oracle.build()
    torch.cuda.set_device(0)
    L = cns._native.lib()
    limit = cns.CNS_STATEMACHINE_NOALLOC_MAX_OPS
    for n, seed, init in ((limit, 21, 0), (12_345, 22, 0xABCD)):
        ops = ci.notify_ops(n, seed=seed)
        ops_d = torch.from_numpy(ops.view(np.int32)).cuda()
        want_trace, want_final = cns.run_statemachine(ops_d, init)          # existing entry point
        trace = torch.full((n, 2), -1, dtype=torch.int32, device="cuda")
        final = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        rc = L.cns_statemachine_run_noalloc(ops_d.data_ptr(), n, init, trace.data_ptr(), final.data_ptr(), None)
        assert rc == cns.CNS_SUCCESS
        torch.cuda.synchronize()
        # integer results: bit-exact, as in every other state-machine test
        assert torch.equal(trace, want_trace)
        assert torch.equal(final, want_final)
        # and the pages' sequential definition, applied op by op by the oracle
        o_trace, o_final = oracle.cnt_statemachine(ops, init)
        np.testing.assert_array_equal(trace.cpu().numpy().view(np.uint32), o_trace)
        assert int(final.cpu().numpy().view(np.uint32)[0]) == o_final


def test_noalloc_state_machine_rejects_sizes_over_its_limit():
    import counted_notify_sync_gb300 as cns

    cns.build()
    L = cns._native.lib()
    over = cns.CNS_STATEMACHINE_NOALLOC_MAX_OPS + 1
    assert L.cns_statemachine_run_noalloc(0x1000, over, 0, 0x2000, 0x3000, None) == cns.CNS_ERR_INVALID_VALUE
    assert L.cns_statemachine_run_noalloc(0x1000, -1, 0, 0x2000, 0x3000, None) == cns.CNS_ERR_INVALID_VALUE


def test_noalloc_state_machine_across_a_device_reset():
    """A plain C program (its own process, so the reset ends only its own
    context) runs the allocation-free entry point before and after
    cudaDeviceReset and checks both traces against cns_statemachine_run."""
    import counted_notify_sync_gb300 as cns
    from counted_notify_sync_gb300 import builder
    lib = cns.build()
    libdir = os.path.dirname(os.path.abspath(lib))
    cuda = builder.cuda_home()
    out = os.path.join(ROOT, "tests", "c_client", "_build", "noalloc_reset")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cudart_dir = next(d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"),
                                  os.path.join(cuda, "targets", "sbsa-linux", "lib"),
                                  os.path.join(cuda, "targets", "x86_64-linux", "lib"))
                      if os.path.exists(os.path.join(d, "libcudart.so")))
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), "-o", out,
                    os.path.join(ROOT, "tests", "c_client", "noalloc_reset.c"),
                    "-L", libdir, "-lcns", "-L", cudart_dir, "-lcudart",
                    f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cudart_dir}"], check=True)
    r = subprocess.run([out], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() in ("ok", "skip"), r.stdout + r.stderr
