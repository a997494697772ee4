"""cns_statemachine_run_noalloc: the op-stream state machine for callers that
may not allocate device memory (for instance a plug-in whose host framework
owns the whole GPU through its own pool, or a loop that cannot afford the
device-wide stalls cudaMalloc can cause).  Its results must be exactly those
of cns_statemachine_run, which takes caller-provided scratch, on two calls in
a row -- the second sees whatever the first left in the library's built-in
scratch array.  This file is collected last on purpose."""
import numpy as np
import pytest

import cns_inputs as ci

pytestmark = pytest.mark.gpu


def test_noalloc_state_machine_matches_scratch_entry_point_twice():
    import torch
    import counted_notify_sync_gb300 as cns

    cns.build()
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


def test_noalloc_state_machine_rejects_sizes_over_its_limit():
    import counted_notify_sync_gb300 as cns

    cns.build()
    L = cns._native.lib()
    over = cns.CNS_STATEMACHINE_NOALLOC_MAX_OPS + 1
    assert L.cns_statemachine_run_noalloc(0x1000, over, 0, 0x2000, 0x3000, None) == cns.CNS_ERR_INVALID_VALUE
    assert L.cns_statemachine_run_noalloc(0x1000, -1, 0, 0x2000, 0x3000, None) == cns.CNS_ERR_INVALID_VALUE
