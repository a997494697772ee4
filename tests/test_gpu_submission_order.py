"""A counted-notify wait submitted (from the host) before the record that
releases it, on another stream ("CANN Runtime CntNotify management API" §5:
the waiting stream and the recording stream are independent; §7 item 6: the
calls are asynchronous).  Whether the wait is released depends on how CUDA
feeds the two streams to the GPU:

  - A running wait kernel never blocks another stream's kernel, so a wait
    submitted first is released by a record submitted after it, whether or
    not the two streams share a hardware queue, as long as nothing else was
    submitted behind the wait on its own stream before the record.
  - Work submitted behind the wait on the wait's stream (the consumer that
    the wait guards) must wait for the wait to end.  When the two streams
    share one hardware queue (CUDA_DEVICE_MAX_CONNECTIONS=1, or more streams
    in use than queues), that dependent launch stalls the queue in front of
    the record, and the wait can only end by its timeout; the record then
    lands afterwards.
  - Under CUDA's lazy module loading (the default) the first launch of a
    kernel can wait for kernels already running: before the library loaded
    its notify kernels when the first notify is created, the very first
    record of a process, submitted behind a running wait, was held back
    until that wait's 1 s timeout.  The default-queue case below is the
    first record and the first wait of its process, so it checks that too.

Each case runs in a fresh process (the queue count is fixed when CUDA
starts), with a 1 s wait timeout, so nothing blocks for longer."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import json, sys, time
sys.path.insert(0, sys.argv[1])
import torch
import counted_notify_sync_gb300 as cns
torch.cuda.set_device(0)
out = {}
for follower in (0, 1):
    rc, n = cns.cntnotify_create(0)
    rc2, other = cns.cntnotify_create(0)
    assert rc == 0 and rc2 == 0
    s_wait, s_rec = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    assert cns.cntnotify_wait_with_timeout(n, s_wait, cns.CNS_WAIT_BIGGER_OR_EQUAL, 1, timeout=1, is_clear=1) == 0
    if follower:   # the consumer the wait guards, on the wait's stream
        assert cns.cntnotify_record(other, s_wait, cns.CNS_REC_ADD, 1) == 0
    assert cns.cntnotify_record(n, s_rec, cns.CNS_REC_ADD, 1) == 0
    torch.cuda.synchronize()
    dt = time.perf_counter() - t0
    _, status, count = cns.cntnotify_query_status(n)
    _, _, other_count = cns.cntnotify_query_status(other)
    out[str(follower)] = {"status": status, "count": count, "other": other_count, "seconds": dt}
    cns.cntnotify_destroy(n)
    cns.cntnotify_destroy(other)
print(json.dumps(out))
"""


def _run(connections):
    import counted_notify_sync_gb300 as cns
    cns.build()
    env = dict(os.environ)
    env.pop("CUDA_DEVICE_MAX_CONNECTIONS", None)
    if connections:
        env["CUDA_DEVICE_MAX_CONNECTIONS"] = str(connections)
    r = subprocess.run([sys.executable, "-c", SCRIPT, ROOT], capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stdout + r.stderr
    return json.loads(r.stdout.strip().splitlines()[-1])


def test_wait_submitted_before_its_record_with_library_defaults():
    """Default queues: released by the later record, with or without the
    guarded consumer behind the wait; the clear leaves 0."""
    res = _run(None)
    for follower in ("0", "1"):
        r = res[follower]
        assert r["status"] == 0 and r["count"] == 0, res
        assert r["seconds"] < 0.5, res
    assert res["1"]["other"] == 1


def test_wait_submitted_before_its_record_on_one_hardware_queue():
    """One hardware queue: without a consumer behind the wait the record still
    releases it; with one, the wait can only end by its timeout (sticky
    status TIMEOUT, nothing cleared) and the record lands after it."""
    res = _run(1)
    r0, r1 = res["0"], res["1"]
    assert r0["status"] == 0 and r0["count"] == 0, res
    assert r1["status"] == 5 and r1["count"] == 1 and r1["other"] == 1, res
    assert r1["seconds"] >= 0.9, res
