"""Counted notifies between devices (cntnotify_enable_peer; CntNotify API §1:
a counted notify also carries notifications between devices).  After the
enable, records, waits and resets on the notify run at system scope, on the
stream's own device.  On one GPU the peer is the notify's own device: the
same system-scope kernels run, and they are checked here against the hand
truth table and the oracle's rules.  With two or more GPUs a stream of device
1 records on, and waits on, a notify of device 0."""
import numpy as np
import pytest

import oracle
from tests.conftest import read_golden
from tests.gpu_helpers import load_user_kernels

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cns():
    import torch
    import counted_notify_sync_gb300 as c
    c.build()
    torch.cuda.set_device(0)
    return c


@pytest.fixture
def peer_notify(cns):
    """A notify of device 0 switched to system scope with device 0 as its peer."""
    rc, h = cns.cntnotify_create(0)
    assert rc == 0
    assert cns.cntnotify_enable_peer(h, 0) == 0
    yield h
    assert cns.cntnotify_destroy(h) == 0


def count_of(cns, h):
    import torch
    torch.cuda.synchronize()
    rc, st, c = cns.cntnotify_query_status(h)
    assert rc == 0
    return st, c


def test_enable_peer_argument_checks(cns):
    import torch
    rc, h = cns.cntnotify_create(0)
    assert rc == 0
    try:
        n = torch.cuda.device_count()
        assert cns.cntnotify_enable_peer(h, -1) == cns.CNS_ERR_INVALID_VALUE
        assert cns.cntnotify_enable_peer(h, n) == cns.CNS_ERR_INVALID_VALUE
        assert cns.cntnotify_enable_peer(h, 64) == cns.CNS_ERR_INVALID_VALUE
        assert cns.cntnotify_enable_peer(h, 0) == 0
        assert cns.cntnotify_enable_peer(h, 0) == 0   # again: nothing changes
    finally:
        cns.cntnotify_destroy(h)
    assert cns.cntnotify_enable_peer(h, 0) == cns.CNS_ERR_INVALID_HANDLE   # destroyed


def test_system_scope_record_truth_table(cns, peer_notify):
    rows = [r for r in read_golden("cntnotify_truth_table.txt") if r[0] == "record"]
    assert len(rows) >= 10
    for _, mode, c, v, want in rows:
        mode, c, v = int(mode, 0), int(c, 0), int(v, 0)
        assert cns.cntnotify_record(peer_notify, None, cns.CNS_REC_SET, c) == 0
        rc = cns.cntnotify_record(peer_notify, None, mode, v)
        if want == "invalid":
            assert rc == cns.CNS_ERR_INVALID_VALUE
            continue
        assert rc == 0
        st, got = count_of(cns, peer_notify)
        exp, ok = oracle.cnt_record(c, mode, v)
        assert ok and got == exp == int(want, 0) and st == 0


@pytest.mark.parametrize("clear", [0, 1])
def test_system_scope_wait_released_rows(cns, peer_notify, clear):
    rows = [r for r in read_golden("cntnotify_truth_table.txt") if r[0] == "wait" and r[4] == "1"]
    assert len(rows) >= 15
    for _, mode, c, v, _ in rows:
        mode, c, v = int(mode, 0), int(c, 0), int(v, 0)
        assert oracle.cnt_wait_satisfied(c, mode, v) == 1
        assert cns.cntnotify_record(peer_notify, None, cns.CNS_REC_SET, c) == 0
        assert cns.cntnotify_wait_with_timeout(peer_notify, None, mode, v, 5, clear) == 0
        st, got = count_of(cns, peer_notify)
        assert st == 0 and got == (0 if clear else c)


def test_system_scope_wait_times_out(cns, peer_notify):
    """A held row (LESS 0 never releases): the sticky status after the 1 s timeout, count untouched."""
    assert cns.cntnotify_record(peer_notify, None, cns.CNS_REC_SET, 7) == 0
    assert cns.cntnotify_wait_with_timeout(peer_notify, None, cns.CNS_WAIT_LESS, 0, 1, 1) == 0
    st, got = count_of(cns, peer_notify)
    assert st == cns.CNS_ERR_TIMEOUT and got == 7


def test_system_scope_reset_and_streams(cns, peer_notify):
    """Stream 1 writes a tensor and records ADD 1 three times; stream 2 waits >= 3 with clear, then copies
    the tensor: it sees stream 1's writes, and the count is cleared.  The records are submitted first."""
    import torch
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    x = torch.zeros(1 << 20, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    with torch.cuda.stream(s1):
        x.fill_(12345)
    for _ in range(3):
        assert cns.cntnotify_record(peer_notify, s1, cns.CNS_REC_ADD, 1) == 0
    assert cns.cntnotify_wait_with_timeout(peer_notify, s2, cns.CNS_WAIT_BIGGER_OR_EQUAL, 3, 5, 1) == 0
    with torch.cuda.stream(s2):
        y = x.clone()
    torch.cuda.synchronize()
    assert int((y == 12345).sum()) == y.numel()
    st, c = count_of(cns, peer_notify)
    assert st == 0 and c == 0
    assert cns.cntnotify_record(peer_notify, s1, cns.CNS_REC_SET, 99) == 0
    assert cns.cntnotify_reset(peer_notify, s1) == 0
    assert count_of(cns, peer_notify) == (0, 0)


CASES = [(c, m, v, clr) for c in (0, 1, 0xFFFFFFFF, 0x0F0F0F0F)
         for m in range(5) for v in (0, 1, 0xFFFFFFFF, 0x0000000F) for clr in (0, 1)]


def test_device_side_system_scope_record_and_wait(cns, peer_notify):
    """cns_cnt_record_sys_dev / cns_cnt_wait_sys_dev in user kernels: each (count, mode, value, isClear)
    releases exactly when the oracle's rule holds (else it runs out after 200 us), and clears only when
    released with isClear; 4096 system-scope ADD 1 records from user threads add up."""
    import torch
    user = load_user_kernels()
    rc, word = cns.cntnotify_get_device_ptr(peer_notify)
    assert rc == 0
    out = torch.zeros(2, dtype=torch.int32, device="cuda")
    for c, m, v, clr in CASES:
        assert user.user_record_sys(word, cns.CNS_REC_SET, c, 1, 1, 1) == 0
        assert user.user_wait_sys(word, m, v, clr, 200_000, out.data_ptr(), out.data_ptr() + 4) == 0
        got_rc, seen = out.cpu().numpy().view(np.uint32).tolist()
        sat = oracle.cnt_wait_satisfied(c, m, v)
        assert got_rc == (0 if sat else cns.CNS_ERR_TIMEOUT), (c, m, v, clr)
        _, now = count_of(cns, peer_notify)
        if sat:
            assert seen == c and now == (0 if clr else c), (c, m, v, clr)
        else:
            assert now == c
    assert user.user_record_sys(word, cns.CNS_REC_SET, 0, 1, 1, 1) == 0
    assert user.user_record_sys(word, cns.CNS_REC_ADD, 1, 64, 32, 2) == 0
    assert count_of(cns, peer_notify) == (0, 4096)
    for m in (-1, 5):
        assert user.user_wait_sys(word, m, 0, 0, 1000, out.data_ptr(), out.data_ptr() + 4) == 0
        assert int(out[0]) == cns.CNS_ERR_INVALID_VALUE


two_gpus = pytest.mark.skipif("__import__('torch').cuda.device_count() < 2", reason="needs two GPUs")


@two_gpus
def test_stream_of_another_device_needs_enable_peer(cns):
    import torch
    rc, h = cns.cntnotify_create(0)
    assert rc == 0
    try:
        s1 = torch.cuda.Stream(device=1)
        assert cns.cntnotify_record(h, s1, cns.CNS_REC_ADD, 1) == cns.CNS_ERR_NO_PEER_ACCESS
        assert cns.cntnotify_wait_with_timeout(h, s1, cns.CNS_WAIT_BIGGER_OR_EQUAL, 1, 1, 0) == \
            cns.CNS_ERR_NO_PEER_ACCESS
        assert cns.cntnotify_reset(h, s1) == cns.CNS_ERR_NO_PEER_ACCESS
    finally:
        cns.cntnotify_destroy(h)


@two_gpus
def test_record_on_device_1_wait_on_device_0(cns):
    """A stream of device 1 records ADD 1 on a notify of device 0 (through the peer mapping) and a stream of
    device 0 waits >= 1 with clear; then the other way round, device 1's stream waiting on device 0's count."""
    import torch
    rc, h = cns.cntnotify_create(0)
    assert rc == 0
    try:
        rc = cns.cntnotify_enable_peer(h, 1)
        if rc == cns.CNS_ERR_NO_PEER_ACCESS:
            pytest.skip("devices 0 and 1 have no peer access")
        assert rc == 0
        s1 = torch.cuda.Stream(device=1)
        s0 = torch.cuda.Stream(device=0)
        assert cns.cntnotify_record(h, s1, cns.CNS_REC_ADD, 1) == 0
        assert cns.cntnotify_wait_with_timeout(h, s0, cns.CNS_WAIT_BIGGER_OR_EQUAL, 1, 5, 1) == 0
        torch.cuda.synchronize(0)
        torch.cuda.synchronize(1)
        rc, st, c = cns.cntnotify_query_status(h)
        assert rc == 0 and st == 0 and c == 0
        assert cns.cntnotify_record(h, s0, cns.CNS_REC_SET, 5) == 0
        assert cns.cntnotify_wait_with_timeout(h, s1, cns.CNS_WAIT_EQUAL, 5, 5, 1) == 0
        torch.cuda.synchronize(0)
        torch.cuda.synchronize(1)
        rc, st, c = cns.cntnotify_query_status(h)
        assert rc == 0 and st == 0 and c == 0
    finally:
        cns.cntnotify_destroy(h)


@pytest.mark.parametrize("scope", [0, 1])
def test_notify_pingpong_probe(cns, scope):
    """The hand-off probe at gpu and system scope: every wait is released, and each count ends at iters."""
    import torch
    lines = torch.zeros(64, dtype=torch.int32, device="cuda")   # two 128-byte lines
    out = torch.zeros(4, dtype=torch.int64, device="cuda")
    assert lines.data_ptr() % 128 == 0
    assert cns.cns_probe_notify_pingpong(scope, 5000, lines, out) == 0
    torch.cuda.synchronize()
    o = out.cpu().numpy()
    assert o[1] == 0 and o[0] > 0
    lw = lines.cpu().numpy()
    assert lw[0] == 5000 and lw[32] == 5000
    assert cns.cns_probe_notify_pingpong(2, 10, lines, out) == cns.CNS_ERR_INVALID_VALUE
