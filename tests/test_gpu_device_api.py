"""The device-side API of include/cns_device.h inside user kernels
(tests/fused/user_kernels.cu, built here into a library of its own): the soft
barrier between ring rounds (one counter, die-local copies, and the
system-scope form for participants on several GPUs) against the sequential
oracle, over a subset of the grid and through the counter's wrap; records from user threads released
by the library's stream wait; device waits on every mode against the oracle's
rule; a grid-wide consumer on cns_cnt_wait_grid_dev against the oracle's
pipeline checksums; and bounded timeouts (a barrier one CTA never reaches, a
count nobody records, a grid-wide wait nobody releases)."""
import numpy as np
import pytest

import cns_inputs as ci
import oracle
from tests.gpu_helpers import from_dev_u32, load_user_kernels, to_dev_u32

pytestmark = pytest.mark.gpu

@pytest.fixture(scope="module")
def cns():
    import torch
    import counted_notify_sync_gb300 as c
    c.build()
    torch.cuda.set_device(0)
    return c


@pytest.fixture(scope="module")
def user(cns):
    return load_user_kernels()


# the three forms of the device-side soft barrier: one counter (cns_syncall_soft), die-local counter copies
# (cns_syncall_soft_die_local), and the system-scope form for participants on several GPUs
# (cns_syncall_soft_sys; one GPU here, the same arithmetic at system scope)
FORMS = {"counter": {}, "die_local": {"die_local": True}, "system_scope": {"sys": True}}


def _ring(cns, user, ctas, P, rounds, start=0, threads=256, short_cta=0xFFFFFFFF, timeout_ns=0, die_local=False,
          sys=False):
    import torch
    v0 = ci.ring_payload(ci.SEED_RING_ROTATE, P, 4)
    b0 = to_dev_u32(np.vstack([v0, np.zeros((ctas - P, 4), np.uint32)]))
    b1 = torch.zeros_like(b0)
    ws = cns.new_workspace(start_value=start, die_local=die_local)
    status = torch.full((ctas,), -1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    launch = user.user_ring_die_local if die_local else user.user_ring_sys if sys else user.user_ring
    rc = launch(ctas, threads, P, rounds, b0.data_ptr(), b1.data_ptr(), ws.data_ptr(), timeout_ns, short_cta,
                status.data_ptr())
    assert rc == 0, rc
    got = from_dev_u32(b0 if rounds % 2 == 0 else b1).reshape(ctas, 4)[:P]
    return v0, got, from_dev_u32(ws), status.cpu().numpy()


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("ctas,P,rounds,threads", [(148, 148, 10001, 256), (8, 8, 1000, 256), (111, 111, 777, 96),
                                                     (148, 64, 2001, 256), (5, 5, 3, 32), (1, 1, 10, 64)])
def test_fused_soft_barrier_ring_matches_oracle(cns, user, ctas, P, rounds, threads, form):
    die_local = form == "die_local"
    v0, got, ws, status = _ring(cns, user, ctas, P, rounds, threads=threads, **FORMS[form])
    want, fc, rc = oracle.syncall_run_ring(oracle.WL_RING_ROTATE, v0, rounds)
    assert rc == oracle.OK
    np.testing.assert_array_equal(got, want)
    assert int(ws[0]) == fc == (rounds * P) % oracle.counter_modulus(P)
    if die_local:
        assert int(ws[1024]) == fc   # the second copy counted every arrival too
    assert (status[:P] == 0).all() and (status[P:] == -1).all()   # CTAs past P never called it


@pytest.mark.parametrize("form", FORMS)
@pytest.mark.parametrize("P", [148, 111, 7])
def test_fused_soft_barrier_through_the_wrap(cns, user, P, form):
    M = oracle.counter_modulus(P)
    start = M - 5 * P
    v0, got, ws, status = _ring(cns, user, P, P, 12, start=start, **FORMS[form])
    want, fc, rc = oracle.syncall_run_ring(oracle.WL_RING_ROTATE, v0, 12, start=start)
    assert rc == oracle.OK
    np.testing.assert_array_equal(got, want)
    assert int(ws[0]) == fc == (start + 12 * P) % M
    assert (status == 0).all()


@pytest.mark.parametrize("form", FORMS)
def test_fused_soft_barrier_times_out_when_a_cta_stops_short(cns, user, form):
    """CTA 5 takes one barrier fewer: the others give up on the last barrier
    after their 20 ms limit, with CNS_ERR_TIMEOUT in every CTA and in the
    workspace's status line, and no CTA is left waiting."""
    P = 8
    v0, got, ws, status = _ring(cns, user, P, P, 4, short_cta=5, timeout_ns=20_000_000, **FORMS[form])
    line = ws[32:36]
    assert int(line[0]) == cns.CNS_ERR_TIMEOUT and int(line[1]) == 1 and int(line[3]) != 5
    assert status[5] == 0
    assert all(status[p] == cns.CNS_ERR_TIMEOUT for p in range(P) if p != 5)


def test_fused_records_released_by_the_library_wait(cns, user):
    import torch
    rc, h = cns.cntnotify_create(0)
    assert rc == 0
    try:
        rc, word = cns.cntnotify_get_device_ptr(h)
        assert rc == 0
        assert user.user_record(word, cns.CNS_REC_ADD, 1, 64, 32, 2) == 0   # 4096 records of ADD 1
        s = torch.cuda.Stream()
        assert cns.cntnotify_wait_with_timeout(h, s, cns.CNS_WAIT_BIGGER_OR_EQUAL, 4096, 5, 1) == 0
        s.synchronize()
        rc, st, c = cns.cntnotify_query_status(h)
        assert rc == 0 and st == 0 and c == 0   # released, then cleared
        assert user.user_record(word, cns.CNS_REC_SET, 0xDEADBEEF, 1, 1, 1) == 0
        assert user.user_record(word, cns.CNS_REC_BIT_AND, 0xFFFF0000, 1, 1, 1) == 0
        assert user.user_record(word, cns.CNS_REC_BIT_OR, 0x0000000F, 1, 1, 1) == 0
        assert user.user_record(word, 3, 0x12345678, 1, 1, 1) == 0   # no such mode: nothing happens
        rc, st, c = cns.cntnotify_query_status(h)
        assert c == ((0xDEADBEEF & 0xFFFF0000) | 0xF)
    finally:
        cns.cntnotify_destroy(h)


CASES = [(c, m, v, clr) for c in (0, 1, 5, 0xFFFFFFFF, 0x0F0F0F0F)
         for m in range(5) for v in (0, 1, 5, 0xFFFFFFFF, 0x0000000F) for clr in (0, 1)]


def test_fused_device_wait_follows_the_rules(cns, user):
    """Each (count, mode, value, isClear): the device wait releases exactly
    when the oracle's rule holds (else it runs out after 200 us), reports the
    count it saw, and clears only when released with isClear."""
    import torch
    rc, h = cns.cntnotify_create(0)
    assert rc == 0
    try:
        rc, word = cns.cntnotify_get_device_ptr(h)
        out = torch.zeros(2, dtype=torch.int32, device="cuda")
        for c, m, v, clr in CASES:
            assert user.user_record(word, cns.CNS_REC_SET, c, 1, 1, 1) == 0
            assert user.user_wait(word, m, v, clr, 200_000, out.data_ptr(), out.data_ptr() + 4) == 0
            got_rc, seen = out.cpu().numpy().view(np.uint32).tolist()
            sat = oracle.cnt_wait_satisfied(c, m, v)
            assert got_rc == (0 if sat else cns.CNS_ERR_TIMEOUT), (c, m, v, clr)
            rc, st, now = cns.cntnotify_query_status(h)
            if sat:
                assert seen == c
                assert now == (0 if clr else c), (c, m, v, clr)
            else:
                assert now == c
    finally:
        cns.cntnotify_destroy(h)


def test_fused_device_wait_rejects_unknown_modes(cns, user):
    import torch
    rc, h = cns.cntnotify_create(0)
    try:
        rc, word = cns.cntnotify_get_device_ptr(h)
        out = torch.zeros(2, dtype=torch.int32, device="cuda")
        for m in (-1, 5, 9):
            assert user.user_wait(word, m, 0, 0, 1000, out.data_ptr(), out.data_ptr() + 4) == 0
            assert int(out[0]) == cns.CNS_ERR_INVALID_VALUE
    finally:
        cns.cntnotify_destroy(h)


# --- the grid-wide wait (cns_cnt_wait_grid_dev) --------------------------------------------

def _lines(n=3):
    import torch
    return [torch.zeros(32, dtype=torch.int32, device="cuda") for _ in range(n)]


@pytest.mark.parametrize("G,threads,words,k,rounds", [(8, 128, 1024, 5, 40), (147, 256, 4096, 1, 20),
                                                       (1, 64, 100, 3, 10), (32, 96, 257, 64, 25)])
def test_grid_wait_consumer_rounds_match_oracle(cns, user, G, threads, words, k, rounds):
    """G consumer CTAs take a grid-wide wait (>= k, clear) per round and each sums the round's area; one
    producer CTA records k per round after the previous call was published: every CTA's sum equals the
    oracle's checksum of its round, each release saw exactly k, and the words end where the protocol
    leaves them."""
    import torch
    count, go, ack = _lines()
    area = torch.zeros(2 * words, dtype=torch.int32, device="cuda")
    sums = torch.zeros(rounds * G, dtype=torch.int32, device="cuda")
    rcs = torch.full((rounds * G,), -1, dtype=torch.int32, device="cuda")
    observed = torch.zeros(rounds, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    rc = user.user_grid_wait(G, threads, count.data_ptr(), go.data_ptr(), ack.data_ptr(), area.data_ptr(), words,
                             k, rounds, 0, sums.data_ptr(), rcs.data_ptr(), observed.data_ptr())
    assert rc == 0, rc
    assert (rcs.cpu().numpy() == 0).all()
    want_cs, _ = oracle.pipeline(1, words, rounds)
    got = from_dev_u32(sums).reshape(rounds, G)
    np.testing.assert_array_equal(got, np.repeat(want_cs[:, None], G, axis=1))
    assert (from_dev_u32(observed) == k).all()
    assert from_dev_u32(count)[0] == 0
    assert tuple(from_dev_u32(go)[:2]) == (rounds, 0)
    assert from_dev_u32(ack)[0] == rounds * G


def test_grid_wait_calls_continue_across_launches(cns, user):
    """A grid that follows another continues the call count: call 0 released by a count of 5 (>= 5, then
    cleared), call 1 by a count of 3 (== 3)."""
    import torch
    count, go, _ = _lines()
    rcs = torch.full((64,), -1, dtype=torch.int32, device="cuda")
    count[0] = 5
    torch.cuda.synchronize()
    assert user.user_grid_wait_only(64, count.data_ptr(), go.data_ptr(), 0, cns.CNS_WAIT_BIGGER_OR_EQUAL, 5,
                                    0, rcs.data_ptr()) == 0
    assert (rcs.cpu().numpy() == 0).all() and from_dev_u32(count)[0] == 0 and from_dev_u32(go)[0] == 1
    count[0] = 3
    rcs.fill_(-1)
    torch.cuda.synchronize()
    assert user.user_grid_wait_only(64, count.data_ptr(), go.data_ptr(), 1, cns.CNS_WAIT_EQUAL, 3, 0,
                                    rcs.data_ptr()) == 0
    assert (rcs.cpu().numpy() == 0).all() and from_dev_u32(count)[0] == 0 and from_dev_u32(go)[0] == 2


def test_grid_wait_times_out_everywhere(cns, user):
    """A count nobody records: CTA 0's wait runs out (2 ms), raises go[1], and every other CTA gives up
    with it; a later call on the same words returns the failure at once."""
    import torch
    count, go, _ = _lines()
    rcs = torch.full((16,), -1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    assert user.user_grid_wait_only(16, count.data_ptr(), go.data_ptr(), 0, cns.CNS_WAIT_BIGGER_OR_EQUAL, 1,
                                    2_000_000, rcs.data_ptr()) == 0
    assert (rcs.cpu().numpy() == cns.CNS_ERR_TIMEOUT).all()
    assert tuple(from_dev_u32(go)[:2]) == (0, cns.CNS_ERR_TIMEOUT)
    count[0] = 1
    rcs.fill_(-1)
    torch.cuda.synchronize()
    assert user.user_grid_wait_only(16, count.data_ptr(), go.data_ptr(), 0, cns.CNS_WAIT_BIGGER_OR_EQUAL, 1,
                                    2_000_000, rcs.data_ptr()) == 0
    assert (rcs.cpu().numpy() == cns.CNS_ERR_TIMEOUT).all() and from_dev_u32(count)[0] == 1


def test_grid_wait_rejects_a_bad_mode(cns, user):
    import torch
    count, go, _ = _lines()
    rcs = torch.full((4,), -1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    assert user.user_grid_wait_only(4, count.data_ptr(), go.data_ptr(), 0, 7, 1, 0, rcs.data_ptr()) == 0
    assert (rcs.cpu().numpy() == cns.CNS_ERR_INVALID_VALUE).all()
    assert tuple(from_dev_u32(go)[:2]) == (0, 0)
