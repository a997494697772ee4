"""CntNotify on the GPU against the CPU oracle: single records and waits from
the hand-built truth table, the op-stream state machine (bit-exact trace),
cross-stream waits, the two-stream counting pipeline and the timeout."""
import numpy as np
import pytest

import cns_inputs as ci
import oracle
from tests.conftest import read_golden
from tests.gpu_helpers import from_dev_u32, to_dev_u32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def cns():
    import torch
    import counted_notify_sync_gb300 as c
    c.build()
    torch.cuda.set_device(0)
    return c


@pytest.fixture
def notify(cns):
    rc, h = cns.cntnotify_create(0)
    assert rc == 0
    yield h
    assert cns.cntnotify_destroy(h) == 0


def count_of(cns, h):
    import torch
    torch.cuda.synchronize()
    rc, st, c = cns.cntnotify_query_status(h)
    assert rc == 0
    return st, c


def test_record_truth_table(cns, notify):
    rows = [r for r in read_golden("cntnotify_truth_table.txt") if r[0] == "record"]
    for _, mode, c, v, want in rows:
        mode, c, v = int(mode, 0), int(c, 0), int(v, 0)
        assert cns.cntnotify_record(notify, None, cns.CNS_REC_SET, c) == 0
        rc = cns.cntnotify_record(notify, None, mode, v)
        if want == "invalid":
            assert rc == cns.CNS_ERR_INVALID_VALUE
            continue
        assert rc == 0
        st, got = count_of(cns, notify)
        exp, ok = oracle.cnt_record(c, mode, v)
        assert ok and got == exp == int(want, 0) and st == 0


@pytest.mark.parametrize("clear", [0, 1])
def test_blocking_wait_released_rows(cns, notify, clear):
    """Every released row of the truth table: the wait returns, and clears if asked."""
    rows = [r for r in read_golden("cntnotify_truth_table.txt") if r[0] == "wait" and r[4] == "1"]
    assert len(rows) >= 15
    for _, mode, c, v, _ in rows:
        mode, c, v = int(mode, 0), int(c, 0), int(v, 0)
        assert oracle.cnt_wait_satisfied(c, mode, v) == 1
        assert cns.cntnotify_record(notify, None, cns.CNS_REC_SET, c) == 0
        assert cns.cntnotify_wait_with_timeout(notify, None, mode, v, 5, clear) == 0
        st, got = count_of(cns, notify)
        assert st == 0 and got == (0 if clear else c)


def test_invalid_wait_mode_rejected(cns, notify):
    assert cns.cntnotify_wait_with_timeout(notify, None, 5, 0, 1, 0) == cns.CNS_ERR_INVALID_VALUE
    assert cns.cntnotify_wait_with_timeout(notify, None, info=None) == cns.CNS_ERR_NULL_PTR
    assert cns.cntnotify_record(notify, None, info=None) == cns.CNS_ERR_NULL_PTR
    assert cns.cntnotify_get_id(notify, out=False)[0] == cns.CNS_ERR_NULL_PTR


def test_usage_example_two_streams(cns, notify):
    """Stream 2 waits for count >= 1 (timeout 10 s, clear); stream 1 records ADD 1."""
    import torch
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    # the record is submitted first: the streams may share one hardware queue
    assert cns.cntnotify_record(notify, s1, cns.CNS_REC_ADD, 1) == 0
    assert cns.cntnotify_wait_with_timeout(notify, s2, cns.CNS_WAIT_BIGGER_OR_EQUAL, 1, 10, 1) == 0
    s1.synchronize()
    s2.synchronize()
    st, c = count_of(cns, notify)
    assert st == 0 and c == 0
    rc, nid = cns.cntnotify_get_id(notify)
    assert rc == 0
    assert cns.cntnotify_reset(notify, s2) == 0


def test_n_producer_streams_fan_in(cns, notify):
    """N producer streams each ADD 1; the waiter uses BIGGER_OR_EQUAL N."""
    import torch
    n = 6
    waiter = torch.cuda.Stream()
    prods = [torch.cuda.Stream() for _ in range(n)]
    for s in prods:
        assert cns.cntnotify_record(notify, s, cns.CNS_REC_ADD, 1) == 0
    assert cns.cntnotify_wait_with_timeout(notify, waiter, cns.CNS_WAIT_BIGGER_OR_EQUAL, n, 10, 0) == 0
    torch.cuda.synchronize()
    st, c = count_of(cns, notify)
    assert st == 0 and c == n


def test_bitmask_multi_signal(cns, notify):
    import torch
    waiter = torch.cuda.Stream()
    bits = [1 << k for k in (0, 3, 9, 31)]
    mask = sum(bits)
    streams = [torch.cuda.Stream() for _ in bits]
    for b, s in zip(bits, streams):
        assert cns.cntnotify_record(notify, s, cns.CNS_REC_BIT_OR, b) == 0
    assert cns.cntnotify_wait_with_timeout(notify, waiter, cns.CNS_WAIT_EQUAL_WITH_BITMASK, mask, 10, 1) == 0
    torch.cuda.synchronize()
    st, c = count_of(cns, notify)
    assert st == 0 and c == 0


def test_wait_timeout_sets_sticky_status(cns, notify):
    """LESS 0 can never be released (the unit-test WaitInfo of the API page)."""
    import time
    t0 = time.time()
    assert cns.cntnotify_wait_with_timeout(notify, None, cns.CNS_WAIT_LESS, 0, 1, 1) == 0
    st, c = count_of(cns, notify)
    assert st == cns.CNS_ERR_TIMEOUT and c == 0
    assert 0.9 < time.time() - t0 < 10
    # the stream and the device keep working
    assert cns.cntnotify_record(notify, None, cns.CNS_REC_ADD, 5) == 0
    assert count_of(cns, notify)[1] == 5


def test_ids_unique_and_destroy_invalidates(cns):
    hs = []
    for _ in range(20):
        rc, h = cns.cntnotify_create(0)
        assert rc == 0
        hs.append(h)
    ids = [cns.cntnotify_get_id(h)[1] for h in hs]
    assert len(set(ids)) == 20
    h = hs.pop()
    assert cns.cntnotify_destroy(h) == 0
    assert cns.cntnotify_destroy(h) == cns.CNS_ERR_INVALID_HANDLE
    assert cns.cntnotify_record(h, None, cns.CNS_REC_ADD, 1) == cns.CNS_ERR_INVALID_HANDLE
    for h in hs:
        assert cns.cntnotify_destroy(h) == 0


def test_pool_exhaustion_and_recovery(cns):
    hs = []
    while True:
        rc, h = cns.cntnotify_create(0)
        if rc != 0:
            break
        hs.append(h)
        assert len(hs) <= 1 << 20
    assert rc == cns.CNS_ERR_RESOURCE and len(hs) >= 1
    assert cns.cntnotify_destroy(hs.pop()) == 0
    rc, h = cns.cntnotify_create(0)
    assert rc == 0
    st, c = count_of(cns, h)        # a reused slot starts clean
    assert st == 0 and c == 0
    hs.append(h)
    for h in hs:
        assert cns.cntnotify_destroy(h) == 0


# --- op-stream state machine ---------------------------------------------------------------

def run_sm(cns, ops, init):
    import torch
    n = ops.shape[0]
    dev = to_dev_u32(ops) if n else torch.empty((0, 4), dtype=torch.int32, device="cuda")
    trace, final = cns.run_statemachine(dev, init)
    return (from_dev_u32(trace) if n else np.zeros((0, 2), np.uint32)), int(from_dev_u32(final)[0])


def test_statemachine_1e6_ops_bit_exact(cns):
    ops = ci.notify_ops(1_000_000)
    got_t, got_f = run_sm(cns, ops, 0)
    want_t, want_f = oracle.cnt_statemachine(ops, 0)
    np.testing.assert_array_equal(got_t, want_t)
    assert got_f == want_f


def test_statemachine_hand_sequence(cns):
    rows = read_golden("cntnotify_sequence.txt")
    ops = np.array([[int(k, 0), int(m, 0), int(v, 0), int(c, 0)] for k, m, v, c, _, _, _ in rows], dtype=np.uint32)
    got_t, got_f = run_sm(cns, ops, 0)
    want = np.array([[int(a, 0), int(o)] for *_, a, o in rows], dtype=np.uint32)
    np.testing.assert_array_equal(got_t, want)


@pytest.mark.parametrize("n", [0, 1, 15, 16, 17, 33, 4097])
def test_statemachine_ragged_lengths(cns, n):
    ops = ci.notify_ops(n, seed=1000 + n)
    got_t, got_f = run_sm(cns, ops, 0xDEAD)
    want_t, want_f = oracle.cnt_statemachine(ops, 0xDEAD)
    np.testing.assert_array_equal(got_t, want_t)
    assert got_f == want_f


def test_statemachine_without_any_set(cns):
    """No SET record at all: the stream is cut only where other ops fix the
    count (an AND that leaves few unknown bits, an OR that sets them, a
    clearing wait decided by the known bits)."""
    ops = ci.notify_ops(50_000, seed=77)
    ops = ops[~((ops[:, 0] == 0) & (ops[:, 1] == 0))]
    got_t, got_f = run_sm(cns, ops, 3)
    want_t, want_f = oracle.cnt_statemachine(ops, 3)
    np.testing.assert_array_equal(got_t, want_t)
    assert got_f == want_f


@pytest.mark.parametrize("n", [5_000, 200_000])
def test_statemachine_one_chain(cns, n):
    """No op ever fixes the count: one dependent chain through every tile."""
    ops = _chain_ops(n, 31)
    got_t, got_f = run_sm(cns, ops, 0xFFFFFFF0)
    want_t, want_f = oracle.cnt_statemachine(ops, 0xFFFFFFF0)
    np.testing.assert_array_equal(got_t, want_t)
    assert got_f == want_f


def _near_fixing_ops(n, seed):
    """Ops that fix, or nearly fix, the count in every way the known-bits
    walk looks at: ANDs with sparse masks and ORs with dense ones (bits fixed
    outright), adds whose carries run through known and unknown bits (small,
    all-ones, one below a power of two, random), and waits whose compare mask
    covers few bits (the bitmask mode, decided early) that clear half the
    time -- with no SET record."""
    ops = ci.notify_ops(n, seed=seed)
    r = ci.splitmix64(seed ^ 0x0F1C5ED, 3 * n).reshape(n, 3)
    lo32 = np.uint64(0xFFFFFFFF)
    rnd = (r[:, 0] & lo32).astype(np.uint32)
    sparse = (rnd & (r[:, 1] >> np.uint64(32)).astype(np.uint32) & (r[:, 2] & lo32).astype(np.uint32))
    dense = rnd | (r[:, 1] & lo32).astype(np.uint32) | (r[:, 2] >> np.uint64(32)).astype(np.uint32)
    pick = (r[:, 0] >> np.uint64(60)).astype(np.int64)          # 0..15
    k = ((r[:, 1] >> np.uint64(27)) & np.uint64(31)).astype(np.uint32)
    below_pow2 = (np.left_shift(np.uint32(1), k, dtype=np.uint32) - np.uint32(1)).astype(np.uint32)
    rec = ops[:, 0] == 0
    mode = np.select([pick < 5, pick < 9, pick < 15], [4, 2, 1], 1).astype(np.uint32)   # AND, OR, ADD
    val = np.select([pick < 5, pick < 9, pick < 11, pick < 13, pick < 14],
                    [sparse, dense, rnd & np.uint32(15), below_pow2, np.uint32(0xFFFFFFFF)], rnd).astype(np.uint32)
    ops[rec, 1] = mode[rec]
    ops[rec, 2] = val[rec]
    wait = ~rec
    bitmask = wait & (pick < 8)
    ops[bitmask, 1] = 4                                            # EQUAL_WITH_BITMASK
    ops[bitmask, 2] = np.where(pick[bitmask] < 4, sparse[bitmask], rnd[bitmask] & np.uint32(7))
    ops[wait, 3] = (pick[wait] & 1).astype(np.uint32)
    return ops


@pytest.mark.parametrize("n,seed", [(3_000, 1), (70_001, 2), (1_000_000, 3)])
def test_statemachine_near_fixing_ops(cns, n, seed):
    """The known-bits cut on ops chosen to sit at its edges (no SET record):
    bit for bit against the sequential oracle."""
    ops = _near_fixing_ops(n, seed)
    assert not ((ops[:, 0] == 0) & (ops[:, 1] == 0)).any()
    got_t, got_f = run_sm(cns, ops, 0x80000001)
    want_t, want_f = oracle.cnt_statemachine(ops, 0x80000001)
    np.testing.assert_array_equal(got_t, want_t)
    assert got_f == want_f


def test_statemachine_fixing_ops_by_hand(cns):
    """Short hand-made streams where a known count is reached without a SET,
    each after a different count: an AND then an OR; an AND, an add whose
    carry stops in known bits, then an OR; a bitmask wait decided by one
    known bit that releases and clears (outcome RELEASED, count 0); and the
    same wait undecided (the count stays unknown)."""
    AND, OR, ADD = 4, 2, 1
    WAIT, EQB = 1, 4
    pad = [[WAIT, 3, 0, 0]] * 9          # waits that fix nothing, to move the ops across chunks
    streams = [
        [[0, AND, 0x3, 0], [0, OR, 0x3, 0]],
        [[0, AND, 0xF0, 0], [0, ADD, 5, 0], [0, OR, 0xF0, 0], [0, ADD, 0xFFFFFFFF, 0]],
        [[0, OR, 1, 0], [WAIT, EQB, 1, 1], [0, ADD, 7, 0]],
        [[0, ADD, 1, 0], [WAIT, EQB, 1, 1], [0, ADD, 7, 0]],
    ]
    for init in (0, 6, 0xFFFFFFFF):
        for st in streams:
            for lead in (0, 3, 7, 8, 15):
                ops = np.array(pad[:lead] + st + pad[:5], dtype=np.uint32).reshape(-1, 4)
                got_t, got_f = run_sm(cns, ops, init)
                want_t, want_f = oracle.cnt_statemachine(ops, init)
                np.testing.assert_array_equal(got_t, want_t)
                assert got_f == want_f


def _fused_limit():
    """Op count that gives every resident CTA exactly one 4096-op tile: 2 CTAs per SM."""
    import torch
    return torch.cuda.get_device_properties(0).multi_processor_count * 2 * 4096


@pytest.mark.parametrize("where", ["at_limit", "over_limit", "three_million"])
def test_statemachine_one_and_several_tiles_per_cta(cns, where):
    """Streams with exactly one 4096-op tile per resident CTA, one tile more
    (a CTA takes a second tile, waiting on a tile of the previous wave), and
    3e6 ops (several waves), bit for bit."""
    lim = _fused_limit()
    n = {"at_limit": lim, "over_limit": lim + 1, "three_million": 3_000_000}[where]
    ops = ci.notify_ops(n, seed=n % 1000)
    got_t, got_f = run_sm(cns, ops, 7)
    want_t, want_f = oracle.cnt_statemachine(ops, 7)
    np.testing.assert_array_equal(got_t, want_t)
    assert got_f == want_f


@pytest.mark.parametrize("n", [17, 1000, 4863, 5000, 100_003, 999_999])
def test_statemachine_spread_over_all_ctas(cns, n):
    """Streams shorter than one 4096-op tile per resident CTA are cut into
    tiles of ceil(n / CTAs) ops (a multiple of 8, at least 16): small tiles,
    tiles that do not divide n, many tiles without a SET; bit for bit."""
    ops = ci.notify_ops(n, seed=n % 997)
    got_t, got_f = run_sm(cns, ops, 5)
    want_t, want_f = oracle.cnt_statemachine(ops, 5)
    np.testing.assert_array_equal(got_t, want_t)
    assert got_f == want_f


def _chain_ops(n, seed):
    """Ops that never fix the count: every record an ADD, no clearing wait (an
    add of a constant to a count with unknown bits leaves them unknown, and a
    wait that does not clear changes nothing)."""
    ops = ci.notify_ops(n, seed=seed)
    ops[ops[:, 0] == 0, 1] = 1
    ops[:, 3] = 0
    return ops


@pytest.mark.parametrize("gap", [1000, 9000, 70000])
def test_statemachine_rare_sets(cns, gap):
    """SET records only every `gap` ops, and no other op that fixes the count:
    chains cross many CTAs (each tile without a SET waits for the one before
    it and replays all its ops)."""
    ops = _chain_ops(400_000, gap)
    ops[::gap, 0] = 0                                    # a SET every `gap` ops
    ops[::gap, 1] = 0
    got_t, got_f = run_sm(cns, ops, 11)
    want_t, want_f = oracle.cnt_statemachine(ops, 11)
    np.testing.assert_array_equal(got_t, want_t)
    assert got_f == want_f


def test_statemachine_back_to_back_calls_reuse_scratch(cns):
    """Consecutive calls on one scratch buffer: the one-pass kernel's link
    words from the earlier call must not be taken by the later one."""
    import torch
    n = 200_000
    scratch = torch.empty(cns.cns_statemachine_scratch_bytes(n) // 4 + 2, dtype=torch.int32, device="cuda")
    for seed in (1, 2, 3):
        ops = ci.notify_ops(n, seed=seed)
        ops_d = to_dev_u32(ops)
        trace = torch.empty((n, 2), dtype=torch.int32, device="cuda")
        final = torch.empty(1, dtype=torch.int32, device="cuda")
        rc = cns._native.lib().cns_statemachine_run(ops_d.data_ptr(), n, seed, trace.data_ptr(), final.data_ptr(),
                                                    scratch.data_ptr(), scratch.numel() * 4, None)
        assert rc == 0
        torch.cuda.synchronize()
        want_t, want_f = oracle.cnt_statemachine(ops, seed)
        np.testing.assert_array_equal(trace.cpu().numpy().view(np.uint32), want_t)
        assert int(final.cpu().numpy().view(np.uint32)[0]) == want_f


@pytest.mark.parametrize("n,kind", [(200_000, "bench"), (1_300_000, "bench"), (300_000, "chain")])
def test_statemachine_replayed_from_a_cuda_graph(cns, n, kind):
    """The call captured once into a CUDA graph and replayed with new ops in the same buffer each time:
    every replay bit for bit against the oracle.  A replay repeats the captured call's link tag, so a
    link word left by the previous replay must never be taken (streams with one tile per CTA, several
    waves of tiles, and one long chain through every tile)."""
    import torch
    streams = [(_chain_ops(n, s) if kind == "chain" else ci.notify_ops(n, seed=s)) for s in (41, 42, 43)]
    d = to_dev_u32(streams[0])
    trace = torch.empty((n, 2), dtype=torch.int32, device="cuda")
    final = torch.empty(1, dtype=torch.int32, device="cuda")
    sb = cns.cns_statemachine_scratch_bytes(n)
    scratch = torch.empty(sb, dtype=torch.uint8, device="cuda")
    side = torch.cuda.Stream()

    def call():
        cns.check(cns.cns_statemachine_run(d, n, 9, trace, final, scratch, sb, torch.cuda.current_stream()),
                  "statemachine")
    with torch.cuda.stream(side):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        call()
    for ops in (streams[1], streams[2], streams[0], streams[1]):
        d.copy_(to_dev_u32(ops))
        g.replay()
        torch.cuda.synchronize()
        want_t, want_f = oracle.cnt_statemachine(ops, 9)
        np.testing.assert_array_equal(from_dev_u32(trace), want_t)
        assert int(from_dev_u32(final)[0]) == want_f


def test_statemachine_noalloc_replayed_from_a_cuda_graph(cns):
    """The allocation-free entry point, captured into a CUDA graph and replayed with new ops."""
    import torch
    n = 250_000
    streams = [ci.notify_ops(n, seed=s) for s in (51, 52)]
    d = to_dev_u32(streams[0])
    trace = torch.empty((n, 2), dtype=torch.int32, device="cuda")
    final = torch.empty(1, dtype=torch.int32, device="cuda")
    L = cns._native.lib()
    side = torch.cuda.Stream()

    def call():
        rc = L.cns_statemachine_run_noalloc(d.data_ptr(), n, 3, trace.data_ptr(), final.data_ptr(),
                                            torch.cuda.current_stream().cuda_stream)
        assert rc == cns.CNS_SUCCESS
    with torch.cuda.stream(side):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        call()
    for ops in (streams[1], streams[0], streams[1]):
        d.copy_(to_dev_u32(ops))
        g.replay()
        torch.cuda.synchronize()
        want_t, want_f = oracle.cnt_statemachine(ops, 3)
        np.testing.assert_array_equal(from_dev_u32(trace), want_t)
        assert int(from_dev_u32(final)[0]) == want_f


def test_statemachine_all_sets_and_invalid_ops(cns):
    ops = ci.notify_ops(3000, seed=5)
    ops[::2, 0] = 0
    ops[::2, 1] = 0
    ops[1::7, 1] = 3          # record mode 3 / wait mode 3
    ops[5::11, 0] = 2         # undefined kind
    ops[6::13, 0] = 1
    ops[6::13, 1] = 9         # undefined wait mode
    got_t, got_f = run_sm(cns, ops, 1)
    want_t, want_f = oracle.cnt_statemachine(ops, 1)
    np.testing.assert_array_equal(got_t, want_t)
    assert got_f == want_f


# --- two-stream counting pipeline --------------------------------------------------------

@pytest.mark.parametrize("consumer_wait", [0, 1])
@pytest.mark.parametrize("areas", [1, 2])
def test_pipeline_4096_tiles_1000_rounds(cns, areas, consumer_wait):
    import torch
    rc, done = cns.cntnotify_create(0)
    rc2, ack = cns.cntnotify_create(0)
    assert rc == rc2 == 0
    try:
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        cfg, rc, checksums, released = cns.run_pipeline(done, ack, 4096, 256, 1000, s1, s2, timeout_s=10,
                                                        areas=areas, consumer_wait=consumer_wait)
        assert rc == 0 and cfg.device_status == 0
        want_cs, want_rel = oracle.pipeline(4096, 256, 1000)
        np.testing.assert_array_equal(from_dev_u32(checksums), want_cs)
        np.testing.assert_array_equal(from_dev_u32(released), want_rel)
        assert cfg.consumer_ctas > 0
        assert count_of(cns, done) == (0, 0) and count_of(cns, ack) == (0, 1000 * cfg.consumer_ctas)
        assert cfg.elapsed_ms > 0 and 0 < cfg.producer_ms <= cfg.elapsed_ms
    finally:
        cns.cntnotify_destroy(done)
        cns.cntnotify_destroy(ack)


@pytest.mark.parametrize("consumer_wait", [0, 1])
@pytest.mark.parametrize("areas", [1, 2])
def test_pipeline_replayed_from_a_cuda_graph(cns, areas, consumer_wait):
    """cns_pipeline_run (sync = 0) captured once into a CUDA graph, the consumer stream joined into the
    capture, and replayed: every replay's checksums and release counts against the oracle, both notifies
    back at their end counts, no timeout."""
    import torch
    rc, done = cns.cntnotify_create(0)
    rc2, ack = cns.cntnotify_create(0)
    assert rc == rc2 == 0
    try:
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        tiles, words, rounds = 4096, 64, 300
        bufs = (torch.empty(areas * tiles * words, dtype=torch.int32, device="cuda"),
                torch.empty(rounds, dtype=torch.int32, device="cuda"),
                torch.empty(rounds, dtype=torch.int32, device="cuda"))
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s1):
            cfg, rc, _, _ = cns.run_pipeline(done, ack, tiles, words, rounds, s1, s2, timeout_s=10, sync=False,
                                             buffers=bufs, areas=areas, consumer_wait=consumer_wait)
        assert rc == 0
        want_cs, want_rel = oracle.pipeline(tiles, words, rounds)
        for _ in range(3):
            bufs[1].zero_()
            bufs[2].zero_()
            g.replay()
            torch.cuda.synchronize()
            np.testing.assert_array_equal(from_dev_u32(bufs[1]), want_cs)
            np.testing.assert_array_equal(from_dev_u32(bufs[2]), want_rel)
            assert count_of(cns, done) == (0, 0)
            assert count_of(cns, ack) == (0, (rounds * cfg.consumer_ctas) % (1 << 32))
    finally:
        cns.cntnotify_destroy(done)
        cns.cntnotify_destroy(ack)


@pytest.mark.parametrize("consumer_wait", [0, 1])
@pytest.mark.parametrize("areas", [0, 1, 2])
def test_pipeline_small_odd_shapes(cns, areas, consumer_wait):
    import torch
    rc, done = cns.cntnotify_create(0)
    rc2, ack = cns.cntnotify_create(0)
    try:
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        cfg, rc, checksums, released = cns.run_pipeline(done, ack, 7, 12, 5, s1, s2, timeout_s=10,
                                                        producer_ctas=3, areas=areas, consumer_wait=consumer_wait)
        assert rc == 0
        want_cs, want_rel = oracle.pipeline(7, 12, 5)
        np.testing.assert_array_equal(from_dev_u32(checksums), want_cs)
        np.testing.assert_array_equal(from_dev_u32(released), want_rel)
    finally:
        cns.cntnotify_destroy(done)
        cns.cntnotify_destroy(ack)


@pytest.mark.parametrize("tiles,tile_words,rounds,producer_ctas", [
    (4096, 256, 20, 1),        # one CTA records all 4096 tiles, 32 lanes at a time
    (4096, 256, 20, 33),       # 124 or 125 tiles per CTA: a ragged last group of lanes
    (4096, 256, 20, 100000),   # more CTAs than the cap and than tiles
    (1000, 4, 30, 0),          # one uint4 per tile
    (40, 8192, 6, 0),          # large tiles, 2048 uint4 each
    (1, 4, 3, 0),              # one tile
])
@pytest.mark.parametrize("consumer_wait", [0, 1])
@pytest.mark.parametrize("areas", [1, 2])
def test_pipeline_producer_grids(cns, tiles, tile_words, rounds, producer_ctas, areas, consumer_wait):
    import torch
    rc, done = cns.cntnotify_create(0)
    rc2, ack = cns.cntnotify_create(0)
    try:
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        cfg, rc, checksums, released = cns.run_pipeline(done, ack, tiles, tile_words, rounds, s1, s2, timeout_s=10,
                                                        producer_ctas=producer_ctas, areas=areas,
                                                        consumer_wait=consumer_wait)
        assert rc == 0 and cfg.device_status == 0
        want_cs, want_rel = oracle.pipeline(tiles, tile_words, rounds)
        np.testing.assert_array_equal(from_dev_u32(checksums), want_cs)
        np.testing.assert_array_equal(from_dev_u32(released), want_rel)
        assert count_of(cns, done) == (0, 0) and count_of(cns, ack) == (0, rounds * cfg.consumer_ctas)
    finally:
        cns.cntnotify_destroy(done)
        cns.cntnotify_destroy(ack)


# --- probes ------------------------------------------------------------------------------------

def test_probes_return_plausible_times(cns):
    import torch
    line = torch.zeros(32, dtype=torch.int32, device="cuda")
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    for kind in (0, 1, 2):
        assert cns.cns_probe_atomic_rtt(kind, sms, sms // 2, 200, line, out) == 0
        torch.cuda.synchronize()
        ns, sm = out.tolist()
        assert 200 * 50 < ns < 200 * 20000 and 0 <= sm < sms
    word = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert cns.cns_probe_same_address_throughput(sms, 256, 10, word) == 0
    torch.cuda.synchronize()
    assert int(word.item()) == sms * 256 * 10


def test_grid_sync_probe_ring_rotate(cns):
    import torch
    v0 = ci.ring_payload(ci.SEED_RING_ROTATE, 148, 4)
    b0 = to_dev_u32(v0)
    b1 = torch.zeros_like(b0)
    assert cns.cns_probe_grid_sync(148, 256, 1001, b0, b1) == 0
    torch.cuda.synchronize()
    np.testing.assert_array_equal(from_dev_u32(b1).reshape(148, 4), np.roll(v0, -1001, axis=0))


@pytest.mark.parametrize("consumer_wait", [0, 1])
@pytest.mark.parametrize("areas", [1, 2])
def test_pipeline_on_one_stream(cns, areas, consumer_wait):
    """Producer and consumer on the same stream: every device wait is then
    already satisfied when it starts, and the result is the same."""
    import torch
    rc, done = cns.cntnotify_create(0)
    rc2, ack = cns.cntnotify_create(0)
    try:
        s = torch.cuda.Stream()
        cfg, rc, checksums, released = cns.run_pipeline(done, ack, 300, 64, 12, s, s, timeout_s=10, areas=areas,
                                                        consumer_wait=consumer_wait)
        assert rc == 0 and cfg.device_status == 0
        want_cs, want_rel = oracle.pipeline(300, 64, 12)
        np.testing.assert_array_equal(from_dev_u32(checksums), want_cs)
        np.testing.assert_array_equal(from_dev_u32(released), want_rel)
    finally:
        cns.cntnotify_destroy(done)
        cns.cntnotify_destroy(ack)


@pytest.mark.parametrize("consumer_wait", [0, 1])
@pytest.mark.parametrize("rounds", [1, 2, 7, 8])
def test_pipeline_two_areas_hold_the_last_two_rounds(cns, rounds, consumer_wait):
    """With two areas, round r writes area r % 2: after the run the area of the
    last round holds its words and the other area those of the round before
    (or is untouched after a single round)."""
    import torch
    tiles, words = 96, 16
    rc, done = cns.cntnotify_create(0)
    rc2, ack = cns.cntnotify_create(0)
    try:
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        buf = torch.full((2 * tiles * words,), 0x5A5A5A5A, dtype=torch.int32, device="cuda")
        cs = torch.empty(rounds, dtype=torch.int32, device="cuda")
        rel = torch.empty(rounds, dtype=torch.int32, device="cuda")
        cfg, rc, checksums, released = cns.run_pipeline(done, ack, tiles, words, rounds, s1, s2, timeout_s=10,
                                                        buffers=(buf, cs, rel), areas=2, consumer_wait=consumer_wait)
        assert rc == 0 and cfg.device_status == 0
        got = from_dev_u32(buf).reshape(2, tiles * words)
        w = np.arange(tiles * words, dtype=np.uint64)
        for r in (rounds - 1, rounds - 2):
            if r >= 0:
                want = np.array([oracle.pipeline_word(int(x), r) for x in w], dtype=np.uint32)
                np.testing.assert_array_equal(got[r % 2], want)
        if rounds == 1:
            assert (got[1] == 0x5A5A5A5A).all()
        want_cs, want_rel = oracle.pipeline(tiles, words, rounds)
        np.testing.assert_array_equal(from_dev_u32(checksums), want_cs)
        np.testing.assert_array_equal(from_dev_u32(released), want_rel)
    finally:
        cns.cntnotify_destroy(done)
        cns.cntnotify_destroy(ack)


def test_pipeline_rejects_bad_area_count(cns):
    import torch
    rc, done = cns.cntnotify_create(0)
    rc2, ack = cns.cntnotify_create(0)
    try:
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        for areas in (-1, 3):
            cfg, rc, _, _ = cns.run_pipeline(done, ack, 8, 4, 2, s1, s2, timeout_s=10, areas=areas)
            assert rc == cns.CNS_ERR_INVALID_VALUE
        for cw in (-1, 2):
            cfg, rc, _, _ = cns.run_pipeline(done, ack, 8, 4, 2, s1, s2, timeout_s=10, areas=2, consumer_wait=cw)
            assert rc == cns.CNS_ERR_INVALID_VALUE
    finally:
        cns.cntnotify_destroy(done)
        cns.cntnotify_destroy(ack)


def _pipeline_configs(n, seed=77):
    rng = np.random.RandomState(seed)
    out = []
    for i in range(n):
        words = 4 * int(rng.randint(1, 2049))                       # 4 .. 8192
        tiles = int(rng.randint(1, max(2, min(6000, (1 << 22) // words))))
        out.append(dict(tiles=tiles, words=words, rounds=int(rng.randint(1, 61)),
                        pctas=int(rng.choice([0, 1, 7, 100, 1000])), areas=int(rng.choice([1, 2])),
                        one_stream=bool(rng.rand() < 0.25), consumer_wait=i % 2))
    return out


@pytest.mark.parametrize("c", _pipeline_configs(24),
                         ids=lambda c: f"t{c['tiles']}w{c['words']}r{c['rounds']}p{c['pctas']}a{c['areas']}"
                                       f"{'s' if c['one_stream'] else 'm'}{'k' if c['consumer_wait'] else ''}")
def test_pipeline_random_configs(cns, c):
    """Seeded random pipelines (tile count, tile size, rounds, producer grid, one or two areas, one or two
    streams, the wait on the stream or in the consumer kernel): every round's checksum and release count equal the oracle's, and the notifies end where
    the protocol leaves them."""
    import torch
    rc, done = cns.cntnotify_create(0)
    rc2, ack = cns.cntnotify_create(0)
    assert rc == rc2 == 0
    try:
        s1 = torch.cuda.Stream()
        s2 = s1 if c["one_stream"] else torch.cuda.Stream()
        cfg, rc, checksums, released = cns.run_pipeline(done, ack, c["tiles"], c["words"], c["rounds"], s1, s2,
                                                        timeout_s=10, producer_ctas=c["pctas"], areas=c["areas"],
                                                        consumer_wait=c["consumer_wait"])
        assert rc == 0 and cfg.device_status == 0
        want_cs, want_rel = oracle.pipeline(c["tiles"], c["words"], c["rounds"])
        np.testing.assert_array_equal(from_dev_u32(checksums), want_cs)
        np.testing.assert_array_equal(from_dev_u32(released), want_rel)
        assert count_of(cns, done) == (0, 0)
        assert count_of(cns, ack) == (0, (c["rounds"] * cfg.consumer_ctas) % (1 << 32))
    finally:
        cns.cntnotify_destroy(done)
        cns.cntnotify_destroy(ack)


@pytest.mark.parametrize("consumer_wait", [0, 1])
@pytest.mark.parametrize("areas", [1, 2])
def test_pipeline_without_released_array(cns, areas, consumer_wait):
    """released_dev is optional: through the C ABI with it NULL, unsynchronised (sync = 0), the
    checksums still match the oracle and the notifies end where the protocol leaves them."""
    import torch
    from counted_notify_sync_gb300 import _native
    rc, done = cns.cntnotify_create(0)
    rc2, ack = cns.cntnotify_create(0)
    try:
        s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
        tiles, words, rounds = 500, 32, 9
        buf = torch.empty(2 * tiles * words, dtype=torch.int32, device="cuda")
        cs = torch.empty(rounds, dtype=torch.int32, device="cuda")
        cfg = _native.Pipeline()
        cfg.done, cfg.ack = done, ack
        cfg.tiles_dev, cfg.checksums_dev, cfg.released_dev = _native.ptr(buf), _native.ptr(cs), None
        cfg.tiles, cfg.tile_words, cfg.rounds = tiles, words, rounds
        cfg.producer_stream = _native.stream_handle(s1)
        cfg.consumer_stream = _native.stream_handle(s2)
        cfg.timeout_s, cfg.sync, cfg.areas, cfg.consumer_wait = 10, 0, areas, consumer_wait
        assert _native.cns_pipeline_run(cfg) == 0
        torch.cuda.synchronize()
        want_cs, _ = oracle.pipeline(tiles, words, rounds)
        np.testing.assert_array_equal(from_dev_u32(cs), want_cs)
        assert count_of(cns, done) == (0, 0) and count_of(cns, ack) == (0, rounds * cfg.consumer_ctas)
    finally:
        cns.cntnotify_destroy(done)
        cns.cntnotify_destroy(ack)


def test_op_chain_probe_applies_the_rule(cns):
    """cns_probe_op_chain applies its 16 ops iters times over to a count that starts at 0: the final count
    and the sum of the outcomes are the oracle's for the same ops repeated."""
    import torch
    ops = ci.notify_ops(16, seed=99)
    ops_d = torch.from_numpy(ops.view(np.int32).copy()).cuda()
    out = torch.zeros(2, dtype=torch.int64, device="cuda")
    assert cns.cns_probe_op_chain(ops_d, 3, out) == 0
    torch.cuda.synchronize()
    ns, packed = (int(v) for v in out.cpu().numpy().view(np.uint64))
    trace, fin = oracle.cnt_statemachine(np.tile(ops, (3, 1)), 0)
    assert packed & 0xFFFFFFFF == fin
    assert packed >> 32 == int(trace[:, 1].astype(np.uint64).sum())
    assert ns > 0
    assert cns.cns_probe_op_chain(ops_d, 0, out) == cns.CNS_ERR_INVALID_VALUE


def test_launch_cost_probe(cns):
    """The host's cost per kernel launch (the pipeline's roofline): positive, a few microseconds at most; bad
    arguments are refused."""
    import torch
    s = torch.cuda.Stream()
    for early in (0, 1):
        rc, us = cns.cns_probe_launch_cost(500, early, s)
        assert rc == 0 and 0.0 < us < 50.0
    assert cns.cns_probe_launch_cost(0, 1, s)[0] == cns.CNS_ERR_INVALID_VALUE
    assert cns.cns_probe_launch_cost(10, 2, s)[0] == cns.CNS_ERR_INVALID_VALUE
