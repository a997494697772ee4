"""Pins for the counted-notify part of the CPU oracle (no GPU)."""
import numpy as np
import pytest

import cns_inputs as ci
import oracle
from tests.conftest import read_golden

U32 = 1 << 32


def _int(s):
    return int(s, 0)


def test_truth_table_from_the_mode_definitions():
    rows = read_golden("cntnotify_truth_table.txt")
    n_rec = n_wait = 0
    for kind, mode, c, v, want in rows:
        mode, c, v = _int(mode), _int(c), _int(v)
        if kind == "record":
            n_rec += 1
            got, ok = oracle.cnt_record(c, mode, v)
            if want == "invalid":
                assert not ok and got == c
            else:
                assert ok and got == _int(want), (mode, hex(c), hex(v))
        else:
            n_wait += 1
            got = oracle.cnt_wait_satisfied(c, mode, v)
            assert got == (-1 if want == "invalid" else int(want)), (mode, hex(c), hex(v))
    assert n_rec >= 20 and n_wait >= 30
    # every defined mode appears
    modes = {(r[0], _int(r[1])) for r in rows}
    for m in (0, 1, 2, 4):
        assert ("record", m) in modes
    for m in range(5):
        assert ("wait", m) in modes


def test_hand_traced_sequence():
    rows = read_golden("cntnotify_sequence.txt")
    ops = np.array([[_int(k), _int(m), _int(v), _int(c)] for k, m, v, c, _, _, _ in rows], dtype=np.uint32)
    want = np.array([[_int(a), int(o)] for *_, a, o in rows], dtype=np.uint32)
    trace, final = oracle.cnt_statemachine(ops, 0)
    np.testing.assert_array_equal(trace, want)
    assert final == int(want[-1, 0])


def test_statemachine_steps_follow_single_op_rules():
    """Every step of a long random stream is one pinned single-op rule."""
    ops = ci.notify_ops(20000)
    trace, final = oracle.cnt_statemachine(ops, 7)
    prev = 7
    for i in range(ops.shape[0]):
        kind, mode, v, clr = (int(x) for x in ops[i])
        if kind == 0:
            nc, ok = oracle.cnt_record(prev, mode, v)
            assert ok and trace[i, 1] == oracle.OUT_RECORD and trace[i, 0] == nc
        else:
            s = oracle.cnt_wait_satisfied(prev, mode, v)
            assert trace[i, 1] == (oracle.OUT_WAIT_RELEASED if s else oracle.OUT_WAIT_HELD)
            assert trace[i, 0] == (0 if (s and clr) else prev)
        prev = int(trace[i, 0])
    assert final == prev


def test_op_stream_exercises_every_wait_outcome():
    ops = ci.notify_ops(1_000_000)
    trace, _ = oracle.cnt_statemachine(ops, 0)
    waits = ops[:, 0] == 1
    for m in range(5):
        sel = waits & (ops[:, 1] == m)
        outs = set(np.unique(trace[sel, 1]).tolist())
        assert outs == {0, 1}, (m, outs)
    assert (trace[:, 1] == oracle.OUT_INVALID).sum() == 0


def test_set_then_add_wraps():
    ops = np.array([[0, 0, 0xFFFFFFFE, 0], [0, 1, 3, 0]], dtype=np.uint32)
    trace, final = oracle.cnt_statemachine(ops, 123)
    assert trace[0, 0] == 0xFFFFFFFE and final == 1


def test_empty_stream_keeps_initial_count():
    trace, final = oracle.cnt_statemachine(np.zeros((0, 4), np.uint32), 0xABC)
    assert trace.shape == (0, 2) and final == 0xABC


def test_pipeline_checksum_closed_form():
    tiles, words, rounds = 4096, 256, 5
    cs, ct = oracle.pipeline(tiles, words, rounds)
    W = tiles * words
    for r in range(rounds):
        # sum_w (w * 2654435761 + r) = 2654435761 * W(W-1)/2 + r W   (mod 2^32)
        assert int(cs[r]) == (2654435761 * (W * (W - 1) // 2) + r * W) % U32
        assert int(ct[r]) == tiles
    assert oracle.pipeline_word(3, 2) == (3 * 2654435761 + 2) % U32
