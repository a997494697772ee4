"""All-interleaving checks of the soft-barrier protocol (no GPU).

The explorer enumerates every order of atomic arrive/poll steps for tiny
participant counts; the wrap-safe arithmetic must be safe and live for every
start value, and the broken variants (a participant that skips a barrier, an
exact-equality poll, the literal unsigned compare at the wrap) must be caught.
"""
import pytest

import oracle
from oracle.protocol import Arith, explore, explore_two_level, sequential_final_counter

U32 = 1 << 32


@pytest.mark.parametrize("P", [1, 2, 3, 4])
@pytest.mark.parametrize("R", [1, 2, 3])
def test_modular_counter_safe_and_live_for_every_start(P, R):
    for mult in (2, 3, 4):
        M = mult * P
        for start in range(0, M, P):
            res = explore(Arith("modular", P, M), R, start)
            assert res.ok and res.completed == 1, (P, R, M, start, res)


@pytest.mark.parametrize("P", [1, 2, 3, 4])
def test_full_width_counter(P):
    M = oracle.counter_modulus(P)
    for start in (0, M - P, M - 2 * P):
        res = explore(Arith("modular", P, M), 3, start)
        assert res.ok and res.completed == 1


def test_oracle_arithmetic_agrees_with_explorer_model():
    # the C oracle's arrive/target/reached are the same functions the explorer uses
    for P, M in [(3, 9), (4, 8), (3, oracle.counter_modulus(3)), (148, oracle.counter_modulus(148))]:
        a = Arith("modular", P, M)
        for before in list(range(0, min(M, 40))) + [M - 1, M - 2, M - P]:
            assert oracle.target_mod(before, P, M) == a.target(before)
            assert oracle.arrive_mod(before, M) == a.arrive(before)
            t = a.target(before)
            for cur in (t, (t + P - 1) % M, (t + P) % M, (t + M - 1) % M, (before + 1) % M):
                assert oracle.reached_mod(cur, t, P, M) == a.reached(cur, t)


def test_skipped_barrier_deadlocks():
    # one participant enters one barrier fewer ("same order, same count", guide §6.2)
    res = explore(Arith("modular", 3, 9), [2, 2, 1])
    assert res.deadlocks > 0 and res.completed == 0


def test_extra_barrier_deadlocks():
    res = explore(Arith("modular", 2, 8), [3, 2])
    assert res.deadlocks > 0


def test_equality_poll_can_miss_the_target():
    res = explore(Arith("equal", 3, 9), 2)
    assert res.deadlocks > 0


def test_literal_unsigned_compare_breaks_at_the_wrap():
    # a 5-bit word stands in for u32: near the wrap the literal target wraps to a
    # small value and `cur >= target` lets participants through early, or hangs
    broken = 0
    for P in (3, 4):
        for start in range(0, 32, P):
            res = explore(Arith("literal", P, 32), 2, start)
            broken += not res.ok
    assert broken > 0
    # far from the wrap the literal form is fine
    assert explore(Arith("literal", 3, U32), 3, 0).ok


def test_start_not_multiple_of_p_breaks():
    res = explore(Arith("modular", 4, 16), 2, 1)
    assert not res.ok


def test_sequential_final_counter():
    a = Arith("modular", 148, oracle.counter_modulus(148))
    assert sequential_final_counter(a, 1000) == 148_000


@pytest.mark.parametrize("P,C", [(2, 1), (2, 2), (4, 2), (4, 4), (6, 3), (6, 2)])
@pytest.mark.parametrize("R", [1, 2, 3])
def test_two_level_barrier_safe_and_live(P, C, R):
    res = explore_two_level(P, C, R)
    assert res.ok and res.completed == 1, res


# --- sense-flip comparison protocol --------------------------------------------------------

from oracle.protocol import explore_flip, flip_final_counter  # noqa: E402


@pytest.mark.parametrize("P", [1, 2, 3, 4])
@pytest.mark.parametrize("R", [1, 2, 3])
def test_flip_barrier_safe_and_live(P, R):
    res = explore_flip(P, R, bits=6)
    assert res.ok and res.completed == 1


def test_flip_barrier_from_the_other_sense():
    assert explore_flip(3, 3, bits=6, start=32).ok


def test_flip_barrier_needs_zero_low_bits():
    res = explore_flip(3, 2, bits=6, start=1)
    assert not res.ok


@pytest.mark.parametrize("wrong", [lambda top, P: top - P, lambda top, P: top - (P - 2), lambda top, P: top])
def test_flip_barrier_wrong_master_constant_is_caught(wrong):
    P, bits = 3, 6
    res = explore_flip(P, 2, bits=bits, master_add=wrong(1 << (bits - 1), P))
    assert not res.ok


def test_flip_barrier_skipped_barrier_deadlocks():
    res = explore_flip(3, [2, 2, 1], bits=6)
    assert res.deadlocks > 0


def test_flip_final_counter():
    assert flip_final_counter(148, 1) == 1 << 31
    assert flip_final_counter(148, 2) == 0
    assert flip_final_counter(148, 3, start=1 << 31) == 0


# --- hard path with one group barrier per round (members poll the counter themselves) -------

from oracle.protocol import explore_hard_one_barrier  # noqa: E402


@pytest.mark.parametrize("P,C", [(2, 1), (2, 2), (4, 2), (4, 4), (6, 2), (6, 3)])
@pytest.mark.parametrize("R", [1, 2, 3])
def test_hard_one_barrier_safe_and_live(P, C, R):
    res = explore_hard_one_barrier(P, C, R)
    assert res.ok and res.completed == 1


@pytest.mark.parametrize("start_mult", [1, 3])
def test_hard_one_barrier_from_an_aligned_start_near_the_wrap(start_mult):
    G = 2
    M = 4 * G
    assert explore_hard_one_barrier(4, 2, 3, M=M, start=M - start_mult * G).ok


def test_hard_one_barrier_misaligned_start_is_caught():
    res = explore_hard_one_barrier(4, 2, 2, start=1)
    assert not res.ok


@pytest.mark.parametrize("step", [0, 1, 3])
def test_hard_one_barrier_wrong_member_prediction_is_caught(step):
    # G = 2: members that step by anything else leave early or never
    assert not explore_hard_one_barrier(4, 2, 3, member_step=step).ok


# --- die-local counter copies (variants 5 and 8) ------------------------------------

# --- the hard path's paired gather / release step (SYNCALL §5.1's intra-block flags) -------

from oracle.protocol import explore_paired  # noqa: E402


@pytest.mark.parametrize("P,C", [(2, 2), (4, 2), (4, 4), (6, 2), (6, 3), (8, 2), (8, 4)])
@pytest.mark.parametrize("R", [1, 2, 3])
def test_paired_step_safe_and_live(P, C, R):
    res = explore_paired(P, C, R)
    assert res.ok and res.completed == 1


@pytest.mark.parametrize("start_mult", [1, 3])
def test_paired_step_from_an_aligned_start_near_the_wrap(start_mult):
    G = 2
    M = 4 * G
    assert explore_paired(4, 2, 3, M=M, start=M - start_mult * G).ok


def test_paired_step_misaligned_start_is_caught():
    assert not explore_paired(4, 2, 2, start=1).ok


@pytest.mark.parametrize("mistake", [{"wait_gather": False}, {"poll_first": False}, {"members_wait": False}])
def test_paired_step_planted_mistakes_are_caught(mistake):
    """A leader that arrives before its members, a leader that releases them before the round is seen, and
    members that do not wait for the release: each lets someone leave a barrier early."""
    res = explore_paired(4, 2, 2, **mistake)
    assert res.safety_violations > 0


from oracle.protocol import explore_die_local  # noqa: E402

NEARS = [(0, 1), (1, 0), (0, 1, 1), (0, 0, 1), (0, 1, 0, 1), (0, 0), (1, 1, 1)]


@pytest.mark.parametrize("near", NEARS)
@pytest.mark.parametrize("R", [1, 2, 3])
def test_die_local_copies_safe_and_live(near, R):
    """Cursor targets after the first barrier and a first barrier whose far
    increment lands after the near one: safe, every epoch right, no deadlock,
    whichever order the two increments of each arrival land in."""
    r = explore_die_local(near, R)
    assert r.ok and r.completed > 0, r


@pytest.mark.parametrize("near", [(0, 1), (0, 1, 1)])
@pytest.mark.parametrize("mult", [1, 2, 3])
def test_die_local_copies_through_the_wrap(near, mult):
    P = len(near)
    M = 4 * P
    r = explore_die_local(near, 3, M=M, start=(M - mult * P) % M)
    assert r.ok and r.completed > 0, r


@pytest.mark.parametrize("near", [(0, 1), (0, 1, 1), (0, 1, 0, 1)])
def test_die_local_target_from_the_returned_value_fails_later(near):
    """Taking every round's target from the near copy's returned value: a
    participant whose near increment lands after another's next-round
    increment computes the next epoch's target and the barrier deadlocks."""
    r = explore_die_local(near, 3, target="formula")
    assert r.epoch_violations > 0 and r.deadlocks > 0


@pytest.mark.parametrize("near", [(0, 1), (0, 0, 1)])
def test_die_local_unordered_first_barrier_fails(near):
    """Cursor targets alone are not enough: with the far increment free to
    land before the near one in the first barrier, that barrier's target (from
    the returned value) can be an epoch ahead."""
    r = explore_die_local(near, 2, target="cursor", safe_first=False)
    assert r.epoch_violations > 0 and r.deadlocks > 0


@pytest.mark.parametrize("near", NEARS)
@pytest.mark.parametrize("R", [1, 2, 3])
@pytest.mark.parametrize("release,near_red", [(False, False), (False, True), (True, True)])
def test_die_local_arrival_forms_safe_and_live(near, R, release, near_red):
    """The arrival-only form (no fence: a participant's next increments may leave while its last ones
    are in flight) and the form whose near increment is fire-and-forget from the second barrier on
    (the participant polls at once): safe, every epoch right, no deadlock."""
    r = explore_die_local(near, R, release=release, near_red=near_red)
    assert r.ok and r.completed > 0, r


@pytest.mark.parametrize("near", [(0, 1), (0, 1, 1)])
@pytest.mark.parametrize("mult", [1, 2, 3])
def test_die_local_fire_and_forget_through_the_wrap(near, mult):
    P = len(near)
    M = 4 * P
    r = explore_die_local(near, 3, M=M, start=(M - mult * P) % M, release=False, near_red=True)
    assert r.ok and r.completed > 0, r


@pytest.mark.parametrize("near", [(0, 1), (0, 0, 1)])
def test_die_local_fire_and_forget_needs_the_ordered_first_barrier(near):
    """The first barrier still takes its target from the returned value, so it still needs the far
    increment ordered after the near one."""
    r = explore_die_local(near, 2, safe_first=False, release=False, near_red=True)
    assert r.epoch_violations > 0 and r.deadlocks > 0


def test_die_local_start_off_the_epoch_grid_is_caught():
    """A count that does not start at a multiple of P (a workspace reused with another P) breaks the
    epochs on the copies: the model reports it, as the library documents for this variant."""
    assert explore_die_local((0, 1, 1), 2).ok
    bad = explore_die_local((0, 1), 2, start=1)
    assert bad.epoch_violations > 0


# --- the two-stream pipeline's handshakes ("CANN Runtime CntNotify" §5) ------------------

from oracle.protocol import explore_pipeline  # noqa: E402


@pytest.mark.parametrize("form", ["in_kernel", "stream"])
@pytest.mark.parametrize("areas", [1, 2])
@pytest.mark.parametrize("K,C,R", [(1, 1, 3), (2, 2, 3), (3, 3, 4), (2, 3, 5), (4, 2, 4)])
def test_pipeline_handshakes_safe_and_live(form, areas, K, C, R):
    """Every interleaving: each read finds its round's data in every tile, each wait releases on
    exactly K records, nothing is stuck, and the run ends at done = 0, ack = R * C."""
    r = explore_pipeline(K, C, R, areas=areas, form=form)
    assert r.ok and r.completed == 1, r


@pytest.mark.parametrize("flag", ["go_gate", "clear_before_go"])
def test_pipeline_in_kernel_wait_rules_are_needed_with_two_areas(flag):
    """Without the previous round's go (or with go published before the clear), CTA 0 of the next
    consumer grid, scheduled early, can take the previous round's count for its own: reads of stale
    tiles, releases on the wrong count, stuck rounds."""
    r = explore_pipeline(2, 2, 3, areas=2, form="in_kernel", **{flag: False})
    assert r.safety_violations > 0 and r.epoch_violations > 0 and r.deadlocks > 0
    # with one area the consumer grids run one after another, and neither rule is needed
    assert explore_pipeline(2, 2, 3, areas=1, form="in_kernel", **{flag: False}).ok


@pytest.mark.parametrize("form", ["in_kernel", "stream"])
def test_pipeline_records_must_wait_for_the_clear(form):
    """Two areas: a record that lands before the previous round's clear is wiped by it."""
    r = explore_pipeline(2, 2, 3, areas=2, form=form, clear_wait=False)
    assert r.epoch_violations > 0 and r.deadlocks > 0


@pytest.mark.parametrize("areas", [1, 2])
def test_pipeline_consumer_ctas_cannot_all_poll_the_count(areas):
    """With more than one consumer CTA polling done and CTA 0 clearing it, a CTA that looks after the
    clear waits for ever: the reason for the go word."""
    assert explore_pipeline(2, 2, 3, areas=areas, all_poll=True).deadlocks > 0
    assert explore_pipeline(2, 1, 3, areas=areas, all_poll=True).ok


# --- the state machine's links between tiles, across launches ----------------------------

from oracle.protocol import explore_links  # noqa: E402

LINK_STARTS = [None, (False, False, False), (True, False, True), (False, True, False, True), (False,) * 4]


@pytest.mark.parametrize("starts", LINK_STARTS)
@pytest.mark.parametrize("launches", [1, 2, 3])
def test_links_taken_words_cleared_are_never_stale(starts, launches):
    """A tile takes its predecessor's link word once it carries the call's tag and sets it to 0: every
    take reads the word its own launch published, even when every launch carries the same tag (a
    CUDA graph replaying one captured call), and every launch completes."""
    T = len(starts) if starts else 3
    r = explore_links(T, launches, starts)
    assert r.ok and r.completed > 0, r


@pytest.mark.parametrize("starts", LINK_STARTS)
def test_links_without_the_clear_go_stale_under_replays(starts):
    """Without the clear, a replay's tile can take the word its predecessor published in the replay
    before (same tag): the model finds it, as the GPU did (wrong trace entries when the ops changed
    between replays)."""
    T = len(starts) if starts else 3
    r = explore_links(T, 2, starts, clear=False)
    assert r.safety_violations > 0


@pytest.mark.parametrize("starts", LINK_STARTS)
def test_links_without_the_clear_hold_with_a_tag_per_call(starts):
    """Calls submitted one by one each carry a new tag, and then the words need no clearing."""
    T = len(starts) if starts else 3
    r = explore_links(T, 3, starts, clear=False, same_tag=False)
    assert r.ok and r.completed > 0, r
