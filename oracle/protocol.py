"""Exhaustive interleaving explorer for the SYNCALL soft-mode epoch barrier.

TEST INFRASTRUCTURE ONLY (see oracle/__init__.py).

Model ("PTO-ISA SYNCALL cross-core barrier guide", lmnt.cn/news/269652, §5.2):
each of P participants runs its barriers one after another; one barrier is

    before = atomic fetch-and-increment(counter)
    target = (before / P + 1) * P
    spin until the counter has reached target

The explorer treats the increment and each successful poll as atomic steps
and enumerates every order in which participants can take them (depth-first,
with a visited-state set).  A failed poll changes nothing, so a polling
participant is simply not enabled until its condition holds.  For every
reachable state it checks

  safety    no participant leaves barrier k before (k+1)*P arrivals happened
            ("any core may continue only after every participant has
            executed the barrier", §2);
  epochs    the values returned to the arrivals of barrier k are exactly
            start + kP .. start + kP + P-1 (mod the cycle length);
  liveness  no reachable state has every unfinished participant blocked.

Counter arithmetic variants:
  "modular"  the wrap-safe reading: counter in Z_M with M a multiple of P,
             target taken mod M, reached <=> (cur - target) mod M < P;
  "literal"  a W-value word (W = 2^bits) with the pages' literal formula and
             an unsigned >= compare, wrapping at W;
  "equal"    modular counter but the poll waits for cur == target exactly.
The last two exist to show that the explorer does catch broken protocols.

The later explorers take the same approach to the library's other
protocols: the two-level (cluster) barrier, the sense-flip counter, the
one-barrier hard path, its paired gather / release step (explore_paired),
the die-local counter copies, the two-stream counted-notify pipeline's
handshakes (explore_pipeline), and the op-stream state machine's link words
between tiles across repeated launches (explore_links).
"""
from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Arith:
    kind: str        # "modular" | "literal" | "equal"
    P: int
    M: int           # cycle length (modular/equal) or word size W (literal)

    def arrive(self, c: int) -> int:
        return (c + 1) % self.M

    def target(self, before: int) -> int:
        return ((before // self.P) + 1) * self.P % self.M

    def reached(self, cur: int, t: int) -> bool:
        if self.kind == "modular":
            return (cur - t) % self.M < self.P
        if self.kind == "equal":
            return cur == t
        if self.kind == "literal":
            return cur >= t
        raise ValueError(self.kind)


@dataclass
class Result:
    states: int = 0
    safety_violations: int = 0
    epoch_violations: int = 0
    deadlocks: int = 0
    completed: int = 0          # terminal states with everyone done

    @property
    def ok(self) -> bool:
        return self.safety_violations == 0 and self.epoch_violations == 0 and self.deadlocks == 0


def explore(arith: Arith, rounds, start: int = 0, max_states: int = 2_000_000) -> Result:
    """Enumerate all interleavings.

    rounds: per-participant barrier count (sequence of length P), or an int for
    all participants.  start: counter value before the first arrival.
    """
    P = arith.P
    if isinstance(rounds, int):
        rounds = [rounds] * P
    rounds = tuple(rounds)
    assert len(rounds) == P
    res = Result()
    # participant state: (k barriers finished, phase 0 = next is arrive /
    # 1 = polling, target)
    init = (start % arith.M, tuple((0, 0, 0) for _ in range(P)))
    seen = set()
    stack = [init]
    while stack:
        state = stack.pop()
        if state in seen:
            continue
        seen.add(state)
        res.states += 1
        if res.states > max_states:
            raise RuntimeError("state space larger than max_states")
        c, parts = state
        arrivals = sum(k + ph for (k, ph, _) in parts)
        succ = []
        for i, (k, ph, t) in enumerate(parts):
            if k == rounds[i]:
                continue
            if ph == 0:
                before = c
                # epochs: the j-th arrival of barrier k gets start + kP + j
                if (before - start - k * P) % arith.M >= P:
                    res.epoch_violations += 1
                nt = arith.target(before)
                nparts = parts[:i] + ((k, 1, nt),) + parts[i + 1:]
                succ.append((arith.arrive(c), nparts))
            elif arith.reached(c, t):
                # leaving barrier k: all (k+1)*P arrivals must have happened
                if arrivals < (k + 1) * P:
                    res.safety_violations += 1
                nparts = parts[:i] + ((k + 1, 0, 0),) + parts[i + 1:]
                succ.append((c, nparts))
        if not succ:
            if all(parts[i][0] == rounds[i] for i in range(P)):
                res.completed += 1
            else:
                res.deadlocks += 1
        stack.extend(succ)
    return res


def sequential_final_counter(arith: Arith, rounds: int, start: int = 0) -> int:
    """Counter after `rounds` barriers taken in participant order (one schedule)."""
    c = start % arith.M
    for _ in range(rounds):
        for _ in range(arith.P):
            c = arith.arrive(c)
    return c


# Two-level (cluster) barrier -------------------------------------------------
#
# The hard path replaces the per-participant arrive with: every member of a
# group of C arrives on a group barrier; the group leader alone arrives on the
# global counter (Pg = number of groups) and polls it; a second group barrier
# releases the members.  The pages' MIX hard path has this shape (the cube core
# waits for its paired vector cores, takes part in the cross-core sync, then
# releases them, §5.1).  The model checks the same safety property at
# participant level.

def explore_two_level(P: int, C: int, rounds: int, M: int | None = None, start: int = 0,
                      max_states: int = 2_000_000) -> Result:
    assert P % C == 0
    G = P // C
    arith = Arith("modular", G, M if M is not None else 4 * G)
    res = Result()
    # member phases: 0 = before group-arrive, 1 = waiting in group barrier 1,
    # 2 = waiting in group barrier 2 (leader: 2 = arrived globally, polling),
    # member k counter.  group state: count in barrier 1, count in barrier 2,
    # generation.  Modelled per participant: (k, phase, target)
    init = (start % arith.M, tuple((0, 0, 0) for _ in range(P)))
    seen = set()
    stack = [init]
    while stack:
        state = stack.pop()
        if state in seen:
            continue
        seen.add(state)
        res.states += 1
        if res.states > max_states:
            raise RuntimeError("state space larger than max_states")
        c, parts = state
        succ = []
        for i, (k, ph, t) in enumerate(parts):
            if k == rounds:
                continue
            g, lead = i // C, (i % C == 0)
            grp = parts[g * C:(g + 1) * C]
            if ph == 0:
                # group barrier 1 arrive
                succ.append((c, parts[:i] + ((k, 1, 0),) + parts[i + 1:]))
            elif ph == 1:
                # group barrier 1 opens when all members of the group are at
                # phase >= 1 of the same barrier k
                if all(m[0] == k and m[1] >= 1 for m in grp):
                    if lead:
                        before = c
                        if (before - start - k * G) % arith.M >= G:
                            res.epoch_violations += 1
                        succ.append((arith.arrive(c), parts[:i] + ((k, 3, arith.target(before)),) + parts[i + 1:]))
                    else:
                        succ.append((c, parts[:i] + ((k, 2, 0),) + parts[i + 1:]))
            elif ph == 3:
                if arith.reached(c, t):
                    succ.append((c, parts[:i] + ((k, 2, 0),) + parts[i + 1:]))
            elif ph == 2:
                # group barrier 2 opens when all members are at phase 2 (leader
                # got there only after its global poll succeeded)
                if all((m[0] == k and m[1] == 2) or m[0] == k + 1 for m in grp):
                    # leaving barrier k: every participant must have arrived
                    if not all(m[0] > k or (m[0] == k and m[1] >= 1) for m in parts):
                        res.safety_violations += 1
                    succ.append((c, parts[:i] + ((k + 1, 0, 0),) + parts[i + 1:]))
        if not succ:
            if all(p[0] == rounds for p in parts):
                res.completed += 1
            else:
                res.deadlocks += 1
        stack.extend(succ)
    return res


# Sense-flip counter --------------------------------------------------------
#
# A comparison protocol, not the pages' arithmetic: the word has `bits` bits
# and its top bit is the sense.  Participant 0 adds 2^(bits-1) - (P-1), every
# other participant adds 1, so one barrier's P additions total exactly
# 2^(bits-1): the low bits return to where they were and the sense flips once
# the last participant has added.  A participant polls until the sense differs
# from the one in the value its own addition returned.  The low bits must be
# 0 at the start (start is 0 or 2^(bits-1)).  The runtime's grid barrier of
# CUDA cooperative groups uses this scheme with bits = 32.

def explore_flip(P: int, rounds, bits: int = 8, start: int = 0, max_states: int = 2_000_000,
                 master_add: int | None = None) -> Result:
    """All interleavings of the sense-flip barrier.  master_add overrides
    participant 0's addition (the tests use it to plant a wrong constant)."""
    W = 1 << bits
    top = W >> 1
    assert P >= 1 and P < top
    m_add = (top - (P - 1)) % W if master_add is None else master_add % W
    if isinstance(rounds, int):
        rounds = [rounds] * P
    rounds = tuple(rounds)
    res = Result()
    init = (start % W, tuple((0, 0, 0) for _ in range(P)))
    seen = set()
    stack = [init]
    while stack:
        state = stack.pop()
        if state in seen:
            continue
        seen.add(state)
        res.states += 1
        if res.states > max_states:
            raise RuntimeError("state space larger than max_states")
        c, parts = state
        arrivals = sum(k + ph for (k, ph, _) in parts)
        succ = []
        for i, (k, ph, s) in enumerate(parts):
            if k == rounds[i]:
                continue
            if ph == 0:
                before = c
                add = m_add if i == 0 else 1
                nparts = parts[:i] + ((k, 1, before & top),) + parts[i + 1:]
                succ.append(((c + add) % W, nparts))
            elif (c & top) != s:
                if arrivals < (k + 1) * P:
                    res.safety_violations += 1
                nparts = parts[:i] + ((k + 1, 0, 0),) + parts[i + 1:]
                succ.append((c, nparts))
        if not succ:
            if all(parts[i][0] == rounds[i] for i in range(P)):
                res.completed += 1
            else:
                res.deadlocks += 1
        stack.extend(succ)
    return res


def flip_final_counter(P: int, rounds: int, bits: int = 32, start: int = 0) -> int:
    """Word after `rounds` complete sense-flip barriers: each adds 2^(bits-1) in total."""
    W = 1 << bits
    return (start + rounds * (W >> 1)) % W


# Hard path with one group barrier per round --------------------------------
#
# The first barrier of a run is the two-level form above, except that the
# leader hands the round's target to its members as the second group barrier
# opens.  From then on a round is: group barrier; the leader arrives on the
# counter; every participant -- leader and members alike -- polls the counter
# for its own target, the members' target being the previous one plus G.  A
# leader whose returned count puts it in another epoch than that prediction
# counts as an epoch violation (the kernel stops the run there).

def explore_hard_one_barrier(P: int, C: int, rounds: int, M: int | None = None, start: int = 0,
                             max_states: int = 2_000_000, member_step: int | None = None) -> Result:
    """All interleavings of the one-barrier hard path.  member_step overrides
    the members' prediction step (G; the tests plant wrong ones)."""
    assert P % C == 0
    G = P // C
    step = G if member_step is None else member_step
    arith = Arith("modular", G, M if M is not None else 4 * G)
    res = Result()
    # participant: (k rounds done, phase, target, cursor)
    #   phase 0 before the group barrier, 1 in it, 3 polling,
    #   2 in the first round's second group barrier
    init = (start % arith.M, tuple((0, 0, 0, 0) for _ in range(P)))
    seen = set()
    stack = [init]

    def arrived(m, k):
        return m[0] > k or (m[0] == k and m[1] >= 1)

    while stack:
        state = stack.pop()
        if state in seen:
            continue
        seen.add(state)
        res.states += 1
        if res.states > max_states:
            raise RuntimeError("state space larger than max_states")
        c, parts = state
        succ = []
        for i, (k, ph, t, cur) in enumerate(parts):
            if k == rounds:
                continue
            g, lead = i // C, (i % C == 0)
            grp = parts[g * C:(g + 1) * C]

            def put(v, nc=c):
                succ.append((nc, parts[:i] + (v,) + parts[i + 1:]))

            if ph == 0:
                put((k, 1, 0, cur))
            elif ph == 1:
                if not all(arrived(m, k) for m in grp):
                    continue
                if lead:
                    before = c
                    if (before - start - k * G) % arith.M >= G:
                        res.epoch_violations += 1
                    tgt = arith.target(before)
                    if k > 0 and tgt != (cur + G) % arith.M:
                        res.epoch_violations += 1
                    put((k, 3, tgt, cur), arith.arrive(c))
                elif k == 0:
                    put((k, 2, 0, cur))          # members wait for the leader's hand-over
                else:
                    put((k, 3, (cur + step) % arith.M, cur))
            elif ph == 3:
                if not arith.reached(c, t):
                    continue
                if k == 0 and lead:
                    put((k, 2, t, t))            # the leader joins the second group barrier
                    continue
                if not all(arrived(m, k) for m in parts):
                    res.safety_violations += 1
                put((k + 1, 0, 0, t))
            elif ph == 2:
                # the first round's second group barrier opens once every member
                # is in it (or already through); the leader reached it holding
                # the round's target, which the members take as their cursor
                if not all((m[0] == 0 and m[1] == 2) or m[0] > 0 for m in grp):
                    continue
                if not all(arrived(m, 0) for m in parts):
                    res.safety_violations += 1
                leader = grp[0]
                tgt = t if lead else (leader[2] if leader[0] == 0 else leader[3])
                put((1, 0, 0, tgt))
        if not succ:
            if all(p[0] == rounds for p in parts):
                res.completed += 1
            else:
                res.deadlocks += 1
        stack.extend(succ)
    return res


# The hard path's paired step -------------------------------------------------
#
# The guide's MIX hard path pairs each AIC core with its AIV cores on
# intra-block flags (SYNCALL §5.1): the AIVs set a flag the AIC waits for, the
# AIC takes part in the cross-core step, then sets a flag each AIV waits for.
# Participant i belongs to group i // C; its rank 0 is the leader.  A member's
# barrier k is one arrival on its leader's gather count, then a wait until the
# leader has released round k.  The leader's barrier k is a wait until all
# C - 1 members have arrived for round k, then the device-wide step on the
# counter (one arrival per group, the pages' arithmetic over the groups), then
# the release of its members.
#
#   wait_gather=False     the leader arrives on the counter without waiting
#                         for its members (a planted mistake)
#   poll_first=False      the leader releases its members before its poll of
#                         the counter has seen the round (a planted mistake)
#   members_wait=False    members leave without waiting for the release (a
#                         planted mistake)

def explore_paired(P: int, C: int, rounds: int, M: int | None = None, start: int = 0,
                   max_states: int = 2_000_000, wait_gather: bool = True, poll_first: bool = True,
                   members_wait: bool = True) -> Result:
    """All interleavings of the paired (gather / release) hard step."""
    assert P % C == 0
    G = P // C
    arith = Arith("modular", G, M if M is not None else 4 * G)
    res = Result()
    # participant: (k barriers finished, phase, target)
    #   member  phase 0 before barrier k, 1 arrived on the gather count, waiting for the release
    #   leader  phase 0 before barrier k, 1 in it waiting for the gather, 3 polling the counter
    # per group: the members' gather arrivals so far, and the rounds released so far
    init = (start % arith.M, (0,) * G, (0,) * G, tuple((0, 0, 0) for _ in range(P)))
    seen = set()
    stack = [init]

    def arrived(m, k):
        return m[0] > k or (m[0] == k and m[1] >= 1)

    while stack:
        state = stack.pop()
        if state in seen:
            continue
        seen.add(state)
        res.states += 1
        if res.states > max_states:
            raise RuntimeError("state space larger than max_states")
        c, gathered, released, parts = state
        succ = []

        def leave(i, k):
            if not all(arrived(m, k) for m in parts):
                res.safety_violations += 1
            return parts[:i] + ((k + 1, 0, 0),) + parts[i + 1:]

        for i, (k, ph, t) in enumerate(parts):
            if k == rounds:
                continue
            g, lead = i // C, (i % C == 0)

            def put(v, nc=c, ng=gathered, nr=released):
                succ.append((nc, ng, nr, parts[:i] + (v,) + parts[i + 1:]))

            if not lead:
                if ph == 0:
                    ng = gathered[:g] + (gathered[g] + 1,) + gathered[g + 1:]
                    put((k, 1, 0), ng=ng)
                elif not members_wait or released[g] >= k + 1:
                    succ.append((c, gathered, released, leave(i, k)))
                continue
            if ph == 0:
                put((k, 1, 0))
            elif ph == 1:
                if wait_gather and gathered[g] < (k + 1) * (C - 1):
                    continue
                before = c
                if (before - start - k * G) % arith.M >= G:
                    res.epoch_violations += 1
                tgt = arith.target(before)
                if poll_first:
                    put((k, 3, tgt), nc=arith.arrive(c))
                else:
                    # the members are released at once; the leader still polls
                    nr = released[:g] + (k + 1,) + released[g + 1:]
                    put((k, 3, tgt), nc=arith.arrive(c), nr=nr)
            elif ph == 3:
                if not arith.reached(c, t):
                    continue
                nr = released[:g] + (max(released[g], k + 1),) + released[g + 1:]
                succ.append((c, gathered, nr, leave(i, k)))
        if not succ:
            if all(p[0] == rounds for p in parts):
                res.completed += 1
            else:
                res.deadlocks += 1
        stack.extend(succ)
    return res


# Die-local counter copies ---------------------------------------------------
#
# Two copies of the counter; participant i calls copy near[i] its near copy.
# One arrival is a fire-and-forget increment of the far copy and a returning
# increment of the near copy, issued together after one release fence: the
# two land in either order, and the far one may still be in flight when the
# participant has left the barrier.  Its next arrival's fence waits for both,
# so a participant has at most one round's increments in flight.  The
# returned old value of the near copy gives the target; the participant then
# polls its near copy (the arrival whose increment completed the round there
# leaves at once).
#
#   target="formula"  target = ((before / P) + 1) * P from the returned value,
#                     in every round (the pages' arithmetic)
#   target="cursor"   from the second round on, the target is the last one
#                     plus P (the formula only in the first round)
#   safe_first=True   in the first round the far increment is issued only
#                     after the near one has returned (a release increment
#                     of the far copy orders it after the near one)
#   release=False     no fence before an arrival (the arrival-only contract):
#                     a participant's next increments may leave while its
#                     last ones are still in flight (one thread's increments
#                     of one copy land in the order they were issued; they
#                     are all +1, so only their number matters here)
#   near_red=True     from the second round on (cursor targets), the near
#                     increment is fire-and-forget too and the participant
#                     polls at once: nothing needs the near copy's old value

def explore_die_local(near, rounds: int, M: int | None = None, start: int = 0, target: str = "cursor",
                      safe_first: bool = True, release: bool = True, near_red: bool = False,
                      max_states: int = 2_000_000) -> Result:
    P = len(near)
    arith = Arith("modular", P, M if M is not None else 4 * P)
    res = Result()
    # participant: (k, phase, target, cursor end or -1, far increments in flight, near ones in flight)
    #   phase 0 between barriers, 1 waiting for the returning near increment, 2 polling
    init = ((start % arith.M, start % arith.M), tuple((0, 0, 0, -1, 0, 0) for _ in range(P)))
    seen = set()
    stack = [init]

    def arrived(m, k):
        return m[0] > k or (m[0] == k and m[1] >= 1)

    while stack:
        state = stack.pop()
        if state in seen:
            continue
        seen.add(state)
        res.states += 1
        if res.states > max_states:
            raise RuntimeError("state space larger than max_states")
        cs, parts = state
        succ = []
        for i, (k, ph, t, cend, pf, pn) in enumerate(parts):
            me, other = near[i], 1 - near[i]

            def put(v, ncs=cs):
                succ.append((ncs, parts[:i] + (v,) + parts[i + 1:]))

            def bump(copy):
                nc = list(cs)
                nc[copy] = arith.arrive(nc[copy])
                return tuple(nc)

            if pf:   # a far increment lands (any time while in flight)
                put((k, ph, t, cend, pf - 1, pn), bump(other))
            if pn and ph != 1:   # a fire-and-forget near increment lands
                put((k, ph, t, cend, pf, pn - 1), bump(me))
            if k == rounds:
                continue
            if ph == 0:
                if release and (pf or pn):
                    continue   # the next arrival's fence waits for the last one's increments
                if near_red and target == "cursor" and cend >= 0:
                    if cend != (start + (k + 1) * P) % arith.M:
                        res.epoch_violations += 1
                    put((k, 2, cend, (cend + P) % arith.M, pf + 1, pn + 1))
                    continue
                if pn:
                    continue   # a returning increment is issued once the last ones have landed
                first_safe = safe_first and k == 0
                put((k, 1, 0, cend, pf + (0 if first_safe else 1), 1))
            elif ph == 1:
                before = cs[me]
                if target == "cursor" and cend >= 0:
                    tgt = cend
                else:
                    tgt = arith.target(before)
                if tgt != (start + (k + 1) * P) % arith.M:
                    res.epoch_violations += 1
                far_now = pf + (1 if (safe_first and k == 0) else 0)
                nxt = (tgt + P) % arith.M
                if arith.reached(arith.arrive(before), tgt):
                    if not all(arrived(m, k) for m in parts):
                        res.safety_violations += 1
                    put((k + 1, 0, 0, nxt, far_now, 0), bump(me))
                else:
                    put((k, 2, tgt, nxt, far_now, 0), bump(me))
            elif ph == 2 and arith.reached(cs[me], t):
                if not all(arrived(m, k) for m in parts):
                    res.safety_violations += 1
                put((k + 1, 0, 0, cend, pf, pn))
        if not succ:
            if all(p[0] == rounds for p in parts):
                res.completed += 1
            else:
                res.deadlocks += 1
        stack.extend(succ)
    return res


def explore_pipeline(tiles: int, consumers: int, rounds: int, areas: int = 2, form: str = "in_kernel",
                     go_gate: bool = True, clear_before_go: bool = True, clear_wait: bool = True,
                     all_poll: bool = False, max_states: int = 3_000_000) -> Result:
    """All interleavings of the two-stream counting pipeline's handshakes
    ("CANN Runtime CntNotify" §5: producers record ADD 1 per tile, the waiter
    waits BIGGER_OR_EQUAL tiles with isClear and continues), as this library
    runs it: `tiles` producer CTAs of one tile each per round, `consumers`
    consumer CTAs, `areas` tile areas, every atomic step taken in any order.

    Words: done (the count), ack (consumer CTAs that finished reading), go
    (form "in_kernel": the last round whose wait has released and cleared),
    and one tag per tile of each area (the round whose data it holds).
    Producer tile j of round r: waits until the consumers that last read its
    area have all recorded on ack (one area: ack >= r * consumers; two:
    ack >= (r - 1) * consumers), stores (tag = r); with two areas it then
    waits for the previous producer grid to complete and for done < tiles;
    then records ADD 1 on done.  With one area a producer grid starts after
    the previous one completes (stream order).
    form "in_kernel": consumer CTA 0 waits for go >= r, then done >= tiles,
    clears done, publishes go = r + 1; the other CTAs wait for go >= r + 1.
    Their start is not ordered at all with two areas (the go gate alone must
    keep them right); with one area a grid starts after the previous one
    completes.  Every CTA then waits for the previous consumer grid to
    complete (two areas), reads its area and records ADD 1 on ack.
    form "stream": a wait task per round polls done >= tiles and clears it;
    it starts after the previous round's wait task has completed and
    completes after the previous consumer grid; the round's consumer CTAs
    start after it completes, read and record on ack.

    Checks: every read finds the round's own data in every tile of its area;
    every wait releases on exactly `tiles` (no record of another round is
    counted or lost); no reachable state is stuck; at the end done = 0 and
    ack = rounds * consumers.  The flags break one rule each, to show that
    the checks see it: go_gate (CTA 0 waits for the previous round's go),
    clear_before_go (the clear comes before the publish), clear_wait (two
    areas: records wait for done < tiles); all_poll = True has every consumer
    CTA poll done itself (and CTA 0 still clear it) instead of waiting for go.
    """
    K, C, R, A = tiles, consumers, rounds, areas
    assert A in (1, 2) and form in ("in_kernel", "stream")
    res = Result()
    # state: (done, ack, go, tags, producers, consumers, waits)
    #   producer phase: 0 start, 1 stored, 2 may record, 3 recorded
    #   consumer phase (in_kernel, CTA 0): 0 start, 1 released (seen checked), 2 cleared, 3 past the wait,
    #   4 read, 5 recorded on ack; other CTAs: 0 start, 3 past the wait, 4, 5
    #   consumer phase (stream): 0 start, 3 past the wait (the task completed), 4, 5
    #   wait task phase (stream): 0 start, 1 released, 2 cleared, 3 completed
    init = (0, 0, 0, tuple(-1 for _ in range(A * K)), tuple(0 for _ in range(R * K)),
            tuple(0 for _ in range(R * C)), tuple(0 for _ in range(R)))
    seen = set()
    stack = [init]
    while stack:
        state = stack.pop()
        if state in seen:
            continue
        seen.add(state)
        res.states += 1
        if res.states > max_states:
            raise RuntimeError("state space larger than max_states")
        done, ack, go, tags, pr, co, wt = state
        succ = []

        def p_complete(r):
            return r < 0 or all(pr[r * K + j] == 3 for j in range(K))

        def c_complete(r):
            return r < 0 or all(co[r * C + c] == 5 for c in range(C))

        def check_seen(v):
            if v != K:
                res.epoch_violations += 1

        for r in range(R):
            for j in range(K):
                i, ph = r * K + j, pr[r * K + j]
                npr = lambda v: pr[:i] + (v,) + pr[i + 1:]  # noqa: E731
                if ph == 0:
                    need = (r - A + 1) * C
                    if (A == 1 and not p_complete(r - 1)) or (r >= A and ack < need):
                        continue
                    nt = tags[:(r % A) * K + j] + (r,) + tags[(r % A) * K + j + 1:]
                    succ.append((done, ack, go, nt, npr(1), co, wt))
                elif ph == 1:
                    if A == 2 and (not p_complete(r - 1) or (clear_wait and done >= K)):
                        continue
                    succ.append((done, ack, go, tags, npr(2), co, wt))
                elif ph == 2:
                    succ.append((done + 1, ack, go, tags, npr(3), co, wt))
            if form == "stream":
                ph = wt[r]
                nwt = lambda v: wt[:r] + (v,) + wt[r + 1:]  # noqa: E731
                if ph == 0 and (r == 0 or wt[r - 1] == 3) and (A == 2 or c_complete(r - 1)) and done >= K:
                    check_seen(done)
                    succ.append((done, ack, go, tags, pr, co, nwt(1)))
                elif ph == 1:
                    succ.append((0, ack, go, tags, pr, co, nwt(2)))
                elif ph == 2 and c_complete(r - 1):
                    succ.append((done, ack, go, tags, pr, co, nwt(3)))
            for c in range(C):
                i, ph = r * C + c, co[r * C + c]
                nco = lambda v: co[:i] + (v,) + co[i + 1:]  # noqa: E731
                if ph == 0:
                    if form == "stream":
                        if wt[r] == 3:
                            succ.append((done, ack, go, tags, pr, nco(3), wt))
                        continue
                    if A == 1 and not c_complete(r - 1):
                        continue
                    if c == 0:
                        if (go_gate and go < r) or done < K:
                            continue
                        check_seen(done)
                        if clear_before_go:
                            succ.append((done, ack, go, tags, pr, nco(1), wt))
                        else:
                            succ.append((done, ack, r + 1, tags, pr, nco(1), wt))
                    elif all_poll:
                        if (go_gate and go < r) or done < K:
                            continue
                        check_seen(done)
                        succ.append((done, ack, go, tags, pr, nco(3), wt))
                    elif go >= r + 1:
                        succ.append((done, ack, go, tags, pr, nco(3), wt))
                elif ph == 1:
                    succ.append((0, ack, go, tags, pr, nco(2), wt))
                elif ph == 2:
                    succ.append((done, ack, max(go, r + 1), tags, pr, nco(3), wt))
                elif ph == 3:
                    if A == 2 and form == "in_kernel" and not c_complete(r - 1):
                        continue
                    if any(tags[(r % A) * K + j] != r for j in range(K)):
                        res.safety_violations += 1
                    succ.append((done, ack, go, tags, pr, nco(4), wt))
                elif ph == 4:
                    succ.append((done, ack + 1, go, tags, pr, nco(5), wt))
        if not succ:
            if all(p == 3 for p in pr) and all(c == 5 for c in co) and all(w in (0, 3) for w in wt) \
                    and (form == "in_kernel" or all(w == 3 for w in wt)):
                res.completed += 1
                if done != 0 or ack != R * C:
                    res.epoch_violations += 1
            else:
                res.deadlocks += 1
        stack.extend(succ)
    return res


# The op-stream state machine's links between tiles, across launches ---------
#
# One launch walks T tiles; tile t's end count goes to the next tile through a
# link word tagged with the launch's tag: the tile publishes the word (after
# taking its predecessor's, if the tile holds no start, else at once), and
# the next tile waits until the word carries the tag, then takes it.  A CUDA
# graph replays a captured launch with the same tag, launch after launch (each
# launch starts once the one before it has ended).  The explorer enumerates
# every order of the tiles' steps within each of L launches and checks that
# every take reads the word its own launch published.
#
#   clear=True    the thread that takes a word sets it to 0 (no launch's tag)
#   starts        per tile, whether it holds a start (publishes before it
#                 waits) or not (its count needs its predecessor's)
#   same_tag      every launch carries the same tag (graph replays); False:
#                 a tag per launch (calls submitted one by one)
#
# Result.safety_violations counts takes of a word another launch published.

def explore_links(T: int, launches: int, starts=None, clear: bool = True, same_tag: bool = True,
                  max_states: int = 2_000_000) -> Result:
    starts = tuple(starts) if starts is not None else tuple(True for _ in range(T))
    res = Result()
    # link word: (tag, launch that published it) or None; tile: (published, taken)
    init = (0, tuple(None for _ in range(T)), tuple((False, False) for _ in range(T)))
    seen = set()
    stack = [init]
    while stack:
        state = stack.pop()
        if state in seen:
            continue
        seen.add(state)
        res.states += 1
        if res.states > max_states:
            raise RuntimeError("state space larger than max_states")
        k, words, tiles = state
        if k == launches:
            res.completed += 1
            continue
        tag = 1 if same_tag else k + 1
        succ = []

        def done(t, pub, took):
            return (pub or t == T - 1) and (took or t == 0)

        if all(done(t, *tiles[t]) for t in range(T)):   # the launch has ended: the next one starts
            succ.append((k + 1, words, tuple((False, False) for _ in range(T))))
        for t in range(T):
            pub, took = tiles[t]

            def put(nw, npub, ntook):
                succ.append((k, nw, tiles[:t] + ((npub, ntook),) + tiles[t + 1:]))

            # publish: a tile with a start at any time (its last stretch needs no earlier count); one
            # without, once it has taken its predecessor's count (tile 0 starts from the call's init)
            if not pub and t < T - 1 and (starts[t] or took or t == 0):
                put(words[:t] + ((tag, k),) + words[t + 1:], True, took)
            # take: once the predecessor's word carries the tag
            if not took and t > 0:
                got = words[t - 1]
                if got is not None and got[0] == tag:
                    if got[1] != k:
                        res.safety_violations += 1
                    nw = words[:t - 1] + (None,) + words[t:] if clear else words
                    put(nw, pub, True)
        if not succ:
            res.deadlocks += 1
        stack.extend(succ)
    return res
