"""Pins for the SYNCALL part of the CPU oracle (no GPU).

Each check ties the oracle to something other than itself: hand-worked
targets, closed forms of the ring payloads, an inverse map, Jacobi fixed
points and the decay of a Fourier mode.
"""
import math

import numpy as np
import pytest

import cns_inputs as ci
import oracle
from tests.conftest import read_golden

U32 = 1 << 32


# --- barrier arithmetic ------------------------------------------------------

def test_targets_match_hand_worked_values():
    rows = read_golden("syncall_targets.txt")
    assert len(rows) >= 20
    for before, P, M, target in rows:
        before, P, M, target = int(before), int(P), int(M), int(target)
        MM = U32 if M == 0 else M
        assert oracle.counter_modulus(P) == MM, (P, M)
        assert oracle.target_mod(before, P, MM) == target, (before, P, M)
        if M == 0:
            # with M = 2^32 the wrap-safe target is the literal u32 formula
            assert oracle.epoch_target(before, P) == target


@pytest.mark.parametrize("P,M", [(1, U32), (2, U32), (3, 4294967295), (4, U32), (8, U32),
                                 (111, 4294967289), (148, 4294967252), (64, U32), (592, 4294967104)])
def test_counter_modulus_hand_values(P, M):
    # M is the largest multiple of P not above 2^32, worked out by hand
    # (e.g. 2^32 / 592 = 7255012.3..., 592 * 7255012 = 4294967104)
    assert oracle.counter_modulus(P) == M
    assert M % P == 0 and M <= U32 and U32 - M < P


def test_reached_window():
    # While polling, the counter is in [before+1, target+P-1]; reached exactly on [target, target+P-1]
    for P, M in [(3, 9), (4, 8), (148, 4294967252), (4, U32)]:
        for before in [0, P - 1, P, M - P, M - 1]:
            t = oracle.target_mod(before, P, M)
            nxt = (before // P + 1) * P
            for d in range(1, nxt - before + P):      # every count the poller can see
                cur = (before + d) % M
                want = (cur - t) % M < P
                # counting arrivals: reached iff d arrivals took the count to the next multiple of P
                assert want == (d >= nxt - before)
                assert oracle.reached_mod(cur, t, P, M) == want


def test_arrive_cycles_through_zm():
    M = oracle.counter_modulus(3)
    assert oracle.arrive_mod(M - 1, M) == 0
    assert oracle.arrive_mod(5, M) == 6
    assert oracle.arrive_mod(U32 - 1, U32) == 0


# --- empty payload: the counter alone ------------------------------------------

@pytest.mark.parametrize("P,R,start", [(1, 5, 0), (8, 1000, 0), (148, 1000, 148 * 7), (3, 10, 4294967295 - 15)])
def test_final_counter_closed_form(P, R, start):
    M = oracle.counter_modulus(P)
    fc, rc = oracle.syncall_run_empty(P, R, start)
    assert rc == oracle.OK
    assert fc == (start + R * P) % M


def test_counter_start_not_multiple_of_p_deadlocks():
    # a workspace that was not zeroed ("counter garbage", troubleshooting table of the guide)
    fc, rc = oracle.syncall_run_empty(4, 3, 1)
    assert rc == oracle.DEADLOCK


def test_wrap_of_the_counter():
    P = 148
    M = oracle.counter_modulus(P)
    start = M - 5 * P
    fc, rc = oracle.syncall_run_empty(P, 12, start)
    assert rc == oracle.OK and fc == 7 * P


# --- ring payloads ---------------------------------------------------------------

def affine_closed_form(v0, R):
    """v_R[p] = 3^R v_0[(p+R)%P] + sum_r 3^(R-1-r) r  (mod 2^32), by induction on R."""
    P = v0.shape[0]
    mul = pow(3, R, U32)
    add = sum(pow(3, R - 1 - r, U32) * r for r in range(R)) % U32
    out = np.empty_like(v0)
    for p in range(P):
        src = v0[(p + R) % P].astype(object)
        out[p] = np.array([(mul * int(x) + add) % U32 for x in src], dtype=np.uint32)
    return out


@pytest.mark.parametrize("P,slots,R", [(1, 3, 7), (2, 5, 4), (3, 1, 11), (8, 256, 1000), (5, 7, 0)])
def test_ring_affine_closed_form(P, slots, R):
    v0 = ci.ring_payload(ci.SEED_RING_AFFINE, P, slots)
    out, fc, rc = oracle.syncall_run_ring(oracle.WL_RING_AFFINE, v0, R)
    assert rc == oracle.OK
    np.testing.assert_array_equal(out, affine_closed_form(v0, R))
    assert fc == (R * P) % oracle.counter_modulus(P)


@pytest.mark.parametrize("P,slots,R", [(148, 4, 100000), (7, 3, 13), (1, 4, 3)])
def test_ring_rotate_closed_form(P, slots, R):
    v0 = ci.ring_payload(ci.SEED_RING_ROTATE, P, slots)
    out, fc, rc = oracle.syncall_run_ring(oracle.WL_RING_ROTATE, v0, R)
    assert rc == oracle.OK
    np.testing.assert_array_equal(out, np.roll(v0, -R, axis=0))
    if (P, R) == (148, 100000):
        assert fc == 14_800_000
        # R mod P = 100: final[p] = init[(p + 100) % 148]
        np.testing.assert_array_equal(out[0], v0[100])


def test_xorshift_hand_value():
    # x = 1: x ^= x<<13 -> 8193; x ^= x>>17 -> 8193; x ^= x<<5 -> 8193 ^ 262176 = 270369
    assert oracle.xorshift32(1) == 270369
    assert oracle.xorshift32(0) == 0


def _xs_inverse(y):
    """Inverse of x ^= x<<13; x ^= x>>17; x ^= x<<5 on uint32 arrays."""
    y = y.astype(np.uint32)
    # undo x ^= x<<5
    x = y.copy()
    for _ in range(7):
        x = y ^ (x << np.uint32(5))
    # undo x ^= x>>17
    x = x ^ (x >> np.uint32(17))
    # undo x ^= x<<13
    z = x.copy()
    for _ in range(3):
        z = x ^ (z << np.uint32(13))
    return z


def test_xorshift_inverse_helper_is_an_inverse():
    x = ci.u32_uniform(99, 10000)
    y = np.array([oracle.xorshift32(int(v)) for v in x[:2000]], dtype=np.uint32)
    np.testing.assert_array_equal(_xs_inverse(y), x[:2000])


@pytest.mark.parametrize("P,slots,R", [(111, 256, 40), (64, 256, 10000), (2, 3, 5)])
def test_xorshift_ring_inverts_to_seed(P, slots, R):
    v0 = ci.ring_payload(ci.SEED_XORSHIFT, P, slots)
    out, fc, rc = oracle.syncall_run_ring(oracle.WL_XORSHIFT, v0, R)
    assert rc == oracle.OK
    v = out.copy()
    for r in range(R - 1, -1, -1):
        # v_{r+1}[p] = xs(v_r[(p+1)%P]) ^ r  =>  v_r[q] = xs^-1(v_{r+1}[q-1] ^ r)
        prev = _xs_inverse(v ^ np.uint32(r))
        v = np.roll(prev, 1, axis=0)
    np.testing.assert_array_equal(v, v0)


# --- Jacobi ----------------------------------------------------------------------

def test_jacobi_constant_is_fixed():
    u0 = np.full(1001, 0.375, dtype=np.float32)
    u, fc, rc = oracle.syncall_run_jacobi(u0, 17, 5)
    assert rc == oracle.OK and fc == 17 * 5
    np.testing.assert_array_equal(u, u0)


def test_jacobi_linear_is_fixed():
    i = np.arange(777, dtype=np.float32)
    u0 = (np.float32(-3.0) + np.float32(2.0) * i).astype(np.float32)
    u, _, _ = oracle.syncall_run_jacobi(u0, 9, 1)
    np.testing.assert_array_equal(u, u0)


@pytest.mark.parametrize("k", [1, 3, 10])
def test_jacobi_fourier_mode_decay(k):
    N, S = 1025, 12
    i = np.arange(N)
    u0 = np.sin(k * math.pi * i / (N - 1)).astype(np.float32)
    u0[0] = 0.0
    u0[-1] = 0.0
    u, _, _ = oracle.syncall_run_jacobi(u0, S, 1)
    want = np.cos(k * math.pi / (N - 1)) ** S * np.sin(k * math.pi * i / (N - 1))
    want[0] = want[-1] = 0.0
    np.testing.assert_allclose(u, want, rtol=0, atol=2e-6)


def test_jacobi_small_hand_case():
    u0 = np.array([1.0, 0.0, 0.0, 0.0, 3.0], dtype=np.float32)
    u, _, _ = oracle.syncall_run_jacobi(u0, 1, 1)
    np.testing.assert_array_equal(u, np.array([1.0, 0.5, 0.0, 1.5, 3.0], dtype=np.float32))
    u, _, _ = oracle.syncall_run_jacobi(u0, 2, 1)
    np.testing.assert_array_equal(u, np.array([1.0, 0.5, 1.0, 1.5, 3.0], dtype=np.float32))


@pytest.mark.parametrize("N", [1, 2, 3, 5, 64, 1000, 4099])
def test_jacobi_points_equal_full_run(N):
    u0 = ci.jacobi_field(N)
    S = 23
    full, _, _ = oracle.syncall_run_jacobi(u0, S, 3)
    idx = ci.sample_indices(7, N, 50)
    np.testing.assert_array_equal(oracle.jacobi_points(u0, S, idx), full[idx])


# --- cross-check of the u32 arithmetic against plain numpy on the field sizes used ---

def test_affine_oracle_matches_numpy_iteration():
    v0 = ci.ring_payload(ci.SEED_RING_AFFINE, 8, 256)
    v = v0.copy()
    for r in range(1000):
        v = (np.roll(v, -1, axis=0) * np.uint32(3) + np.uint32(r)).astype(np.uint32)
    out, _, _ = oracle.syncall_run_ring(oracle.WL_RING_AFFINE, v0, 1000)
    np.testing.assert_array_equal(out, v)
