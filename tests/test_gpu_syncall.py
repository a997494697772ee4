"""SYNCALL on the GPU against the CPU oracle (bit-exact for every u32 round
and counter; the fp32 Jacobi within 1e-5 relative and in fact bit-exact)."""
import numpy as np
import pytest

import cns_inputs as ci
import oracle
from tests.gpu_helpers import from_dev_u32, to_dev_f32, to_dev_u32

pytestmark = pytest.mark.gpu

SOFT, HARD = 1, 0
AIV, AIC, MIX = 0, 1, 2


@pytest.fixture(scope="module")
def cns():
    import torch
    import counted_notify_sync_gb300 as c
    c.build()
    torch.cuda.set_device(0)
    return c


# Word offsets (int32) of the counters in a die-local workspace: soft counter, hard counter, and their
# second copies 4 KB further on.
COUNTER_WORDS = (0, 64, 1024, 1024 + 64)


def garble_counters(ws, value):
    """Counter garbage written over an initialised workspace's counters (not through the library): the
    base count that the workspace check reads still says 0, so the run starts and the counts desynchronise
    the epochs."""
    for w in COUNTER_WORDS:
        ws[w] = value


def run_ring(cns, mode, core, wl, launch_ctas, v0, rounds, used=0, ratio=0, start=0, threads=256,
             cluster_dim=0, timeout_ms=0, check=True, variant=0, garble=None, launch_flags=0, ws=None, hard_step=0):
    import torch
    P, slots = v0.shape
    b0 = to_dev_u32(v0) if v0.size else None
    b1 = torch.zeros_like(b0) if v0.size else None
    if ws is None:
        ws = cns.new_workspace(start_value=start, participants=P, elems=slots)
    if garble is not None:
        garble_counters(ws, garble)
    group = (1 + (ratio or 1)) if core == MIX else 1
    status = torch.zeros(launch_ctas * group, dtype=torch.int32, device="cuda")
    d, rc = cns.run_syncall(mode, core, wl, launch_ctas, b0, b1, rounds, used_cores=used, aiv_ratio=ratio,
                            elems=slots, threads=threads, cluster_dim=cluster_dim, workspace=ws,
                            cta_status=status, timeout_ms=timeout_ms, check=check, variant=variant,
                            launch_flags=launch_flags, hard_step=hard_step)
    torch.cuda.synchronize()
    final = from_dev_u32(b1 if rounds & 1 else b0).reshape(P, slots) if v0.size else v0.copy()
    return d, rc, final, status.cpu().numpy()


def expect_ring(wl, v0, rounds, start=0):
    out, fc, rc = oracle.syncall_run_ring(wl, v0, rounds, start)
    assert rc == oracle.OK
    return out, fc


# --- ring-affine, 8 participants (256 uint32 each, 1000 rounds) --------------------------

def test_ring_affine_p8_1000_rounds(cns):
    v0 = ci.ring_payload(ci.SEED_RING_AFFINE, 8, 256)
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_RING_AFFINE, 8, v0, 1000)
    want, fc = expect_ring(oracle.WL_RING_AFFINE, v0, 1000)
    np.testing.assert_array_equal(got, want)
    assert d.final_counter == fc == 8000 and d.device_status == 0
    assert d.participants == 8 and d.grid_ctas == 8
    assert (st == cns.CNS_CTA_DONE).all()


@pytest.mark.parametrize("P,slots,R,threads", [(3, 7, 5, 32), (5, 1030, 17, 256), (1, 4, 9, 64), (2, 0, 4, 32),
                                                (13, 4096, 3, 1024), (16, 9, 2, 96)])
def test_ring_affine_ragged_shapes(cns, P, slots, R, threads):
    v0 = ci.ring_payload(ci.SEED_RING_AFFINE + P, P, slots)
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_RING_AFFINE, P, v0, R, threads=threads)
    want, fc = expect_ring(oracle.WL_RING_AFFINE, v0, R)
    np.testing.assert_array_equal(got, want)
    assert d.final_counter == fc


def test_zero_rounds_leaves_everything(cns):
    v0 = ci.ring_payload(1, 4, 8)
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_RING_AFFINE, 4, v0, 0)
    np.testing.assert_array_equal(got, v0)
    assert d.final_counter == 0


# --- ring-rotate, 148 participants, 100000 rounds, soft and hard -------------------------

@pytest.mark.parametrize("mode,variant", [(SOFT, 0), (HARD, 0), (SOFT, 5), (HARD, 5)])
def test_ring_rotate_p148_100000_rounds(cns, mode, variant):
    """The full ring-rotate configuration against the oracle, in the guide's
    form (variant 0) and in the bench's headline form (variant 5, die-local
    counter copies)."""
    v0 = ci.ring_payload(ci.SEED_RING_ROTATE, 148, 4)
    d, rc, got, st = run_ring(cns, mode, AIV, cns.CNS_WL_RING_ROTATE, 148, v0, 100000, variant=variant)
    want, fc = expect_ring(oracle.WL_RING_ROTATE, v0, 100000)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(got, np.roll(v0, -100000, axis=0))
    assert d.device_status == 0 and (st == cns.CNS_CTA_DONE).all()
    if mode == SOFT:
        assert d.final_counter == fc == 14_800_000 and d.cluster_used == 1
    else:
        assert d.cluster_used in (1, 2, 4)
        assert d.final_counter == 100000 * (148 // d.cluster_used)


@pytest.mark.parametrize("C", [1, 2, 4])
def test_hard_explicit_cluster_dims(cns, C):
    v0 = ci.ring_payload(7, 16, 12)
    d, rc, got, st = run_ring(cns, HARD, AIV, cns.CNS_WL_RING_AFFINE, 16, v0, 301, cluster_dim=C)
    want, _ = expect_ring(oracle.WL_RING_AFFINE, v0, 301)
    np.testing.assert_array_equal(got, want)
    assert d.cluster_used == C and d.final_counter == 301 * (16 // C)


# --- MIX role classes and the used_cores subset (xorshift payload) --------------------------

@pytest.mark.parametrize("mode", [SOFT, HARD])
def test_mix_37_groups_ratio_2(cns, mode):
    v0 = ci.ring_payload(ci.SEED_XORSHIFT, 111, 256)
    d, rc, got, st = run_ring(cns, mode, MIX, cns.CNS_WL_XORSHIFT, 37, v0, 10000, ratio=2)
    want, fc = expect_ring(oracle.WL_XORSHIFT, v0, 10000)
    np.testing.assert_array_equal(got, want)
    assert d.participants == 111 and d.grid_ctas == 111
    roles = st >> 8
    np.testing.assert_array_equal(roles, (np.arange(111) % 3 == 0).astype(np.int32))
    assert ((st & 0xFF) == cns.CNS_CTA_DONE).all()
    if mode == SOFT:
        assert d.final_counter == fc
    else:
        assert d.cluster_used == 3 and d.final_counter == 10000 * 37


def test_mix_default_ratio_is_one(cns):
    v0 = ci.ring_payload(11, 10, 8)
    d, rc, got, st = run_ring(cns, SOFT, MIX, cns.CNS_WL_XORSHIFT, 5, v0, 33, ratio=0)
    want, _ = expect_ring(oracle.WL_XORSHIFT, v0, 33)
    np.testing.assert_array_equal(got, want)
    assert d.participants == 10


def test_used_cores_subset_64_of_148(cns):
    import torch
    v0 = ci.ring_payload(ci.SEED_XORSHIFT, 64, 256)
    b0 = to_dev_u32(v0)
    b1 = torch.zeros_like(b0)
    ws = cns.new_workspace()
    status = torch.zeros(148, dtype=torch.int32, device="cuda")
    d, rc = cns.run_syncall(SOFT, AIV, cns.CNS_WL_XORSHIFT, 148, b0, b1, 10000, used_cores=64, elems=256,
                            workspace=ws, cta_status=status)
    got = from_dev_u32(b0).reshape(64, 256)
    want, fc = expect_ring(oracle.WL_XORSHIFT, v0, 10000)
    np.testing.assert_array_equal(got, want)
    st = status.cpu().numpy()
    assert (st[:64] == cns.CNS_CTA_DONE).all() and (st[64:] == cns.CNS_CTA_IDLE).all()
    assert d.final_counter == fc == 640000 and d.participants == 64


@pytest.mark.parametrize("mode", [SOFT, HARD])
def test_aic_only(cns, mode):
    v0 = ci.ring_payload(5, 24, 64)
    d, rc, got, st = run_ring(cns, mode, AIC, cns.CNS_WL_RING_AFFINE, 24, v0, 99)
    want, _ = expect_ring(oracle.WL_RING_AFFINE, v0, 99)
    np.testing.assert_array_equal(got, want)
    assert ((st >> 8) == 1).all()


# --- counter arithmetic -------------------------------------------------------------------

def test_empty_payload_counter_only(cns):
    ws = cns.new_workspace()
    d, rc = cns.run_syncall(SOFT, AIV, cns.CNS_WL_EMPTY, 148, None, None, 5000, workspace=ws)
    fc, _ = oracle.syncall_run_empty(148, 5000)
    assert d.final_counter == fc == 740000


@pytest.mark.parametrize("P", [148, 3, 111])
def test_counter_wraps_through_zm(cns, P):
    M = oracle.counter_modulus(P)
    start = M - 5 * P
    v0 = ci.ring_payload(9, P, 4)
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_RING_AFFINE, P, v0, 12, start=start)
    want, fc = expect_ring(oracle.WL_RING_AFFINE, v0, 12, start)
    np.testing.assert_array_equal(got, want)
    assert d.final_counter == fc == 7 * P


def test_workspace_reused_across_runs(cns):
    ws = cns.new_workspace()
    total = 0
    for R in (10, 1, 77):
        d, rc = cns.run_syncall(SOFT, AIV, cns.CNS_WL_EMPTY, 37, None, None, R, workspace=ws)
        total += R
        assert d.final_counter == 37 * total


# --- Jacobi -------------------------------------------------------------------------------

def run_jacobi(cns, u0, sweeps, ctas, mode=SOFT, threads=256, variant=0, hard_step=0):
    import torch
    b0 = to_dev_f32(u0)
    b1 = torch.zeros_like(b0)
    ws = cns.new_workspace()
    d, rc = cns.run_syncall(mode, AIV, cns.CNS_WL_JACOBI, ctas, b0, b1, sweeps, elems=u0.size,
                            threads=threads, workspace=ws, variant=variant, hard_step=hard_step)
    out = (b1 if sweeps & 1 else b0).cpu().numpy()
    return d, out


@pytest.mark.parametrize("N,sweeps,ctas,threads", [(100003, 20, 37, 256), (4099, 7, 5, 64), (5, 3, 2, 32),
                                                   (1, 2, 1, 32), (2, 5, 3, 32), (64, 11, 20, 32),
                                                   (1 << 20, 9, 592, 256)])
def test_jacobi_small_bit_exact(cns, N, sweeps, ctas, threads):
    u0 = ci.jacobi_field(N)
    d, got = run_jacobi(cns, u0, sweeps, ctas, threads=threads)
    want, fc, rc = oracle.syncall_run_jacobi(u0, sweeps, ctas)
    np.testing.assert_allclose(got, want, rtol=1e-5, atol=0)
    np.testing.assert_array_equal(got, want)
    assert d.final_counter == fc


@pytest.mark.parametrize("variant", [0, 1, 5, 6])
@pytest.mark.parametrize("cols_per_cta,extra", [(0, 3), (1, 0), (1, 2), (2, 1), (3, 0), (2050, 3)])
@pytest.mark.parametrize("sweeps", [1, 2, 7])
def test_jacobi_split_phase_chunk_shapes(cns, variant, cols_per_cta, extra, sweeps):
    """The soft Jacobi runs its sweeps split-phase (interior before the wait,
    first/last column and tail after it): chunks of 0, 1, 2, 3 and >2 tiles of
    float4 columns, with and without a scalar tail, for several variants."""
    import torch
    ctas = 37
    N = 4 * (cols_per_cta * ctas + (5 if cols_per_cta == 0 else 0)) + extra
    u0 = ci.jacobi_field(N, seed=cols_per_cta * 10 + extra)
    b0 = to_dev_f32(u0)
    b1 = torch.zeros_like(b0)
    ws = cns.new_workspace()
    d, rc = cns.run_syncall(SOFT, AIV, cns.CNS_WL_JACOBI, ctas, b0, b1, sweeps, elems=N, threads=128, workspace=ws,
                            variant=variant)
    got = (b1 if sweeps & 1 else b0).cpu().numpy()
    want, fc, orc = oracle.syncall_run_jacobi(u0, sweeps, ctas)
    np.testing.assert_array_equal(got, want)
    assert rc == 0 and d.device_status == 0


def test_jacobi_hard_path(cns):
    u0 = ci.jacobi_field(200003)
    d, got = run_jacobi(cns, u0, 10, 64, mode=HARD)
    want, _, _ = oracle.syncall_run_jacobi(u0, 10, 64)
    np.testing.assert_array_equal(got, want)


@pytest.fixture(scope="module")
def jacobi_full_size_oracle():
    """The oracle's whole field after 200 sweeps of N = 2^26 points on 592 participants (about 20 s on one
    host core), computed once for the full-size tests below."""
    N, S, C = 1 << 26, 200, 592
    u0 = ci.jacobi_field(N)
    want, fc, rc = oracle.syncall_run_jacobi(u0, S, C)
    assert rc == oracle.OK and fc == S * C
    return u0, want


@pytest.mark.parametrize("mode,variant", [(SOFT, 0), (SOFT, 2), (SOFT, 5), (HARD, 5)])
def test_jacobi_full_size_whole_field(cns, jacobi_full_size_oracle, mode, variant):
    """The full Jacobi configuration -- 2^26 fp32 points, 592 persistent CTAs,
    200 sweeps with a barrier between sweeps -- compared with the oracle on
    every point: bit for bit (the bar is 1e-5 relative).  The variants the
    bench measures, and the hard path."""
    u0, want = jacobi_full_size_oracle
    d, got = run_jacobi(cns, u0, 200, 592, mode=mode, variant=variant)
    assert d.device_status == 0
    if mode == SOFT:
        assert d.final_counter == 200 * 592
    np.testing.assert_allclose(got, want, rtol=1e-5, atol=0)
    np.testing.assert_array_equal(got, want)


def test_jacobi_full_size_sampled(cns):
    """2^26 points, 592 CTAs, 200 sweeps: sampled points from the oracle's
    light-cone evaluation, plus chunk edges and both ends."""
    N, S, C = 1 << 26, 200, 592
    u0 = ci.jacobi_field(N)
    d, got = run_jacobi(cns, u0, S, C)
    assert d.device_status == 0 and d.final_counter == S * C
    n4 = N // 4
    edges = []
    for p in range(0, C, 37):
        j0 = p * (n4 // C) + min(p, n4 % C)
        edges += [4 * j0 - 1, 4 * j0, 4 * j0 + 3, 4 * j0 + 4]
    idx = np.unique(np.concatenate([ci.sample_indices(3, N, 300), np.clip(np.array(edges), 0, N - 1)]))
    want = oracle.jacobi_points(u0, S, idx)
    np.testing.assert_allclose(got[idx], want, rtol=1e-5, atol=0)
    np.testing.assert_array_equal(got[idx], want)
    assert got[0] == u0[0] and got[-1] == u0[-1]


# --- host buffers through the same call -----------------------------------------------------

def test_host_in_host_out(cns):
    import torch
    v0 = ci.ring_payload(ci.SEED_RING_ROTATE, 148, 4)
    hin = torch.from_numpy(v0.view(np.int32).copy()).pin_memory()
    hout = torch.empty_like(hin).pin_memory()
    b0 = torch.empty(148 * 4, dtype=torch.int32, device="cuda")
    b1 = torch.empty_like(b0)
    ws = cns.new_workspace()
    d, rc = cns.run_syncall(SOFT, AIV, cns.CNS_WL_RING_ROTATE, 148, b0, b1, 1001, elems=4, workspace=ws,
                            host_in=hin, host_out=hout)
    np.testing.assert_array_equal(hout.numpy().view(np.uint32).reshape(148, 4), np.roll(v0, -1001, axis=0))


# --- failures reported as status, never a hang ---------------------------------------------

def test_unzeroed_workspace_times_out_and_context_survives(cns):
    """A counter at 1 ("counter garbage", written behind the library's back so
    that the workspace check passes) puts the participants in different epochs;
    the bounded poll gives up."""
    v0 = ci.ring_payload(3, 4, 4)
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_RING_AFFINE, 4, v0, 3, garble=1, timeout_ms=300,
                              check=False)
    assert rc == cns.CNS_ERR_TIMEOUT and d.device_status == cns.CNS_ERR_TIMEOUT
    assert ((st & 0xFF) == cns.CNS_CTA_ABORTED).any()
    # the device still works
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_RING_AFFINE, 4, v0, 3)
    want, _ = expect_ring(oracle.WL_RING_AFFINE, v0, 3)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("variant", [0, 1, 4])
@pytest.mark.parametrize("rounds", [1, 3, 6])
def test_hard_path_unzeroed_workspace_times_out(cns, variant, rounds):
    """The hard path with a counter garbled to 1: the clusters' leaders fall into
    different epochs and the bounded waits give up.  A CTA that stops takes its
    whole cluster with it at the next cluster barrier, so the run ends (no CTA
    is left at a cluster barrier) and reports the timeout.  (Not the die-local
    variant: each copy sees the arrivals in its own order, so a misaligned
    start need not put anyone in a later epoch there.)"""
    v0 = ci.ring_payload(3, 8, 4)
    d, rc, got, st = run_ring(cns, HARD, AIV, cns.CNS_WL_RING_AFFINE, 8, v0, rounds, garble=1, timeout_ms=300,
                              cluster_dim=4, check=False, variant=variant)
    assert rc == cns.CNS_ERR_TIMEOUT and d.device_status == cns.CNS_ERR_TIMEOUT
    assert ((st & 0xFF) == cns.CNS_CTA_ABORTED).any()
    # CTAs of one cluster agree
    assert len(set((st[:4] & 0xFF).tolist())) == 1 and len(set((st[4:] & 0xFF).tolist())) == 1


def test_hard_path_long_run_with_many_clusters(cns):
    """Members follow the epochs themselves after the first round: a long run on
    37 clusters of 4 lands exactly where the oracle does, near the wrap too."""
    P = 148
    v0 = ci.ring_payload(11, P, 8)
    Pc = 37
    M = oracle.counter_modulus(Pc)
    d, rc, got, st = run_ring(cns, HARD, AIV, cns.CNS_WL_XORSHIFT, P, v0, 5001, start=M - 7 * Pc, cluster_dim=4)
    want, _ = expect_ring(oracle.WL_XORSHIFT, v0, 5001)
    np.testing.assert_array_equal(got, want)
    assert d.device_status == 0 and d.final_counter == (M - 7 * Pc + 5001 * Pc) % M
    assert (st == cns.CNS_CTA_DONE).all()


def test_grid_that_cannot_be_resident_is_refused(cns):
    import torch
    ws = cns.new_workspace()
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    d, rc = cns.run_syncall(SOFT, AIV, cns.CNS_WL_EMPTY, sms * 64 + 1, None, None, 1, threads=1024, workspace=ws,
                            check=False)
    assert rc == cns.CNS_ERR_NOT_RESIDENT


# --- barrier variants: same results, every wait form ----------------------------------------

VARIANTS = [0, 1, 2, 3, 4, 5]


@pytest.mark.parametrize("variant", VARIANTS)
@pytest.mark.parametrize("mode", [SOFT, HARD])
def test_variants_ring_rotate_148(cns, variant, mode):
    v0 = ci.ring_payload(ci.SEED_RING_ROTATE, 148, 4)
    d, rc, got, st = run_ring(cns, mode, AIV, cns.CNS_WL_RING_ROTATE, 148, v0, 20001, variant=variant)
    np.testing.assert_array_equal(got, np.roll(v0, -20001, axis=0))
    assert d.device_status == 0 and (st == cns.CNS_CTA_DONE).all()
    assert d.final_counter == 20001 * (148 if mode == SOFT else 148 // d.cluster_used)


@pytest.mark.parametrize("variant", VARIANTS)
def test_variants_affine_and_mix(cns, variant):
    v0 = ci.ring_payload(ci.SEED_RING_AFFINE, 8, 256)
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_RING_AFFINE, 8, v0, 1000, variant=variant)
    want, fc = expect_ring(oracle.WL_RING_AFFINE, v0, 1000)
    np.testing.assert_array_equal(got, want)
    v1 = ci.ring_payload(ci.SEED_XORSHIFT, 111, 256)
    d, rc, got, st = run_ring(cns, HARD, MIX, cns.CNS_WL_XORSHIFT, 37, v1, 2000, ratio=2, variant=variant)
    want, _ = expect_ring(oracle.WL_XORSHIFT, v1, 2000)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("variant", VARIANTS)
def test_variants_wrap_and_jacobi(cns, variant):
    P = 111
    M = oracle.counter_modulus(P)
    v0 = ci.ring_payload(9, P, 4)
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_RING_AFFINE, P, v0, 12, start=M - 5 * P, variant=variant)
    want, fc = expect_ring(oracle.WL_RING_AFFINE, v0, 12, M - 5 * P)
    np.testing.assert_array_equal(got, want)
    assert d.final_counter == fc
    import torch
    u0 = ci.jacobi_field(300007)
    b0 = to_dev_f32(u0)
    b1 = torch.zeros_like(b0)
    ws = cns.new_workspace()
    cns.run_syncall(SOFT, AIV, cns.CNS_WL_JACOBI, 592, b0, b1, 8, elems=u0.size, workspace=ws, variant=variant)
    want, _, _ = oracle.syncall_run_jacobi(u0, 8, 592)
    np.testing.assert_array_equal(b0.cpu().numpy(), want)


@pytest.mark.parametrize("variant", [v for v in VARIANTS if v != 5])
def test_variants_time_out_cleanly(cns, variant):
    """A single counter garbled to 1 behind the library's back ends the run in a
    timeout.  The die-local variant is left out: each of its copies sees the
    arrivals in its own order, so a garbled count need not leave anyone behind
    there (the workspace check below guards its start)."""
    v0 = ci.ring_payload(3, 4, 4)
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_RING_AFFINE, 4, v0, 3, garble=1, timeout_ms=200,
                              check=False, variant=variant)
    assert rc == cns.CNS_ERR_TIMEOUT


# --- the workspace check ("counter garbage", SYNCALL guide §8) -----------------------------

@pytest.mark.parametrize("mode", [SOFT, HARD])
@pytest.mark.parametrize("variant", [0, 2, 5])
@pytest.mark.parametrize("start", [1, 3, 0xFFFFFFFF])
def test_misaligned_start_is_refused_before_any_arrival(cns, mode, variant, start):
    """A workspace initialised with a start that is not a multiple of P (P = 4
    participants, or 2 clusters of 2): refused with INVALID_VALUE at once, every
    CTA aborted, and no counter moved -- the die-local variant included, which
    could otherwise release participants early."""
    v0 = ci.ring_payload(3, 4, 4)
    # an even round count: the result would be in buffer 0, which holds the input untouched
    d, rc, got, st = run_ring(cns, mode, AIV, cns.CNS_WL_RING_AFFINE, 4, v0, 4, start=start, timeout_ms=2000,
                              check=False, variant=variant, cluster_dim=2 if mode == HARD else 0)
    assert rc == cns.CNS_ERR_INVALID_VALUE and d.device_status == cns.CNS_ERR_INVALID_VALUE
    assert d.elapsed_ms < 100.0
    assert ((st & 0xFF) == cns.CNS_CTA_ABORTED).all()
    assert d.final_counter == start
    np.testing.assert_array_equal(got, v0)


def test_die_local_misaligned_start_ends(cns):
    """The die-local variant from a misaligned start never reports success: the
    workspace check refuses it before anyone arrives."""
    v0 = ci.ring_payload(3, 4, 4)
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_RING_AFFINE, 4, v0, 3, start=1, timeout_ms=200,
                              check=False, variant=5)
    assert rc != 0 and rc == cns.CNS_ERR_INVALID_VALUE


@pytest.mark.parametrize("variant", [0, 5])
def test_workspace_reused_with_another_participant_count(cns, variant):
    """Runs continue on one workspace from where the last one left the counter;
    a run whose P does not divide that count is refused, one whose P does runs
    exactly as the oracle does from that start."""
    import torch
    ws = cns.new_workspace()
    v4 = ci.ring_payload(21, 4, 8)
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_XORSHIFT, 4, v4, 3, ws=ws, variant=variant)
    assert rc == 0 and d.final_counter == 12
    v5 = ci.ring_payload(22, 5, 8)
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_XORSHIFT, 5, v5, 4, ws=ws, variant=variant, check=False)
    assert rc == cns.CNS_ERR_INVALID_VALUE and d.final_counter == 12
    np.testing.assert_array_equal(got, v5)
    # the refusal raised the status: initialise a fresh one at the count the P = 4 run left
    ws = cns.new_workspace(start_value=12)
    v6 = ci.ring_payload(23, 6, 8)
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_XORSHIFT, 6, v6, 7, ws=ws, variant=variant)
    want, fc = expect_ring(oracle.WL_XORSHIFT, v6, 7, start=12)
    np.testing.assert_array_equal(got, want)
    assert d.final_counter == fc == 12 + 42
    # and a second run on it continues from 54
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_XORSHIFT, 6, v6, 5, ws=ws, variant=variant)
    want, fc = expect_ring(oracle.WL_XORSHIFT, v6, 5, start=54)
    np.testing.assert_array_equal(got, want)
    assert d.final_counter == fc == 84


@pytest.mark.parametrize("mode", [SOFT, HARD])
def test_zeroed_workspace_is_accepted_and_garbage_refused(cns, mode):
    """A workspace zeroed by the caller (the guide's own preparation, §4.1)
    works without syncall_workspace_init; one full of garbage is refused."""
    import torch
    v0 = ci.ring_payload(5, 8, 4)
    ws = torch.zeros(cns.CNS_SYNCALL_WORKSPACE_BYTES // 4, dtype=torch.int32, device="cuda")
    d, rc, got, st = run_ring(cns, mode, AIV, cns.CNS_WL_RING_ROTATE, 8, v0, 10, ws=ws,
                              cluster_dim=2 if mode == HARD else 0)
    np.testing.assert_array_equal(got, np.roll(v0, -10, axis=0))
    g = torch.from_numpy(ci.ring_payload(99, 1, cns.CNS_SYNCALL_WORKSPACE_BYTES // 4)[0].view(np.int32).copy())
    ws = g.cuda()
    d, rc, got, st = run_ring(cns, mode, AIV, cns.CNS_WL_RING_ROTATE, 8, v0, 10, ws=ws, check=False,
                              cluster_dim=2 if mode == HARD else 0)
    assert rc == cns.CNS_ERR_INVALID_VALUE
    np.testing.assert_array_equal(got, v0)


def test_sense_flip_tags_the_workspace(cns):
    """After a sense-flip run the count is no longer on the pages' epoch grid:
    the other variants refuse the workspace, the sense-flip variant goes on."""
    v0 = ci.ring_payload(6, 8, 4)
    ws = cns.new_workspace()
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_RING_ROTATE, 8, v0, 3, ws=ws, variant=6)
    assert rc == 0
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_RING_ROTATE, 8, v0, 3, ws=ws, variant=0, check=False)
    assert rc == cns.CNS_ERR_INVALID_VALUE


# --- the hard path takes its cluster shape from the launch it got ---------------------------

@pytest.mark.parametrize("variant", [0, 2, 5, 6])
@pytest.mark.parametrize("wl", ["rotate", "xorshift"])
def test_hard_path_without_the_cluster_attribute(cns, variant, wl):
    """The hard kernel launched without the cluster attribute (as a tool's
    replay may launch it): each CTA is a cluster of its own, the kernel counts
    the clusters itself, and the run is exact and fast (no timeout)."""
    P = 148
    R = 3001
    v0 = ci.ring_payload(ci.SEED_RING_ROTATE, P, 4)
    code = cns.CNS_WL_RING_ROTATE if wl == "rotate" else cns.CNS_WL_XORSHIFT
    d, rc, got, st = run_ring(cns, HARD, AIV, code, P, v0, R, cluster_dim=4, variant=variant,
                              launch_flags=cns.CNS_LAUNCH_NO_CLUSTER_ATTR)
    want, _ = expect_ring(oracle.WL_RING_ROTATE if wl == "rotate" else oracle.WL_XORSHIFT, v0, R)
    np.testing.assert_array_equal(got, want)
    assert rc == 0 and d.device_status == 0 and d.cluster_used == 1
    if variant != 6:
        assert d.final_counter == (R * P) % oracle.counter_modulus(P)
    assert (st == cns.CNS_CTA_DONE).all()
    assert d.elapsed_ms < 1000.0
    # the same workspace, now with clusters: the base count R * 148 is a multiple of 37 clusters too
    if variant != 6:
        d, rc, got, st = run_ring(cns, HARD, AIV, code, P, v0, R, cluster_dim=4, variant=variant)
        assert rc == 0 and d.cluster_used == 4
        np.testing.assert_array_equal(got, want)


def test_launch_flags_outside_the_defined_bits_are_refused(cns):
    v0 = ci.ring_payload(3, 4, 4)
    d, rc, got, st = run_ring(cns, HARD, AIV, cns.CNS_WL_RING_ROTATE, 4, v0, 3, check=False, launch_flags=4)
    assert rc == cns.CNS_ERR_INVALID_VALUE


@pytest.mark.parametrize("mode", [SOFT, HARD])
def test_launch_without_the_cooperative_attribute(cns, mode):
    """The residency check alone (no cooperative attribute): exact, and the hard path keeps its clusters."""
    R = 3001
    v0 = ci.ring_payload(ci.SEED_RING_ROTATE, 148, 4)
    d, rc, got, st = run_ring(cns, mode, AIV, cns.CNS_WL_RING_ROTATE, 148, v0, R, variant=5,
                              launch_flags=cns.CNS_LAUNCH_NO_COOPERATIVE_ATTR)
    want, _ = expect_ring(oracle.WL_RING_ROTATE, v0, R)
    np.testing.assert_array_equal(got, want)
    assert rc == 0 and d.device_status == 0
    if mode == HARD:
        assert d.cluster_used == 2 and d.final_counter == R * 74


# --- the hard path's paired-mbarrier step (the guide's intra-block flags, §5.1) -------------

PAIRED = 1


@pytest.mark.parametrize("variant", [0, 2, 5, 6])
@pytest.mark.parametrize("C", [2, 4])
def test_paired_step_ring_rotate_148(cns, variant, C):
    """Members meet their cluster's rank 0 on shared-memory mbarriers; only rank 0 touches the counter."""
    R = 20001
    v0 = ci.ring_payload(ci.SEED_RING_ROTATE, 148, 4)
    d, rc, got, st = run_ring(cns, HARD, AIV, cns.CNS_WL_RING_ROTATE, 148, v0, R, cluster_dim=C, variant=variant,
                              hard_step=PAIRED)
    want, _ = expect_ring(oracle.WL_RING_ROTATE, v0, R)
    np.testing.assert_array_equal(got, want)
    assert rc == 0 and d.device_status == 0 and d.cluster_used == C
    if variant != FLIP:
        assert d.final_counter == (R * (148 // C)) % oracle.counter_modulus(148 // C)
    assert (st == cns.CNS_CTA_DONE).all()


def test_paired_step_mix_37x3_and_affine(cns):
    """MIX (37 groups of 1 AIC + 2 AIV CTAs, one cluster each) with the xorshift payload, and a ring-affine
    run with ragged rows, both against the oracle."""
    v0 = ci.ring_payload(ci.SEED_XORSHIFT, 111, 256)
    d, rc, got, st = run_ring(cns, HARD, MIX, cns.CNS_WL_XORSHIFT, 37, v0, 10000, ratio=2, hard_step=PAIRED)
    want, _ = expect_ring(oracle.WL_XORSHIFT, v0, 10000)
    np.testing.assert_array_equal(got, want)
    assert d.cluster_used == 3 and d.final_counter == 10000 * 37
    np.testing.assert_array_equal(st >> 8, (np.arange(111) % 3 == 0).astype(np.int32))
    v0 = ci.ring_payload(7, 16, 13)
    d, rc, got, st = run_ring(cns, HARD, AIV, cns.CNS_WL_RING_AFFINE, 16, v0, 301, cluster_dim=8, hard_step=PAIRED)
    want, _ = expect_ring(oracle.WL_RING_AFFINE, v0, 301)
    np.testing.assert_array_equal(got, want)
    assert d.cluster_used == 8 and d.final_counter == 301 * 2


def test_paired_step_jacobi(cns):
    u0 = ci.jacobi_field(200003)
    d, got = run_jacobi(cns, u0, 10, 64, mode=HARD, hard_step=PAIRED)
    want, _, _ = oracle.syncall_run_jacobi(u0, 10, 64)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("rounds", [1, 3, 6])
def test_paired_step_unzeroed_workspace_times_out(cns, rounds):
    """A garbled counter puts the clusters' rank-0 CTAs in different epochs: their bounded waits give up,
    each releases its members with the stop flag, and every CTA of a cluster reports the same outcome."""
    v0 = ci.ring_payload(3, 8, 4)
    d, rc, got, st = run_ring(cns, HARD, AIV, cns.CNS_WL_RING_AFFINE, 8, v0, rounds, garble=1, timeout_ms=300,
                              cluster_dim=4, check=False, hard_step=PAIRED)
    assert rc == cns.CNS_ERR_TIMEOUT and d.device_status == cns.CNS_ERR_TIMEOUT
    assert ((st & 0xFF) == cns.CNS_CTA_ABORTED).any()
    assert len(set((st[:4] & 0xFF).tolist())) == 1 and len(set((st[4:] & 0xFF).tolist())) == 1
    d, rc, got, st = run_ring(cns, HARD, AIV, cns.CNS_WL_RING_AFFINE, 8, v0, 5, cluster_dim=4, hard_step=PAIRED)
    want, _ = expect_ring(oracle.WL_RING_AFFINE, v0, 5)
    np.testing.assert_array_equal(got, want)


def test_paired_step_without_the_cluster_attribute(cns):
    """Clusters of one: rank 0 has no members and arrives for itself."""
    R = 3001
    v0 = ci.ring_payload(ci.SEED_RING_ROTATE, 148, 4)
    d, rc, got, st = run_ring(cns, HARD, AIV, cns.CNS_WL_RING_ROTATE, 148, v0, R, cluster_dim=4,
                              launch_flags=cns.CNS_LAUNCH_NO_CLUSTER_ATTR, hard_step=PAIRED)
    want, _ = expect_ring(oracle.WL_RING_ROTATE, v0, R)
    np.testing.assert_array_equal(got, want)
    assert rc == 0 and d.cluster_used == 1 and d.final_counter == (R * 148) % oracle.counter_modulus(148)


def test_paired_step_is_refused_where_it_has_no_meaning(cns):
    v0 = ci.ring_payload(3, 4, 4)
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_RING_ROTATE, 4, v0, 3, check=False, hard_step=PAIRED)
    assert rc == cns.CNS_ERR_INVALID_VALUE
    d, rc, got, st = run_ring(cns, HARD, AIV, cns.CNS_WL_RING_ROTATE, 4, v0, 3, check=False, hard_step=2)
    assert rc == cns.CNS_ERR_INVALID_VALUE


# --- sense-flip comparison variant (not the guide's arithmetic) ---------------------------

from oracle.protocol import flip_final_counter  # noqa: E402

FLIP = 6
SENSE = 1 << 31


@pytest.mark.parametrize("mode", [SOFT, HARD])
@pytest.mark.parametrize("start", [0, SENSE])
def test_sense_flip_ring_rotate_148(cns, mode, start):
    v0 = ci.ring_payload(ci.SEED_RING_ROTATE, 148, 4)
    d, rc, got, st = run_ring(cns, mode, AIV, cns.CNS_WL_RING_ROTATE, 148, v0, 20001, start=start, variant=FLIP)
    np.testing.assert_array_equal(got, np.roll(v0, -20001, axis=0))
    assert rc == 0 and d.device_status == 0 and (st == cns.CNS_CTA_DONE).all()
    assert d.final_counter == flip_final_counter(148, 20001, start=start) == start ^ SENSE


def test_sense_flip_affine_mix_and_jacobi(cns):
    import torch
    v0 = ci.ring_payload(ci.SEED_RING_AFFINE, 8, 256)
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_RING_AFFINE, 8, v0, 1000, variant=FLIP)
    want, _ = expect_ring(oracle.WL_RING_AFFINE, v0, 1000)
    np.testing.assert_array_equal(got, want)
    assert d.final_counter == 0
    v1 = ci.ring_payload(ci.SEED_XORSHIFT, 111, 256)
    d, rc, got, st = run_ring(cns, HARD, MIX, cns.CNS_WL_XORSHIFT, 37, v1, 2000, ratio=2, variant=FLIP)
    want, _ = expect_ring(oracle.WL_XORSHIFT, v1, 2000)
    np.testing.assert_array_equal(got, want)
    v2 = ci.ring_payload(ci.SEED_XORSHIFT, 64, 256)
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_XORSHIFT, 148, v2, 999, used=64, variant=FLIP)
    want, _ = expect_ring(oracle.WL_XORSHIFT, v2, 999)
    np.testing.assert_array_equal(got, want)
    assert d.final_counter == SENSE
    u0 = ci.jacobi_field(300007)
    b0 = to_dev_f32(u0)
    b1 = torch.zeros_like(b0)
    ws = cns.new_workspace()
    d, rc = cns.run_syncall(SOFT, AIV, cns.CNS_WL_JACOBI, 592, b0, b1, 8, elems=u0.size, workspace=ws, variant=FLIP)
    want, _, _ = oracle.syncall_run_jacobi(u0, 8, 592)
    np.testing.assert_array_equal(b0.cpu().numpy(), want)


@pytest.mark.parametrize("mode", [SOFT, HARD])
def test_sense_flip_rejects_a_foreign_count(cns, mode):
    """A workspace whose count has low bits no round of the scheme produces
    (left, say, by a run of another variant) stops the run with INVALID_VALUE."""
    v0 = ci.ring_payload(3, 148, 4)
    d, rc, got, st = run_ring(cns, mode, AIV, cns.CNS_WL_RING_ROTATE, 148, v0, 50, start=0x12345678, check=False,
                              variant=FLIP)
    assert rc == cns.CNS_ERR_INVALID_VALUE and d.device_status == cns.CNS_ERR_INVALID_VALUE
    assert ((st & 0xFF) == cns.CNS_CTA_ABORTED).all()


# --- arrival-only variant (the guide's bare contract), empty rounds only -------------------

@pytest.mark.parametrize("variant", [7, 8])
@pytest.mark.parametrize("mode", [SOFT, HARD])
@pytest.mark.parametrize("start_rounds", [(0, 10001), ("wrap", 500)])
def test_arrival_only_empty_rounds(cns, mode, start_rounds, variant):
    import torch
    start, R = start_rounds
    P = 148
    Pc = P if mode == SOFT else None
    ws = cns.new_workspace()
    d, rc = cns.run_syncall(mode, AIV, cns.CNS_WL_EMPTY, P, None, None, 1, workspace=ws, variant=variant)
    Pc = P if mode == SOFT else P // d.cluster_used
    M = oracle.counter_modulus(Pc)
    s0 = 0 if start == 0 else M - 3 * Pc
    ws = cns.new_workspace(start_value=s0)
    status = torch.zeros(P, dtype=torch.int32, device="cuda")
    d, rc = cns.run_syncall(mode, AIV, cns.CNS_WL_EMPTY, P, None, None, R, workspace=ws, cta_status=status,
                            variant=variant)
    assert rc == 0 and d.device_status == 0
    assert d.final_counter == (s0 + R * Pc) % M
    assert (status.cpu().numpy() == cns.CNS_CTA_DONE).all()


@pytest.mark.parametrize("variant", [7, 8])
def test_arrival_only_refused_with_a_payload(cns, variant):
    v0 = ci.ring_payload(3, 8, 4)
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_RING_AFFINE, 8, v0, 3, check=False, variant=variant)
    assert rc == cns.CNS_ERR_INVALID_VALUE


@pytest.mark.parametrize("mode", [SOFT, HARD])
def test_jacobi_unzeroed_workspace_times_out(cns, mode):
    """Jacobi sweeps (split phase on the soft path, fused on the hard path)
    with the counter garbled to 1: the bounded waits end the run with a timeout,
    and the device keeps working."""
    import torch
    u0 = ci.jacobi_field(100003, seed=5)
    b0 = to_dev_f32(u0)
    b1 = torch.zeros_like(b0)
    ws = cns.new_workspace()
    garble_counters(ws, 1)
    d, rc = cns.run_syncall(mode, AIV, cns.CNS_WL_JACOBI, 16, b0, b1, 6, elems=u0.size, workspace=ws,
                            timeout_ms=300, check=False, cluster_dim=4 if mode == HARD else 0)
    assert rc == cns.CNS_ERR_TIMEOUT and d.device_status == cns.CNS_ERR_TIMEOUT
    d, got = run_jacobi(cns, u0, 4, 16, mode=mode)
    want, _, _ = oracle.syncall_run_jacobi(u0, 4, 16)
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("mode", [SOFT, HARD])
def test_largest_resident_grid(cns, mode):
    """The most CTAs the GPU holds at once (32 per SM at 32 threads on the soft
    path; fewer in clusters): every participant arrives every round, and the
    xorshift ring comes out exact.  Larger grids are refused before launch."""
    import torch
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    # 32 is the hardware's CTA limit per SM; clusters allow fewer (the library
    # measured 8 per SM for clusters of 1 and 2, 4 for clusters of 4)
    for per_sm in (32, 16, 8, 4, 2, 1):
        P = sms * per_sm
        v0 = ci.ring_payload(77, P, 4)
        d, rc, got, st = run_ring(cns, mode, AIV, cns.CNS_WL_XORSHIFT, P, v0, 40, threads=32,
                                  cluster_dim=4 if mode == HARD else 0, check=False)
        if rc != cns.CNS_ERR_NOT_RESIDENT:
            break
    want, fc = expect_ring(oracle.WL_XORSHIFT, v0, 40)
    np.testing.assert_array_equal(got, want)
    assert rc == 0 and d.device_status == 0 and d.grid_ctas == P
    Pc = P if mode == SOFT else P // d.cluster_used
    assert d.final_counter == (40 * Pc) % oracle.counter_modulus(Pc)
    if per_sm == 32:   # a cluster more than 32 CTAs per SM can never be resident: refused before launch
        d, rc, got, st = run_ring(cns, mode, AIV, cns.CNS_WL_XORSHIFT, P + 4, ci.ring_payload(77, P + 4, 4), 1,
                                  threads=32, cluster_dim=4 if mode == HARD else 0, check=False)
        assert rc == cns.CNS_ERR_NOT_RESIDENT


def test_new_workspace_is_aligned_for_die_local_copies(cns):
    for _ in range(4):
        ws = cns.new_workspace()
        assert ws.data_ptr() % cns.CNS_SYNCALL_DIE_LOCAL_ALIGN == 0
        assert ws.numel() * 4 == cns.CNS_SYNCALL_WORKSPACE_MIRROR_BYTES
        ws = cns.new_workspace(mirror=False)
        assert ws.data_ptr() % cns.CNS_SYNCALL_DIE_LOCAL_ALIGN == 0
        assert ws.numel() * 4 == cns.CNS_SYNCALL_WORKSPACE_DIE_LOCAL_BYTES


# --- rounds on thread 0 alone, and the die-local payload copies ----------------------------

def _both_buffers(cns, wl, v0, R, variant, ws_bytes_kind, mode=SOFT, threads=256):
    import torch
    P = v0.shape[0]
    b0 = to_dev_u32(v0)
    b1 = torch.zeros_like(b0)
    if ws_bytes_kind == "mirror":
        ws = cns.new_workspace()
    elif ws_bytes_kind == "sized":
        ws = cns.new_workspace(participants=P, elems=v0.shape[1])
    elif ws_bytes_kind == "die_local":
        ws = cns.new_workspace(mirror=False)
    else:
        ws = cns.new_workspace(die_local=False)
    status = torch.zeros(P, dtype=torch.int32, device="cuda")
    d, rc = cns.run_syncall(mode, AIV, wl, P, b0, b1, R, elems=v0.shape[1], workspace=ws, cta_status=status,
                            variant=variant, threads=threads)
    assert rc == 0 and d.device_status == 0 and (status.cpu().numpy() == cns.CNS_CTA_DONE).all()
    M = oracle.counter_modulus(P)
    if mode == SOFT:
        assert d.final_counter == (R * P) % M
    return from_dev_u32(b0).reshape(P, -1), from_dev_u32(b1).reshape(P, -1)


WLS = {"rotate": (2, oracle.WL_RING_ROTATE), "affine": (1, oracle.WL_RING_AFFINE), "xorshift": (3, oracle.WL_XORSHIFT)}


@pytest.mark.parametrize("wl", sorted(WLS))
@pytest.mark.parametrize("P", [1, 2, 3, 148, 255, 256, 600])
@pytest.mark.parametrize("R", [1, 2, 3, 8, 1001])
def test_one_uint4_rings_through_the_payload_copies(cns, wl, P, R):
    """Rows of one uint4 on the die-local variant with a mirror-size workspace
    (per-die payload copies up to 255 participants; more run without them) and
    with one sized for the run (copies in as many 8 KB pairs as the rows
    need): both caller buffers end as the oracle's last two states -- buffer
    R & 1 holds round R's state and the other round R - 1's -- exactly as on a
    plain die-local workspace and on the guide's counter poll."""
    code, owl = WLS[wl]
    v0 = ci.ring_payload(31 + P, P, 4)
    states = {R: expect_ring(owl, v0, R)[0], R - 1: expect_ring(owl, v0, R - 1)[0] if R > 1 else v0}
    for kind, variant in (("mirror", 5), ("sized", 5), ("die_local", 5), ("plain", 0)):
        b0, b1 = _both_buffers(cns, code, v0, R, variant, kind)
        fin, prev = (b1, b0) if R & 1 else (b0, b1)
        np.testing.assert_array_equal(fin, states[R], err_msg=kind)
        np.testing.assert_array_equal(prev, states[R - 1], err_msg=kind)


@pytest.mark.parametrize("mode", [SOFT, HARD])
@pytest.mark.parametrize("wl", sorted(WLS))
@pytest.mark.parametrize("P,slots", [(1, 8), (3, 12), (8, 256), (111, 256), (5, 1020), (8, 1024), (4, 6)])
@pytest.mark.parametrize("R", [1, 2, 1001])
def test_longer_rows_through_the_payload_copies(cns, mode, wl, P, slots, R):
    """Rows of several uint4 (up to 1020 words: 255 uint4, one row per block pair) through the per-die
    copies on a workspace sized for them, on both paths: both caller buffers end as the oracle's last two
    states.  Rows of 1024 words, or of a length that is not a multiple of 4, run without copies."""
    code, owl = WLS[wl]
    v0 = ci.ring_payload(7 * P + slots, P, slots)
    states = {R: expect_ring(owl, v0, R)[0], R - 1: expect_ring(owl, v0, R - 1)[0] if R > 1 else v0}
    b0, b1 = _both_buffers(cns, code, v0, R, 5, "sized", mode=mode)
    fin, prev = (b1, b0) if R & 1 else (b0, b1)
    np.testing.assert_array_equal(fin, states[R])
    np.testing.assert_array_equal(prev, states[R - 1])


@pytest.mark.parametrize("mode", [SOFT, HARD])
@pytest.mark.parametrize("threads", [32, 64])
def test_rows_longer_than_the_cta_through_the_payload_copies(cns, mode, threads):
    """Rows of 255 uint4 moved by CTAs of 32 or 64 threads (each thread loops over several uint4 of the row)
    through the per-die copies: exact against the oracle."""
    v0 = ci.ring_payload(404, 6, 1020)
    want, _ = expect_ring(oracle.WL_XORSHIFT, v0, 77)
    b0, b1 = _both_buffers(cns, cns.CNS_WL_XORSHIFT, v0, 77, 5, "sized", mode=mode, threads=threads)
    np.testing.assert_array_equal(b1, want)


def test_subset_rows_through_the_payload_copies(cns):
    """64 participants of a 148-CTA launch with 1 KB rows through the per-die copies (the others idle):
    exact against the oracle, and the workspace sized for the 64 participants is enough."""
    v0 = ci.ring_payload(ci.SEED_XORSHIFT, 64, 256)
    import torch
    b0 = to_dev_u32(np.vstack([v0, np.zeros((84, 256), np.uint32)]))
    b1 = torch.zeros_like(b0)
    ws = cns.new_workspace(participants=64, elems=256)
    d, rc = cns.run_syncall(SOFT, AIV, cns.CNS_WL_XORSHIFT, 148, b0, b1, 1001, used_cores=64, elems=256,
                            workspace=ws, variant=5)
    want, fc = expect_ring(oracle.WL_XORSHIFT, v0, 1001)
    np.testing.assert_array_equal(from_dev_u32(b1).reshape(148, 256)[:64], want)
    assert rc == 0 and d.final_counter == fc


@pytest.mark.parametrize("variant", [0, 1, 2, 5, 6])
@pytest.mark.parametrize("slots", [0, 1, 4])
def test_solo_rounds_every_variant(cns, variant, slots):
    """Rounds that thread 0 runs alone (no payload, one word or one uint4 per
    row) with every data-carrying variant: exact against the oracle over 3001
    rounds of 148 participants."""
    v0 = ci.ring_payload(5, 148, slots)
    d, rc, got, st = run_ring(cns, SOFT, AIV, cns.CNS_WL_XORSHIFT, 148, v0, 3001, variant=variant)
    want, fc = expect_ring(oracle.WL_XORSHIFT, v0, 3001)
    np.testing.assert_array_equal(got, want)
    assert d.device_status == 0 and (st == cns.CNS_CTA_DONE).all()


@pytest.mark.parametrize("offset", [0, 1024, 4096, 5120, 128])
@pytest.mark.parametrize("mode", [SOFT, HARD])
def test_die_local_results_do_not_depend_on_placement(cns, offset, mode):
    """Die-local copies on a workspace at any 128-byte-aligned place: where the copies land decides only
    whether they share a die (the speed), never the result."""
    import torch
    big = torch.zeros(1 << 16, dtype=torch.int32, device="cuda")
    skip = ((-big.data_ptr()) % 8192 + offset) // 4
    ws = big[skip:skip + cns.CNS_SYNCALL_WORKSPACE_DIE_LOCAL_BYTES // 4]
    assert cns.syncall_workspace_init(ws, ws.numel() * 4, 0, None) == 0
    v0 = ci.ring_payload(ci.SEED_RING_ROTATE, 148, 4)
    b0 = to_dev_u32(v0)
    b1 = torch.zeros_like(b0)
    d, rc = cns.run_syncall(mode, AIV, cns.CNS_WL_RING_ROTATE, 148, b0, b1, 3001, elems=4, workspace=ws,
                            variant=cns.CNS_BARRIER_DIE_LOCAL)
    assert rc == 0 and d.device_status == 0
    np.testing.assert_array_equal(from_dev_u32(b1).reshape(148, 4), np.roll(v0, -3001, axis=0))
    assert d.final_counter == 3001 * (148 if mode == SOFT else 148 // d.cluster_used)


# --- the headline round with phase stamps (cns_probe_round_phases) -------------------------

def test_round_phase_probe(cns):
    """The stamped copy of the headline round computes the same ring as syncall_run; its stamps come in
    phase order for every CTA and round, and the bench's budget adds up to the mean round."""
    import torch
    import bench
    P, R, K = 148, 3001, 256
    v0 = ci.ring_payload(ci.SEED_RING_ROTATE, P, 4)
    b0 = to_dev_u32(v0)
    b1 = torch.zeros_like(b0)
    ws = cns.new_workspace()
    st = torch.zeros(K * P * 8, dtype=torch.int64, device="cuda")
    assert cns.cns_probe_round_phases(P, 256, R, K, b0, b1, ws, st) == 0
    torch.cuda.synchronize()
    want, fc = expect_ring(oracle.WL_RING_ROTATE, v0, R)
    np.testing.assert_array_equal(from_dev_u32(b1).reshape(P, 4), want)
    t = st.cpu().numpy().reshape(K, P, 8)
    assert (np.diff(t, axis=2) >= 0).all()
    assert (t[1:, :, 0] >= t[:-1, :, 7]).all()     # a round starts after the last one closed (the stamps'
    b = bench.round_budget(t)                      # bookkeeping in between)
    parts = sum(b[k] for k in bench.PHASES)
    assert abs(parts - b["round"]) < 1.0
    assert b["probe_bookkeeping"] >= 0.0
    assert abs(b["wait_for_last_arrival"] + b["wait_landing_and_detection"] - b["wait"]) < 1.0
    assert 100.0 < b["round"] < 100000.0
    # the same on a workspace without room for the payload copies (the caller's buffers every round)
    ws8 = cns.new_workspace(mirror=False)
    b0.copy_(to_dev_u32(v0))
    assert cns.cns_probe_round_phases(P, 256, R, K, b0, b1, ws8, st) == 0
    np.testing.assert_array_equal(from_dev_u32(b1).reshape(P, 4), want)
    # bad arguments are refused before any launch
    assert cns.cns_probe_round_phases(P, 256, 10, 20, b0, b1, ws, st) == cns.CNS_ERR_INVALID_VALUE
    assert cns.cns_probe_round_phases(P, 256, R, 2000, b0, b1, ws, st) == cns.CNS_ERR_INVALID_VALUE


def test_release_fence_probe(cns):
    """The fence-cost probe runs, refuses a misaligned region, and finds a release after a store on the other
    die dearer than one after a store on the SM's own die (its two blocks sit on different dies)."""
    import torch
    import bench
    f = bench.probe_release_fence(cns, torch, iters=300)
    assert 0 < f["after_nothing"] < f["after_a_store_on_the_other_die"]
    assert f["after_a_store_on_its_die"] < f["after_a_store_on_the_other_die"]
    raw = torch.zeros(4096, dtype=torch.int32, device="cuda")
    off = ((-raw.data_ptr()) % 8192 + 4096) // 4
    out = torch.zeros(3, dtype=torch.int64, device="cuda")
    assert cns.cns_probe_release_fence(raw[off:], 10, out) == cns.CNS_ERR_INVALID_VALUE
    assert cns.cns_probe_release_fence(raw, 0, out) == cns.CNS_ERR_INVALID_VALUE   # no samples


# --- the run captured into a CUDA graph --------------------------------------------------

@pytest.mark.parametrize("mode,variant,wl,P,slots", [
    (SOFT, 5, "rotate", 148, 4),        # the headline's solo rounds through the per-die copies
    (SOFT, 5, "xorshift", 64, 256),     # 1 KB rows through the copies, every thread moving them
    (SOFT, 0, "affine", 8, 256),        # the guide's counter poll, no copies
    (HARD, 5, "rotate", 148, 4),        # clusters of 2, one arrival per cluster
])
def test_syncall_replayed_from_a_cuda_graph(cns, mode, variant, wl, P, slots):
    """syncall_run captured once into a CUDA graph and replayed with a new payload in buf0 each time:
    every replay's result against the oracle, and the counter carrying on from replay to replay."""
    import torch
    wl_c = {"rotate": cns.CNS_WL_RING_ROTATE, "xorshift": cns.CNS_WL_XORSHIFT, "affine": cns.CNS_WL_RING_AFFINE}[wl]
    wl_o = {"rotate": oracle.WL_RING_ROTATE, "xorshift": oracle.WL_XORSHIFT, "affine": oracle.WL_RING_AFFINE}[wl]
    R = 1001
    payloads = [ci.ring_payload(seed, P, slots) for seed in (61, 62, 63)]
    b0 = to_dev_u32(payloads[0])
    b1 = torch.zeros_like(b0)
    ws = cns.new_workspace(participants=P, elems=slots)
    side = torch.cuda.Stream()

    def call():
        cns.run_syncall(mode, AIV, wl_c, P, b0, b1, R, elems=slots, workspace=ws, variant=variant, sync=False,
                        stream=torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        call()
    runs = 1
    for v in (payloads[1], payloads[2], payloads[0]):
        b0.copy_(to_dev_u32(v))
        g.replay()
        torch.cuda.synchronize()
        runs += 1
        want, _ = expect_ring(wl_o, v, R)
        np.testing.assert_array_equal(from_dev_u32(b1).reshape(P, slots), want)
        rc, soft, hard, st = cns.syncall_read_workspace(ws)
        assert rc == 0 and st == 0
        arrivals = P if mode == SOFT else P // 2
        counter = soft if mode == SOFT else hard
        assert counter == (runs * R * arrivals) % oracle.counter_modulus(arrivals)
