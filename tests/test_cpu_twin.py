"""The multithreaded CPU timing twin computes what the sequential oracle
computes: ring rounds, Jacobi sweeps (bit for bit, the same fp32 expression),
and the pipeline's checksums, for several thread counts."""
import numpy as np
import pytest

import cns_inputs as ci
import oracle
from oracle import twin


@pytest.mark.parametrize("wl", [twin.RING_AFFINE, twin.RING_ROTATE, twin.XORSHIFT])
@pytest.mark.parametrize("P,slots,rounds,threads", [(8, 256, 50, 3), (148, 4, 37, 4), (5, 7, 11, 8), (1, 3, 4, 2)])
def test_twin_ring_matches_oracle(wl, P, slots, rounds, threads):
    v0 = ci.ring_payload(ci.SEED_RING_ROTATE, P, slots)
    got, sec, fc = twin.syncall_ring(wl, v0, rounds, threads)
    want, _, rc = oracle.syncall_run_ring(wl, v0, rounds)
    assert rc == oracle.OK
    np.testing.assert_array_equal(got, want)
    assert fc == rounds * min(threads, P) and sec >= 0


@pytest.mark.parametrize("n,sweeps,threads", [(1000, 20, 3), (4097, 7, 4), (2, 3, 2), (1, 2, 1), (33, 4, 8)])
def test_twin_jacobi_matches_oracle(n, sweeps, threads):
    u0 = ci.jacobi_field(n, seed=77)
    got, sec = twin.jacobi(u0, sweeps, threads)
    want, _, rc = oracle.syncall_run_jacobi(u0, sweeps, 4)
    assert rc == oracle.OK
    np.testing.assert_array_equal(got, want)


@pytest.mark.parametrize("areas", [1, 2])
@pytest.mark.parametrize("tiles,tile_words,rounds", [(64, 8, 5), (7, 12, 9), (1, 4, 3), (300, 16, 40)])
def test_twin_pipeline_matches_oracle(tiles, tile_words, rounds, areas):
    cs, sec = twin.pipeline(tiles, tile_words, rounds, areas)
    want, _ = oracle.pipeline(tiles, tile_words, rounds)
    np.testing.assert_array_equal(cs, want)


def test_twin_rejects_bad_arguments():
    with pytest.raises(RuntimeError):
        twin.syncall_ring(9, np.zeros((2, 2), np.uint32), 1, 1)
    with pytest.raises(RuntimeError):
        twin.pipeline(0, 4, 1)
    with pytest.raises(RuntimeError):
        twin.pipeline(4, 4, 1, areas=3)
