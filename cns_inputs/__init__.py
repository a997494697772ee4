"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module draws random numbers and nothing else: it holds none of the
barrier, payload or counted-notify arithmetic.  Both the CPU oracle and the
CUDA path read the arrays made here, so a parity test compares the two on
identical data.

Generator: SplitMix64 (G. L. Steele, D. Lea, C. H. Flood, "Fast splittable
pseudorandom number generators", OOPSLA 2014), in the widely used form with
the golden-ratio increment 0x9E3779B97F4A7C15 and the output mix
z ^= z>>30; z *= 0xBF58476D1CE4E5B9; z ^= z>>27; z *= 0x94D049BB133111EB;
z ^= z>>31.  Element i of a stream with seed s is the output for the state
s + (i+1)*increment, so any slice can be regenerated without the prefix.
"""
from __future__ import annotations

import numpy as np

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)

# Per-workload seeds.
SEED_RING_AFFINE = 0xC0FFEE01
SEED_RING_ROTATE = 0xC0FFEE02
SEED_XORSHIFT = 0xC0FFEE03
SEED_JACOBI = 0xC0FFEE04
SEED_NOTIFY_OPS = 0xC0FFEE05


def splitmix64(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """n consecutive SplitMix64 outputs (uint64) of the stream `seed`, from index `offset`."""
    if n < 0:
        raise ValueError("n must be >= 0")
    idx = np.arange(offset + 1, offset + n + 1, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * _GAMMA
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
        z = z ^ (z >> np.uint64(31))
    return z


def u32_uniform(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Uniform uint32 over [0, 2^32): the high 32 bits of each SplitMix64 output."""
    return (splitmix64(seed, n, offset) >> np.uint64(32)).astype(np.uint32)


def f32_uniform_pm1(seed: int, n: int, offset: int = 0) -> np.ndarray:
    """Uniform float32 on [-1, 1): ((x >> 40) * 2^-24) * 2 - 1, every step exact in fp32."""
    top24 = (splitmix64(seed, n, offset) >> np.uint64(40)).astype(np.float32)
    return (top24 * np.float32(2.0 ** -24)) * np.float32(2.0) - np.float32(1.0)


def ring_payload(seed: int, participants: int, slots: int) -> np.ndarray:
    """[participants, slots] uint32 payload, seeded uniform."""
    return u32_uniform(seed, participants * slots).reshape(participants, slots)


def jacobi_field(n: int, seed: int = SEED_JACOBI) -> np.ndarray:
    """Length-n float32 field, seeded U[-1, 1)."""
    return f32_uniform_pm1(seed, n)


# Counted-notify operation stream --------------------------------------------
#
# One op is four uint32 words: kind (0 = record, 1 = try-wait), mode, value,
# is_clear.  Record modes are drawn from {0, 1, 2, 4}, wait modes from 0..4.
OP_RECORD = 0
OP_WAIT = 1
RECORD_MODES = np.array([0, 1, 2, 4], dtype=np.uint32)


def notify_ops(n: int, seed: int = SEED_NOTIFY_OPS) -> np.ndarray:
    """[n, 4] uint32 op stream for the counted-notify state machine.

    kind: record or try-wait, 1/2 each.  mode: uniform over the valid set of
    that kind.  value: 1/2 small in [0, 16), 1/4 uniform uint32, 1/4 a bit
    pattern (a single bit, a low mask 2^k - 1, or the complement of a single
    bit).  is_clear: 1 with probability 1/8, on waits only.  Small values keep
    the counter near values that the waits compare against, so every wait
    mode is satisfied for part of the stream and not for the rest.
    """
    r = splitmix64(seed, 6 * n).reshape(n, 6) if n else np.zeros((0, 6), np.uint64)
    lo32 = np.uint64(0xFFFFFFFF)
    kind = (r[:, 0] >> np.uint64(63)).astype(np.uint32)
    rec_mode = RECORD_MODES[(r[:, 1] >> np.uint64(62)).astype(np.int64)]
    wait_mode = ((r[:, 1] & lo32) % np.uint64(5)).astype(np.uint32)
    mode = np.where(kind == OP_RECORD, rec_mode, wait_mode).astype(np.uint32)

    cls = (r[:, 2] >> np.uint64(62)).astype(np.int64)          # 0,1 small; 2 uniform; 3 pattern
    small = (r[:, 3] & np.uint64(15)).astype(np.uint32)
    uni = (r[:, 3] >> np.uint64(32)).astype(np.uint32)
    k = ((r[:, 4] >> np.uint64(8)) & np.uint64(31)).astype(np.uint32)
    pat_kind = (r[:, 4] & np.uint64(3)).astype(np.int64)
    one = np.uint32(1)
    single = np.left_shift(one, k, dtype=np.uint32)
    lowmask = np.where(k == 0, np.uint32(0xFFFFFFFF), single - one).astype(np.uint32)
    notbit = np.bitwise_not(single).astype(np.uint32)
    pattern = np.where(pat_kind == 0, single, np.where(pat_kind == 1, lowmask, np.where(pat_kind == 2, notbit, single)))
    value = np.where(cls <= 1, small, np.where(cls == 2, uni, pattern)).astype(np.uint32)

    clear = ((r[:, 5] >> np.uint64(61)) == np.uint64(0)).astype(np.uint32)
    clear = np.where(kind == OP_WAIT, clear, np.uint32(0)).astype(np.uint32)
    return np.stack([kind, mode, value, clear], axis=1).astype(np.uint32)


def sample_indices(seed: int, n_total: int, k: int) -> np.ndarray:
    """k sorted distinct-ish indices in [0, n_total), plus both ends, for sampled checks."""
    if n_total <= 0:
        return np.zeros(0, dtype=np.int64)
    draws = (splitmix64(seed ^ 0x5A5A5A5A, k) % np.uint64(n_total)).astype(np.int64)
    ends = np.array([0, n_total - 1], dtype=np.int64)
    return np.unique(np.concatenate([draws, ends]))
