"""CPU oracle for the counted-notify / SYNCALL hot path.

TEST INFRASTRUCTURE ONLY: imported by the tests, by ``__graft_entry__.smoke``
and by the benchmark's CPU-baseline leg, never by the product package.  The
arithmetic lives in ``cns_oracle.c`` (plain sequential C) and in
``protocol.py`` (the barrier-protocol interleaving explorer); this module
builds the C part with gcc and wraps it for numpy arrays.

Parity status of each function (what pins it; see tests/test_oracle_*.py):
  epoch_target / target_mod / reached_mod   closed form + all-interleaving
                                            brute force (protocol.py)
  syncall_run (ring workloads)              closed forms (affine, rotate),
                                            xorshift inverse + hand value
  syncall_run (Jacobi), jacobi_points       fixed points, Fourier-mode decay,
                                            point sampler vs full sweep
  cnt_record / cnt_wait_satisfied           hand-built truth table (golden)
  cnt_statemachine                          golden sequences + per-op table
  pipeline                                  closed-form checksum
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cns_oracle.c")
_LIB = os.path.join(_HERE, "liboracle_cns.so")
_lock = threading.Lock()
_lib = None

WL_EMPTY, WL_RING_AFFINE, WL_RING_ROTATE, WL_XORSHIFT, WL_JACOBI = 0, 1, 2, 3, 4
REC_SET, REC_ADD, REC_OR, REC_AND = 0, 1, 2, 4
WAIT_LESS, WAIT_EQUAL, WAIT_BIGGER, WAIT_BGE, WAIT_MASK = 0, 1, 2, 3, 4
OUT_WAIT_HELD, OUT_WAIT_RELEASED, OUT_RECORD, OUT_INVALID = 0, 1, 2, 3
OK, DEADLOCK, BAD_ARG = 0, 1, 2


def build(force: bool = False) -> str:
    """Compile cns_oracle.c into liboracle_cns.so (gcc, -O2, no FP contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
           "-Wall", "-Wextra", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def lib() -> ctypes.CDLL:
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = ctypes.CDLL(_LIB)
            u32, u64, i64, i32 = ctypes.c_uint32, ctypes.c_uint64, ctypes.c_int64, ctypes.c_int
            vp = ctypes.c_void_p
            L.oracle_epoch_target.argtypes = [u32, u32]
            L.oracle_epoch_target.restype = u32
            L.oracle_counter_modulus.argtypes = [u32]
            L.oracle_counter_modulus.restype = u64
            L.oracle_arrive_mod.argtypes = [u32, u64]
            L.oracle_arrive_mod.restype = u32
            L.oracle_target_mod.argtypes = [u32, u32, u64]
            L.oracle_target_mod.restype = u32
            L.oracle_reached_mod.argtypes = [u32, u32, u32, u64]
            L.oracle_reached_mod.restype = i32
            L.oracle_xorshift32.argtypes = [u32]
            L.oracle_xorshift32.restype = u32
            L.oracle_syncall_run.argtypes = [i32, u32, u64, u32, vp, i64, vp, i64, vp]
            L.oracle_syncall_run.restype = i32
            L.oracle_jacobi_points.argtypes = [vp, i64, i64, vp, i64, vp]
            L.oracle_jacobi_points.restype = i32
            L.oracle_cnt_record.argtypes = [u32, u32, u32, vp]
            L.oracle_cnt_record.restype = i32
            L.oracle_cnt_wait_satisfied.argtypes = [u32, u32, u32]
            L.oracle_cnt_wait_satisfied.restype = i32
            L.oracle_cnt_statemachine.argtypes = [vp, i64, u32, vp, vp]
            L.oracle_cnt_statemachine.restype = None
            L.oracle_pipeline_word.argtypes = [i64, u64]
            L.oracle_pipeline_word.restype = u32
            L.oracle_pipeline.argtypes = [i64, i64, i64, vp, vp]
            L.oracle_pipeline.restype = None
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p) if a is not None and a.size else None


# SYNCALL barrier arithmetic -------------------------------------------------

def epoch_target(before: int, P: int) -> int:
    return lib().oracle_epoch_target(before, P)


def counter_modulus(P: int) -> int:
    return lib().oracle_counter_modulus(P)


def arrive_mod(c: int, M: int) -> int:
    return lib().oracle_arrive_mod(c, M)


def target_mod(before: int, P: int, M: int) -> int:
    return lib().oracle_target_mod(before, P, M)


def reached_mod(cur: int, target: int, P: int, M: int) -> bool:
    return bool(lib().oracle_reached_mod(cur, target, P, M))


def xorshift32(x: int) -> int:
    return lib().oracle_xorshift32(x)


def syncall_run_ring(workload: int, state: np.ndarray, rounds: int, start: int = 0):
    """Run `rounds` payload+barrier rounds on a [P, slots] uint32 ring state.

    Returns (final_state, final_counter, status)."""
    st = np.ascontiguousarray(state, dtype=np.uint32).copy()
    P, slots = st.shape
    fc = np.zeros(1, dtype=np.uint32)
    rc = lib().oracle_syncall_run(workload, P, rounds, start, _ptr(st), slots, None, 0, _ptr(fc))
    return st, int(fc[0]), rc


def syncall_run_empty(P: int, rounds: int, start: int = 0):
    fc = np.zeros(1, dtype=np.uint32)
    rc = lib().oracle_syncall_run(WL_EMPTY, P, rounds, start, None, 0, None, 0, _ptr(fc))
    return int(fc[0]), rc


def syncall_run_jacobi(u0: np.ndarray, sweeps: int, P: int, start: int = 0):
    """Run `sweeps` Jacobi sweeps, a P-participant barrier after each.

    Returns (field, final_counter, status)."""
    u = np.ascontiguousarray(u0, dtype=np.float32).copy()
    fc = np.zeros(1, dtype=np.uint32)
    rc = lib().oracle_syncall_run(WL_JACOBI, P, sweeps, start, None, 0, _ptr(u), u.size, _ptr(fc))
    return u, int(fc[0]), rc


def jacobi_points(u0: np.ndarray, sweeps: int, idx: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(u0, dtype=np.float32)
    ix = np.ascontiguousarray(idx, dtype=np.int64)
    out = np.zeros(ix.size, dtype=np.float32)
    rc = lib().oracle_jacobi_points(_ptr(u), u.size, sweeps, _ptr(ix), ix.size, _ptr(out))
    if rc != OK:
        raise ValueError("oracle_jacobi_points: bad argument")
    return out


# CntNotify --------------------------------------------------------------------

def cnt_record(c: int, mode: int, v: int):
    """(new_count, ok) for one record."""
    out = ctypes.c_uint32(0)
    rc = lib().oracle_cnt_record(c, mode, v, ctypes.byref(out))
    return int(out.value), rc == 0


def cnt_wait_satisfied(c: int, mode: int, v: int) -> int:
    return lib().oracle_cnt_wait_satisfied(c, mode, v)


def cnt_statemachine(ops: np.ndarray, init: int = 0):
    """Apply an [n, 4] op stream. Returns (trace [n, 2] uint32, final count)."""
    o = np.ascontiguousarray(ops, dtype=np.uint32).reshape(-1, 4)
    n = o.shape[0]
    trace = np.zeros((n, 2), dtype=np.uint32)
    fin = np.zeros(1, dtype=np.uint32)
    lib().oracle_cnt_statemachine(_ptr(o), n, init, _ptr(trace), _ptr(fin))
    return trace, int(fin[0])


def pipeline_word(w: int, r: int) -> int:
    return lib().oracle_pipeline_word(w, r)


def pipeline(tiles: int, tile_words: int, rounds: int):
    """(checksums[rounds], release_counts[rounds]) of the two-stream pipeline."""
    cs = np.zeros(rounds, dtype=np.uint32)
    ct = np.zeros(rounds, dtype=np.uint32)
    lib().oracle_pipeline(tiles, tile_words, rounds, _ptr(cs), _ptr(ct))
    return cs, ct
