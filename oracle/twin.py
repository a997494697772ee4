"""Multithreaded CPU timing twin (``cns_cpu_twin.c``): the SYNCALL ring and
Jacobi rounds on T host threads with the pages' epoch barrier, and the
counted-notify pipeline on two host threads.

TEST AND BASELINE INFRASTRUCTURE ONLY: used by the CPU tests (checked there
against the sequential oracle) and by the benchmark's CPU-baseline leg, never
by the product package.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "cns_cpu_twin.c")
_LIB = os.path.join(_HERE, "libcns_cpu_twin.so")
_lock = threading.Lock()
_lib = None

RING_AFFINE, RING_ROTATE, XORSHIFT = 1, 2, 3


def build(force: bool = False) -> str:
    """Compile cns_cpu_twin.c into libcns_cpu_twin.so (gcc, -O2, pthreads, no FP contraction)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-pthread", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
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
            u32, i64, i32, vp = ctypes.c_uint32, ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
            dp = ctypes.POINTER(ctypes.c_double)
            up = ctypes.POINTER(ctypes.c_uint32)
            L.twin_syncall_ring.argtypes = [i32, u32, i64, i32, vp, vp, i64, dp, up]
            L.twin_syncall_ring.restype = i32
            L.twin_jacobi.argtypes = [vp, vp, i64, i64, i32, dp]
            L.twin_jacobi.restype = i32
            L.twin_pipeline.argtypes = [i64, i32, i64, i32, vp, dp]
            L.twin_pipeline.restype = i32
            _lib = L
    return _lib


def host_threads() -> int:
    """Threads the twin uses: every core this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def syncall_ring(wl: int, v0: np.ndarray, rounds: int, threads: int):
    """(final [P][slots] uint32, seconds, final barrier count) of `rounds` ring rounds."""
    v0 = np.ascontiguousarray(v0, dtype=np.uint32)
    P, slots = v0.shape
    b = [v0.copy(), np.zeros_like(v0)]
    sec = ctypes.c_double()
    fc = ctypes.c_uint32()
    rc = lib().twin_syncall_ring(wl, P, rounds, threads, b[0].ctypes.data, b[1].ctypes.data, slots,
                                 ctypes.byref(sec), ctypes.byref(fc))
    if rc != 0:
        raise RuntimeError(f"twin_syncall_ring: {rc}")
    return b[rounds & 1], sec.value, fc.value


def jacobi(u0: np.ndarray, sweeps: int, threads: int):
    """(field after `sweeps` sweeps, seconds)."""
    u0 = np.ascontiguousarray(u0, dtype=np.float32)
    b = [u0.copy(), np.empty_like(u0)]
    sec = ctypes.c_double()
    rc = lib().twin_jacobi(b[0].ctypes.data, b[1].ctypes.data, u0.size, sweeps, threads, ctypes.byref(sec))
    if rc != 0:
        raise RuntimeError(f"twin_jacobi: {rc}")
    return b[sweeps & 1], sec.value


def pipeline(tiles: int, tile_words: int, rounds: int, areas: int = 1):
    """(checksums[rounds], seconds) of the two-thread pipeline over `areas` tile areas."""
    cs = np.zeros(rounds, dtype=np.uint32)
    sec = ctypes.c_double()
    rc = lib().twin_pipeline(tiles, tile_words, rounds, areas, cs.ctypes.data, ctypes.byref(sec))
    if rc != 0:
        raise RuntimeError(f"twin_pipeline: {rc}")
    return cs, sec.value
