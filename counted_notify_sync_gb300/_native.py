"""ctypes binding of libcns (include/cns.h): argument marshalling only.

Every function here keeps the C name and returns the C status code; tensors
are passed as their device (or pinned host) addresses and streams as their
cudaStream_t.  All work happens in the CUDA library.  If libcns.so is absent
the first call raises: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os
import threading
from ctypes import (POINTER, Structure, c_char_p, c_double, c_float, c_int, c_int32, c_int64, c_size_t, c_uint8, c_uint32,
                    c_uint64, c_void_p)

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libcns.so")

# --- constants (cns.h) ---------------------------------------------------------
CNS_SUCCESS = 0
CNS_ERR_INVALID_VALUE = 1
CNS_ERR_NULL_PTR = 2
CNS_ERR_INVALID_HANDLE = 3
CNS_ERR_RESOURCE = 4
CNS_ERR_TIMEOUT = 5
CNS_ERR_NOT_RESIDENT = 6
CNS_ERR_CUDA = 7
CNS_ERR_ARCH = 8
CNS_ERR_NO_PEER_ACCESS = 9

CNS_SYNCALL_HARD = 0
CNS_SYNCALL_SOFT = 1
CNS_AIV_ONLY = 0
CNS_AIC_ONLY = 1
CNS_MIX = 2
CNS_WL_EMPTY = 0
CNS_WL_RING_AFFINE = 1
CNS_WL_RING_ROTATE = 2
CNS_WL_XORSHIFT = 3
CNS_WL_JACOBI = 4
CNS_SYNCALL_LINE_BYTES = 128
CNS_SYNCALL_WORKSPACE_BYTES = 512
CNS_BARRIER_COUNTER_ACQUIRE = 0
CNS_BARRIER_LAST_SKIPS = 1
CNS_BARRIER_RELAXED_POLL = 2
CNS_BARRIER_BACKOFF = 3
CNS_BARRIER_FLAG_BROADCAST = 4
CNS_BARRIER_DIE_LOCAL = 5
CNS_BARRIER_SENSE_FLIP = 6
CNS_BARRIER_ARRIVAL_ONLY = 7
CNS_BARRIER_ARRIVAL_ONLY_DIE_LOCAL = 8
CNS_SYNCALL_REPLICA_OFFSET = 4096
CNS_SYNCALL_WORKSPACE_DIE_LOCAL_BYTES = 8192
CNS_SYNCALL_DIE_LOCAL_ALIGN = 8192
CNS_SYNCALL_WORKSPACE_MIRROR_BYTES = 24576
CNS_SYNCALL_MIRROR_MAX_P = 255
CNS_CTA_DONE = 1
CNS_CTA_IDLE = 2
CNS_CTA_ABORTED = 4
CNS_LAUNCH_NO_CLUSTER_ATTR = 1
CNS_LAUNCH_NO_COOPERATIVE_ATTR = 2
CNS_HARD_STEP_CLUSTER_BARRIER = 0
CNS_HARD_STEP_PAIRED_MBARRIER = 1

CNS_REC_SET = 0
CNS_REC_ADD = 1
CNS_REC_BIT_OR = 2
CNS_REC_BIT_AND = 4
CNS_WAIT_LESS = 0
CNS_WAIT_EQUAL = 1
CNS_WAIT_BIGGER = 2
CNS_WAIT_BIGGER_OR_EQUAL = 3
CNS_WAIT_EQUAL_WITH_BITMASK = 4
CNS_OUT_WAIT_HELD = 0
CNS_OUT_WAIT_RELEASED = 1
CNS_OUT_RECORD = 2
CNS_OUT_INVALID = 3
CNS_PIPE_WAIT_STREAM = 0
CNS_PIPE_WAIT_IN_KERNEL = 1


class CnsError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{what}: {error_string(code)} ({code})" if what else f"{error_string(code)} ({code})")


# --- structs (layout mirrors cns.h) ------------------------------------------------
class SyncallData(Structure):
    _fields_ = [
        ("workload", c_int32), ("launch_ctas", c_int32), ("threads", c_int32), ("cluster_dim", c_int32),
        ("buf0_dev", c_void_p), ("buf1_dev", c_void_p), ("elems", c_int64), ("workspace_dev", c_void_p),
        ("cta_status_dev", c_void_p), ("stream", c_void_p), ("timeout_ms", c_uint32), ("sync", c_int32),
        ("host_in", c_void_p), ("host_out", c_void_p), ("elapsed_ms", c_float), ("final_counter", c_uint32),
        ("device_status", c_int32), ("grid_ctas", c_int32), ("participants", c_int32), ("cluster_used", c_int32),
        ("barrier_variant", c_int32), ("workspace_bytes", c_uint32), ("launch_flags", c_uint32), ("hard_step", c_int32),
    ]


class RecordInfo(Structure):
    _fields_ = [("mode", c_int32), ("value", c_uint32)]


class WaitInfo(Structure):
    _fields_ = [("mode", c_int32), ("value", c_uint32), ("timeout", c_uint32), ("is_clear", c_uint8),
                ("rev", c_uint8 * 3)]


class Pipeline(Structure):
    _fields_ = [
        ("done", c_void_p), ("ack", c_void_p), ("tiles_dev", c_void_p), ("checksums_dev", c_void_p),
        ("released_dev", c_void_p), ("tiles", c_int64), ("tile_words", c_int32), ("producer_ctas", c_int32),
        ("rounds", c_int64), ("producer_stream", c_void_p), ("consumer_stream", c_void_p), ("timeout_s", c_uint32),
        ("sync", c_int32), ("elapsed_ms", c_float), ("producer_ms", c_float), ("device_status", c_int32),
        ("consumer_ctas", c_int32), ("areas", c_int32), ("consumer_wait", c_int32),
    ]


_SIGS = {
    "syncall_workspace_init": (c_int, [c_void_p, c_size_t, c_uint32, c_void_p]),
    "syncall_workspace_bytes": (c_int, [c_int32, c_int64, POINTER(c_size_t)]),
    "syncall_run": (c_int, [c_int, c_int, c_int32, c_int32, c_int64, POINTER(SyncallData)]),
    "syncall_read_workspace": (c_int, [c_void_p, c_void_p, POINTER(c_uint32), POINTER(c_uint32), POINTER(c_int32)]),
    "cntnotify_create": (c_int, [POINTER(c_void_p), c_uint64]),
    "cntnotify_record": (c_int, [c_void_p, c_void_p, POINTER(RecordInfo)]),
    "cntnotify_wait_with_timeout": (c_int, [c_void_p, c_void_p, POINTER(WaitInfo)]),
    "cntnotify_reset": (c_int, [c_void_p, c_void_p]),
    "cntnotify_get_id": (c_int, [c_void_p, POINTER(c_uint32)]),
    "cntnotify_destroy": (c_int, [c_void_p]),
    "cntnotify_get_device_ptr": (c_int, [c_void_p, POINTER(c_void_p)]),
    "cntnotify_query_status": (c_int, [c_void_p, POINTER(c_int32), POINTER(c_uint32)]),
    "cntnotify_enable_peer": (c_int, [c_void_p, c_int]),
    "cns_statemachine_scratch_bytes": (c_size_t, [c_int64]),
    "cns_statemachine_run": (c_int, [c_void_p, c_int64, c_uint32, c_void_p, c_void_p, c_void_p, c_size_t, c_void_p]),
    "cns_statemachine_run_noalloc": (c_int, [c_void_p, c_int64, c_uint32, c_void_p, c_void_p, c_void_p]),
    "cns_pipeline_run": (c_int, [POINTER(Pipeline)]),
    "cns_probe_atomic_rtt": (c_int, [c_int, c_int32, c_int32, c_int32, c_void_p, c_void_p, c_void_p]),
    "cns_probe_same_address_throughput": (c_int, [c_int32, c_int32, c_int32, c_void_p, c_void_p]),
    "cns_probe_grid_sync": (c_int, [c_int32, c_int32, c_int64, c_void_p, c_void_p, c_void_p]),
    "cns_probe_op_chain": (c_int, [c_void_p, c_int32, c_void_p, c_void_p]),
    "cns_probe_launch_cost": (c_int, [c_int32, c_int32, POINTER(c_double), c_void_p]),
    "cns_probe_release_fence": (c_int, [c_void_p, c_int32, c_void_p, c_void_p]),
    "cns_probe_notify_pingpong": (c_int, [c_int, c_int32, c_void_p, c_void_p, c_void_p]),
    "cns_probe_round_phases": (c_int, [c_int32, c_int32, c_int64, c_int32, c_void_p, c_void_p, c_void_p, c_size_t,
                                       c_void_p, c_void_p]),
    "cns_version": (c_int, [POINTER(c_int32), POINTER(c_int32)]),
    "cns_error_string": (c_char_p, [c_int]),
}

_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded libcns.so, with signatures set.  Raises if it was not built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"libcns.so is not built ({LIB_PATH}); run `python -m counted_notify_sync_gb300.builder`")
            L = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in _SIGS.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def exported_names():
    return list(_SIGS)


# --- marshalling helpers -------------------------------------------------------------

def ptr(x) -> int | None:
    """Address of a tensor / numpy array / int / None."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    if hasattr(x, "ctypes"):
        return x.ctypes.data
    raise TypeError(f"cannot take the address of {type(x)}")


def stream_handle(s) -> int | None:
    """cudaStream_t of a torch stream, an int handle, or None (default stream)."""
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


def error_string(code: int) -> str:
    try:
        return lib().cns_error_string(code).decode()
    except RuntimeError:
        return f"error {code}"


def check(code: int, what: str = "") -> None:
    if code != CNS_SUCCESS:
        raise CnsError(code, what)


# --- the C entry points, same names ----------------------------------------------------

def syncall_workspace_init(ws, nbytes: int, start_value: int = 0, stream=None) -> int:
    return lib().syncall_workspace_init(ptr(ws), nbytes, start_value, stream_handle(stream))


def syncall_run(mode: int, core_type: int, used_cores: int, aiv_ratio: int, rounds: int, data: SyncallData) -> int:
    return lib().syncall_run(mode, core_type, used_cores, aiv_ratio, rounds, ctypes.byref(data))


def syncall_read_workspace(ws, stream=None):
    """(code, soft_counter, hard_counter, status)"""
    sc, hc, st = c_uint32(0), c_uint32(0), c_int32(0)
    rc = lib().syncall_read_workspace(ptr(ws), stream_handle(stream), ctypes.byref(sc), ctypes.byref(hc),
                                      ctypes.byref(st))
    return rc, sc.value, hc.value, st.value


def cntnotify_create(flag: int = 0):
    """(code, handle)"""
    h = c_void_p(None)
    rc = lib().cntnotify_create(ctypes.byref(h), flag)
    return rc, h.value


def cntnotify_record(h, stream, mode: int | None = None, value: int = 0, info: RecordInfo | None = None) -> int:
    if info is None and mode is not None:
        info = RecordInfo(mode, value)
    return lib().cntnotify_record(h, stream_handle(stream), ctypes.byref(info) if info is not None else None)


def cntnotify_wait_with_timeout(h, stream, mode: int | None = None, value: int = 0, timeout: int = 0,
                                is_clear: int = 0, info: WaitInfo | None = None) -> int:
    if info is None and mode is not None:
        info = WaitInfo(mode, value, timeout, is_clear)
    return lib().cntnotify_wait_with_timeout(h, stream_handle(stream), ctypes.byref(info) if info is not None else None)


def cntnotify_reset(h, stream=None) -> int:
    return lib().cntnotify_reset(h, stream_handle(stream))


def cntnotify_get_id(h, out: bool = True):
    """(code, id); out=False passes a NULL id pointer."""
    v = c_uint32(0)
    rc = lib().cntnotify_get_id(h, ctypes.byref(v) if out else None)
    return rc, v.value


def cntnotify_destroy(h) -> int:
    return lib().cntnotify_destroy(h)


def cntnotify_get_device_ptr(h):
    p = c_void_p(None)
    rc = lib().cntnotify_get_device_ptr(h, ctypes.byref(p))
    return rc, p.value


def cntnotify_query_status(h):
    """(code, sticky status, count)"""
    st, c = c_int32(0), c_uint32(0)
    rc = lib().cntnotify_query_status(h, ctypes.byref(st), ctypes.byref(c))
    return rc, st.value, c.value


def syncall_workspace_bytes(participants: int, elems: int, out: bool = True):
    """(code, bytes); out=False passes a NULL bytes pointer."""
    v = c_size_t(0)
    rc = lib().syncall_workspace_bytes(participants, elems, ctypes.byref(v) if out else None)
    return rc, v.value


def cntnotify_enable_peer(h, peer_device: int) -> int:
    return lib().cntnotify_enable_peer(h, peer_device)


def cns_probe_launch_cost(launches: int, early: int = 1, stream=None):
    """(code, host microseconds per kernel launch)"""
    v = c_double(0.0)
    rc = lib().cns_probe_launch_cost(launches, early, ctypes.byref(v), stream_handle(stream))
    return rc, v.value


def cns_probe_release_fence(region, iters: int, out, stream=None) -> int:
    return lib().cns_probe_release_fence(ptr(region), iters, ptr(out), stream_handle(stream))


def cns_probe_notify_pingpong(scope: int, iters: int, lines, out, stream=None) -> int:
    return lib().cns_probe_notify_pingpong(scope, iters, ptr(lines), ptr(out), stream_handle(stream))


def cns_statemachine_scratch_bytes(n: int) -> int:
    return lib().cns_statemachine_scratch_bytes(n)


def cns_statemachine_run(ops, n: int, init: int, trace, final, scratch, scratch_bytes: int, stream=None) -> int:
    return lib().cns_statemachine_run(ptr(ops), n, init, ptr(trace), ptr(final), ptr(scratch), scratch_bytes,
                                      stream_handle(stream))


CNS_STATEMACHINE_NOALLOC_MAX_OPS = 2097152


def cns_statemachine_run_noalloc(ops, n: int, init: int, trace, final, stream=None) -> int:
    return lib().cns_statemachine_run_noalloc(ptr(ops), n, init, ptr(trace), ptr(final), stream_handle(stream))


def cns_pipeline_run(cfg: Pipeline) -> int:
    return lib().cns_pipeline_run(ctypes.byref(cfg))


def cns_probe_atomic_rtt(kind: int, grid: int, probe_cta: int, iters: int, line, out, stream=None) -> int:
    return lib().cns_probe_atomic_rtt(kind, grid, probe_cta, iters, ptr(line), ptr(out), stream_handle(stream))


def cns_probe_same_address_throughput(grid: int, threads: int, iters: int, word, stream=None) -> int:
    return lib().cns_probe_same_address_throughput(grid, threads, iters, ptr(word), stream_handle(stream))


def cns_probe_grid_sync(ctas: int, threads: int, rounds: int, buf0, buf1, stream=None) -> int:
    return lib().cns_probe_grid_sync(ctas, threads, rounds, ptr(buf0), ptr(buf1), stream_handle(stream))


def cns_probe_op_chain(ops, iters: int, out, stream=None) -> int:
    return lib().cns_probe_op_chain(ptr(ops), iters, ptr(out), stream_handle(stream))


def cns_probe_round_phases(ctas: int, threads: int, rounds: int, stamp_rounds: int, buf0, buf1, workspace, stamps,
                           stream=None, workspace_bytes: int | None = None) -> int:
    if workspace_bytes is None:
        workspace_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0
    return lib().cns_probe_round_phases(ctas, threads, rounds, stamp_rounds, ptr(buf0), ptr(buf1), ptr(workspace),
                                        workspace_bytes, ptr(stamps), stream_handle(stream))


def cns_version():
    v, sm = c_int32(0), c_int32(0)
    rc = lib().cns_version(ctypes.byref(v), ctypes.byref(sm))
    return rc, v.value, sm.value
