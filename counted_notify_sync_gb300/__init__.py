"""counted_notify_sync_gb300: SYNCALL epoch barrier and CntNotify on GB300.

The C ABI (include/cns.h, libcns.so) does all the work; this package is the
thin Python side: ``_native`` mirrors the C entry points one to one, and the
helpers below allocate device buffers with PyTorch and marshal arguments.
"""
from __future__ import annotations

from . import _native
from ._native import *  # noqa: F401,F403  (C names and constants)

__all__ = [n for n in dir(_native) if not n.startswith("_")] + [
    "build", "new_workspace", "run_syncall", "run_statemachine", "run_pipeline",
]


def build(force: bool = False, verbose: bool = False) -> str:
    from .builder import build as _b
    return _b(force=force, verbose=verbose)


def _torch():
    import torch
    if not torch.cuda.is_available():
        raise RuntimeError("counted_notify_sync_gb300 needs a CUDA device")
    return torch


def new_workspace(device=None, start_value: int = 0, stream=None, die_local: bool = True, mirror: bool = True,
                  participants: int | None = None, elems: int | None = None):
    """An initialised SYNCALL workspace on `device`, usable by every barrier variant.  With die_local (the
    default) it starts on a CNS_SYNCALL_DIE_LOCAL_ALIGN boundary, so that the two copies of each counter sit
    on different dies, and has room for the die-local variant's per-die payload copies: of rows of one uint4
    and up to CNS_SYNCALL_MIRROR_MAX_P participants (CNS_SYNCALL_WORKSPACE_MIRROR_BYTES), or, given
    participants and elems, of that ring (syncall_workspace_bytes).  mirror=False gives
    CNS_SYNCALL_WORKSPACE_DIE_LOCAL_BYTES, die_local=False the minimal CNS_SYNCALL_WORKSPACE_BYTES."""
    torch = _torch()
    if not die_local:
        ws = torch.empty(_native.CNS_SYNCALL_WORKSPACE_BYTES // 4, dtype=torch.int32, device=device or "cuda")
    else:
        nbytes = _native.CNS_SYNCALL_WORKSPACE_MIRROR_BYTES if mirror else _native.CNS_SYNCALL_WORKSPACE_DIE_LOCAL_BYTES
        if mirror and participants is not None and elems is not None:
            rc, need = _native.syncall_workspace_bytes(participants, elems)
            _native.check(rc, "syncall_workspace_bytes")
            nbytes = max(nbytes, need)
        align = _native.CNS_SYNCALL_DIE_LOCAL_ALIGN
        raw = torch.empty((nbytes + align) // 4, dtype=torch.int32, device=device or "cuda")
        skip = (-raw.data_ptr()) % align // 4
        ws = raw[skip:skip + nbytes // 4]   # a view: keeps `raw` alive
    _native.check(_native.syncall_workspace_init(ws, ws.numel() * 4, start_value, stream), "syncall_workspace_init")
    return ws


def run_syncall(mode, core_type, workload, launch_ctas, buf0, buf1, rounds, *, used_cores=0, aiv_ratio=0,
                elems=0, threads=256, cluster_dim=0, timeout_ms=0, workspace=None, cta_status=None,
                stream=None, sync=True, host_in=None, host_out=None, check=True, variant=0, launch_flags=0,
                hard_step=0):
    """Call syncall_run with device buffers (torch tensors); returns the filled SyncallData and the code."""
    d = _native.SyncallData()
    d.workload = workload
    d.launch_ctas = launch_ctas
    d.threads = threads
    d.cluster_dim = cluster_dim
    d.buf0_dev = _native.ptr(buf0)
    d.buf1_dev = _native.ptr(buf1)
    d.elems = elems
    d.workspace_dev = _native.ptr(workspace)
    d.cta_status_dev = _native.ptr(cta_status)
    d.stream = _native.stream_handle(stream)
    d.timeout_ms = timeout_ms
    d.sync = 1 if sync else 0
    d.host_in = _native.ptr(host_in)
    d.host_out = _native.ptr(host_out)
    d.barrier_variant = variant
    d.launch_flags = launch_flags
    d.hard_step = hard_step
    d.workspace_bytes = workspace.numel() * workspace.element_size() if hasattr(workspace, "numel") else 0
    rc = _native.syncall_run(mode, core_type, used_cores, aiv_ratio, rounds, d)
    if check and rc != _native.CNS_SUCCESS:
        raise _native.CnsError(rc, "syncall_run")
    return d, rc


def run_statemachine(ops_dev, init: int, stream=None):
    """Apply an [n, 4] int32 device op stream; returns (trace [n, 2] int32, final [1] int32) device tensors."""
    torch = _torch()
    n = ops_dev.shape[0]
    trace = torch.empty((n, 2), dtype=torch.int32, device=ops_dev.device)
    final = torch.empty(1, dtype=torch.int32, device=ops_dev.device)
    sb = _native.cns_statemachine_scratch_bytes(n)
    scratch = torch.empty(max(sb, 8), dtype=torch.uint8, device=ops_dev.device)
    _native.check(_native.cns_statemachine_run(ops_dev if n else None, n, init, trace if n else None, final,
                                               scratch, scratch.numel(), stream), "cns_statemachine_run")
    return trace, final


def run_pipeline(done, ack, tiles: int, tile_words: int, rounds: int, producer_stream, consumer_stream,
                 timeout_s: int = 10, producer_ctas: int = 0, sync: bool = True, buffers=None, areas: int = 1,
                 consumer_wait: int = 0):
    """Run the two-stream counting pipeline; returns (Pipeline struct, code, checksums, released).
    areas = 2 alternates the rounds between two tile areas (the tile buffer then holds both);
    consumer_wait = 1 (CNS_PIPE_WAIT_IN_KERNEL) has the consumer kernel take the wait itself."""
    torch = _torch()
    if buffers is None:
        tiles_buf = torch.empty(max(1, areas) * tiles * tile_words, dtype=torch.int32, device="cuda")
        checksums = torch.empty(rounds, dtype=torch.int32, device="cuda")
        released = torch.empty(rounds, dtype=torch.int32, device="cuda")
    else:
        tiles_buf, checksums, released = buffers
    cfg = _native.Pipeline()
    cfg.done = done
    cfg.ack = ack
    cfg.tiles_dev = _native.ptr(tiles_buf)
    cfg.checksums_dev = _native.ptr(checksums)
    cfg.released_dev = _native.ptr(released)
    cfg.tiles = tiles
    cfg.tile_words = tile_words
    cfg.producer_ctas = producer_ctas
    cfg.rounds = rounds
    cfg.producer_stream = _native.stream_handle(producer_stream)
    cfg.consumer_stream = _native.stream_handle(consumer_stream)
    cfg.timeout_s = timeout_s
    cfg.sync = 1 if sync else 0
    cfg.areas = areas
    cfg.consumer_wait = consumer_wait
    rc = _native.cns_pipeline_run(cfg)
    return cfg, rc, checksums, released
