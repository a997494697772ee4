"""The C ABI without a GPU: the library loads, exports every function cns.h
declares, the Python structs match the C layout, and argument / handle errors
come back as codes before any CUDA call."""
import ctypes
import os
import re
import subprocess

import pytest

import counted_notify_sync_gb300 as cns
from counted_notify_sync_gb300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "cns.h")


@pytest.fixture(scope="module")
def built():
    cns.build()
    return _native.lib()


def declared_functions():
    src = open(HEADER, encoding="utf-8").read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*([a-z_][a-z0-9_]*)\s*\(", src, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_named_entry_points():
    names = declared_functions()
    for n in ["syncall_workspace_init", "syncall_run", "cntnotify_create", "cntnotify_record",
              "cntnotify_wait_with_timeout", "cntnotify_reset", "cntnotify_get_id", "cntnotify_destroy"]:
        assert n in names
    assert len(names) >= 18


def test_library_exports_every_declared_symbol(built):
    for n in declared_functions():
        assert hasattr(built, n), n
    assert set(declared_functions()) == set(_native.exported_names())


def test_version(built):
    rc, v, sm = cns.cns_version()
    assert rc == 0 and sm == 103 and v >= 100


def _c_layout():
    prog = r"""
#include <stdio.h>
#include <stddef.h>
#include "cns.h"
#define F(T, m) printf(#T "." #m " %zu\n", offsetof(T, m))
int main(void) {
  printf("cns_syncall_data_t %zu\n", sizeof(cns_syncall_data_t));
  F(cns_syncall_data_t, buf0_dev); F(cns_syncall_data_t, elems); F(cns_syncall_data_t, stream);
  F(cns_syncall_data_t, timeout_ms); F(cns_syncall_data_t, host_in); F(cns_syncall_data_t, elapsed_ms);
  F(cns_syncall_data_t, final_counter); F(cns_syncall_data_t, cluster_used); F(cns_syncall_data_t, barrier_variant);
  F(cns_syncall_data_t, workspace_bytes); F(cns_syncall_data_t, launch_flags); F(cns_syncall_data_t, hard_step);
  printf("cns_record_info_t %zu\n", sizeof(cns_record_info_t));
  printf("cns_wait_info_t %zu\n", sizeof(cns_wait_info_t));
  F(cns_wait_info_t, is_clear);
  printf("cns_pipeline_t %zu\n", sizeof(cns_pipeline_t));
  F(cns_pipeline_t, tiles); F(cns_pipeline_t, rounds); F(cns_pipeline_t, timeout_s);
  F(cns_pipeline_t, elapsed_ms); F(cns_pipeline_t, device_status); F(cns_pipeline_t, consumer_ctas);
  F(cns_pipeline_t, areas); F(cns_pipeline_t, consumer_wait);
  return 0;
}
"""
    wd = os.path.join(ROOT, "counted_notify_sync_gb300", "_build")
    os.makedirs(wd, exist_ok=True)
    c = os.path.join(wd, "layout.c")
    exe = os.path.join(wd, "layout")
    with open(c, "w") as f:
        f.write(prog)
    subprocess.run(["gcc", "-std=c11", "-I", os.path.dirname(HEADER), "-o", exe, c], check=True)
    out = subprocess.run([exe], check=True, capture_output=True, text=True).stdout
    return dict(line.rsplit(" ", 1) for line in out.strip().splitlines())


def test_ctypes_structs_match_c_layout():
    lay = {k: int(v) for k, v in _c_layout().items()}
    S, P, W = _native.SyncallData, _native.Pipeline, _native.WaitInfo
    assert lay["cns_syncall_data_t"] == ctypes.sizeof(S)
    for f in ["buf0_dev", "elems", "stream", "timeout_ms", "host_in", "elapsed_ms", "final_counter",
              "cluster_used", "barrier_variant", "workspace_bytes", "launch_flags", "hard_step"]:
        assert lay[f"cns_syncall_data_t.{f}"] == getattr(S, f).offset, f
    assert lay["cns_record_info_t"] == ctypes.sizeof(_native.RecordInfo) == 8
    assert lay["cns_wait_info_t"] == ctypes.sizeof(W) == 16
    assert lay["cns_wait_info_t.is_clear"] == W.is_clear.offset
    assert lay["cns_pipeline_t"] == ctypes.sizeof(P)
    for f in ["tiles", "rounds", "timeout_s", "elapsed_ms", "device_status", "consumer_ctas", "areas",
              "consumer_wait"]:
        assert lay[f"cns_pipeline_t.{f}"] == getattr(P, f).offset, f


# --- errors decided before any CUDA call ("CANN Runtime CntNotify" §4, §6.3) ---------

def test_create_checks(built):
    assert _native.lib().cntnotify_create(None, 0) == cns.CNS_ERR_NULL_PTR
    rc, h = cns.cntnotify_create(1)          # flag is reserved, must be 0
    assert rc == cns.CNS_ERR_INVALID_VALUE and h is None


def test_invalid_handles(built):
    bogus = ctypes.c_void_p(0x1234).value
    for h in (None, bogus):
        assert cns.cntnotify_record(h, None, cns.CNS_REC_ADD, 1) == cns.CNS_ERR_INVALID_HANDLE
        assert cns.cntnotify_wait_with_timeout(h, None, cns.CNS_WAIT_LESS, 0, 0, 1) == cns.CNS_ERR_INVALID_HANDLE
        assert cns.cntnotify_reset(h) == cns.CNS_ERR_INVALID_HANDLE
        assert cns.cntnotify_get_id(h)[0] == cns.CNS_ERR_INVALID_HANDLE
        assert cns.cntnotify_destroy(h) == cns.CNS_ERR_INVALID_HANDLE
        assert cns.cntnotify_get_device_ptr(h)[0] == cns.CNS_ERR_INVALID_HANDLE
        assert cns.cntnotify_query_status(h)[0] == cns.CNS_ERR_INVALID_HANDLE
        assert cns.cntnotify_enable_peer(h, 0) == cns.CNS_ERR_INVALID_HANDLE


def test_syncall_argument_checks(built):
    L = _native.lib()
    assert L.syncall_run(cns.CNS_SYNCALL_SOFT, 0, 0, 0, 10, None) == cns.CNS_ERR_NULL_PTR
    d = _native.SyncallData()
    d.launch_ctas = 8
    d.workload = cns.CNS_WL_EMPTY
    assert cns.syncall_run(7, 0, 0, 0, 1, d) == cns.CNS_ERR_INVALID_VALUE          # mode
    assert cns.syncall_run(1, 3, 0, 0, 1, d) == cns.CNS_ERR_INVALID_VALUE          # core type
    assert cns.syncall_run(1, 0, 0, 0, -1, d) == cns.CNS_ERR_INVALID_VALUE         # rounds
    assert cns.syncall_run(1, 0, 9, 0, 1, d) == cns.CNS_ERR_INVALID_VALUE          # used_cores > launched
    assert cns.syncall_run(1, 0, 0, 0, 1, d) == cns.CNS_ERR_NULL_PTR               # no workspace
    d.workspace_dev = 0x1000 + 64
    assert cns.syncall_run(1, 0, 0, 0, 1, d) == cns.CNS_ERR_INVALID_VALUE          # misaligned workspace
    d.workspace_dev = 0x1000
    d.workload, d.elems = cns.CNS_WL_RING_AFFINE, 4
    assert cns.syncall_run(1, 0, 0, 0, 1, d) == cns.CNS_ERR_NULL_PTR               # no payload buffers
    d.buf0_dev, d.buf1_dev = 0x2008, 0x3000
    assert cns.syncall_run(1, 0, 0, 0, 1, d) == cns.CNS_ERR_INVALID_VALUE          # misaligned payload
    d.workload = 9
    assert cns.syncall_run(1, 0, 0, 0, 1, d) == cns.CNS_ERR_INVALID_VALUE          # workload
    d.workload, d.threads = cns.CNS_WL_EMPTY, 48
    assert cns.syncall_run(1, 0, 0, 0, 1, d) == cns.CNS_ERR_INVALID_VALUE          # threads
    d.threads, d.cluster_dim = 256, 3
    assert cns.syncall_run(0, 0, 0, 0, 1, d) == cns.CNS_ERR_INVALID_VALUE          # 3 does not divide 8
    assert cns.syncall_run(0, cns.CNS_MIX, 0, 8, 1, d) == cns.CNS_ERR_INVALID_VALUE  # cluster of 9
    d.cluster_dim, d.barrier_variant = 0, 9
    assert cns.syncall_run(1, 0, 0, 0, 1, d) == cns.CNS_ERR_INVALID_VALUE          # barrier variant
    wl = d.workload
    d.barrier_variant, d.workload = cns.CNS_BARRIER_ARRIVAL_ONLY, cns.CNS_WL_RING_AFFINE
    assert cns.syncall_run(1, 0, 0, 0, 1, d) == cns.CNS_ERR_INVALID_VALUE          # arrival only orders no data
    d.workload = wl
    d.barrier_variant, d.workspace_bytes = cns.CNS_BARRIER_DIE_LOCAL, 512
    assert cns.syncall_run(1, 0, 0, 0, 1, d) == cns.CNS_ERR_INVALID_VALUE          # die-local needs 8 KB
    d.barrier_variant, d.workspace_bytes = 0, 256
    assert cns.syncall_run(1, 0, 0, 0, 1, d) == cns.CNS_ERR_INVALID_VALUE          # workspace too small
    d.workspace_bytes, d.hard_step = 0, cns.CNS_HARD_STEP_PAIRED_MBARRIER
    assert cns.syncall_run(1, 0, 0, 0, 1, d) == cns.CNS_ERR_INVALID_VALUE          # paired step on the soft path
    d.hard_step = 2
    assert cns.syncall_run(0, 0, 0, 0, 1, d) == cns.CNS_ERR_INVALID_VALUE          # no such hard step
    d.hard_step = 0
    assert L.syncall_workspace_init(None, 512, 0, None) == cns.CNS_ERR_NULL_PTR
    assert L.syncall_workspace_init(0x1000, 511, 0, None) == cns.CNS_ERR_INVALID_VALUE


def test_statemachine_and_pipeline_argument_checks(built):
    L = _native.lib()
    # one 128-byte line per tile: at most ceil(n / 16) tiles, and at most max(ceil(n / 4096), 4096)
    assert cns.cns_statemachine_scratch_bytes(0) == 0
    assert cns.cns_statemachine_scratch_bytes(17) == 2 * 128
    assert cns.cns_statemachine_scratch_bytes(16 * 4096) == 4096 * 128
    assert cns.cns_statemachine_scratch_bytes(1_000_000) == 4096 * 128
    assert cns.cns_statemachine_scratch_bytes(4096 * 5000 + 1) == 5001 * 128
    assert L.cns_statemachine_run(None, -1, 0, None, None, None, 0, None) == cns.CNS_ERR_INVALID_VALUE
    assert L.cns_statemachine_run(None, 4, 0, None, 0x1000, None, 0, None) == cns.CNS_ERR_NULL_PTR
    assert L.cns_statemachine_run(0x1008, 4, 0, 0x2000, 0x3000, 0x4000, 8, None) == cns.CNS_ERR_INVALID_VALUE
    assert L.cns_statemachine_run(0x1000, 40, 0, 0x2000, 0x3000, 0x4000, 8, None) == cns.CNS_ERR_INVALID_VALUE
    assert L.cns_pipeline_run(None) == cns.CNS_ERR_NULL_PTR
    assert cns.cns_pipeline_run(_native.Pipeline()) == cns.CNS_ERR_INVALID_HANDLE
    assert cns.cns_probe_atomic_rtt(0, 1, 0, 1, None, None) == cns.CNS_ERR_NULL_PTR
    assert cns.cns_probe_atomic_rtt(3, 1, 0, 1, 0x1000, 0x2000) == cns.CNS_ERR_INVALID_VALUE


def test_no_device_is_an_error_not_a_crash(built):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    rc, h = cns.cntnotify_create(0)
    assert rc in (cns.CNS_ERR_CUDA, cns.CNS_ERR_ARCH) and h is None


def test_error_strings(built):
    assert cns.error_string(cns.CNS_ERR_TIMEOUT) == "timeout"
    assert cns.error_string(12345) == "unknown error"


def test_python_constants_match_the_header():
    """Every integer #define of cns.h has the same value in the binding."""
    import re
    src = open(HEADER, encoding="utf-8").read()
    found = 0
    for name, val in re.findall(r"^#define (CNS_[A-Z0-9_]+) \(?(\d+)u?\)?", src, flags=re.M):
        if hasattr(_native, name):
            assert getattr(_native, name) == int(val), name
            found += 1
    assert found >= 10
    assert _native.CNS_SYNCALL_DIE_LOCAL_ALIGN == 8192
    assert (_native.CNS_PIPE_WAIT_STREAM, _native.CNS_PIPE_WAIT_IN_KERNEL) == (0, 1)


def test_workspace_bytes_for_the_payload_copies(built):
    """The die-local workspace size that makes room for the per-die payload copies (host only)."""
    rows = lambda slots: 255 // (slots // 4)   # noqa: E731  (rows per 4 KB block)
    for P, slots in [(148, 4), (255, 4), (256, 4), (8, 256), (111, 256), (5, 1020), (4864, 4)]:
        rc, nbytes = cns.syncall_workspace_bytes(P, slots)
        pairs = -(-P // rows(slots))
        assert rc == 0 and nbytes == cns.CNS_SYNCALL_WORKSPACE_DIE_LOCAL_BYTES + 2 * pairs * 8192
    for P, slots in [(8, 1024), (8, 6), (8, 0)]:
        assert cns.syncall_workspace_bytes(P, slots) == (0, cns.CNS_SYNCALL_WORKSPACE_DIE_LOCAL_BYTES)
    assert cns.syncall_workspace_bytes(148, 4)[1] == cns.CNS_SYNCALL_WORKSPACE_MIRROR_BYTES
    assert cns.syncall_workspace_bytes(0, 4)[0] == cns.CNS_ERR_INVALID_VALUE
    assert cns.syncall_workspace_bytes(8, -1)[0] == cns.CNS_ERR_INVALID_VALUE
    assert cns.syncall_workspace_bytes(8, 4, out=False)[0] == cns.CNS_ERR_NULL_PTR
