"""Helpers for the GPU tests: move uint32 / float32 numpy arrays to and from
the device bit for bit (torch has no full uint32 dtype, so int32 views), and
build and load the user kernels of tests/fused/ (test-only kernels written on
include/cns_device.h)."""
import ctypes
import os
import subprocess

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
USER_SRC = os.path.join(ROOT, "tests", "fused", "user_kernels.cu")
USER_OUT = os.path.join(ROOT, "tests", "fused", "_build", "libcns_user_kernels.so")


def to_dev_u32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint32).view(np.int32)).cuda()


def to_dev_f32(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def from_dev_u32(t):
    return t.cpu().numpy().view(np.uint32)


def load_user_kernels():
    """tests/fused/user_kernels.cu as a shared library (built with nvcc for sm_103a when missing or older than
    its sources), with the ctypes signatures of its entry points."""
    from counted_notify_sync_gb300 import builder
    hdrs = [os.path.join(ROOT, "include", n) for n in ("cns_device.h", "cns.h")]
    newest = max(os.path.getmtime(p) for p in [USER_SRC, *hdrs])
    if not os.path.exists(USER_OUT) or os.path.getmtime(USER_OUT) < newest:
        os.makedirs(os.path.dirname(USER_OUT), exist_ok=True)
        tmp = USER_OUT + f".tmp{os.getpid()}"
        nvcc = os.path.join(builder.cuda_home(), "bin", "nvcc")
        subprocess.run([nvcc, *builder.ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                        "-I", os.path.join(ROOT, "include"), "-o", tmp, USER_SRC], check=True)
        os.replace(tmp, USER_OUT)
    L = ctypes.CDLL(USER_OUT)
    i32, u32, i64, u64, vp = ctypes.c_int32, ctypes.c_uint32, ctypes.c_int64, ctypes.c_uint64, ctypes.c_void_p
    L.user_ring.argtypes = [i32, i32, u32, i64, vp, vp, vp, u64, u32, vp]
    L.user_ring_die_local.argtypes = [i32, i32, u32, i64, vp, vp, vp, u64, u32, vp]
    L.user_ring_sys.argtypes = [i32, i32, u32, i64, vp, vp, vp, u64, u32, vp]
    L.user_record.argtypes = [vp, ctypes.c_int, u32, i32, i32, ctypes.c_int]
    L.user_wait.argtypes = [vp, ctypes.c_int, u32, ctypes.c_int, u64, vp, vp]
    L.user_record_sys.argtypes = [vp, ctypes.c_int, u32, i32, i32, ctypes.c_int]
    L.user_wait_sys.argtypes = [vp, ctypes.c_int, u32, ctypes.c_int, u64, vp, vp]
    L.user_grid_wait.argtypes = [i32, i32, vp, vp, vp, vp, ctypes.c_int, u32, ctypes.c_int, u64, vp, vp, vp]
    L.user_grid_wait_only.argtypes = [i32, vp, vp, u32, ctypes.c_int, u32, u64, vp]
    for f in (L.user_ring, L.user_ring_die_local, L.user_ring_sys, L.user_record, L.user_wait, L.user_record_sys, L.user_wait_sys,
              L.user_grid_wait, L.user_grid_wait_only):
        f.restype = ctypes.c_int
    return L
