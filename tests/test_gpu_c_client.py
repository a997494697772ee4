"""The C ABI from a plain C program, no Python in between: tests/c_client/client.c
is compiled with gcc against include/cns.h, linked with libcns.so and the CUDA
runtime, and run (soft and hard rings, the paired hard step, workspaces sized
for the per-die payload copies, and counted notifies at gpu and at system
scope); it checks its own results against closed forms and prints "ok"."""
import os
import subprocess

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_program_uses_the_library():
    import counted_notify_sync_gb300 as cns
    from counted_notify_sync_gb300 import builder
    lib = cns.build()
    libdir = os.path.dirname(os.path.abspath(lib))
    cuda = builder.cuda_home()
    out = os.path.join(ROOT, "tests", "c_client", "_build", "client")
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cudart_dir = next(d for d in (os.path.join(cuda, "lib64"), os.path.join(cuda, "lib"),
                                  os.path.join(cuda, "targets", "sbsa-linux", "lib"),
                                  os.path.join(cuda, "targets", "x86_64-linux", "lib"))
                      if os.path.exists(os.path.join(d, "libcudart.so")))
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-Wextra", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(cuda, "include"), "-o", out, os.path.join(ROOT, "tests", "c_client", "client.c"),
                    "-L", libdir, "-lcns", "-L", cudart_dir, "-lcudart",
                    f"-Wl,-rpath,{libdir}", f"-Wl,-rpath,{cudart_dir}"], check=True)
    r = subprocess.run([out], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
