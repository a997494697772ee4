"""include/cns_device.h stands on its own: it compiles for sm_103a in a
translation unit that includes nothing else, the test-only user kernels built
on it compile, and a plain C compiler sees only cns.h's declarations."""
import os
import subprocess

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INC = os.path.join(ROOT, "include")


def _nvcc():
    from counted_notify_sync_gb300 import builder
    return os.path.join(builder.cuda_home(), "bin", "nvcc"), builder.ARCH


def test_device_header_compiles_alone(tmp_path):
    nvcc, arch = _nvcc()
    src = tmp_path / "alone.cu"
    src.write_text('#include "cns_device.h"\n'
                   "__global__ void k(uint32_t *w, void *ws, int *rc)\n"
                   "{\n"
                   "    cns_cnt_record_dev(w, CNS_REC_ADD, 1u);\n"
                   "    rc[0] = cns_cnt_wait_dev(w, CNS_WAIT_BIGGER_OR_EQUAL, 1u, 1, 0, nullptr);\n"
                   "    rc[1] = cns_syncall_soft(ws, gridDim.x, 0);\n"
                   "    rc[2] = cns_cnt_wait_grid_dev(w, w + 32, 0u, CNS_WAIT_BIGGER_OR_EQUAL, 1u, 1, 0, nullptr);\n"
                   "}\n")
    subprocess.run([nvcc, *arch, "-std=c++17", "-I", INC, "-c", "-o", str(tmp_path / "alone.o"), str(src)],
                   check=True)


def test_user_kernels_compile(tmp_path):
    nvcc, arch = _nvcc()
    subprocess.run([nvcc, *arch, "-std=c++17", "-I", INC, "-c", "-o", str(tmp_path / "u.o"),
                    os.path.join(ROOT, "tests", "fused", "user_kernels.cu")], check=True)


def test_device_header_is_plain_c_without_cuda(tmp_path):
    src = tmp_path / "c.c"
    src.write_text('#include "cns_device.h"\nint main(void) { return CNS_SUCCESS; }\n')
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", INC, "-o", str(tmp_path / "c"), str(src)],
                   check=True)
