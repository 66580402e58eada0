"""The C ABI header compiles as strict C11 and as C++17, and a C program
built against it and linked with libq.so calls it: argument validation
runs on the host (no device is touched)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
LIB_DIR = os.path.join(ROOT, "nvfp4_quantization_current_gb300")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "q.h"

int main(void)
{
    if (q_abi_version() != 4) return 1;
    /* K = 24 is not a multiple of 16: rejected on the host, nothing launched */
    q_status s = q_nvfp4((const void *)0x10000, Q_BF16, 16, 24, Q_B1x16, Q_RN, 0, 0,
                         (uint8_t *)0x10000, (uint8_t *)0x10000, NULL, NULL, (float *)0x10000,
                         Q_AMAX_COMPUTE, (float *)0x10000, NULL, NULL);
    if (s != Q_ERR_SHAPE) return 2;
    if (strstr(q_last_error(), "q_nvfp4") == NULL) return 3;
    printf("ok %s\n", q_last_error());
    return 0;
}
"""


@pytest.mark.parametrize("cc,flags", [("gcc", ["-x", "c", "-std=c11", "-pedantic"]),
                                      ("g++", ["-x", "c++", "-std=c++17", "-pedantic"])])
def test_header_compiles(tmp_path, cc, flags):
    if shutil.which(cc) is None:
        pytest.skip(f"{cc} not found")
    src = tmp_path / "use_q.c"
    src.write_text('#include "q.h"\nint q_header_probe(void) { return (int)Q_ERR_CUDA + (int)Q_HIST_MOST_RECENT; }\n')
    r = subprocess.run([cc, *flags, "-Wall", "-Wextra", "-Werror", "-I", INCLUDE, "-c", str(src), "-o",
                        str(tmp_path / "use_q.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_c_program_links_and_validates(tmp_path):
    lib = os.path.join(LIB_DIR, "libq.so")
    if shutil.which("gcc") is None or not os.path.exists(lib):
        pytest.skip("gcc or libq.so missing")
    src = tmp_path / "main.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "main"
    r = subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", INCLUDE, str(src), "-o", str(exe),
                        "-L", LIB_DIR, "-lq", "-Wl,-rpath," + LIB_DIR], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, (r.returncode, r.stdout, r.stderr)
    assert r.stdout.startswith("ok ")
