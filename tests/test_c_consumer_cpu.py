"""The boundary as a C program sees it (CPU only): lf_decode.h compiles as
strict C99 and C++11, and a C program linked against liblf_decode.so gets
the version, status strings and host-side argument errors without a GPU."""
import os
import shutil
import subprocess

import pytest

from decode_kv_cache_step_gb300 import build as lfbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")

C_PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "lf_decode.h"

int main(void) {
    static unsigned short buf[4096] __attribute__((aligned(256)));
    int32_t slots[4] = {0, 0, 0, 0};
    lf_step_handle* h = NULL;
    if (lf_version() != 100) return 1;
    if (strcmp(lf_status_string(LF_OK), "LF_OK") != 0) return 2;
    /* A missing q is refused on the host, before any CUDA call. */
    if (lf_decode_step(NULL, buf, buf, slots, buf, buf, slots, buf, slots, 1, 4, 2, 64, 16, 2,
                       0.125f, NULL) != LF_ERR_INVALID_ARG) return 3;
    if (lf_last_error()[0] == '\0') return 4;
    if (lf_step_prepare(buf, buf, buf, slots, buf, buf, slots, buf, slots, 1, 4, 2, 96, 16, 2,
                        0.125f, NULL, &h) != LF_ERR_UNSUPPORTED || h != NULL) return 5;
    if (lf_step_run(NULL) != LF_ERR_INVALID_ARG) return 6;
    if (lf_step_destroy(NULL) != LF_OK) return 7;
    puts("ok");
    return 0;
}
"""


def _cc(name):
    path = shutil.which(name)
    if path is None:
        pytest.skip(f"{name} not found")
    return path


def test_header_is_strict_c99_and_cxx11(tmp_path):
    src = tmp_path / "h.c"
    src.write_text('#include "lf_decode.h"\nint lf_probe(void) { return LF_MAX_TOPK; }\n')
    subprocess.run([_cc("gcc"), "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-c",
                    str(src), "-I", INCLUDE, "-o", str(tmp_path / "h.o")], check=True)
    srcpp = tmp_path / "h.cpp"
    srcpp.write_text('#include "lf_decode.h"\nint lf_probe() { return LF_MAX_TOPK; }\n')
    subprocess.run([_cc("g++"), "-std=c++11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-c",
                    str(srcpp), "-I", INCLUDE, "-o", str(tmp_path / "hpp.o")], check=True)


def test_c_program_links_and_runs_without_a_gpu(tmp_path):
    if not os.path.exists(lfbuild.LIB_PATH):
        pytest.skip("liblf_decode.so is not built")
    src = tmp_path / "consumer.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "consumer"
    lib_dir = os.path.dirname(lfbuild.LIB_PATH)
    subprocess.run([_cc("gcc"), "-std=gnu99", "-Wall", "-Werror", str(src), "-I", INCLUDE,
                    "-L", lib_dir, "-llf_decode", f"-Wl,-rpath,{lib_dir}", "-o", str(exe)],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", (r.returncode, r.stdout, r.stderr)
