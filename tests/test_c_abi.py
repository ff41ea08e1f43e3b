"""The C ABI from C: include/fa.h compiles as strict C11 on its own, and a plain C program (no Python,
no torch) builds against libfa and the CUDA runtime's C API; on a GPU it runs one fa_fwd and one
fa_decode_splitkv (ragged chunks) and checks both against the oracle's C library."""
import os
import subprocess

import pytest

import attention_forward_05_gb300 as fa
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = "/usr/local/cuda"


def test_header_is_plain_c11(tmp_path):
    src = tmp_path / "h.c"
    src.write_text('#include "fa.h"\nint main(void) { return fa_status_string(FA_OK)[0] == 0; }\n')
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-fsyntax-only",
                    "-I", os.path.join(ROOT, "include"), str(src)], check=True)


def _build_consumer(out_dir) -> str:
    exe = os.path.join(str(out_dir), "fa_c_consumer")
    lib_dir = os.path.dirname(fa.lib_path())
    ora = oracle.build()
    subprocess.run(["gcc", "-std=c11", "-O2", "-Wall", "-Werror", "-o", exe,
                    os.path.join(ROOT, "tests", "c", "fa_c_consumer.c"),
                    "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
                    fa.lib_path(), ora, "-L", os.path.join(CUDA, "lib64"), "-lcudart", "-lm",
                    "-Wl,-rpath," + lib_dir + ":" + os.path.dirname(ora) + ":" + os.path.join(CUDA, "lib64")],
                   check=True)
    return exe


def test_c_consumer_builds(tmp_path):
    fa.lib()  # builds libfa if needed
    assert os.path.exists(_build_consumer(tmp_path))


@pytest.mark.gpu
def test_c_consumer_runs(tmp_path):
    r = subprocess.run([_build_consumer(tmp_path)], capture_output=True, text=True, timeout=300)
    print(r.stdout, r.stderr)
    assert r.returncode == 0, r.stdout + r.stderr
