"""CPU: the C ABI from plain C.  `include/bsa.h` compiles as C and as C++,
and a small C program linked against libbsa.so calls the library's host-side
entry points (version, status strings, argument validation) with no GPU."""

import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA_INC = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "bsa.h"

int main(void) {
  if (bsa_version() < 100) return 10;
  const char* s = bsa_status_string(BSA_ERR_UNSUPPORTED);
  if (s == NULL || strlen(s) == 0) return 11;
  /* null pointers and a bad head dim are refused on the host, before any device work */
  if (tra_forward(NULL, NULL, NULL, NULL, 1, 1, 16, 64, 1.0f, 2.0f, BSA_BF16, 0) != BSA_ERR_NULLPTR) return 12;
  char buf[64];
  void* p = (void*)(((size_t)buf + 15) & ~(size_t)15);
  if (tra_forward(p, p, p, p, 1, 1, 16, 100, 1.0f, 2.0f, BSA_BF16, 0) != BSA_ERR_UNSUPPORTED) return 13;
  if (nsa_select_forward(p, p, p, NULL, p, NULL, 1, 16, 1, 128, 128, 64, 4, 0) != BSA_ERR_NULLPTR) return 14;
  printf("ok %d\n", bsa_version());
  return 0;
}
"""


def _cc():
    return shutil.which("gcc") or shutil.which("cc")


@pytest.mark.skipif(_cc() is None or not os.path.isdir(CUDA_INC), reason="needs gcc and the CUDA headers")
@pytest.mark.parametrize("lang", ["c", "c++"])
def test_header_compiles(lang, tmp_path):
    cc = _cc() if lang == "c" else (shutil.which("g++") or pytest.skip("no g++"))
    r = subprocess.run([cc, "-fsyntax-only", "-x", lang, "-I", CUDA_INC, os.path.join(ROOT, "include", "bsa.h")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


@pytest.mark.skipif(_cc() is None or not os.path.isdir(CUDA_INC), reason="needs gcc and the CUDA headers")
def test_c_program_calls_the_library(tmp_path):
    from block_sparse_attention_tra_gb300 import build

    lib = build.build()
    src = tmp_path / "consumer.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(lib)
    r = subprocess.run([_cc(), str(src), "-o", str(exe), "-I", os.path.join(ROOT, "include"), "-I", CUDA_INC,
                        "-L", libdir, "-lbsa", "-Wl,-rpath," + libdir], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert out.returncode == 0, (out.returncode, out.stderr)
    assert out.stdout.startswith("ok ")
