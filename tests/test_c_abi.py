"""The C ABI from C itself: include/sdpa.h compiles as strict C99 and C++17, a C program
links against the built library and gets the documented behaviour from it (version, struct
size, workspace sizing of a valid problem, and an error status plus message for an invalid
one).  No GPU is needed: these calls validate and size on the host only."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_SOURCE = r"""
#include <stdio.h>
#include <string.h>
#include "sdpa.h"

static void strides(sdpa_strides_t* s, int64_t h, int64_t n, int64_t d) {
  s->b = h * n * d; s->h = n * d; s->s = d; s->d = 1;
}

int main(void) {
  sdpa_problem_t p;
  size_t bytes = 0;
  sdpa_status_t st;
  if (sdpa_version() < 100) return 10;
  if (sdpa_problem_struct_size() != sizeof(sdpa_problem_t)) return 11;
  memset(&p, 0, sizeof p);
  p.b = 2; p.h_q = 8; p.h_kv = 2; p.s_q = 1000; p.s_kv = 1000; p.d = 128;
  p.in_dtype = SDPA_DTYPE_BF16; p.out_dtype = SDPA_DTYPE_BF16;
  p.attn_scale = 0.08838834764831845f; p.causal = 1;
  strides(&p.q, 8, 1000, 128); strides(&p.o, 8, 1000, 128);
  strides(&p.dout, 8, 1000, 128); strides(&p.dq, 8, 1000, 128);
  strides(&p.k, 2, 1000, 128); strides(&p.v, 2, 1000, 128);
  strides(&p.dk, 2, 1000, 128); strides(&p.dv, 2, 1000, 128);
  st = sdpa_workspace_size(&p, 0, &bytes);
  if (st != SDPA_OK || bytes != 0) return 12;            /* the forward pass needs none */
  st = sdpa_workspace_size(&p, 1, &bytes);
  if (st != SDPA_OK || bytes == 0) return 13;
  printf("bwd_workspace %zu\n", bytes);
  p.h_kv = 3;                                            /* 8 query heads do not group by 3 */
  st = sdpa_workspace_size(&p, 1, &bytes);
  if (st != SDPA_ERR_INVALID_ARG) return 14;
  if (strlen(sdpa_last_error_string()) == 0) return 15;
  printf("error %s\n", sdpa_last_error_string());
  return 0;
}
"""


@pytest.fixture(scope="module")
def lib_path():
    import attention_flashattention_sdpa_gb300 as m
    return m.LIB_PATH


def _compiler(name):
    path = shutil.which(name)
    if path is None:
        pytest.skip(f"{name} not found")
    return path


@pytest.mark.parametrize("lang,flags", [("c", ["-std=c99", "-pedantic"]), ("c++", ["-std=c++17", "-pedantic"])])
def test_header_compiles_warning_free(tmp_path, lang, flags):
    src = tmp_path / ("h.c" if lang == "c" else "h.cpp")
    src.write_text('#include "sdpa.h"\nint probe(void) { return (int)sizeof(sdpa_problem_t); }\n')
    cc = _compiler("gcc" if lang == "c" else "g++")
    subprocess.run([cc, *flags, "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"), "-c",
                    str(src), "-o", str(tmp_path / "h.o")], check=True)


def test_c_program_links_and_gets_documented_results(tmp_path, lib_path):
    src = tmp_path / "abi.c"
    src.write_text(C_SOURCE)
    exe = tmp_path / "abi"
    libdir = os.path.dirname(lib_path)
    subprocess.run([_compiler("gcc"), "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), lib_path, f"-Wl,-rpath,{libdir}"], check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0, f"exit {r.returncode}: {r.stdout} {r.stderr}"
    lines = r.stdout.splitlines()
    assert lines[0].startswith("bwd_workspace ") and int(lines[0].split()[1]) > 0
    assert lines[1].startswith("error ") and "h_kv" in lines[1]
