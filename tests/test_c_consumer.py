"""The boundary as a C program sees it: include/fa.h compiles as strict C99
(-Wall -Wextra -pedantic -Werror), a program that references every entry
point the header declares links against libfa.so, and the calls that fail
argument checks return their codes without touching a GPU."""

import os
import shutil
import subprocess

import pytest

from tiled_attention_07_gb300 import fa

from test_abi import HEADER, header_symbols

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include "fa.h"
#include <stdio.h>

typedef void (*fn)(void);
static const fn every_entry_point[] = {
%(refs)s
};

int main(void) {
  int bad = 0;
  /* head dim 96 is not supported: rejected before any CUDA call */
  fa_status s = fa_fwd(0, 0, 0, 0, 0, 1, 1, 128, 128, 96, 0.125f, 0, FA_BF16, 0);
  bad |= s != FA_ERR_UNSUPPORTED;
  /* a sequence longer than FA_MAX_SEQLEN */
  s = fa_fwd(0, 0, 0, 0, 0, 1, 1, FA_MAX_SEQLEN + 1, 128, 64, 0.125f, 0, FA_BF16, 0);
  bad |= s != FA_ERR_INVALID_ARG;
  /* workspace size of the bench shape: 2 float32 per padded query row */
  bad |= fa_bwd_workspace_bytes(4, 32, 8192, 8192, 80) != (size_t)2 * 4 * 4 * 32 * 8192;
  printf("%%s %%s %%d\n", fa_version(), fa_status_string(FA_ERR_WORKSPACE),
         (int)(sizeof every_entry_point / sizeof every_entry_point[0]));
  return bad;
}
"""


@pytest.fixture(scope="module")
def libfa():
    if not os.path.exists(fa.LIB_PATH):
        from tiled_attention_07_gb300 import build
        build.build()
    return fa.LIB_PATH


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_c99_program_links_and_calls(libfa, tmp_path):
    syms = header_symbols()
    refs = ",\n".join(f"  (fn){s}" for s in syms)
    src = tmp_path / "consumer.c"
    src.write_text(PROGRAM % {"refs": refs})
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(libfa)
    cmd = ["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.dirname(HEADER), str(src),
           "-L", libdir, "-lfa", f"-Wl,-rpath,{libdir}", "-o", str(exe)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    words = r.stdout.split()
    assert words[0] == fa.fa_version()
    assert words[1].startswith("FA_ERR_WORKSPACE")
    assert int(words[-1]) == len(syms)
