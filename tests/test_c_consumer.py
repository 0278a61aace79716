"""The C ABI from a plain C99 program (CPU): include/ssfwd.h compiles as C with
-Wall -Werror, and a program linked against libssfwd.so calls the
validation-only entry points (no CUDA call is made on these inputs) and gets
the documented statuses. This checks the boundary without Python or torch
types in between."""
import os
import shutil
import subprocess
import tempfile

import pytest

from state_space_model_03_gb300 import build as ssbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

C_PROGRAM = r"""
#include <stdint.h>
#include <stdio.h>
#include <string.h>
#include "ssfwd.h"

int main(void) {
  ss_fwd_params p;
  ss_bwd_params q;
  ss_fwd_complex_params x;
  int64_t bytes = -1;
  memset(&p, 0, sizeof(p));
  memset(&q, 0, sizeof(q));
  memset(&x, 0, sizeof(x));
  printf("version %d %d\n", ss_abi_version(), SS_ABI_VERSION);
  printf("null %d\n", ss_fwd_validate(NULL));
  p.abi_version = SS_ABI_VERSION - 1;
  printf("stale %d\n", ss_fwd_validate(&p));
  p.abi_version = SS_ABI_VERSION;
  p.in_dtype = SS_BF16; p.bc_dtype = SS_BF16; p.bc_mode = SS_BC_VARIABLE;
  p.batch = 2; p.dim = 64; p.seqlen = 0; p.dstate = 65; p.ngroups = 1;
  printf("dstate %d\n", ss_fwd_validate(&p));
  p.dstate = 16;
  printf("empty %d\n", ss_fwd_validate(&p));
  q.abi_version = SS_ABI_VERSION;
  q.in_dtype = SS_F32; q.bc_dtype = SS_F32; q.bc_mode = SS_BC_FIXED;
  q.batch = 1; q.dim = 4; q.seqlen = 300; q.dstate = 8;
  printf("bwd_null %d\n", ss_bwd_validate(&q));
  q.seqlen = 0;  /* fake, never dereferenced addresses for the required operands */
  q.A = (const float *)(uintptr_t)0x10000; q.A_stride[0] = 8; q.A_stride[1] = 1;
  q.dA = (float *)(uintptr_t)0x20000; q.dB = (float *)(uintptr_t)0x30000; q.dC = (float *)(uintptr_t)0x40000;
  {
    const int st = ss_bwd_workspace_size(&q, &bytes);  /* before reading bytes */
    printf("bwd_ws %d %d\n", st, (int)bytes);
  }
  x.abi_version = SS_ABI_VERSION;
  x.in_dtype = SS_F16; x.bc_dtype = SS_BF16; x.bc_mode = SS_BC_VARIABLE;
  x.batch = 1; x.dim = 4; x.seqlen = 8; x.dstate = 4; x.ngroups = 1;
  printf("cx_dtype %d\n", ss_fwd_complex_validate(&x));
  printf("text %s\n", ss_status_string(SS_ERR_ALIAS));
  return 0;
}
"""


def test_c_program_against_the_library():
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    lib = ssbuild.build()
    libdir = os.path.dirname(lib)
    with tempfile.TemporaryDirectory() as tmp:
        src = os.path.join(tmp, "consumer.c")
        exe = os.path.join(tmp, "consumer")
        with open(src, "w") as f:
            f.write(C_PROGRAM)
        subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
                        src, "-o", exe, "-L", libdir, "-lssfwd", "-Wl,-rpath," + libdir], check=True)
        r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    got = dict(line.split(" ", 1) for line in r.stdout.strip().splitlines())
    v = got["version"].split()
    assert v[0] == v[1]
    assert got["null"] == "1"          # SS_ERR_NULL
    assert got["stale"] == "10"        # SS_ERR_VERSION
    assert got["dstate"] == "7"        # SS_ERR_UNSUPPORTED
    assert got["empty"] == "0"         # seqlen 0: nothing to check beyond the shape
    assert got["bwd_null"] == "1"      # required gradients missing
    assert got["bwd_ws"] == "0 0"      # an empty sequence needs no workspace
    assert got["cx_dtype"] == "3"      # SS_ERR_DTYPE: fp16 inputs with bf16 B/C
    assert "overlaps" in got["text"]
