"""Builds libssfwd.so in-tree (state_space_model_03_gb300/_build/) with nvcc
for sm_103a only. Translation units compile in parallel; the library links the
CUDA runtime statically and reaches the driver's tensor-map encoder through the
runtime's driver entry-point query, so it needs no libcuda at link time.
"""
from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT = os.path.join(PKG, "_build")
LIB = os.path.join(OUT, "libssfwd.so")
SOURCES = ["ssfwd_api.cu", "ss_fwd_f32.cu", "ss_fwd_f16.cu", "ss_fwd_bf16.cu", "ss_fwd_lane.cu", "ss_state_update.cu", "ss_conv1d.cu", "ss_bwd.cu", "ss_fwd_complex.cu"]
HEADERS = ["ss_dispatch.h", "ss_fwd_kernel.cuh", "ss_fwd_instances.cuh"]
NVCC = os.environ.get("NVCC", "nvcc")
FLAGS = ["-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-lineinfo",
         "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "include"), "-I", CSRC]


def _stale(obj: str, src: str) -> bool:
    if not os.path.exists(obj):
        return True
    deps = [src] + [os.path.join(os.path.dirname(src), h) for h in HEADERS] + [os.path.join(ROOT, "include", "ssfwd.h")]
    return any(os.path.getmtime(d) > os.path.getmtime(obj) for d in deps)


def build(force: bool = False, verbose: bool = False, out_dir: str = OUT, extra_flags=(), csrc: str = CSRC) -> str:
    """Compile the library into out_dir/libssfwd.so from the sources in csrc;
    extra_flags (e.g. -D knobs) are passed to every nvcc compile."""
    os.makedirs(out_dir, exist_ok=True)
    lib = os.path.join(out_dir, "libssfwd.so")
    jobs = []
    for src in SOURCES:
        s = os.path.join(csrc, src)
        o = os.path.join(out_dir, src.replace(".cu", ".o"))
        if force or _stale(o, s):
            jobs.append((s, o))

    def compile_one(job):
        s, o = job
        cmd = [NVCC, *FLAGS, "-I", csrc, *extra_flags, "-c", s, "-o", o + ".tmp"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {s}:\n{r.stdout}\n{r.stderr}")
        os.replace(o + ".tmp", o)
        if verbose:
            print(r.stderr, file=sys.stderr)

    if jobs:
        with ThreadPoolExecutor(len(jobs)) as ex:
            list(ex.map(compile_one, jobs))
    objs = [os.path.join(out_dir, s.replace(".cu", ".o")) for s in SOURCES]
    if force or jobs or not os.path.exists(lib):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [NVCC, "-shared", "-gencode", "arch=compute_103a,code=sm_103a", "-cudart", "static",
               "-o", tmp, *objs]
        subprocess.run(cmd, check=True, capture_output=True, text=True)
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
