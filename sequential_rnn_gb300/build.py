"""Build the in-tree shared library libsrnn.so for sm_103a.

Each CUDA translation unit is compiled in parallel with nvcc
(-gencode arch=compute_103a,code=sm_103a), then linked with the static CUDA
runtime into sequential_rnn_gb300/libsrnn.so.  Objects go to
sequential_rnn_gb300/_build/.  Usage:  python -m sequential_rnn_gb300.build

The bounds-check variant (-DRNN_BOUNDS_CHECK: every computed index checked,
violations reported as RNN_ERR_BOUNDS) goes to libsrnn_bc.so via
_build_bc/:  python -m sequential_rnn_gb300.build -bc
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libsrnn.so")
LIB_BC = os.path.join(PKG, "libsrnn_bc.so")

SOURCES = ["capi.cu", "plan.cu", "runtime.cu", "fwd_f32.cu", "fwd_bf16_lstm.cu", "fwd_bf16_gru.cu", "fwd_bf16_slstm.cu",
           "floor.cu", "bwd_cell.cu", "grad_weights.cu", "tc_gemm.cu", "tc_gemm_pair.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def build(verbose: bool = False, force: bool = False, bounds_check: bool = False) -> str:
    bdir = BUILD + "_bc" if bounds_check else BUILD
    lib = LIB_BC if bounds_check else LIB
    flags = FLAGS + (["-DRNN_BOUNDS_CHECK"] if bounds_check else [])
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    srcs = [s for s in SOURCES if os.path.exists(os.path.join(CSRC, s))]
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(ROOT, "include", "rnn.h")]
    newest_dep = max(os.path.getmtime(f) for f in deps)
    procs = []
    objs = []
    for s in srcs:
        obj = os.path.join(bdir, s.replace(".cu", ".o"))
        objs.append(obj)
        if not force and os.path.exists(obj) and os.path.getmtime(obj) >= newest_dep:
            continue
        cmd = [cc, *ARCH, *flags, "-c", os.path.join(CSRC, s), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((s, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
    failed = []
    for s, p in procs:
        out, _ = p.communicate()
        if p.returncode != 0:
            failed.append((s, out.decode(errors="replace")))
        elif verbose and out:
            print(out.decode(errors="replace"))
    if failed:
        msg = "\n".join(f"--- {s}\n{o}" for s, o in failed)
        raise RuntimeError(f"nvcc failed:\n{msg}")
    if force or not os.path.exists(lib) or any(os.path.getmtime(o) > os.path.getmtime(lib) for o in objs):
        cmd = [cc, *ARCH, "-shared", "-o", lib + ".tmp", *objs, "-cudart", "static"]
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
        os.replace(lib + ".tmp", lib)
    return lib


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv, bounds_check="-bc" in sys.argv))
