"""Build libmoe.so in-tree with nvcc for sm_103a (GB300).

    python -m token_dispatch_gb300.build [--verbose]

Every ``csrc/*.cu`` is compiled in parallel to an object under ``_build/`` and
linked into ``token_dispatch_gb300/libmoe.so`` against the shared CUDA runtime.
``ptxas -v`` resource usage (registers, spills, shared memory) is kept in
``_build/ptxas.log``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libmoe.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def cuda_lib_dir(nv: str) -> str:
    root = os.path.dirname(os.path.dirname(os.path.realpath(nv)))
    for d in ("lib64", "lib", os.path.join("targets", "sbsa-linux", "lib"),
              os.path.join("targets", "x86_64-linux", "lib")):
        p = os.path.join(root, d)
        if os.path.exists(os.path.join(p, "libcudart.so")):
            return p
    return os.path.join(root, "lib64")


def _compile(nv: str, src: str, obj: str) -> tuple[str, int, str]:
    cmd = [nv, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-fvisibility=hidden",
           "-Xptxas", "-v", "--expt-relaxed-constexpr", "-I", os.path.dirname(PKG),
           "-c", src, "-o", obj]
    p = subprocess.run(cmd, capture_output=True, text=True)
    return src, p.returncode, p.stdout + p.stderr


def build(verbose: bool = False, force: bool = False) -> str:
    nv = nvcc()
    os.makedirs(BUILD, exist_ok=True)
    sources = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    headers = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    headers.append(os.path.join(os.path.dirname(PKG), "include", "moe.h"))
    newest_header = max(os.path.getmtime(h) for h in headers if os.path.exists(h))
    jobs = []
    for f in sources:
        src = os.path.join(CSRC, f)
        obj = os.path.join(BUILD, f[:-3] + ".o")
        stale = force or not os.path.exists(obj) or os.path.getmtime(obj) < max(os.path.getmtime(src), newest_header)
        jobs.append((src, obj, stale))
    logs = []
    with cf.ThreadPoolExecutor(max_workers=min(8, max(1, len(jobs)))) as ex:
        futs = [ex.submit(_compile, nv, s, o) for s, o, stale in jobs if stale]
        for fu in futs:
            src, rc, out = fu.result()
            logs.append(f"== {os.path.basename(src)}\n{out}")
            if rc != 0:
                raise RuntimeError(f"nvcc failed for {src}:\n{out}")
    if logs:
        with open(os.path.join(BUILD, "ptxas.log"), "w") as fh:
            fh.write("\n".join(logs))
        if verbose:
            print("\n".join(logs))
    objs = [o for _, o, _ in jobs]
    if force or logs or not os.path.exists(LIB) or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs):
        libdir = cuda_lib_dir(nv)
        cmd = [nv, *ARCH, "-shared", "-cudart", "shared", "-o", LIB, *objs,
               "-Xlinker", f"-rpath={libdir}", "-L", libdir]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode != 0:
            raise RuntimeError(f"link failed:\n{p.stdout}{p.stderr}")
    return LIB


if __name__ == "__main__":
    print(build(verbose="--verbose" in sys.argv, force="--force" in sys.argv))
