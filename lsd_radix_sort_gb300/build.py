"""Build ``liblsdrs.so`` (the C-ABI sort library) in-tree for sm_103a.

Each ``csrc/*.cu`` translation unit is compiled by nvcc in parallel, then
linked into ``lsd_radix_sort_gb300/_build/liblsdrs.so`` against the shared
CUDA runtime (so that it shares the runtime PyTorch loads).

    python -m lsd_radix_sort_gb300.build [--force] [--verbose-ptxas]
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
ROOT = os.path.dirname(HERE)
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(BUILD, "liblsdrs.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
              "--expt-relaxed-constexpr", "-I", INCLUDE]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def cuda_lib_dir() -> str:
    base = os.path.dirname(os.path.dirname(os.path.realpath(nvcc())))
    for d in ("lib64", "lib", "targets/sbsa-linux/lib", "targets/x86_64-linux/lib"):
        p = os.path.join(base, d)
        if os.path.exists(os.path.join(p, "libcudart.so")) or os.path.isdir(p):
            return p
    return "/usr/local/cuda/lib64"


def sources() -> list[str]:
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "lsdrs.h"))
    files.append(os.path.abspath(__file__))
    return max(os.path.getmtime(f) for f in files)


def up_to_date() -> bool:
    return os.path.exists(LIB) and os.path.getmtime(LIB) >= _deps_mtime()


def build(force: bool = False, verbose_ptxas: bool = False, jobs: int | None = None,
          defines: list[str] | None = None, out: str | None = None) -> str:
    """Compile and link; ``defines``/``out`` build a variant library elsewhere."""
    lib = out or LIB
    if not force and not defines and out is None and up_to_date():
        return LIB
    bdir = os.path.dirname(lib) if out else BUILD
    os.makedirs(bdir, exist_ok=True)
    dflags = [f"-D{d}" for d in (defines or [])]
    srcs = sources()
    extra = ["-Xptxas", "-v"] if verbose_ptxas else []

    def compile_one(src: str):
        obj = os.path.join(bdir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc(), *ARCH, *NVCC_FLAGS, *dflags, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    jobs = jobs or min(len(srcs), os.cpu_count() or 1)
    with ThreadPoolExecutor(jobs) as ex:
        results = list(ex.map(compile_one, srcs))
    failed = [(s, r) for s, _, r in results if r.returncode != 0]
    for s, _, r in results:
        if verbose_ptxas or r.returncode != 0:
            sys.stderr.write(f"== {os.path.basename(s)}\n{r.stdout}{r.stderr}")
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(os.path.basename(s) for s, _ in failed))
    tmp = lib + f".tmp{os.getpid()}"
    libdir = cuda_lib_dir()
    cmd = [nvcc(), *ARCH, "-shared", "-cudart", "shared", "-o", tmp,
           *[o for _, o, _ in results], "-Xlinker", f"-rpath,{libdir}"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, lib)
    return lib


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("--verbose-ptxas", action="store_true")
    ap.add_argument("-D", dest="defines", action="append", default=[])
    ap.add_argument("--out", default=None)
    args = ap.parse_args()
    print(build(force=args.force, verbose_ptxas=args.verbose_ptxas, defines=args.defines,
                out=args.out))


if __name__ == "__main__":
    main()
