"""Build libtg.so in-tree: one nvcc per translation unit in parallel, then link.

Only sm_103a is targeted (-gencode arch=compute_103a,code=sm_103a). The host
part (packer) is plain portable C++17, so the same sources build on x86_64
and aarch64 hosts. The CUDA runtime is linked shared so the process uses one
runtime together with PyTorch.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtg.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cpp")))


def headers():
    out = [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    out += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    return out


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(p) > t for p in sources() + headers() + [__file__, os.path.join(CSRC, "tgpy.c")])


def build(force: bool = False, verbose: bool = False, extra=()) -> str:
    if not force and not _stale():
        return LIB
    nvcc = _nvcc()
    os.makedirs(BUILD, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(BUILD, os.path.basename(src) + ".o")
        if src.endswith(".cu"):
            cmd = [nvcc, *ARCH, *COMMON, *extra, "-c", src, "-o", obj]
        else:
            cmd = [nvcc, *COMMON, "-x", "c++", "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError(f"compile failed: {src}")
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = LIB + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "shared", "-o", tmp, *objs, "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode:
        sys.stderr.write(" ".join(cmd) + "\n" + r.stdout + r.stderr)
        raise RuntimeError("link failed")
    os.replace(tmp, LIB)
    _build_tgpy()
    return LIB


def _build_tgpy() -> None:
    """The optional CPython call path to tg_gemv_i8 (csrc/tgpy.c), linked against the
    in-tree libtg.so; skipped with a note if there is no C compiler or no Python headers
    (the binding then calls through ctypes)."""
    import sysconfig
    src = os.path.join(CSRC, "tgpy.c")
    out = os.path.join(PKG, "_tgpy" + (sysconfig.get_config_var("EXT_SUFFIX") or ".so"))
    inc = sysconfig.get_paths().get("include", "")
    cc = os.environ.get("CC") or shutil.which("gcc") or shutil.which("cc")
    if not cc or not os.path.exists(os.path.join(inc, "Python.h")):
        sys.stderr.write("note: _tgpy not built (no C compiler or Python headers); the binding uses ctypes\n")
        return
    tmp = out + f".tmp{os.getpid()}"
    cmd = [cc, "-O2", "-shared", "-fPIC", "-I", inc, "-I", INCLUDE, src, "-o", tmp, "-L", PKG, "-l:libtg.so",
           "-Wl,-rpath,$ORIGIN"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode:
        sys.stderr.write("note: _tgpy not built; the binding uses ctypes\n" + " ".join(cmd) + "\n" + r.stderr[-2000:])
        return
    os.replace(tmp, out)


if __name__ == "__main__":
    extra = [a for a in sys.argv[1:] if a.startswith("-X") or a.startswith("--")]
    extra = [a for a in extra if a not in ("--force", "--verbose")]
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv, extra=extra))
