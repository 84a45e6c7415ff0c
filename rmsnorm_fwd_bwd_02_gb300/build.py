"""Build librmsnorm.so (the C-ABI CUDA library) in-tree for sm_103a.

Each translation unit under csrc/ is compiled by nvcc in parallel into
_build/, then linked into rmsnorm_fwd_bwd_02_gb300/librmsnorm.so. A unit is
rebuilt when it, any header under csrc/ or include/, or this file is newer
than its object. No cmake; plain nvcc with one -gencode.

    python -m rmsnorm_fwd_bwd_02_gb300.build [--force] [--ptxas-verbose]
"""
import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "librmsnorm.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "-I" + INCLUDE, "-I" + CSRC]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _newest_dep_mtime():
    deps = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(
        os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    deps.append(os.path.abspath(__file__))
    return max(os.path.getmtime(d) for d in deps)


def _compile(src, obj, extra):
    cmd = [_nvcc()] + NVCC_FLAGS + extra + ["-c", src, "-o", obj + ".tmp"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n"
                           f"{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    os.replace(obj + ".tmp", obj)
    return r.stdout + r.stderr


def build(force: bool = False, ptxas_verbose: bool = False, jobs: int = 0) -> str:
    os.makedirs(BUILD, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    dep_t = _newest_dep_mtime()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    todo = []
    objs = []
    for s in sources:
        o = os.path.join(BUILD, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if (force or ptxas_verbose or not os.path.exists(o)
                or os.path.getmtime(o) < max(dep_t, os.path.getmtime(s))):
            todo.append((s, o))
    logs = []
    if todo:
        n = jobs or min(len(todo), os.cpu_count() or 4)
        with ThreadPoolExecutor(max_workers=n) as ex:
            for log in ex.map(lambda so: _compile(so[0], so[1], extra), todo):
                logs.append(log)
    if (todo or not os.path.exists(LIB)
            or os.path.getmtime(LIB) < max(os.path.getmtime(o) for o in objs)):
        tmp = LIB + ".tmp.%d" % os.getpid()
        cmd = [_nvcc()] + ARCH + ["-shared", "-o", tmp] + objs
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, LIB)
    if ptxas_verbose:
        sys.stdout.write("".join(logs))
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv,
                ptxas_verbose="--ptxas-verbose" in sys.argv))
