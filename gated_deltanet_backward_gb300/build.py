"""Builds libgdn.so (the C-ABI library) for sm_103a with nvcc.

Each translation unit under csrc/ is compiled in parallel, then linked into a
shared library next to this file.  Re-running rebuilds only what changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT = os.path.join(HERE, "libgdn.so")
OBJ = os.path.join(HERE, "_build")
SOURCES = ["gdn_api.cu", "gdn_fwd.cu", "gdn_bwd.cu", "gdn_tc_fwd.cu", "gdn_tc_bwd.cu",
           "gdn_tc_kda.cu", "gdn_noalloc.cu", "gdn_decode.cu", "gdn_neighbours.cu",
           "gdn_context.cu", "gdn_kda.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(cuda, "bin", "nvcc")
    return path if os.path.exists(path) else (shutil.which("nvcc") or "nvcc")


def _flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE,
                   "-I", CSRC, "--expt-relaxed-constexpr"] + list(extra)


def _headers():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))] + [
        os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]


def _stale(target, deps):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(verbose: bool = False, extra_flags=(), force: bool = False) -> str:
    os.makedirs(OBJ, exist_ok=True)
    nvcc = _nvcc()
    hdrs = _headers()
    jobs = []
    objs = []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(OBJ, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s, __file__] + hdrs):
            jobs.append([nvcc] + _flags(extra_flags) + ["-c", s, "-o", o])

    def run(cmd):
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed:\n%s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)

    with cf.ThreadPoolExecutor(max_workers=max(1, len(jobs))) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(OUT, objs):
        tmp = OUT + ".tmp%d" % os.getpid()
        run([nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", tmp] + objs)
        os.replace(tmp, OUT)
    return OUT


def build_variant(out_path: str, defines, sources=("gdn_tc_fwd.cu", "gdn_tc_bwd.cu"),
                  verbose: bool = False) -> str:
    """A second copy of the library at out_path whose `sources` are compiled with extra
    preprocessor definitions (e.g. {"GDN_FLAG_WAIT_LIMIT_NS": 0}); the other translation
    units are the regular build's objects.  Builds the regular library first."""
    build(verbose=verbose)
    nvcc = _nvcc()
    work = os.path.dirname(os.path.abspath(out_path))
    os.makedirs(work, exist_ok=True)
    dflags = ["-D%s=%s" % (k, v) for k, v in sorted(dict(defines).items())]
    objs = []
    for src in SOURCES:
        if src in sources:
            o = os.path.join(work, src.replace(".cu", ".variant.o"))
            cmd = [nvcc] + _flags(dflags) + ["-c", os.path.join(CSRC, src), "-o", o]
            r = subprocess.run(cmd, capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError("nvcc failed:\n%s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
            objs.append(o)
        else:
            objs.append(os.path.join(OBJ, src.replace(".cu", ".o")))
    cmd = [nvcc] + ARCH + ["-shared", "-cudart", "shared", "-o", out_path] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s%s" % (" ".join(cmd), r.stdout, r.stderr))
    return out_path


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, force="-f" in sys.argv))
