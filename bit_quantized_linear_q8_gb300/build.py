"""Builds libbq8.so in-tree for sm_103a (GB300).

Each ``csrc/*.cu`` is compiled in parallel with one ``-gencode`` (compute_103a ->
sm_103a), then linked with ``nvcc -shared``.  The CUDA runtime is linked statically
(nvcc's default), so the library depends only on the driver.  Re-running is cheap:
objects newer than every source and header are reused.
"""
import concurrent.futures as cf
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(OUT_DIR, "libbq8.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-I" + INCLUDE, "-I" + CSRC] + ARCH


def _nvcc():
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(INCLUDE, "*.h"))


def _compile(src, obj, verbose):
    cmd = [_nvcc(), "-c", src, "-o", obj] + NVCC_FLAGS + (["-Xptxas", "-v"] if verbose else [])
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
    return r.stderr


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(OUT_DIR, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    newest_hdr = max([os.path.getmtime(h) for h in _headers()] + [0])
    jobs = []
    for s in srcs:
        obj = os.path.join(OUT_DIR, os.path.basename(s)[:-3] + ".o")
        stale = force or not os.path.exists(obj) or os.path.getmtime(obj) < max(os.path.getmtime(s), newest_hdr)
        jobs.append((s, obj, stale))
    logs = []
    with cf.ThreadPoolExecutor(max_workers=min(8, len(jobs) or 1)) as ex:
        futs = [ex.submit(_compile, s, o, verbose) for s, o, stale in jobs if stale]
        for f in futs:
            logs.append(f.result())
    objs = [o for _, o, _ in jobs]
    if force or any(st for _, _, st in jobs) or not os.path.exists(LIB):
        tmp = LIB + ".tmp.%d" % os.getpid()
        cmd = [_nvcc(), "-shared", "-o", tmp] + objs + ARCH + ["-Xcompiler", "-fPIC"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc link failed:\n%s\n%s" % (r.stdout, r.stderr))
        os.replace(tmp, LIB)
    if verbose:
        for line in logs:
            sys.stdout.write(line)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
