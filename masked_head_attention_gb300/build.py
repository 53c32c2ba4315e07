"""Build libmha.so (the CUDA kernels and the C ABI) in-tree for sm_103a.

Each .cu translation unit is compiled in parallel with nvcc, then linked into
masked_head_attention_gb300/_lib/libmha.so.  Rebuilds only when a source or
header is newer than the library.
"""
import concurrent.futures as cf
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT_DIR = os.path.join(HERE, "_lib")
LIB = os.path.join(OUT_DIR, "libmha.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC = os.environ.get("NVCC", "nvcc")


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return (_sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h"))
            + glob.glob(os.path.join(ROOT, "include", "*.h")) + [os.path.abspath(__file__)])


def _flags(extra):
    return ["-O3", "-std=c++17", *ARCH, "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler",
            "-fvisibility=hidden", "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include"),
            *extra]


def up_to_date(lib=LIB):
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(d) <= t for d in _deps())


def build(force=False, verbose=False, extra=(), lib=LIB, ptxas_info=False):
    """Compile and link; returns the library path."""
    if not force and not extra and up_to_date(lib):
        return lib
    os.makedirs(OUT_DIR, exist_ok=True)
    flags = _flags(list(extra) + (["-Xptxas", "-v"] if ptxas_info else []))
    objs = []
    jobs = []
    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        for src in _sources():
            obj = os.path.join(OUT_DIR, os.path.basename(src)[:-3] + ".o")
            objs.append(obj)
            cmd = [NVCC, *flags, "-c", src, "-o", obj]
            jobs.append(ex.submit(subprocess.run, cmd, capture_output=True, text=True))
        results = [j.result() for j in jobs]
    for src, r in zip(_sources(), results):
        if verbose or ptxas_info or r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed on %s" % os.path.basename(src))
    tmp = lib + ".tmp%d" % os.getpid()
    link = [NVCC, "-shared", *ARCH, "-o", tmp, *objs, "-lcudart_static", "-ldl", "-lpthread", "-lrt"]
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("link failed")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
