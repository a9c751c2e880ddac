"""Builds libtrfn.so in-tree: CUDA kernels for sm_103a plus the host C ABI.

`python -m image_preprocessing_gb300.build` (or `__graft_entry__.build()`)
compiles each translation unit in parallel with nvcc and links one shared
library next to this file.  No cmake; a rebuild happens only when a source
or header is newer than the library.
"""
import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtrfn.so")
# the same library with the tiled kernel's bounds and alignment checks
# compiled in (-DTRFN_BOUNDS=1): a failed check sets bit 1 of the device
# status word and skips the access; for tests, never for measurements
LIB_BOUNDS = os.path.join(PKG, "libtrfn_bounds.so")
CHECKED_SOURCE = "fused_norm.cu"
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def _sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def _stale():
    if not os.path.exists(LIB) or not os.path.exists(LIB_BOUNDS):
        return True
    t = min(os.path.getmtime(LIB), os.path.getmtime(LIB_BOUNDS))
    deps = _sources() + glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(INCLUDE, "*.h"))
    return any(os.path.getmtime(d) > t for d in deps)


def _compile(src, checked=False):
    obj = os.path.join(BUILD, os.path.basename(src) + (".bounds.o" if checked else ".o"))
    cmd = [_nvcc(), "-c", *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
           "-I", INCLUDE, "-I", CSRC, "-o", obj, src]
    if checked:
        cmd[2:2] = ["-DTRFN_BOUNDS=1"]
    if src.endswith(".cu"):
        cmd[2:2] = ["-Xptxas", "-v", "--expt-relaxed-constexpr"]
    if os.path.basename(src) == "sampler.cpp":
        # the sampler's binary32 arithmetic must round each operation on its own
        cmd[2:2] = ["-Xcompiler", "-ffp-contract=off"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("compile failed: %s\n%s\n%s" % (" ".join(cmd), r.stdout, r.stderr))
    return obj, r.stderr


def build_library(force=False, verbose=False):
    """Compile and link libtrfn.so; return its path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD, exist_ok=True)
    srcs = _sources()
    checked_src = os.path.join(CSRC, CHECKED_SOURCE)
    jobs = [(s, False) for s in srcs] + [(checked_src, True)]
    with cf.ThreadPoolExecutor(max_workers=max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
        results = list(ex.map(lambda j: _compile(*j), jobs))
    with open(os.path.join(BUILD, "ptxas.log"), "w") as f:
        for (obj, log), (src, checked) in zip(results, jobs):
            if not checked:
                f.write("== %s\n%s\n" % (os.path.basename(src), log))
    plain = [o for (o, _), (_, checked) in zip(results, jobs) if not checked]
    bounds = [o for (o, _), (src, checked) in zip(results, jobs)
              if checked or os.path.basename(src) != CHECKED_SOURCE]
    for lib, objs in ((LIB, plain), (LIB_BOUNDS, bounds)):
        tmp = lib + ".tmp%d" % os.getpid()
        cmd = [_nvcc(), "-shared", *ARCH, "-o", tmp] + objs + ["-lpthread", "-ldl", "-lrt"]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("link failed: %s\n%s\n%s" % (" ".join(cmd), r.stdout, r.stderr))
        os.replace(tmp, lib)
    if verbose:
        for (obj, log), (src, checked) in zip(results, jobs):
            if log.strip() and not checked:
                print("==", os.path.basename(src))
                print(log)
    return LIB


if __name__ == "__main__":
    print(build_library(force="--force" in sys.argv, verbose="-v" in sys.argv))
