"""Builds libvr.so in-tree: one nvcc process per translation unit, in
parallel, for sm_103a only, then one link.  Run ``python -m
double_binary_tree_gb300.build`` or call ``build()``.

The bounds-checked build libvr_debug.so (every kernel access checked against
its call's buffers; -DVR_DEBUG_BOUNDS) is compiled from the same sources in
the same parallel batch (``build(debug=True)`` builds both)."""

import os
import platform
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIB = os.path.join(HERE, "libvr.so")
LIB_DEBUG = os.path.join(HERE, "libvr_debug.so")
SOURCES = ["topology.cc", "api.cc", "kernels_f32.cu", "kernels_f16.cu", "kernels_bf16.cu",
           "kernels_copy.cu", "kernels_ablation.cu", "noalloc.cu", "jit.cc",
           "costmodel.cc", "options.cc", "graphlog.cc"]
HEADERS = ["common.h", "host.h", "fold.cuh", "kernels.cuh", "staged.cuh", "ablation.cuh",
           "gather.cuh", "bounds.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _build_dir(debug=False):
    return os.path.join(HERE, "_build", platform.machine() + ("-debug" if debug else ""))


def _stamp(debug=False):
    return os.path.join(_build_dir(debug), "libvr.stamp")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "vr.h"))
    files.append(os.path.abspath(__file__))
    return files


def is_fresh(debug=False):
    """True when the library (the bounds-checked one when `debug`) was built
    on this machine type after every source."""
    lib = LIB_DEBUG if debug else LIB
    if not (os.path.exists(lib) and os.path.exists(_stamp(debug))):
        return False
    t = os.path.getmtime(_stamp(debug))
    return all(os.path.getmtime(f) <= t for f in _inputs()) and os.path.getmtime(lib) <= t + 5


def build(force=False, verbose=False, ptxas_info=False, debug=False):
    """Compile and link libvr.so unless it is fresh (and libvr_debug.so too
    when `debug`).  Returns the path of libvr.so."""
    variants = [v for v in ([False, True] if debug else [False]) if force or not is_fresh(v)]
    if not variants:
        return LIB
    nvcc = _nvcc()
    common = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "-I" + INCLUDE,
              "-I" + CSRC] + ARCH
    if ptxas_info:
        common += ["-Xptxas", "-v"]
    # extra flags for tuning experiments (e.g. -DVR_MIN_BLOCKS_RING=2)
    common += os.environ.get("VR_NVCC_FLAGS", "").split()
    procs, objs = [], {v: [] for v in variants}
    for v in variants:
        bdir = _build_dir(v)
        os.makedirs(bdir, exist_ok=True)
        for src in SOURCES:
            obj = os.path.join(bdir, src + ".o")
            objs[v].append(obj)
            cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", obj] + common
            if v:
                cmd.append("-DVR_DEBUG_BOUNDS=1")
            if verbose:
                print(" ".join(cmd), file=sys.stderr)
            procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE,
                                                stderr=subprocess.STDOUT)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        text = out.decode(errors="replace")
        if p.returncode != 0:
            failed.append("%s:\n%s" % (src, text))
        elif verbose or ptxas_info:
            sys.stderr.write(text)
    if failed:
        raise RuntimeError("nvcc failed\n" + "\n".join(failed))
    for v in variants:
        lib = LIB_DEBUG if v else LIB
        tmp = lib + ".tmp"
        link = [nvcc, "-shared", "-o", tmp] + objs[v] + ARCH + ["-cudart", "static", "-ldl"]
        r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
        if r.returncode != 0:
            raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
        os.replace(tmp, lib)
        with open(_stamp(v), "w") as f:
            f.write(platform.machine() + "\n")
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv,
          ptxas_info="--ptxas" in sys.argv, debug="--debug" in sys.argv)
    print(LIB)
