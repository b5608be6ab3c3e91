"""Builds libvr.so in-tree: one nvcc process per translation unit, in
parallel, for sm_103a only, then one link.  Run ``python -m
double_binary_tree_gb300.build`` or call ``build()``."""

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
SOURCES = ["topology.cc", "api.cc", "kernels_f32.cu", "kernels_f16.cu", "kernels_bf16.cu",
           "kernels_copy.cu", "kernels_ablation.cu", "noalloc.cu", "jit.cc",
           "costmodel.cc", "options.cc", "graphlog.cc"]
HEADERS = ["common.h", "host.h", "fold.cuh", "kernels.cuh", "staged.cuh", "ablation.cuh", "gather.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _build_dir():
    return os.path.join(HERE, "_build", platform.machine())


def _stamp():
    return os.path.join(_build_dir(), "libvr.stamp")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "vr.h"))
    files.append(os.path.abspath(__file__))
    return files


def is_fresh():
    """True when libvr.so was built on this machine type after every source."""
    if not (os.path.exists(LIB) and os.path.exists(_stamp())):
        return False
    t = os.path.getmtime(_stamp())
    return all(os.path.getmtime(f) <= t for f in _inputs()) and os.path.getmtime(LIB) <= t + 5


def build(force=False, verbose=False, ptxas_info=False):
    """Compile and link libvr.so unless it is fresh.  Returns its path."""
    if not force and is_fresh():
        return LIB
    nvcc = _nvcc()
    bdir = _build_dir()
    os.makedirs(bdir, exist_ok=True)
    common = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-O2", "-I" + INCLUDE,
              "-I" + CSRC] + ARCH
    if ptxas_info:
        common += ["-Xptxas", "-v"]
    # extra flags for tuning experiments (e.g. -DVR_MIN_BLOCKS_RING=2)
    common += os.environ.get("VR_NVCC_FLAGS", "").split()
    procs, objs = [], []
    for src in SOURCES:
        obj = os.path.join(bdir, src + ".o")
        objs.append(obj)
        cmd = [nvcc, "-c", os.path.join(CSRC, src), "-o", obj] + common
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)))
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
    tmp = LIB + ".tmp"
    link = [nvcc, "-shared", "-o", tmp] + objs + ARCH + ["-cudart", "static", "-ldl"]
    r = subprocess.run(link, stdout=subprocess.PIPE, stderr=subprocess.STDOUT)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + r.stdout.decode(errors="replace"))
    os.replace(tmp, LIB)
    with open(_stamp(), "w") as f:
        f.write(platform.machine() + "\n")
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv,
          ptxas_info="--ptxas" in sys.argv)
    print(LIB)
