"""Build the CUDA library (libgpt2.so) in-tree for sm_103a with nvcc.

Each source is compiled to its own object in parallel (objects under
_build/ beside the package), then the objects are linked into one shared
library.

Usage: python -m gpt_transformer_train_b300.build   (or build() from Python)
"""
import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OBJ = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libgpt2.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-ffp-contract=off"]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))


def headers():
    return glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))


def needs_build():
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    return any(os.path.getmtime(d) > t for d in sources() + headers())


def _obj(src):
    return os.path.join(OBJ, os.path.basename(src) + ".o")


def _compile(src, verbose):
    cmd = [NVCC, *ARCH, *FLAGS, "-I" + os.path.join(ROOT, "include"), "-c", src, "-o", _obj(src)]
    if verbose:
        cmd.insert(1, "-Xptxas=-v")
    r = subprocess.run(cmd, capture_output=True, text=True)
    return src, r.returncode, r.stdout + r.stderr


def build(force=False, verbose=False):
    if not force and not needs_build():
        return LIB
    os.makedirs(OBJ, exist_ok=True)
    hdr_t = max(os.path.getmtime(h) for h in headers())
    todo = [s for s in sources() if force or verbose or not os.path.exists(_obj(s)) or
            os.path.getmtime(_obj(s)) < max(os.path.getmtime(s), hdr_t)]
    with ThreadPoolExecutor(max_workers=max(1, min(len(todo), os.cpu_count() or 4))) as ex:
        results = list(ex.map(lambda s: _compile(s, verbose), todo))
    failed = [(s, out) for s, rc, out in results if rc != 0]
    for s, rc, out in results:
        if out.strip():  # errors, warnings, and with verbose the ptxas report
            sys.stderr.write(out)
    if failed:
        raise RuntimeError("nvcc failed building " + ", ".join(os.path.basename(s) for s, _ in failed))
    cmd = [NVCC, *ARCH, "-shared", "-o", LIB + ".tmp", *[_obj(s) for s in sources()], "-lpthread"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("nvcc failed linking libgpt2.so")
    os.replace(LIB + ".tmp", LIB)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIB)
