"""Build ``libtq.so`` (the C-ABI library) in-tree for sm_103a with nvcc.

    python -m decode_attention_21_b300.build [--debug]

Compiles every ``csrc/*.cu`` / ``csrc/*.cpp`` into one shared library next to
this file, statically linked against the CUDA runtime so it loads on a
machine without a GPU driver (the symbol-export tests run there).
"""
import argparse
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
OUT = os.path.join(HERE, "libtq.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc():
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def build(debug=False, verbose=False, out=OUT):
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    objdir = os.path.join(HERE, "_build")
    os.makedirs(objdir, exist_ok=True)
    common = ARCH + ["-std=c++17", "-lineinfo", "-O3", "-Xcompiler", "-fPIC,-O2",
                     "-I" + os.path.join(ROOT, "include"), "-I" + CSRC]
    if debug:
        common += ["-DTQ_DEBUG"]
    if verbose:
        common += ["-Xptxas", "-v"]
    objs = []
    for s in srcs:
        o = os.path.join(objdir, os.path.basename(s) + ".o")
        cmd = [nvcc()] + common + ["-c", s, "-o", o]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if verbose or r.returncode:
            sys.stderr.write(r.stdout + r.stderr)
        if r.returncode:
            raise RuntimeError("nvcc failed on " + s)
        objs.append(o)
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", out] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("link failed")
    return out


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("--debug", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    a = ap.parse_args()
    print(build(a.debug, a.verbose))
