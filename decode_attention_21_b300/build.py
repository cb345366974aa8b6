"""Build ``libtq.so`` (the C-ABI library) in-tree for sm_103a with nvcc.

    python -m decode_attention_21_b300.build [-v]

Compiles every ``csrc/*.cu`` / ``csrc/*.cpp`` into one shared library next to
this file, statically linked against the CUDA runtime so it loads on a
machine without a GPU driver (the symbol-export tests run there).
"""
import argparse
import concurrent.futures
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


def build(verbose=False, out=OUT):
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    objdir = os.path.join(HERE, "_build")
    os.makedirs(objdir, exist_ok=True)
    common = ARCH + ["-std=c++17", "-lineinfo", "-O3", "-Xcompiler", "-fPIC,-O2",
                     "-I" + os.path.join(ROOT, "include"), "-I" + CSRC]
    if verbose:
        common += ["-Xptxas", "-v"]
    def compile_one(s):
        o = os.path.join(objdir, os.path.basename(s) + ".o")
        r = subprocess.run([nvcc()] + common + ["-c", s, "-o", o], capture_output=True, text=True)
        return s, o, r

    objs = []
    with concurrent.futures.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 1)) as ex:
        for s, o, r in ex.map(compile_one, srcs):
            if verbose or r.returncode:
                sys.stderr.write(r.stdout + r.stderr)
            if r.returncode:
                raise RuntimeError("nvcc failed on " + s)
            objs.append(o)
    cmd = [nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", out] + objs + ["-ldl"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode:
        sys.stderr.write(r.stdout + r.stderr)
        raise RuntimeError("link failed")
    return out


if __name__ == "__main__":
    ap = argparse.ArgumentParser()
    ap.add_argument("-v", "--verbose", action="store_true")
    a = ap.parse_args()
    print(build(verbose=a.verbose))
