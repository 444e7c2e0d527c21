"""Build liba4w4.so in-tree: nvcc for sm_103a only, translation units in parallel.

    python -m mxfp4_a4w4_gemm_gb300.build        (or __graft_entry__.build())

Objects go to ``_build/`` at the repository root and the library to
``mxfp4_a4w4_gemm_gb300/_lib/liba4w4.so``; both are git-ignored.  The library
is rebuilt unless a stamp file beside it records the same build key: a SHA-256
of every source and header, this file, the nvcc flags, the compiler's version
line and the machine architecture.  File modification times play no part, so
a copied tree with preserved or skewed times cannot reuse a stale binary, and
a library built on another architecture is never taken.
"""

import hashlib
import os
import platform
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OBJDIR = os.path.join(ROOT, "_build")
LIBDIR = os.path.join(PKG, "_lib")
LIB = os.path.join(LIBDIR, "liba4w4.so")
STAMP = LIB + ".key"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC,
                     "--expt-relaxed-constexpr"]


def nvcc():
    home = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    path = os.path.join(home, "bin", "nvcc")
    return path if os.path.exists(path) else "nvcc"


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE)]
    return sorted(files) + [os.path.abspath(__file__)]


def _nvcc_version():
    try:
        out = subprocess.run([nvcc(), "--version"], stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True).stdout
    except OSError:
        return "nvcc missing"
    lines = [ln for ln in out.splitlines() if "release" in ln]
    return lines[-1] if lines else out.strip()


def build_key(extra_flags=()):
    """SHA-256 over the sources, headers, build script, flags, nvcc version and machine."""
    h = hashlib.sha256()
    for f in _deps():
        h.update(os.path.relpath(f, ROOT).encode() + b"\0")
        with open(f, "rb") as fh:
            h.update(fh.read())
    h.update(repr((NVCC_FLAGS, list(extra_flags))).encode())
    h.update(_nvcc_version().encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def up_to_date(key):
    """True when the library exists and its stamp records `key`."""
    if not (os.path.exists(LIB) and os.path.exists(STAMP)):
        return False
    with open(STAMP) as fh:
        return fh.read().strip() == key


def build(force=False, verbose=False, extra_flags=()):
    """Compile every CUDA source for sm_103a and link liba4w4.so.  Returns its path."""
    key = build_key(extra_flags)
    if not force and up_to_date(key):
        return LIB
    os.makedirs(OBJDIR, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    procs = []
    objs = []
    for src in sources():
        obj = os.path.join(OBJDIR, os.path.basename(src)[:-3] + ".o")
        objs.append(obj)
        cmd = [nvcc()] + NVCC_FLAGS + list(extra_flags) + ["-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if verbose or p.returncode != 0:
            sys.stdout.write(out)
        if p.returncode != 0:
            failed.append(src)
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(os.path.basename(f) for f in failed))
    tmp = LIB + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lpthread", "-ldl", "-lrt"]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        sys.stdout.write(r.stdout)
        raise RuntimeError("linking liba4w4.so failed")
    os.replace(tmp, LIB)
    with open(STAMP + ".tmp", "w") as fh:
        fh.write(key + "\n")
    os.replace(STAMP + ".tmp", STAMP)
    return LIB


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose=True,
          extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else ())
    print(LIB)
