"""Build the codec's shared library (libcachegen.so) in-tree with nvcc for
sm_103a. The translation units compile in parallel; the result is reused
while the sources, headers and flags are unchanged."""
from __future__ import annotations

import hashlib
import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(OUT_DIR, "libcachegen.so")

SOURCES = ["cachegen_kernels.cu", "cachegen_api.cu", "cachegen_noalloc.cu", "cachegen_int8.cu"]
HEADERS = [os.path.join(CSRC, "cg_internal.h"), os.path.join(INCLUDE, "cachegen.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xptxas", "-v",
         "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    cand = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "bin", "nvcc")
    return cand if os.path.exists(cand) else "nvcc"


def _digest() -> str:
    h = hashlib.sha256()
    for p in [os.path.join(CSRC, s) for s in SOURCES] + HEADERS:
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(ARCH + FLAGS).encode())
    return h.hexdigest()


def _compile(out_dir: str, lib: str, defines=()) -> str:
    nvcc = _nvcc()
    extra = ["-D" + d for d in defines]
    procs, objs = [], []
    for s in SOURCES:
        obj = os.path.join(out_dir, s.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [nvcc] + ARCH + FLAGS + extra + ["-c", os.path.join(CSRC, s), "-o", obj]
        procs.append((cmd, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT,
                                            text=True)))
    log = []
    for cmd, p in procs:
        out, _ = p.communicate()
        log.append(out)
        if p.returncode != 0:
            raise RuntimeError("nvcc failed:\n" + " ".join(cmd) + "\n" + out)
    tmp = lib + f".tmp{os.getpid()}"
    link = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(link, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n" + " ".join(link) + "\n" + r.stdout + r.stderr)
    os.replace(tmp, lib)
    with open(os.path.join(out_dir, "ptxas.log"), "w") as f:
        f.write("\n".join(log))
    return "\n".join(log)


def _build_into(out_dir: str, defines=(), force: bool = False, verbose: bool = False) -> str:
    os.makedirs(out_dir, exist_ok=True)
    lib = os.path.join(out_dir, "libcachegen.so")
    stamp = os.path.join(out_dir, "libcachegen.stamp")
    dig = " ".join([_digest()] + list(defines))
    if not force and os.path.exists(lib) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == dig:
                return lib
    log = _compile(out_dir, lib, defines)
    with open(stamp, "w") as f:
        f.write(dig)
    if verbose:
        sys.stdout.write(log)
    return lib


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile libcachegen.so (if stale) and return its path."""
    return _build_into(OUT_DIR, (), force, verbose)


def build_test_variant(name: str, defines) -> str:
    """A library compiled with test-only macros (cachegen_kernels.cu names
    them: each forces a rarely taken path, an exact fallback or a bounded
    wait that runs out), in _build/<name>/. For the tests; the product
    library never sets them."""
    return _build_into(os.path.join(OUT_DIR, name), tuple(defines))


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True))
