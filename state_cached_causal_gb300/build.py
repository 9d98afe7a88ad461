"""Build libcconv.so (sm_103a) in-tree with nvcc.

Each ``csrc/*.cu`` translation unit compiles in parallel to an object under
``_build/``; the objects link into ``state_cached_causal_gb300/libcconv.so``.
An object is rebuilt when its source, a header it may include, or the flags
change.
"""
from __future__ import annotations

import concurrent.futures as cf
import hashlib
import os
import shutil
import subprocess

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libcconv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                 "-Xcompiler", "-fvisibility=hidden",
                 "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc():
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _headers():
    hs = [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cuh", ".h"))]
    hs += [os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")]
    return sorted(hs)


def _digest(src, extra_flags):
    h = hashlib.sha256()
    for p in [src] + _headers():
        with open(p, "rb") as f:
            h.update(f.read())
    h.update(" ".join(CFLAGS + extra_flags).encode())
    return h.hexdigest()[:16]


def _compile(nvcc, src, extra_flags, verbose):
    name = os.path.splitext(os.path.basename(src))[0]
    obj = os.path.join(BUILD, f"{name}.{_digest(src, extra_flags)}.o")
    if os.path.exists(obj):
        return obj
    for f in os.listdir(BUILD):   # objects of older versions of this source
        if f.startswith(name + ".") and f.endswith(".o"):
            try:
                os.remove(os.path.join(BUILD, f))
            except OSError:
                pass
    tmp = obj + f".{os.getpid()}.tmp"
    cmd = [nvcc] + CFLAGS + extra_flags + ["-c", src, "-o", tmp]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr)
    os.replace(tmp, obj)
    return obj


def build(verbose: bool = False, extra_flags=None, jobs: int | None = None) -> str:
    """Compile every CUDA source and link libcconv.so; return its path."""
    extra_flags = list(extra_flags or [])
    os.makedirs(BUILD, exist_ok=True)
    nvcc = _nvcc()
    srcs = _sources()
    jobs = jobs or min(len(srcs), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, extra_flags, verbose), srcs))
    stamp = os.path.join(BUILD, "link." + hashlib.sha256(
        "".join(objs).encode()).hexdigest()[:16])
    if os.path.exists(LIB) and os.path.exists(stamp):
        return LIB
    tmp = LIB + f".{os.getpid()}.tmp"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    for f in os.listdir(BUILD):
        if f.startswith("link."):
            os.remove(os.path.join(BUILD, f))
    open(stamp, "w").close()
    return LIB


def build_cca_variant(out_dir: str, extra_flags) -> str:
    """The CCA entry points alone (``cca_qk_conv.cu`` and the status strings),
    compiled with extra nvcc flags into ``out_dir/libcconv_cca.so``: the tests
    build one with a short pipeline-wait limit (``-DCCA_WAIT_CYCLES=...``) to
    run the kernel's timeout path."""
    os.makedirs(out_dir, exist_ok=True)
    nvcc = _nvcc()
    objs = []
    for name in ("cca_qk_conv.cu", "abi.cu"):
        obj = os.path.join(out_dir, name + ".o")
        cmd = [nvcc] + CFLAGS + list(extra_flags) + ["-c", os.path.join(CSRC, name), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {name}:\n{r.stdout}\n{r.stderr}")
        objs.append(obj)
    lib = os.path.join(out_dir, "libcconv_cca.so")
    r = subprocess.run([nvcc] + ARCH + ["-shared", "-o", lib] + objs, capture_output=True,
                       text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return lib


if __name__ == "__main__":
    print(build(verbose=True))
