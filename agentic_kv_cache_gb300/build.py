"""Build libakv.so in-tree for sm_103a (GB300) with nvcc.

Each translation unit is compiled in parallel, then linked into
``agentic_kv_cache_gb300/libakv.so`` (CUDA runtime linked statically, so the
library only needs the driver at run time).  Rebuilds only when a source or
header is newer than the library.

The checked variant ``libakv_checked.so`` is the same sources compiled with
-DAKV_CHECKED: every kernel checks the descriptors it reads (pages inside the
pool, row ranges inside a page, segments and runs inside their tables, query
rows inside Q) and records AKV_ERR_DEVICE instead of touching memory they do
not name.  It is built with ``checked=True`` or when the environment sets
AKV_CHECKED=1, which also makes the binding load it.

    python -m agentic_kv_cache_gb300.build [--force] [--verbose] [--checked]
"""
import concurrent.futures
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libakv.so")
BUILD_CHECKED = os.path.join(HERE, "_build_checked")
LIB_CHECKED = os.path.join(HERE, "libakv_checked.so")


def checked_from_env():
    return os.environ.get("AKV_CHECKED", "") == "1"

SOURCES = ["engine.cpp", "kv_write.cu", "repos_rotate.cu", "segment_attn.cu", "segment_attn_mla.cu", "repos_noalloc.cu", "compact_copy.cu", "attn_mass.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def nvcc():
    path = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(path):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libakv.so")
    return path


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES]
    files += [os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".h", ".cuh"))]
    files.append(os.path.join(INCLUDE, "akv.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date(lib=LIB):
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def _compile(src, verbose, extra, build_dir=BUILD):
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    lang = ["-x", "cu"] if src.endswith(".cu") else ["-x", "c++"]
    cmd = [nvcc()] + ARCH + FLAGS + extra + lang + ["-c", src, "-o", obj]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed on {os.path.basename(src)}:\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)
    return obj


def build(force=False, verbose=False, extra_flags=(), checked=None):
    """Compile and link libakv.so (checked: libakv_checked.so, -DAKV_CHECKED; None: from the
    AKV_CHECKED environment variable); returns its path."""
    if checked is None:
        checked = checked_from_env()
    lib, build_dir = (LIB_CHECKED, BUILD_CHECKED) if checked else (LIB, BUILD)
    extra = list(extra_flags) + (["-DAKV_CHECKED"] if checked else [])
    if not force and up_to_date(lib):
        return lib
    os.makedirs(build_dir, exist_ok=True)
    srcs = [os.path.join(CSRC, s) for s in SOURCES]
    with concurrent.futures.ThreadPoolExecutor(max_workers=len(srcs)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose, extra, build_dir), srcs))
    tmp = lib + ".tmp"
    cmd = [nvcc()] + ARCH + ["-shared", "-o", tmp] + objs + ["-lrt", "-ldl", "-lpthread"]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv,
                checked=True if "--checked" in sys.argv else None))
