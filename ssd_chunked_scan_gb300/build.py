"""Build libssd.so (the CUDA library behind include/ssd.h) in-tree.

Each translation unit under csrc/ is compiled for sm_103a only, in parallel,
then linked into ``ssd_chunked_scan_gb300/_lib/libssd.so``.  Objects go to
``ssd_chunked_scan_gb300/_build/``.  A unit is rebuilt when it or any header
is newer than its object.

``build_lib(check=True)`` builds the debug variant instead: the same sources
with ``-DSSD_CHECK`` (every global index tested against its buffer's size; a
failure sets the device check word, reported by ssd_last_device_error as
SSD_ERR_CHECK), objects in ``_build/check/``, library ``_lib/libssd_check.so``.
The binding loads it when the environment variable SSD_LIB_VARIANT is "check".
"""
import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIBDIR = os.path.join(HERE, "_lib")
LIB = os.path.join(LIBDIR, "libssd.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc():
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def _newest_header():
    hdrs = glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(ROOT, "include", "*.h"))
    return max((os.path.getmtime(h) for h in hdrs), default=0.0)


def _compile(src, force, extra, bdir):
    obj = os.path.join(bdir, os.path.basename(src).replace(".cu", ".o"))
    if (not force and os.path.exists(obj)
            and os.path.getmtime(obj) >= max(os.path.getmtime(src), _newest_header())):
        return obj, False
    cmd = [_nvcc()] + ARCH + FLAGS + extra + ["-c", src, "-o", obj]
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}")
    return obj, True


def lib_path(check: bool = False) -> str:
    return os.path.join(LIBDIR, "libssd_check.so" if check else "libssd.so")


def build_lib(force: bool = False, verbose: bool = False, extra=(), check: bool = False) -> str:
    bdir = os.path.join(BUILD, "check") if check else BUILD
    lib = lib_path(check)
    extra = list(extra) + (["-DSSD_CHECK"] if check else [])
    os.makedirs(bdir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    with ThreadPoolExecutor(max_workers=max(1, min(len(srcs), os.cpu_count() or 1))) as ex:
        res = list(ex.map(lambda s: _compile(s, force, extra, bdir), srcs))
    objs = [o for o, _ in res]
    rebuilt = any(r for _, r in res)
    if rebuilt or not os.path.exists(lib):
        cmd = [_nvcc()] + ARCH + ["-shared", "-o", lib] + objs
        r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}")
    if verbose:
        print(lib)
    return lib


if __name__ == "__main__":
    build_lib(force="--force" in sys.argv, verbose=True, check="--check" in sys.argv)
