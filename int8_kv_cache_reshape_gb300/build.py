"""Build ``libkvq.so`` (the C-ABI library) in-tree with nvcc for sm_103a.

Each translation unit under ``csrc/`` compiles in parallel to an object in
``_build/``; the objects link into ``libkvq.so`` next to this file, with the
CUDA runtime linked statically.  Rebuilds only what changed.
"""
from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import platform
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build", platform.machine())
LIB = os.path.join(HERE, "libkvq.so")
# The bounds-checked build (-DKVQ_CHECKED=1): same sources, its own objects.
BUILD_CHECKED = os.path.join(HERE, "_build", platform.machine() + "-checked")
LIB_CHECKED = os.path.join(HERE, "libkvq_checked.so")
# The prefill on CTA pairs (-DKVQ_PREFILL_PAIR=1), a build option.
BUILD_PAIR = os.path.join(HERE, "_build", platform.machine() + "-pair")
LIB_PAIR = os.path.join(HERE, "libkvq_pair.so")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libkvq.so")


def _headers_mtime() -> float:
    hs = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh"))
    hs += glob.glob(os.path.join(INCLUDE, "*.h"))
    return max(os.path.getmtime(h) for h in hs)


def _compile(src: str, force: bool, extra, build_dir: str = BUILD) -> str:
    obj = os.path.join(build_dir, os.path.basename(src) + ".o")
    if (not force and os.path.exists(obj)
            and os.path.getmtime(obj) >= max(os.path.getmtime(src), _headers_mtime())):
        return obj
    tmp = obj + f".tmp{os.getpid()}"
    cmd = [_nvcc()] + NVCC_FLAGS + list(extra) + ["-c", src, "-o", tmp]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {os.path.basename(src)}:\n{res.stdout}{res.stderr}")
    os.replace(tmp, obj)
    if os.environ.get("KVQ_BUILD_VERBOSE"):
        print(res.stdout + res.stderr)
    return obj


def build(force: bool = False, extra_flags=(), jobs: int = 0, checked: bool = False,
          pair: bool = False) -> str:
    """Compile and link libkvq.so (checked: libkvq_checked.so, the
    bounds-checked build; pair: libkvq_pair.so, the prefill on CTA pairs);
    returns its path."""
    assert not (checked and pair)
    build_dir, lib = ((BUILD_CHECKED, LIB_CHECKED) if checked else (BUILD_PAIR, LIB_PAIR) if pair
                      else (BUILD, LIB))
    extra = (list(extra_flags) + (["-DKVQ_CHECKED=1"] if checked else [])
             + (["-DKVQ_PREFILL_PAIR=1"] if pair else []))
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    jobs = jobs or min(len(srcs), os.cpu_count() or 4)
    with cf.ThreadPoolExecutor(jobs) as ex:
        objs = list(ex.map(lambda s: _compile(s, force, extra, build_dir), srcs))
    stamp = os.path.join(build_dir, "libkvq.stamp")
    if (force or not os.path.exists(lib) or not os.path.exists(stamp)
            or os.path.getmtime(lib) < max(os.path.getmtime(o) for o in objs)):
        tmp = lib + f".tmp{os.getpid()}"
        cmd = [_nvcc()] + ARCH + ["-shared", "-cudart", "static", "-o", tmp] + objs
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"link failed:\n{res.stdout}{res.stderr}")
        os.replace(tmp, lib)
        with open(stamp, "w") as f:     # marks the library as built on this machine
            f.write(platform.machine() + "\n")
    return lib


if __name__ == "__main__":
    print(build())
