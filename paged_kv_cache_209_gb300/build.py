"""Build libpkv.so in-tree: every .cu (and host-only .cpp) under csrc/,
compiled for sm_103a.

Usage: ``python -m paged_kv_cache_209_gb300.build`` (or call ``build()``).
Objects go to ``_build/`` beside this file; the shared library lands next to
this file as ``libpkv.so``. Translation units compile in parallel; a unit is
rebuilt only when it or a header is newer than its object.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libpkv.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
         "--expt-relaxed-constexpr"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _newest_header() -> float:
    hdrs = glob.glob(os.path.join(CSRC, "*.h")) + glob.glob(os.path.join(CSRC, "*.cuh")) + \
        glob.glob(os.path.join(INCLUDE, "*.h"))
    return max((os.path.getmtime(h) for h in hdrs), default=0.0)


def _compile(src: str, obj: str, extra: list[str]) -> tuple[str, int, str]:
    cmd = [_nvcc(), *ARCH, *FLAGS, "-I", INCLUDE, "-I", CSRC, *extra, "-c", src, "-o", obj]
    p = subprocess.run(cmd, capture_output=True, text=True)
    return src, p.returncode, (p.stdout + p.stderr)


def build(verbose: bool = False, ptxas_info: bool = False, force: bool = False,
          defines: dict | None = None, out_dir: str | None = None) -> str:
    """Compile and link ``libpkv.so``; returns its path. Raises on failure.

    ``defines`` adds ``-D`` build-time knobs (e.g. ``{"PKV_TC_STAGES": 12}``);
    with ``out_dir`` the objects and the library go there instead of in-tree.
    """
    build_dir = BUILD if out_dir is None else os.path.join(out_dir, "_build")
    lib_path = LIB if out_dir is None else os.path.join(out_dir, "libpkv.so")
    os.makedirs(build_dir, exist_ok=True)
    sources = sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cpp")))
    hdr_time = _newest_header()
    extra = ["-Xptxas", "-v"] if ptxas_info else []
    extra += [f"-D{k}={v}" for k, v in (defines or {}).items()]
    jobs = []
    objs = []
    for src in sources:
        obj = os.path.join(build_dir, os.path.splitext(os.path.basename(src))[0] + ".o")
        objs.append(obj)
        stale = force or ptxas_info or not os.path.exists(obj) or \
            os.path.getmtime(obj) < max(os.path.getmtime(src), hdr_time)
        if stale:
            jobs.append((src, obj))
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
            for src, rc, log in ex.map(lambda j: _compile(j[0], j[1], extra), jobs):
                if verbose or ptxas_info or rc:
                    sys.stderr.write(f"== {os.path.basename(src)} (rc={rc})\n{log}")
                if rc:
                    raise RuntimeError(f"nvcc failed on {src}")
    if jobs or force or not os.path.exists(lib_path) or \
            os.path.getmtime(lib_path) < max(os.path.getmtime(o) for o in objs):
        cmd = [_nvcc(), *ARCH, "-shared", "-o", lib_path, *objs]
        p = subprocess.run(cmd, capture_output=True, text=True)
        if p.returncode:
            raise RuntimeError("link failed:\n" + p.stdout + p.stderr)
    return lib_path


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv, force="-f" in sys.argv))
