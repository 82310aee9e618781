"""Build the route library (``_build/libroute.so``) for sm_103a with nvcc.

The translation units compile in parallel; ptxas resource usage (registers,
spills, shared memory) is written to ``_build/ptxas.log``.

``build(debug=True)`` builds the same sources with ``-DROUTE_DEBUG`` into
``_build/debug/libroute_debug.so``: every computed global index is checked
in the kernels, and a failed check is reported through the device status
word (``route_device_status`` returns ROUTE_ERR_DEVICE_BOUNDS) instead of
faulting.  The binding loads it when the environment sets ROUTE_DEBUG_LIB=1.
"""

from __future__ import annotations

import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libroute.so")
DEBUG_BUILD = os.path.join(BUILD, "debug")
DEBUG_LIB = os.path.join(DEBUG_BUILD, "libroute_debug.so")
INCLUDE = os.path.join(ROOT, "include")

SOURCES = ["decode_kernel.cu", "prefill_kernel.cu", "topk_kernel.cu", "stage_kernel.cu",
           "route_api.cu"]
HEADERS = ["common.cuh", "sm103_ptx.cuh", "topk16.cuh", "twofloat.cuh"]

NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                "-Xptxas", "-v", "-I", INCLUDE, "-I", CSRC]


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(INCLUDE, "route.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    return any(os.path.getmtime(f) > t for f in _inputs())


def _compile(src: str, build_dir: str, extra: list) -> tuple[str, str]:
    obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
    cmd = [NVCC] + FLAGS + extra + ["-c", os.path.join(CSRC, src), "-o", obj]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{res.stdout}\n{res.stderr}")
    return obj, res.stderr


def _link(objs: list, lib: str) -> None:
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [NVCC] + ARCH + ["-shared", "-o", tmp] + objs + ["-cudart", "static"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, lib)


def build(force: bool = False, verbose: bool = False, debug: bool = False,
          both: bool = False) -> str:
    """Build the release library (or, with debug=True, the checked one; with
    both=True, both at once, their translation units in parallel).  Returns
    the path of the release library (of the debug one with debug=True)."""
    targets = [(LIB, BUILD, [])] if not debug or both else []
    if debug or both:
        targets.append((DEBUG_LIB, DEBUG_BUILD, ["-DROUTE_DEBUG"]))
    todo = [(lib, d, x) for lib, d, x in targets if force or _stale(lib)]
    if todo:
        for _, d, _ in todo:
            os.makedirs(d, exist_ok=True)
        jobs = [(src, d, x) for _, d, x in todo for src in SOURCES]
        with ThreadPoolExecutor(max_workers=len(jobs)) as pool:
            results = list(pool.map(lambda j: _compile(*j), jobs))
        for k, (lib, d, _) in enumerate(todo):
            part = results[k * len(SOURCES):(k + 1) * len(SOURCES)]
            with open(os.path.join(d, "ptxas.log"), "w") as f:
                for (o, log), src in zip(part, SOURCES):
                    f.write(f"==== {src}\n{log}\n")
            _link([o for o, _ in part], lib)
        if verbose:
            print(open(os.path.join(todo[0][1], "ptxas.log")).read())
    return DEBUG_LIB if debug and not both else LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv, debug="--debug" in sys.argv,
                both="--both" in sys.argv))
