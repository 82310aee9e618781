"""The C ABI from a plain C program (tests/c/route_abi_check.c): no Python
binding and no PyTorch on the path, device memory from the CUDA runtime; one
decode and one prefill step checked against the oracle, which the program
links (test code only), and two host steps in flight together checked
against route_step."""

import os
import subprocess

import pytest

import latent_projection_top_gb300 as route
import oracle
from latent_projection_top_gb300 import builder

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_plain_c_program_on_the_abi(tmp_path):
    lib = route.build()
    ora = oracle.build()
    cuda = os.path.dirname(os.path.dirname(builder.NVCC))
    exe = str(tmp_path / "route_abi_check")
    # the library the binding loads (the checked one under ROUTE_DEBUG_LIB=1),
    # linked by its path
    lib_dirs = [os.path.dirname(lib), os.path.dirname(ora), os.path.join(cuda, "lib64")]
    cmd = ["gcc", "-std=c11", "-O2", "-Wall", "-o", exe, os.path.join(HERE, "c", "route_abi_check.c"),
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(cuda, "include"), lib, ora]
    for d in lib_dirs:
        cmd += ["-L", d, f"-Wl,-rpath,{d}"]
    cmd += ["-lcudart", "-lm"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr[-3000:]
    run = subprocess.run([exe], capture_output=True, text=True, timeout=600)
    assert run.returncode == 0, run.stdout[-2000:] + run.stderr[-2000:]
    for line in ("decode 8 rows: ok", "prefill 264 rows: ok", "host steps, two in flight: ok"):
        assert line in run.stdout, run.stdout
