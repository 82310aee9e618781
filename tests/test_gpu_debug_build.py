"""The bounds-checked library (built with -DROUTE_DEBUG; see builder.py):
every computed global index in the kernels is checked before its access, and
a failed check sets a status bit that route_device_status reports as
ROUTE_ERR_DEVICE_BOUNDS, instead of faulting.  It stands in for a memory
checker (the pages' stress runs rely on poisoned memory for the same
purpose).  A child process loads it (ROUTE_DEBUG_LIB=1) and runs decode and
prefill steps at small shapes, ragged ones included; every check must pass
and every output must equal the release library's bits."""

import os
import subprocess
import sys
import tempfile

import numpy as np
import pytest
import torch

import latent_projection_top_gb300 as route
from gpu_util import DEV, bank, require_gpu, to_dev_bf16

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CASES = [("decode", "decode_r8", 8), ("decode", "decode_sweep", 20), ("decode", "decode_r1", 1),
         ("prefill", "prefill_r1024", 40), ("prefill", "prefill_r1024", 300)]

CHILD = r"""
import os, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, os.path.join({root!r}, "tests"))
import numpy as np, torch
import latent_projection_top_gb300 as route
from gpu_util import DEV, bank, to_dev_bf16
assert route.LIB_PATH.endswith("libroute_debug.so")
out = {{}}
for mode, wk, rows in {cases!r}:
    h, wl, wr = bank(wk, 0)
    m = route.DECODE if mode == "decode" else route.PREFILL
    with route.Plan(m, rows) as plan:
        o = [torch.empty((rows, route.N_LATENT), dtype=torch.bfloat16, device=DEV),
             torch.empty((rows, route.N_EXPERTS), dtype=torch.float32, device=DEV),
             torch.empty((rows, route.TOPK), dtype=torch.int32, device=DEV),
             torch.empty((rows, route.TOPK), dtype=torch.float32, device=DEV),
             torch.empty((rows,), dtype=torch.float32, device=DEV)]
        for _ in range(2):
            route.route_step_sumsq(plan, to_dev_bf16(np.ascontiguousarray(h[:rows])),
                                   to_dev_bf16(wl), to_dev_bf16(wr), *o)
        route.route_device_status(plan)  # raises on any failed bounds check
    for i, t in enumerate(o):
        out[f"{{wk}}_{{rows}}_{{i}}"] = t.view(torch.uint8).cpu().numpy()
np.savez({path!r}, **out)
print("debug library ok", len(out))
"""


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def test_debug_library_runs_clean_and_matches_release():
    route.build(debug=True)
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "debug_out.npz")
        env = dict(os.environ, ROUTE_DEBUG_LIB="1")
        res = subprocess.run([sys.executable, "-c", CHILD.format(root=ROOT, cases=CASES, path=path)],
                             env=env, capture_output=True, text=True, timeout=600)
        assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
        got = dict(np.load(path))
    for mode, wk, rows in CASES:
        h, wl, wr = bank(wk, 0)
        m = route.DECODE if mode == "decode" else route.PREFILL
        with route.Plan(m, rows) as plan:
            o = [torch.empty((rows, route.N_LATENT), dtype=torch.bfloat16, device=DEV),
                 torch.empty((rows, route.N_EXPERTS), dtype=torch.float32, device=DEV),
                 torch.empty((rows, route.TOPK), dtype=torch.int32, device=DEV),
                 torch.empty((rows, route.TOPK), dtype=torch.float32, device=DEV),
                 torch.empty((rows,), dtype=torch.float32, device=DEV)]
            route.route_step_sumsq(plan, to_dev_bf16(np.ascontiguousarray(h[:rows])), to_dev_bf16(wl),
                                   to_dev_bf16(wr), *o)
            route.route_device_status(plan)
        for i, t in enumerate(o):
            assert np.array_equal(t.view(torch.uint8).cpu().numpy(), got[f"{wk}_{rows}_{i}"]), \
                f"{wk} {rows} rows: output {i} differs between the debug and release libraries"


SHARD_CASES = [(8, 40), (16, 8), (8, 20), (2, 1), (7, 300)]

SHARD_RUN = r"""
def shard_outputs(W, rows):
    import numpy as np, torch
    import latent_projection_top_gb300 as route
    from gpu_util import DEV, bank, to_dev_bf16
    h, wl, wr = bank("prefill_r3072", 0)
    NL, NE = route.shard_columns(W)
    hd = to_dev_bf16(np.ascontiguousarray(h[:rows]))
    cid = torch.empty((W, rows, route.TOPK), dtype=torch.int32, device=DEV)
    clg = torch.empty((W, rows, route.TOPK), dtype=torch.float32, device=DEV)
    out = []
    for s in range(W):
        lat = torch.empty((rows, NL), dtype=torch.bfloat16, device=DEV)
        lg = torch.empty((rows, NE), dtype=torch.float32, device=DEV)
        with route.ShardPlan(rows, s, W) as plan:
            route.route_shard_step(plan, hd, to_dev_bf16(np.ascontiguousarray(wl[:, s * NL:(s + 1) * NL])),
                                   to_dev_bf16(np.ascontiguousarray(wr[:, s * NE:(s + 1) * NE])),
                                   lat, lg, cid[s], clg[s])
            route.route_device_status(plan)  # raises on any failed bounds check
        out += [lat, lg]
    ids = torch.empty((rows, route.TOPK), dtype=torch.int32, device=DEV)
    w = torch.empty((rows, route.TOPK), dtype=torch.float32, device=DEV)
    route.route_merge_candidates(cid, clg, ids, w)
    torch.cuda.synchronize()
    return [t.view(torch.uint8).cpu().numpy() for t in out + [cid, clg, ids, w]]
"""

SHARD_CHILD = r"""
import os, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, os.path.join({root!r}, "tests"))
import numpy as np
import latent_projection_top_gb300 as route
assert route.LIB_PATH.endswith("libroute_debug.so")
{run}
out = {{}}
for W, rows in {cases!r}:
    for i, a in enumerate(shard_outputs(W, rows)):
        out[f"W{{W}}_{{rows}}_{{i}}"] = a
np.savez({path!r}, **out)
print("debug library ok", len(out))
"""


def test_debug_library_runs_column_shards_clean():
    """Shard plans store only their own columns (the store maps and the
    validity of a column are sized to the shard): every index of the shard
    kernels and the merge is checked, outputs equal the release library's."""
    route.build(debug=True)
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "debug_shards.npz")
        env = dict(os.environ, ROUTE_DEBUG_LIB="1")
        code = SHARD_CHILD.format(root=ROOT, run=SHARD_RUN, cases=SHARD_CASES, path=path)
        res = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True,
                             timeout=600)
        assert res.returncode == 0, res.stdout[-2000:] + res.stderr[-4000:]
        got = dict(np.load(path))
    ns = {}
    exec(SHARD_RUN, ns)
    for W, rows in SHARD_CASES:
        for i, a in enumerate(ns["shard_outputs"](W, rows)):
            assert np.array_equal(a, got[f"W{W}_{rows}_{i}"]), \
                f"W = {W}, {rows} rows: output {i} differs between the debug and release libraries"
