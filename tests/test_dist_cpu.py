"""Multi-process paths on CPU processes (gloo backend), no GPU involved: the
benchmark's replica path (the barrier, the max over ranks of the timed
interval, the whole-job throughput, the reference arm's one-rank rule) and
the column-shard candidate exchange and merge."""

import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.abspath(os.path.join(os.path.dirname(__file__), ".."))

CHILD = """
import json, sys
sys.path.insert(0, {root!r})
import bench
d = bench.Dist()
d.barrier()
mine = 1.0 + 2.0 * d.rank            # rank 0 timed 1 ms, rank 1 timed 3 ms
m = d.max(mine)
v = bench.whole_job_rows_per_s(d.world, 100, 8, m)
d.barrier()
print(json.dumps({{"rank": d.rank, "world": d.world, "max": m, "value": v}}))
d.close()
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank: int, world: int, port: int) -> dict:
    return dict(os.environ, RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world),
                MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), CUDA_VISIBLE_DEVICES="")


def test_two_replicas_share_the_slowest_time():
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", CHILD.format(root=ROOT)], env=_env(r, 2, port),
                              stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True)
             for r in range(2)]
    outs = [p.communicate(timeout=180) for p in procs]
    for p, (_, err) in zip(procs, outs):
        assert p.returncode == 0, err[-2000:]
    res = [json.loads(out.strip().splitlines()[-1]) for out, _ in outs]
    assert sorted(r["rank"] for r in res) == [0, 1]
    for r in res:
        assert r["world"] == 2 and r["max"] == 3.0
        # 2 replicas x 100 layers x 8 rows over the slowest replica's 3 ms
        assert abs(r["value"] - 2 * 100 * 8 / 3e-3) <= 1e-9 * r["value"]


def test_reference_arm_runs_on_rank_zero_only():
    env = _env(1, 2, _free_port())
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert p.returncode == 0, p.stderr[-2000:]
    assert p.stdout.strip() == ""


def test_recorded_traffic_only_for_the_profiled_sources(tmp_path, monkeypatch):
    """roofline.traffic comes from the committed ncu summary only while the
    kernel's sources hash to the value recorded with it; otherwise null."""
    sys.path.insert(0, ROOT)
    import bench
    sha = bench.kernel_source_sha("decode_stream_kernel")
    prof = tmp_path / "profiles"
    prof.mkdir()
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_sha", lambda k: sha)
    rec = {"decode_stream_kernel:decode_r8": {"dram_bytes_per_launch": 123, "source_sha": sha}}
    (prof / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("decode_stream_kernel", "decode_r8") == 123.0
    assert bench.recorded_traffic("decode_stream_kernel", "decode_r1") is None
    rec["decode_stream_kernel:decode_r8"]["source_sha"] = "0" * 16
    (prof / "traffic.json").write_text(json.dumps(rec))
    assert bench.recorded_traffic("decode_stream_kernel", "decode_r8") is None


SHARD_CHILD = """
import json, sys
sys.path.insert(0, {root!r})
import numpy as np, torch, torch.distributed as dist
import latent_projection_top_gb300 as route
import oracle
dist.init_process_group("gloo")
r, W = dist.get_rank(), dist.get_world_size()
rows, E = 48, route.N_EXPERTS
NE = E // W
rng = np.random.default_rng(2024)          # the same full logit rows on every rank
lg = rng.standard_normal((rows, E)).astype(np.float32)
for i in range(rows):
    if i % 3 == 0:                         # equal logits in every shard at the 16th place
        v = lg[i, np.argsort(-lg[i], kind="stable")[15]]
        lg[i, [s * NE + 5 for s in range(W)]] = v
    elif i % 3 == 1:                       # NaN, -0 and +0 across the shards
        lg[i, rng.choice(E, 40, replace=False)] = np.nan
        lg[i, [s * NE + 1 for s in range(W)]] = np.float32(-0.0)
        lg[i, [s * NE + 2 for s in range(W)]] = np.float32(0.0)
        lg[i, rng.choice(E, 850, replace=False)] = np.nan
# this rank's shard: its experts' logits and its local top-16 (global ids)
part = np.ascontiguousarray(lg[:, r * NE:(r + 1) * NE])
local, _ = oracle.topk(part)
cids = torch.from_numpy((local + r * NE).astype(np.int32))
clg = torch.from_numpy(np.take_along_axis(part, local, axis=1))
g_ids, g_lg = route.gather_candidates(cids, clg)   # the exchange: [W, rows, 16]
# the merge rule on the gathered candidates: rank order over the W x 16 of a
# row.  Laid out shard after shard and in rank order inside a shard, a
# candidate's position orders equal logits exactly as its id does, so the
# oracle's top-16 over positions is the merge.
flat_ids = g_ids.permute(1, 0, 2).reshape(rows, W * 16).numpy()
flat_lg = np.ascontiguousarray(g_lg.permute(1, 0, 2).reshape(rows, W * 16).numpy())
pos, w = oracle.topk(flat_lg)
ids = np.take_along_axis(flat_ids, pos, axis=1)
ids_o, w_o = oracle.topk(lg)
layout = all(bool((g_ids[s].numpy() // NE == s).all()) for s in range(W))
print(json.dumps({{"rank": r, "layout": layout, "ids": bool(np.array_equal(ids, ids_o)),
                  "weights": bool(np.array_equal(w.view(np.uint32), w_o.view(np.uint32)))}}))
dist.destroy_process_group()
"""


@pytest.mark.parametrize("world", [2, 4])
def test_candidate_exchange_and_merge_across_ranks(world):
    """Column shards on `world` gloo ranks: each rank's local top-16, the
    candidate all-gather of the package (gather_candidates) and the merge
    rule give exactly the top-16 and weights of the whole logit row."""
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", SHARD_CHILD.format(root=ROOT)],
                              env=_env(r, world, port), stdout=subprocess.PIPE,
                              stderr=subprocess.PIPE, text=True)
             for r in range(world)]
    outs = [p.communicate(timeout=300) for p in procs]
    for p, (_, err) in zip(procs, outs):
        assert p.returncode == 0, err[-2000:]
    res = [json.loads(out.strip().splitlines()[-1]) for out, _ in outs]
    assert sorted(r["rank"] for r in res) == list(range(world))
    for r in res:
        assert r["layout"] and r["ids"] and r["weights"], r


PAIRED_CHILD = """
import json, sys
sys.path.insert(0, {root!r})
import numpy as np, torch, torch.distributed as dist
import latent_projection_top_gb300 as route
dist.init_process_group("gloo")
r, W = dist.get_rank(), dist.get_world_size()
rows = 20
NL, NE = route.N_LATENT // W, route.N_EXPERTS // W
g = torch.Generator().manual_seed(7)                 # the same whole layer on every rank
lat = torch.randn(rows, route.N_LATENT, generator=g).to(torch.bfloat16)
lg = torch.randn(rows, route.N_EXPERTS, generator=g)
lg[0, 3] = float("nan"); lg[1, 5] = -0.0            # bits travel unchanged
mine_lat = lat[:, r * NL:(r + 1) * NL].clone()
mine_lg = lg[:, r * NE:(r + 1) * NE].clone()
got_lat, got_lg = route.gather_latent_logits(mine_lat, mine_lg)
ok_lat = bool(torch.equal(got_lat.view(torch.int16), lat.view(torch.int16)))
ok_lg = bool(torch.equal(got_lg.view(torch.int32), lg.view(torch.int32)))
shape = list(got_lat.shape) == [rows, route.N_LATENT] and list(got_lg.shape) == [rows, route.N_EXPERTS]
print(json.dumps({{"rank": r, "latent": ok_lat, "logits": ok_lg, "shape": shape}}))
dist.destroy_process_group()
"""


@pytest.mark.parametrize("world", [2, 4])
def test_paired_gather_of_latent_and_logit_columns(world):
    """The paired gather (gather_latent_logits): each rank's latent and logit
    columns in one all-gather, stitched back into the whole layer's tensors
    bit for bit (NaN and -0 included) on every rank."""
    port = _free_port()
    procs = [subprocess.Popen([sys.executable, "-c", PAIRED_CHILD.format(root=ROOT)],
                              env=_env(r, world, port), stdout=subprocess.PIPE,
                              stderr=subprocess.PIPE, text=True)
             for r in range(world)]
    outs = [p.communicate(timeout=300) for p in procs]
    for p, (_, err) in zip(procs, outs):
        assert p.returncode == 0, err[-2000:]
    res = [json.loads(out.strip().splitlines()[-1]) for out, _ in outs]
    assert sorted(r["rank"] for r in res) == list(range(world))
    for r in res:
        assert r["latent"] and r["logits"] and r["shape"], r
