"""The benchmark's replica path on two CPU processes (gloo backend): the
barrier, the max over ranks of the timed interval and the whole-job
throughput, and the reference arm's one-rank rule -- no GPU involved."""

import json
import os
import socket
import subprocess
import sys

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
