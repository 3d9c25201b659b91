"""The benchmark's N > 1 path on CPU, two gloo ranks (no GPU): each GPU runs an
independent replica, so the only cross-rank steps are the barrier around the
timed region, the max of the ranks' times, and rank 0 alone printing (and,
for the reference arm, alone doing the work)."""
import json
import os
import socket
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _env(rank, world, port):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world), RANK=str(rank),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)


def _replica_rank(rank, world, port, out_dir):
    _env(rank, world, port)
    import bench
    w, r, _ = bench.dist_init(world)
    assert (w, r) == (world, rank)
    bench.barrier(w)
    slowest = bench.max_over_ranks(w, 10.0 + rank)   # per-rank timed milliseconds
    tokens = w * 274 * 5 / (slowest / 1e3)            # whole-job tokens over the slowest rank's time
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"slowest": slowest, "tokens": tokens}, f)
    torch.distributed.destroy_process_group()


def test_two_replicas_take_the_slowest_rank(tmp_path):
    port = _free_port()
    mp.spawn(_replica_rank, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    res = [json.load(open(tmp_path / f"r{r}.json")) for r in range(2)]
    assert res[0] == res[1]
    assert res[0]["slowest"] == 11.0
    assert res[0]["tokens"] == pytest.approx(2 * 274 * 5 / 0.011)


def _reference_rank(rank, world, port, out_dir):
    _env(rank, world, port)
    import contextlib
    import io
    import types
    import bench
    from chunked_prefill_hybrid_gb300 import workloads
    workloads.llama13b_hybrid = lambda seed=2: workloads.tiny(seed)  # a small batch: the logic, not the size
    buf = io.StringIO()
    args = types.SimpleNamespace(gpus=world, steps=1, warmup=3, ref_seconds=0.05)
    with contextlib.redirect_stdout(buf):
        rc = bench.run_reference(args)
    with open(os.path.join(out_dir, f"ref{rank}.json"), "w") as f:
        json.dump({"rc": rc, "out": buf.getvalue()}, f)
    torch.distributed.destroy_process_group()


def test_reference_arm_runs_on_rank_zero_only(tmp_path):
    port = _free_port()
    mp.spawn(_reference_rank, args=(2, port, str(tmp_path)), nprocs=2, join=True)
    r0 = json.load(open(tmp_path / "ref0.json"))
    r1 = json.load(open(tmp_path / "ref1.json"))
    assert r0["rc"] == 0 and r1["rc"] == 0
    assert r1["out"] == ""
    lines = [l for l in r0["out"].splitlines() if l.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
