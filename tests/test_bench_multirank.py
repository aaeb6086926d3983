"""The bench's multi-rank path on CPU: two gloo ranks, max over ranks of the step times
and the whole-job value (every rank's bytes over the slowest rank's time); the launcher
that `bench.py --gpus N` uses when started without one (torch.distributed.run, N ranks),
with each rank's own batch (replica r of the workload) and the reductions across them."""
import json
import os
import socket
import subprocess

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        step_ms, attn_ms = bench.max_over_ranks([1.0 + rank, 5.0 - rank], dist, "cpu")
        q.put((rank, step_ms, attn_ms, bench.job_gbs(world, 1e9, step_ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, step_ms, attn_ms, gbs in got:
        assert step_ms == 2.0 and attn_ms == 5.0  # the slowest rank's numbers on every rank
        assert gbs == pytest.approx(2 * 1e9 / 2e-3 / 1e9)


def test_single_rank_passthrough():
    import bench

    assert bench.max_over_ranks([3, 4]) == [3.0, 4.0]
    assert bench.job_gbs(1, 2e9, 1.0) == pytest.approx(2000.0)


def test_launcher_runs_ranks_with_their_own_batches():
    import bench
    import workloads

    probe = os.path.join(os.path.dirname(os.path.abspath(__file__)), "multirank_probe.py")
    cmd = bench.launch_command(2, [], script=probe)
    assert cmd[1:3] == ["-m", "torch.distributed.run"] and "--nproc-per-node=2" in cmd
    assert "--master-addr=127.0.0.1" in cmd
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=300, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    wls = [workloads.build(3, replica=i) for i in range(2)]
    assert line["world"] == 2
    assert line["seeds"] == [w.seed for w in wls] and wls[0].seed != wls[1].seed
    assert line["step_ms"] == 2.0  # the slower rank's
    assert line["job_bytes"] == sum(sum(w.meta["final_lens"]) * w.spec.kv_token_bytes for w in wls)


def test_bench_without_launcher_reexecs_itself(monkeypatch):
    import bench

    seen = []
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench.subprocess, "call", lambda cmd: seen.append(cmd) or 0)
    assert bench.main(["--gpus", "4", "--steps", "7", "--warmup", "3"]) == 0
    cmd = seen[0]
    assert "--nproc-per-node=4" in cmd and cmd[-6:] == ["--gpus", "4", "--steps", "7", "--warmup", "3"]
    assert os.path.basename(cmd[-7]) == "bench.py"
    with pytest.raises(SystemExit):
        bench.main(["--gpus", "2", "--workload", "mixed"])
