"""The multi-GPU path of the decode step is replicas only (a step exchanges
nothing between GPUs): bench.py under torchrun runs one replica per rank,
takes the slowest rank's time and reports the whole job's throughput.  Those
host steps run here as two gloo ranks on the CPU, and the reference arm's
ranks other than 0 do no work."""
import json
import multiprocessing as mp
import os
import socket
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _replica(rank, world, port, local_ms, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        r, w, _ = bench.dist_env()
        slowest = bench.max_over_ranks(local_ms[rank], w)
        q.put((r, w, slowest, bench.job_rate(4 * 100, w, slowest)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_report_the_slowest_rank_and_the_whole_job():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    local_ms = [3.0, 5.5]
    procs = [ctx.Process(target=_replica, args=(r, 2, port, local_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1] and all(g[1] == 2 for g in got)
    assert all(g[2] == 5.5 for g in got)  # every rank agrees on the slowest replica
    # 2 replicas x 400 units in 5.5 ms
    assert all(abs(g[3] - 2 * 400 / 5.5e-3) < 1e-6 for g in got)


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(7.25, 1) == 7.25
    assert bench.job_rate(10, 1, 2.0) == 5000.0


def test_reference_arm_ranks_other_than_zero_do_nothing(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    args = type("A", (), {"workload": "tiny", "steps": 1, "warmup": 1})()
    assert bench.run_reference(args) is None
    assert capsys.readouterr().out == ""


def test_reference_arm_line(monkeypatch, capsys):
    """Rank 0 of the reference arm prints one JSON line in the contract's form
    (the oracle on the host cores, tiny workload)."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    args = type("A", (), {"workload": "tiny", "steps": 2, "warmup": 1})()
    bench.run_reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 1 and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
