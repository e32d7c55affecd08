"""The multi-rank bench harness on CPU: world_size-2 gloo ranks exercise
bench.py's rank handling (env parsing, barrier, max over ranks) without a
GPU.  Each rank quantizes its own batch in the real run (weak scaling, no
collective on the data path); only the timing aggregation is collective."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    r, w, lr = bench.dist_env()
    dist.init_process_group("gloo", rank=r, world_size=w)
    bench.barrier(w)
    mx = bench.max_over_ranks(1.5 + rank, w)     # rank 1 is the slow one
    bench.barrier(w)
    dist.destroy_process_group()
    q.put((r, w, lr, mx))


def test_two_rank_max_over_ranks_and_barrier():
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
    assert got == [(0, 2, 0, 2.5), (1, 2, 1, 2.5)]


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    bench.barrier(1)


def test_reference_arm_rank_gate(monkeypatch, capsys):
    """Under torchrun only rank 0 runs the reference arm; other ranks exit
    quietly without work."""
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"])
    assert capsys.readouterr().out == ""


def test_reference_arm_json_contract(monkeypatch, capsys):
    """Rank 0's reference arm (the oracle on host cores) prints one JSON line
    with the contract's keys: the arm's own e2e with no host-device bytes, a
    cpu_baseline describing the run, and the workload named in config."""
    import json
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "3"])
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["steps"] == 1 and d["warmup"] == 3 and d["n_gpus"] == 1
    assert d["value"] > 0 and d["higher_is_better"] is True and d["unit"] == "GB/s"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["value"] == d["value"]
    assert d["cpu_baseline"]["cores"] >= 1 and d["cpu_baseline"]["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert d["config"]["workload"]


def test_gpus_flag_starts_that_many_ranks():
    """`bench.py --gpus 2` outside torchrun relaunches itself as two ranks;
    both start (each announces itself on stderr) and rank 0 alone prints the
    JSON line, with n_gpus 2.  The reference arm needs no GPU."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK")}
    res = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
                          "--steps", "1", "--warmup", "3"], capture_output=True, text=True, env=env, timeout=600)
    assert res.returncode == 0, res.stderr[-2000:]
    assert "bench: rank 0 of 2" in res.stderr and "bench: rank 1 of 2" in res.stderr
    lines = [ln for ln in res.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1 and json.loads(lines[0])["n_gpus"] == 2


def test_gpus_flag_must_match_world_size(monkeypatch):
    """Under a launcher, --gpus must equal WORLD_SIZE: a mismatch is refused
    (exit status 2) instead of silently running another number of ranks."""
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit) as ei:
        bench.main(["--impl", "reference", "--gpus", "3", "--steps", "1", "--warmup", "3"])
    assert ei.value.code == 2
