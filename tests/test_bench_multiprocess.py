"""Host-side multi-rank logic of bench.py on CPU: two gloo ranks (the N > 1
launch runs one replica per GPU; here the replicas are CPU processes)."""

import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # each rank's timed region; the job's time is the slowest rank's
        t = bench.max_over_ranks(10.0 * (rank + 1), world, torch.device("cpu"))
        q.put((rank, t, bench.dist_env()))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_rank_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert [g[1] for g in got] == [20.0, 20.0]
    assert [g[2] for g in got] == [(0, 2, 0), (1, 2, 1)]


def test_reference_arm_prints_nothing_on_nonzero_ranks(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup = 1, 0
    bench.run_reference(A())
    assert capsys.readouterr().out == ""


def test_single_process_defaults():
    import bench
    for k in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        os.environ.pop(k, None)
    assert bench.dist_env() == (0, 1, 0)
    assert bench.max_over_ranks(3.5, 1, torch.device("cpu")) == 3.5


def test_kernel_source_hash_ignores_comments_but_not_code(monkeypatch, tmp_path):
    """The committed DRAM traffic is keyed by this hash: editing a comment
    must keep it, editing code must change it."""
    import bench
    csrc = tmp_path / "tensor_transformer_mlp_columnparallel_gb300" / "csrc"
    csrc.mkdir(parents=True)
    f = csrc / "k.cu"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "KERNEL_FAMILIES", {"gemm": ("k.cu",)})
    f.write_text("// kernel\nint x = 1;  // one\n\n")
    h0 = bench.kernel_source_hash("gemm")
    f.write_text("// the kernel, reworded\n\nint x = 1;    // still one\n")
    assert bench.kernel_source_hash("gemm") == h0
    f.write_text("// kernel\nint x = 2;  // one\n")
    assert bench.kernel_source_hash("gemm") != h0


def test_reference_arm_line_on_rank_zero(monkeypatch, capsys):
    """Rank 0 times the float64 oracle on a small shape and prints one line
    with the contract's keys and the same `config` our arm prints."""
    import json
    import bench
    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    args = bench.parse(["--impl", "reference", "--steps", "2", "--warmup", "1",
                        "--shape", "96,256,512,4"])
    bench.run_reference(args)
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 1 and line["steps"] == 2
    assert line["config"] == bench.line_config(bench.workload_config(args), "splitk", 1)
    assert line["value"] > 0 and line["e2e"]["h2d_bytes_per_step"] == 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1
    assert "96 of 96 tokens" in cb["sample"]
