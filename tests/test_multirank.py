"""The N > 1 host path of the benchmark on CPU: two gloo ranks, each with its own replica,
agree on the slowest rank's step time and report whole-job tokens/s (weak scaling); --gpus N
either starts N ranks under torchrun or refuses a mismatched WORLD_SIZE."""
import os
import socket

import pytest


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms_local = [1.5, 2.25][rank]
    ms, value = bench.aggregate_over_ranks(ms_local, 256)
    # each rank's replica: the same workload and its own byte count; the line's fields
    import synth
    wl = synth.tiny()
    algo = bench.algorithmic(wl, num_sms=152)
    head = bench.headline_fields(ms_local, wl.T)
    out.put((rank, ms, value, head, algo["base_gemm"]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted((q.get(timeout=10) for _ in range(2)), key=lambda r: r[0])
    for rank, ms, value, head, base_bytes in res:
        assert ms == 2.25
        assert value == pytest.approx(2 * 256 / 2.25e-3)
        assert head["n_gpus"] == 2 and head["ms_per_step"] == 2.25 and head["parallelism"] == "replicas x2"
        assert head["value"] == pytest.approx(2 * 16 / 2.25e-3)
    assert res[0][4] == res[1][4]                          # identical replicas


def test_gpus_flag_starts_torchrun_without_a_world(monkeypatch):
    import bench
    calls = []
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench.subprocess, "call", lambda cmd: calls.append(cmd) or 0)
    assert bench.main(["--gpus", "2", "--steps", "3"]) == 0
    cmd = calls[0]
    assert cmd[1:4] == ["-m", "torch.distributed.run", "--nnodes=1"] and "--nproc-per-node=2" in cmd
    assert "127.0.0.1" in cmd and cmd[-4:] == ["--gpus", "2", "--steps", "3"]


def test_gpus_flag_refuses_a_mismatched_world(monkeypatch):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "1")
    with pytest.raises(SystemExit, match="WORLD_SIZE=1"):
        bench.main(["--gpus", "4"])


def test_reference_arm_on_a_non_zero_rank_does_nothing(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")

    class A:
        workload, steps, warmup, layers = "tiny", 1, 3, 32
    assert bench.run_reference(A()) == 0
    assert capsys.readouterr().out == ""
