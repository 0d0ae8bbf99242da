"""The multi-GPU host logic of bench.py on CPU ranks (gloo, world size 2): every rank runs its
own sequences (replicas, no collective on the data path) and the timing is the maximum over
ranks."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    w, r, _ = bench.dist_env()
    bench.barrier(w)
    t = bench.max_over_ranks(10.0 + 5.0 * rank, w)
    q.put((r, w, t, bench.sequence_of_rank(r)))
    dist.destroy_process_group()


def test_two_cpu_ranks_take_the_max_time_and_distinct_sequences():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    assert [o[0] for o in out] == [0, 1]
    assert all(o[1] == 2 for o in out)
    assert all(o[2] == 15.0 for o in out)
    assert len({o[3] for o in out}) == 2


def test_reference_arm_other_ranks_do_nothing(monkeypatch, capsys):
    import bench
    from weight_mlp_layers_swiglu_b300.inputs import WORKLOADS

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")

    class A:
        steps, warmup, gpus = 3, 3, 2

    assert bench.run_reference(A, WORKLOADS["tiny_fp32"]) == 0
    assert capsys.readouterr().out == ""


def test_reference_arm_line_on_rank0(monkeypatch, capsys):
    import json

    import bench
    from weight_mlp_layers_swiglu_b300.inputs import WORKLOADS

    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")

    class A:
        steps, warmup, gpus = 3, 3, 1

    assert bench.run_reference(A, WORKLOADS["tiny_fp32"]) == 0
    line = json.loads(capsys.readouterr().out.strip())
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
