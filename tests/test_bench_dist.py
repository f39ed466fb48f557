"""bench.py's multi-process bookkeeping on CPU: two gloo ranks, as torchrun
would launch them, agree on the maximum time over ranks and on the whole-job
value; the reference arm runs on rank 0 alone."""

import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench

    d = bench.Dist(backend="gloo")
    assert (d.rank, d.world) == (rank, world)
    d.barrier()
    elapsed_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    m = d.max(elapsed_ms)
    out[rank] = (m, bench.aggregate_value(m, 100, d.world))
    d.barrier()
    d.close()


def test_two_gloo_ranks_take_the_max_and_the_whole_job_value():
    world, port = 2, _free_port()
    with mp.Manager() as mgr:
        out = mgr.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0] == res[1]
    m, value = res[0]
    assert m == 15.0
    # 2 replicas x 100 layer-steps in 15 ms: 75 us per layer-step for the job
    assert value == pytest.approx(75.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench

    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "0"]) == 0
    assert capsys.readouterr().out == ""


def test_profile_summaries_are_readable_by_the_bench():
    """Every kernel summary under profiles/ gives the command that made it, the
    digest of the kernel sources it was taken on and its DRAM bytes per launch, in
    the form bench.py reads; the launch list exists."""
    sys.path.insert(0, ROOT)
    import bench

    prof = os.path.join(ROOT, "profiles")
    names = sorted(f for f in os.listdir(prof) if f.endswith(".md"))
    assert "launches_prop_llama8b_32k_b1.md" in names
    for f in names:
        text = open(os.path.join(prof, f)).read()
        assert "ncu " in text and "--clock-control none" in text, f
        if f.startswith("launches_"):
            continue
        fields = {}
        for line in text.splitlines():
            if ":" in line and line.strip().startswith("- "):
                k, v = line.strip()[2:].split(":", 1)
                fields[k.strip()] = v.strip().strip("`")
        assert len(fields.get("source_digest", "")) == 16, f
        assert float(fields["dram_bytes_per_launch"]) > 0, f
    # the whole call's and pass 1's summaries are the ones the bench line uses
    for kernel in ("prop_call", "prop_pass1"):
        assert os.path.exists(os.path.join(prof, f"{kernel}_llama8b_32k_b1.md"))
    assert len(bench.source_digest()) == 16
