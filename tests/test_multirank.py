"""The N > 1 host path of bench.py on CPU, with two gloo ranks: the job's time
is the slowest rank's, its rate all ranks' units over that time (replicas,
weak scaling), and the reference arm runs on rank 0 only."""
import socket

import torch
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, port, elapsed, q):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=2)
    try:
        q.put((rank,) + bench.job_rate(elapsed[rank], 100, 2, torch.device("cpu")))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_job_rate_is_all_units_over_the_slowest_of_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    elapsed = (0.5, 2.0)
    ps = [ctx.Process(target=_rank, args=(r, port, elapsed, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, rate in got:
        assert slowest == 2.0
        assert rate == 2 * 100 / 2.0


def test_job_rate_single_rank_needs_no_group():
    assert bench.job_rate(0.25, 10, 1, torch.device("cpu")) == (0.25, 40.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    import synth
    cfg = synth.with_cache(synth.CONFIGS["tiny"])

    class A:
        steps, warmup, seed = 2, 1, 0

    assert bench.run_reference(A, cfg) is None
    assert capsys.readouterr().out == ""
