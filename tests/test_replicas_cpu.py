"""The N > 1 path of bench.py on CPU: world-size-2 gloo ranks agree on the
slowest rank's step time and count both ranks' tokens; the reference arm
prints from rank 0 only."""
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


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    from quantized_verification_gb300 import replicas
    replicas.barrier()
    ms_max, rate = replicas.job_step_time_and_rate(2.0 + rank, tokens_per_step=5, device="cpu")
    out[rank] = (ms_max, rate, replicas.world_size())
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_and_count_all_tokens():
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        port = _free_port()
        mp.start_processes(_rank_main, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
        res = dict(out)
    assert set(res) == {0, 1}
    for rank in (0, 1):
        ms_max, rate, w = res[rank]
        assert w == 2
        assert ms_max == pytest.approx(3.0)                   # rank 1 was slower
        assert rate == pytest.approx(2 * 5 / 3.0e-3)          # both ranks' tokens over that time


def test_single_process_is_world_one():
    from quantized_verification_gb300 import replicas
    ms_max, rate = replicas.job_step_time_and_rate(4.0, tokens_per_step=5, device="cpu")
    assert replicas.world_size() == 1 and ms_max == 4.0 and rate == pytest.approx(5 / 4.0e-3)


def test_reference_arm_prints_on_rank_zero_only(capsys):
    import importlib.util
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(root, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)

    class A:
        steps, warmup = 1, 0
    assert bench.run_reference(A(), rank=1, world=2) == 0
    assert capsys.readouterr().out == ""
