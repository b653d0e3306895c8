"""Host logic of bench.py, without a GPU: the whole-job aggregation over ranks (two gloo ranks on
CPU, the way torchrun launches one replica per GPU), the summary of the clock samples taken during
the timed region, and the reference arm's rule that only rank 0 runs."""
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, t_ms, tokens, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    import torch.distributed as dist
    import bench as b
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        q.put((rank, b.aggregate(t_ms[rank], tokens[rank], dist, "cpu")))
    finally:
        dist.destroy_process_group()


def _run_ranks(t_ms, tokens):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, len(t_ms), port, t_ms, tokens, q)) for r in range(len(t_ms))]
    for p in procs:
        p.start()
    out = {}
    for _ in procs:
        r, v = q.get(timeout=120)
        out[r] = v
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return out


def test_aggregate_two_gloo_ranks_takes_slowest_time_and_all_tokens():
    out = _run_ranks([10.0, 12.5], [100, 90])
    assert out[0] == out[1] == (12.5, 190)


def test_aggregate_without_process_group_is_local():
    assert bench.aggregate(3.5, 42) == (3.5, 42)


def test_clock_summary_median_max_and_reasons():
    cs = bench.ClockSampler(0)
    cs.lines = [
        "0, 2070, 2070, 900.5, 0x0000000000000000, Not Active, Not Active, Not Active, Not Active",
        "0, 2055, 2070, 1390.2, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "0, 2040, 2070, 1399.0, 0x0000000000000004, Not Active, Not Active, Not Active, Active",
        "garbled line",
    ]
    s = cs.summary()
    assert s == {"sm_mhz": 2055.0, "sm_max_mhz": 2070.0, "reasons": ["sw_power_cap"], "samples": 3}


def test_clock_summary_flags_thermal_and_unsampled():
    cs = bench.ClockSampler(0)
    cs.lines = ["0, 1800, 2070, 1400, 0x40, Not Active, Active, Not Active, Not Active"]
    assert cs.summary()["reasons"] == ["hw_thermal_slowdown"]
    cs.lines = []
    assert cs.summary()["reasons"] == ["unsampled"]


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")

    def boom():
        raise AssertionError("a rank other than 0 ran the oracle")

    monkeypatch.setattr(bench, "OraclePool", boom)
    args = bench.argparse.Namespace(warmup=1, steps=1, gpus=2)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""


def test_oracle_pool_wave_counts_the_requests_accepted_tokens():
    """One wave of the CPU legs' worker pool (two spawned single-thread workers splitting the query
    heads) returns the request's accepted tokens as the oracle's accept gives them, and positive wall
    and worker times."""
    import oracle as O
    from workloads import configs, gen
    w = configs.scaled(configs.mixed_serving(), ctx_div=128, batch=2, vocab=2000)
    pool = bench.OraclePool(2)
    try:
        for b in range(2):
            wall, cpu, n = pool.wave(w, b)
            dr, lg = gen.request_logits(w, 0, b)
            assert n == O.accept(lg.numpy(), dr.numpy(), w.L[b])[1]
            assert wall > 0 and cpu > 0
    finally:
        pool.close()


def test_interval_coverage():
    """The overlap figure: the part of a copy interval under the union of compute intervals."""
    assert bench._covered((0.0, 10.0), [(2.0, 4.0), (3.0, 6.0), (8.0, 20.0)]) == pytest.approx(0.6)
    assert bench._covered((0.0, 10.0), []) == 0.0
    assert bench._covered((5.0, 6.0), [(0.0, 100.0)]) == pytest.approx(1.0)
