"""The multi-rank timing path of bench.py on CPU: two gloo ranks (127.0.0.1)
reduce their timings to the slowest rank's, the whole-job rate counts every
rank's units, and the reference arm does no work on ranks other than 0."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        # rank r took (10 + r) ms for the device-timed loop and (20 - r) ms end to end
        ms, ms_e2e = bench.max_over_ranks([10.0 + rank, 20.0 - rank], dist)
        out.put((rank, ms, ms_e2e, bench.whole_job_rate(1000, world, ms)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_and_count_every_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms, ms_e2e, rate in res:
        assert ms == 11.0 and ms_e2e == 20.0
        assert rate == pytest.approx(2 * 1000 / 11e-3)


def test_one_rank_passes_values_through():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([3, 4.5]) == [3.0, 4.5]
    assert bench.whole_job_rate(500, 1, 250.0) == pytest.approx(2000.0)


def test_reference_arm_does_no_work_off_rank_0(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.run_reference(None) is None
    assert capsys.readouterr().out == ""


def test_reference_arm_prints_the_contract_line(monkeypatch, capsys):
    """Rank 0 of the reference arm prints one JSON line with the keys the
    driver reads (the oracle on a small layer shape here, so the CPU suite
    stays fast; the line's shape is the same at page scale)."""
    import json
    import types
    sys.path.insert(0, ROOT)
    import bench
    from quantized_expert_ffn_gemv_gb300 import synth
    sh = synth.SMALL
    monkeypatch.setattr(synth, "PAGE", sh)
    monkeypatch.setattr(bench, "H", sh.H)
    monkeypatch.setattr(bench, "E", sh.E)
    monkeypatch.setattr(bench, "K", sh.k)
    monkeypatch.setattr(bench, "I", sh.I)
    monkeypatch.setattr(bench, "host_cores", lambda: 2)
    for v in ("RANK", "WORLD_SIZE", "LOCAL_RANK"):
        monkeypatch.delenv(v, raising=False)
    bench.run_reference(types.SimpleNamespace(steps=2, warmup=1))
    lines = [l for l in capsys.readouterr().out.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["value"] > 0 and d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 1
    assert d["higher_is_better"] is True and d["vs_baseline"] is None
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 2
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}
    assert "workload" in d["config"]
