"""Host-side logic of bench.py without a GPU: algorithmic counts, the committed-traffic lookup, the
max-over-ranks aggregation across two gloo ranks on CPU, and the reference arm's JSON line."""
import json
import multiprocessing as mp
import os
import socket

import pytest

import bench


def test_algorithmic_counts_prefill_4096():
    b, f = bench.algorithmic(4096, 16, 32, True)
    # q, k at 16 key heads + v + g + beta + o (bf16) + S0 in + S_T out
    assert b == 2 * 4096 * 16 * 128 * 2 + 4096 * 32 * 128 * 2 * 2 + 2 * 4096 * 32 * 4 + 2 * 32 * 128 * 128 * 4
    assert b == 105_906_176
    per_head_chunk = 5 * 2 * 64 * 64 * 128 + 3 * 2 * 64 * 128 * 128 + 64 ** 3 / 3
    assert abs(per_head_chunk - 11.62e6) < 0.01e6
    assert f == pytest.approx(32 * 64 * per_head_chunk)


def test_profiled_traffic_requires_matching_sources(tmp_path, monkeypatch):
    prof = tmp_path / "profiles"
    prof.mkdir()
    (prof / "dram_traffic_x.md").write_text(
        f"sources: {bench.source_digest()}\ndram bytes per step: 1234\n| gdr_a | 1000 |\n| gdr_b | 234 |\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    os.makedirs(tmp_path / "gated_deltanet_rule_gb300", exist_ok=True)
    os.symlink(os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                            "gated_deltanet_rule_gb300", "csrc"), tmp_path / "gated_deltanet_rule_gb300" / "csrc")
    total, per = bench.profiled_traffic("x")
    assert total == 1234 and per == {"gdr_a": 1000, "gdr_b": 234}
    (prof / "dram_traffic_x.md").write_text("sources: 0000000000000000\ndram bytes per step: 1234\n")
    assert bench.profiled_traffic("x") == (None, None)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    seconds = [2.0, 5.0][rank]
    value, tmax = bench.aggregate(4096 * 10, seconds)
    bench.barrier()
    q.put((rank, value, tmax))
    dist.destroy_process_group()


def test_aggregate_max_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, tmax in out:
        assert tmax == 5.0                              # slowest rank sets the time
        assert value == pytest.approx(2 * 4096 * 10 / 5.0)


def test_reference_arm_line(monkeypatch, capsys):
    monkeypatch.setitem(bench.WORKLOADS, "tiny", (128, 8, 16, True, "R1"))
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"])
    line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["metric"] == bench.METRIC and line["unit"] == "tokens/s"
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]


def test_reference_arm_nonzero_rank_prints_nothing(monkeypatch, capsys):
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setitem(bench.WORKLOADS, "tiny", (128, 8, 16, True, "R1"))
    bench.main(["--impl", "reference", "--workload", "tiny", "--steps", "1", "--warmup", "3"])
    assert capsys.readouterr().out.strip() == ""
