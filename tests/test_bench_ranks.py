"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each timing its
own replica; the job's time is the slowest rank's and its throughput counts
every rank's rows. The reference arm prints from rank 0 only."""

import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = 10.0 + 5.0 * rank                  # rank 1 is the slow one
        got = bench.max_over_ranks(ms, world, torch.device("cpu"))
        dist.barrier()
        out[rank] = (got, bench.job_throughput(4, 100, world, got))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank_main, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0
    # 4 rows x 100 steps on each of 2 ranks in 15 ms
    assert res[0][1] == pytest.approx(4 * 100 * 2 / 0.015)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(12.5, 1, None) == 12.5
    assert bench.job_throughput(1, 1000, 1, 23.4) == pytest.approx(1000 / 0.0234)


def test_reference_arm_prints_from_rank_zero_only(capsys):
    class A:  # the fields reference_main reads
        workload, steps, warmup, gpus = "decode", 1, 0, 2
    bench.reference_main(A, rank=1, world=2)
    assert capsys.readouterr().out == ""


def test_reference_arm_json_line():
    """`bench.py --impl reference` times the oracle on the host and prints one
    JSON line with the keys the bench contract asks for."""
    import json
    import subprocess
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]


def test_traffic_record_attaches_only_on_current_sources(tmp_path, monkeypatch):
    """A DRAM-traffic record is attached to a roofline only when it was taken on
    the kernel sources as they are now (same source hash), for the same path
    and workload."""
    import json

    sha = bench.source_sha(bench.KERNEL_SOURCES["gemm_tc"])
    (tmp_path / "profiles").mkdir()
    rec_file = tmp_path / "profiles" / "ncu_traffic.json"
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "source_sha", lambda paths: sha)

    def attached(records, workload="prefill4096"):
        rec_file.write_text(json.dumps(records))
        r = {"path": "gemm_tc", "roofline": {}}
        bench.attach_traffic(r, workload)
        return r["roofline"]["traffic"], r["roofline"]["kernel_source_sha"]

    good = {"gemm_tc:prefill4096": {"dram_bytes_per_launch": 123.0, "source_sha": sha}}
    assert attached(good) == (123.0, sha)
    stale = {"gemm_tc:prefill4096": {"dram_bytes_per_launch": 123.0, "source_sha": "0" * 16}}
    assert attached(stale) == (None, sha)
    assert attached(good, workload="decode64") == (None, sha)
    rec_file.unlink()
    r = {"path": "gemm_tc", "roofline": {}}
    bench.attach_traffic(r, "prefill4096")
    assert r["roofline"]["traffic"] is None
