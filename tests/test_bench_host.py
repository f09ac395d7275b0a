"""The bench's host-side pieces on CPU: the multi-rank reductions it uses
for max-over-ranks timing (gloo, world size 2) and the reference arm's JSON
line (the CPU oracle timed on a bounded sample)."""

import io
import json
import os
import sys
from contextlib import redirect_stdout

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    r, w = bench.dist_init("gloo")
    bench.barrier()
    mx = bench.reduce_scalar(10.0 + r, "max")
    sm = bench.reduce_scalar(1.5 * (r + 1), "sum")
    q.put((r, w, mx, sm))
    import torch.distributed as dist
    dist.destroy_process_group()


def test_max_and_sum_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[0] for r in res] == [0, 1]
    assert all(r[1] == 2 and r[2] == 11.0 and r[3] == 4.5 for r in res)


def test_single_process_reductions_are_identity():
    import bench
    assert bench.reduce_scalar(3.25, "max") == 3.25
    bench.barrier()


def test_reference_arm_prints_one_json_line():
    import bench
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3", "--reference-budget", "3"])
    lines = [ln for ln in buf.getvalue().splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    assert d["metric"] == bench.METRIC and d["steps"] == 3


def test_reference_arm_other_ranks_exit_without_work(monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    buf = io.StringIO()
    with redirect_stdout(buf):
        bench.main(["--impl", "reference", "--steps", "3", "--warmup", "3"])
    assert buf.getvalue() == ""


def test_warmup_below_three_is_refused():
    import bench
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])


def test_traffic_is_reported_only_for_the_captured_source(monkeypatch, tmp_path):
    # the committed ncu summary is used while the kernel's sources hash to the captured value,
    # scaled to the launch by algorithmic bytes; a changed source or a missing entry gives None
    # (the sources' real hashes are not checked here: a kernel edited since its capture simply
    # reports no traffic until it is captured again)
    import json

    import bench

    rec = json.load(open(os.path.join(ROOT, "profiles", "ncu_traffic.json")))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel: rec[kernel]["source_sha256"])
    for kernel, r in rec.items():
        got = bench.ncu_traffic(kernel, r["algorithmic_bytes_per_launch"])
        assert got == pytest.approx(r["dram_bytes_per_launch"])
        assert bench.ncu_traffic(kernel, 2 * r["algorithmic_bytes_per_launch"]) == pytest.approx(
            2 * r["dram_bytes_per_launch"])
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel: "0" * 64)
    assert all(bench.ncu_traffic(k, 1.0) is None for k in rec)
    assert bench.ncu_traffic("no_such_kernel", 1.0) is None
