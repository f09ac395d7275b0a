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


def _synthetic_full(bench, world=1):
    """A result dict shaped like run_ours' with every detail leg filled in
    (long enough that printing it whole would run to tens of KB)."""
    rows = {"one_shot": 1 << 30, "two_shot": 9 << 27, "ring": 5 << 30, "ll": 80 << 20, "ll128": 44 << 20}
    sweep_row = {"bytes_per_rank": 1 << 20, "us": 4.1, "hbm_GB/s": 4055.0, "frac_of_peak": 0.6, "graph_us": 4.06}
    return {
        "metric": bench.METRIC, "value": 6969.7, "unit": "GB/s", "n_gpus": world, "steps": 300, "warmup": 5,
        "ms_per_step": 0.79, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": "n8_bf16_S64MiB_prefill+n8_f32_P1MiB_ll", "n_ranks": 8, "bytes_per_rank": 64 << 20,
                   "payload": "bf16 N(0,1), fp32 accumulation", "ll_payload_bytes_per_rank": 1 << 20,
                   "rows": list(rows), "bytes_per_step": sum(rows.values()), "bytes_per_step_by_row": rows,
                   "l2": "inputs larger than L2", "parallelism": "single GPU"},
        "frac_of_peak": 1.02, "frac_of_8tbs": 0.87,
        "roofline": {"bound": "hbm", "kernel": "ring_rs_step", "achieved": 6970.1, "peak": 6791.7, "unit": "GB/s",
                     "frac": 1.0263, "traffic": 304.7e6, "bytes_per_launch": 316.4e6, "us_per_launch": 45.35,
                     "peak_source": "measured (MEASURED_PEAKS.json hbm_gbs: torch copy, read+write bytes)",
                     "dram_achieved": 6718.9, "dram_frac": 0.9893},
        "kernels": {f"k{i}": {"share": 0.1, "GB/s": 6000.0} for i in range(12)},
        "gpu_launches": 6900, "launch_timing": {"steps_sampled": 30},
        "clocks": {"sm_mhz": 2070.0, "sm_max_mhz": 2070.0, "reasons": [], "samples": 40, "in_timed_region": 5,
                   "power_w_max": 820.0},
        "e2e": {"value": 1555.0, "unit": "GB/s", "ms_per_step": 3.6, "steps": 20, "h2d_bytes_per_step": 545 << 20,
                "d2h_bytes_per_step": 554 << 20, "pipelining": "3 buffer sets", "host_link_GB/s": {"h2d": 210.0}},
        "cpu_baseline": {"value": 2.49, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "oracle on n=8 bf16 2048 KiB per rank + LL/LL128 32 KiB fp32 payloads "
                                   "(1/32 of the step), 15 passes in 10.2 s, single-threaded C" * 3},
        "cpu_parallel": {"value": 12.9}, "cpu_calls": {"one_shot": {"ms": 15.6}},
        "sweep": {"one_shot": [sweep_row] * 12, "two_shot": [sweep_row] * 12},
        "fused_epilogue": [{"tokens": 1, "hidden": 4096, "fused_us": 3.8}] * 8,
        "variants": {f"v{i}": [sweep_row] * 4 for i in range(13)},
        "ll_sweep": {"ll": [sweep_row] * 18, "ll128": [sweep_row] * 18},
        "n16_sweep": {"columns": [], "bf16/ring": [[1024, 51.0, 1.0, 34.1, False]] * 19},
    }


def test_headline_line_is_short_and_carries_the_contract_keys(tmp_path):
    import bench
    full = _synthetic_full(bench)
    assert len(json.dumps(full)) > 8000          # printing the whole result would not fit a short tail
    path = bench.write_details(full, str(tmp_path / "d" / "details.json"))
    line = bench.headline(full, path)
    text = json.dumps(line)
    assert len(text.encode()) < 2048 and "\n" not in text
    d = json.loads(text)
    assert d["value"] > 0 and d["metric"] == bench.METRIC and d["unit"] == "GB/s"
    for k in ("n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling", "vs_baseline", "dtype",
              "data", "config", "roofline", "cpu_baseline", "e2e", "clocks", "gpu_launches"):
        assert k in d, k
    assert d["config"]["workload"] == full["config"]["workload"]
    rf = d["roofline"]
    assert rf["bound"] == "hbm" and rf["peak"] > 0 and rf["frac"] == pytest.approx(rf["achieved"] / rf["peak"], 1e-3)
    assert rf["dram_frac"] == pytest.approx(rf["dram_achieved"] / rf["peak"], 1e-3)
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["e2e"]["h2d_bytes_per_step"] > 0 and d["e2e"]["d2h_bytes_per_step"] > 0
    assert d["e2e"]["value"] != d["value"]
    assert set(d["clocks"]) == {"sm_mhz", "sm_max_mhz", "reasons"}
    # the details file holds everything, and parses back
    back = json.load(open(tmp_path / "d" / "details.json"))
    assert back["n16_sweep"] == json.loads(json.dumps(full["n16_sweep"]))


def test_headline_tolerates_absent_legs():
    import bench
    full = _synthetic_full(bench)
    full.update(e2e=None, cpu_baseline=None, clocks=None)
    full["roofline"].update(traffic=None, dram_achieved=None, dram_frac=None)
    d = json.loads(json.dumps(bench.headline(full, None)))
    assert d["e2e"] is None and d["cpu_baseline"] is None and d["roofline"]["dram_frac"] is None


def test_dram_rate_and_l2_marking():
    import bench
    r = bench.dram_rate(300e6, 50.0, 6000.0)
    assert r["dram_achieved"] == pytest.approx(6000.0) and r["dram_frac"] == pytest.approx(1.0)
    assert bench.dram_rate(None, 50.0, 6000.0) == {"dram_achieved": None, "dram_frac": None}
    assert bench.mark_l2({"hbm_GB/s": 7000.0}, 6800.0)["l2_assisted"] is True
    assert "l2_assisted" not in bench.mark_l2({"hbm_GB/s": 6700.0}, 6800.0)


def test_model_step_bytes_match_the_library_plan():
    # the oracle legs count bytes from the closed forms, without loading the CUDA library;
    # the GPU arm counts them from the library's own plan: both must agree
    import bench
    from all_reduce_reduction_rank_gb300 import build as arbuild
    arbuild.build()
    for N, c in ((32 << 20, 1 << 18), (1 << 10, 30), (4099, 7)):
        assert bench.step_bytes_model(8, N, 2, c) == bench.step_bytes(8, N, 2, c)


def test_reference_arm_does_not_load_the_cuda_library():
    # the reference arm is the oracle alone: run it in a fresh interpreter and check
    # that libar_gb300.so was never mapped
    import subprocess
    code = ("import sys, io, contextlib; sys.path.insert(0, %r); import bench\n"
            "buf = io.StringIO()\n"
            "with contextlib.redirect_stdout(buf):\n"
            "    bench.main(['--impl', 'reference', '--steps', '3', '--warmup', '3', '--reference-budget', '2'])\n"
            "maps = open('/proc/self/maps').read()\n"
            "print('LOADED' if 'libar_gb300' in maps else 'CLEAN')\n" % ROOT)
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr
    assert out.stdout.strip().splitlines()[-1] == "CLEAN"
