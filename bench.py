#!/usr/bin/env python3
"""Benchmark of the emulated sum all-reduce on one GB300 (per GPU).

Metric: all-reduce HBM GB/s (algorithmic bytes / device time), and its
fraction of the measured HBM peak, n = 8 ranks, bf16.

One step = one pass of every row of the hot path over one batch:
  batch   n = 8 rank buffers of S = 64 MiB bf16, N(0,1) (the prefill
          workload's largest size: 4096 tokens x hidden 8192), plus n = 8
          fp32 payloads of 1 MiB, U[-1,1] (the LL workload's largest size)
  rows    one-shot, two-shot (reduce-scatter + all-gather) and the
          2(n-1)-step ring over the bf16 batch; LL and LL128 pack ->
          flag-checked reduce -> unpack over the fp32 payloads (fresh step id
          per pass).  Argument checks and planning run inside every call.
`value` = all algorithmic HBM bytes of K steps on all ranks / max-over-ranks
device time.  The 1.3 GiB per-step working set is 10x the 129 MB L2, so no
flush is needed between steps.  Per-kernel times come from the library's
own launch record (CUDA events on the launching stream, AR_OPT_TIMING).

The run ends with ONE short JSON line (under 2 KB): the headline value, the
roofline of the dominant kernel (algorithmic and DRAM rates), the oracle
timed on the host (cpu_baseline), the end-to-end leg through host buffers
(e2e) and the SM clocks seen during the timed region.  Everything else it
measures goes to a details file (--details; by default bench_details.json
beside this file; relative paths are taken from here): a decode/prefill sweep of one-shot and
two-shot, the fused all-reduce + RMSNorm epilogue, every all-reduce call
side by side (variants), the LL payload sweep, the n = 16 doubling sweep,
the per-kernel table and the other CPU legs (cpu_parallel, cpu_calls).
Rows whose algorithmic rate is above the measured copy peak are marked
l2_assisted.

--impl reference times the CPU oracle instead (the reference arm), on a
bounded sample of the same workload.  Multi-GPU runs (torchrun) are
independent replicas: the path has no exchange between GPUs.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

MiB = 1 << 20
METRIC = "all-reduce HBM GB/s & % of GB300 HBM peak vs msg size, n=8 bf16"
NOMINAL_PEAK_GBS = 8000.0        # the ~8 TB/s HBM3e figure the target is stated against
FALLBACK_PEAK_GBS = 6800.0       # profiling recipe fallback when no measured peak is present


# --------------------------------------------------------------------------
# distributed plumbing (replicas: a barrier and max/sum of scalars only)
# --------------------------------------------------------------------------

def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("WORLD_SIZE", 1)), int(os.environ.get("LOCAL_RANK", 0))


def dist_init(backend: str):
    import torch.distributed as dist
    rank, world, _ = dist_env()
    if world > 1 and not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return rank, world


def reduce_scalar(x: float, op: str = "max") -> float:
    """max / sum of a host scalar over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX if op == "max" else dist.ReduceOp.SUM)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# --------------------------------------------------------------------------
# workload bookkeeping
# --------------------------------------------------------------------------

def step_bytes(n: int, N: int, e: int, ll_count: int) -> dict:
    """Algorithmic HBM bytes of every row of one step, from the library's plan."""
    import all_reduce_reduction_rank_gb300 as ar
    rows = {}
    for name, op in (("one_shot", ar.AR_OP_ONE_SHOT), ("two_shot", ar.AR_OP_TWO_SHOT), ("ring", ar.AR_OP_RING)):
        t = ar.ar_plan(op, n, N, {4: "f32", 2: "bf16"}[e])
        rows[name] = t.hbm_read_bytes + t.hbm_write_bytes
    for kind, (pk, rd, up) in (("ll", (ar.AR_OP_LL_PACK, ar.AR_OP_LL_REDUCE, ar.AR_OP_LL_UNPACK)),
                               ("ll128", (ar.AR_OP_LL128_PACK, ar.AR_OP_LL128_REDUCE, ar.AR_OP_LL128_UNPACK))):
        b = 0
        for op in (pk, rd, up):          # pack / unpack over all n buffers in one call
            t = ar.ar_plan(op, n, ll_count, "f32")
            b += t.hbm_read_bytes + t.hbm_write_bytes
        rows[kind] = b
    return rows


def step_bytes_model(n: int, N: int, e: int, ll_count: int) -> dict:
    """The same per-row bytes from the oracle's closed forms (oracle/model.py),
    for the legs that run the oracle and must not load the CUDA library."""
    from oracle import model
    rows = {"one_shot": sum(model.hbm_one_shot(n, N, e)), "two_shot": sum(model.hbm_two_shot(n, N, e)),
            "ring": sum(model.hbm_ring(n, N, e))}
    rows["ll"] = sum(model.hbm_ll_pack(ll_count)) * n + sum(model.hbm_ll_reduce(n, ll_count)) + \
        sum(model.hbm_ll_unpack(ll_count)) * n
    rows["ll128"] = sum(model.hbm_ll128_pack(ll_count)) * n + sum(model.hbm_ll128_reduce(n, ll_count)) + \
        sum(model.hbm_ll128_unpack(ll_count)) * n
    return rows


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured (MEASURED_PEAKS.json hbm_gbs: torch copy, read+write bytes)"
    except Exception:
        return FALLBACK_PEAK_GBS, "fallback (6.8 TB/s, earlier GB300 copy measurement)"


KERNEL_SOURCES = {
    "one_shot": ["one_shot.cu"], "reduce_scatter": ["two_shot.cu"], "all_gather": ["two_shot.cu"],
    "ring_rs_step": ["ring.cu"], "ring_ag_step": ["ring.cu"],
    "ll_pack": ["ll.cu"], "ll_unpack": ["ll.cu"], "ll_reduce": ["ll.cu"],
    "ll128_pack": ["ll.cu"], "ll128_unpack": ["ll.cu"], "ll128_reduce": ["ll.cu"],
    "allreduce_rmsnorm": ["rmsnorm.cu"], "push": ["one_shot_modes.cu"], "push_reduce": ["one_shot_modes.cu"],
    "copyin": ["one_shot_modes.cu"], "ring_rs_step_rounded": ["ring.cu"], "tree_level": ["tree.cu"],
    "ring_persistent": ["ring_persistent.cu"], "ring_cluster": ["ring_cluster.cu"], "tree_fused": ["tree.cu"],
    "ring_fused": ["ring_fused.cu"], "ring_rounded_fused": ["ring_fused.cu"], "two_shot": ["two_shot.cu"],
}


def kernel_source_hash(kernel: str) -> str:
    csrc = os.path.join(ROOT, "all_reduce_reduction_rank_gb300", "csrc")
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel] + ["common.cuh", "internal.h"]:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def ncu_traffic(kernel: str, bytes_per_launch: float):
    """DRAM bytes per launch from the committed ncu summary, scaled to this
    launch by algorithmic bytes; None when there is none or the kernel's
    source changed since the capture."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)[kernel]
    except Exception:
        return None
    if rec.get("source_sha256") != kernel_source_hash(kernel):
        return None
    scale = bytes_per_launch / float(rec["algorithmic_bytes_per_launch"])
    return float(rec["dram_bytes_per_launch"]) * scale


# --------------------------------------------------------------------------
# clocks during the timed region
# --------------------------------------------------------------------------

class ClockSampler:
    FIELDS = ("timestamp,pci.bus_id,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, bus_id: int | None):
        self.bus_id = bus_id
        self.rows = []
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        t0 = time.time()
        while not self.rows and time.time() - t0 < 5:   # wait for the first sample
            time.sleep(0.02)

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append((time.time(), [c.strip() for c in line.split(",")]))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float, t1: float) -> dict | None:
        if not self.rows:
            return None
        rows = [r for t, r in self.rows if len(r) >= 10]
        if self.bus_id is not None:
            mine = [r for r in rows if _bus_number(r[1]) == self.bus_id]
            rows = mine or rows
        timed = [r for (t, r) in self.rows if t0 <= t <= t1 and r in rows]
        use = timed if len(timed) >= 1 else rows
        sm = [float(r[2]) for r in use if _isnum(r[2])]
        mx = [float(r[3]) for r in use if _isnum(r[3])]
        reasons = sorted({name for r in use for name, v in zip(self.REASONS, r[6:10]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(use), "in_timed_region": len(timed),
                "power_w_max": max((float(r[4]) for r in use if _isnum(r[4])), default=None)}


def _isnum(s):
    try:
        float(s)
        return True
    except ValueError:
        return False


def _bus_number(bus_id: str):
    try:
        return int(bus_id.split(":")[-2], 16)
    except Exception:
        return None


# --------------------------------------------------------------------------
# our arm
# --------------------------------------------------------------------------

class Workload:
    """Device buffers of one batch and the pre-marshalled C-ABI calls of a step."""

    def __init__(self, n: int, S: int, ll_count: int, dev, seed: int):
        import ctypes

        import torch

        import all_reduce_reduction_rank_gb300 as ar
        import workloads

        self.n, self.S, self.N, self.ll_count, self.dev = n, S, S // 2, ll_count, dev
        self.ins = workloads.rank_inputs_device(n, self.N, "bf16", "normal", seed, device=dev)
        self.outs = [torch.empty_like(t) for t in self.ins]
        self.pay = workloads.rank_inputs_device(n, ll_count, "f32", "uniform", seed + 1, device=dev)
        lb, l128 = ar.ar_ll_bytes(4 * ll_count), ar.ar_ll128_bytes(4 * ll_count)
        mk = lambda nb: [torch.zeros(nb, dtype=torch.uint8, device=dev) for _ in range(n)]
        self.ll_lines, self.ll_red, self.l128_lines, self.l128_red = mk(lb), mk(lb), mk(l128), mk(l128)
        self.ll_dst = [torch.zeros(ll_count, dtype=torch.float32, device=dev) for _ in range(n)]
        self.l128_dst = [torch.zeros(ll_count, dtype=torch.float32, device=dev) for _ in range(n)]
        self.h = ar.ar_create(n, S)
        self.stream = torch.cuda.Stream(device=dev)
        self.s = ctypes.c_void_p(self.stream.cuda_stream)
        P = lambda ts: (ctypes.c_void_p * n)(*[t.data_ptr() for t in ts])
        self.p_in, self.p_out = P(self.ins), P(self.outs)
        self.p_ll, self.p_llr = P(self.ll_lines), P(self.ll_red)
        self.p_l128, self.p_l128r = P(self.l128_lines), P(self.l128_red)
        self.p_pay = P(self.pay)
        self.p_lld, self.p_l128d = P(self.ll_dst), P(self.l128_dst)
        self.L = ar.lib()
        self.step_id = 0
        self.launches_per_step = None   # counted by count_launches()

    def calls(self, k: int):
        """The step's C-ABI calls, in order, for step id k."""
        L, h, s, N, c = self.L, self.h, self.s, self.N, self.ll_count
        return (lambda: L.ar_one_shot(h, self.p_in, self.p_out, N, 1, s),
                lambda: L.ar_two_shot(h, self.p_in, self.p_out, N, 1, s),
                lambda: L.ar_ring(h, self.p_in, self.p_out, N, 1, s),
                lambda: L.ar_ll_pack_n(h, self.p_pay, self.p_ll, c, k, s),
                lambda: L.ar_ll_reduce(h, self.p_ll, self.p_llr, c, k, s),
                lambda: L.ar_ll_unpack_n(h, self.p_llr, self.p_lld, c, k, s),
                lambda: L.ar_ll128_pack_n(h, self.p_pay, self.p_l128, c, k, s),
                lambda: L.ar_ll128_reduce(h, self.p_l128, self.p_l128r, c, k, s),
                lambda: L.ar_ll128_unpack_n(h, self.p_l128r, self.p_l128d, c, k, s))

    def count_launches(self) -> int:
        """Run one (untimed) step and add up the kernels each call reports
        (ar_traffic), so the count follows the forms the options select."""
        import all_reduce_reduction_rank_gb300 as ar
        self.step_id += 1
        total = 0
        for call in self.calls(self.step_id):
            ar.check(call(), "step call")
            total += ar.ar_traffic(self.h).launches
        self.launches_per_step = total
        return total

    def run(self):
        L, h, s, n, N, c = self.L, self.h, self.s, self.n, self.N, self.ll_count
        self.step_id += 1
        k = self.step_id
        rc = L.ar_one_shot(h, self.p_in, self.p_out, N, 1, s)
        rc |= L.ar_two_shot(h, self.p_in, self.p_out, N, 1, s)
        rc |= L.ar_ring(h, self.p_in, self.p_out, N, 1, s)
        rc |= L.ar_ll_pack_n(h, self.p_pay, self.p_ll, c, k, s)
        rc |= L.ar_ll_reduce(h, self.p_ll, self.p_llr, c, k, s)
        rc |= L.ar_ll_unpack_n(h, self.p_llr, self.p_lld, c, k, s)
        rc |= L.ar_ll128_pack_n(h, self.p_pay, self.p_l128, c, k, s)
        rc |= L.ar_ll128_reduce(h, self.p_l128, self.p_l128r, c, k, s)
        rc |= L.ar_ll128_unpack_n(h, self.p_l128r, self.p_l128d, c, k, s)
        if rc:
            raise RuntimeError(f"a C-ABI call failed in step {k}")

    def close(self):
        import all_reduce_reduction_rank_gb300 as ar
        ar.check(ar.ar_destroy(self.h), "ar_destroy")


def time_steps(wl, K: int, before_step=None) -> tuple[float, float]:
    """Device ms of exactly K steps, bracketed by a barrier + synchronize, and
    the host ms spent issuing them."""
    import torch
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    ev0.record(wl.stream)
    t0 = time.perf_counter()
    for i in range(K):
        if before_step is not None:
            before_step(i)
        wl.run()
    host_ms = 1e3 * (time.perf_counter() - t0)
    ev1.record(wl.stream)
    torch.cuda.synchronize()
    barrier()
    return ev0.elapsed_time(ev1), host_ms


def per_kernel(records, K: int, peak: float) -> dict:
    agg = {}
    for name, _op, ms, b, launches in records:
        a = agg.setdefault(name, {"launches": 0, "ms": 0.0, "bytes": 0})
        a["launches"] += launches
        a["ms"] += ms
        a["bytes"] += b
    total = sum(a["ms"] for a in agg.values()) or 1.0
    out = {}
    for name, a in agg.items():
        gbs = a["bytes"] / (a["ms"] * 1e-3) / 1e9 if a["ms"] > 0 else None
        out[name] = {"launches_per_step": a["launches"] / K, "us_per_launch": 1e3 * a["ms"] / a["launches"],
                     "bytes_per_launch": a["bytes"] / a["launches"], "GB/s": gbs,
                     "frac_of_peak": gbs / peak if gbs else None, "share": a["ms"] / total}
    return out


def sweep(wl, peak: float, batches: int = 7, min_calls: int = 64) -> dict:
    """one-shot and two-shot over the decode and prefill message sizes (n = 8,
    bf16).  Each rank's 64 MiB input and output buffers are cut into slots of
    the message size; a batch issues back-to-back calls on successive slots
    (the batch's calls touch 1 GiB between two uses of a slot, so no call finds
    its data in the 129 MB L2) and is timed with one pair of CUDA events, which
    also avoids the ~2 us resolution of timing a single short call.  Reported:
    the median over batches of the time per call."""
    import ctypes

    import torch

    import all_reduce_reduction_rank_gb300 as ar
    import workloads

    sizes = sorted({2 * c for c in workloads.CONFIGS[2]["counts"]} | {2 * c for c in workloads.CONFIGS[3]["counts"]})
    res = {"one_shot": [], "two_shot": []}
    n = wl.n
    for S in sizes:
        if S > wl.S:
            continue
        N = S // 2
        slots = wl.S // S
        P = lambda ts, k: (ctypes.c_void_p * n)(*[t.data_ptr() + k * S for t in ts])
        pin = [P(wl.ins, k) for k in range(slots)]
        pout = [P(wl.outs, k) for k in range(slots)]
        calls = max(min_calls, slots)
        for algo, call, op in (("one_shot", wl.L.ar_one_shot, ar.AR_OP_ONE_SHOT),
                               ("two_shot", wl.L.ar_two_shot, ar.AR_OP_TWO_SHOT)):
            t = ar.ar_plan(op, n, N, "bf16")
            b = t.hbm_read_bytes + t.hbm_write_bytes
            for k in range(min(slots, 4)):
                ar.check(call(wl.h, pin[k], pout[k], N, 1, wl.s), algo)
            per_call = []
            for _ in range(batches):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(wl.stream)
                for i in range(calls):
                    call(wl.h, pin[i % slots], pout[i % slots], N, 1, wl.s)
                e1.record(wl.stream)
                e1.synchronize()
                per_call.append(e0.elapsed_time(e1) / calls)
            ar.check(ar.ar_status(wl.h), algo)
            ms = statistics.median(per_call)
            gbs = b / (ms * 1e-3) / 1e9
            algbw = S / (ms * 1e-3) / 1e9
            row = {"bytes_per_rank": S, "us": round(ms * 1e3, 3), "hbm_GB/s": round(gbs, 1),
                   "frac_of_peak": round(gbs / peak, 4), "algbw_GB/s": round(algbw, 1),
                   "busbw_GB/s": round(algbw * 2 * (n - 1) / n, 1), "calls_per_batch": calls, "batches": batches}
            if S <= GRAPH_MAX_BYTES:
                row["graph_us"] = round(_graph_us(wl.stream, lambda i: call(wl.h, pin[i % slots], pout[i % slots],
                                                                            N, 1, wl.s)), 3)
                ar.check(ar.ar_status(wl.h), algo)
            res[algo].append(mark_l2(row, peak))
    return res


def fused_epilogue(wl, peak: float, batches: int = 7, calls: int = 200) -> list:
    """ar_allreduce_rmsnorm on the decode shapes (n = 8 bf16, tokens {1, 8,
    32, 64} x hidden {4096, 8192}), beside ar_one_shot on the same shape: the
    fused epilogue's cost over a bare all-reduce.  Back-to-back calls on
    rotating slots of the 64 MiB rank buffers, one event pair per batch."""
    import ctypes

    import torch

    import all_reduce_reduction_rank_gb300 as ar

    n, out = wl.n, []
    res = torch.randn(64 * 8192, device=wl.dev).to(torch.bfloat16)
    res_out = torch.empty_like(res)
    w = torch.rand(8192, device=wl.dev).to(torch.bfloat16)
    for T in (1, 8, 32, 64):
        for H in (4096, 8192):
            S = T * H * 2
            slots = min(wl.S // S, 4096)
            P = lambda ts, k: (ctypes.c_void_p * n)(*[t.data_ptr() + k * S for t in ts])
            pin = [P(wl.ins, k) for k in range(slots)]
            pout = [P(wl.outs, k) for k in range(slots)]
            row = {"tokens": T, "hidden": H}
            for name in ("fused", "one_shot"):
                def call(k):
                    if name == "fused":
                        return wl.L.ar_allreduce_rmsnorm(wl.h, pin[k], res.data_ptr(), w.data_ptr(),
                                                         ctypes.c_float(1e-6), pout[k], res_out.data_ptr(), T, H, 1,
                                                         wl.s)
                    return wl.L.ar_one_shot(wl.h, pin[k], pout[k], T * H, 1, wl.s)
                ar.check(call(0), name)
                per = []
                for _ in range(batches):
                    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                    e0.record(wl.stream)
                    for i in range(calls):
                        call(i % slots)
                    e1.record(wl.stream)
                    e1.synchronize()
                    per.append(e0.elapsed_time(e1) / calls)
                us = statistics.median(per) * 1e3
                b = (2 * n + 2) * S + H * 2 if name == "fused" else 2 * n * S
                row[name + "_us"] = round(us, 3)
                row[name + "_GB/s"] = round(b / (us * 1e-6) / 1e9, 1)
                row[name + "_graph_us"] = round(_graph_us(wl.stream, lambda i: call(i % slots)), 3)
            ar.check(ar.ar_status(wl.h), "fused epilogue")
            out.append(row)
    return out


def _batched_us(stream, fn, calls: int, batches: int) -> float:
    """Median over batches of the device time per call of `calls` back-to-back
    calls fn(i), one CUDA event pair per batch, µs."""
    import torch
    per = []
    for _ in range(batches):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(calls):
            fn(i)
        e1.record(stream)
        e1.synchronize()
        per.append(e0.elapsed_time(e1) / calls)
    return statistics.median(per) * 1e3


GRAPH_MAX_BYTES = 8 * MiB   # messages up to this size are also timed from a CUDA graph


def _graph_us(stream, fn, in_graph: int = 20, replays: int = 10, batches: int = 5) -> float:
    """Device time per call with the host out of the way: `in_graph` calls
    fn(i) captured once into a CUDA graph on `stream`, replayed back to back;
    median over batches, us.  Small calls issued one by one from Python are
    bound by the host's issue rate (ctypes + launch, ~3 us a call on a
    GB300 machine's Grace CPU), which the replay removes."""
    import torch
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(in_graph):
            fn(i)
    g.replay()
    torch.cuda.synchronize()
    per = []
    for _ in range(batches):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(replays):
                g.replay()
        e1.record(stream)
        e1.synchronize()
        per.append(e0.elapsed_time(e1) * 1e3 / (in_graph * replays))
    del g
    return statistics.median(per)


def ll_sweep(wl, peak: float, batches: int = 5) -> dict:
    """The LL / LL128 workload over its payload sizes (n = 8 fp32 payloads of
    8 B .. 1 MiB per rank, doubling): one pass = batched pack of the n
    payloads, the flag-checked reduce, batched unpack, with a fresh step id
    per pass.  Reported per size: µs per pass, payload GB/s (n P / t), the
    lines' wire efficiency and the algorithmic HBM GB/s of the three calls
    (all from back-to-back passes issued from Python), and the device time
    per pass replayed from a CUDA graph."""
    import all_reduce_reduction_rank_gb300 as ar
    import workloads

    n, L, h, s = wl.n, wl.L, wl.h, wl.s
    out = {"ll": [], "ll128": []}
    step = [1 << 20]
    for count in workloads.CONFIGS[4]["counts"]:
        P = 4 * count
        for kind in ("ll", "ll128"):
            if kind == "ll":
                calls = (L.ar_ll_pack_n, L.ar_ll_reduce, L.ar_ll_unpack_n)
                lines, red, dst = wl.p_ll, wl.p_llr, wl.p_lld
                ops = (ar.AR_OP_LL_PACK, ar.AR_OP_LL_REDUCE, ar.AR_OP_LL_UNPACK)
                wire = P / ar.ar_ll_bytes(P)
            else:
                calls = (L.ar_ll128_pack_n, L.ar_ll128_reduce, L.ar_ll128_unpack_n)
                lines, red, dst = wl.p_l128, wl.p_l128r, wl.p_l128d
                ops = (ar.AR_OP_LL128_PACK, ar.AR_OP_LL128_REDUCE, ar.AR_OP_LL128_UNPACK)
                wire = P / ar.ar_ll128_bytes(P)

            def one(_i, calls=calls, lines=lines, red=red, dst=dst):
                step[0] += 1
                k = step[0]
                calls[0](h, wl.p_pay, lines, count, k, s)
                calls[1](h, lines, red, count, k, s)
                calls[2](h, red, dst, count, k, s)

            b = 0
            for op in ops:
                t = ar.ar_plan(op, n, count, "f32")
                b += t.hbm_read_bytes + t.hbm_write_bytes
            one(0)
            us = _batched_us(wl.stream, one, 200 if P <= 64 * 1024 else 50, batches)
            ar.check(ar.ar_status(h), kind + " sweep")
            # device time per pass: 20 passes (their step ids fixed at capture) replayed from a graph
            gus = _graph_us(wl.stream, one)
            ar.check(ar.ar_status(h), kind + " sweep, graph")
            out[kind].append(mark_l2({"payload_bytes": P, "us_per_pass": round(us, 3),
                                      "graph_us_per_pass": round(gus, 3),
                                      "payload_GB/s": round(n * P / (us * 1e-6) / 1e9, 2),
                                      "wire_efficiency": round(wire, 4), "hbm_GB/s": round(b / (us * 1e-6) / 1e9, 1),
                                      "frac_of_peak": round(b / (us * 1e-6) / 1e9 / peak, 4)}, peak))
    return out


def n16_sweep(dev, peak: float, batches: int = 3) -> dict:
    """The n = 16 doubling sweep (bf16 and fp16, 1 KiB .. 256 MiB per rank):
    ring, one-shot and two-shot.  Inputs are 16 device buffers of 256 MiB;
    smaller messages rotate over slots of them so that back-to-back calls do
    not find their data in L2.  µs per call and algorithmic HBM GB/s of
    back-to-back calls issued from Python, and (up to 8 MiB) the device time
    per call replayed from a CUDA graph."""
    import ctypes

    import torch

    import all_reduce_reduction_rank_gb300 as ar
    import workloads

    n = 16
    top = 256 * MiB
    ins = workloads.rank_inputs_device(n, top // 2, "bf16", "normal_over_n", workloads.seed_of(5), device=dev)
    outs = [torch.empty_like(t) for t in ins]
    h = ar.ar_create(n, top)
    stream = torch.cuda.Stream(device=dev)
    sp = ctypes.c_void_p(stream.cuda_stream)
    L = ar.lib()
    res = {}
    try:
        for dtype in ("bf16", "f16"):
            dt = ar.DTYPES[dtype]
            for name, call, op in (("ring", L.ar_ring, ar.AR_OP_RING), ("one_shot", L.ar_one_shot, ar.AR_OP_ONE_SHOT),
                                   ("two_shot", L.ar_two_shot, ar.AR_OP_TWO_SHOT)):
                rows = []
                for count in workloads.CONFIGS[5]["counts"]:
                    S = 2 * count
                    slots = top // S
                    P = lambda ts, k: (ctypes.c_void_p * n)(*[t.data_ptr() + k * S for t in ts])
                    nslot = min(slots, 256)
                    pin = [P(ins, k * (slots // nslot)) for k in range(nslot)]
                    pout = [P(outs, k * (slots // nslot)) for k in range(nslot)]
                    calls = max(8, min(nslot, 256))

                    def one(i, call=call, pin=pin, pout=pout, count=count):
                        call(h, pin[i % nslot], pout[i % nslot], count, dt, sp)

                    ar.check(call(h, pin[0], pout[0], count, dt, sp), name)
                    us = _batched_us(stream, one, calls, batches)
                    t = ar.ar_plan(op, n, count, dtype)
                    gbs = (t.hbm_read_bytes + t.hbm_write_bytes) / (us * 1e-6) / 1e9
                    gus = round(_graph_us(stream, one), 3) if S <= GRAPH_MAX_BYTES else None
                    rows.append([S, round(us, 2), round(gbs, 1), gus, gbs > peak])
                ar.check(ar.ar_status(h), name)
                res[f"{dtype}/{name}"] = rows
    finally:
        ar.ar_destroy(h)
    return {"columns": ["bytes_per_rank", "us", "hbm_GB/s", "graph_us", "l2_assisted"], "peak": peak, **res}


VARIANT_SIZES = (64 * 1024, 1 * MiB, 8 * MiB, 64 * MiB)
NOALLOC_MAX_BYTES = 8 * MiB   # ar_ring_noalloc's static scratch holds n = 8 bf16 up to this per rank
E2E_SETS = 3   # device buffer sets the e2e leg rotates over
E2E_WINDOWS = 3   # timed regions of the e2e leg; the median is reported


def variants(wl, peak: float, batches: int = 5, min_calls: int = 32) -> dict:
    """Every all-reduce call of the library on the same n = 8 bf16 buffers, at
    64 KiB, 1 MiB, 8 MiB and 64 MiB per rank: one-shot, its push and copy-in
    forms, two-shot, the ring (one launch per step), the ring with hop
    rounding, the persistent single-launch LL128 ring (global-memory inboxes,
    and over a thread-block cluster), the pairwise tree, the one-pass forms,
    and the handle-free ring (ar_ring_noalloc, up to its 8 MiB limit).
    Timing as in `sweep` (back-to-back calls on rotating slots, one event pair
    per batch, median of the batches); bytes are each call's algorithmic HBM
    bytes (ar_plan)."""
    import ctypes

    import torch

    import all_reduce_reduction_rank_gb300 as ar

    n, L, h = wl.n, wl.L, wl.h
    for opt in (ar.AR_OPT_PUSH_STAGING, ar.AR_OPT_REGISTERED, ar.AR_OPT_PERSISTENT):
        ar.check(ar.ar_set_option(h, opt, 1), "variant buffers")
    algos = (("one_shot", L.ar_one_shot, ar.AR_OP_ONE_SHOT),
             ("one_shot_push", L.ar_one_shot_push, ar.AR_OP_ONE_SHOT_PUSH),
             ("one_shot_copyin", L.ar_one_shot_copyin, ar.AR_OP_ONE_SHOT_COPYIN),
             ("two_shot", L.ar_two_shot, ar.AR_OP_TWO_SHOT),
             ("two_shot_two_launches", L.ar_two_shot, ar.AR_OP_TWO_SHOT),
             ("two_shot_tile_flags", L.ar_two_shot, ar.AR_OP_TWO_SHOT),
             ("ring", L.ar_ring, ar.AR_OP_RING),
             ("ring_rounded", L.ar_ring_rounded, ar.AR_OP_RING_ROUNDED),
             ("ring_persistent", L.ar_ring_persistent, ar.AR_OP_RING_PERSISTENT),
             ("ring_cluster", L.ar_ring_cluster, ar.AR_OP_RING_CLUSTER),
             ("ring_fused", L.ar_ring_fused, ar.AR_OP_RING_FUSED),
             ("ring_rounded_fused", L.ar_ring_rounded_fused, ar.AR_OP_RING_ROUNDED_FUSED),
             ("tree", L.ar_tree, ar.AR_OP_TREE),
             ("tree_fused", L.ar_tree_fused, ar.AR_OP_TREE_FUSED),
             # the handle-free ring (static scratch, up to 8 MiB per rank at n = 8 bf16)
             ("ring_noalloc", lambda _h, pi, po, cnt, dt, st: L.ar_ring_noalloc(n, pi, po, cnt, dt, st),
              ar.AR_OP_RING))
    res = {a[0]: [] for a in algos}
    for S in VARIANT_SIZES:
        if S > wl.S:
            continue
        N = S // 2
        slots = wl.S // S
        P = lambda ts, k: (ctypes.c_void_p * n)(*[t.data_ptr() + k * S for t in ts])
        pin = [P(wl.ins, k) for k in range(slots)]
        pout = [P(wl.outs, k) for k in range(slots)]
        calls = max(min_calls, min(slots, 4096))
        for name, call, op in algos:
            if name == "ring_noalloc" and S > NOALLOC_MAX_BYTES:
                continue
            # two-shot as its default form, and forced to its other two forms
            ar.check(ar.ar_set_option(h, ar.AR_OPT_TWO_SHOT_IMPL,
                                      {"two_shot_two_launches": 1, "two_shot_tile_flags": 3}.get(name, 0)))
            t = ar.ar_plan(op, n, N, "bf16")
            b = t.hbm_read_bytes + t.hbm_write_bytes
            for k in range(min(slots, 4)):
                ar.check(call(h, pin[k], pout[k], N, 1, wl.s), name)
            per_call = []
            for _ in range(batches):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(wl.stream)
                for i in range(calls):
                    call(h, pin[i % slots], pout[i % slots], N, 1, wl.s)
                e1.record(wl.stream)
                e1.synchronize()
                per_call.append(e0.elapsed_time(e1) / calls)
            ar.check(ar.ar_status(h), name)
            ms = statistics.median(per_call)
            gbs = b / (ms * 1e-3) / 1e9
            algbw = S / (ms * 1e-3) / 1e9
            row = {"bytes_per_rank": S, "us": round(ms * 1e3, 3), "hbm_GB/s": round(gbs, 1),
                   "frac_of_peak": round(gbs / peak, 4), "algbw_GB/s": round(algbw, 1),
                   "launches": t.launches if name == "ring_noalloc" else ar.ar_traffic(h).launches,
                   "calls_per_batch": calls}
            if S <= GRAPH_MAX_BYTES:
                row["graph_us"] = round(_graph_us(wl.stream, lambda i: call(h, pin[i % slots], pout[i % slots],
                                                                            N, 1, wl.s)), 3)
                ar.check(ar.ar_status(h), name)
            res[name].append(mark_l2(row, peak))
    ar.check(ar.ar_set_option(h, ar.AR_OPT_TWO_SHOT_IMPL, 0))
    for opt in (ar.AR_OPT_PUSH_STAGING, ar.AR_OPT_REGISTERED, ar.AR_OPT_PERSISTENT):
        ar.check(ar.ar_set_option(h, opt, 0), "variant buffers")
    return res


def e2e_leg(wl, K: int, bytes_per_step: int) -> dict:
    """The same step through the public API with HOST buffers: every step
    copies its inputs from pinned host memory, runs, and reads its results
    (the n all-reduced buffers and the n LL and LL128 unpacked payloads) back.

    Steps rotate over E2E_SETS device buffer sets, each with its own stream
    (copy in -> the step's calls -> copy out, in order on that stream), so
    one step's copies overlap the other sets' calls and copies in the other
    direction; every step still moves all of its own bytes in and out."""
    import torch
    n = wl.n
    extra = [Workload(n, wl.S, wl.ll_count, wl.dev, seed=1004 + i) for i in range(E2E_SETS - 1)]
    sets = (wl, *extra)
    h_in = [torch.empty_like(t, device="cpu").pin_memory() for t in wl.ins]
    h_pay = [torch.empty_like(t, device="cpu").pin_memory() for t in wl.pay]
    for h, d in zip(h_in + h_pay, wl.ins + wl.pay):
        h.copy_(d)
    h_outs = [[torch.empty_like(t, device="cpu").pin_memory() for t in w.outs + w.ll_dst + w.l128_dst]
              for w in sets]
    h2d = sum(t.numel() * t.element_size() for t in h_in + h_pay)
    d2h = sum(t.numel() * t.element_size() for t in h_outs[0])

    def one(i):
        w, hout = sets[i % len(sets)], h_outs[i % len(sets)]
        with torch.cuda.stream(w.stream):
            for h, d in zip(h_in + h_pay, w.ins + w.pay):
                d.copy_(h, non_blocking=True)
            w.run()
            for h, d in zip(hout, w.outs + w.ll_dst + w.l128_dst):
                h.copy_(d, non_blocking=True)

    for i in range(2 * len(sets)):   # every set's buffers and copies touched twice before timing
        one(i)
    torch.cuda.synchronize()

    def window() -> tuple[float, float]:
        """One timed region of K steps: device ms (events, max over ranks) and host issue ms."""
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier()
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        ev0.record(wl.stream)
        for w in extra:
            w.stream.wait_event(ev0)
        for i in range(K):
            one(i)
        for w in extra:
            done = torch.cuda.Event()
            done.record(w.stream)
            wl.stream.wait_event(done)
        ev1.record(wl.stream)
        t1 = time.perf_counter()
        torch.cuda.synchronize()
        return reduce_scalar(ev0.elapsed_time(ev1), "max"), (t1 - t0) * 1e3

    # E2E_WINDOWS timed regions, the median reported: the leg issues ~50 host calls per step from
    # Python, and a region that met a busy host (one run on a shared box: 6.4 ms per step with
    # the host link measured at its usual rate right after) would otherwise set the figure alone
    # one untimed region first: on one box the first region after the warm-up passes read 7.4 ms
    # per step and the next two 3.5 ms
    window()
    wins = [window() for _ in range(E2E_WINDOWS)]
    import all_reduce_reduction_rank_gb300 as ar
    for w in sets:
        ar.check(ar.ar_status(w.h), "e2e status")
    link = _host_link(wl, h_in + h_pay, h_outs[0], sets[1] if len(sets) > 1 else wl)
    for w in extra:
        w.close()
    ms = statistics.median(d for d, _ in wins) / K
    world = dist_env()[1]
    return {"value": round(world * bytes_per_step / (ms * 1e-3) / 1e9, 2), "unit": "GB/s",
            "ms_per_step": round(ms, 4), "steps": K, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "windows": [{"ms_per_step": round(d / K, 4), "host_issue_ms_per_step": round(hst / K, 4)}
                        for d, hst in wins],
            "pipelining": f"{E2E_SETS} buffer sets on {E2E_SETS} streams: copy in, calls, copy out per step; "
                          f"median of {E2E_WINDOWS} timed regions of {K} steps",
            "host_link_GB/s": link}


def _host_link(wl, h_in, h_out, other) -> dict:
    """This machine's pinned host<->device copy rates, measured on the e2e
    leg's own buffers after its timed region: the step's inputs host->device,
    its outputs device->host, and both at once on two streams (median of 3,
    GB/s).  The e2e figure is bound by these, which vary from machine to
    machine."""
    import torch

    d_in = wl.ins + wl.pay
    d_out = wl.outs + wl.ll_dst + wl.l128_dst
    b_in = sum(t.numel() * t.element_size() for t in h_in)
    b_out = sum(t.numel() * t.element_size() for t in h_out)

    def timed(fn):
        per = []
        for _ in range(3):
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(wl.stream)
            fn()
            e1.record(wl.stream)
            torch.cuda.synchronize()
            per.append(e0.elapsed_time(e1) * 1e-3)
        return statistics.median(per)

    def h2d(stream=None):
        with torch.cuda.stream(stream or wl.stream):
            for h, d in zip(h_in, d_in):
                d.copy_(h, non_blocking=True)

    def d2h(stream=None):
        with torch.cuda.stream(stream or wl.stream):
            for h, d in zip(h_out, d_out):
                h.copy_(d, non_blocking=True)

    def both():
        done = torch.cuda.Event()
        other.stream.wait_stream(wl.stream)
        h2d(wl.stream)
        d2h(other.stream)
        done.record(other.stream)
        wl.stream.wait_event(done)

    t_in, t_out, t_both = timed(h2d), timed(d2h), timed(both)
    return {"h2d": round(b_in / t_in / 1e9, 1), "d2h": round(b_out / t_out / 1e9, 1),
            "both": round((b_in + b_out) / t_both / 1e9, 1)}


def run_ours(args):
    import torch

    import all_reduce_reduction_rank_gb300 as ar

    rank, world = dist_init("nccl")
    local = dist_env()[2]
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    ar.lib()                                   # fails loudly if the library is not built
    n, S, ll_count = 8, args.size_mib * MiB, (1 * MiB) // 4
    wl = Workload(n, S, ll_count, dev, seed=1003)
    ar.check(ar.ar_set_option(wl.h, ar.AR_OPT_ONE_SHOT_IMPL, args.one_shot_impl))
    ar.check(ar.ar_set_option(wl.h, ar.AR_OPT_CTAS_PER_SM, args.ctas_per_sm))
    ar.check(ar.ar_set_option(wl.h, ar.AR_OPT_TWO_SHOT_IMPL, args.two_shot_impl))
    wl.count_launches()
    peak, peak_src = measured_peak()
    rows = step_bytes(n, wl.N, 2, ll_count)
    bytes_step = sum(rows.values())
    for _ in range(args.warmup):
        wl.run()
    torch.cuda.synchronize()
    ar.check(ar.ar_status(wl.h), "warm-up status")
    # per-launch events on every k-th timed step only (each event pair costs a
    # little device time between launches); the others run unrecorded
    every = max(1, args.timing_every)
    sampled = (args.steps + every - 1) // every
    ar.check(ar.ar_set_option(wl.h, ar.AR_OPT_TIMING, min(1 << 20, wl.launches_per_step * sampled)))
    # (a ring phase's n-1 launches share one record, so this is more than enough)
    L = ar.lib()

    def sample(i):
        L.ar_set_option(wl.h, ar.AR_OPT_TIMING_PAUSE, 0 if i % every == 0 else 1)

    try:
        bus = torch.cuda.get_device_properties(dev).pci_bus_id
    except Exception:
        bus = None
    clocks = ClockSampler(bus)
    clocks.start()
    t_wall0 = time.time()
    ms, host_ms = time_steps(wl, args.steps, sample)
    t_wall1 = time.time()
    clocks.stop()
    records = ar.ar_timing(wl.h)
    ar.check(ar.ar_status(wl.h), "timed-region status")
    ar.check(ar.ar_set_option(wl.h, ar.AR_OPT_TIMING, 0))
    ms_max = reduce_scalar(ms, "max")
    total_bytes = reduce_scalar(bytes_step * args.steps, "sum")
    value = total_bytes / (ms_max * 1e-3) / 1e9
    kernels = per_kernel(records, sampled, peak)
    # launches in the timed region: the sampled steps' from their records (a step that records runs
    # the ring's pieces on one stream, fewer launches than the two-stream steps), the others' from
    # the untimed counting step
    gpu_launches = wl.launches_per_step * (args.steps - sampled) + sum(r[4] for r in records)
    dom = max(kernels, key=lambda k: kernels[k]["share"])
    dk = kernels[dom]
    traffic = ncu_traffic(dom, dk["bytes_per_launch"])
    roofline = {"bound": "hbm", "kernel": dom, "achieved": round(dk["GB/s"], 1), "peak": peak, "unit": "GB/s",
                "frac": round(dk["GB/s"] / peak, 4), "traffic": traffic,
                "bytes_per_launch": dk["bytes_per_launch"], "us_per_launch": round(dk["us_per_launch"], 3),
                "peak_source": peak_src}
    roofline.update(dram_rate(traffic, dk["us_per_launch"], peak))

    # the end-to-end leg first: a leg that allocates and frees gigabytes of device memory (the
    # variants leg's optional buffers) measured to slow the next timed region by up to a quarter
    e2e = e2e_leg(wl, max(3, min(args.steps, args.e2e_steps)), bytes_step) if args.e2e else None
    sw = sweep(wl, peak) if args.sweep else None
    fe = fused_epilogue(wl, peak) if args.sweep else None
    lls = ll_sweep(wl, peak) if args.sweep else None
    va = variants(wl, peak) if args.sweep else None
    n16 = n16_sweep(dev, peak) if args.sweep else None
    cpu = cpu_par = cpu_calls = None
    if world == 1 and rank == 0 and args.cpu_baseline:
        cpu = cpu_baseline(seconds=args.cpu_seconds)
        cpu_par = cpu_parallel(seconds=args.cpu_seconds)
        cpu_calls = calls_cpu() if args.sweep else None
    wl.close()
    full = {
        "metric": METRIC, "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_max / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"n8_bf16_S{args.size_mib}MiB_prefill+n8_f32_P1MiB_ll", "n_ranks": n,
                   "bytes_per_rank": S, "payload": "bf16 N(0,1), fp32 accumulation",
                   "ll_payload_bytes_per_rank": 4 * ll_count,
                   "rows": ["one_shot", "two_shot", "ring", "ll(pack,reduce,unpack)", "ll128(pack,reduce,unpack)"],
                   "bytes_per_step": bytes_step, "bytes_per_step_by_row": rows,
                   "l2": "inputs larger than L2: 1.3 GiB touched per step vs 129 MB L2; no flush",
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
        "frac_of_peak": round(value / world / peak, 4), "frac_of_8tbs": round(value / world / NOMINAL_PEAK_GBS, 4),
        "roofline": roofline, "kernels": kernels, "gpu_launches": gpu_launches,
        "launch_timing": {"steps_sampled": sampled, "every": every, "records": len(records),
                          "launches_recorded": sum(r[4] for r in records)},
        "host_issue_ms_per_step": round(host_ms / args.steps, 4),
        "clocks": clocks.summary(t_wall0, t_wall1), "e2e": e2e, "cpu_baseline": cpu, "cpu_parallel": cpu_par,
        "cpu_calls": cpu_calls, "sweep": sw, "fused_epilogue": fe, "variants": va, "ll_sweep": lls,
        "n16_sweep": n16,
    }
    if rank == 0:
        path = write_details(full, args.details)
        print(json.dumps(headline(full, path)), flush=True)


def dram_rate(traffic, us_per_launch: float, peak: float) -> dict:
    """The dominant kernel's DRAM rate beside its algorithmic one: ncu's
    DRAM bytes per launch over the same average launch time.  An algorithmic
    rate above the copy peak with a DRAM rate below it means L2 served part
    of the algorithmic bytes."""
    if traffic is None or not us_per_launch:
        return {"dram_achieved": None, "dram_frac": None}
    a = traffic / (us_per_launch * 1e-6) / 1e9
    return {"dram_achieved": round(a, 1), "dram_frac": round(a / peak, 4)}


def mark_l2(row: dict, peak: float, key: str = "hbm_GB/s") -> dict:
    """Flag a row whose algorithmic rate is above the measured copy peak:
    such a rate is only reachable with part of its bytes served by L2."""
    v = row.get(key)
    if v is not None and v > peak:
        row["l2_assisted"] = True
    return row


HEADLINE_MAX_BYTES = 2000


def headline(full: dict, details_path: str | None) -> dict:
    """The one JSON line the run ends with: the headline figures only (the
    sweeps and per-kernel tables go to the details file).  Kept under
    HEADLINE_MAX_BYTES so that a reader keeping the tail of stdout has it
    whole."""
    cfg = full["config"]
    rf = full.get("roofline") or {}
    keep_rf = ("bound", "kernel", "achieved", "peak", "unit", "frac", "traffic", "bytes_per_launch",
               "us_per_launch", "dram_achieved", "dram_frac")
    cpu = full.get("cpu_baseline")
    e2e = full.get("e2e")
    clk = full.get("clocks")
    line = {k: full[k] for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                                 "higher_is_better", "scaling", "vs_baseline", "dtype", "data")}
    line["config"] = {"workload": cfg["workload"], "n_ranks": cfg["n_ranks"], "bytes_per_rank": cfg["bytes_per_rank"],
                      "ll_payload_bytes_per_rank": cfg["ll_payload_bytes_per_rank"],
                      "bytes_per_step": cfg["bytes_per_step"], "l2": "no flush: 1.3 GiB per step > 129 MB L2",
                      "parallelism": cfg["parallelism"]}
    line["frac_of_peak"] = full.get("frac_of_peak")
    line["frac_of_8tbs"] = full.get("frac_of_8tbs")
    line["roofline"] = {k: rf.get(k) for k in keep_rf}
    if rf.get("peak_source"):
        line["roofline"]["peak_source"] = "measured" if rf["peak_source"].startswith("measured") else "fallback"
    line["cpu_baseline"] = None if cpu is None else {
        "value": cpu["value"], "unit": cpu["unit"], "cores": cpu["cores"], "kind": cpu["kind"],
        "sample": cpu["sample"][:200]}
    line["e2e"] = None if e2e is None else {
        k: e2e[k] for k in ("value", "unit", "ms_per_step", "h2d_bytes_per_step", "d2h_bytes_per_step")}
    line["clocks"] = None if clk is None else {k: clk.get(k) for k in ("sm_mhz", "sm_max_mhz", "reasons")}
    line["gpu_launches"] = full["gpu_launches"]
    line["details"] = details_path
    if len(json.dumps(line)) > HEADLINE_MAX_BYTES:      # never expected; keep the line whole regardless
        line["cpu_baseline"] and line["cpu_baseline"].update(sample=line["cpu_baseline"]["sample"][:60])
        line["details"] = os.path.basename(details_path) if details_path else None
    return line


def write_details(full: dict, path: str | None) -> str | None:
    """Everything the run measured (sweeps, variants, per-kernel table, CPU
    legs) as one JSON file; returns its path, or None if it cannot be
    written (the headline line is printed regardless)."""
    if not path:
        return None
    if not os.path.isabs(path):
        path = os.path.join(ROOT, path)
    try:
        os.makedirs(os.path.dirname(path), exist_ok=True)
        with open(path, "w") as f:
            json.dump(full, f, indent=1)
    except OSError as exc:
        print(f"bench: details not written ({exc})", file=sys.stderr)
        return None
    return os.path.relpath(path, ROOT)


# --------------------------------------------------------------------------
# the oracle on the host (CPU baseline / reference arm)
# --------------------------------------------------------------------------

def oracle_sample(scale_div: int, seed: int = 1003):
    """The step's rows at 1/scale_div of the workload, run by the oracle."""
    import oracle
    import workloads
    n = 8
    N = (64 * MiB // 2) // scale_div
    c = ((1 * MiB) // 4) // scale_div
    xs = workloads.rank_inputs(n, N, "bf16", "normal", seed)
    ps = workloads.payload_f32(n, c, seed + 1)
    rows = step_bytes_model(n, N, 2, c)

    def run(step_id: int):
        oracle.all_reduce(xs, "bf16")
        oracle.all_gather(oracle.reduce_scatter(xs, "bf16"), "bf16")
        oracle.ring(xs, "bf16")
        red, _ = oracle.ll_reduce([oracle.ll_pack(p, step_id) for p in ps], c, step_id)
        for r in red:
            oracle.ll_unpack(r, c, step_id)
        red, _ = oracle.ll128_reduce([oracle.ll128_pack(p, step_id) for p in ps], c, step_id)
        for r in red:
            oracle.ll128_unpack(r, c, step_id)

    desc = f"oracle on n=8 bf16 {2 * N // 1024} KiB per rank + LL/LL128 {4 * c // 1024} KiB fp32 payloads (1/{scale_div} of the step)"
    return run, sum(rows.values()), desc


def cpu_baseline(seconds: float = 10.0, scale_div: int = 32) -> dict:
    run, b, desc = oracle_sample(scale_div)
    run(1)
    reps, t0 = 0, time.perf_counter()
    while True:
        run(2 + reps)
        reps += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": round(reps * b / dt / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{desc}, {reps} passes in {dt:.1f} s, single-threaded C"}


def cpu_parallel(seconds: float = 10.0, scale_div: int = 32) -> dict:
    """The same oracle sample split by element range over every host core
    (threads; the oracle's C routines run without the GIL): each thread does
    one-shot, two-shot (the reduce-scatter sums then the all-gather copies),
    the ring (its per-element order statement, which the literal step
    simulation is pinned to) and the LL / LL128 pack -> reduce -> unpack of
    its range.  A second CPU figure beside the single-threaded oracle."""
    from concurrent.futures import ThreadPoolExecutor

    import numpy as np

    import oracle
    import workloads
    n = 8
    N = (64 * MiB // 2) // scale_div
    c = ((1 * MiB) // 4) // scale_div
    xs = workloads.rank_inputs(n, N, "bf16", "normal", 1003)
    ps = workloads.payload_f32(n, c, 1004)
    C = oracle.chunk_elems(n, N, "bf16")
    chunk = (np.arange(N) // C).astype(np.int32)
    b = sum(step_bytes_model(n, N, 2, c).values())
    cores = os.cpu_count() or 1
    # element ranges: multiples of 30 words keep LL128 lines whole
    def ranges(total, align):
        per = -(-total // cores)
        per = -(-per // align) * align
        return [(lo, min(total, lo + per)) for lo in range(0, total, per)]
    xr, pr = ranges(N, 8), ranges(c, 30)

    def work(t, step_id):
        if t < len(xr):
            lo, hi = xr[t]
            cols = [x[lo:hi] for x in xs]
            oracle.all_reduce(cols, "bf16")
            oracle.all_reduce(cols, "bf16")            # two-shot: the same sums, then copies
            oracle.ring_order_sum(cols, chunk[lo:hi], "bf16")
        if t < len(pr):
            lo, hi = pr[t]
            sub = [p[lo:hi] for p in ps]
            red, _ = oracle.ll_reduce([oracle.ll_pack(p, step_id) for p in sub], hi - lo, step_id)
            for r in red:
                oracle.ll_unpack(r, hi - lo, step_id)
            red, _ = oracle.ll128_reduce([oracle.ll128_pack(p, step_id) for p in sub], hi - lo, step_id)
            for r in red:
                oracle.ll128_unpack(r, hi - lo, step_id)

    threads = max(len(xr), len(pr))
    with ThreadPoolExecutor(max_workers=threads) as pool:
        list(pool.map(lambda t: work(t, 1), range(threads)))
        reps, t0 = 0, time.perf_counter()
        while True:
            list(pool.map(lambda t: work(t, 2 + reps), range(threads)))
            reps += 1
            if time.perf_counter() - t0 >= seconds:
                break
        dt = time.perf_counter() - t0
    return {"value": round(reps * b / dt / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle routines, element-range parallel",
            "sample": f"the cpu_baseline sample (1/{scale_div} of the step) over {threads} threads, "
                      f"{reps} passes in {dt:.1f} s"}


def calls_cpu(min_seconds: float = 0.5) -> dict:
    """The oracle beside each all-reduce call of the variants leg and beside
    the fused epilogue: n = 8 bf16 at 1 MiB per rank (the epilogue at
    64 tokens x 8192), timed single-threaded on the host, GB/s of the same
    algorithmic bytes the GPU figures use (ar_plan)."""
    import numpy as np

    import all_reduce_reduction_rank_gb300 as ar
    import oracle
    import workloads
    n, N = 8, (1 * MiB) // 2
    xs = workloads.rank_inputs(n, N, "bf16", "normal_over_n", 1003)
    rows = {}

    def timed(fn):
        fn()
        reps, t0 = 0, time.perf_counter()
        while True:
            fn()
            reps += 1
            if time.perf_counter() - t0 >= min_seconds:
                return (time.perf_counter() - t0) / reps

    for name, fn, op in (("one_shot", lambda: oracle.all_reduce(xs, "bf16"), ar.AR_OP_ONE_SHOT),
                         ("one_shot_push", lambda: oracle.all_reduce(xs, "bf16"), ar.AR_OP_ONE_SHOT_PUSH),
                         ("one_shot_copyin", lambda: oracle.all_reduce(xs, "bf16"), ar.AR_OP_ONE_SHOT_COPYIN),
                         ("two_shot", lambda: oracle.all_gather(oracle.reduce_scatter(xs, "bf16"), "bf16"),
                          ar.AR_OP_TWO_SHOT),
                         ("ring", lambda: oracle.ring(xs, "bf16"), ar.AR_OP_RING),
                         ("ring_rounded", lambda: oracle.ring_rounded(xs, "bf16"), ar.AR_OP_RING_ROUNDED),
                         ("ring_persistent", lambda: oracle.ring(xs, "bf16"), ar.AR_OP_RING_PERSISTENT),
                         ("ring_cluster", lambda: oracle.ring(xs, "bf16"), ar.AR_OP_RING_CLUSTER),
                         ("ring_fused", lambda: oracle.ring(xs, "bf16"), ar.AR_OP_RING_FUSED),
                         ("ring_rounded_fused", lambda: oracle.ring_rounded(xs, "bf16"),
                          ar.AR_OP_RING_ROUNDED_FUSED),
                         ("tree", lambda: oracle.tree(xs, "bf16"), ar.AR_OP_TREE),
                         ("tree_fused", lambda: oracle.tree(xs, "bf16"), ar.AR_OP_TREE_FUSED)):
        t = ar.ar_plan(op, n, N, "bf16")
        sec = timed(fn)
        rows[name] = {"bytes_per_rank": 2 * N, "ms": round(sec * 1e3, 3),
                      "GB/s": round((t.hbm_read_bytes + t.hbm_write_bytes) / sec / 1e9, 3)}
    T, H = 64, 8192
    xr = workloads.rank_inputs(n, T * H, "bf16", "normal", 1005)
    res = workloads.rank_inputs(1, T * H, "bf16", "normal", 1006)[0]
    w = workloads.rank_inputs(1, H, "bf16", "uniform", 1007)[0]
    sec = timed(lambda: oracle.allreduce_rmsnorm(xr, res, w, 1e-6, T, H, "bf16"))
    S = T * H * 2
    rows["allreduce_rmsnorm"] = {"tokens": T, "hidden": H, "ms": round(sec * 1e3, 3),
                                 "GB/s": round(((2 * n + 2) * S + 2 * H) / sec / 1e9, 3)}
    return {"kind": "oracle", "cores": 1, "sample": "n=8 bf16, 1 MiB per rank; epilogue 64 x 8192", **rows}


def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return                                   # rank 0 alone runs the reference arm
    budget = args.reference_budget / max(1, args.steps + args.warmup)   # seconds per step
    div = 1024
    run, b, desc = oracle_sample(div)
    t0 = time.perf_counter()
    run(1)
    t_small = time.perf_counter() - t0
    while div > 8 and t_small * 2 <= budget:
        div //= 2
        t_small *= 2
    run, b, desc = oracle_sample(div)
    for i in range(args.warmup):
        run(1 + i)
    t0 = time.perf_counter()
    for i in range(args.steps):
        run(1000 + i)
    dt = time.perf_counter() - t0
    value = args.steps * b / dt / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": {"workload": f"n8_bf16_S{args.size_mib}MiB_prefill+n8_f32_P1MiB_ll", "n_ranks": 8,
                       "sample_scale": f"1/{div}"},
            "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": desc},
            "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=300)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--size-mib", type=int, default=64, help="bytes per rank of the bf16 batch, MiB")
    p.add_argument("--no-sweep", dest="sweep", action="store_false")
    p.add_argument("--no-e2e", dest="e2e", action="store_false")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--timing-every", type=int, default=10,
                   help="record per-launch events on every k-th timed step")
    p.add_argument("--one-shot-impl", type=int, default=0, help="AR_OPT_ONE_SHOT_IMPL (0 auto, 1, 2)")
    p.add_argument("--ctas-per-sm", type=int, default=0, help="AR_OPT_CTAS_PER_SM (0 auto)")
    p.add_argument("--two-shot-impl", type=int, default=0,
                   help="AR_OPT_TWO_SHOT_IMPL (0 auto, 1 two launches, 2 one launch with a per-tile CTA "
                        "barrier, 3 one launch with per-tile flags between CTAs)")
    p.add_argument("--no-cpu-baseline", dest="cpu_baseline", action="store_false")
    p.add_argument("--cpu-seconds", type=float, default=10.0)
    p.add_argument("--details", default="bench_details.json",
                   help="JSON file for everything beyond the headline line (sweeps, variants, per-kernel "
                        "table, CPU legs); '' for none")
    p.add_argument("--reference-budget", type=float, default=150.0,
                   help="seconds the reference arm's warm-up + timed steps should take in all")
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
