"""Pins for the closed forms: the pages' printed table and worked exercises
(stored under tests/golden/ with their citations), and brute-force counts."""

import math
import os

import pytest

from oracle import model

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]


def _kv(fields):
    it = iter(fields[1:])
    return {k: v for k, v in zip(it, it)}


def test_alpha_beta_table_reproduces_printed_values():
    rows = _rows("alpha_beta_table.txt")
    head = {r[0]: r[1] for r in rows if r[0] in ("n", "beta", "alpha")}
    n, beta, alpha = int(head["n"]), float(head["beta"]), float(head["alpha"])
    algos = model.alpha_beta(n, beta, alpha)
    names = ["ring", "tree", "one-shot", "two-shot", "NVLS"]
    checked = 0
    for r in rows:
        if r[0] == "row":
            S = int(r[1])
            t = {k: f(S) * 1e6 for k, f in algos.items()}
            for name, printed in zip(names, r[2:7]):
                assert f"{t[name]:.1f}" == printed, (S, name, t[name])
            assert model.fastest_without_nvls(t) == r[7]
            checked += 1
        elif r[0] == "ring1g":
            S = int(r[1])
            t = algos["ring"](S)
            assert f"{t * 1e3:.2f}" == r[2]
            assert f"{S / t / 1e9:.0f}" == r[3]
            assert f"{model.busbw(S / t, n) / 1e9:.0f}" == r[4]
    assert checked == 5


def test_busbw_exercise():
    (row,) = [r for r in _rows("exercises.txt") if r[0] == "busbw_exercise"]
    kv = _kv(row)
    n, bb, S = int(kv["n"]), float(kv["busbw"]), int(kv["bytes"])
    ar_alg = bb / model.BUS_FACTOR["all_reduce"](n)
    ag_alg = bb / model.BUS_FACTOR["all_gather"](n)
    assert f"{ar_alg / 1e9:.1f}" == kv["ar_algbw"]
    assert f"{ag_alg / 1e9:.0f}" == kv["ag_algbw"]
    assert f"{model.time_from_busbw(S, bb, n) * 1e3:.1f}" == kv["ar_ms"]
    assert f"{model.time_from_busbw(S, bb, n, 'all_gather') * 1e3:.2f}" == kv["ag_ms"]


def test_crossover_exercise():
    rows = {r[0]: _kv(r) for r in _rows("exercises.txt")}
    kv = rows["crossover"]
    n, a, b = int(kv["n"]), float(kv["alpha"]), float(kv["beta"])
    assert (n - 1) * (1 - 2 / n) == pytest.approx(float(kv["denom"]))
    s = model.one_two_shot_crossover(n, b, a)
    assert f"{s / 1e3:.0f}" == kv["kb"]
    # at S* the two model times agree
    t = model.alpha_beta(n, b, a)
    assert t["one-shot"](s) == pytest.approx(t["two-shot"](s), rel=1e-12)
    assert model.one_two_shot_crossover(int(rows["crossover_none"]["n"]), b, a) is None


def test_tp_exercise():
    rows = {r[0]: _kv(r) for r in _rows("exercises.txt")}
    d = rows["tp_decode"]
    n, S, bw = int(d["n"]), float(d["bytes"]), float(d["bw"])
    assert f"{model.link_bytes_ring(n, S) / bw * 1e6:.2f}" == d["us"]
    p = rows["tp_prefill"]
    S = float(p["bytes"])
    sent = model.link_bytes_ring(int(p["n"]), S)
    assert f"{sent / 1e6:.0f}" == p["sent_mb"]
    assert f"{sent / float(p['bw']) * 1e3:.2f}" == p["ms"]


@pytest.mark.parametrize("n", [2, 3, 8, 16])
def test_link_traffic_closed_forms(n):
    S = 1 << 20
    assert model.link_bytes_one_shot(n, S) == (n - 1) * S
    assert model.link_bytes_two_shot(n, S) == pytest.approx(2 * (n - 1) / n * S)
    assert model.link_bytes_ring(n, S) == pytest.approx(model.link_bytes_two_shot(n, S))
    assert model.steps_ring(n) == 2 * (n - 1)
    # "2(p-1) S/p -> about 2S as p grows, almost independent of the card count"
    assert model.link_bytes_ring(1024, S) == pytest.approx(2 * S, rel=1e-2)
    # two ranks: one-shot and two-shot move the same bytes (no crossover)
    if n == 2:
        assert model.link_bytes_one_shot(n, S) == model.link_bytes_two_shot(n, S)


def _brute_ring_bytes(n, N, e):
    """Count the ring's HBM bytes step by step over the actual chunk lengths."""
    q = 16 // e
    C = -(-(-(-N // n)) // q) * q
    length = [max(0, min((c + 1) * C, N) - min(c * C, N)) for c in range(n)]
    rd = wr = 0
    for s in range(n - 1):
        for r in range(n):
            L = length[(r - s) % n]
            rd += (e if s == 0 else 4) * L + e * L
            wr += (e if s == n - 2 else 4) * L
    for s in range(n - 1):
        for r in range(n):
            L = length[(r + 1 - s) % n]
            rd += e * L
            wr += e * L
    return rd, wr


@pytest.mark.parametrize("n", [2, 3, 8, 16])
@pytest.mark.parametrize("N,e", [(1, 2), (1000, 2), (4099, 4), (1 << 20, 2), (77, 4)])
def test_ring_hbm_bytes_brute_force(n, N, e):
    assert model.hbm_ring(n, N, e) == _brute_ring_bytes(n, N, e)


def test_hbm_closed_forms_small_cases():
    assert model.hbm_one_shot(8, 10, 2) == (160, 160)
    assert model.hbm_two_shot(8, 10, 2) == (180, 160)
    assert sum(model.hbm_two_shot(8, 10, 2)) == (2 * 8 + 1) * 20
    assert model.hbm_ll_reduce(8, 3) == (192, 192)
    assert model.hbm_ll128_pack(31) == (124, 256)
    assert math.isclose(sum(model.hbm_ll_pack(1000)), 3 * 4000)
