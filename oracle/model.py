"""Closed forms the pages state -- TEST INFRASTRUCTURE ONLY (part of the oracle).

Sources:
- handbook chapter "集合通信：NCCL 的算法、协议与推理框架的定制 all-reduce":
  §算法 (per-rank traffic of ring, one-shot and two-shot; the alpha-beta model
  of ring / tree / one-shot / two-shot / NVLS and its printed table),
  §读懂 nccl-tests (algbw = S / t; busbw = algbw x 2(n-1)/n for all-reduce,
  (n-1)/n for all-gather and reduce-scatter, 1 for broadcast),
  §练习 exercise 1 (busbw -> time) and exercise 2 (one-shot / two-shot
  crossover S* = 2 alpha beta / ((n-1)(1 - 2/n))).
- handbook chapter "多 GPU 与 NCCL", §ring all-reduce (each rank sends
  2(p-1) S/p bytes over 2(p-1) steps).

The last block gives the HBM bytes each emulated step must move on one GPU
(n rank buffers of S = N e bytes in one HBM), derived from the same steps:
one-shot reads n S and writes n S; two-shot adds the reduced chunk's write
and re-read; the ring keeps fp32 partials between hops.
"""

from __future__ import annotations

import math


# --- per-rank link traffic and step counts --------------------------------

def link_bytes_one_shot(n: int, S: float) -> float:
    """Each rank reads the full buffer of each of the other n-1 ranks."""
    return (n - 1) * S


def link_bytes_two_shot(n: int, S: float) -> float:
    """Reduce-scatter reads (n-1) S/n, all-gather reads (n-1) S/n."""
    return 2 * (n - 1) / n * S


def link_bytes_ring(n: int, S: float) -> float:
    """Each rank sends one S/n chunk in each of 2(n-1) steps."""
    return 2 * (n - 1) * S / n


def steps_one_shot(n: int) -> int:
    return 1


def steps_two_shot(n: int) -> int:
    return 2


def steps_ring(n: int) -> int:
    return 2 * (n - 1)


# --- nccl-tests bandwidths -------------------------------------------------

BUS_FACTOR = {
    "all_reduce": lambda n: 2 * (n - 1) / n,
    "all_gather": lambda n: (n - 1) / n,
    "reduce_scatter": lambda n: (n - 1) / n,
    "broadcast": lambda n: 1.0,
}


def algbw(S: float, t: float) -> float:
    return S / t


def busbw(algbw_value: float, n: int, op: str = "all_reduce") -> float:
    return algbw_value * BUS_FACTOR[op](n)


def time_from_busbw(S: float, busbw_value: float, n: int, op: str = "all_reduce") -> float:
    """Invert busbw = (S / t) x factor for the time of one operation."""
    return S * BUS_FACTOR[op](n) / busbw_value


# --- the alpha-beta model ----------------------------------------------------

def alpha_beta(n: int, beta: float, alpha: float) -> dict:
    """t(S) of one all-reduce of S bytes per rank, per algorithm."""
    return {
        "ring": lambda S: 2 * (n - 1) * alpha + 2 * (n - 1) / n * S / beta,
        "tree": lambda S: 2 * math.log2(n) * alpha + 2 * S / beta,
        "one-shot": lambda S: 2 * alpha + (n - 1) * S / beta,
        "two-shot": lambda S: 4 * alpha + 2 * (n - 1) / n * S / beta,
        "NVLS": lambda S: 2 * alpha + S / beta,
    }


def fastest_without_nvls(times: dict) -> str:
    return min((k for k in times if k != "NVLS"), key=times.get)


def one_two_shot_crossover(n: int, beta: float, alpha: float) -> float | None:
    """S where 2a + (n-1)S/b = 4a + 2(n-1)/n S/b; none at n = 2 (same traffic)."""
    denom = (n - 1) * (1 - 2 / n)
    return None if denom == 0 else 2 * alpha * beta / denom


# --- HBM bytes of the single-GPU emulation ---------------------------------

def hbm_one_shot(n: int, N: int, e: int) -> tuple[int, int]:
    """(read, write): read n S, write n S."""
    return n * N * e, n * N * e


def hbm_two_shot(n: int, N: int, e: int) -> tuple[int, int]:
    """Reduce-scatter reads n S and writes S; all-gather reads S, writes (n-1) S."""
    return (n + 1) * N * e, n * N * e


def hbm_ring(n: int, N: int, e: int) -> tuple[int, int]:
    """fp32 partials between hops.  In every step the n transfers cover each
    chunk once, so the per-step bytes depend on N only.  Reduce-scatter:
    step 0 reads two payloads, later steps an fp32 partial and a payload;
    steps before the last write an fp32 partial, the last writes the payload.
    All-gather: n-1 steps of one payload read and one payload write."""
    if n == 2:
        return 2 * e * N + e * N, e * N + e * N
    read = 2 * e * N + (n - 2) * (4 + e) * N + (n - 1) * e * N
    write = (n - 2) * 4 * N + e * N + (n - 1) * e * N
    return read, write


def hbm_ll_pack(count: int) -> tuple[int, int]:
    return 4 * count, 8 * count


def hbm_ll_unpack(count: int) -> tuple[int, int]:
    return 8 * count, 4 * count


def hbm_ll_reduce(n: int, count: int) -> tuple[int, int]:
    return n * 8 * count, n * 8 * count


def ll128_lines(count: int) -> int:
    return (count + 29) // 30


def hbm_ll128_pack(count: int) -> tuple[int, int]:
    return 4 * count, 128 * ll128_lines(count)


def hbm_ll128_unpack(count: int) -> tuple[int, int]:
    return 128 * ll128_lines(count), 4 * count


def hbm_ll128_reduce(n: int, count: int) -> tuple[int, int]:
    return n * 128 * ll128_lines(count), n * 128 * ll128_lines(count)


def hbm_ring_rounded(n: int, N: int, e: int) -> tuple[int, int]:
    """Partials in the payload type: every reduce-scatter step reads two
    payloads and writes one; every all-gather step reads one and writes one."""
    return 2 * e * N * (n - 1) + e * N * (n - 1), e * N * (n - 1) + e * N * (n - 1)


def hbm_tree(n: int, N: int, e: int) -> tuple[int, int]:
    """log2(n) levels; each reads and writes every rank's buffer once."""
    levels = n.bit_length() - 1
    return levels * n * e * N, levels * n * e * N
