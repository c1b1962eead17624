"""Measurement arithmetic (host only): latency floor, bandwidth, roofline.

Latency floor: "Every Microsecond Matters", Sec. VI, models the speed-of-light
latency of a small push AllReduce as 2 L2 round trips plus one remote store:
    L_SoL = 2 * L_L2_RTT + L_remote_store.
On one GPU, L_L2_RTT is the per-hop time of a dependent L2 pointer chase and
L_remote_store is half the round trip of a cross-SM store/poll ping-pong
(include/rra_probe.h).

Bandwidth: an AllReduce of M bytes per rank over N ranks must read every
input once and write every output once: 2 N M bytes of compulsory HBM
traffic (scratch is meant to stay in L2).  "busbw" is the nccl-tests style
figure M/t * 2(N-1)/N, reported for context only.
"""
from __future__ import annotations


def sol_floor_ns(l2_rtt_ns: float, store_poll_ns: float) -> float:
    return 2.0 * l2_rtt_ns + store_poll_ns


def algorithmic_bytes(nranks: int, bytes_per_rank: int) -> int:
    return 2 * nranks * bytes_per_rank


def hbm_gbs(nranks: int, bytes_per_rank: int, seconds: float) -> float:
    return algorithmic_bytes(nranks, bytes_per_rank) / seconds / 1e9


def busbw_gbs(nranks: int, bytes_per_rank: int, seconds: float) -> float:
    return bytes_per_rank / seconds * 2.0 * (nranks - 1) / nranks / 1e9


def median(xs):
    s = sorted(xs)
    n = len(s)
    if n == 0:
        return float("nan")
    return s[n // 2] if n % 2 else 0.5 * (s[n // 2 - 1] + s[n // 2])


def percentile(xs, q: float):
    s = sorted(xs)
    if not s:
        return float("nan")
    k = min(len(s) - 1, max(0, int(round(q / 100.0 * (len(s) - 1)))))
    return s[k]
