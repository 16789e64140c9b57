"""FLOP and byte counts used to report throughput and roofline fractions.

FLOPs follow the usual attention convention: forward 4 B H N^2 d (two contractions of
2 N^2 d each per head), halved under the causal mask; backward 2.5 x forward.
Algorithmic bytes are the compulsory HBM traffic of each kernel: every input read once and
every output written once ("flash ~ 4Nd" of the CUDA lesson 06 page); re-reads of K/V by
several query blocks are served by L2 and are not counted.
"""
from __future__ import annotations


def fwd_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    f = 4.0 * B * H * N * N * d
    return 0.5 * f if causal else f


def bwd_flops(B: int, H: int, N: int, d: int, causal: bool) -> float:
    return 2.5 * fwd_flops(B, H, N, d, causal)


def fwd_bytes(B: int, H: int, N: int, d: int, elem: int) -> float:
    """Read Q, K, V; write O and the fp32 LSE."""
    return B * H * N * (4 * d * elem + 4)


def bwd_bytes(B: int, H: int, N: int, d: int, elem: int) -> float:
    """Read Q, K, V, O, dO, LSE; write dQ, dK, dV (Delta and the base-2 LSE round trip
    through the workspace: 2 x 4 bytes written and read once more per row)."""
    return B * H * N * (8 * d * elem + 4 + 16)


def preprocess_bytes(B: int, H: int, N: int, d: int, elem: int) -> float:
    """Backward preprocess: read O, dO and LSE; write Delta and the base-2 LSE."""
    return B * H * N * (2 * d * elem + 4 + 8)


def standard_attention_intermediate_bytes(N: int, elem: int = 2) -> float:
    """Standard attention writes S and P once and reads them once: 4 N^2 elements."""
    return 4.0 * N * N * elem


def lesson06_hbm_elements(N: int, d: int) -> tuple[float, float]:
    """(naive, flash) HBM element counts of the lesson-06 model: 4N^2 + 4Nd and 4Nd."""
    return 4.0 * N * N + 4.0 * N * d, 4.0 * N * d
