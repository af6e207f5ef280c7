"""Work counts for the W4A16 skinny GEMM, used to turn times into rates.

FLOPs are the dense product's multiply-adds, 2 per weight per row of X:
``2 * rows * N * K``.  Dequantisation work is not counted.  This is the
convention of the throughput tables on "Add Triton BF16xINT4 rowwise GEMM for
ROCm gfx942/gfx950" ("Performance"), where time x TFLOP/s reproduces
2 * (total rows) * N * K for the grouped and batched ops.

Algorithmic bytes are what one call must move at least once between HBM and
the SMs: packed W (N*K/2), bf16 scales (N*K/G*2), X (2*rows*K) and Y
(2*rows*N).  A split-K workspace, re-reads and padding are not counted, so
this is stricter than the pages' GB/s figures, which also count workspace
traffic and per-group metadata.
"""
from __future__ import annotations


def flops(rows: int, N: int, K: int) -> int:
    return 2 * int(rows) * int(N) * int(K)


def weight_bytes(N: int, K: int, G: int = 128) -> int:
    return int(N) * int(K) // 2 + int(N) * (int(K) // int(G)) * 2


def algorithmic_bytes(rows: int, N: int, K: int, G: int = 128) -> int:
    return weight_bytes(N, K, G) + 2 * int(rows) * int(K) + 2 * int(rows) * int(N)


def grouped_algorithmic_bytes(num_groups: int, M_total: int, N: int, K: int, G: int = 128) -> int:
    return (int(num_groups) * weight_bytes(N, K, G) + 2 * int(M_total) * int(K)
            + 2 * int(M_total) * int(N))


def roofline_seconds(flop: float, nbytes: float, peak_flops: float, peak_bytes_per_s: float) -> float:
    """The slower of the byte time and the FLOP time."""
    return max(nbytes / peak_bytes_per_s, flop / peak_flops)
