"""Seeded synthetic inputs for the W4A16 skinny GEMM (tests and benchmark).

This module only draws random data and writes it in the operand formats; it
holds none of the GEMM's arithmetic, so both the CUDA path's tests and the CPU
oracle can take their inputs from it without sharing method code.

Operand formats:
  * X: bf16 bit patterns, uint16 ``[M, K]``, row-major.
  * W: canonical int4 packing, uint8 ``[N, K/2]``: byte ``j`` of row ``n``
    holds the code for ``k = 2j`` in bits 0-3 and ``k = 2j+1`` in bits 4-7
    (the pairing of low nibble / even K on "Add Triton BF16xINT4 rowwise GEMM
    for ROCm gfx942/gfx950", "Implementation").
  * scales: bf16 bit patterns, uint16 ``[N, K/G]``.
  * M_sizes: int32 ``[num_groups]``.

Value recipe (one seed per call, NumPy PCG64, draws in this order): X from
N(0, 1); codes uniform integers in [0, 15]; scales uniform in [0.005, 0.02];
group sizes multinomial(M_total, uniform), redrawn while any group is empty.
fp32 draws become bf16 by round-to-nearest-even.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

GROUP = 128


def f32_to_bf16_bits(a) -> np.ndarray:
    """Round binary32 values to bf16 (nearest, ties to even); returns uint16.

    Inputs are finite by construction here, so no NaN handling is needed.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return ((u + bias) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def pack_codes(codes: np.ndarray) -> np.ndarray:
    """[N, K] codes in [0, 15] -> canonical packed uint8 [N, K/2]."""
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    if c.shape[-1] % 2:
        raise ValueError("K must be even to pack two codes per byte")
    return (c[..., 0::2] | (c[..., 1::2] << 4)).astype(np.uint8)


@dataclass
class GemmInputs:
    x: np.ndarray        # uint16 [M, K] bf16 bits
    w_canon: np.ndarray  # uint8  [N, K/2]
    scales: np.ndarray   # uint16 [N, K/G] bf16 bits
    M: int
    N: int
    K: int
    G: int = GROUP


@dataclass
class GroupedInputs:
    x: np.ndarray        # uint16 [M_total, K]
    w_canon: np.ndarray  # uint8  [num_groups, N, K/2]
    scales: np.ndarray   # uint16 [num_groups, N, K/G]
    m_sizes: np.ndarray  # int32  [num_groups]
    num_groups: int
    M_total: int
    N: int
    K: int
    G: int = GROUP


def _draw_x(rng, M, K):
    return f32_to_bf16_bits(rng.standard_normal((M, K), dtype=np.float32))


def _draw_codes(rng, shape):
    return rng.integers(0, 16, size=shape, dtype=np.uint8)


def _draw_scales(rng, shape):
    return f32_to_bf16_bits(rng.uniform(0.005, 0.02, size=shape).astype(np.float32))


def make_gemm_inputs(M: int, N: int, K: int, G: int = GROUP, seed: int = 0) -> GemmInputs:
    if K % G:
        raise ValueError("K must be a multiple of the group size")
    rng = np.random.default_rng(seed)
    x = _draw_x(rng, M, K)
    w = pack_codes(_draw_codes(rng, (N, K)))
    s = _draw_scales(rng, (N, K // G))
    return GemmInputs(x=x, w_canon=w, scales=s, M=M, N=N, K=K, G=G)


def make_zeros(N: int, K: int, G: int = GROUP, seed: int = 0) -> np.ndarray:
    """Zero points for the asymmetric variant: uint8 [N, K/G], uniform integers
    0..15, from a generator of their own (seed + 7919), so the other inputs of
    a seed are unchanged."""
    rng = np.random.default_rng(seed + 7919)
    return rng.integers(0, 16, size=(N, K // G), dtype=np.uint8)


def draw_group_sizes(rng, num_groups: int, M_total: int) -> np.ndarray:
    while True:
        sizes = rng.multinomial(M_total, [1.0 / num_groups] * num_groups)
        if M_total < num_groups or np.all(sizes > 0):
            return sizes.astype(np.int32)


def make_grouped_inputs(num_groups: int, M_total: int, N: int, K: int, G: int = GROUP,
                        seed: int = 0, m_sizes=None) -> GroupedInputs:
    if K % G:
        raise ValueError("K must be a multiple of the group size")
    rng = np.random.default_rng(seed)
    x = _draw_x(rng, M_total, K)
    w = pack_codes(_draw_codes(rng, (num_groups, N, K)))
    s = _draw_scales(rng, (num_groups, N, K // G))
    if m_sizes is None:
        m_sizes = draw_group_sizes(rng, num_groups, M_total)
    return GroupedInputs(x=x, w_canon=w, scales=s, m_sizes=np.asarray(m_sizes, np.int32),
                         num_groups=num_groups, M_total=M_total, N=N, K=K, G=G)


# Named workloads and their sizes.  The group size is 128 throughout.
WORKLOADS = {
    "tiny": [(4, 256, 512)],
    "decode_gemv": [(1, 8192, 8192), (1, 17408, 5120)],
    "decode_sweep_gate_up": [(m, 19456, 2560) for m in (1, 8, 16, 32, 64, 128)],
    "decode_sweep_down": [(m, 2560, 9728) for m in (1, 8, 16, 32, 64, 128)],
    "prefill": [(1322, 19456, 2560), (1322, 2560, 9728)],
    # Longer prefills on the same projections: the end-to-end prefill of the
    # gfx1151 page runs about 2858 tokens, the rowwise-GEMM page's prefill rows
    # use 2048 and 4096.
    "prefill_long": [(m, n, k) for m in (2048, 2858, 4096) for (n, k) in ((19456, 2560), (2560, 9728))],
}
GROUPED_WORKLOAD = dict(num_groups=8, M_total=4096, N=2048, K=4096)
