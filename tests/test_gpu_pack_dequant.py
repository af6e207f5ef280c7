"""GPU: the pack layout is bit-exact against its NumPy model, and the kernels'
register dequantisation is bit-exact against the oracle (fp32 and bf16)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bf16_activation_quantized_gb300 as w4
import oracle
from bf16_activation_quantized_gb300 import synthetic as syn

from gpu_util import DeviceProblem, bf16_to_u16, dev_u16_as_bf16, dev_u8, layout_model, require_gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("N,K", [(256, 512), (300, 640), (16, 128), (7, 256), (129, 128),
                                 (2560, 9728)])
def test_pack_layout_bit_exact(N, K):
    inp = syn.make_gemm_inputs(1, N, K, seed=N + K)
    wp = w4.pack(dev_u8(inp.w_canon))
    got = wp.cpu().numpy().view(np.uint32)
    assert np.array_equal(got, layout_model(inp.w_canon, N, K))


def _all_codes_problem(scale_bits: np.ndarray):
    """One row per scale pattern, every code 0..15 repeated along one group."""
    N, K = scale_bits.shape[0], 128
    codes = np.tile(np.arange(16, dtype=np.uint8), (N, K // 16))
    # shuffle the column order per row so each code visits every slot position
    rng = np.random.default_rng(0)
    for r in range(0, N, 97):
        rng.shuffle(codes[r])
    return syn.pack_codes(codes), scale_bits.reshape(N, 1).astype(np.uint16), N, K


def _scale_patterns(lo=None, hi=None, below=None):
    bits = np.arange(0x0080, 0x7F80, dtype=np.uint16)
    vals = (bits.astype(np.uint32) << 16).view(np.float32)
    keep = np.ones_like(vals, dtype=bool)
    if lo is not None:
        keep &= vals >= lo
    if hi is not None:
        keep &= vals <= hi
    if below is not None:
        keep &= vals < below
    return bits[keep]


@pytest.mark.parametrize("which", ["input_range", "all_normal"])
def test_dequant_fp32_bit_exact_exhaustive(which):
    sb = _scale_patterns(0.005, 0.02) if which == "input_range" else _scale_patterns(below=2.0 ** 120)
    w, s, N, K = _all_codes_problem(sb)
    got = w4.dequant_fp32(w4.pack(dev_u8(w)), dev_u16_as_bf16(s)).cpu().numpy()
    ref = oracle.dequant_f32(w, s, N, K)
    assert np.array_equal(got.view(np.uint32), ref.view(np.uint32))


@pytest.mark.parametrize("which", ["input_range", "all_normal"])
def test_dequant_bf16_bit_exact_exhaustive(which):
    sb = _scale_patterns(0.005, 0.02) if which == "input_range" else _scale_patterns(below=2.0 ** 120)
    w, s, N, K = _all_codes_problem(sb)
    got = bf16_to_u16(w4.dequant_bf16(w4.pack(dev_u8(w)), dev_u16_as_bf16(s)))
    ref = oracle.dequant_bf16(w, s, N, K)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("N,K,seed", [(300, 640, 1), (19456, 2560, 0)])
def test_dequant_random_positions(N, K, seed):
    inp = syn.make_gemm_inputs(1, N, K, seed=seed)
    p = DeviceProblem(inp)
    got32 = w4.dequant_fp32(p.w_packed, p.scales).cpu().numpy()
    got16 = bf16_to_u16(w4.dequant_bf16(p.w_packed, p.scales))
    rng = np.random.default_rng(seed)
    rows = rng.integers(0, N, 64)
    rows = np.concatenate([rows, [0, N - 1]])
    ref32 = oracle.dequant_f32(inp.w_canon[rows], inp.scales[rows], len(rows), K)
    ref16 = oracle.dequant_bf16(inp.w_canon[rows], inp.scales[rows], len(rows), K)
    assert np.array_equal(got32[rows].view(np.uint32), ref32.view(np.uint32))
    assert np.array_equal(got16[rows], ref16)
