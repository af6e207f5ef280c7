"""GPU parity of longer prefills (2048, 2858 and 4096 tokens) on the prefill
projections, through the planner's choice (the tensor arm): every token on a
sample of output features against the fp64 oracle, plus a ragged token count
whose last token tile is partial, and square and wide shapes whose default
plan takes narrower token tiles."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bf16_activation_quantized_gb300 as w4
import oracle
from bf16_activation_quantized_gb300 import synthetic as syn

from gpu_util import bf16_to_f64, dev_u16_as_bf16, dev_u8, poisoned_gemm, require_gpu
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("M,N,K", syn.WORKLOADS["prefill_long"] + [(2857, 2560, 9728)])
def test_prefill_long_sampled(M, N, K):
    assert w4.plan(M, N, K)["arm"] == "tensor"
    inp = syn.make_gemm_inputs(M, N, K, seed=M % 7)
    y = poisoned_gemm(dev_u16_as_bf16(inp.x), w4.pack(dev_u8(inp.w_canon)), dev_u16_as_bf16(inp.scales))
    torch.cuda.synchronize()
    rng = np.random.default_rng(M + N)
    cols = np.unique(np.r_[rng.choice(N, 48, replace=False), 0, 127, 128, N - 1])
    ref = oracle.gemm(inp.x, inp.w_canon[cols], inp.scales[cols], M, len(cols), K)
    assert_close(bf16_to_f64(y)[:, cols], ref, what=f"{M}x{N}x{K}")


# Shapes whose default plan takes plain or separate-epilogue tiles of 160 or
# 192 tokens with several tiles per CTA (4096- to 19456-wide weights).
@pytest.mark.parametrize("M,N,K", [(1024, 19456, 2560), (2048, 4096, 4096), (1024, 7168, 8192)])
def test_narrow_tile_plans_sampled(M, N, K):
    plan = w4.plan(M, N, K)
    assert plan["arm"] == "tensor" and plan["tile_tokens"] in (160, 192)
    inp = syn.make_gemm_inputs(M, N, K, seed=N % 11)
    y = poisoned_gemm(dev_u16_as_bf16(inp.x), w4.pack(dev_u8(inp.w_canon)), dev_u16_as_bf16(inp.scales))
    torch.cuda.synchronize()
    rng = np.random.default_rng(M + K)
    cols = np.unique(np.r_[rng.choice(N, 48, replace=False), 0, 127, 128, N - 1])
    ref = oracle.gemm(inp.x, inp.w_canon[cols], inp.scales[cols], M, len(cols), K)
    assert_close(bf16_to_f64(y)[:, cols], ref, what=f"{M}x{N}x{K}")
