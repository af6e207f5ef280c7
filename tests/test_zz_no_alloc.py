"""GPU: w4a16_gemm_noalloc, the entry point for callers that cannot allocate
device memory (a plugin handed only inputs and outputs, or code under CUDA
graph capture), matches w4a16_gemm through the C ABI on two calls in a row.

This file is collected last so that a run stopping at its first failure has
already run every other test."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle

from bf16_activation_quantized_gb300 import _lib
from bf16_activation_quantized_gb300 import synthetic as syn

from gpu_util import DeviceProblem, bf16_to_f64, require_gpu
from parity import assert_close

pytestmark = pytest.mark.gpu

SCRATCH_MAX = 4 << 20


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def _gemm_with_workspace(L, p, M, N, K, out):
    nb = ctypes.c_size_t(0)
    assert L.w4a16_workspace_bytes(M, N, K, 128, ctypes.byref(nb)) == 0
    ws = torch.empty(max(nb.value, 16), dtype=torch.uint8, device="cuda")
    st = L.w4a16_gemm(p.x.data_ptr(), p.w_packed.data_ptr(), p.scales.data_ptr(), out.data_ptr(),
                      M, N, K, 128, ws.data_ptr(), ws.numel(), None)
    assert st == 0
    torch.cuda.synchronize()
    return nb.value


# Shapes whose split-K scratch stays within 4 MiB for any split the planner can
# choose (at most K/128 slices of M x N fp32).
@pytest.mark.parametrize("M,N,K", [(1, 8192, 8192), (8, 2048, 4096), (4, 256, 512)])
def test_noalloc_matches_gemm_twice(M, N, K):
    L = _lib.lib()
    p = DeviceProblem(syn.make_gemm_inputs(M, N, K, seed=11))
    ref = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    need = _gemm_with_workspace(L, p, M, N, K, ref)
    assert need <= SCRATCH_MAX
    i = p.inp
    yref = oracle.gemm(i.x, i.w_canon, i.scales, M, N, K)
    for _ in range(2):
        out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = L.w4a16_gemm_noalloc(p.x.data_ptr(), p.w_packed.data_ptr(), p.scales.data_ptr(),
                                  out.data_ptr(), M, N, K, 128, None)
        assert st == 0
        torch.cuda.synchronize()
        # Same plan, same kernels: the same bits as w4a16_gemm, and the oracle's
        # values within the GEMM tolerance.
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
        assert_close(bf16_to_f64(out), yref, what=f"noalloc M{M} N{N} K{K}")


def test_noalloc_rejects_shapes_beyond_its_scratch():
    L = _lib.lib()
    nb = ctypes.c_size_t(0)
    # The first decode or prefill workload shape whose plan needs more split-K
    # scratch than the array holds.
    shape = None
    for M, N, K in ((16, 19456, 2560), (8, 19456, 2560), (16, 17408, 5120), (16, 8192, 8192),
                    (512, 7168, 8192), (16, 2560, 9728), (128, 2560, 9728), (16, 8192, 16384)):
        assert L.w4a16_workspace_bytes(M, N, K, 128, ctypes.byref(nb)) == 0
        if nb.value > SCRATCH_MAX:
            shape = (M, N, K)
            break
    assert shape is not None, "no candidate shape needs more than the scratch array"
    M, N, K = shape
    out = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros(N * K // 2, dtype=torch.uint8, device="cuda")
    s = torch.zeros((N, K // 128), dtype=torch.bfloat16, device="cuda")
    st = L.w4a16_gemm_noalloc(x.data_ptr(), w.data_ptr(), s.data_ptr(), out.data_ptr(),
                              M, N, K, 128, None)
    assert st == 3          # W4A16_ERR_WORKSPACE_TOO_SMALL: nothing launched
    torch.cuda.synchronize()
    assert not bool(out.any())
