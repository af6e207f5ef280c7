"""GPU: the failure path of the decode arm, made to run without faulting the GPU.

W4A16_FLAG_TEST_STALL launches the K-slice decode kernel with no weight copies
and a 1 ms wait limit, so every bounded wait runs out.  The kernel must then
end on its own, record W4A16_ERROR_WAIT_TIMEOUT in the device error word
(read through the C ABI's w4a16_read_error_word), and leave NaN -- never a
plausible stale value -- in every output it owns, both when it writes Y itself
and when its NaN partial sums pass through the split-K reduce.  The context
stays usable: a normal call right after matches the oracle."""
from __future__ import annotations

import ctypes

import pytest
import torch

import bf16_activation_quantized_gb300 as w4
import oracle
from bf16_activation_quantized_gb300 import _lib
from bf16_activation_quantized_gb300 import synthetic as syn

from gpu_util import DeviceProblem, bf16_to_f64, poisoned_gemm, require_gpu
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


@pytest.mark.parametrize("M,N,K,split", [(1, 2048, 2048, 1), (4, 2048, 4096, 4), (16, 1024, 2048, 2),
                                         (3, 300, 1024, 8)])
def test_stalled_decode_kernel_reports_and_poisons(M, N, K, split):
    p = DeviceProblem(syn.make_gemm_inputs(M, N, K, seed=5))
    plan = w4.plan(M, N, K, arm="decode", split_k=split, decode_kernel="k_slices")
    assert plan["split_k"] == split
    ws = torch.zeros(max(plan["workspace_bytes"], 16), dtype=torch.uint8, device="cuda")
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    assert w4.read_error_word(clear=True) == 0
    w4.gemm(p.x, p.w_packed, p.scales, out=y, workspace=ws, arm="decode", split_k=split,
            test_stall=True)
    word = w4.read_error_word(clear=True)
    assert word & w4.ERROR_WAIT_TIMEOUT, f"error word {word:#x}"
    assert bool(torch.isnan(y.float()).all()), "an incomplete output is not NaN"
    # The context is still usable and the next call is correct.
    y2 = poisoned_gemm(p.x, p.w_packed, p.scales)
    torch.cuda.synchronize()
    i = p.inp
    assert_close(bf16_to_f64(y2), oracle.gemm(i.x, i.w_canon, i.scales, M, N, K),
                 what=f"call after a stall {M}x{N}x{K}")


def test_read_error_word_through_the_c_abi():
    L = _lib.lib()
    v = ctypes.c_int(-1)
    assert L.w4a16_read_error_word(ctypes.byref(v), 1) == 0
    assert v.value == 0
    p = DeviceProblem(syn.make_gemm_inputs(1, 256, 512, seed=1))
    w4.gemm(p.x, p.w_packed, p.scales, arm="decode", decode_kernel="k_slices", test_stall=True,
            workspace=torch.zeros(1 << 16, dtype=torch.uint8, device="cuda"))
    # Without clearing, the bit stays; clearing returns it once more, then 0.
    assert L.w4a16_read_error_word(ctypes.byref(v), 0) == 0 and v.value == w4.ERROR_WAIT_TIMEOUT
    assert L.w4a16_read_error_word(ctypes.byref(v), 1) == 0 and v.value == w4.ERROR_WAIT_TIMEOUT
    assert L.w4a16_read_error_word(ctypes.byref(v), 1) == 0 and v.value == 0


@pytest.mark.parametrize("kw", [dict(arm="tensor"), dict(arm="decode", decode_kernel="whole_k")])
def test_stall_mode_exists_only_for_the_k_slice_kernel(kw):
    p = DeviceProblem(syn.make_gemm_inputs(4, 256, 512, seed=2))
    with pytest.raises(w4.W4A16Error) as e:
        w4.gemm(p.x, p.w_packed, p.scales, test_stall=True, **kw)
    assert e.value.status == 2          # W4A16_ERR_UNSUPPORTED, nothing launched
    assert w4.read_error_word(clear=True) == 0
