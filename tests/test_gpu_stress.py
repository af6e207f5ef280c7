"""GPU: repeated calls of every decode workload shape are bit-identical.

A self-checking stress run.  Each shape runs 200 calls in one process: 100
with Y and the split-K workspace refilled with NaN before every call (an
output a kernel skipped would show up), and 100 launched back to back without
synchronisation, each into its own output buffer with one shared workspace,
with and without resident weights (programmatic dependent launch lets each
call start while the previous one still runs).  Every result must equal the
first bit for bit, the first must match the oracle, and the device error word
(checked after every GPU test) must stay 0."""
from __future__ import annotations

import pytest
import torch

import bf16_activation_quantized_gb300 as w4
import oracle
from bf16_activation_quantized_gb300 import synthetic as syn

from gpu_util import DeviceProblem, bf16_to_f64, poisoned_gemm, require_gpu
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


SHAPES = ([(1, 8192, 8192), (1, 17408, 5120)]
          + [(m, n, k) for (n, k) in ((19456, 2560), (2560, 9728)) for m in (1, 8, 16)])


@pytest.mark.parametrize("M,N,K", SHAPES)
def test_two_hundred_calls_are_bit_identical(M, N, K):
    p = DeviceProblem(syn.make_gemm_inputs(M, N, K, seed=3))
    first = poisoned_gemm(p.x, p.w_packed, p.scales)
    torch.cuda.synchronize()
    i = p.inp
    assert_close(bf16_to_f64(first), oracle.gemm(i.x, i.w_canon, i.scales, M, N, K),
                 what=f"stress {M}x{N}x{K}")
    ref = first.view(torch.int16)
    plan = w4.plan(M, N, K)
    ws = torch.empty(max(plan["workspace_bytes"], 16), dtype=torch.uint8, device="cuda")
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    bad = []
    for it in range(100):
        out.fill_(float("nan"))
        ws.view(torch.float32)[: ws.numel() // 4].fill_(float("nan"))
        w4.gemm(p.x, p.w_packed, p.scales, out=out, workspace=ws)
        if not torch.equal(out.view(torch.int16), ref):
            bad.append(("refilled", it))
    for resident in (False, True):
        outs = [torch.empty((M, N), dtype=torch.bfloat16, device="cuda") for _ in range(50)]
        for o in outs:
            w4.gemm(p.x, p.w_packed, p.scales, out=o, workspace=ws, resident_weights=resident)
        torch.cuda.synchronize()
        bad += [("back to back", resident, j) for j, o in enumerate(outs)
                if not torch.equal(o.view(torch.int16), ref)]
    assert not bad, f"{len(bad)} of 200 calls differ from the first ({plan}): {bad[:5]}"
