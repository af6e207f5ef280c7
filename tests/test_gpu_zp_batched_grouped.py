"""GPU parity of the zero-point variant (dequant = scale * (code - z)) in the
batched and the grouped product against the fp64 oracle's gemm_zp, applied
entry by entry (batched) and group by group on each group's rows (grouped);
and z = 8 everywhere reproducing the symmetric launches bit for bit."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bf16_activation_quantized_gb300 as w4
import oracle
from bf16_activation_quantized_gb300 import synthetic as syn

from gpu_util import bf16_to_f64, dev_u16_as_bf16, dev_u8, poisoned_gemm_batched, require_gpu
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def stacked(inps, zs):
    x = torch.stack([dev_u16_as_bf16(i.x) for i in inps])
    s = torch.stack([dev_u16_as_bf16(i.scales) for i in inps])
    w = torch.stack([w4.pack(dev_u8(i.w_canon)) for i in inps])
    z = torch.stack([dev_u8(zz) for zz in zs])
    return x, w, s, z


@pytest.mark.parametrize("B,M,N,K,G,kw", [
    (3, 1, 2048, 1024, 128, {}),
    (2, 8, 300, 640, 64, {}),
    (2, 16, 2560, 2560, 128, {}),
    (3, 1, 2048, 1024, 32, dict(arm="decode", split_k=4, decode_kernel="k_slices")),
    (2, 128, 2048, 2560, 128, {}),
    (3, 40, 300, 640, 32, {}),
    (2, 96, 384, 1024, 64, dict(arm="tensor", split_k=2)),
])
def test_batched_zero_points_match_the_oracle_per_entry(B, M, N, K, G, kw):
    inps = [syn.make_gemm_inputs(M, N, K, G=G, seed=10 + b) for b in range(B)]
    zs = [syn.make_zeros(N, K, G, seed=10 + b) for b in range(B)]
    x, w, s, z = stacked(inps, zs)
    y = poisoned_gemm_batched(x, w, s, zeros=z, **kw)
    torch.cuda.synchronize()
    plan = w4.plan_batched(B, M, N, K, group_size=G, zero_points=True, **kw)
    for b in range(B):
        ref = oracle.gemm_zp(inps[b].x, inps[b].w_canon, inps[b].scales, zs[b], M, N, K, G=G)
        assert_close(bf16_to_f64(y[b]), ref, what=f"zp entry {b} of {B}x{M}x{N}x{K} G={G} {plan}")


@pytest.mark.parametrize("M,kw", [(1, dict(arm="decode", split_k=2, decode_kernel="k_slices")),
                                  (64, dict(arm="tensor"))])
def test_batched_zero_point_eight_matches_symmetric_bits(M, kw):
    B, N, K = 2, 384, 2048
    inps = [syn.make_gemm_inputs(M, N, K, seed=20 + b) for b in range(B)]
    x, w, s, z = stacked(inps, [np.full((N, K // 128), 8, np.uint8)] * B)
    a = w4.gemm_batched(x, w, s, **kw)
    b = w4.gemm_batched(x, w, s, zeros=z, **kw)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def grouped_zeros(g, seed):
    return np.stack([syn.make_zeros(g.N, g.K, g.G, seed=seed + i) for i in range(g.num_groups)])


def run_grouped(g, zeros):
    x = dev_u16_as_bf16(g.x)
    s = dev_u16_as_bf16(g.scales)
    wp = torch.cat([w4.pack(dev_u8(g.w_canon[i])) for i in range(g.num_groups)])
    ms = torch.from_numpy(np.asarray(g.m_sizes, dtype=np.int32).copy()).cuda()
    out = torch.full((g.M_total, g.N), float("nan"), dtype=torch.bfloat16, device="cuda")
    zd = None if zeros is None else dev_u8(zeros)
    y, status = w4.gemm_grouped(x, wp, s, ms, out=out, zeros=zd)
    torch.cuda.synchronize()
    return y, int(status[0].item())


@pytest.mark.parametrize("NG,M_total,N,K,G,sizes", [
    (3, 100, 256, 512, 128, [40, 0, 60]),
    (4, 77, 300, 640, 64, [1, 33, 3, 40]),
    (2, 300, 384, 1024, 32, None),
])
def test_grouped_zero_points_match_the_oracle_per_group(NG, M_total, N, K, G, sizes):
    g = syn.make_grouped_inputs(NG, M_total, N, K, G=G, seed=NG + M_total, m_sizes=sizes)
    zeros = grouped_zeros(g, 30)
    y, status = run_grouped(g, zeros)
    assert status == 0
    y = bf16_to_f64(y)
    starts = np.concatenate([[0], np.cumsum(g.m_sizes)[:-1]])
    for i in range(NG):
        lo, hi = int(starts[i]), int(starts[i] + g.m_sizes[i])
        if hi == lo:
            continue
        ref = oracle.gemm_zp(g.x[lo:hi], g.w_canon[i], g.scales[i], zeros[i], hi - lo, N, K, G=G)
        assert_close(y[lo:hi], ref, what=f"grouped zp group {i} of {NG}, G={G}")


def test_grouped_zero_points_workload_sampled():
    spec = syn.GROUPED_WORKLOAD
    g = syn.make_grouped_inputs(spec["num_groups"], spec["M_total"], spec["N"], spec["K"], seed=0)
    zeros = grouped_zeros(g, 40)
    y, status = run_grouped(g, zeros)
    assert status == 0
    y = bf16_to_f64(y)
    assert np.all(np.isfinite(y))
    starts = np.concatenate([[0], np.cumsum(g.m_sizes)[:-1]])
    rng = np.random.default_rng(3)
    cols = np.unique(np.concatenate([rng.choice(spec["N"], 64, replace=False), [0, spec["N"] - 1]]))
    for i in range(g.num_groups):
        lo, hi = int(starts[i]), int(starts[i] + g.m_sizes[i])
        ref = oracle.gemm_zp(g.x[lo:hi], g.w_canon[i][cols], g.scales[i][cols], zeros[i][cols],
                             hi - lo, len(cols), spec["K"])
        assert_close(y[lo:hi][:, cols], ref, what=f"grouped zp workload group {i}")


def test_grouped_zero_point_eight_matches_symmetric_bits():
    g = syn.make_grouped_inputs(3, 200, 384, 1024, seed=7, m_sizes=[70, 0, 130])
    a, sa = run_grouped(g, None)
    b, sb = run_grouped(g, np.full((3, 384, 1024 // 128), 8, np.uint8))
    assert sa == sb == 0
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
