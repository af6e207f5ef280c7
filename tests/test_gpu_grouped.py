"""GPU parity of the grouped product (one launch, device-side M_sizes) against
the oracle, including empty groups and the clamping rules of the status word."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bf16_activation_quantized_gb300 as w4
import oracle
from bf16_activation_quantized_gb300 import synthetic as syn

from gpu_util import bf16_to_f64, dev_u16_as_bf16, dev_u8, require_gpu
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def device_grouped(g):
    x = dev_u16_as_bf16(g.x)
    s = dev_u16_as_bf16(g.scales)
    wp = torch.cat([w4.pack(dev_u8(g.w_canon[i])) for i in range(g.num_groups)])
    ms = torch.from_numpy(np.asarray(g.m_sizes, dtype=np.int32).copy()).cuda()
    return x, wp, s, ms


def run_grouped(g, fill=None):
    x, wp, s, ms = device_grouped(g)
    out = torch.full((g.M_total, g.N), float("nan") if fill is None else fill,
                     dtype=torch.bfloat16, device="cuda")
    y, status = w4.gemm_grouped(x, wp, s, ms, out=out)
    torch.cuda.synchronize()
    return bf16_to_f64(y), int(status[0].item())


@pytest.mark.parametrize("G,M_total,N,K,sizes", [
    (3, 100, 256, 512, [40, 0, 60]),
    (4, 77, 300, 640, [1, 33, 3, 40]),
    (1, 50, 256, 256, [50]),
    (5, 500, 128, 384, None),
])
def test_grouped_small(G, M_total, N, K, sizes):
    g = syn.make_grouped_inputs(G, M_total, N, K, seed=G + M_total, m_sizes=sizes)
    y, status = run_grouped(g)
    assert status == 0
    ref = oracle.gemm_grouped(g.x, g.w_canon, g.scales, g.m_sizes, M_total, N, K)
    assert_close(y, ref, what=f"grouped G{G}")


def test_grouped_workload_sampled():
    spec = syn.GROUPED_WORKLOAD
    g = syn.make_grouped_inputs(spec["num_groups"], spec["M_total"], spec["N"], spec["K"], seed=0)
    y, status = run_grouped(g)
    assert status == 0
    starts = np.concatenate([[0], np.cumsum(g.m_sizes)[:-1]])
    rng = np.random.default_rng(1)
    cols = np.unique(np.concatenate([rng.choice(spec["N"], 96, replace=False), [0, spec["N"] - 1]]))
    for i in range(g.num_groups):
        lo, hi = int(starts[i]), int(starts[i] + g.m_sizes[i])
        ref = oracle.gemm(g.x[lo:hi], g.w_canon[i][cols], g.scales[i][cols], hi - lo, len(cols),
                          spec["K"])
        assert_close(y[lo:hi][:, cols], ref, what=f"grouped workload group {i}")
    assert np.all(np.isfinite(y))


def test_grouped_status_and_clamping():
    # negative size -> treated as empty (bit 0); sum past M_total -> cut (bit 1)
    g = syn.make_grouped_inputs(3, 60, 256, 256, seed=3, m_sizes=[20, -5, 70])
    y, status = run_grouped(g)
    assert status == 3
    ref = oracle.gemm_grouped(g.x, g.w_canon, g.scales, g.m_sizes, 60, 256, 256)
    assert_close(y, ref, what="clamped")
    # sizes summing below M_total: trailing rows are left untouched
    h = syn.make_grouped_inputs(2, 64, 256, 256, seed=4, m_sizes=[10, 20])
    yh, st = run_grouped(h, fill=7.0)
    assert st == 0
    assert np.all(yh[30:] == 7.0)
    refh = oracle.gemm_grouped(h.x, h.w_canon, h.scales, h.m_sizes, 64, 256, 256)
    assert_close(yh[:30], refh[:30], what="short sizes")


def test_grouped_equals_plain_per_group():
    g = syn.make_grouped_inputs(3, 96, 256, 512, seed=5, m_sizes=[32, 32, 32])
    y, _ = run_grouped(g)
    x, wp, s, _ = device_grouped(g)
    nb = w4.packed_weight_bytes(256, 512)
    for i in range(3):
        # same tile (32 tokens) and no K split: the same MMA sequence per output
        yi = w4.gemm(x[32 * i:32 * (i + 1)], wp[i * nb:(i + 1) * nb], s[i], arm="tensor",
                     split_k=1, tile_tokens=32)
        torch.cuda.synchronize()
        assert np.array_equal(bf16_to_f64(yi), y[32 * i:32 * (i + 1)])


def test_grouped_graph_replay():
    g = syn.make_grouped_inputs(4, 200, 256, 512, seed=6)
    x, wp, s, ms = device_grouped(g)
    out = torch.empty((200, 256), dtype=torch.bfloat16, device="cuda")
    status = torch.zeros(4, dtype=torch.int32, device="cuda")
    w4.gemm_grouped(x, wp, s, ms, out=out, status=status)
    torch.cuda.synchronize()
    eager = bf16_to_f64(out).copy()
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.graph(gr):
        w4.gemm_grouped(x, wp, s, ms, out=out, status=status)
    out.zero_()
    gr.replay()
    torch.cuda.synchronize()
    assert np.array_equal(bf16_to_f64(out), eager)
    # new sizes in device memory are picked up by the replay without host sync
    ms.copy_(torch.tensor([50, 50, 50, 50], dtype=torch.int32))
    gr.replay()
    torch.cuda.synchronize()
    ref = oracle.gemm_grouped(g.x, g.w_canon, g.scales, [50, 50, 50, 50], 200, 256, 512)
    assert_close(bf16_to_f64(out), ref, what="graph replay with new sizes")
