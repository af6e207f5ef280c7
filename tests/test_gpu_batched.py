"""GPU parity of the batched product (one launch over B independent products of
one shape) against the fp64 oracle per entry, and against separate calls."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bf16_activation_quantized_gb300 as w4
import oracle
from bf16_activation_quantized_gb300 import synthetic as syn

from gpu_util import bf16_to_f64, bf16_to_u16, dev_u16_as_bf16, dev_u8, poisoned_gemm_batched, require_gpu
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


class Batch:
    """B seeded problems of one shape, stacked on the GPU as the batched op takes them."""

    def __init__(self, B, M, N, K, seed=0):
        self.inps = [syn.make_gemm_inputs(M, N, K, seed=seed + b) for b in range(B)]
        self.B, self.M, self.N, self.K = B, M, N, K
        self.x = torch.stack([dev_u16_as_bf16(i.x) for i in self.inps])
        self.scales = torch.stack([dev_u16_as_bf16(i.scales) for i in self.inps])
        self.w = torch.stack([w4.pack(dev_u8(i.w_canon)) for i in self.inps])

    def reference(self, b, cols=None):
        i = self.inps[b]
        if cols is None:
            return oracle.gemm(i.x, i.w_canon, i.scales, self.M, self.N, self.K)
        return oracle.gemm(i.x, i.w_canon[cols], i.scales[cols], self.M, len(cols), self.K)

    def run(self, **kw):
        y = poisoned_gemm_batched(self.x, self.w, self.scales, **kw)
        torch.cuda.synchronize()
        return y


SHAPES = [(3, 1, 2048, 1024), (2, 8, 300, 640), (4, 16, 2560, 2560), (2, 5, 129, 384),
          (2, 128, 2048, 5120), (3, 40, 300, 640), (2, 300, 1024, 1024), (2, 1, 8192, 8192)]


@pytest.mark.parametrize("B,M,N,K", SHAPES)
def test_batched_matches_the_oracle_per_entry(B, M, N, K):
    bt = Batch(B, M, N, K)
    y = bt.run()
    plan = w4.plan_batched(B, M, N, K)
    for b in range(B):
        assert_close(bf16_to_f64(y[b]), bt.reference(b), what=f"entry {b} of {B}x{M}x{N}x{K} {plan}")


@pytest.mark.parametrize("B,M,N,K,opts", [
    (3, 1, 2048, 1024, dict(arm="decode", split_k=4, decode_kernel="k_slices")),
    (2, 16, 2560, 2560, dict(arm="decode", split_k=5, decode_kernel="k_slices")),
    (2, 8, 300, 640, dict(arm="decode", split_k=1, decode_kernel="k_slices")),
    (2, 128, 2048, 5120, dict(arm="tensor", tile_tokens=128, split_k=1)),
    (3, 40, 300, 640, dict(arm="tensor", tile_tokens=32, split_k=5)),
    (2, 300, 1024, 1024, dict(arm="tensor", tile_tokens=96, split_k=2)),
])
def test_batched_equals_separate_calls_bit_for_bit(B, M, N, K, opts):
    # With the same slices and tiles every entry is computed exactly as on its own.
    bt = Batch(B, M, N, K, seed=7)
    y = bf16_to_u16(bt.run(**opts))
    for b in range(B):
        one = w4.gemm(bt.x[b], bt.w[b], bt.scales[b], **opts)
        torch.cuda.synchronize()
        assert np.array_equal(y[b], bf16_to_u16(one))


def test_batched_whole_k_kernel():
    bt = Batch(3, 1, 2048, 2048, seed=11)
    y = bt.run(arm="decode", decode_kernel="whole_k")
    assert w4.plan_batched(3, 1, 2048, 2048, arm="decode", decode_kernel="whole_k")["whole_k"]
    for b in range(3):
        assert_close(bf16_to_f64(y[b]), bt.reference(b), what=f"whole-K entry {b}")


def test_batch_of_one_is_the_plain_call():
    bt = Batch(1, 4, 1024, 2048, seed=3)
    y = bf16_to_u16(bt.run())
    one = w4.gemm(bt.x[0], bt.w[0], bt.scales[0])
    torch.cuda.synchronize()
    assert np.array_equal(y[0], bf16_to_u16(one))


def test_batched_in_a_graph_replays_exactly():
    bt = Batch(2, 16, 2560, 2560, seed=5)
    eager = bf16_to_u16(bt.run())
    out = torch.empty((2, 16, 2560), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        w4.gemm_batched(bt.x, bt.w, bt.scales, out=out)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        w4.gemm_batched(bt.x, bt.w, bt.scales, out=out, resident_weights=True)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bf16_to_u16(out), eager)


def test_batched_workload_sampled():
    # Two 2048x7168x8192 products through the planner's choice (160-token
    # tensor tiles, several per CTA): every token on a sample of features.
    B, M, N, K = 2, 2048, 7168, 8192
    assert w4.plan_batched(B, M, N, K)["arm"] == "tensor"
    bt = Batch(B, M, N, K, seed=21)
    y = bt.run()
    rng = np.random.default_rng(5)
    cols = np.unique(np.r_[rng.choice(N, 40, replace=False), 0, 127, 128, N - 1])
    for b in range(B):
        assert_close(bf16_to_f64(y[b])[:, cols], bt.reference(b, cols), what=f"entry {b} of {B}x{M}x{N}x{K}")
