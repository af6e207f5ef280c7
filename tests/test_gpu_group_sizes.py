"""GPU parity at scale-group sizes 64 and 32 (G columns per scale; the gfx1151
page's "Benchmark results (per-GEMM)" use group_size=32): both arms, every
decode slice width the planner may pick, split-K, the grouped and batched
ops, and the bit-exact dequantisation probes.  Same bar as every GEMM test
(tests/parity.py) against the fp64 oracle called with the same G."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bf16_activation_quantized_gb300 as w4
import oracle
from bf16_activation_quantized_gb300 import synthetic as syn

from gpu_util import bf16_to_f64, bf16_to_u16, dev_u16_as_bf16, dev_u8, poisoned_gemm, require_gpu
from parity import assert_close

pytestmark = pytest.mark.gpu

GS = [64, 32]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def device(inp):
    return (dev_u16_as_bf16(inp.x), w4.pack(dev_u8(inp.w_canon)), dev_u16_as_bf16(inp.scales))


def check(M, N, K, G, seed=0, cols=None, **kw):
    inp = syn.make_gemm_inputs(M, N, K, G=G, seed=seed)
    x, wp, s = device(inp)
    y = poisoned_gemm(x, wp, s, **kw)
    torch.cuda.synchronize()
    got = bf16_to_f64(y)
    if cols is None:
        ref = oracle.gemm(inp.x, inp.w_canon, inp.scales, M, N, K, G=G)
        assert_close(got, ref, what=f"{M}x{N}x{K} G={G} {kw}")
    else:
        ref = oracle.gemm(inp.x, inp.w_canon[cols], inp.scales[cols], M, len(cols), K, G=G)
        assert_close(got[:, cols], ref, what=f"{M}x{N}x{K} G={G} {kw} sampled")
    return y


@pytest.mark.parametrize("G", GS)
@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (4, 2560, 1024), (8, 300, 640), (13, 200, 384),
                                   (16, 2560, 1024), (1, 640, 2048)])
def test_decode_auto(M, N, K, G):
    assert w4.plan(M, N, K, group_size=G)["arm"] == "decode"
    assert not w4.plan(M, N, K, group_size=G)["whole_k"]
    check(M, N, K, G)


@pytest.mark.parametrize("G", GS)
@pytest.mark.parametrize("M", [1, 9])
@pytest.mark.parametrize("split", [1, 2, 4, 8, 16])
def test_decode_every_slice_width(M, G, split):
    # K = 2048 is 16 blocks of 128: splits 16, 8, 4, 2, 1 give slices of 1 to
    # 16 blocks, clamped to the register limit of 16 (8 for two token octets)
    # scales per row and slice.
    check(M, 384, 2048, G, seed=split, arm="decode", split_k=split)


@pytest.mark.parametrize("G", GS)
def test_decode_refuses_whole_k_kernel(G):
    inp = syn.make_gemm_inputs(2, 256, 512, G=G)
    x, wp, s = device(inp)
    with pytest.raises(w4.W4A16Error):
        w4.gemm(x, wp, s, decode_kernel="whole_k")


@pytest.mark.parametrize("G", GS)
def test_decode_resident_weights(G):
    check(3, 1280, 1536, G, resident_weights=True)


@pytest.mark.parametrize("G", GS)
@pytest.mark.parametrize("M,N,K,kw", [(64, 512, 1024, {}), (200, 300, 640, {}),
                                      (128, 2560, 1024, {"split_k": 2}),
                                      (96, 384, 512, {"tile_tokens": 32}),
                                      (33, 256, 768, {"arm": "tensor", "tile_tokens": 256}),
                                      (5, 256, 512, {"arm": "tensor"})])
def test_tensor_arm(M, N, K, G, kw):
    if M > 16:
        assert w4.plan(M, N, K, group_size=G, **kw)["arm"] == "tensor"
    check(M, N, K, G, arm="tensor", **{k: v for k, v in kw.items() if k != "arm"})


@pytest.mark.parametrize("G", GS)
def test_tensor_arm_repeated_scales_bit_identical_to_128(G):
    # The tensor arm rounds scale * (code - 8) once to bf16 per weight; with
    # each 128-wide group's scale repeated over its sub-groups every operand,
    # and so every output bit, is that of the G = 128 call.
    M, N, K = 96, 640, 1280
    inp = syn.make_gemm_inputs(M, N, K, seed=5)
    x, wp, s = device(inp)
    rep = dev_u16_as_bf16(np.repeat(inp.scales, 128 // G, axis=1))
    a = w4.gemm(x, wp, s, arm="tensor")
    b = w4.gemm(x, wp, rep, arm="tensor")
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_decode_headline_shape_g32_sampled():
    check(1, 8192, 8192, 32, cols=np.r_[0:64, 4000:4064, 8128:8192])


def test_prefill_shape_g32_sampled():
    rng = np.random.default_rng(1)
    cols = np.unique(np.r_[rng.choice(19456, 128, replace=False), 0, 19455])
    check(1322, 19456, 2560, 32, cols=cols)


@pytest.mark.parametrize("G", GS)
def test_deterministic(G):
    inp = syn.make_gemm_inputs(4, 2560, 1024, G=G, seed=3)
    x, wp, s = device(inp)
    a = w4.gemm(x, wp, s, split_k=4)
    b = w4.gemm(x, wp, s, split_k=4)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("G", GS)
def test_grouped(G):
    g = syn.make_grouped_inputs(4, 200, 384, 512, G=G, seed=G, m_sizes=[30, 0, 101, 69])
    x = dev_u16_as_bf16(g.x)
    s = dev_u16_as_bf16(g.scales)
    wp = torch.cat([w4.pack(dev_u8(g.w_canon[i])) for i in range(g.num_groups)])
    ms = torch.from_numpy(np.asarray(g.m_sizes, dtype=np.int32).copy()).cuda()
    y, status = w4.gemm_grouped(x, wp, s, ms)
    torch.cuda.synchronize()
    assert int(status[0].item()) == 0
    ref = oracle.gemm_grouped(g.x, g.w_canon, g.scales, g.m_sizes, 200, 384, 512, G=G)
    assert_close(bf16_to_f64(y), ref, what=f"grouped G={G}")


@pytest.mark.parametrize("G", GS)
@pytest.mark.parametrize("M", [4, 64])
def test_batched(G, M):
    inps = [syn.make_gemm_inputs(M, 384, 768, G=G, seed=10 + b) for b in range(3)]
    x = torch.stack([dev_u16_as_bf16(i.x) for i in inps])
    wp = torch.stack([w4.pack(dev_u8(i.w_canon)) for i in inps])
    s = torch.stack([dev_u16_as_bf16(i.scales) for i in inps])
    y = w4.gemm_batched(x, wp, s)
    torch.cuda.synchronize()
    for b, i in enumerate(inps):
        ref = oracle.gemm(i.x, i.w_canon, i.scales, M, 384, 768, G=G)
        assert_close(bf16_to_f64(y[b]), ref, what=f"batched G={G} entry {b}")


@pytest.mark.parametrize("G", GS)
def test_dequant_bit_exact(G):
    N, K = 200, 640
    inp = syn.make_gemm_inputs(1, N, K, G=G, seed=7)
    wp = w4.pack(dev_u8(inp.w_canon))
    s = dev_u16_as_bf16(inp.scales)
    got32 = w4.dequant_fp32(wp, s, group_size=G).cpu().numpy()
    got16 = bf16_to_u16(w4.dequant_bf16(wp, s, group_size=G))
    assert np.array_equal(got32, oracle.dequant_f32(inp.w_canon, inp.scales, N, K, G=G))
    assert np.array_equal(got16, oracle.dequant_bf16(inp.w_canon, inp.scales, N, K, G=G))


def test_scales_shape_selects_group_size():
    inp = syn.make_gemm_inputs(2, 256, 512, G=32)
    x, wp, s = device(inp)
    with pytest.raises(ValueError):
        w4.gemm(x, wp, s[:, :10])              # K / 10 is not a group size
    with pytest.raises(ValueError):
        w4.gemm(x, wp, s[:, :2].contiguous())  # G = 256 is not served


@pytest.mark.parametrize("G", GS + [128])
@pytest.mark.parametrize("M,arm", [(3, "decode"), (80, "tensor")])
def test_scales_only_2_byte_aligned(G, M, arm):
    # Scales at an address that is a multiple of 2 but not of 4: both arms
    # fall back from their vector scale loads to one load per scale.
    inp = syn.make_gemm_inputs(M, 384, 1024, G=G, seed=12)
    x, wp, s = device(inp)
    buf = torch.empty(s.numel() + 1, dtype=torch.bfloat16, device="cuda")
    s_odd = buf[1:].view(s.shape)
    s_odd.copy_(s)
    assert s_odd.data_ptr() % 4 == 2
    y = w4.gemm(x, wp, s_odd, arm=arm)
    torch.cuda.synchronize()
    ref = oracle.gemm(inp.x, inp.w_canon, inp.scales, M, 384, 1024, G=G)
    assert_close(bf16_to_f64(y), ref, what=f"odd scales G={G} {arm}")


@pytest.mark.parametrize("G", [64, 32])
@pytest.mark.parametrize("kw", [dict(arm="decode"), dict(arm="decode", split_k=4), dict(arm="tensor")])
def test_all_eights_give_exact_zeros(G, kw):
    # Every weight is scale * (8 - 8) = 0: Y_ref is 0 and so is the bound.
    M, N, K = 6, 260, 1024
    inp = syn.make_gemm_inputs(M, N, K, G=G, seed=8)
    inp.w_canon[:] = 0x88
    x, wp, s = device(inp)
    y = bf16_to_f64(poisoned_gemm(x, wp, s, **kw))
    assert np.all(y == 0.0), f"G={G} {kw}: max |y| {np.max(np.abs(y))}"
