"""GPU parity of the zero-point variant (dequant = scale * (code - z), z a
4-bit integer per row and scale group) against the fp64 oracle's gemm_zp:
both arms, group sizes 128/64/32, forced splits, unaligned zero points, the
bit-exact dequant probes, and z = 8 reproducing the symmetric kernels bit
for bit under the same plan."""
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

GS = [128, 64, 32]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


def device(inp, z):
    return (dev_u16_as_bf16(inp.x), w4.pack(dev_u8(inp.w_canon)), dev_u16_as_bf16(inp.scales),
            dev_u8(z))


def check(M, N, K, G, seed=0, cols=None, **kw):
    inp = syn.make_gemm_inputs(M, N, K, G=G, seed=seed)
    z = syn.make_zeros(N, K, G, seed=seed)
    x, wp, s, zd = device(inp, z)
    y = poisoned_gemm(x, wp, s, zeros=zd, **kw)
    torch.cuda.synchronize()
    got = bf16_to_f64(y)
    if cols is None:
        ref = oracle.gemm_zp(inp.x, inp.w_canon, inp.scales, z, M, N, K, G=G)
        assert_close(got, ref, what=f"zp {M}x{N}x{K} G={G} {kw}")
    else:
        ref = oracle.gemm_zp(inp.x, inp.w_canon[cols], inp.scales[cols], z[cols], M, len(cols), K, G=G)
        assert_close(got[:, cols], ref, what=f"zp {M}x{N}x{K} G={G} {kw} sampled")


@pytest.mark.parametrize("G", GS)
@pytest.mark.parametrize("M,N,K", [(1, 256, 512), (4, 2560, 1024), (13, 200, 384), (16, 2560, 1024),
                                   (8, 300, 640)])
def test_decode(M, N, K, G):
    assert w4.plan(M, N, K, group_size=G, zero_points=True)["arm"] == "decode"
    check(M, N, K, G)


@pytest.mark.parametrize("G", GS)
@pytest.mark.parametrize("M", [1, 9])
@pytest.mark.parametrize("split", [1, 4, 16])
def test_decode_forced_splits(M, G, split):
    check(M, 384, 2048, G, seed=split, arm="decode", split_k=split, resident_weights=True)


@pytest.mark.parametrize("G", GS)
@pytest.mark.parametrize("M,N,K,kw", [(64, 512, 1024, {}), (200, 300, 640, {}),
                                      (128, 2560, 1024, {"split_k": 2}),
                                      (96, 384, 512, {"tile_tokens": 32}),
                                      (5, 256, 512, {})])
def test_tensor(M, N, K, G, kw):
    check(M, N, K, G, arm="tensor", **kw)


def test_decode_headline_shape_sampled():
    check(1, 8192, 8192, 128, cols=np.r_[0:64, 8128:8192])


@pytest.mark.parametrize("G", [128, 32])
def test_prefill_shape_sampled(G):
    rng = np.random.default_rng(2)
    check(1322, 19456, 2560, G, cols=np.unique(np.r_[rng.choice(19456, 96, replace=False), 0, 19455]))


@pytest.mark.parametrize("G", GS)
@pytest.mark.parametrize("M,kw", [(1, {"arm": "decode", "split_k": 4}), (96, {"arm": "tensor"})])
def test_zero_point_eight_matches_symmetric_bits(M, G, kw):
    # Same plan on both calls (forced); with z = 8 the zero-point chain starts
    # from the same correction and the tensor arm subtracts the same 136.
    inp = syn.make_gemm_inputs(M, 384, 2048, G=G, seed=4)
    x, wp, s, zd = device(inp, np.full((384, 2048 // G), 8, dtype=np.uint8))
    a = w4.gemm(x, wp, s, **kw)
    b = w4.gemm(x, wp, s, zeros=zd, **kw)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("G", [128, 32])
@pytest.mark.parametrize("M,arm", [(3, "decode"), (80, "tensor")])
def test_unaligned_zero_points(G, M, arm):
    inp = syn.make_gemm_inputs(M, 384, 1024, G=G, seed=8)
    z = syn.make_zeros(384, 1024, G, seed=8)
    x, wp, s, zd = device(inp, z)
    buf = torch.empty(zd.numel() + 1, dtype=torch.uint8, device="cuda")
    z_odd = buf[1:].view(zd.shape)
    z_odd.copy_(zd)
    y = w4.gemm(x, wp, s, zeros=z_odd, arm=arm)
    torch.cuda.synchronize()
    ref = oracle.gemm_zp(inp.x, inp.w_canon, inp.scales, z, M, 384, 1024, G=G)
    assert_close(bf16_to_f64(y), ref, what=f"odd zeros G={G} {arm}")


@pytest.mark.parametrize("G", GS)
def test_dequant_bit_exact(G):
    N, K = 200, 640
    inp = syn.make_gemm_inputs(1, N, K, G=G, seed=9)
    z = syn.make_zeros(N, K, G, seed=9) | np.uint8(0xA0)      # high bits are ignored
    wp = w4.pack(dev_u8(inp.w_canon))
    s = dev_u16_as_bf16(inp.scales)
    got32 = w4.dequant_fp32(wp, s, group_size=G, zeros=dev_u8(z)).cpu().numpy()
    got16 = bf16_to_u16(w4.dequant_bf16(wp, s, group_size=G, zeros=dev_u8(z)))
    assert np.array_equal(got32, oracle.dequant_zp_f32(inp.w_canon, inp.scales, z, N, K, G=G))
    assert np.array_equal(got16, oracle.dequant_zp_bf16(inp.w_canon, inp.scales, z, N, K, G=G))


def test_zero_points_shape_checked():
    inp = syn.make_gemm_inputs(2, 256, 512)
    x, wp, s, zd = device(inp, syn.make_zeros(256, 512))
    with pytest.raises(ValueError):
        w4.gemm(x, wp, s, zeros=zd[:, :1].contiguous())


@pytest.mark.parametrize("G", [128, 64, 32])
@pytest.mark.parametrize("kw", [dict(arm="decode"), dict(arm="decode", split_k=4), dict(arm="tensor")])
def test_codes_equal_to_their_zero_points_give_exact_zeros(G, kw):
    # code = z everywhere: every weight is scale * 0, Y_ref is 0, and the
    # bound is 0, so the output must be exactly 0 for every zero point.
    M, N, K = 6, 260, 1024
    inp = syn.make_gemm_inputs(M, N, K, G=G, seed=9)
    rng = np.random.default_rng(9)
    zg = rng.integers(0, 16, size=(N, K // G)).astype(np.uint8)
    codes = np.repeat(zg, G, axis=1)                      # [N][K]: code(n, k) = z(n, k / G)
    inp.w_canon[:] = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    x, wp, s, zd = device(inp, zg)
    y = bf16_to_f64(poisoned_gemm(x, wp, s, zeros=zd, **kw))
    assert np.all(y == 0.0), f"G={G} {kw}: max |y| {np.max(np.abs(y))}"
