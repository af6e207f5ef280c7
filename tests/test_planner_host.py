"""The planner's rules, checked on the CPU through w4a16_plan_for_sms (plans
for a GB300's 152 SMs without a GPU): dispatch by token count, slice caps for
32/64-column groups and zero points, the whole-K kernel's scope, workspace
sizes, the split-K choices measured on GB300, and determinism."""
from __future__ import annotations

import ctypes

import pytest

from bf16_activation_quantized_gb300 import _lib

SMS = 152
OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def L():
    from bf16_activation_quantized_gb300 import build as build_mod
    build_mod.build()
    return _lib.lib()


def plan(L, M, N, K, G=128, batch=1, arm=0, split_k=0, tile=0, flags=0, sms=SMS):
    info = _lib.PlanInfo()
    o = _lib.Options(arm, split_k, tile, flags)
    st = L.w4a16_plan_for_sms(sms, batch, M, N, K, G, ctypes.byref(o), ctypes.byref(info))
    return st, info


SHAPES = [(1, 8192, 8192), (1, 17408, 5120), (1, 19456, 2560), (8, 2560, 9728), (16, 19456, 2560),
          (4, 256, 512), (13, 300, 640), (2, 2560, 1024)]


def test_arguments(L):
    assert plan(L, 1, 256, 512, sms=-1)[0] == INVALID
    assert plan(L, 1, 256, 512, sms=5000)[0] == INVALID
    assert plan(L, 1, 256, 500)[0] == INVALID
    assert plan(L, 1, 256, 512, G=16)[0] == UNSUPPORTED
    st, info = plan(L, 2, 256, 512, batch=2, flags=8)                 # batched zero points
    assert st == OK and info.arm == 1 and not info.whole_k


@pytest.mark.parametrize("M", [1, 8, 16, 17, 32, 1322])
def test_dispatch_by_token_count(L, M):
    st, info = plan(L, M, 2560, 9728)
    assert st == OK
    assert info.arm == (1 if M <= 16 else 2)


@pytest.mark.parametrize("G", [128, 64, 32])
@pytest.mark.parametrize("zp", [False, True])
@pytest.mark.parametrize("M,N,K", SHAPES)
def test_decode_slice_caps(L, M, N, K, G, zp):
    # A slice's scale groups of a row stay in registers: at most 16 (one token
    # octet) or 8 (two), halved with zero points; slices divide K exactly.
    st, info = plan(L, M, N, K, G=G, flags=8 if zp else 0)
    assert st == OK and info.arm == 1
    blocks = K // 128
    assert blocks % info.split_k == 0
    gps = blocks // info.split_k
    cap = (16 if M <= 8 else 8) // (128 // G) // (2 if zp else 1)
    if info.whole_k:
        assert G == 128 and not zp and info.split_k == 1
    else:
        assert gps <= cap, (gps, cap)
    assert info.workspace_bytes == (info.split_k * M * N * 4 if info.split_k > 1 else 0)


@pytest.mark.parametrize("G", [64, 32])
def test_whole_k_kernel_only_for_128_column_symmetric_groups(L, G):
    assert plan(L, 1, 19456, 2560)[1].whole_k                      # the measured winner at G=128
    assert not plan(L, 1, 19456, 2560, G=G)[1].whole_k
    assert not plan(L, 1, 19456, 2560, flags=8)[1].whole_k
    assert plan(L, 1, 19456, 2560, G=G, flags=2)[0] == UNSUPPORTED   # forced whole-K refused
    assert plan(L, 1, 19456, 2560, flags=8 | 2)[0] == UNSUPPORTED


def test_headline_plans(L):
    # The decode GEMV shapes' plans on a GB300 (the figures quoted for them).
    st, a = plan(L, 1, 8192, 8192)
    assert st == OK and a.arm == 1 and a.split_k == 1 and a.whole_k and a.ctas == 256
    st, b = plan(L, 1, 17408, 5120)
    assert st == OK and b.arm == 1 and b.split_k == 1 and b.whole_k and b.ctas == 272
    st, c = plan(L, 1322, 19456, 2560)
    assert st == OK and c.arm == 2 and c.split_k == 1 and c.tile_tokens == 192 and c.ctas == SMS


@pytest.mark.parametrize("M,N,K", [(512, 7168, 8192), (2048, 8192, 8192), (1024, 2560, 9728)])
def test_split_drain_keeps_these_unsplit(L, M, N, K):
    # Measured on GB300: splitting these in wide plain-epilogue tiles was
    # 11-32 % slower than the unsplit plans.
    st, info = plan(L, M, N, K)
    assert st == OK and info.arm == 2 and info.split_k == 1


def test_planning_is_deterministic_and_scales_with_sms(L):
    a = plan(L, 1, 8192, 8192)[1]
    b = plan(L, 1, 8192, 8192)[1]
    assert (a.split_k, a.ctas) == (b.split_k, b.ctas)
    small = plan(L, 1, 8192, 8192, sms=16)[1]
    assert small.ctas <= 2 * 16 * max(1, small.split_k)
    big = plan(L, 1322, 19456, 2560, sms=16)[1]
    assert big.ctas <= 2 * 16


def test_batched_plans_share_the_slots(L):
    one = plan(L, 4, 8192, 3584)[1]
    four = plan(L, 4, 8192, 3584, batch=4)[1]
    assert four.arm == one.arm == 1
    assert four.workspace_bytes == (four.split_k * 4 * 4 * 8192 * 4 if four.split_k > 1 else 0)


@pytest.mark.parametrize("M,N,K", [(1322, 19456, 2560), (64, 2560, 9728), (200, 300, 640),
                                   (4096, 2560, 9728), (33, 8192, 8192)])
def test_tensor_tiles_are_valid(L, M, N, K):
    st, info = plan(L, M, N, K)
    assert st == OK and info.arm == 2
    assert 32 <= info.tile_tokens <= 256 and info.tile_tokens % 32 == 0
    assert 1 <= info.ctas <= 2 * SMS
    blocks = K // 128
    assert 1 <= info.split_k <= min(blocks, 16)
    assert info.workspace_bytes == (info.split_k * M * N * 4 if info.split_k > 1 else 0)


@pytest.mark.parametrize("tile", [32, 64, 128, 192, 256])
def test_forced_tile_is_honoured(L, tile):
    st, info = plan(L, 300, 2560, 1024, arm=2, tile=tile)
    assert st == OK and info.tile_tokens == tile


@pytest.mark.parametrize("bad", [16, 48, 288, -32])
def test_bad_forced_tiles_are_refused(L, bad):
    assert plan(L, 300, 2560, 1024, arm=2, tile=bad)[0] != OK


def test_forced_tile_on_the_decode_arm_is_refused(L):
    assert plan(L, 4, 2560, 1024, arm=1, tile=64)[0] == INVALID


@pytest.mark.parametrize("request_,want", [(1, 1), (2, 2), (3, 4), (5, 8), (8, 8), (16, 16), (40, 16)])
def test_forced_decode_split_rounds_up_to_a_slice_count(L, request_, want):
    # K = 2048 is 16 blocks; slices hold 1, 2, 4, 8 or 16 of them, and a request
    # becomes the nearest feasible count from above (16 at most).
    st, info = plan(L, 1, 384, 2048, arm=1, split_k=request_, flags=4)
    assert st == OK and info.split_k == want


def test_forced_tensor_split(L):
    for sk in (1, 2, 5, 20):
        st, info = plan(L, 128, 2560, 2560, arm=2, split_k=sk)
        assert st == OK and info.split_k == min(sk, 20)


def test_forced_arms(L):
    assert plan(L, 1, 2560, 1024, arm=2)[1].arm == 2            # one token on the tensor arm
    assert plan(L, 64, 2560, 1024, arm=1)[1].arm == 1           # 64 tokens on the decode arm
    assert plan(L, 1, 2560, 1024, arm=7)[0] == INVALID


def test_whole_k_refused_where_it_does_not_fit(L):
    # The whole-K kernel takes up to 16 tokens (two octets; their X columns
    # travel in each ring stage, which must hold at least three stages next
    # to the CTA's scales in shared memory).
    assert plan(L, 2, 2560, 8192, flags=2)[1].whole_k
    assert plan(L, 8, 2560, 8192, flags=2)[1].whole_k
    assert plan(L, 16, 2560, 9728, flags=2)[1].whole_k
    assert plan(L, 17, 256, 512, flags=2)[0] == UNSUPPORTED
    assert plan(L, 16, 256, 131072, flags=2)[0] == UNSUPPORTED     # X and scales: < 3 stages
    assert plan(L, 1, 256, 262144, flags=2)[0] == UNSUPPORTED      # the scales alone


def test_gate_up_at_16_tokens_takes_the_whole_k_kernel(L):
    # Two token octets per dequantised fragment: 304 CTAs of 64 rows.
    st, info = plan(L, 16, 19456, 2560)
    assert st == OK and info.arm == 1 and info.whole_k and info.ctas == 2 * SMS


def test_python_plan_for_sms_needs_no_gpu():
    import bf16_activation_quantized_gb300 as w4
    p = w4.plan(1, 8192, 8192, sms=SMS)
    assert p == {"arm": "decode", "split_k": 1, "tile_tokens": 8, "ctas": 256,
                 "workspace_bytes": 0, "whole_k": True}
    assert w4.plan(1, 8192, 8192, sms=SMS, decode_kernel="k_slices")["split_k"] == 8
    assert w4.plan(1322, 19456, 2560, sms=SMS)["tile_tokens"] == 192
    assert w4.plan(1, 19456, 2560, sms=SMS, group_size=32, zero_points=True)["whole_k"] is False
    with pytest.raises(w4.W4A16Error):
        w4.plan(1, 256, 512, sms=SMS, group_size=16)


# Tensor-arm plans pinned by measurements on GB300 (graphs of back-to-back
# calls, rotating weights).  Each case names the plan that measured fastest
# among the tile widths and splits tried for it.
@pytest.mark.parametrize("M,N,K,bt,split", [
    # long prefills: separate-epilogue 192-token tiles beat plain 256-token ones
    # (2048x19456x2560 127 vs 158 us, 4096x19456x2560 247 vs 312 us,
    # 2048x8192x8192 172 vs 203 us)
    (2048, 19456, 2560, 192, 1), (4096, 19456, 2560, 192, 1), (2048, 8192, 8192, 192, 1),
    (1322, 19456, 2560, 192, 1), (1322, 2560, 9728, 192, 1),
    # unsplit 160-token tiles beat split 2 (78.0 vs 88.4 us: 42 MB of partials)
    (2048, 2560, 9728, 160, 1),
    # one tile per CTA: the plain 256-token form, unsplit (split 4 measured 47 % slower)
    (512, 7168, 8192, 256, 1),
    # split 2 beats split 16 (19.4 vs 27.5 us); unsplit 64-token tiles beat split 3 (7.3 vs 11.9 us)
    (33, 8192, 8192, 64, 2), (300, 2560, 1024, 64, 1),
    # several tiles per CTA: plain tiles above 192 tokens lose to narrower ones
    # (1024x19456x2560 192: 68.9 vs 256: 79.7 us; 512x19456x2560 37.4 vs 40.9 us;
    # 2048x4096x4096 160: 52.1 vs 256: 58.0 us; 2048x7168x8192 161.3 vs 163.4 us;
    # 1024x7168x8192 160: 96.5 vs 224: 103.4 us)
    (1024, 19456, 2560, 192, 1), (512, 19456, 2560, 192, 1), (2048, 4096, 4096, 160, 1),
    (2048, 7168, 8192, 160, 1), (1024, 7168, 8192, 160, 1),
])
def test_measured_tensor_plans(L, M, N, K, bt, split):
    st, info = plan(L, M, N, K)
    assert st == OK and info.arm == 2
    assert (info.tile_tokens, info.split_k) == (bt, split), (info.tile_tokens, info.split_k)
