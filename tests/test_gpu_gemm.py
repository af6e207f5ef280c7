"""GPU parity of the GEMM against the fp64 oracle, on the workloads' shapes, with
every arm and split forced, edge cases, determinism and graph replay.

Bar (float): |y - yref| <= 8e-3*|yref| + 2e-3*max|yref| element-wise and
cosine >= 0.99999 (tests/parity.py).  Full outputs are compared wherever the
oracle finishes in seconds; for the 1322-token prefill shapes the oracle
computes a sample of output features (every token), chosen at random plus the
first and last feature."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import bf16_activation_quantized_gb300 as w4
import oracle
from bf16_activation_quantized_gb300 import _lib
from bf16_activation_quantized_gb300 import synthetic as syn

from gpu_util import DeviceProblem, bf16_to_f64, bf16_to_u16, poisoned_gemm, require_gpu
from parity import assert_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    require_gpu()


_cache = {}


def problem(M, N, K, seed=0):
    key = (M, N, K, seed)
    if key not in _cache:
        if len(_cache) > 6:
            _cache.clear()
            torch.cuda.empty_cache()
        _cache[key] = DeviceProblem(syn.make_gemm_inputs(M, N, K, seed=seed))
    return _cache[key]


def reference(p, cols=None):
    i = p.inp
    if cols is None:
        if getattr(p, "_ref", None) is None:
            p._ref = oracle.gemm(i.x, i.w_canon, i.scales, i.M, i.N, i.K)
        return p._ref
    return oracle.gemm(i.x, i.w_canon[cols], i.scales[cols], i.M, len(cols), i.K)


def sample_cols(N, count=192, seed=0):
    rng = np.random.default_rng(seed + N)
    cols = np.unique(np.concatenate([rng.choice(N, size=min(count, N), replace=False),
                                     [0, N - 1]]))
    return cols


def run(p, **kw):
    y = poisoned_gemm(p.x, p.w_packed, p.scales, **kw)
    torch.cuda.synchronize()
    return y


# ------------------------------------------------------------- the workloads
TINY = [(4, 256, 512)]
DECODE = [(1, 8192, 8192), (1, 17408, 5120)]
SWEEP = [(m, n, k) for (n, k) in ((19456, 2560), (2560, 9728)) for m in (1, 8, 16, 32, 64, 128)]
PREFILL = [(1322, 19456, 2560), (1322, 2560, 9728)]


@pytest.mark.parametrize("M,N,K", TINY + DECODE + SWEEP)
def test_workload_full_output(M, N, K):
    p = problem(M, N, K)
    y = run(p)
    assert_close(bf16_to_f64(y), reference(p), what=f"M{M} N{N} K{K} {w4.plan(M, N, K)}")


@pytest.mark.parametrize("M,N,K", PREFILL)
def test_prefill_sampled_features(M, N, K):
    p = problem(M, N, K)
    y = bf16_to_f64(run(p))
    cols = sample_cols(N)
    assert_close(y[:, cols], reference(p, cols), what=f"M{M} N{N} K{K}")
    assert np.all(np.isfinite(y))


# ------------------------------------------------------- forced arms / splits
@pytest.mark.parametrize("M", [1, 3, 8, 9, 16])
@pytest.mark.parametrize("split_k", [1, 2, 3, 5])
def test_decode_arm_every_split(M, split_k):
    N, K = 300, 640        # 3 tiles with a ragged last tile, 5 groups
    p = problem(M, N, K, seed=M)
    y = run(p, arm="decode", split_k=split_k, decode_kernel="k_slices")
    plan = w4.plan(M, N, K, arm="decode", split_k=split_k, decode_kernel="k_slices")
    # 5 groups: every slice holds one group, whatever split is requested
    assert plan["split_k"] == 5
    assert_close(bf16_to_f64(y), reference(p), what=f"decode M{M} SK{split_k}")


@pytest.mark.parametrize("M", [1, 5, 8, 12, 16])
@pytest.mark.parametrize("split_k", [1, 2, 4, 8])
def test_decode_arm_slice_sizes(M, split_k):
    N, K = 300, 1024       # 8 groups: slices of 8, 4, 2 and 1 groups
    p = problem(M, N, K, seed=M + 100)
    y = run(p, arm="decode", split_k=split_k, decode_kernel="k_slices")
    assert w4.plan(M, N, K, arm="decode", split_k=split_k, decode_kernel="k_slices")["split_k"] == split_k
    assert_close(bf16_to_f64(y), reference(p), what=f"decode M{M} SK{split_k}")


@pytest.mark.parametrize("M", [1, 3, 8, 12])
def test_decode_arm_sixteen_group_slices(M):
    N, K = 300, 2048       # 16 groups: one 16-group slice for up to 8 tokens, else two of 8
    p = problem(M, N, K, seed=M + 200)
    y = run(p, arm="decode", split_k=1, decode_kernel="k_slices")
    assert w4.plan(M, N, K, arm="decode", split_k=1, decode_kernel="k_slices")["split_k"] == (1 if M <= 8 else 2)
    assert_close(bf16_to_f64(y), reference(p), what=f"decode M{M} one slice")


@pytest.mark.parametrize("M,N,K", [(1, 19456, 2560), (16, 2560, 9728), (8, 8192, 8192)])
@pytest.mark.parametrize("split_k", [1, 4, 16])
def test_decode_arm_splits_on_workload_shapes(M, N, K, split_k):
    p = problem(M, N, K)
    y = run(p, arm="decode", split_k=split_k, decode_kernel="k_slices")
    assert_close(bf16_to_f64(y), reference(p), what=f"decode M{M} N{N} K{K} SK{split_k}")


@pytest.mark.parametrize("M", [1, 16, 17, 32, 33, 64, 100, 300])
@pytest.mark.parametrize("tile_tokens", [32, 96, 256])
@pytest.mark.parametrize("split_k", [1, 2, 5])
def test_tensor_arm_tiles_and_splits(M, tile_tokens, split_k):
    N, K = 300, 640        # 3 weight tiles with a ragged last one, 5 groups
    p = problem(M, N, K, seed=M + 1)
    y = run(p, arm="tensor", split_k=split_k, tile_tokens=tile_tokens)
    plan = w4.plan(M, N, K, arm="tensor", split_k=split_k, tile_tokens=tile_tokens)
    assert plan["arm"] == "tensor" and plan["tile_tokens"] == tile_tokens
    assert plan["split_k"] == split_k
    assert_close(bf16_to_f64(y), reference(p), what=f"tensor M{M} BT{tile_tokens} SK{split_k}")


@pytest.mark.parametrize("M,N,K", [(32, 19456, 2560), (128, 2560, 9728), (1322, 2560, 9728)])
@pytest.mark.parametrize("tile_tokens", [64, 224])
def test_tensor_arm_workload_shapes(M, N, K, tile_tokens):
    p = problem(M, N, K)
    y = bf16_to_f64(run(p, arm="tensor", tile_tokens=tile_tokens))
    cols = sample_cols(N, 128)
    assert_close(y[:, cols], reference(p, cols), what=f"tensor M{M} N{N} K{K} BT{tile_tokens}")


def test_tensor_arm_matches_bf16_operand_exactly_on_one_group():
    # With unit activations on one column and K = 128 the output is the bf16
    # weight operand itself (one product, exact accumulation): compare bits.
    M, N, K = 32, 256, 128
    inp = syn.make_gemm_inputs(M, N, K, seed=9)
    inp.x[:] = 0
    for m in range(M):
        inp.x[m, (m * 5) % K] = 0x3F80
    p = DeviceProblem(inp)
    y = bf16_to_u16(run(p, arm="tensor"))
    wq = oracle.dequant_bf16(inp.w_canon, inp.scales, N, K)
    for m in range(M):
        assert np.array_equal(y[m], wq[:, (m * 5) % K])


@pytest.mark.parametrize("M", [17, 40, 100])
def test_decode_arm_many_token_blocks(M):
    p = problem(M, 256, 512, seed=M)
    y = run(p, arm="decode")
    assert_close(bf16_to_f64(y), reference(p), what=f"decode M{M}")


# ------------------------------------------------------------------ edge cases
@pytest.mark.parametrize("M,N,K", [(1, 1, 128), (2, 7, 128), (1, 16, 128), (5, 129, 256),
                                   (3, 200, 65536 // 8), (16, 136, 1024)])
def test_edge_shapes(M, N, K):
    p = problem(M, N, K, seed=7)
    y = run(p)
    assert_close(bf16_to_f64(y), reference(p), what=f"edge M{M} N{N} K{K}")


def test_empty_m_is_a_noop():
    p = problem(4, 256, 512)
    out = torch.full((0, 256), 1.0, dtype=torch.bfloat16, device="cuda")
    x0 = p.x[:0]
    L = _lib.lib()
    st = L.w4a16_gemm(x0.data_ptr(), p.w_packed.data_ptr(), p.scales.data_ptr(), out.data_ptr(),
                      0, 256, 512, 128, None, 0, None)
    assert st == 0


def _bf16_bits_to_f64(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32).astype(np.float64)


def test_all_eights_and_zero_scales_give_zero():
    # Every weight is scale * (8 - 8) = 0, or has a zero scale: Y_ref is 0, so
    # the bound |y - y_ref| <= 8e-3 |y_ref| + 2e-3 max|y_ref| is 0 and every
    # arm, kernel and split must return exact zeros.  (The decode arm removes
    # the 1024 + 8 offset of its fp16 operands exactly, before the MMA.)
    M, N, K = 5, 300, 640
    inp = syn.make_gemm_inputs(M, N, K, seed=3)
    inp.w_canon[:] = 0x88
    p = DeviceProblem(inp)
    for kw in (dict(arm="tensor"), dict(arm="tensor", split_k=5), dict(arm="decode"),
               dict(arm="decode", split_k=5), dict(arm="decode", split_k=1)):
        y = bf16_to_f64(run(p, **kw))
        assert np.all(y == 0.0), f"{kw}: max |y| {np.max(np.abs(y))}"
    inp2 = syn.make_gemm_inputs(M, N, K, seed=4)
    inp2.scales[:] = 0
    p2 = DeviceProblem(inp2)
    for kw in (dict(arm="tensor"), dict(arm="decode"), dict(arm="decode", split_k=5)):
        assert np.all(bf16_to_f64(run(p2, **kw)) == 0.0), kw


def test_unit_scales_one_hot_is_exact():
    M, N, K = 4, 300, 640
    inp = syn.make_gemm_inputs(M, N, K, seed=4)
    inp.scales[:] = 0x3F80
    inp.x[:] = 0
    ks = [0, 77, 128, 639]
    for m, k0 in enumerate(ks):
        inp.x[m, k0] = 0x3F80
    p = DeviceProblem(inp)
    y = bf16_to_f64(run(p))
    codes = np.empty((N, K), dtype=np.int64)
    codes[:, 0::2] = inp.w_canon & 0xF
    codes[:, 1::2] = inp.w_canon >> 4
    for m, k0 in enumerate(ks):
        assert np.array_equal(y[m], (codes[:, k0] - 8).astype(np.float64))


# ------------------------------------------------- determinism / graph replay
@pytest.mark.parametrize("M,N,K", [(1, 8192, 8192), (16, 2560, 9728), (4, 256, 512)])
def test_repeat_is_bit_exact(M, N, K):
    p = problem(M, N, K)
    a = bf16_to_u16(run(p))
    for _ in range(3):
        assert np.array_equal(bf16_to_u16(run(p)), a)


@pytest.mark.parametrize("M,N,K", [(1, 8192, 8192), (16, 2560, 9728)])
def test_cuda_graph_replay_matches_eager(M, N, K):
    p = problem(M, N, K)
    eager = bf16_to_u16(run(p))
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    need = w4.plan(M, N, K)["workspace_bytes"]
    ws = torch.empty(max(need, 16), dtype=torch.uint8, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        w4.gemm(p.x, p.w_packed, p.scales, out=out, workspace=ws)    # warm-up on the side stream
    torch.cuda.current_stream().wait_stream(s)
    out.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        w4.gemm(p.x, p.w_packed, p.scales, out=out, workspace=ws)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bf16_to_u16(out), eager)


def test_workspace_too_small_is_rejected_before_launch():
    M, N, K = 16, 2560, 9728         # a split-K plan: it needs a workspace
    p = problem(M, N, K)
    need = w4.plan(M, N, K)["workspace_bytes"]
    assert need > 0
    out = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    L = _lib.lib()
    st = L.w4a16_gemm(p.x.data_ptr(), p.w_packed.data_ptr(), p.scales.data_ptr(), out.data_ptr(),
                      M, N, K, 128, ws.data_ptr(), need - 4, None)
    assert st == 3
    st = L.w4a16_gemm(p.x.data_ptr(), p.w_packed.data_ptr(), p.scales.data_ptr(), out.data_ptr(),
                      M, N, K, 128, None, 0, None)
    assert st == 3
    torch.cuda.synchronize()
    assert torch.count_nonzero(out).item() == 0          # nothing was launched
    nb = ctypes.c_size_t(0)
    assert L.w4a16_workspace_bytes(M, N, K, 128, ctypes.byref(nb)) == 0 and nb.value == need


@pytest.mark.parametrize("M,N,K", [(1, 8192, 8192), (16, 2560, 9728), (3, 300, 640)])
def test_partials_then_reduce_equals_gemm(M, N, K):
    p = problem(M, N, K)
    full = bf16_to_u16(run(p))
    plan = w4.plan(M, N, K)
    ws = torch.empty(max(plan["workspace_bytes"], 16), dtype=torch.uint8, device="cuda")
    out = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    sk = w4.gemm_partials(p.x, p.w_packed, p.scales, out=out, workspace=ws)
    assert sk == plan["split_k"]
    if sk > 1:
        assert torch.count_nonzero(out).item() == 0
        parts = ws[: sk * M * N * 4].view(torch.float32).view(sk, M, N)
        # the partial slices sum (in fp64) to the oracle within the bar
        assert_close(parts.double().sum(0).cpu().numpy(), reference(p), what="partials")
        w4.splitk_reduce(parts, out=out)
    torch.cuda.synchronize()
    assert np.array_equal(bf16_to_u16(out), full)


# ---------------------------------------------------------------- split-K reduce
@pytest.mark.parametrize("S,M,N", [(1, 4, 256), (3, 5, 300), (8, 1, 19456), (16, 2, 7)])
def test_splitk_reduce_bit_exact(S, M, N):
    # Dyadic partial sums (multiples of 2^-12 below 2^8) add exactly in fp32, so the
    # only rounding is the final one to bf16, which the oracle does in fp64.
    rng = np.random.default_rng(S * 1000 + N)
    ws = (rng.integers(-2 ** 19, 2 ** 19, size=(S, M, N)) * 2.0 ** -12).astype(np.float32)
    got = bf16_to_u16(w4.splitk_reduce(torch.from_numpy(ws).cuda()))
    ref = oracle.sum_slices(ws)
    expect = np.array([oracle.f64_to_bf16(v) for v in ref.ravel()], dtype=np.uint16).reshape(M, N)
    assert np.array_equal(got, expect)


# ------------------------------------------------------------ resident weights
@pytest.mark.parametrize("M,N,K,arm", [(1, 8192, 8192, None), (16, 2560, 9728, None), (3, 300, 640, None),
                                       (8, 19456, 2560, None), (64, 2048, 2048, "tensor"),
                                       (256, 1536, 4096, "tensor"), (40, 640, 1280, "tensor")])
def test_resident_weights_give_the_same_bits(M, N, K, arm):
    # The flag only moves the weight stream ahead of the dependency wait.
    p = problem(M, N, K)
    a = bf16_to_u16(run(p, arm=arm))
    b = bf16_to_u16(run(p, arm=arm, resident_weights=True))
    assert np.array_equal(a, b)


@pytest.mark.parametrize("M,arm", [(1, None), (64, "tensor")])
def test_resident_weights_chain_reads_x_after_the_previous_call(M, arm):
    # A chain of layers on one stream inside one graph, through two ping-pong
    # buffers: the Y of one call is the X of the next, and each call writes
    # the buffer the call before it read as X.  Each call streams its weights
    # early but must read X, and write Y, only after the call before it has
    # completed.
    K = 2048
    layers = [DeviceProblem(syn.make_gemm_inputs(M, K, K, seed=50 + i)) for i in range(4)]
    x0 = layers[0].x.clone()
    bufs = [torch.empty((M, K), dtype=torch.bfloat16, device="cuda") for _ in range(2)]

    def chain(resident):
        bufs[0].copy_(x0)
        outs = []
        for i, lp in enumerate(layers):
            x, y = bufs[i % 2], bufs[(i + 1) % 2]
            w4.gemm(x, lp.w_packed, lp.scales, out=y, arm=arm, resident_weights=resident)
            outs.append(y.clone())
        return outs

    eager = [bf16_to_u16(y) for y in chain(False)]
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        chain(True)                                    # warm-up on the side stream
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        outs = chain(True)
    for _ in range(3):
        for y in outs:
            y.zero_()
        g.replay()
        torch.cuda.synchronize()
        for y, e in zip(outs, eager):
            assert np.array_equal(bf16_to_u16(y), e)
    # and the chain itself is right: the last layer against the oracle, fed the
    # previous layer's bf16 output
    xin = bf16_to_u16(outs[-2]).reshape(M, K)
    last = layers[-1].inp
    ref = oracle.gemm(xin, last.w_canon, last.scales, M, K, K)
    assert_close(bf16_to_f64(outs[-1]), ref, what="chain")


# ------------------------------------------------------ whole-K decode kernel
WHOLE_K = [(1, 8192, 8192), (1, 17408, 5120), (1, 19456, 2560), (1, 2560, 9728), (2, 8192, 8192),
           (4, 4096, 4096), (8, 2048, 2048), (3, 300, 640), (1, 7, 256), (5, 129, 384), (1, 256, 128),
           # two token octets (9..16 tokens), ragged octets and rows
           (9, 2048, 2048), (16, 19456, 2560), (16, 2560, 9728), (13, 300, 1024), (16, 4096, 4096),
           (11, 129, 384)]


@pytest.mark.parametrize("M,N,K", WHOLE_K)
def test_whole_k_kernel_full_output(M, N, K):
    # Every CTA covers all of K for a few 16-row blocks; its warps split K and
    # add their parts in shared memory.
    p = problem(M, N, K)
    pl = w4.plan(M, N, K, arm="decode", decode_kernel="whole_k")
    assert pl["whole_k"] and pl["split_k"] == 1 and pl["workspace_bytes"] == 0
    y = run(p, arm="decode", decode_kernel="whole_k")
    assert_close(bf16_to_f64(y), reference(p), what=f"whole-K M{M} N{N} K{K} {pl}")
    again = run(p, arm="decode", decode_kernel="whole_k", resident_weights=True)
    assert np.array_equal(bf16_to_u16(again), bf16_to_u16(y))


def test_whole_k_kernel_refuses_what_it_cannot_stage():
    # More than 16 tokens, or X columns and scales that leave fewer than three
    # ring stages in a CTA's shared memory, are refused when forced.
    for M, N, K in ((17, 256, 512), (16, 256, 131072), (1, 256, 262144)):
        with pytest.raises(w4.W4A16Error):
            w4.plan(M, N, K, arm="decode", decode_kernel="whole_k")
    assert not w4.plan(1, 8192, 8192, decode_kernel="k_slices")["whole_k"]


def test_whole_k_kernel_in_a_graph_replays_exactly():
    M, N, K = 1, 8192, 8192
    p = problem(M, N, K)
    eager = bf16_to_u16(run(p, arm="decode", decode_kernel="whole_k"))
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        w4.gemm(p.x, p.w_packed, p.scales, out=out, arm="decode", decode_kernel="whole_k")
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(3):
            w4.gemm(p.x, p.w_packed, p.scales, out=out, arm="decode", decode_kernel="whole_k",
                    resident_weights=True)
    for _ in range(2):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bf16_to_u16(out), eager)


def test_whole_k_all_eights_give_zero():
    # All codes 8: every weight is 0, so Y_ref is 0 and the output must be
    # exactly 0 (the offset of the fp16 operands is removed exactly).
    M, N, K = 1, 1024, 4096
    inp = syn.make_gemm_inputs(M, N, K, seed=3)
    inp.w_canon[:] = 0x88
    p = DeviceProblem(inp)
    y = bf16_to_f64(run(p, arm="decode", decode_kernel="whole_k"))
    assert np.all(y == 0.0), f"max |y| {np.max(np.abs(y))}"
