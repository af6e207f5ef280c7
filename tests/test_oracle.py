"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself:
  * fixtures written from the pages (tests/golden/*.txt, each with its source);
  * an independent NumPy brute force (vectorised unpack -> dense fp64 W -> X @ W^T);
  * exact invariants of the definition (all-eights, one-hot, scaling, linearity,
    grouped = concatenation of plain products);
  * exhaustive dequant over all codes and every bf16 scale in the input range;
  * mutation checks: a copy of oracle.c with a planted mistake (swapped nibbles,
    wrong offset, wrong group index, dropped term, flipped sign, transposed
    operand) must fail at least one of these pins.
"""
from __future__ import annotations

import ctypes
import os
import re
import struct
import subprocess

import numpy as np
import pytest

import oracle
from bf16_activation_quantized_gb300 import metrics
from bf16_activation_quantized_gb300 import synthetic as syn

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ----------------------------------------------------------------- brute force
def np_bf16(bits):
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def np_codes(w_canon, K):
    lo = (w_canon & 0x0F).astype(np.int64)
    hi = (w_canon >> 4).astype(np.int64)
    codes = np.empty(w_canon.shape[:-1] + (K,), dtype=np.int64)
    codes[..., 0::2] = lo
    codes[..., 1::2] = hi
    return codes


def np_dense(w_canon, scales, K, G=128):
    s = np.repeat(np_bf16(scales), G, axis=-1)
    return s * (np_codes(w_canon, K) - 8).astype(np.float64)


def np_gemm(x, w_canon, scales, K, G=128):
    return np_bf16(x) @ np_dense(w_canon, scales, K, G).T


def read_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


# --------------------------------------------------------------- page fixtures
def test_golden_nibble_order():
    rows = [r.split() for r in read_rows("nibble_order.txt")]
    bytes_ = np.array([[int(r[0], 16) for r in rows]], dtype=np.uint8)
    K = 2 * bytes_.shape[1]
    for j, r in enumerate(rows):
        assert oracle.nibble(bytes_, K, 0, 2 * j) == int(r[1])
        assert oracle.nibble(bytes_, K, 0, 2 * j + 1) == int(r[2])
    # The generator writes the same packing.
    codes = np.array([[int(r[1]), int(r[2])] for r in rows], dtype=np.uint8).reshape(1, -1)
    assert np.array_equal(syn.pack_codes(codes), bytes_)


def test_golden_magic_constants():
    for r in read_rows("magic_dequant.txt"):
        bits, value = r.split()
        assert oracle.bf16_to_f64(int(bits, 16)) == float(value)
    # scale * ((128 + n) - 136) equals the oracle's dequantised weight for every code.
    minus136 = oracle.bf16_to_f64(0xC308)
    K = 128
    codes = np.tile(np.arange(16, dtype=np.uint8), K // 16).reshape(1, K)
    w = syn.pack_codes(codes)
    for sbits in (0x3F80, 0x3C23, 0x3BA4, 0x4100):
        sc = np.array([[sbits]], dtype=np.uint16)
        dq = oracle.dequant_f64(w, sc, 1, K)
        s = oracle.bf16_to_f64(sbits)
        for k in range(K):
            n = int(codes[0, k])
            assert dq[0, k] == s * (oracle.bf16_to_f64(0x4300 | n) + minus136)


def test_golden_group_starts():
    for r in read_rows("group_starts.txt"):
        sizes, starts = r.split("|")
        sizes = [int(v) for v in sizes.split()]
        starts = [int(v) for v in starts.split()]
        assert list(oracle.group_starts(sizes)) == starts


def test_golden_page_flop_convention():
    """2 * rows * N * K over the printed time reproduces the printed TFLOP/s."""
    for r in read_rows("page_throughput_rows.txt"):
        op, count, rows_each, N, K, us, tf = r.split()
        rows = int(count) * int(rows_each)
        tflops = metrics.flops(rows, int(N), int(K)) / (float(us) * 1e-6) / 1e12
        assert abs(tflops - float(tf)) <= 0.05 + 1e-3 * float(tf), (r, tflops)


# ------------------------------------------------------------- bf16 encodings
def test_bf16_decode_matches_struct():
    rng = np.random.default_rng(1)
    for bits in list(rng.integers(0, 0x7F80, 2000)) + [0, 1, 0x0080, 0x7F7F, 0x8001]:
        f = struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0]
        assert oracle.bf16_to_f64(int(bits)) == f


@pytest.mark.parametrize("value,bits", [
    (1.0, 0x3F80),
    (1.0 + 2.0 ** -8, 0x3F80),            # halfway between 0x3F80 and 0x3F81 -> even
    (1.0 + 3 * 2.0 ** -8, 0x3F82),        # halfway between 0x3F81 and 0x3F82 -> even
    (1.0 + 2.0 ** -8 + 2.0 ** -30, 0x3F81),
    (-2.5, 0xC020),
    (0.0, 0x0000),
    (-0.0, 0x8000),
    (2.0 ** -133, 0x0001),                # smallest subnormal
    (2.0 ** -134, 0x0000),                # half of it: tie -> even (zero)
    (3 * 2.0 ** -134, 0x0002),            # 1.5 quanta: tie -> even (2)
    (3.4e38, 0x7F80),                     # rounds past the largest finite -> inf
])
def test_f64_to_bf16_rne(value, bits):
    assert oracle.f64_to_bf16(value) == bits


# ---------------------------------------------------------------- brute force
@pytest.mark.parametrize("M,N,K,seed", [(1, 16, 128, 0), (3, 33, 256, 1), (4, 256, 512, 0),
                                        (5, 7, 384, 2)])
def test_oracle_matches_numpy_bruteforce(M, N, K, seed):
    inp = syn.make_gemm_inputs(M, N, K, seed=seed)
    y = oracle.gemm(inp.x, inp.w_canon, inp.scales, M, N, K)
    ref = np_gemm(inp.x, inp.w_canon, inp.scales, K)
    scale = max(np.max(np.abs(ref)), 1e-300)
    assert np.max(np.abs(y - ref)) <= 1e-12 * scale


# Group sizes 32 and 64: the gfx1151 page benchmarks group_size=32 ("Benchmark
# results (per-GEMM)"); the scale of weight (n, k) is scale[n][k / G].
@pytest.mark.parametrize("G", [32, 64])
@pytest.mark.parametrize("M,N,K,seed", [(1, 16, 128, 0), (3, 33, 256, 1), (5, 7, 384, 2)])
def test_oracle_matches_numpy_bruteforce_small_groups(M, N, K, G, seed):
    inp = syn.make_gemm_inputs(M, N, K, G=G, seed=seed)
    assert inp.scales.shape == (N, K // G)
    y = oracle.gemm(inp.x, inp.w_canon, inp.scales, M, N, K, G=G)
    ref = np_gemm(inp.x, inp.w_canon, inp.scales, K, G)
    scale = max(np.max(np.abs(ref)), 1e-300)
    assert np.max(np.abs(y - ref)) <= 1e-12 * scale


@pytest.mark.parametrize("G", [32, 64])
def test_small_groups_with_repeated_scales_equal_128(G):
    # Every weight keeps its value when each 128-wide group's scale is repeated
    # over its 128 / G sub-groups, and the k order of the sum is unchanged: the
    # results agree bit for bit.
    M, N, K = 3, 24, 384
    inp = syn.make_gemm_inputs(M, N, K, seed=9)
    rep = np.repeat(inp.scales, 128 // G, axis=1)
    a = oracle.gemm(inp.x, inp.w_canon, inp.scales, M, N, K)
    b = oracle.gemm(inp.x, inp.w_canon, rep, M, N, K, G=G)
    assert np.array_equal(a, b)
    assert np.array_equal(oracle.dequant_f64(inp.w_canon, inp.scales, N, K),
                          oracle.dequant_f64(inp.w_canon, rep, N, K, G=G))


@pytest.mark.parametrize("G", [32, 64])
def test_one_hot_picks_the_sub_group_scale(G):
    # Distinct power-of-two scales per (row, group), X one-hot at k0:
    # Y[m][n] = 2^(e(n, k0 / G)) * (code(n, k0) - 8) exactly (closed form).
    M, N, K = 1, 12, 256
    inp = syn.make_gemm_inputs(M, N, K, G=G, seed=10)
    n_g = K // G
    e = (np.arange(N)[:, None] * 3 + np.arange(n_g)[None, :]) % 11 - 5      # exponents -5..5
    scales = ((127 + e) << 7).astype(np.uint16)                              # bf16 2^e
    codes = np_codes(inp.w_canon, K)
    for k0 in [0, G - 1, G, 2 * G + 5, K - 1]:
        x = np.zeros((M, K), dtype=np.uint16)
        x[0, k0] = 0x3F80
        y = oracle.gemm(x, inp.w_canon, scales, M, N, K, G=G)
        want = np.ldexp(1.0, e[:, k0 // G]) * (codes[:, k0] - 8)
        assert np.array_equal(y[0], want)


@pytest.mark.parametrize("G", [32, 64])
def test_grouped_small_groups_is_concatenation_of_plain(G):
    inp = syn.make_grouped_inputs(3, 40, 24, 256, G=G, seed=11)
    y = oracle.gemm_grouped(inp.x, inp.w_canon, inp.scales, inp.m_sizes, 40, 24, 256, G=G)
    starts = np.concatenate([[0], np.cumsum(inp.m_sizes)[:-1]])
    for g in range(3):
        r0, r1 = starts[g], starts[g] + inp.m_sizes[g]
        ref = np_gemm(inp.x[r0:r1], inp.w_canon[g], inp.scales[g], 256, G)
        assert np.max(np.abs(y[r0:r1] - ref)) <= 1e-12 * max(np.max(np.abs(ref)), 1e-300)


def test_oracle_dequant_matches_numpy():
    inp = syn.make_gemm_inputs(1, 40, 384, seed=3)
    d = oracle.dequant_f64(inp.w_canon, inp.scales, 40, 384)
    assert np.array_equal(d, np_dense(inp.w_canon, inp.scales, 384))


def test_oracle_gemm_cols_sample():
    inp = syn.make_gemm_inputs(2, 64, 256, seed=4)
    full = oracle.gemm(inp.x, inp.w_canon, inp.scales, 2, 64, 256)
    part = oracle.gemm_cols(inp.x, inp.w_canon, inp.scales, 2, 64, 256, 10, 30)
    assert np.array_equal(part[:, 10:30], full[:, 10:30])
    assert np.all(np.isnan(part[:, :10])) and np.all(np.isnan(part[:, 30:]))


def test_thread_count_does_not_change_result():
    inp = syn.make_gemm_inputs(3, 48, 256, seed=5)
    a = oracle.gemm(inp.x, inp.w_canon, inp.scales, 3, 48, 256, threads=1)
    b = oracle.gemm(inp.x, inp.w_canon, inp.scales, 3, 48, 256, threads=4)
    assert np.array_equal(a, b)


# ------------------------------------------------------------------ invariants
def test_all_eights_gives_zero():
    inp = syn.make_gemm_inputs(3, 20, 256, seed=6)
    w = np.full_like(inp.w_canon, 0x88)
    y = oracle.gemm(inp.x, w, inp.scales, 3, 20, 256)
    assert np.all(y == 0.0)


def test_unit_scales_one_hot_reproduces_codes():
    M, N, K = 4, 24, 256
    inp = syn.make_gemm_inputs(M, N, K, seed=7)
    ones = np.full_like(inp.scales, 0x3F80)
    codes = np_codes(inp.w_canon, K)
    for m, k0 in enumerate([0, 1, 130, 255]):
        x = np.zeros((M, K), dtype=np.uint16)
        x[m, k0] = 0x3F80
        y = oracle.gemm(x, inp.w_canon, ones, M, N, K)
        assert np.array_equal(y[m], (codes[:, k0] - 8).astype(np.float64))
        others = np.delete(y, m, axis=0)
        assert np.all(others == 0.0)


def test_scaling_scales_by_two_is_exact():
    inp = syn.make_gemm_inputs(2, 32, 384, seed=8)
    y = oracle.gemm(inp.x, inp.w_canon, inp.scales, 2, 32, 384)
    s2 = (inp.scales.astype(np.uint32) + 0x80).astype(np.uint16)    # exponent + 1
    y2 = oracle.gemm(inp.x, inp.w_canon, s2, 2, 32, 384)
    assert np.array_equal(y2, 2.0 * y)


def test_scaling_x_by_power_of_two_is_exact():
    inp = syn.make_gemm_inputs(2, 32, 256, seed=9)
    y = oracle.gemm(inp.x, inp.w_canon, inp.scales, 2, 32, 256)
    x4 = (inp.x.astype(np.uint32) + (2 << 7)).astype(np.uint16)     # exponent + 2
    y4 = oracle.gemm(x4, inp.w_canon, inp.scales, 2, 32, 256)
    assert np.array_equal(y4, 4.0 * y)


def test_linearity_in_x():
    M, N, K = 3, 16, 256
    inp = syn.make_gemm_inputs(M, N, K, seed=10)
    x1 = inp.x.copy()
    x2 = inp.x.copy()
    x1[:, 1::2] = 0
    x2[:, 0::2] = 0
    y = oracle.gemm(inp.x, inp.w_canon, inp.scales, M, N, K)
    y1 = oracle.gemm(x1, inp.w_canon, inp.scales, M, N, K)
    y2 = oracle.gemm(x2, inp.w_canon, inp.scales, M, N, K)
    assert np.max(np.abs(y - (y1 + y2))) <= 1e-13 * np.max(np.abs(y))


def test_linearity_in_scales():
    M, N, K = 2, 16, 384
    inp = syn.make_gemm_inputs(M, N, K, seed=11)
    s1 = inp.scales.copy()
    s2 = inp.scales.copy()
    s1[:, 1:] = 0
    s2[:, :1] = 0
    y = oracle.gemm(inp.x, inp.w_canon, inp.scales, M, N, K)
    y1 = oracle.gemm(inp.x, inp.w_canon, s1, M, N, K)
    y2 = oracle.gemm(inp.x, inp.w_canon, s2, M, N, K)
    assert np.max(np.abs(y - (y1 + y2))) <= 1e-13 * np.max(np.abs(y))


# --------------------------------------------------------------------- grouped
def test_grouped_one_group_is_plain():
    g = syn.make_grouped_inputs(1, 5, 24, 256, seed=12)
    yg = oracle.gemm_grouped(g.x, g.w_canon, g.scales, g.m_sizes, 5, 24, 256)
    yp = oracle.gemm(g.x, g.w_canon[0], g.scales[0], 5, 24, 256)
    assert np.array_equal(yg, yp)


def test_grouped_is_concatenation_of_plain():
    g = syn.make_grouped_inputs(4, 23, 16, 256, seed=13)
    yg = oracle.gemm_grouped(g.x, g.w_canon, g.scales, g.m_sizes, 23, 16, 256)
    starts = np.concatenate([[0], np.cumsum(g.m_sizes)[:-1]])
    for i in range(4):
        lo, hi = int(starts[i]), int(starts[i] + g.m_sizes[i])
        yp = oracle.gemm(g.x[lo:hi], g.w_canon[i], g.scales[i], hi - lo, 16, 256)
        assert np.array_equal(yg[lo:hi], yp)
        # and against the brute force
        ref = np_gemm(g.x[lo:hi], g.w_canon[i], g.scales[i], 256)
        assert np.max(np.abs(yg[lo:hi] - ref)) <= 1e-12 * max(np.max(np.abs(ref)), 1e-300)


def test_grouped_clamping_rules():
    g = syn.make_grouped_inputs(3, 10, 8, 128, seed=14, m_sizes=[4, -2, 9])
    y = oracle.gemm_grouped(g.x, g.w_canon, g.scales, g.m_sizes, 10, 8, 128)
    # group 1 is empty (negative -> 0), group 2 starts at 4 and is cut at M_total.
    ref0 = np_gemm(g.x[0:4], g.w_canon[0], g.scales[0], 128)
    ref2 = np_gemm(g.x[4:10], g.w_canon[2], g.scales[2], 128)
    assert np.allclose(y[0:4], ref0, rtol=0, atol=1e-12)
    assert np.allclose(y[4:10], ref2, rtol=0, atol=1e-12)
    h = syn.make_grouped_inputs(2, 10, 8, 128, seed=15, m_sizes=[3, 4])
    yh = oracle.gemm_grouped(h.x, h.w_canon, h.scales, h.m_sizes, 10, 8, 128)
    assert np.all(np.isnan(yh[7:]))        # rows no group covers are untouched


def test_multinomial_group_sizes():
    g = syn.make_grouped_inputs(8, 4096, 16, 128, seed=0)
    assert int(g.m_sizes.sum()) == 4096 and np.all(g.m_sizes > 0)


# ---------------------------------------------------------- dequant exhaustive
def _all_scale_patterns(lo=0.005, hi=0.02):
    bits = np.arange(0x0080, 0x7F80, dtype=np.uint16)          # positive normals
    vals = np_bf16(bits)
    rng_bits = bits[(vals >= lo) & (vals <= hi)]
    return bits, rng_bits


def test_dequant_exact_all_codes_and_scales():
    all_bits, _ = _all_scale_patterns()
    # every positive normal bf16 below 2^120 (products stay finite in binary32)
    scales = all_bits[np_bf16(all_bits) < 2.0 ** 120].reshape(-1, 1)
    N, K = scales.shape[0], 128
    codes = np.tile(np.arange(16, dtype=np.uint8), (N, K // 16))
    w = syn.pack_codes(codes)
    d32 = oracle.dequant_f32(w, scales, N, K)
    expect = np_bf16(scales) * (codes.astype(np.float64) - 8.0)
    assert np.array_equal(d32.astype(np.float64), expect)        # binary32 holds it exactly


def _independent_bf16_rne(v):
    """RNE to bf16 for values exact in binary32 (by neighbour comparison)."""
    f = np.asarray(v, dtype=np.float32)
    u = f.view(np.uint32)
    lo = (u >> 16).astype(np.uint32)
    lo_val = (lo << 16).view(np.float32).astype(np.float64)
    hi = lo + 1
    hi_val = (hi << 16).view(np.float32).astype(np.float64)
    x = f.astype(np.float64)
    dlo = np.abs(x - lo_val)
    dhi = np.abs(hi_val - x)
    pick_hi = (dhi < dlo) | ((dhi == dlo) & ((lo & 1) == 1))
    return np.where(pick_hi, hi, lo).astype(np.uint16)


def test_dequant_bf16_rounding_all_codes_and_scales():
    _, scales = _all_scale_patterns()
    scales = scales.reshape(-1, 1)
    N, K = scales.shape[0], 128
    codes = np.tile(np.arange(16, dtype=np.uint8), (N, K // 16))
    w = syn.pack_codes(codes)
    got = oracle.dequant_bf16(w, scales, N, K)
    prod = np_bf16(scales) * (codes.astype(np.float64) - 8.0)
    assert np.array_equal(got, _independent_bf16_rne(prod))


def test_sum_slices_order():
    ws = np.array([[1e8, 1.0], [1.0, 2.0], [-1e8, 3.0]], dtype=np.float32)
    out = oracle.sum_slices(ws)
    assert out[0] == 1.0 and out[1] == 6.0


# -------------------------------------------------------------- mutation pins
MUTANTS = {
    "swap_nibbles": ("(k % 2 == 0) ? (byte & 0x0F) : (byte >> 4)",
                     "(k % 2 == 0) ? (byte >> 4) : (byte & 0x0F)"),
    "offset_7": ("oracle_nibble(w_canon, K, n, k) - 8", "oracle_nibble(w_canon, K, n, k) - 7"),
    "group_index": ("scales[n * (K / G) + k / G]", "scales[n * (K / G) + k / (2 * G)]"),
    "group_fixed_128": ("scales[n * (K / G) + k / G]", "scales[n * (K / G) + k / 128]"),
    "dropped_term": ("for (long k = 0; k < K; ++k)\n                acc += oracle_bf16_to_f64(x[m * K + k])",
                     "for (long k = 1; k < K; ++k)\n                acc += oracle_bf16_to_f64(x[m * K + k])"),
    "sign": ("acc += oracle_bf16_to_f64(x[m * K + k]) *\n                       oracle_weight(w_canon",
             "acc -= oracle_bf16_to_f64(x[m * K + k]) *\n                       oracle_weight(w_canon"),
    "transposed_x": ("oracle_bf16_to_f64(x[m * K + k]) *\n                       oracle_weight(w_canon",
                     "oracle_bf16_to_f64(x[(k % M) * K + (m % K)]) *\n                       oracle_weight(w_canon"),
}


def _build_mutant(tmp_path, name):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = MUTANTS[name]
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    src = src.replace(old, new, 1)
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(src)
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", str(c), "-o", str(so), "-lm"],
                   check=True)
    lib = ctypes.CDLL(str(so))
    P, L, I = ctypes.c_void_p, ctypes.c_long, ctypes.c_int
    lib.oracle_gemm_f64.argtypes = [P, P, P, L, L, L, L, P, I]
    lib.oracle_nibble.argtypes = [P, L, L, L]
    lib.oracle_nibble.restype = I
    return lib


def _mutant_fails_pins(lib):
    def gemm(x, w, s, M, N, K, G=128):
        y = np.zeros((M, N))
        lib.oracle_gemm_f64(x.ctypes.data_as(ctypes.c_void_p), w.ctypes.data_as(ctypes.c_void_p),
                            s.ctypes.data_as(ctypes.c_void_p), M, N, K, G,
                            y.ctypes.data_as(ctypes.c_void_p), 1)
        return y
    # pin 1: golden nibble order
    rows = [r.split() for r in read_rows("nibble_order.txt")]
    b = np.array([[int(r[0], 16) for r in rows]], dtype=np.uint8)
    for j, r in enumerate(rows):
        if lib.oracle_nibble(b.ctypes.data_as(ctypes.c_void_p), 2 * b.shape[1], 0, 2 * j) != int(r[1]):
            return True
    # pin 2: brute force on a small shape, at group sizes 128 and 32
    for G in (128, 32):
        inp = syn.make_gemm_inputs(3, 16, 256, G=G, seed=21)
        y = gemm(inp.x, inp.w_canon, inp.scales, 3, 16, 256, G)
        ref = np_gemm(inp.x, inp.w_canon, inp.scales, 256, G)
        if not (np.max(np.abs(y - ref)) <= 1e-12 * np.max(np.abs(ref))):
            return True
    return False


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(tmp_path, name):
    lib = _build_mutant(tmp_path, name)
    assert _mutant_fails_pins(lib), f"planted mistake {name} slipped through the pins"


# ------------------------------------------------------- zero points (variant)
def np_gemm_zp(x, w_canon, scales, zeros, K, G):
    s = np.repeat(np_bf16(scales), G, axis=-1)
    z = np.repeat((zeros & 0x0F).astype(np.int64), G, axis=-1)
    return np_bf16(x) @ (s * (np_codes(w_canon, K) - z).astype(np.float64)).T


@pytest.mark.parametrize("G", [128, 64, 32])
@pytest.mark.parametrize("M,N,K,seed", [(1, 16, 128, 0), (3, 33, 256, 1), (5, 7, 384, 2)])
def test_oracle_zp_matches_numpy_bruteforce(M, N, K, G, seed):
    inp = syn.make_gemm_inputs(M, N, K, G=G, seed=seed)
    z = syn.make_zeros(N, K, G, seed=seed)
    y = oracle.gemm_zp(inp.x, inp.w_canon, inp.scales, z, M, N, K, G=G)
    ref = np_gemm_zp(inp.x, inp.w_canon, inp.scales, z, K, G)
    assert np.max(np.abs(y - ref)) <= 1e-12 * max(np.max(np.abs(ref)), 1e-300)


@pytest.mark.parametrize("G", [128, 32])
def test_zero_point_eight_is_symmetric(G):
    inp = syn.make_gemm_inputs(3, 40, 384, G=G, seed=13)
    eights = np.full((40, 384 // G), 8, dtype=np.uint8)
    assert np.array_equal(oracle.gemm_zp(inp.x, inp.w_canon, inp.scales, eights, 3, 40, 384, G=G),
                          oracle.gemm(inp.x, inp.w_canon, inp.scales, 3, 40, 384, G=G))


def test_zero_point_one_hot_closed_form():
    # Unit scales, X one-hot at k0: Y[m][n] = code(n, k0) - z(n, k0 / G) exactly.
    M, N, K, G = 1, 20, 256, 32
    inp = syn.make_gemm_inputs(M, N, K, G=G, seed=14)
    z = syn.make_zeros(N, K, G, seed=14)
    ones = np.full_like(inp.scales, 0x3F80)
    codes = np_codes(inp.w_canon, K)
    for k0 in [0, 31, 32, 100, 255]:
        x = np.zeros((M, K), dtype=np.uint16)
        x[0, k0] = 0x3F80
        y = oracle.gemm_zp(x, inp.w_canon, ones, z, M, N, K, G=G)
        assert np.array_equal(y[0], (codes[:, k0] - z[:, k0 // G]).astype(np.float64))


def test_codes_equal_to_zero_point_give_zero():
    inp = syn.make_gemm_inputs(2, 24, 256, seed=15)
    for zval in (0, 3, 15):
        w = np.full_like(inp.w_canon, zval * 0x11)
        z = np.full((24, 2), zval, dtype=np.uint8)
        assert np.all(oracle.gemm_zp(inp.x, w, inp.scales, z, 2, 24, 256) == 0.0)


def test_zero_point_high_bits_ignored():
    inp = syn.make_gemm_inputs(2, 24, 256, G=64, seed=16)
    z = syn.make_zeros(24, 256, 64, seed=16)
    a = oracle.gemm_zp(inp.x, inp.w_canon, inp.scales, z, 2, 24, 256, G=64)
    b = oracle.gemm_zp(inp.x, inp.w_canon, inp.scales, z | 0xF0, 2, 24, 256, G=64)
    assert np.array_equal(a, b)


def test_dequant_zp_matches_numpy():
    inp = syn.make_gemm_inputs(1, 40, 384, G=32, seed=17)
    z = syn.make_zeros(40, 384, 32, seed=17)
    d = oracle.dequant_zp_f32(inp.w_canon, inp.scales, z, 40, 384, G=32)
    s = np.repeat(np_bf16(inp.scales), 32, axis=-1)
    ref = s * (np_codes(inp.w_canon, 384) - np.repeat(z.astype(np.int64), 32, axis=-1))
    assert np.array_equal(d.astype(np.float64), ref)
    b = oracle.dequant_zp_bf16(inp.w_canon, inp.scales, z, 40, 384, G=32)
    assert np.array_equal(b, np.vectorize(oracle.f64_to_bf16)(ref).astype(np.uint16))


ZP_MUTANTS = {
    "zero_ignored": ("- (int)(zeros[gi] & 0x0F)", "- 8"),
    "zero_sign": ("(oracle_nibble(w_canon, K, n, k) - (int)(zeros[gi] & 0x0F))",
                  "(oracle_nibble(w_canon, K, n, k) + (int)(zeros[gi] & 0x0F))"),
    "zero_index": ("long gi = n * (K / G) + k / G;", "long gi = n * (K / G) + k / (2 * G);"),
}


@pytest.mark.parametrize("name", sorted(ZP_MUTANTS))
def test_planted_zero_point_mistake_is_caught(tmp_path, name):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    old, new = ZP_MUTANTS[name]
    assert src.count(old) == 1, f"mutation site for {name} not found"
    c = tmp_path / f"{name}.c"
    so = tmp_path / f"{name}.so"
    c.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-O1", "-fopenmp", "-fPIC", "-shared", str(c), "-o", str(so), "-lm"],
                   check=True)
    lib = ctypes.CDLL(str(so))
    P, L, I = ctypes.c_void_p, ctypes.c_long, ctypes.c_int
    lib.oracle_gemm_zp_f64.argtypes = [P, P, P, P, L, L, L, L, P, I]
    M, N, K, G = 3, 16, 256, 32
    inp = syn.make_gemm_inputs(M, N, K, G=G, seed=22)
    z = syn.make_zeros(N, K, G, seed=22)
    y = np.zeros((M, N))
    lib.oracle_gemm_zp_f64(*(a.ctypes.data_as(P) for a in (inp.x, inp.w_canon, inp.scales, z)),
                           M, N, K, G, y.ctypes.data_as(P), 1)
    ref = np_gemm_zp(inp.x, inp.w_canon, inp.scales, z, K, G)
    assert not np.max(np.abs(y - ref)) <= 1e-12 * np.max(np.abs(ref)), f"{name} slipped through"
