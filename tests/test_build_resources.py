"""Resource report of the sm_103a build (ptxas -v, kept in _build/ptxas.log by
the build): the kernels on the measured paths must not spill and must fit the
occupancy their launches are sized for -- a build-level guard against
performance regressions, checked without a GPU."""
from __future__ import annotations

import os
import re

import pytest

from bf16_activation_quantized_gb300 import build as build_mod


@pytest.fixture(scope="module")
def report():
    build_mod.build()
    path = os.path.join(build_mod.BUILD, "ptxas.log")
    if not os.path.exists(path):      # a library built before the log existed
        build_mod.build(force=True)
    text = open(path).read()
    out = {}
    name = None
    for line in text.splitlines():
        m = re.search(r"Compiling entry function '(\S+)'", line)
        if m:
            name = m.group(1)
            continue
        if name and "spill stores" in line:
            out.setdefault(name, {})["spill"] = int(re.search(r"(\d+) bytes spill stores", line).group(1))
        if name and re.search(r"Used \d+ registers", line):
            out.setdefault(name, {})["regs"] = int(re.search(r"Used (\d+) registers", line).group(1))
            name = None
    assert out, "no kernels in the ptxas report"
    return out


def find(report, pattern):
    hits = {k: v for k, v in report.items() if re.search(pattern, k)}
    assert hits, f"no kernel matches {pattern}"
    return hits


def _source_int(path, name):
    text = open(os.path.join(build_mod.CSRC, path)).read()
    return int(re.search(rf"constexpr int {name} = (\d+);", text).group(1))


def tensor_threads(sep):
    # Dequantiser teams of four warps, the two producers and the MMA issuer,
    # plus the epilogue warps of the separate-epilogue form.
    teams = _source_int("internal.h", "kTensorTeamsSep" if sep else "kTensorTeamsPlain")
    team_warps = _source_int("tensor.cu", "kTcTeamWarps")
    epi_warps = _source_int("tensor.cu", "kTcEpiWarps") if sep else 0
    return (team_warps * teams + 3 + epi_warps) * 32


@pytest.mark.parametrize("gps", [4, 8])
def test_headline_decode_kernels_do_not_spill(report, gps):
    # decode_kernel<MT=1, GPS, split, SUB=1>: the decode GEMV step's two launches
    for name, r in find(report, rf"13decode_kernelILi1ELi{gps}ELb1ELi1E").items():
        assert r["spill"] == 0, name
        assert fits(r["regs"], 2 * 9), name    # two 288-thread CTAs per SM


def fits(regs, warps_per_sm):
    # Each of the SM's four sub-partitions holds 16384 registers for the
    # warps placed on it (up to ceil(warps / 4)); a warp's registers are
    # granted in units of 256.
    per_warp = -(-regs * 32 // 256) * 256
    return -(-warps_per_sm // 4) * per_warp <= 16384


def test_every_decode_kernel_fits_two_ctas_per_sm(report):
    # eight consumer warps and a producer warp, two CTAs per SM
    warps = {"slices": _source_int("decode_slices.cuh", "kDecodeWarps") + 1,
             "rows": _source_int("decode_rows.cu", "kRowsWarps") + 1}
    assert warps == {"slices": 9, "rows": 9}
    for kind, pattern in (("slices", r"decode_(zp_)?kernel"), ("rows", r"decode_rows_kernel")):
        for name, r in find(report, pattern).items():
            assert fits(r["regs"], 2 * warps[kind]), name


def test_symmetric_decode_kernels_do_not_spill(report):
    # every symmetric K-slice form and the whole-K kernel; the zero-point
    # forms may spill a few bytes at the two-CTA register cap
    for name, r in find(report, r"13decode_kernel|decode_rows_kernel").items():
        assert r["spill"] == 0, name


def test_tensor_thread_counts():
    assert (tensor_threads(False), tensor_threads(True)) == (608, 480)


def test_tensor_kernels_fit_their_occupancy(report):
    # one CTA per SM
    for name, r in find(report, r"tc_gemm_(zp_)?kernel").items():
        sep = re.search(r"tc_gemm_kernelILb[01]ELb1E|tc_gemm_zp_kernelILb[01]ELb1E", name) is not None
        assert fits(r["regs"], tensor_threads(sep) // 32), name


def test_prefill_tensor_kernels_do_not_spill(report):
    # the symmetric kernels at 128-column groups (prefill, grouped, batched)
    for name, r in find(report, r"tc_gemm_kernelILb[01]ELb[01]ELb[01]ELi1E").items():
        assert r["spill"] == 0, name
