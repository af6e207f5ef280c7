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


@pytest.mark.parametrize("gps", [4, 8])
def test_headline_decode_kernels_do_not_spill(report, gps):
    # decode_kernel<MT=1, GPS, split, SUB=1>: the decode GEMV step's two launches
    for name, r in find(report, rf"13decode_kernelILi1ELi{gps}ELb1ELi1E").items():
        assert r["spill"] == 0, name
        assert r["regs"] <= 112, name          # two 288-thread CTAs per SM


def test_every_decode_kernel_fits_two_ctas_per_sm(report):
    for name, r in find(report, r"decode_(zp_)?kernel|decode_wk_kernel").items():
        assert r["regs"] * 288 * 2 <= 65536, name


def test_tensor_kernels_fit_their_occupancy(report):
    for name, r in find(report, r"tc_gemm_(zp_)?kernel").items():
        sep = re.search(r"tc_gemm_kernelILb[01]ELb1E|tc_gemm_zp_kernelILb[01]ELb1E", name) is not None
        threads, ctas = (448, 1) if sep else (320, 2)
        assert r["regs"] * threads * ctas <= 65536, name


def test_prefill_tensor_kernels_do_not_spill(report):
    # the symmetric kernels at 128-column groups (prefill, grouped, batched)
    for name, r in find(report, r"tc_gemm_kernelILb[01]ELb[01]ELb[01]ELi1E").items():
        assert r["spill"] == 0, name
