"""The C ABI library loads, exports what include/w4a16.h declares, and rejects
bad arguments on the host before touching CUDA (no GPU needed)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

from bf16_activation_quantized_gb300 import _lib
from bf16_activation_quantized_gb300 import build as build_mod

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "w4a16.h")

OK, INVALID, UNSUPPORTED, WS_SMALL, CUDA_ERR = 0, 1, 2, 3, 4


@pytest.fixture(scope="module")
def L():
    build_mod.build()
    return _lib.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(w4a16_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("w4a16_gemm", "w4a16_gemm_grouped", "w4a16_pack_weights",
                     "w4a16_dequant_fp32", "w4a16_splitk_reduce"):
        assert required in names


def test_every_declared_symbol_is_exported(L):
    for name in declared_functions():
        assert hasattr(L, name), f"{name} declared in w4a16.h but not exported"


def test_binding_covers_the_header():
    assert sorted(_lib.SIGNATURES) == declared_functions()


def test_library_does_not_need_libcudart_or_libcuda(L):
    # The runtime is linked statically and the driver is opened lazily, so the
    # library loads on a machine without a GPU.
    maps = open("/proc/self/maps").read()
    assert "libw4a16.so" in maps


def test_host_only_queries(L):
    assert L.w4a16_layout_version() == 2
    assert L.w4a16_packed_weight_bytes(8192, 8192) == 8192 * 4096
    assert L.w4a16_packed_weight_bytes(200, 256) == 256 * 128      # rows padded to 128
    assert L.w4a16_packed_weight_bytes(1, 128) == 128 * 64
    assert L.w4a16_packed_weight_bytes(0, 128) == 0
    assert L.w4a16_packed_weight_bytes(16, 100) == 0
    assert L.w4a16_packed_weight_bytes(16, 64) == 0
    for code in range(5):
        assert L.w4a16_status_string(code)
    assert L.w4a16_status_string(99) == b"unknown status"


FAKE = 0x10000  # a 16-byte-aligned non-null address; never dereferenced on these paths


def gemm(L, X=FAKE, W=FAKE, S=FAKE, Y=FAKE, M=4, N=256, K=512, G=128, ws=None, wsb=0):
    return L.w4a16_gemm(X, W, S, Y, M, N, K, G, ws, wsb, None)


def test_gemm_argument_checks(L):
    # group sizes 128, 64 and 32 are served (M == 0 needs no device); others are not
    for G in (128, 64, 32):
        assert gemm(L, M=0, G=G) == OK
    for G in (16, 96, 256, 0, -128):
        assert gemm(L, G=G) == UNSUPPORTED
    assert gemm(L, K=500) == INVALID
    assert gemm(L, K=0) == INVALID
    assert gemm(L, K=64) == INVALID
    assert gemm(L, N=0) == INVALID
    assert gemm(L, M=-1) == INVALID
    assert gemm(L, X=None) == INVALID
    assert gemm(L, W=None) == INVALID
    assert gemm(L, S=None) == INVALID
    assert gemm(L, Y=None) == INVALID
    assert gemm(L, X=FAKE + 8) == INVALID       # X must be 16-byte aligned
    assert gemm(L, W=FAKE + 4) == INVALID       # W must be 16-byte aligned
    assert gemm(L, Y=FAKE + 1) == INVALID       # Y must be 2-byte aligned
    assert gemm(L, S=FAKE + 1) == INVALID
    # M == 0 is a no-op that succeeds without any CUDA call, even with null pointers.
    assert gemm(L, M=0, X=None, Y=None) == OK


def test_other_entry_points_check_arguments(L):
    assert L.w4a16_pack_weights(None, FAKE, 16, 128, None) == INVALID
    assert L.w4a16_pack_weights(FAKE, FAKE, 16, 100, None) == INVALID
    assert L.w4a16_pack_weights(FAKE, FAKE + 8, 16, 128, None) == INVALID
    assert L.w4a16_dequant_fp32(FAKE, FAKE, None, 16, 128, 128, None) == INVALID
    assert L.w4a16_dequant_fp32(FAKE, FAKE, FAKE, 16, 128, 256, None) == UNSUPPORTED
    assert L.w4a16_dequant_fp32(FAKE, FAKE, FAKE, 16, 128, 48, None) == UNSUPPORTED
    assert L.w4a16_dequant_bf16(None, FAKE, FAKE, 16, 128, 128, None) == INVALID
    assert L.w4a16_splitk_reduce(None, FAKE, 2, 4, 4, None) == INVALID
    assert L.w4a16_splitk_reduce(FAKE, FAKE, 0, 4, 4, None) == INVALID
    assert L.w4a16_splitk_reduce(FAKE + 4, FAKE, 2, 4, 4, None) == INVALID
    assert L.w4a16_splitk_reduce(FAKE, FAKE, 2, 0, 4, None) == OK
    nb = ctypes.c_size_t(0)
    assert L.w4a16_grouped_workspace_bytes(8, 4096, 2048, 4096, 128, ctypes.byref(nb)) == OK
    assert nb.value >= 4
    assert L.w4a16_grouped_workspace_bytes(0, 4096, 2048, 4096, 128, ctypes.byref(nb)) == INVALID
    assert L.w4a16_grouped_workspace_bytes(8, 4096, 2048, 4096, 256, ctypes.byref(nb)) == UNSUPPORTED
    assert L.w4a16_grouped_workspace_bytes(8, 4096, 2048, 4096, 32, ctypes.byref(nb)) == OK
    assert L.w4a16_workspace_bytes(1, 256, 512, 128, None) == INVALID
    assert L.w4a16_gemm_grouped(None, FAKE, FAKE, FAKE, FAKE, 8, 64, 256, 512, 128, FAKE, 16,
                                None) == INVALID


def test_plan_without_a_gpu_reports_cuda_error(L):
    # Planning needs the device's SM count; with no GPU that is a CUDA error, not a crash.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        pytest.skip("a GPU is present")
    info = _lib.PlanInfo()
    assert L.w4a16_plan(1, 256, 512, 128, None, ctypes.byref(info)) == CUDA_ERR


def test_options_are_checked_before_the_device_is_queried(L):
    # Unknown flag bits, bad arms and bad tile sizes are host-side errors.
    info = _lib.PlanInfo()
    for o, want in ((_lib.Options(0, 0, 0, 32), INVALID), (_lib.Options(0, 0, 0, 1 << 30), INVALID),
                    (_lib.Options(0, 0, 0, 16 | 2), UNSUPPORTED),
                    (_lib.Options(0, 0, 0, 2 | 4), INVALID),
                    (_lib.Options(7, 0, 0, 0), INVALID), (_lib.Options(0, -1, 0, 0), INVALID),
                    (_lib.Options(2, 0, 48, 0), UNSUPPORTED)):
        assert L.w4a16_plan(1, 256, 512, 128, ctypes.byref(o), ctypes.byref(info)) == want


def test_header_flag_values_match_the_binding():
    import bf16_activation_quantized_gb300 as w4
    text = open(HEADER).read()
    for name, value in (("RESIDENT_WEIGHTS", 1), ("DECODE_WHOLE_K", 2), ("DECODE_K_SLICES", 4),
                        ("ZERO_POINTS", 8), ("TEST_STALL", 16)):
        assert re.search(rf"W4A16_FLAG_{name}\s*=\s*{value}\b", text)
        assert getattr(w4, f"FLAG_{name}") == value


def test_batched_entry_points_check_arguments(L):
    info = _lib.PlanInfo()
    for batch in (0, -1, 1025):
        assert L.w4a16_plan_batched(batch, 4, 256, 512, 128, None, ctypes.byref(info)) == INVALID
    assert L.w4a16_plan_batched(2, 4, 256, 512, 256, None, ctypes.byref(info)) == UNSUPPORTED
    assert L.w4a16_plan_batched(2, 4, 256, 500, 128, None, ctypes.byref(info)) == INVALID
    # batch * M beyond 2^24 rows
    assert L.w4a16_plan_batched(1024, 1 << 15, 256, 512, 128, None, ctypes.byref(info)) == INVALID
    FAKE = 1 << 20
    assert L.w4a16_gemm_batched(None, FAKE, FAKE, FAKE, 2, 4, 256, 512, 128, None, 0, None, None) == INVALID
    assert L.w4a16_gemm_batched(FAKE, FAKE, FAKE, FAKE, 0, 4, 256, 512, 128, None, 0, None, None) == INVALID
    # M == 0: nothing to do, nothing launched, no GPU needed
    assert L.w4a16_gemm_batched(None, None, None, None, 2, 0, 256, 512, 128, None, 0, None, None) == OK


def test_zero_point_entry_points_check_arguments(L):
    FAKE = 1 << 20
    zp = _lib.Options(0, 0, 0, 8)
    # zeros are required; the flag alone (without a zeros pointer) is refused
    assert L.w4a16_gemm_zp(FAKE, FAKE, FAKE, None, FAKE, 4, 256, 512, 128, None, 0, None, None) == INVALID
    assert L.w4a16_gemm_ex(FAKE, FAKE, FAKE, FAKE, 4, 256, 512, 128, None, 0, ctypes.byref(zp),
                           None) == INVALID
    assert L.w4a16_gemm_zp(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 512, 256, None, 0, None, None) == UNSUPPORTED
    assert L.w4a16_gemm_zp(FAKE, FAKE, FAKE, FAKE, FAKE, 4, 256, 500, 128, None, 0, None, None) == INVALID
    assert L.w4a16_gemm_zp(None, None, None, None, None, 0, 256, 512, 32, None, 0, None, None) == OK
    # the batched and grouped forms also require their zeros pointer
    assert L.w4a16_gemm_batched_zp(FAKE, FAKE, FAKE, None, FAKE, 2, 4, 256, 512, 128, None, 0, None,
                                   None) == INVALID
    assert L.w4a16_gemm_grouped_zp(FAKE, FAKE, FAKE, None, FAKE, FAKE, 8, 64, 256, 512, 128, FAKE, 16,
                                   None) == INVALID
    assert L.w4a16_dequant_zp_fp32(FAKE, FAKE, None, FAKE, 16, 128, 128, None) == INVALID
    assert L.w4a16_dequant_zp_bf16(FAKE, FAKE, FAKE, FAKE, 16, 128, 48, None) == UNSUPPORTED


def test_python_binding_refuses_cpu_tensors():
    # No CPU path: host tensors are an error before any library call.
    import torch
    import bf16_activation_quantized_gb300 as w4
    x = torch.zeros(2, 256, dtype=torch.bfloat16)
    wp = torch.zeros(256 * 128, dtype=torch.uint8)
    s = torch.zeros(256, 2, dtype=torch.bfloat16)
    for call in (lambda: w4.gemm(x, wp, s),
                 lambda: w4.gemm(x, wp, s, zeros=torch.zeros(256, 2, dtype=torch.uint8)),
                 lambda: w4.pack(torch.zeros(256, 128, dtype=torch.uint8)),
                 lambda: w4.dequant_fp32(wp, s),
                 lambda: w4.gemm_batched(x[None], wp[None], s[None])):
        with pytest.raises(ValueError):
            call()


def test_binding_fails_loudly_without_the_library(tmp_path, monkeypatch):
    from bf16_activation_quantized_gb300 import _lib as lib_mod
    monkeypatch.setattr(lib_mod, "_lib", None)
    monkeypatch.setattr(lib_mod, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        lib_mod.lib()


def test_header_error_bits_match_the_binding():
    import bf16_activation_quantized_gb300 as w4
    text = open(HEADER).read()
    assert re.search(r"W4A16_ERROR_WAIT_TIMEOUT\s*=\s*1\b", text)
    assert w4.ERROR_WAIT_TIMEOUT == 1


def test_read_error_word_checks_its_pointer(L):
    # A null output pointer is refused before the device is touched.
    assert L.w4a16_read_error_word(None, 0) == INVALID
