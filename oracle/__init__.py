"""CPU fp64 oracle for the W4A16 skinny GEMM -- test infrastructure only.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The product path (the CUDA library and its
Python binding) never does, and the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over output
elements); this module only compiles it with gcc and marshals NumPy arrays
through ctypes.  Every function follows the definition of the op:
``Y = X . dequant(W)^T`` with ``dequant(W)[n, k] = scale[n, k // G] * (nib - 8)``
("[ROCm][Kernel] W4A16 skinny GEMM: hand-asm kernel for gfx1151", section 1
"Magic-constant bf16 dequant"; nibble order from "Add Triton BF16xINT4 rowwise
GEMM for ROCm gfx942/gfx950", "Implementation", "Fused A-operand dot"; group
row starts from its "Native fused grouped kernel" paragraph).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, -fopenmp)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        L = ctypes.c_long
        I = ctypes.c_int
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_f64.restype = ctypes.c_double
        lib.oracle_f64_to_bf16.argtypes = [ctypes.c_double]
        lib.oracle_f64_to_bf16.restype = ctypes.c_uint16
        lib.oracle_nibble.argtypes = [P, L, L, L]
        lib.oracle_nibble.restype = I
        lib.oracle_weight.argtypes = [P, P, L, L, L, L]
        lib.oracle_weight.restype = ctypes.c_double
        for name in ("oracle_dequant_f64", "oracle_dequant_f32", "oracle_dequant_bf16"):
            getattr(lib, name).argtypes = [P, P, L, L, L, P]
            getattr(lib, name).restype = None
        lib.oracle_gemm_f64.argtypes = [P, P, P, L, L, L, L, P, I]
        lib.oracle_gemm_f64.restype = None
        lib.oracle_gemm_cols_f64.argtypes = [P, P, P, L, L, L, L, L, L, P, I]
        lib.oracle_gemm_cols_f64.restype = None
        lib.oracle_group_starts.argtypes = [P, L, P]
        lib.oracle_group_starts.restype = None
        lib.oracle_gemm_grouped_f64.argtypes = [P, P, P, P, L, L, L, L, L, P, I]
        lib.oracle_gemm_grouped_f64.restype = None
        lib.oracle_sum_slices_f64.argtypes = [P, L, L, P]
        lib.oracle_sum_slices_f64.restype = None
        lib.oracle_weight_zp.argtypes = [P, P, P, L, L, L, L]
        lib.oracle_weight_zp.restype = ctypes.c_double
        for name in ("oracle_dequant_zp_f32", "oracle_dequant_zp_bf16"):
            getattr(lib, name).argtypes = [P, P, P, L, L, L, P]
            getattr(lib, name).restype = None
        lib.oracle_gemm_zp_f64.argtypes = [P, P, P, P, L, L, L, L, P, I]
        lib.oracle_gemm_zp_f64.restype = None
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = I
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a):
    return np.ascontiguousarray(a, dtype=np.uint16)


def _u8(a):
    return np.ascontiguousarray(a, dtype=np.uint8)


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def bf16_to_f64(bits: int) -> float:
    return float(_load().oracle_bf16_to_f64(int(bits)))


def f64_to_bf16(value: float) -> int:
    return int(_load().oracle_f64_to_bf16(float(value)))


def nibble(w_canon: np.ndarray, K: int, n: int, k: int) -> int:
    w = _u8(w_canon)
    return int(_load().oracle_nibble(_ptr(w), K, n, k))


def dequant_f64(w_canon, scales, N, K, G=128) -> np.ndarray:
    w, s = _u8(w_canon), _u16(scales)
    out = np.empty((N, K), dtype=np.float64)
    _load().oracle_dequant_f64(_ptr(w), _ptr(s), N, K, G, _ptr(out))
    return out


def dequant_f32(w_canon, scales, N, K, G=128) -> np.ndarray:
    w, s = _u8(w_canon), _u16(scales)
    out = np.empty((N, K), dtype=np.float32)
    _load().oracle_dequant_f32(_ptr(w), _ptr(s), N, K, G, _ptr(out))
    return out


def dequant_bf16(w_canon, scales, N, K, G=128) -> np.ndarray:
    """bf16 bit patterns of round-to-nearest-even(scale * (nib - 8))."""
    w, s = _u8(w_canon), _u16(scales)
    out = np.empty((N, K), dtype=np.uint16)
    _load().oracle_dequant_bf16(_ptr(w), _ptr(s), N, K, G, _ptr(out))
    return out


def gemm(x, w_canon, scales, M, N, K, G=128, threads: int = 0) -> np.ndarray:
    """Y[M, N] in fp64; x holds bf16 bit patterns [M, K]."""
    x, w, s = _u16(x), _u8(w_canon), _u16(scales)
    y = np.zeros((M, N), dtype=np.float64)
    _load().oracle_gemm_f64(_ptr(x), _ptr(w), _ptr(s), M, N, K, G, _ptr(y), threads)
    return y


def gemm_cols(x, w_canon, scales, M, N, K, n_lo, n_hi, G=128, threads: int = 0) -> np.ndarray:
    """Columns [n_lo, n_hi) of Y (the rest stay NaN): a bounded sample."""
    x, w, s = _u16(x), _u8(w_canon), _u16(scales)
    y = np.full((M, N), np.nan, dtype=np.float64)
    _load().oracle_gemm_cols_f64(_ptr(x), _ptr(w), _ptr(s), M, N, K, G, n_lo, n_hi,
                                 _ptr(y), threads)
    return y


def gemm_zp(x, w_canon, scales, zeros, M, N, K, G=128, threads: int = 0) -> np.ndarray:
    """Y[M, N] in fp64 with a zero point per scale group:
    dequant = scale[n, k // G] * (nib - (zeros[n, k // G] & 15)); zeros uint8 [N, K/G]."""
    x, w, s, z = _u16(x), _u8(w_canon), _u16(scales), _u8(zeros)
    y = np.zeros((M, N), dtype=np.float64)
    _load().oracle_gemm_zp_f64(_ptr(x), _ptr(w), _ptr(s), _ptr(z), M, N, K, G, _ptr(y), threads)
    return y


def dequant_zp_f32(w_canon, scales, zeros, N, K, G=128) -> np.ndarray:
    w, s, z = _u8(w_canon), _u16(scales), _u8(zeros)
    out = np.empty((N, K), dtype=np.float32)
    _load().oracle_dequant_zp_f32(_ptr(w), _ptr(s), _ptr(z), N, K, G, _ptr(out))
    return out


def dequant_zp_bf16(w_canon, scales, zeros, N, K, G=128) -> np.ndarray:
    """bf16 bit patterns of round-to-nearest-even(scale * (nib - zero))."""
    w, s, z = _u8(w_canon), _u16(scales), _u8(zeros)
    out = np.empty((N, K), dtype=np.uint16)
    _load().oracle_dequant_zp_bf16(_ptr(w), _ptr(s), _ptr(z), N, K, G, _ptr(out))
    return out


def group_starts(m_sizes) -> np.ndarray:
    ms = np.ascontiguousarray(m_sizes, dtype=np.int32)
    out = np.empty(ms.shape[0], dtype=np.int64)
    _load().oracle_group_starts(_ptr(ms), ms.shape[0], _ptr(out))
    return out


def gemm_grouped(x, w_canon, scales, m_sizes, M_total, N, K, G=128, threads: int = 0,
                 fill: float = np.nan) -> np.ndarray:
    """Grouped Y[M_total, N] in fp64; rows no group covers hold ``fill``."""
    x, w, s = _u16(x), _u8(w_canon), _u16(scales)
    ms = np.ascontiguousarray(m_sizes, dtype=np.int32)
    y = np.full((M_total, N), fill, dtype=np.float64)
    _load().oracle_gemm_grouped_f64(_ptr(x), _ptr(w), _ptr(s), _ptr(ms), ms.shape[0],
                                    M_total, N, K, G, _ptr(y), threads)
    return y


def sum_slices(ws: np.ndarray) -> np.ndarray:
    """Sum of fp32 split-K slices ws[S, ...] in ascending slice order, fp64."""
    w = np.ascontiguousarray(ws, dtype=np.float32)
    S = w.shape[0]
    count = int(np.prod(w.shape[1:]))
    out = np.empty(w.shape[1:], dtype=np.float64)
    _load().oracle_sum_slices_f64(_ptr(w), S, count, _ptr(out))
    return out
