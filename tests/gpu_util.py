"""Helpers for the GPU tests: moving seeded NumPy inputs to the device and back,
a NumPy model of the packed weight layout, and the oracle comparison."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import bf16_activation_quantized_gb300 as w4
from bf16_activation_quantized_gb300 import build as build_mod


def require_gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build_mod.build()


NAN_BF16 = float("nan")


def _nan_workspace(nbytes: int) -> torch.Tensor:
    """A workspace whose every fp32 word is NaN (16-byte aligned, >= 16 bytes)."""
    n = max(16, (nbytes + 15) // 16 * 16)
    return torch.full((n // 4,), float("nan"), dtype=torch.float32, device="cuda").view(torch.uint8)


def poisoned_gemm(x, w_packed, scales, **kw):
    """w4.gemm with Y and the split-K workspace filled with NaN before the call,
    so an output the kernels skipped shows up as NaN instead of a stale value."""
    M, K = x.shape
    N = scales.shape[0]
    G = K // scales.shape[1]
    zeros = kw.get("zeros")
    plan = w4.plan(M, N, K, arm=kw.get("arm"), split_k=kw.get("split_k", 0),
                   tile_tokens=kw.get("tile_tokens", 0), decode_kernel=kw.get("decode_kernel"),
                   group_size=G, zero_points=zeros is not None)
    if "out" not in kw:
        kw["out"] = torch.full((M, N), NAN_BF16, dtype=torch.bfloat16, device=x.device)
    if "workspace" not in kw:
        kw["workspace"] = _nan_workspace(plan["workspace_bytes"])
    return w4.gemm(x, w_packed, scales, **kw)


def poisoned_gemm_batched(x, w_packed, scales, **kw):
    """w4.gemm_batched with Y and the workspace filled with NaN before the call."""
    B, M, K = x.shape
    N = scales.shape[1]
    G = K // scales.shape[2]
    plan = w4.plan_batched(B, M, N, K, arm=kw.get("arm"), split_k=kw.get("split_k", 0),
                           tile_tokens=kw.get("tile_tokens", 0),
                           decode_kernel=kw.get("decode_kernel"), group_size=G,
                           zero_points=kw.get("zeros") is not None)
    if "out" not in kw:
        kw["out"] = torch.full((B, M, N), NAN_BF16, dtype=torch.bfloat16, device=x.device)
    if "workspace" not in kw:
        kw["workspace"] = _nan_workspace(plan["workspace_bytes"])
    return w4.gemm_batched(x, w_packed, scales, **kw)


def dev_u16_as_bf16(bits: np.ndarray) -> torch.Tensor:
    a = np.ascontiguousarray(bits, dtype=np.uint16).view(np.int16)
    return torch.from_numpy(a.copy()).view(torch.bfloat16).cuda()


def dev_u8(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.uint8).copy()).cuda()


def bf16_to_u16(t: torch.Tensor) -> np.ndarray:
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    bits = bf16_to_u16(t)
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


class DeviceProblem:
    """One seeded problem resident on the GPU (canonical weights packed there)."""

    def __init__(self, inp):
        self.inp = inp
        self.x = dev_u16_as_bf16(inp.x)
        self.scales = dev_u16_as_bf16(inp.scales)
        self.w_canon = dev_u8(inp.w_canon)
        self.w_packed = w4.pack(self.w_canon)


def layout_model(w_canon: np.ndarray, N: int, K: int) -> np.ndarray:
    """Independent NumPy model of the packed layout (uint32 words).

    Tiles of 128 rows x 64 columns, 4096 bytes each, tile-major then chunk;
    inside, 8 blocks of 16 rows; lane L = 4g + t holds 4 words; word j covers
    rows {g, g+8} and columns 64*chunk + 16j + 4t + {0..3} with nibble slots
    (bit: row, column offset) 0:g,0 4:g+8,0 8:g,2 12:g+8,2 16:g,1 20:g+8,1
    24:g,3 28:g+8,3.  Padding rows hold code 8."""
    n_pad = (N + 127) // 128 * 128
    codes = np.full((n_pad, K), 8, dtype=np.uint32)
    codes[:N, 0::2] = w_canon & 0x0F
    codes[:N, 1::2] = w_canon >> 4
    T, KC = n_pad // 128, K // 64
    tile, chunk, block, lane, j = np.meshgrid(np.arange(T), np.arange(KC), np.arange(8),
                                              np.arange(32), np.arange(4), indexing="ij")
    g, t = lane // 4, lane % 4
    r0 = tile * 128 + block * 16 + g
    r1 = r0 + 8
    k = chunk * 64 + 16 * j + 4 * t
    w = (codes[r0, k] | (codes[r1, k] << 4) | (codes[r0, k + 2] << 8) | (codes[r1, k + 2] << 12)
         | (codes[r0, k + 1] << 16) | (codes[r1, k + 1] << 20) | (codes[r0, k + 3] << 24)
         | (codes[r1, k + 3] << 28))
    return w.astype(np.uint32).reshape(-1)
