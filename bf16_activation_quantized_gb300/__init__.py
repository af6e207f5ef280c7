"""W4A16 skinny GEMM for GB300 (sm_103a): Python binding of the C ABI.

``Y[M, N] = X[M, K] . dequant(W)[N, K]^T`` with bf16 X and Y, int4 W packed two
codes per byte (low nibble = even k), one bf16 scale per G weights along K
(G = 128, 64 or 32, read off the scales' shape [N, K/G]),
``dequant = scale * (code - 8)``, fp32 accumulation.

Every function here only checks tensor metadata, allocates outputs and
workspaces with torch, and calls the C ABI on the current torch stream: all
arithmetic runs in the library's CUDA kernels.  There is no CPU path; a call
with CPU tensors or without the built library raises.
"""
from __future__ import annotations

import ctypes
import threading

import torch

from . import _lib
from ._lib import Options, PlanInfo, W4A16Error

GROUP = 128                  # default scale group size
GROUP_SIZES = (128, 64, 32)
ARM_AUTO, ARM_DECODE, ARM_TENSOR = 0, 1, 2
_ARMS = {None: ARM_AUTO, "auto": ARM_AUTO, "decode": ARM_DECODE, "tensor": ARM_TENSOR}

__all__ = ["GROUP", "pack", "gemm", "gemm_partials", "gemm_grouped", "gemm_batched", "plan_batched", "dequant_fp32", "dequant_bf16",
           "splitk_reduce", "plan", "packed_weight_bytes", "layout_version", "read_error_word",
           "ERROR_WAIT_TIMEOUT", "W4A16Error"]


def _stream_ptr(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def _need_cuda(t: torch.Tensor, name: str, dtype=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


FLAG_RESIDENT_WEIGHTS = 1
FLAG_DECODE_WHOLE_K = 2
FLAG_DECODE_K_SLICES = 4
FLAG_ZERO_POINTS = 8
FLAG_TEST_STALL = 16
ERROR_WAIT_TIMEOUT = 1       # error-word bit: a bounded wait in a kernel ran out
_KERNELS = {None: 0, "auto": 0, "whole_k": FLAG_DECODE_WHOLE_K, "k_slices": FLAG_DECODE_K_SLICES}


def _group_size(K: int, cols: int, what: str) -> int:
    """G from K and the scales' last dimension K / G (the library rejects G
    other than 128, 64 and 32)."""
    if cols <= 0 or K % cols or (K // cols) not in GROUP_SIZES:
        raise ValueError(f"{what} must have K/G columns with G in {GROUP_SIZES} (K={K}, got {cols})")
    return K // cols


def _opts(arm, split_k, tile_tokens, resident_weights=False, decode_kernel=None, zero_points=False,
          test_stall=False):
    if arm not in _ARMS:
        raise ValueError(f"arm must be one of {list(_ARMS)}")
    if decode_kernel not in _KERNELS:
        raise ValueError(f"decode_kernel must be one of {list(_KERNELS)}")
    flags = ((FLAG_RESIDENT_WEIGHTS if resident_weights else 0) | _KERNELS[decode_kernel]
             | (FLAG_ZERO_POINTS if zero_points else 0) | (FLAG_TEST_STALL if test_stall else 0))
    return Options(_ARMS[arm], int(split_k), int(tile_tokens), flags)


_ws_lock = threading.Lock()
_ws_cache: dict = {}


def _workspace(device, nbytes: int) -> torch.Tensor:
    """A grow-only scratch buffer per device (contents need no initialisation)."""
    key = torch.device(device).index
    with _ws_lock:
        buf = _ws_cache.get(key)
        if buf is None or buf.numel() < nbytes:
            buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
            _ws_cache[key] = buf
        return buf


# Host-side answers that depend only on the shape, the options and the device
# (the plan depends on the device's SM count), cached so that a call costs one
# library call.
_plan_cache: dict = {}
_pwb_cache: dict = {}


def _workspace_need(M: int, N: int, K: int, G: int, o: Options, dev_index: int) -> int:
    key = (M, N, K, G, o.arm, o.split_k, o.tile_tokens, o.flags, dev_index)
    need = _plan_cache.get(key)
    if need is None:
        info = PlanInfo()
        _lib.check(_lib.lib().w4a16_plan(M, N, K, G, ctypes.byref(o), ctypes.byref(info)),
                   "w4a16_plan")
        need = int(info.workspace_bytes)
        _plan_cache[key] = need
    return need


def _plan_dict(info: PlanInfo) -> dict:
    return {"arm": {1: "decode", 2: "tensor"}.get(info.arm, info.arm), "split_k": info.split_k,
            "tile_tokens": info.tile_tokens, "ctas": info.ctas,
            "workspace_bytes": int(info.workspace_bytes), "whole_k": bool(info.whole_k)}


def layout_version() -> int:
    return int(_lib.lib().w4a16_layout_version())


def read_error_word(clear: bool = True, device=None) -> int:
    """The device error word (w4a16_read_error_word): OR of the ERROR_* bits
    the kernels recorded since it was last cleared; 0 means no kernel gave up.
    Waits for all work on the device first; ``clear`` resets the word."""
    v = ctypes.c_int(0)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        _lib.check(_lib.lib().w4a16_read_error_word(ctypes.byref(v), 1 if clear else 0),
                   "w4a16_read_error_word")
    return int(v.value)


def packed_weight_bytes(N: int, K: int) -> int:
    key = (N, K)
    nb = _pwb_cache.get(key)
    if nb is None:
        nb = _pwb_cache[key] = int(_lib.lib().w4a16_packed_weight_bytes(N, K))
    return nb


def pack(w_canon: torch.Tensor) -> torch.Tensor:
    """Canonical uint8 [N, K/2] (CUDA) -> packed uint8 buffer for the kernels."""
    _need_cuda(w_canon, "w_canon", torch.uint8)
    N, half_k = w_canon.shape
    K = 2 * half_k
    nbytes = packed_weight_bytes(N, K)
    if nbytes == 0:
        raise ValueError(f"unsupported weight shape N={N} K={K} (K must be a multiple of 128)")
    out = torch.empty(nbytes, dtype=torch.uint8, device=w_canon.device)
    with torch.cuda.device(w_canon.device):
        _lib.check(_lib.lib().w4a16_pack_weights(w_canon.data_ptr(), out.data_ptr(), N, K,
                                                 _stream_ptr(w_canon.device)), "w4a16_pack_weights")
    return out


def plan(M: int, N: int, K: int, arm=None, split_k: int = 0, tile_tokens: int = 0,
         device=None, decode_kernel=None, group_size: int = GROUP,
         zero_points: bool = False, sms: int | None = None) -> dict:
    """What the dispatcher picks for this shape on the (current) device, or,
    with ``sms``, on a device with that many SMs (host only, no GPU needed)."""
    info = PlanInfo()
    o = _opts(arm, split_k, tile_tokens, decode_kernel=decode_kernel, zero_points=zero_points)
    if sms is not None:
        _lib.check(_lib.lib().w4a16_plan_for_sms(int(sms), 1, M, N, K, group_size, ctypes.byref(o),
                                                 ctypes.byref(info)), "w4a16_plan_for_sms")
        return _plan_dict(info)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        _lib.check(_lib.lib().w4a16_plan(M, N, K, group_size, ctypes.byref(o), ctypes.byref(info)),
                   "w4a16_plan")
    return _plan_dict(info)


def gemm(x: torch.Tensor, w_packed: torch.Tensor, scales: torch.Tensor, *, arm=None,
         split_k: int = 0, tile_tokens: int = 0, out: torch.Tensor | None = None,
         workspace: torch.Tensor | None = None, resident_weights: bool = False,
         decode_kernel=None, zeros: torch.Tensor | None = None,
         test_stall: bool = False) -> torch.Tensor:
    """Y = X . dequant(W)^T.  x: bf16 [M, K]; scales: bf16 [N, K/G]; returns bf16 [M, N].

    ``zeros`` (uint8 [N, K/G], low four bits) selects the zero-point variant,
    dequant = scale * (code - z) (w4a16_gemm_zp); without it z is 8.

    ``resident_weights=True`` promises that no kernel still running on the
    current stream writes ``w_packed`` or ``scales`` (W4A16_FLAG_RESIDENT_WEIGHTS):
    the call may then start streaming them before the previous kernel ends.
    ``decode_kernel`` ("whole_k" or "k_slices") forces the decode arm's kernel.
    ``test_stall`` (tests only, W4A16_FLAG_TEST_STALL) makes the decode kernel's
    bounded waits run out: the outputs become NaN and the error word is set."""
    _need_cuda(x, "x", torch.bfloat16)
    _need_cuda(scales, "scales", torch.bfloat16)
    _need_cuda(w_packed, "w_packed", torch.uint8)
    M, K = x.shape
    N = scales.shape[0]
    G = _group_size(K, scales.shape[1], "scales [N, K/G]")
    if w_packed.numel() < packed_weight_bytes(N, K):
        raise ValueError("w_packed is smaller than packed_weight_bytes(N, K)")
    if zeros is not None:
        _need_cuda(zeros, "zeros", torch.uint8)
        if tuple(zeros.shape) != tuple(scales.shape):
            raise ValueError("zeros must be uint8 [N, K/G], the shape of scales")
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=x.device)
    else:
        _need_cuda(out, "out", torch.bfloat16)
    o = _opts(arm, split_k, tile_tokens, resident_weights, decode_kernel, zeros is not None,
              test_stall)
    L = _lib.lib()
    dev = x.device
    switch = dev.index != torch.cuda.current_device()
    if switch:
        prev = torch.cuda.current_device()
        torch.cuda.set_device(dev)
    try:
        need = _workspace_need(M, N, K, G, o, dev.index)
        if workspace is None:
            ws = _workspace(dev, need) if need else None
        else:
            ws = workspace
        ws_ptr = ws.data_ptr() if ws is not None else None
        ws_bytes = ws.numel() * ws.element_size() if ws is not None else 0
        stream = torch.cuda.current_stream(dev).cuda_stream
        if zeros is None:
            _lib.check(L.w4a16_gemm_ex(x.data_ptr(), w_packed.data_ptr(), scales.data_ptr(),
                                       out.data_ptr(), M, N, K, G, ws_ptr, ws_bytes,
                                       ctypes.byref(o), stream), "w4a16_gemm_ex")
        else:
            _lib.check(L.w4a16_gemm_zp(x.data_ptr(), w_packed.data_ptr(), scales.data_ptr(),
                                       zeros.data_ptr(), out.data_ptr(), M, N, K, G, ws_ptr,
                                       ws_bytes, ctypes.byref(o), stream), "w4a16_gemm_zp")
    finally:
        if switch:
            torch.cuda.set_device(prev)
    return out


def gemm_partials(x: torch.Tensor, w_packed: torch.Tensor, scales: torch.Tensor, *,
                  out: torch.Tensor, workspace: torch.Tensor, arm=None, split_k: int = 0,
                  tile_tokens: int = 0, resident_weights: bool = False) -> int:
    """First launch of gemm() only (see w4a16_gemm_partials); returns SPLIT_K.

    With SPLIT_K > 1 the fp32 partial sums land in ``workspace`` as
    [SPLIT_K, M, N] and ``out`` is untouched; splitk_reduce() finishes the call."""
    _need_cuda(x, "x", torch.bfloat16)
    _need_cuda(scales, "scales", torch.bfloat16)
    _need_cuda(w_packed, "w_packed", torch.uint8)
    _need_cuda(out, "out", torch.bfloat16)
    _need_cuda(workspace, "workspace")
    M, K = x.shape
    N = scales.shape[0]
    G = _group_size(K, scales.shape[1], "scales [N, K/G]")
    o = _opts(arm, split_k, tile_tokens, resident_weights)
    sk = ctypes.c_int(0)
    with torch.cuda.device(x.device):
        _lib.check(_lib.lib().w4a16_gemm_partials(
            x.data_ptr(), w_packed.data_ptr(), scales.data_ptr(), out.data_ptr(), M, N, K, G,
            workspace.data_ptr(), workspace.numel() * workspace.element_size(), ctypes.byref(o),
            ctypes.byref(sk), _stream_ptr(x.device)), "w4a16_gemm_partials")
    return int(sk.value)


def plan_batched(batch: int, M: int, N: int, K: int, arm=None, split_k: int = 0,
                 tile_tokens: int = 0, device=None, decode_kernel=None,
                 group_size: int = GROUP, zero_points: bool = False) -> dict:
    """What the dispatcher picks for a batch of ``batch`` products of shape (M, N, K)."""
    info = PlanInfo()
    o = _opts(arm, split_k, tile_tokens, decode_kernel=decode_kernel, zero_points=zero_points)
    with torch.cuda.device(device if device is not None else torch.cuda.current_device()):
        _lib.check(_lib.lib().w4a16_plan_batched(batch, M, N, K, group_size, ctypes.byref(o),
                                                 ctypes.byref(info)), "w4a16_plan_batched")
    return _plan_dict(info)


def gemm_batched(x: torch.Tensor, w_packed: torch.Tensor, scales: torch.Tensor, *, arm=None,
                 split_k: int = 0, tile_tokens: int = 0, out: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None, resident_weights: bool = False,
                 decode_kernel=None, zeros: torch.Tensor | None = None) -> torch.Tensor:
    """Y[b] = X[b] . dequant(W[b])^T for every b in one launch.

    x: bf16 [B, M, K]; w_packed: uint8 [B, packed_weight_bytes(N, K)] (or the same
    bytes flat); scales: bf16 [B, N, K/G]; returns bf16 [B, M, N].  ``zeros``
    (uint8 [B, N, K/G]) selects the zero-point variant (w4a16_gemm_batched_zp)."""
    _need_cuda(x, "x", torch.bfloat16)
    _need_cuda(scales, "scales", torch.bfloat16)
    _need_cuda(w_packed, "w_packed", torch.uint8)
    if x.dim() != 3 or scales.dim() != 3:
        raise ValueError("x must be [B, M, K] and scales [B, N, K/G]")
    B, M, K = x.shape
    N = scales.shape[1]
    if scales.shape[0] != B:
        raise ValueError("scales must be [B, N, K/G]")
    G = _group_size(K, scales.shape[2], "scales [B, N, K/G]")
    if w_packed.numel() < B * packed_weight_bytes(N, K):
        raise ValueError("w_packed is smaller than B * packed_weight_bytes(N, K)")
    if out is None:
        out = torch.empty((B, M, N), dtype=torch.bfloat16, device=x.device)
    else:
        _need_cuda(out, "out", torch.bfloat16)
    if zeros is not None:
        _need_cuda(zeros, "zeros", torch.uint8)
        if tuple(zeros.shape) != tuple(scales.shape):
            raise ValueError("zeros must be uint8 [B, N, K/G], the shape of scales")
    o = _opts(arm, split_k, tile_tokens, resident_weights, decode_kernel, zeros is not None)
    with torch.cuda.device(x.device):
        info = PlanInfo()
        _lib.check(_lib.lib().w4a16_plan_batched(B, M, N, K, G, ctypes.byref(o), ctypes.byref(info)),
                   "w4a16_plan_batched")
        need = int(info.workspace_bytes)
        ws = workspace if workspace is not None else (_workspace(x.device, need) if need else None)
        args = (ws.data_ptr() if ws is not None else None,
                ws.numel() * ws.element_size() if ws is not None else 0, ctypes.byref(o),
                _stream_ptr(x.device))
        if zeros is None:
            _lib.check(_lib.lib().w4a16_gemm_batched(
                x.data_ptr(), w_packed.data_ptr(), scales.data_ptr(), out.data_ptr(), B, M, N, K, G,
                *args), "w4a16_gemm_batched")
        else:
            _lib.check(_lib.lib().w4a16_gemm_batched_zp(
                x.data_ptr(), w_packed.data_ptr(), scales.data_ptr(), zeros.data_ptr(),
                out.data_ptr(), B, M, N, K, G, *args), "w4a16_gemm_batched_zp")
    return out


def gemm_grouped(x: torch.Tensor, w_packed: torch.Tensor, scales: torch.Tensor,
                 m_sizes: torch.Tensor, *, out: torch.Tensor | None = None,
                 status: torch.Tensor | None = None, zeros: torch.Tensor | None = None):
    """Grouped product in one launch.

    x: bf16 [M_total, K]; w_packed: num_groups packed blocks; scales: bf16
    [num_groups, N, K/G]; m_sizes: int32 [num_groups] on the device (never
    read on the host).  ``zeros`` (uint8 [num_groups, N, K/G]) selects the
    zero-point variant (w4a16_gemm_grouped_zp).  Returns (Y bf16 [M_total, N],
    status int32 tensor whose element 0 the kernel sets; 0 = sizes consistent)."""
    _need_cuda(x, "x", torch.bfloat16)
    _need_cuda(scales, "scales", torch.bfloat16)
    _need_cuda(w_packed, "w_packed", torch.uint8)
    _need_cuda(m_sizes, "m_sizes", torch.int32)
    M_total, K = x.shape
    NG, N, kg = scales.shape
    if m_sizes.numel() != NG:
        raise ValueError("scales must be [num_groups, N, K/G] and m_sizes [num_groups]")
    G = _group_size(K, kg, "scales [num_groups, N, K/G]")
    if w_packed.numel() < NG * packed_weight_bytes(N, K):
        raise ValueError("w_packed is smaller than num_groups * packed_weight_bytes(N, K)")
    if out is None:
        out = torch.empty((M_total, N), dtype=torch.bfloat16, device=x.device)
    L = _lib.lib()
    with torch.cuda.device(x.device):
        nb = ctypes.c_size_t(0)
        _lib.check(L.w4a16_grouped_workspace_bytes(NG, M_total, N, K, G, ctypes.byref(nb)),
                   "w4a16_grouped_workspace_bytes")
        if status is None:
            status = torch.empty(max(4, (nb.value + 3) // 4), dtype=torch.int32, device=x.device)
        if zeros is None:
            _lib.check(L.w4a16_gemm_grouped(x.data_ptr(), w_packed.data_ptr(), scales.data_ptr(),
                                            m_sizes.data_ptr(), out.data_ptr(), NG, M_total, N, K,
                                            G, status.data_ptr(), status.numel() * 4,
                                            _stream_ptr(x.device)), "w4a16_gemm_grouped")
        else:
            _need_cuda(zeros, "zeros", torch.uint8)
            if tuple(zeros.shape) != tuple(scales.shape):
                raise ValueError("zeros must be uint8 [num_groups, N, K/G], the shape of scales")
            _lib.check(L.w4a16_gemm_grouped_zp(x.data_ptr(), w_packed.data_ptr(), scales.data_ptr(),
                                               zeros.data_ptr(), m_sizes.data_ptr(), out.data_ptr(),
                                               NG, M_total, N, K, G, status.data_ptr(),
                                               status.numel() * 4, _stream_ptr(x.device)),
                       "w4a16_gemm_grouped_zp")
    return out, status


def dequant_fp32(w_packed: torch.Tensor, scales: torch.Tensor,
                 group_size: int = GROUP, zeros: torch.Tensor | None = None) -> torch.Tensor:
    """fp32 [N, K] = scale * (code - 8), computed by the kernels' bit trick;
    scales bf16 [N, K/G] with G = group_size; with ``zeros`` (uint8 [N, K/G])
    scale * (code - z)."""
    _need_cuda(w_packed, "w_packed", torch.uint8)
    _need_cuda(scales, "scales", torch.bfloat16)
    N, kg = scales.shape
    K = kg * group_size
    out = torch.empty((N, K), dtype=torch.float32, device=scales.device)
    with torch.cuda.device(scales.device):
        if zeros is None:
            _lib.check(_lib.lib().w4a16_dequant_fp32(w_packed.data_ptr(), scales.data_ptr(),
                                                     out.data_ptr(), N, K, group_size,
                                                     _stream_ptr(scales.device)), "w4a16_dequant_fp32")
        else:
            _need_cuda(zeros, "zeros", torch.uint8)
            _lib.check(_lib.lib().w4a16_dequant_zp_fp32(w_packed.data_ptr(), scales.data_ptr(),
                                                        zeros.data_ptr(), out.data_ptr(), N, K,
                                                        group_size, _stream_ptr(scales.device)),
                       "w4a16_dequant_zp_fp32")
    return out


def dequant_bf16(w_packed: torch.Tensor, scales: torch.Tensor,
                 group_size: int = GROUP, zeros: torch.Tensor | None = None) -> torch.Tensor:
    """bf16 [N, K] = round_nearest_even(scale * (code - 8)): the tensor arm's
    operand; scales bf16 [N, K/G] with G = group_size; with ``zeros``
    scale * (code - z)."""
    _need_cuda(w_packed, "w_packed", torch.uint8)
    _need_cuda(scales, "scales", torch.bfloat16)
    N, kg = scales.shape
    K = kg * group_size
    out = torch.empty((N, K), dtype=torch.bfloat16, device=scales.device)
    with torch.cuda.device(scales.device):
        if zeros is None:
            _lib.check(_lib.lib().w4a16_dequant_bf16(w_packed.data_ptr(), scales.data_ptr(),
                                                     out.data_ptr(), N, K, group_size,
                                                     _stream_ptr(scales.device)), "w4a16_dequant_bf16")
        else:
            _need_cuda(zeros, "zeros", torch.uint8)
            _lib.check(_lib.lib().w4a16_dequant_zp_bf16(w_packed.data_ptr(), scales.data_ptr(),
                                                        zeros.data_ptr(), out.data_ptr(), N, K,
                                                        group_size, _stream_ptr(scales.device)),
                       "w4a16_dequant_zp_bf16")
    return out


def splitk_reduce(ws: torch.Tensor, out: torch.Tensor | None = None) -> torch.Tensor:
    """bf16 [M, N] = sum over slices of fp32 ws [S, M, N] (slices in order)."""
    _need_cuda(ws, "ws", torch.float32)
    S, M, N = ws.shape
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=ws.device)
    with torch.cuda.device(ws.device):
        _lib.check(_lib.lib().w4a16_splitk_reduce(ws.data_ptr(), out.data_ptr(), S, M, N,
                                                  _stream_ptr(ws.device)), "w4a16_splitk_reduce")
    return out
