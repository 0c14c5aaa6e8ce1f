"""Thin ctypes binding over ``libsage.so`` (the C ABI in ``include/sage.h``).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels. Tensors are PyTorch CUDA tensors; outputs and scratch are allocated
with torch when the caller does not pass them. Calls are enqueued on the
current torch stream. A non-OK status raises ``SageError``. Importing this
module raises if the library has not been built.
"""
from __future__ import annotations

import ctypes
import math
import os
import re
from typing import Optional, Sequence, Tuple

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libsage.so")
HEADER_PATH = os.path.join(os.path.dirname(_PKG), "include", "sage.h")

FMT_INT8 = 0   # SAGE_FMT_QK_INT8_V_FP8
FMT_MXFP4 = 1  # SAGE_FMT_QK_MXFP4_V_FP8
FMT_FP8 = 2    # SAGE_FMT_QK_FP8_V_FP8
FMT_MXFP4H = 3  # SAGE_FMT_QK_MXFP4H_V_FP8 (Hadamard-rotated MXFP4)
FMT_MXFP4_V4 = 4  # SAGE_FMT_QK_MXFP4_V_MXFP4 (MXFP4 Q/K, V and P)

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libsage.so is not built ({LIB_PATH}); run __graft_entry__.build()")

_lib = ctypes.CDLL(LIB_PATH)


class Strides(ctypes.Structure):
    _fields_ = [("b", ctypes.c_int64), ("n", ctypes.c_int64), ("h", ctypes.c_int64)]


class AttnOptions(ctypes.Structure):
    _fields_ = [("num_splits", ctypes.c_int32), ("cta_mode", ctypes.c_int32),
                ("k_mean", ctypes.c_void_p), ("delta_s", ctypes.c_void_p),
                ("wait_cycles", ctypes.c_int64), ("test_withhold_v", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class HostAttention(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int), ("B", ctypes.c_int64), ("Nq", ctypes.c_int64),
                ("Nk", ctypes.c_int64), ("H", ctypes.c_int64), ("D", ctypes.c_int64),
                ("q", ctypes.c_void_p), ("k", ctypes.c_void_p), ("v", ctypes.c_void_p),
                ("o", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("k_lens", ctypes.c_void_p),
                ("softmax_scale", ctypes.c_float), ("smooth_k", ctypes.c_int32),
                ("smooth_q", ctypes.c_int32), ("heads_per_group", ctypes.c_int32),
                ("num_splits", ctypes.c_int32), ("cta_mode", ctypes.c_int32)]


_P, _I64, _I32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
_lib.sage_quantized_bytes.restype = ctypes.c_size_t
_lib.sage_quantized_bytes.argtypes = [_I32, _I32, _I64, _I64, _I64, _I64]
_lib.sage_workspace_bytes.restype = ctypes.c_size_t
_lib.sage_workspace_bytes.argtypes = [_I32, _I32, _I64, _I64, _I64, _I64, _I64, _I32]
_lib.sage_quantize_qk.restype = _I32
_lib.sage_quantize_qk.argtypes = [_I32, _P, Strides, _I64, _I64, _I64, _I64, _P, _P, _P, _P]
_lib.sage_quantize_v.restype = _I32
_lib.sage_quantize_v.argtypes = [_P, Strides, _I64, _I64, _I64, _I64, _P, _P, _P, _P,
                                 ctypes.c_size_t, _P]
_lib.sage_quantize_v_mxfp4.restype = _I32
_lib.sage_quantize_v_mxfp4.argtypes = [_P, Strides, _I64, _I64, _I64, _I64, _P, _P, _P, _P]
_lib.sage_quantize_qkv.restype = _I32
_lib.sage_quantize_qkv.argtypes = [_I32, _P, Strides, _P, Strides, _P, Strides, _I64, _I64, _I64,
                                   _I64, _I64, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_size_t,
                                   _P]
_lib.sage_quantize_q_smooth.restype = _I32
_lib.sage_quantize_q_smooth.argtypes = [_I32, _P, Strides, _I64, _I64, _I64, _I64, _P, _P, _P, _P]
_lib.sage_delta_s.restype = _I32
_lib.sage_delta_s.argtypes = [_I32, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64, _P, _P]
_lib.sage_quantize_k_smooth.restype = _I32
_lib.sage_quantize_k_smooth.argtypes = [_I32, _P, Strides, _I64, _I64, _I64, _I64, _P, _P, _P, _P,
                                        _P, ctypes.c_size_t, _P]
_lib.sage_attn_fwd.restype = _I32
_lib.sage_attn_fwd.argtypes = [_I32, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64, _I64,
                               ctypes.c_float, _I32, _P, Strides, _P, _P, ctypes.c_size_t,
                               ctypes.POINTER(AttnOptions), _P]
_lib.sage_attention_host_workspace_bytes.restype = ctypes.c_size_t
_lib.sage_attention_host_workspace_bytes.argtypes = [ctypes.POINTER(HostAttention)]
_lib.sage_attention_host.restype = _I32
_lib.sage_attention_host.argtypes = [ctypes.POINTER(HostAttention), _P, ctypes.c_size_t, _P]
_lib.sage_status_string.restype = ctypes.c_char_p
_lib.sage_status_string.argtypes = [_I32]
_lib.sage_last_device_status.restype = _I32
_lib.sage_last_device_status.argtypes = [_P]
_lib.sage_version.restype = ctypes.c_char_p
_lib.sage_version.argtypes = []


class SageError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_lib.sage_status_string(status).decode()} ({status})")


def _check(st: int, where: str):
    if st != 0:
        raise SageError(st, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _bnhd_strides(x: torch.Tensor) -> Strides:
    if x.dim() != 4 or x.stride(3) != 1:
        raise ValueError("expected a [B, N, H, D] tensor with unit stride along D")
    return Strides(x.stride(0), x.stride(1), x.stride(2))


def header_symbols() -> Sequence[str]:
    """Function names declared in include/sage.h."""
    text = open(HEADER_PATH).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\*?(sage_\w+)\s*\(", text, re.M)))


def library() -> ctypes.CDLL:
    return _lib


def sage_version() -> str:
    return _lib.sage_version().decode()


def sage_quantized_bytes(fmt: int, which: int, B: int, N: int, H: int, D: int = 128) -> int:
    return int(_lib.sage_quantized_bytes(fmt, which, B, N, H, D))


def sage_workspace_bytes(op: int, fmt: int, B: int, H: int, Nq: int, Nk: int, D: int = 128,
                         num_splits: int = 0) -> int:
    return int(_lib.sage_workspace_bytes(op, fmt, B, H, Nq, Nk, D, num_splits))


def attn_splits(B: int, H: int, Nq: int, Nk: int, num_splits: int = 0) -> int:
    """KV split count sage_attn_fwd uses (derived from its workspace size)."""
    ws = sage_workspace_bytes(2, FMT_INT8, B, H, Nq, Nk, 128, num_splits)
    return 1 if ws == 0 else ws // (B * H * Nq * 129 * 4)


def pad128(n: int) -> int:
    return (n + 127) // 128 * 128


def _lens_tensor(lens, device) -> Optional[torch.Tensor]:
    if lens is None:
        return None
    if isinstance(lens, torch.Tensor):
        return lens.to(device=device, dtype=torch.int32).contiguous()
    return torch.tensor(list(lens), dtype=torch.int32, device=device)


def sage_quantize_qk(x: torch.Tensor, fmt: int = FMT_INT8, lens=None,
                     out: Optional[torch.Tensor] = None,
                     scale: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Quantize BF16 Q or K ``[B, N, H, D]``.

    INT8: returns (codes held as float16 ``[B, H, Npad, D]``, float32 scales
    ``[B, H, Npad/128]``). MXFP4: (uint8 ``[B, H, Npad, D/2]``, uint8 E8M0
    ``[B, H, Npad, D/32]``; the rotated MXFP4 format has the same layout).
    FP8: (uint8 E4M3 ``[B, H, Npad, D]``, float32 scales ``[B, H, Npad/128]``).
    """
    B, N, H, D = x.shape
    Np = pad128(N)
    if out is None:
        if fmt == FMT_INT8:
            out = torch.empty((B, H, Np, D), dtype=torch.float16, device=x.device)
        elif fmt == FMT_FP8:
            out = torch.empty((B, H, Np, D), dtype=torch.uint8, device=x.device)
        else:
            out = torch.empty((B, H, Np, D // 2), dtype=torch.uint8, device=x.device)
    if scale is None:
        scale = (torch.empty((B, H, Np, D // 32), dtype=torch.uint8, device=x.device)
                 if fmt in (FMT_MXFP4, FMT_MXFP4H, FMT_MXFP4_V4)
                 else torch.empty((B, H, Np // 128), dtype=torch.float32, device=x.device))
    ln = _lens_tensor(lens, x.device)
    _check(_lib.sage_quantize_qk(fmt, _ptr(x), _bnhd_strides(x), B, N, H, D, _ptr(ln), _ptr(out),
                                 _ptr(scale), _stream()), "sage_quantize_qk")
    return out, scale


def sage_quantize_v(v: torch.Tensor, lens=None, out: Optional[torch.Tensor] = None,
                    scale: Optional[torch.Tensor] = None,
                    workspace: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Quantize BF16 V ``[B, N, H, D]`` to FP8 E4M3 ``[B, H, Npad, D]`` (uint8) + scales."""
    B, N, H, D = v.shape
    Np = pad128(N)
    if out is None:
        out = torch.empty((B, H, Np, D), dtype=torch.uint8, device=v.device)
    if scale is None:
        scale = torch.empty((B, H, D), dtype=torch.float32, device=v.device)
    need = sage_workspace_bytes(1, FMT_INT8, B, H, N, N, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=v.device)
    ln = _lens_tensor(lens, v.device)
    _check(_lib.sage_quantize_v(_ptr(v), _bnhd_strides(v), B, N, H, D, _ptr(ln), _ptr(out),
                                _ptr(scale), _ptr(workspace), workspace.numel(), _stream()),
           "sage_quantize_v")
    return out, scale


def _qk_outputs(fmt: int, B: int, N: int, H: int, D: int, dev):
    Np = pad128(N)
    if fmt == FMT_INT8:
        return (torch.empty((B, H, Np, D), dtype=torch.float16, device=dev),
                torch.empty((B, H, Np // 128), dtype=torch.float32, device=dev))
    if fmt == FMT_FP8:
        return (torch.empty((B, H, Np, D), dtype=torch.uint8, device=dev),
                torch.empty((B, H, Np // 128), dtype=torch.float32, device=dev))
    return (torch.empty((B, H, Np, D // 2), dtype=torch.uint8, device=dev),
            torch.empty((B, H, Np, D // 32), dtype=torch.uint8, device=dev))


def sage_quantize_v_mxfp4(v: torch.Tensor, lens=None, out: Optional[torch.Tensor] = None,
                          scale: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Quantize BF16 V ``[B, N, H, D]`` to MXFP4 along tokens: packed E2M1
    ``[B, H, D, Npad/2]`` (uint8) + E8M0 bytes ``[B, H, Npad/128, D, 4]``."""
    B, N, H, D = v.shape
    Np = pad128(N)
    if out is None:
        out = torch.empty((B, H, D, Np // 2), dtype=torch.uint8, device=v.device)
    if scale is None:
        scale = torch.empty((B, H, Np // 128, D, 4), dtype=torch.uint8, device=v.device)
    ln = _lens_tensor(lens, v.device)
    _check(_lib.sage_quantize_v_mxfp4(_ptr(v), _bnhd_strides(v), B, N, H, D, _ptr(ln), _ptr(out),
                                      _ptr(scale), _stream()), "sage_quantize_v_mxfp4")
    return out, scale


def sage_quantize_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, fmt: int = FMT_INT8,
                      k_lens=None, outs=None, workspace: Optional[torch.Tensor] = None):
    """Quantize Q, K, V in one library call (bit-identical to the three separate
    calls). Returns ((q_q, q_scale), (k_q, k_scale), (v_q, v_scale)); `outs` may
    supply those six tensors."""
    B, Nq, H, D = q.shape
    Nk = k.shape[1]
    dev = q.device
    if outs is None:
        (qq, qs), (kq, ks) = _qk_outputs(fmt, B, Nq, H, D, dev), _qk_outputs(fmt, B, Nk, H, D, dev)
        if fmt == FMT_MXFP4_V4:
            vq = torch.empty((B, H, D, pad128(Nk) // 2), dtype=torch.uint8, device=dev)
            vs = torch.empty((B, H, pad128(Nk) // 128, D, 4), dtype=torch.uint8, device=dev)
        else:
            vq = torch.empty((B, H, pad128(Nk), D), dtype=torch.uint8, device=dev)
            vs = torch.empty((B, H, D), dtype=torch.float32, device=dev)
    else:
        (qq, qs), (kq, ks), (vq, vs) = outs
    need = sage_workspace_bytes(1, fmt, B, H, Nk, Nk, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    ln = _lens_tensor(k_lens, dev)
    _check(_lib.sage_quantize_qkv(fmt, _ptr(q), _bnhd_strides(q), _ptr(k), _bnhd_strides(k),
                                  _ptr(v), _bnhd_strides(v), B, Nq, Nk, H, D, _ptr(ln), _ptr(qq),
                                  _ptr(qs), _ptr(kq), _ptr(ks), _ptr(vq), _ptr(vs),
                                  _ptr(workspace), workspace.numel(), _stream()),
           "sage_quantize_qkv")
    return (qq, qs), (kq, ks), (vq, vs)


def sage_quantize_q_smooth(q: torch.Tensor, out: Optional[torch.Tensor] = None,
                           scale: Optional[torch.Tensor] = None,
                           q_mean: Optional[torch.Tensor] = None):
    """Q smoothing + INT8 quantization of BF16 Q ``[B, N, H, D]``: (codes held as
    float16 ``[B, H, Npad, D]``, float32 block scales ``[B, H, Npad/128]``,
    float32 block channel means ``[B, H, Npad/128, D]``)."""
    B, N, H, D = q.shape
    Np = pad128(N)
    dev = q.device
    if out is None:
        out = torch.empty((B, H, Np, D), dtype=torch.float16, device=dev)
    if scale is None:
        scale = torch.empty((B, H, Np // 128), dtype=torch.float32, device=dev)
    if q_mean is None:
        q_mean = torch.empty((B, H, Np // 128, D), dtype=torch.float32, device=dev)
    _check(_lib.sage_quantize_q_smooth(FMT_INT8, _ptr(q), _bnhd_strides(q), B, N, H, D, _ptr(out),
                                       _ptr(scale), _ptr(q_mean), _stream()),
           "sage_quantize_q_smooth")
    return out, scale, q_mean


def sage_delta_s(q_mean: torch.Tensor, k_q: torch.Tensor, k_scale: torch.Tensor, *, Nq: int,
                 Nk: int, k_mean: Optional[torch.Tensor] = None,
                 out: Optional[torch.Tensor] = None) -> torch.Tensor:
    """Q smoothing's logit correction dS ``[B, H, Nq_pad/128, Nk_pad]`` (float32)."""
    B, H = k_q.shape[0], k_q.shape[1]
    if out is None:
        out = torch.empty((B, H, pad128(Nq) // 128, pad128(Nk)), dtype=torch.float32,
                          device=k_q.device)
    _check(_lib.sage_delta_s(FMT_INT8, _ptr(q_mean), _ptr(k_q), _ptr(k_scale), _ptr(k_mean), B, H,
                             Nq, Nk, 128, _ptr(out), _stream()), "sage_delta_s")
    return out


def sage_quantize_k_smooth(k: torch.Tensor, lens=None, out: Optional[torch.Tensor] = None,
                           scale: Optional[torch.Tensor] = None,
                           k_mean: Optional[torch.Tensor] = None,
                           workspace: Optional[torch.Tensor] = None):
    """K smoothing + INT8 quantization of BF16 K ``[B, N, H, D]``: returns (codes
    held as float16 ``[B, H, Npad, D]``, float32 block scales ``[B, H, Npad/128]``,
    float32 channel means ``[B, H, D]``); pass the means to sage_attn_fwd(k_mean=)."""
    B, N, H, D = k.shape
    Np = pad128(N)
    dev = k.device
    if out is None:
        out = torch.empty((B, H, Np, D), dtype=torch.float16, device=dev)
    if scale is None:
        scale = torch.empty((B, H, Np // 128), dtype=torch.float32, device=dev)
    if k_mean is None:
        k_mean = torch.empty((B, H, D), dtype=torch.float32, device=dev)
    need = sage_workspace_bytes(3, FMT_INT8, B, H, N, N, D)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=dev)
    ln = _lens_tensor(lens, dev)
    _check(_lib.sage_quantize_k_smooth(FMT_INT8, _ptr(k), _bnhd_strides(k), B, N, H, D, _ptr(ln),
                                       _ptr(out), _ptr(scale), _ptr(k_mean), _ptr(workspace),
                                       workspace.numel(), _stream()), "sage_quantize_k_smooth")
    return out, scale, k_mean


def sage_attn_fwd(fmt: int, q_q, q_scale, k_q, k_scale, v_q, v_scale, *, Nq: int, Nk: int,
                  k_lens=None, softmax_scale: Optional[float] = None, causal: int = 0,
                  out: Optional[torch.Tensor] = None, return_lse: bool = True,
                  lse: Optional[torch.Tensor] = None, num_splits: int = 0,
                  workspace: Optional[torch.Tensor] = None, k_mean: Optional[torch.Tensor] = None,
                  delta_s: Optional[torch.Tensor] = None, wait_cycles: int = 0,
                  test_withhold_v: bool = False, cta_mode: int = 0):
    """Attention forward on quantized operands. Returns (O ``[B, Nq, H, D]`` bf16, LSE or None).
    k_mean: the channel means from sage_quantize_k_smooth when K was smoothed.
    wait_cycles / test_withhold_v: sage_attn_options_t's wait bound and its
    testing-only withheld V loads. cta_mode: 0 library choice, 1 one-CTA tiles,
    2 two-CTA tiles (cta_group::2 pairs)."""
    B, H = q_q.shape[0], q_q.shape[1]
    D = 128
    dev = q_q.device
    if out is None:
        out = torch.empty((B, Nq, H, D), dtype=torch.bfloat16, device=dev)
    if return_lse and lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=dev)
    need = sage_workspace_bytes(2, fmt, B, H, Nq, Nk, D, num_splits)
    if need > 0 and (workspace is None or workspace.numel() < need):
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    ln = _lens_tensor(k_lens, dev)
    opts = AttnOptions(num_splits, int(cta_mode), None if k_mean is None else k_mean.data_ptr(),
                       None if delta_s is None else delta_s.data_ptr(), int(wait_cycles),
                       int(bool(test_withhold_v)), 0)
    sc = -1.0 if softmax_scale is None else float(softmax_scale)
    _check(_lib.sage_attn_fwd(fmt, _ptr(q_q), _ptr(q_scale), _ptr(k_q), _ptr(k_scale), _ptr(v_q),
                              _ptr(v_scale), _ptr(ln), B, H, Nq, Nk, D, sc, causal, _ptr(out),
                              _bnhd_strides(out), _ptr(lse if return_lse else None),
                              _ptr(workspace), 0 if workspace is None else workspace.numel(),
                              ctypes.byref(opts), _stream()), "sage_attn_fwd")
    return out, (lse if return_lse else None)


def sage_last_device_status() -> int:
    """Synchronise the current stream and read/clear the device status word."""
    return int(_lib.sage_last_device_status(_stream()))


def sage_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, fmt: int = FMT_INT8,
                   k_lens=None, softmax_scale: Optional[float] = None, num_splits: int = 0,
                   return_lse: bool = True, smooth_k: bool = False, smooth_q: bool = False,
                   cta_mode: int = 0):
    """Quantize Q/K/V (one sage_quantize_qkv call) and attend. smooth_q (INT8
    only) quantizes Q with sage_quantize_q_smooth and adds sage_delta_s's
    correction to the logits. smooth_k
    (INT8 only) quantizes K with sage_quantize_k_smooth and passes its channel
    means to the attention call."""
    B, Nq, H, D = q.shape
    Nk = k.shape[1]
    km = ds = None
    if smooth_k or smooth_q:
        if smooth_q:
            qq, qs, qm = sage_quantize_q_smooth(q)
        else:
            qq, qs = sage_quantize_qk(q, fmt)
        if smooth_k:
            kq, ks, km = sage_quantize_k_smooth(k, lens=k_lens)
        else:
            kq, ks = sage_quantize_qk(k, fmt, lens=k_lens)
        vq, vs = sage_quantize_v(v, lens=k_lens)
        if smooth_q:
            ds = sage_delta_s(qm, kq, ks, Nq=Nq, Nk=Nk, k_mean=km)
    else:
        (qq, qs), (kq, ks), (vq, vs) = sage_quantize_qkv(q, k, v, fmt, k_lens=k_lens)
    return sage_attn_fwd(fmt, qq, qs, kq, ks, vq, vs, Nq=Nq, Nk=Nk, k_lens=k_lens,
                         softmax_scale=softmax_scale, num_splits=num_splits,
                         return_lse=return_lse, k_mean=km, delta_s=ds, cta_mode=cta_mode)


def _host_desc(q, k, v, o, lse, lens, fmt, softmax_scale, smooth_k, smooth_q, heads_per_group,
               num_splits, cta_mode) -> HostAttention:
    B, Nq, H, D = q.shape
    addr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    return HostAttention(fmt, B, Nq, k.shape[1], H, D, addr(q), addr(k), addr(v), addr(o),
                         addr(lse), addr(lens),
                         float(softmax_scale) if softmax_scale else 0.0, int(smooth_k),
                         int(smooth_q), int(heads_per_group), int(num_splits), int(cta_mode))


def sage_attention_host_workspace_bytes(B: int, Nq: int, Nk: int, H: int, *, fmt: int = FMT_INT8,
                                        D: int = 128, smooth_k: bool = False,
                                        smooth_q: bool = False, heads_per_group: int = 0,
                                        num_splits: int = 0, cta_mode: int = 0,
                                        k_lens: bool = False, lse: bool = True) -> int:
    """Device workspace of sage_attention_host for these sizes (0 if invalid)."""
    one = 1  # non-null placeholders: only sizes are read
    d = HostAttention(fmt, B, Nq, Nk, H, D, one, one, one, one, one if lse else None,
                      one if k_lens else None, 0.0, int(smooth_k), int(smooth_q),
                      int(heads_per_group), int(num_splits), int(cta_mode))
    return int(_lib.sage_attention_host_workspace_bytes(ctypes.byref(d)))


def sage_attention_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, fmt: int = FMT_INT8,
                        k_lens=None, softmax_scale: Optional[float] = None, num_splits: int = 0,
                        smooth_k: bool = False, smooth_q: bool = False, cta_mode: int = 0,
                        heads_per_group: int = 0, out: Optional[torch.Tensor] = None,
                        lse: Optional[torch.Tensor] = None, return_lse: bool = True,
                        workspace: Optional[torch.Tensor] = None):
    """sage_attention on HOST tensors (contiguous BF16 [B, N, H, D] on the CPU,
    page-locked for copy/compute overlap): the library copies head groups in,
    quantizes and attends them, and copies O (and LSE) out, pipelined. Stream
    ordered on the current CUDA stream: synchronise it before reading the
    outputs. Returns host (o, lse)."""
    for t in (q, k, v):
        if t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous BF16 host tensors")
    B, Nq, H, D = q.shape
    Nk = k.shape[1]
    pin = q.is_pinned()
    if out is None:
        out = torch.empty((B, Nq, H, D), dtype=torch.bfloat16, pin_memory=pin)
    if lse is None and return_lse:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, pin_memory=pin)
    lens = None
    if k_lens is not None:
        lens = torch.as_tensor(k_lens, dtype=torch.int32).contiguous()
        if lens.is_cuda:
            raise ValueError("k_lens must be a host tensor or a sequence")
    d = _host_desc(q, k, v, out, lse, lens, fmt, softmax_scale, smooth_k, smooth_q,
                   heads_per_group, num_splits, cta_mode)
    need = int(_lib.sage_attention_host_workspace_bytes(ctypes.byref(d)))
    if need == 0:
        raise SageError(-1, "sage_attention_host_workspace_bytes")
    if workspace is None or workspace.numel() * workspace.element_size() < need:
        workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
    _check(_lib.sage_attention_host(ctypes.byref(d), _ptr(workspace), need, _stream()),
           "sage_attention_host")
    return out, lse


def int8_codes(x_q: torch.Tensor) -> torch.Tensor:
    """INT8 codes from the FP16-held quantized Q/K layout."""
    return x_q.to(torch.int8)
