"""CPU oracle for quantized (Sage-style) attention forward — TEST INFRASTRUCTURE.

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package. It is a ctypes wrapper over ``sage_oracle.cpp`` (plain
C++, FP64 arithmetic) and shares nothing with the CUDA library.

Parity pins live in ``tests/test_oracle.py``; every function below is pinned
there against brute force, closed forms, invariants or a library routine.

Arrays: BF16 inputs are passed as ``numpy.uint16`` bit patterns with shape
``[B, N, H, D]`` (any strides, unit stride along D).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sage_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")

LOG2E = 1.4426950408889634


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` with g++ (IEEE arithmetic, no contraction)."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= max(os.path.getmtime(_SRC),
                                              os.path.getmtime(os.path.join(_HERE, "sage_oracle.h")))):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
           "-ffp-contract=off", "-fno-fast-math", "-o", tmp, _SRC]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


_lib = None


def _L():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P, I64, I32, D = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_double
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_encode.argtypes = [D]
        lib.oracle_e4m3_decode.restype = D
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_e2m1_encode.restype = ctypes.c_uint8
        lib.oracle_e2m1_encode.argtypes = [D]
        lib.oracle_e2m1_decode.restype = D
        lib.oracle_e2m1_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_int8_quantize_value.restype = I32
        lib.oracle_int8_quantize_value.argtypes = [ctypes.c_float, ctypes.c_float]
        lib.oracle_bf16_from_double.restype = ctypes.c_uint16
        lib.oracle_bf16_from_double.argtypes = [D]
        q_args = [P, I64, I64, I64, I64, I64, I64, I64, P, P, P]
        for name in ("oracle_quantize_int8", "oracle_quantize_v_fp8", "oracle_quantize_mxfp4",
                     "oracle_quantize_fp8_qk", "oracle_quantize_mxfp4_hadamard",
                     "oracle_quantize_v_mxfp4"):
            getattr(lib, name).restype = None
            getattr(lib, name).argtypes = q_args
        lib.oracle_k_mean.restype = None
        lib.oracle_k_mean.argtypes = [P, I64, I64, I64, I64, I64, I64, I64, P, P]
        lib.oracle_quantize_int8_smooth.restype = None
        lib.oracle_quantize_int8_smooth.argtypes = [P, I64, I64, I64, I64, I64, I64, I64, P, P, P,
                                                    P]
        lib.oracle_k_mean_lse_term.restype = None
        lib.oracle_k_mean_lse_term.argtypes = [P, P, P, I64, I64, I64, I64, D, P, I64, P]
        lib.oracle_fwht128.restype = None
        lib.oracle_fwht128.argtypes = [P, P, I64]
        lib.oracle_attention.restype = None
        lib.oracle_attention.argtypes = [I32, P, P, P, P, P, P, P, I64, I64, I64, I64, I64, D,
                                         P, I64, P, P, P, I32, P, I32]
        lib.oracle_quantize_int8_qsmooth.restype = None
        lib.oracle_quantize_int8_qsmooth.argtypes = [P, I64, I64, I64, I64, I64, I64, I64, P, P, P,
                                                     P]
        lib.oracle_delta_s.restype = None
        lib.oracle_delta_s.argtypes = [P, P, P, P, I64, I64, I64, I64, I64, P]
        lib.oracle_attention_exact.restype = None
        lib.oracle_attention_exact.argtypes = [P, I64, I64, I64, P, I64, I64, I64, P, I64, I64,
                                               I64, P, I64, I64, I64, I64, I64, D, P, I64, P, P,
                                               I32]
        for name in ("oracle_p8_final",):
            getattr(lib, name).restype = None
            getattr(lib, name).argtypes = [P, I64, P]
        lib.oracle_p8_online.restype = None
        lib.oracle_p8_online.argtypes = [P, I64, I64, P]
        _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _bnhd(x: np.ndarray):
    assert x.dtype == np.uint16 and x.ndim == 4 and x.strides[3] == 2, "BF16 bits [B,N,H,D], unit D stride"
    B, N, H, D = x.shape
    sb, sn, sh = (s // 2 for s in x.strides[:3])
    return B, N, H, D, sb, sn, sh


def _lens(lens) -> Optional[np.ndarray]:
    return None if lens is None else np.ascontiguousarray(np.asarray(lens, dtype=np.int32))


def pad128(n: int) -> int:
    return (n + 127) // 128 * 128


# ------------------------------------------------------------------ scalars
def e4m3_encode(x: float) -> int:
    return int(_L().oracle_e4m3_encode(float(x)))


def e4m3_decode(c: int) -> float:
    return float(_L().oracle_e4m3_decode(int(c)))


def e2m1_encode(x: float) -> int:
    return int(_L().oracle_e2m1_encode(float(x)))


def e2m1_decode(c: int) -> float:
    return float(_L().oracle_e2m1_decode(int(c)))


def int8_quantize_value(x: float, s: float) -> int:
    return int(_L().oracle_int8_quantize_value(float(x), float(s)))


def bf16_from_double(x: float) -> int:
    return int(_L().oracle_bf16_from_double(float(x)))


# ------------------------------------------------------------------ quantize
def quantize_int8(x: np.ndarray, lens=None) -> Tuple[np.ndarray, np.ndarray]:
    """INT8 codes [B,H,Npad,D] and FP32 block scales [B,H,Npad/128]."""
    B, N, H, D, sb, sn, sh = _bnhd(x)
    Np = pad128(N)
    q = np.zeros((B, H, Np, D), np.int8)
    s = np.zeros((B, H, Np // 128), np.float32)
    ln = _lens(lens)
    _L().oracle_quantize_int8(_ptr(x), sb, sn, sh, B, N, H, D, _ptr(ln), _ptr(q), _ptr(s))
    return q, s


def quantize_v_fp8(v: np.ndarray, lens=None) -> Tuple[np.ndarray, np.ndarray]:
    """E4M3 codes [B,H,D,Npad] (token-contiguous) and FP32 scales [B,H,D]."""
    B, N, H, D, sb, sn, sh = _bnhd(v)
    Np = pad128(N)
    v8 = np.zeros((B, H, D, Np), np.uint8)
    sv = np.zeros((B, H, D), np.float32)
    ln = _lens(lens)
    _L().oracle_quantize_v_fp8(_ptr(v), sb, sn, sh, B, N, H, D, _ptr(ln), _ptr(v8), _ptr(sv))
    return v8, sv


def quantize_v_mxfp4(v: np.ndarray, lens=None) -> Tuple[np.ndarray, np.ndarray]:
    """MXFP4 V along tokens: codes [B,H,D,Npad/2] (token 2i in the low nibble)
    and E8M0 bytes [B,H,Npad/128,D,4] (32-token blocks, per 128-token tile)."""
    B, N, H, D, sb, sn, sh = _bnhd(v)
    Np = pad128(N)
    c = np.zeros((B, H, D, Np // 2), np.uint8)
    e = np.zeros((B, H, Np // 128, D, 4), np.uint8)
    ln = _lens(lens)
    _L().oracle_quantize_v_mxfp4(_ptr(v), sb, sn, sh, B, N, H, D, _ptr(ln), _ptr(c), _ptr(e))
    return c, e


def fwht128(x: np.ndarray) -> np.ndarray:
    """Binary32 fast Walsh-Hadamard transform of the last axis (length 128)."""
    xin = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty_like(xin)
    _L().oracle_fwht128(_ptr(xin), _ptr(out), xin.size // 128)
    return out


def quantize_mxfp4_hadamard(x: np.ndarray, lens=None) -> Tuple[np.ndarray, np.ndarray]:
    """MXFP4 codes [B,H,Npad,D/2] and E8M0 scales [B,H,Npad,D/32] of the
    Hadamard-rotated rows; pair with softmax_scale / 128 in attention()."""
    B, N, H, D, sb, sn, sh = _bnhd(x)
    Np = pad128(N)
    c = np.zeros((B, H, Np, D // 2), np.uint8)
    e = np.zeros((B, H, Np, D // 32), np.uint8)
    ln = _lens(lens)
    _L().oracle_quantize_mxfp4_hadamard(_ptr(x), sb, sn, sh, B, N, H, D, _ptr(ln), _ptr(c),
                                        _ptr(e))
    return c, e


def k_mean(x: np.ndarray, lens=None) -> np.ndarray:
    """Per-(b,h,channel) K mean over the valid tokens, float32 [B,H,D], from the
    exact fixed-point sum (grid 2^(E-40), E the exponent of the channel maximum)."""
    B, N, H, D, sb, sn, sh = _bnhd(x)
    mu = np.zeros((B, H, D), np.float32)
    ln = _lens(lens)
    _L().oracle_k_mean(_ptr(x), sb, sn, sh, B, N, H, D, _ptr(ln), _ptr(mu))
    return mu


def quantize_int8_smooth(x: np.ndarray, lens=None) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """K smoothing then INT8: (codes [B,H,Npad,D], block scales [B,H,Npad/128],
    channel means [B,H,D]) with codes/scales those of (float)k - mean."""
    B, N, H, D, sb, sn, sh = _bnhd(x)
    Np = pad128(N)
    mu = k_mean(x, lens=lens)
    q = np.zeros((B, H, Np, D), np.int8)
    s = np.zeros((B, H, Np // 128), np.float32)
    ln = _lens(lens)
    _L().oracle_quantize_int8_smooth(_ptr(x), sb, sn, sh, B, N, H, D, _ptr(ln), _ptr(mu), _ptr(q),
                                     _ptr(s))
    return q, s, mu


def quantize_int8_qsmooth(x: np.ndarray, lens=None):
    """Q smoothing then INT8: (codes [B,H,Npad,D], block scales [B,H,Npad/128],
    block channel means [B,H,Npad/128,D])."""
    B, N, H, D, sb, sn, sh = _bnhd(x)
    Np = pad128(N)
    q = np.zeros((B, H, Np, D), np.int8)
    s = np.zeros((B, H, Np // 128), np.float32)
    m = np.zeros((B, H, Np // 128, D), np.float32)
    ln = _lens(lens)
    _L().oracle_quantize_int8_qsmooth(_ptr(x), sb, sn, sh, B, N, H, D, _ptr(ln), _ptr(q), _ptr(s),
                                      _ptr(m))
    return q, s, m


def delta_s(k8: np.ndarray, k_scale: np.ndarray, q_mean: np.ndarray, *, Nq: int, Nk: int,
            k_mean=None) -> np.ndarray:
    """dS [B,H,Nq_pad/128,Nk_pad] float64: q_grid . (dequantized K + K's channel means),
    q_grid the block means on the 16-bit grid 2^(E-13) (see q_grid())."""
    B, H, _, D = k8.shape
    out = np.zeros((B, H, pad128(Nq) // 128, pad128(Nk)), np.float64)
    ka, sa, qa = (np.ascontiguousarray(a) for a in (k8, k_scale, q_mean))
    km = None if k_mean is None else np.ascontiguousarray(k_mean, dtype=np.float32)
    _L().oracle_delta_s(_ptr(ka), _ptr(sa), _ptr(km), _ptr(qa), B, H, Nq, Nk, D, _ptr(out))
    return out


def q_grid(q_mean: np.ndarray) -> np.ndarray:
    """The block means as dS uses them: per block, E = exponent of the largest
    |mean|, values rounded (nearest even) to multiples of 2^(E - 13)."""
    qm = np.asarray(q_mean, dtype=np.float32)
    amax = np.abs(qm).max(axis=-1, keepdims=True)
    e = ((amax.view(np.uint32) >> 23) & 0xFF).astype(np.int64)
    E = np.maximum(e, 1) - 127
    return np.rint(qm.astype(np.float64) * np.exp2(13.0 - E)) * np.exp2(E - 13.0)


def k_mean_lse_term(q: np.ndarray, q_scale: np.ndarray, mu: np.ndarray, *, Nq: int,
                    softmax_scale: Optional[float] = None, rows=None) -> np.ndarray:
    """softmax_scale * (s_q q8_i) . mu for every (b, h, evaluated row): the
    per-row logit offset that K smoothing removes, [B,H,nrows] float64."""
    B, H, _, D = q.shape
    c = 1.0 / math.sqrt(D) if softmax_scale is None or softmax_scale <= 0 else float(softmax_scale)
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    nr = Nq if r is None else len(r)
    out = np.zeros((B, H, nr), np.float64)
    qa, sa, ma = (np.ascontiguousarray(a) for a in (q, q_scale, mu))
    _L().oracle_k_mean_lse_term(_ptr(qa), _ptr(sa), _ptr(ma), B, H, Nq, D, c, _ptr(r), nr,
                                _ptr(out))
    return out


def quantize_fp8_qk(x: np.ndarray, lens=None) -> Tuple[np.ndarray, np.ndarray]:
    """E4M3 codes [B,H,Npad,D] and FP32 block scales [B,H,Npad/128] (absmax/448)."""
    B, N, H, D, sb, sn, sh = _bnhd(x)
    Np = pad128(N)
    q = np.zeros((B, H, Np, D), np.uint8)
    s = np.zeros((B, H, Np // 128), np.float32)
    ln = _lens(lens)
    _L().oracle_quantize_fp8_qk(_ptr(x), sb, sn, sh, B, N, H, D, _ptr(ln), _ptr(q), _ptr(s))
    return q, s


def quantize_mxfp4(x: np.ndarray, lens=None) -> Tuple[np.ndarray, np.ndarray]:
    """Packed E2M1 codes [B,H,Npad,D/2] and E8M0 scales [B,H,Npad,D/32]."""
    B, N, H, D, sb, sn, sh = _bnhd(x)
    Np = pad128(N)
    c = np.zeros((B, H, Np, D // 2), np.uint8)
    e = np.zeros((B, H, Np, D // 32), np.uint8)
    ln = _lens(lens)
    _L().oracle_quantize_mxfp4(_ptr(x), sb, sn, sh, B, N, H, D, _ptr(ln), _ptr(c), _ptr(e))
    return c, e


# ------------------------------------------------------------------ attention
def attention(fmt: int, q, q_scale, k, k_scale, v8, sv, *, Nq: int, Nk: int, D: int = 128,
              softmax_scale: Optional[float] = None, k_lens=None, rows=None,
              want_weights: bool = False, nthreads: int = 0, k_mean=None, delta_s=None,
              logits32: bool = False):
    """Quantized attention. fmt 0: INT8 Q/K; fmt 1: MXFP4 Q/K; fmt 2: E4M3 Q/K (V E4M3);
    fmt 4: MXFP4 Q/K with MXFP4 V (quantize_v_mxfp4) and MXFP4 P per 32 keys.

    logits32 (fmt 0 only): form the logits in binary32, the precision in which
    the INT8 format decides its FP8 P codes (see oracle_attention in
    sage_oracle.h); the default forms them in binary64.

    delta_s (fmt 0 only): the Q smoothing correction of delta_s(), added to every
    logit of the rows of each 128-query block.
    k_mean (fmt 0 only): the channel means that K smoothing subtracted before
    quantizing K; O is that of the smoothed logits and LSE adds back the
    per-row term softmax_scale * q^ . mean (k_mean_lse_term).

    Returns (o [B,H,nrows,D] float64, lse [B,H,nrows] float64, w or None).
    """
    B, H = q.shape[0], q.shape[1]
    c = 1.0 / math.sqrt(D) if softmax_scale is None or softmax_scale <= 0 else float(softmax_scale)
    arrs = [np.ascontiguousarray(a) for a in (q, q_scale, k, k_scale, v8, sv)]
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    nr = Nq if r is None else len(r)
    o = np.zeros((B, H, nr, D), np.float64)
    lse = np.zeros((B, H, nr), np.float64)
    w = np.zeros((B, H, nr, Nk), np.float64) if want_weights else None
    ln = _lens(k_lens)
    ds = None if delta_s is None else np.ascontiguousarray(delta_s, dtype=np.float64)
    assert ds is None or fmt == 0, "Q smoothing is defined for the INT8 Q/K format"
    assert not logits32 or fmt == 0, "binary32 logits are defined for the INT8 Q/K format"
    _L().oracle_attention(fmt, *(_ptr(a) for a in arrs), _ptr(ln), B, H, Nq, Nk, D, c, _ptr(r),
                          nr, _ptr(o), _ptr(lse), _ptr(w), nthreads, _ptr(ds), int(logits32))
    if k_mean is not None:
        assert fmt == 0, "K smoothing is defined for the INT8 Q/K format"
        lse = lse + k_mean_lse_term(q, q_scale, k_mean, Nq=Nq, softmax_scale=c, rows=r)
    return o, lse, w


def attention_exact(q: np.ndarray, k: np.ndarray, v: np.ndarray, *, softmax_scale=None,
                    k_lens=None, rows=None, nthreads: int = 0):
    """Unquantized FP64 softmax attention of BF16 inputs [B,N,H,D]."""
    B, Nq, H, D, qsb, qsn, qsh = _bnhd(q)
    _, Nk, _, _, ksb, ksn, ksh = _bnhd(k)
    _, _, _, _, vsb, vsn, vsh = _bnhd(v)
    c = 1.0 / math.sqrt(D) if softmax_scale is None or softmax_scale <= 0 else float(softmax_scale)
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    nr = Nq if r is None else len(r)
    o = np.zeros((B, H, nr, D), np.float64)
    lse = np.zeros((B, H, nr), np.float64)
    ln = _lens(k_lens)
    _L().oracle_attention_exact(_ptr(q), qsb, qsn, qsh, _ptr(k), ksb, ksn, ksh, _ptr(v), vsb, vsn,
                                vsh, _ptr(ln), B, H, Nq, Nk, D, c, _ptr(r), nr, _ptr(o), _ptr(lse),
                                nthreads)
    return o, lse


def p8_final(t: np.ndarray) -> np.ndarray:
    t = np.ascontiguousarray(t, dtype=np.float64)
    out = np.zeros_like(t)
    _L().oracle_p8_final(_ptr(t), len(t), _ptr(out))
    return out


def p8_online(t: np.ndarray, tile: int) -> np.ndarray:
    t = np.ascontiguousarray(t, dtype=np.float64)
    out = np.zeros_like(t)
    _L().oracle_p8_online(_ptr(t), len(t), tile, _ptr(out))
    return out


def bf16_round(o: np.ndarray) -> np.ndarray:
    """Round float64 values to BF16 (returned as uint16 bit patterns)."""
    f = np.vectorize(bf16_from_double, otypes=[np.uint16])
    return f(o)
