"""Shared helpers for the parity tests: run the oracle on the same seeded inputs
as the CUDA path and compare within the stated tolerances
(O: max-abs 1e-2 and cosine >= 0.9999; LSE: 1e-3 absolute; quantized tensors
and scales bit-exact)."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
from precision_attention_diffusion_sage_gb300.inputs import bf16_bits

O_MAX_ABS = 1e-2
O_MIN_COS = 0.9999
LSE_MAX_ABS = 1e-3


def oracle_quantize(fmt, q, k, v, k_lens=None):
    qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
    if fmt == 0:
        qz = oracle.quantize_int8(qb)
        kz = oracle.quantize_int8(kb, lens=k_lens)
    elif fmt == 2:
        qz = oracle.quantize_fp8_qk(qb)
        kz = oracle.quantize_fp8_qk(kb, lens=k_lens)
    elif fmt == 3:
        qz = oracle.quantize_mxfp4_hadamard(qb)
        kz = oracle.quantize_mxfp4_hadamard(kb, lens=k_lens)
    else:  # MXFP4 Q/K (formats 1 and 4)
        qz = oracle.quantize_mxfp4(qb)
        kz = oracle.quantize_mxfp4(kb, lens=k_lens)
    vz = oracle.quantize_v_mxfp4(vb, lens=k_lens) if fmt == 4 else oracle.quantize_v_fp8(vb, lens=k_lens)
    return qz, kz, vz


def oracle_attention_format(fmt, softmax_scale=None, D=128):
    """The oracle attention call for a library format: the rotated MXFP4
    format holds MXFP4 codes of QH and KH, whose logits (QH)(KH)^T are 128
    times QK^T, so it is MXFP4 attention with the multiplier divided by 128."""
    if fmt != 3:
        return fmt, softmax_scale
    c = 1.0 / math.sqrt(D) if softmax_scale is None or softmax_scale <= 0 else softmax_scale
    return 1, c / 128.0


def gpu_codes(fmt, x_q):
    """Host numpy view of the GPU's quantized Q/K data in the oracle's format."""
    if fmt == 0:
        return x_q.to(torch.int8).cpu().numpy()
    return x_q.cpu().numpy()


def assert_qk_equal(fmt, gpu_q, gpu_s, ref_q, ref_s):
    np.testing.assert_array_equal(gpu_codes(fmt, gpu_q), ref_q)
    gs = gpu_s.cpu().numpy()
    if fmt in (0, 2):  # float block scales, compared bit for bit
        np.testing.assert_array_equal(gs.view(np.uint32), ref_s.view(np.uint32))
    else:
        np.testing.assert_array_equal(gs, ref_s)


def assert_v_equal(gpu_v, gpu_s, ref_v, ref_s):
    """V codes and scales bit for bit: FP32 channel scales (E4M3 V) or E8M0
    bytes (MXFP4 V). The library's E4M3 V is token-major [B, H, Npad, D]; the
    oracle writes [B, H, D, Npad], so the comparison transposes the GPU's."""
    gs = gpu_s.cpu().numpy()
    if ref_s.dtype == np.uint8:
        np.testing.assert_array_equal(gpu_v.cpu().numpy(), ref_v)
        np.testing.assert_array_equal(gs, ref_s)
    else:
        np.testing.assert_array_equal(gpu_v.transpose(-1, -2).cpu().numpy(), ref_v)
        np.testing.assert_array_equal(gs.view(np.uint32), ref_s.view(np.uint32))


def compare_attention(o_gpu, lse_gpu, o_ref, lse_ref, rows=None):
    """o_gpu [B,Nq,H,D] bf16 (device), lse_gpu [B,H,Nq]; refs [B,H,nr,D] / [B,H,nr].
    Returns (max_abs, cosine, lse_max_abs)."""
    og = o_gpu.float().cpu().permute(0, 2, 1, 3).numpy().astype(np.float64)
    lg = lse_gpu.cpu().numpy().astype(np.float64)
    if rows is not None:
        og = og[:, :, rows]
        lg = lg[:, :, rows]
    max_abs = float(np.abs(og - o_ref).max()) if og.size else 0.0
    den = math.sqrt(float((og * og).sum()) * float((o_ref * o_ref).sum()))
    cos = float((og * o_ref).sum()) / den if den > 0 else 1.0
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lg), fin), "LSE finiteness differs"
    lse_err = float(np.abs(lg[fin] - lse_ref[fin]).max()) if fin.any() else 0.0
    return max_abs, cos, lse_err


def assert_attention_close(o_gpu, lse_gpu, o_ref, lse_ref, rows=None):
    max_abs, cos, lse_err = compare_attention(o_gpu, lse_gpu, o_ref, lse_ref, rows)
    assert max_abs <= O_MAX_ABS, f"O max-abs {max_abs}"
    assert cos >= O_MIN_COS, f"O cosine {cos}"
    assert lse_err <= LSE_MAX_ABS, f"LSE max-abs {lse_err}"
    return max_abs, cos, lse_err
