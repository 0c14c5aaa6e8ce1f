"""Pins against the values the pages print (tests/golden/printed_values.txt):
the base-2 softmax constant, the head dimension and masking the boundary
accepts, and the operand formats of the oracle and the library."""
import ctypes
import math
import os

import numpy as np
import scipy.special

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "printed_values.txt")


def _bf16(x):
    """BF16 bit patterns of float values (round to nearest even)."""
    import torch
    from precision_attention_diffusion_sage_gb300.inputs import bf16_bits
    return bf16_bits(torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16))


def _printed():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                name, value = line.split(None, 1)
                vals[name] = value
    return vals


def test_printed_log2e_is_the_double_nearest_log2_e():
    l2e = float(_printed()["MHA_V4_LOG2E"])
    assert l2e == math.log2(math.e)
    assert abs(l2e * math.log(2.0) - 1.0) < 2 ** -52
    assert oracle.LOG2E == l2e


def test_oracle_softmax_in_base_2_matches_natural_logsumexp():
    """Two keys with exact integer logits S = 17 and S = -5 under an INT8 Q
    code of 1: the oracle's base-2 softmax (t = S c log2e, LSE = (M + log2 l)
    ln 2) must give the natural-log logsumexp of c S, and weights e^{cS}
    normalised, whatever the page's constant makes of the exponent."""
    D = 128
    q = np.zeros((1, 1, 128, D), np.int8)
    k = np.zeros((1, 1, 128, D), np.int8)
    q[0, 0, 0, 0] = 1
    k[0, 0, 0, 0], k[0, 0, 1, 0] = 17, -5
    qs = np.ones((1, 1, 1), np.float32)
    ks = np.ones((1, 1, 1), np.float32)
    v8 = np.zeros((1, 1, D, 128), np.uint8)
    sv = np.zeros((1, 1, D), np.float32)
    c = 0.125
    o, lse, w = oracle.attention(0, q, qs, k, ks, v8, sv, Nq=1, Nk=2, softmax_scale=c,
                                 want_weights=True)
    logits = np.array([17.0 * c, -5.0 * c])
    assert abs(lse[0, 0, 0] - scipy.special.logsumexp(logits)) < 1e-12
    # the weights are the P8-coded probabilities over l (E4M3 rounding of
    # p 2^8 stays within 2^-4 relative)
    p = scipy.special.softmax(logits)
    assert np.all(np.abs(w[0, 0, 0] - p) <= p * 2.0 ** -4)


def test_boundary_takes_the_printed_head_dim_and_masking():
    from precision_attention_diffusion_sage_gb300 import build as sage_build
    sage_build.build()
    from precision_attention_diffusion_sage_gb300 import binding
    g = _printed()
    D = int(g["HEAD_DIM"])
    assert D == 128
    # the quantized layouts exist for the printed head dimension only
    assert binding.sage_quantized_bytes(0, 0, 1, 256, 1, D) > 0
    assert binding.sage_quantized_bytes(0, 0, 1, 256, 1, D // 2) == 0
    assert binding.sage_quantized_bytes(0, 0, 1, 256, 1, 2 * D) == 0
    # non-causal only: a causal request is refused before any launch
    assert int(g["CAUSAL"]) == 0
    lib = binding.library()
    S = binding.Strides(0, 0, 0)
    fake = ctypes.c_void_p(1 << 20)
    assert lib.sage_attn_fwd(0, fake, fake, fake, fake, fake, fake, None, 1, 1, 128, 128, D,
                             -1.0, 1, fake, S, None, None, 0, None, None) == -2


def test_formats_cover_the_printed_operands():
    """The library's format enum has the printed combinations: INT8 Q/K with
    FP8 P V, MXFP4 (E2M1) Q/K, BF16 output; the oracle codes the same types."""
    from precision_attention_diffusion_sage_gb300 import binding
    g = _printed()
    assert (g["QK_OPERAND"], g["PV_OPERAND"], g["OUTPUT"]) == ("INT8", "FP8", "BF16")
    assert g["MX_QK_OPERAND"] == "MXFP4_E2M1"
    text = open(binding.HEADER_PATH).read()
    assert "SAGE_FMT_QK_INT8_V_FP8" in text and "SAGE_FMT_QK_MXFP4_V_FP8" in text
    # INT8 codes stay within +-127 and E2M1 codes are nibbles of the eight
    # magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}
    x = np.linspace(-3.0, 3.0, 128 * 128).reshape(1, 128, 1, 128)
    xb = _bf16(x)
    codes, _ = oracle.quantize_int8(xb)
    assert codes.min() >= -127 and codes.max() <= 127
    mx, _ = oracle.quantize_mxfp4(xb)
    assert mx.dtype == np.uint8
