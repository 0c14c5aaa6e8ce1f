"""Host-only checks of the C-ABI library: it builds, loads without a GPU,
exports every entry point the header declares, sizes buffers as documented
and rejects invalid calls before any launch."""
import ctypes
import re

import pytest

from precision_attention_diffusion_sage_gb300 import build as sage_build

sage_build.build()
from precision_attention_diffusion_sage_gb300 import binding  # noqa: E402


def test_exports_every_header_symbol():
    names = binding.header_symbols()
    assert {"sage_quantize_qk", "sage_quantize_v", "sage_attn_fwd"} <= set(names)
    lib = binding.library()
    for n in names:
        assert hasattr(lib, n), n


def test_header_has_no_torch_types():
    text = open(binding.HEADER_PATH).read()
    for token in ("at::", "torch::", "Tensor", "#include <torch", "c10::"):
        assert token not in text, token
    assert 'extern "C"' in text


def test_quantized_bytes():
    B, N, H, D = 2, 300, 3, 128
    Np = 384
    assert binding.sage_quantized_bytes(0, 0, B, N, H, D) == B * H * Np * D * 2
    assert binding.sage_quantized_bytes(0, 1, B, N, H, D) == B * H * 3 * 4
    assert binding.sage_quantized_bytes(1, 0, B, N, H, D) == B * H * Np * 64
    assert binding.sage_quantized_bytes(1, 1, B, N, H, D) == B * H * Np * 4
    assert binding.sage_quantized_bytes(0, 2, B, N, H, D) == B * H * D * Np
    assert binding.sage_quantized_bytes(0, 3, B, N, H, D) == B * H * D * 4
    assert binding.sage_quantized_bytes(0, 0, B, N, H, 64) == 0      # D must be 128
    assert binding.sage_quantized_bytes(2, 0, B, N, H, D) == B * H * Np * D       # FP8 codes
    assert binding.sage_quantized_bytes(2, 1, B, N, H, D) == B * H * 3 * 4        # FP8 block scales
    assert binding.sage_quantized_bytes(3, 0, B, N, H, D) == B * H * Np * 64      # rotated MXFP4
    assert binding.sage_quantized_bytes(3, 1, B, N, H, D) == B * H * Np * 4
    assert binding.sage_quantized_bytes(7, 0, B, N, H, D) == 0       # unknown format


def test_workspace_bytes():
    assert binding.sage_workspace_bytes(0, 0, 1, 2, 256, 256) == 0
    assert binding.sage_workspace_bytes(1, 0, 1, 2, 1000, 1000) == 1 * 2 * 128 * 4  # channel maxima
    # forced splits: [splits][B][H][Nq][D] partial O + [splits][B][H][Nq] LSE, FP32
    assert binding.sage_workspace_bytes(2, 0, 1, 2, 256, 1024, 128, 3) == 3 * 2 * 256 * 129 * 4
    assert binding.sage_workspace_bytes(2, 0, 1, 2, 256, 1024, 128, 1) == 0
    # large grids need no split
    assert binding.sage_workspace_bytes(2, 0, 1, 40, 14040, 14040) == 0
    # K smoothing: an int64 sum and a binary32 maximum per channel; INT8 only
    assert binding.sage_workspace_bytes(3, 0, 2, 3, 300, 300) == 2 * 3 * 128 * 12
    assert binding.sage_workspace_bytes(3, 1, 2, 3, 300, 300) == 0


def _status(name):
    return {"SAGE_OK": 0, "SAGE_ERR_INVALID_ARG": -1, "SAGE_ERR_UNSUPPORTED": -2,
            "SAGE_ERR_WORKSPACE": -3}[name]


def test_host_validation_rejects_before_launch():
    lib = binding.library()
    S = binding.Strides(0, 0, 0)
    fake = ctypes.c_void_p(1 << 20)
    # D != 128 and causal are unsupported
    assert lib.sage_quantize_qk(0, fake, S, 1, 128, 1, 64, None, fake, fake, None) == -2
    assert lib.sage_attn_fwd(0, fake, fake, fake, fake, fake, fake, None, 1, 1, 128, 128, 128,
                             -1.0, 1, fake, S, None, None, 0, None, None) == -2
    # unknown format
    assert lib.sage_quantize_qk(9, fake, S, 1, 128, 1, 128, None, fake, fake, None) == -2
    # null / misaligned pointers and bad strides
    assert lib.sage_quantize_qk(0, None, S, 1, 128, 1, 128, None, fake, fake, None) == -1
    assert lib.sage_quantize_qk(0, ctypes.c_void_p((1 << 20) + 2), S, 1, 128, 1, 128, None, fake,
                                fake, None) == -1
    assert lib.sage_quantize_qk(0, fake, binding.Strides(0, 130, 0), 1, 128, 1, 128, None, fake,
                                fake, None) == -1
    # empty inputs
    assert lib.sage_quantize_qk(0, fake, S, 1, 0, 1, 128, None, fake, fake, None) == -1
    # V quantization needs its workspace
    assert lib.sage_quantize_v(fake, S, 1, 1000, 1, 128, None, fake, fake, None, 0, None) == -3
    # attention with a forced split and no workspace
    opts = binding.AttnOptions(4, 0)
    assert lib.sage_attn_fwd(0, fake, fake, fake, fake, fake, fake, None, 1, 1, 128, 1024, 128,
                             -1.0, 0, fake, S, None, None, 0, ctypes.byref(opts), None) == -3
    # K smoothing: INT8 only, needs its workspace and an aligned mean output
    ws = ctypes.c_void_p(1 << 24)
    assert lib.sage_quantize_k_smooth(1, fake, S, 1, 128, 1, 128, None, fake, fake, fake, ws,
                                      1 << 20, None) == -2
    assert lib.sage_quantize_k_smooth(0, fake, S, 1, 128, 1, 128, None, fake, fake, fake, None,
                                      0, None) == -3
    assert lib.sage_quantize_k_smooth(0, fake, S, 1, 128, 1, 128, None, fake, fake,
                                      ctypes.c_void_p((1 << 20) + 4), ws, 1 << 20, None) == -1
    # the channel means only go with the INT8 format, 16-byte aligned
    opts = binding.AttnOptions(1, 0, 1 << 20)
    assert lib.sage_attn_fwd(1, fake, fake, fake, fake, fake, fake, None, 1, 1, 128, 128, 128,
                             -1.0, 0, fake, S, None, None, 0, ctypes.byref(opts), None) == -2
    opts = binding.AttnOptions(1, 0, (1 << 20) + 4)
    assert lib.sage_attn_fwd(0, fake, fake, fake, fake, fake, fake, None, 1, 1, 128, 128, 128,
                             -1.0, 0, fake, S, None, None, 0, ctypes.byref(opts), None) == -1


def test_wait_bound_options_validated_before_launch():
    """The per-call wait bound and the testing-only withheld V loads are
    checked on the host: bound in [0, 2^31], withholding only with an explicit
    bound of at most 2^24 cycles, the reserved word zero."""
    lib = binding.library()
    S = binding.Strides(0, 0, 0)
    fake = ctypes.c_void_p(1 << 20)

    def call(**kw):
        opts = binding.AttnOptions(1, 0, None, None, kw.get("wait", 0), kw.get("withhold", 0),
                                   kw.get("reserved", 0))
        return lib.sage_attn_fwd(0, fake, fake, fake, fake, fake, fake, None, 1, 1, 128, 128, 128,
                                 -1.0, 0, fake, S, None, None, 0, ctypes.byref(opts), None)

    assert call(wait=-1) == -1
    assert call(wait=(1 << 31) + 1) == -1
    assert call(withhold=1) == -1                      # needs an explicit bound
    assert call(withhold=1, wait=(1 << 24) + 1) == -1  # and a short one
    assert call(withhold=2, wait=1 << 16) == -1
    assert call(reserved=1) == -1


def test_cta_mode_validated_before_launch():
    """cta_mode: 0, 1 or 2; 2-CTA tiles only for INT8 / FP8 Q/K with more
    than one query tile and no dS."""
    lib = binding.library()
    S = binding.Strides(0, 0, 0)
    fake = ctypes.c_void_p(1 << 20)

    def call(fmt, mode, Nq=256, ds=None):
        opts = binding.AttnOptions(1, mode, None, ds)
        return lib.sage_attn_fwd(fmt, fake, fake, fake, fake, fake, fake, None, 1, 1, Nq, 256, 128,
                                 -1.0, 0, fake, S, None, None, 0, ctypes.byref(opts), None)

    assert call(0, 3) == -1 and call(0, -1) == -1
    assert call(1, 2) == -2                 # MXFP4 Q/K
    assert call(4, 2) == -2                 # MXFP4 Q/K, V and P
    assert call(0, 2, Nq=128) == -2         # one query tile
    assert call(0, 2, ds=1 << 20) == -2     # Q smoothing's dS


def test_status_strings():
    lib = binding.library()
    for code in range(-7, 1):
        assert lib.sage_status_string(code).decode().startswith("SAGE_")
    assert binding.sage_version().startswith("libsage")


def test_new_entry_points_validate_before_launch():
    """The quantize / dS entry points reject bad formats, shapes, pointers and
    workspaces on the host, before any launch (no GPU is touched)."""
    lib = binding.library()
    S = binding.Strides(0, 0, 0)
    fake = ctypes.c_void_p(1 << 20)
    odd = ctypes.c_void_p((1 << 20) + 4)
    # Q smoothing and dS: INT8 only, D = 128, aligned outputs
    assert lib.sage_quantize_q_smooth(2, fake, S, 1, 128, 1, 128, fake, fake, fake, None) == -2
    assert lib.sage_quantize_q_smooth(0, fake, S, 1, 128, 1, 64, fake, fake, fake, None) == -2
    assert lib.sage_quantize_q_smooth(0, fake, S, 1, 128, 1, 128, fake, fake, odd, None) == -1
    assert lib.sage_delta_s(1, fake, fake, fake, None, 1, 1, 128, 128, 128, fake, None) == -2
    assert lib.sage_delta_s(0, fake, fake, fake, None, 1, 1, 0, 128, 128, fake, None) == -1
    assert lib.sage_delta_s(0, fake, fake, fake, None, 1, 1, 128, 128, 128, odd, None) == -1
    # MXFP4 V: D = 128 and aligned data
    assert lib.sage_quantize_v_mxfp4(fake, S, 1, 128, 1, 64, None, fake, fake, None) == -2
    assert lib.sage_quantize_v_mxfp4(odd, S, 1, 128, 1, 128, None, fake, fake, None) == -1
    # one-call quantization: unknown format, empty K, missing FP8 workspace
    assert lib.sage_quantize_qkv(9, fake, S, fake, S, fake, S, 1, 128, 128, 1, 128, None, fake,
                                 fake, fake, fake, fake, fake, None, 0, None) == -2
    assert lib.sage_quantize_qkv(0, fake, S, fake, S, fake, S, 1, 128, 0, 1, 128, None, fake,
                                 fake, fake, fake, fake, fake, None, 0, None) == -1
    assert lib.sage_quantize_qkv(0, fake, S, fake, S, fake, S, 1, 128, 128, 1, 128, None, fake,
                                 fake, fake, fake, fake, fake, None, 0, None) == -3
    # dS only goes with the INT8 format
    opts = binding.AttnOptions(1, 0, None, 1 << 20)
    assert lib.sage_attn_fwd(2, fake, fake, fake, fake, fake, fake, None, 1, 1, 128, 128, 128,
                             -1.0, 0, fake, S, None, None, 0, ctypes.byref(opts), None) == -2


def test_format4_byte_counts():
    B, N, H, D = 2, 300, 3, 128
    Np = 384
    assert binding.sage_quantized_bytes(4, 0, B, N, H, D) == B * H * Np * 64      # E2M1 Q/K
    assert binding.sage_quantized_bytes(4, 1, B, N, H, D) == B * H * Np * 4       # E8M0 Q/K
    assert binding.sage_quantized_bytes(4, 2, B, N, H, D) == B * H * D * Np // 2  # E2M1 V^T
    assert binding.sage_quantized_bytes(4, 3, B, N, H, D) == B * H * Np * D // 32  # E8M0 V
    assert binding.sage_workspace_bytes(1, 4, B, H, N, N) == 0                     # no V maxima


def _host_desc(**kw):
    d = dict(fmt=0, B=1, Nq=300, Nk=500, H=5, D=128, q=1 << 20, k=1 << 20, v=1 << 20, o=1 << 20,
             lse=1 << 20, k_lens=None, softmax_scale=0.0, smooth_k=0, smooth_q=0,
             heads_per_group=0, num_splits=0, cta_mode=0)
    d.update(kw)
    return binding.HostAttention(**d)


def test_host_attention_workspace_and_validation():
    """sage_attention_host: its workspace is two slots of one head group's
    buffers plus the key lengths (no CUDA call), and invalid calls are
    rejected before any CUDA call."""
    lib = binding.library()
    size = lambda **kw: lib.sage_attention_host_workspace_bytes(ctypes.byref(_host_desc(**kw)))  # noqa: E731
    B, Nq, Nk, D = 1, 300, 500, 128
    r = lambda x: (x + 255) // 256 * 256  # noqa: E731
    # one head per group, INT8: BF16 Q/K/V, codes, scales, V scales, O, LSE
    slot = (r(B * Nq * D * 2) + 2 * r(B * Nk * D * 2) + r(384 * D * 2) + r(3 * 4) + r(512 * D * 2)
            + r(4 * 4) + r(512 * D) + r(D * 4) + r(B * Nq * D * 2) + r(Nq * 4) + r(D * 4))
    assert size(heads_per_group=1, num_splits=1) == 2 * slot + 256
    # the split count is resolved for the whole shape; each group holds its partials
    splits = 3
    assert size(heads_per_group=1, num_splits=splits) == 2 * (slot + r(splits * Nq * (D + 1) * 4)) + 256
    # grows with the group; by default about 5 groups, or about 20 when each
    # head's attention outlasts its copies several times over (long sequences)
    assert size(heads_per_group=2) > size(heads_per_group=1)
    assert size(heads_per_group=0) == size(heads_per_group=1)  # H = 5 -> 5 groups of 1
    assert size(H=40) == size(H=40, heads_per_group=8)
    assert size(H=40, Nq=65520, Nk=65520) == size(H=40, Nq=65520, Nk=65520, heads_per_group=2)
    # smoothing adds its buffers; invalid descriptions size to 0
    assert size(smooth_k=1, smooth_q=1) > size()
    for bad in (dict(D=64), dict(fmt=9), dict(smooth_k=1, fmt=1), dict(heads_per_group=6),
                dict(heads_per_group=-1), dict(q=None), dict(o=None), dict(num_splits=65),
                dict(cta_mode=3), dict(Nq=0), dict(smooth_q=2)):
        assert size(**bad) == 0, bad
    assert lib.sage_attention_host_workspace_bytes(None) == 0
    # the call itself: the same checks, then the workspace, before any CUDA call
    call = lambda ws, n, **kw: lib.sage_attention_host(ctypes.byref(_host_desc(**kw)), ws, n, None)  # noqa: E731
    ws = ctypes.c_void_p(1 << 24)
    assert lib.sage_attention_host(None, ws, 1 << 30, None) == -1
    assert call(ws, 1 << 30, D=64) == -2
    assert call(ws, 1 << 30, smooth_q=1, fmt=2) == -2
    assert call(ws, 1 << 30, heads_per_group=9) == -1
    assert call(ws, 1 << 30, softmax_scale=float("inf")) == -1
    assert call(None, 1 << 30) == -3
    assert call(ws, size() - 1) == -3
    assert call(ctypes.c_void_p((1 << 24) + 16), 1 << 30) == -3  # 256-byte alignment
