"""Seeded synthetic workloads shared by the tests, the benchmark and the smoke check.

This module only draws random inputs; it holds none of the method's arithmetic.
Every workload is BF16 Q/K/V in ``[B, N, H, D]`` layout, drawn as FP32 standard
normals from a seeded ``torch.Generator`` and rounded to BF16, with the
per-workload structure below (diffusion-transformer attention shapes: image and
video DiT self-attention, long video sequences, 8K block-scaled and
cross-attention cases).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    seed: int
    fmt: int = 0                      # 0: INT8, 1: MXFP4, 2: FP8, 3: rotated MXFP4 Q/K (V FP8);
                                      # 4: MXFP4 Q/K, V and P
    structure: str = "plain"
    smooth_k: bool = False            # K smoothing (INT8 only): channel means removed from K
    smooth_q: bool = False            # Q smoothing (INT8 only): block means removed, dS added
    k_lens: Optional[List[int]] = field(default=None)
    D: int = 128

    @property
    def flops(self) -> float:
        """4*B*H*Nq*Nk*D with Nk summed over the batch for ragged keys."""
        nk_sum = sum(self.k_lens) if self.k_lens else self.B * self.Nk
        return 4.0 * self.H * self.Nq * nk_sum * self.D


WORKLOADS = {
    # small case: per-(head, channel) K offset ~ N(0, std 2) (outlier channels)
    "tiny": Workload("tiny", 1, 2, 256, 256, seed=0, structure="k_offset_std2"),
    # image DiT self-attention: 4096 image + 512 text tokens, 4 of 128 K channels x8
    "image_dit": Workload("image_dit", 1, 24, 4608, 4608, seed=1, structure="k_channels_x8"),
    # video DiT self-attention, per-(head, channel) K mean ~ N(0, 1)
    "video_dit": Workload("video_dit", 1, 40, 14040, 14040, seed=2, structure="k_mean"),
    # long video self-attention
    "long_video": Workload("long_video", 1, 40, 65520, 65520, seed=3),
    # block-scaled (MXFP4 Q/K) self-attention at 8K
    "mxfp4_self": Workload("mxfp4_self", 2, 24, 8192, 8192, seed=4, fmt=1),
    # cross-attention to 512 text tokens, dense and ragged per-batch key lengths
    "cross": Workload("cross", 2, 24, 8192, 512, seed=4),
    "cross_ragged": Workload("cross_ragged", 2, 24, 8192, 512, seed=4, k_lens=[512, 300]),
    "cross_ragged_mxfp4": Workload("cross_ragged_mxfp4", 2, 24, 8192, 512, seed=4, fmt=1,
                                   k_lens=[512, 300]),
    # FP8 E4M3 Q/K (the pages' FP8 QK^T / FP8 PV format) on the image and video shapes
    "image_dit_fp8": Workload("image_dit_fp8", 1, 24, 4608, 4608, seed=1, fmt=2,
                              structure="k_channels_x8"),
    "video_dit_fp8": Workload("video_dit_fp8", 1, 40, 14040, 14040, seed=2, fmt=2,
                              structure="k_mean"),
    # video DiT with K smoothing: the per-channel K means (the workload's
    # structure) taken out of K before INT8 quantization
    "video_dit_ksmooth": Workload("video_dit_ksmooth", 1, 40, 14040, 14040, seed=2,
                                  structure="k_mean", smooth_k=True),
    # MXFP4 Q/K with MXFP4 V and P (the FP4 P V format) on the 8K shape
    "mxfp4_v4_self": Workload("mxfp4_v4_self", 2, 24, 8192, 8192, seed=4, fmt=4),
    # video DiT with Q and K smoothing (Q block means out, dS in the logits)
    "video_dit_qksmooth": Workload("video_dit_qksmooth", 1, 40, 14040, 14040, seed=2,
                                   structure="k_mean", smooth_k=True, smooth_q=True),
    # Hadamard-rotated MXFP4 Q/K on the 8K shape, with the outlier-channel K
    # structure the rotation is meant to spread
    "mxfp4h_self": Workload("mxfp4h_self", 2, 24, 8192, 8192, seed=4, fmt=3,
                            structure="k_channels_x8"),
}


def make_qkv(w: Workload, device: str = "cpu", seed: Optional[int] = None):
    """Draw (q, k, v) as contiguous BF16 tensors ``[B, N, H, D]`` on ``device``."""
    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)
    f32 = dict(dtype=torch.float32, device=device, generator=g)
    q = torch.randn(w.B, w.Nq, w.H, w.D, **f32)
    k = torch.randn(w.B, w.Nk, w.H, w.D, **f32)
    v = torch.randn(w.B, w.Nk, w.H, w.D, **f32)
    if w.structure == "k_offset_std2":
        k += 2.0 * torch.randn(1, 1, w.H, w.D, **f32)
    elif w.structure == "k_channels_x8":
        ch = torch.randperm(w.D, generator=g, device=device)[:4]
        k[..., ch] *= 8.0
    elif w.structure == "k_mean":
        k += torch.randn(1, 1, w.H, w.D, **f32)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def bf16_bits(t: torch.Tensor):
    """Host numpy uint16 view of a BF16 tensor (keeps the strides)."""
    t = t.detach().cpu()
    return t.view(torch.int16).numpy().view("uint16")
