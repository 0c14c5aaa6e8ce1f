"""sage_attention_host (host-resident Q/K/V, head groups pipelined through
copy-in, quantize + attend and copy-out) against the same library calls on
the whole device tensors: O and LSE must be equal bit for bit, since every
scale, code and row depends on its own head only and the split count and
tile mode are resolved for the whole shape."""
import pytest
import torch

from precision_attention_diffusion_sage_gb300.inputs import Workload, make_qkv

pytestmark = pytest.mark.gpu

binding = None


@pytest.fixture(scope="module", autouse=True)
def _lib():
    global binding
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from precision_attention_diffusion_sage_gb300 import build as sage_build
    sage_build.build()
    from precision_attention_diffusion_sage_gb300 import binding as b
    binding = b
    yield


def _device_reference(q, k, v, **kw):
    o, lse = binding.sage_attention(q.cuda(), k.cuda(), v.cuda(), **kw)
    torch.cuda.synchronize()
    assert binding.sage_last_device_status() == 0
    return o.cpu(), lse.cpu()


# fmt, B, H, Nq, Nk, k_lens, heads_per_group, splits, smooth_k, smooth_q, cta_mode
CASES = [
    (0, 2, 5, 300, 700, [700, 413], 2, 0, False, False, 0),
    (0, 1, 3, 256, 129, None, 0, 3, False, False, 0),
    (2, 1, 4, 257, 300, None, 3, 0, False, False, 0),
    (1, 1, 3, 200, 256, [100], 1, 0, False, False, 0),
    (3, 1, 2, 128, 384, None, 1, 0, False, False, 0),
    (4, 1, 3, 300, 300, None, 2, 0, False, False, 0),
    (0, 1, 3, 384, 300, [211], 2, 0, True, True, 0),
    (0, 2, 3, 200, 160, [0, 160], 0, 0, False, True, 0),
    (0, 1, 4, 512, 512, None, 3, 0, False, False, 2),
    (0, 1, 9, 640, 1000, None, 0, 0, True, False, 0),
    (0, 1, 1, 1, 1, None, 0, 0, False, False, 0),
    (2, 3, 2, 129, 2, [2, 0, 1], 1, 0, False, False, 0),
]


@pytest.mark.parametrize("case", CASES)
def test_host_pipeline_equals_device_calls(case):
    fmt, B, H, Nq, Nk, lens, hpg, splits, sk, sq, cta = case
    w = Workload("case", B, H, Nq, Nk, seed=11 * H + Nq, structure="k_mean")
    q, k, v = (t.pin_memory() for t in make_qkv(w))
    kw = dict(fmt=fmt, k_lens=lens, num_splits=splits, smooth_k=sk, smooth_q=sq, cta_mode=cta)
    ro, rl = _device_reference(q, k, v, **kw)
    o, lse = binding.sage_attention_host(q, k, v, heads_per_group=hpg, **kw)
    torch.cuda.synchronize()
    assert binding.sage_last_device_status() == 0
    assert torch.equal(o.view(torch.int16), ro.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), rl.view(torch.int32))


def test_host_pipeline_pageable_memory_side_stream_and_no_lse():
    """Pageable host buffers (copies without overlap), a side CUDA stream and
    no LSE output give the same O; the call is ordered on that stream."""
    w = Workload("case", 1, 6, 333, 500, seed=3)
    q, k, v = make_qkv(w)
    ro, _ = _device_reference(q, k, v)
    side = torch.cuda.Stream()
    with torch.cuda.stream(side):
        o, lse = binding.sage_attention_host(q, k, v, heads_per_group=4, return_lse=False)
    side.synchronize()
    assert lse is None
    assert torch.equal(o.view(torch.int16), ro.view(torch.int16))


def test_host_pipeline_full_size_long_video_heads():
    """The long-video shape (65520 tokens) on 4 of its heads, 2 per group,
    against the device calls."""
    w = Workload("case", 1, 4, 65520, 65520, seed=0)
    q, k, v = (t.pin_memory() for t in make_qkv(w))
    ro, rl = _device_reference(q, k, v)
    o, lse = binding.sage_attention_host(q, k, v, heads_per_group=2)
    torch.cuda.synchronize()
    assert binding.sage_last_device_status() == 0
    assert torch.equal(o.view(torch.int16), ro.view(torch.int16))
    assert torch.equal(lse.view(torch.int32), rl.view(torch.int32))
