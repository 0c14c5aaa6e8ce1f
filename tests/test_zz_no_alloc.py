"""sage_quantize_v_noalloc: the entry point for callers that cannot allocate
device memory (their framework owns all device memory, or their memory plan is
fixed up front). It keeps its scratch in a fixed array inside the library.
Checked here, through the C ABI, against sage_quantize_v with a caller-owned
workspace, on two calls in a row (different shapes and data, so a stale array
would show). Collected last on purpose; it passes alone and after the others.
"""
import ctypes

import pytest
import torch

from precision_attention_diffusion_sage_gb300.inputs import Workload, make_qkv

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from precision_attention_diffusion_sage_gb300 import build as sage_build
    sage_build.build()
    from precision_attention_diffusion_sage_gb300 import binding
    return binding


def _noalloc(binding, v, lens):
    B, N, H, D = v.shape
    Np = binding.pad128(N)
    out = torch.full((B, H, Np, D), 0xAB, dtype=torch.uint8, device=v.device)
    scale = torch.full((B, H, D), -1.0, dtype=torch.float32, device=v.device)
    ln = None if lens is None else torch.tensor(lens, dtype=torch.int32, device=v.device)
    f = binding.library().sage_quantize_v_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, binding.Strides, ctypes.c_int64, ctypes.c_int64,
                  ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p]
    st = f(ctypes.c_void_p(v.data_ptr()), binding.Strides(*v.stride()[:3]), B, N, H, D,
           None if ln is None else ctypes.c_void_p(ln.data_ptr()), ctypes.c_void_p(out.data_ptr()),
           ctypes.c_void_p(scale.data_ptr()),
           ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, binding.library().sage_status_string(st)
    return out, scale


def test_noalloc_matches_workspace_path_twice(lib):
    """The first call leaves channel maxima about 100 times larger than the
    second call's in every word the second call uses (at least as many
    (batch, head) pairs, V scaled by 100), so a second call that skipped the
    clear of the shared array would keep the first call's scales."""
    cases = [(Workload("a", 2, 4, 1000, 1000, seed=91), [1000, 700], 100.0),
             (Workload("b", 2, 3, 3000, 3000, seed=92), [2500, 3000], 1.0)]
    for w, lens, gain in cases:
        _, _, v = make_qkv(w)
        v = (v.float() * gain).to(torch.bfloat16).cuda()
        got_q, got_s = _noalloc(lib, v, lens)
        ref_q, ref_s = lib.sage_quantize_v(v, lens=lens)
        torch.cuda.synchronize()
        assert lib.sage_last_device_status() == 0
        assert torch.equal(got_q, ref_q)
        assert torch.equal(got_s.view(torch.int32), ref_s.view(torch.int32))


def test_noalloc_rejects_oversize(lib):
    v = torch.zeros((1, 128, 1, 128), dtype=torch.bfloat16, device="cuda")
    f = lib.library().sage_quantize_v_noalloc
    f.restype = ctypes.c_int
    # B * H * 128 words beyond the 8 MiB array (B * H > 16384): rejected before any launch
    st = f(ctypes.c_void_p(v.data_ptr()), lib.Strides(0, 0, 0), 2, 128, 8200, 128, None,
           ctypes.c_void_p(v.data_ptr()), ctypes.c_void_p(v.data_ptr()), None)
    assert st == -3  # SAGE_ERR_WORKSPACE
