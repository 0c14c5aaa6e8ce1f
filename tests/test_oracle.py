"""Pins for the CPU oracle: every oracle function is checked against something
other than itself — brute force over the format tables, a library routine
(torch's float8/bfloat16 conversions, SDPA, scipy's logsumexp/softmax),
closed forms and invariants — so that a dropped term, a wrong sign, index or
layout fails at least one test.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from precision_attention_diffusion_sage_gb300.inputs import WORKLOADS, Workload, bf16_bits, make_qkv

L2E = 1.4426950408889634


# ------------------------------------------------------------------ format tables
def _e4m3_table():
    """(code, value) for every finite E4M3 code, decoded by torch's float8_e4m3fn."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    vals = torch.from_numpy(codes).view(torch.float8_e4m3fn).double().numpy()
    return codes, vals


def _nearest_even(x, codes, vals, max_mag):
    """Brute force: the table value nearest to x; ties to the even code."""
    a = min(abs(x), max_mag)
    mags = np.abs(vals)
    d = np.abs(mags - a)
    best = d.min()
    cand = [int(c) & 0x7F for c, v, dd in zip(codes, vals, d) if dd == best and v >= 0]
    even = [c for c in cand if c % 2 == 0]
    mag_code = even[0] if even else cand[0]
    return mag_code


def test_e4m3_decode_matches_torch():
    codes, vals = _e4m3_table()
    for c, v in zip(codes, vals):
        assert oracle.e4m3_decode(int(c)) == v
    assert math.isnan(oracle.e4m3_decode(0x7F))


def test_e4m3_encode_bruteforce_and_torch():
    codes, vals = _e4m3_table()
    pos = sorted(set(float(v) for v in vals if v >= 0))
    xs = list(pos)
    xs += [(a + b) / 2 for a, b in zip(pos[:-1], pos[1:])]        # exact ties
    xs += [a * (1 + 1e-9) for a in pos[1:]] + [a * (1 - 1e-9) for a in pos[1:]]
    rng = np.random.default_rng(0)
    xs += list(np.exp2(rng.uniform(-12, 9.5, 2000)))
    xs += [449.0, 463.9, 464.0, 500.0, 1e6, float("inf")]
    for x in xs:
        for s in (1.0, -1.0):
            got = oracle.e4m3_encode(s * x)
            want_mag = _nearest_even(x, codes, vals, 448.0)
            want = want_mag | (0x80 if s < 0 else 0)
            assert got == want, (s * x, got, want)
            if x <= 448.0:  # torch's conversion is RNE without saturation
                t = torch.tensor([s * x], dtype=torch.float64).to(torch.float8_e4m3fn)
                assert int(t.view(torch.uint8)[0]) == got, (s * x,)


def test_e4m3_hand_cases():
    # OCP E4M3: 1.0 = 0.0111.000, 448 = 0.1111.110, 2^-9 = 0.0000.001, 2^-6 = 0.0001.000
    assert oracle.e4m3_encode(1.0) == 0x38
    assert oracle.e4m3_encode(448.0) == 0x7E
    assert oracle.e4m3_encode(2.0 ** -9) == 0x01
    assert oracle.e4m3_encode(2.0 ** -6) == 0x08
    assert oracle.e4m3_encode(1.0625) == 0x38       # tie -> even mantissa (1.0)
    assert oracle.e4m3_encode(1.1875) == 0x3A       # tie -> even mantissa (1.25)
    assert oracle.e4m3_encode(2.0 ** -10) == 0x00   # subnormal tie -> 0
    assert oracle.e4m3_encode(-(2.0 ** -10)) == 0x80
    assert oracle.e4m3_encode(1e9) == 0x7E          # saturation
    assert oracle.e4m3_encode(256.0) == 0x78


E2M1 = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def test_e2m1_bruteforce():
    codes = np.arange(16, dtype=np.uint8)
    vals = np.array([E2M1[c & 7] * (-1 if c & 8 else 1) for c in codes])
    for c in codes:
        assert oracle.e2m1_decode(int(c)) == vals[c]
    xs = list(E2M1) + [(a + b) / 2 for a, b in zip(E2M1[:-1], E2M1[1:])]
    xs += list(np.random.default_rng(1).uniform(0, 8, 3000)) + [6.5, 7.0, 100.0]
    for x in xs:
        for s in (1.0, -1.0):
            mag = _nearest_even(x, codes[:8], vals[:8], 6.0)
            want = mag | (0x8 if s < 0 else 0)
            assert oracle.e2m1_encode(s * x) == want, (s * x,)


def test_e2m1_hand_cases():
    # ties to even mantissa: 0.25->0, 0.75->1.0, 1.25->1.0, 1.75->2, 2.5->2, 3.5->4, 5->4
    for x, c in [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6),
                 (7.0, 7), (6.0, 7), (0.5, 1), (3.0, 5)]:
        assert oracle.e2m1_encode(x) == c, x
    assert oracle.e2m1_encode(-0.1) == 0x8


def test_int8_value_hand_cases():
    assert oracle.int8_quantize_value(2.5, 1.0) == 2      # ties to even
    assert oracle.int8_quantize_value(3.5, 1.0) == 4
    assert oracle.int8_quantize_value(-2.5, 1.0) == -2
    assert oracle.int8_quantize_value(-200.0, 1.0) == -127  # symmetric clamp
    s = np.float32(3.0) / np.float32(127.0)
    assert oracle.int8_quantize_value(3.0, float(s)) == 127
    assert oracle.int8_quantize_value(-3.0, float(s)) == -127


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(2)
    xs = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-5, 5, 3000),
                         [0.0, -0.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1e-40, 3e38]])
    want = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_round(xs)
    np.testing.assert_array_equal(got, want)


# ------------------------------------------------------------------ quantization
def _tiny(lens=None, seed=None, N=None):
    w = WORKLOADS["tiny"]
    if N is not None:
        w = Workload("t", w.B, w.H, N, N, seed=w.seed, structure=w.structure)
    q, k, v = make_qkv(w, seed=seed)
    return w, q, k, v


def _f32(x_bits):
    return (x_bits.astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("N,lens", [(256, None), (300, None), (300, [173])])
def test_quantize_int8(N, lens):
    w, q, k, v = _tiny(N=N)
    x = bf16_bits(k)
    codes, scale = oracle.quantize_int8(x, lens=lens)
    xf = _f32(x)  # [B,N,H,D]
    B, _, H, D = xf.shape
    nv = lens[0] if lens else N
    for b in range(B):
        for h in range(H):
            for blk in range(scale.shape[2]):
                n0, n1 = blk * 128, min(blk * 128 + 128, nv)
                blkx = xf[b, n0:n1, h, :]
                amax = np.float32(np.abs(blkx).max()) if n1 > n0 else np.float32(0)
                s = np.float32(amax / np.float32(127.0))
                assert scale[b, h, blk] == s
                c = codes[b, h, blk * 128:(blk + 1) * 128].astype(np.int32)
                assert np.all(c[max(0, n1 - n0):] == 0)          # padding / past lens
                if n1 > n0:
                    cc = c[:n1 - n0]
                    assert np.abs(cc).max() == 127                # the absmax maps to 127
                    err = np.abs(blkx.astype(np.float64) - cc * np.float64(s))
                    # half a step, plus the binary32 rounding of x/s (|x/s| <= 127, 2^-24 relative)
                    assert err.max() <= s * (0.5 + 127 * 2.0 ** -24)
                    ref = np.clip(np.rint(blkx / s), -127, 127)   # numpy binary32 division
                    np.testing.assert_array_equal(cc, ref)


@pytest.mark.parametrize("N,lens", [(256, None), (300, [211]), (129, None)])
def test_quantize_fp8_qk(N, lens):
    """FP8 E4M3 Q/K: absmax/448 per 128-token block (binary32 division) and the
    E4M3 encoding of the binary32 quotient, checked against numpy's division
    and torch's float32 -> float8_e4m3fn conversion."""
    w, q, k, v = _tiny(N=N)
    x = bf16_bits(k)
    codes, scale = oracle.quantize_fp8_qk(x, lens=lens)
    xf = _f32(x)
    B, _, H, D = xf.shape
    nv = lens[0] if lens else N
    assert codes.shape == (B, H, oracle.pad128(N), D) and scale.shape == (B, H, oracle.pad128(N) // 128)
    for b in range(B):
        for h in range(H):
            for blk in range(scale.shape[2]):
                n0, n1 = blk * 128, min(blk * 128 + 128, nv)
                c = codes[b, h, blk * 128:(blk + 1) * 128]
                assert np.all(c[max(0, n1 - n0):] == 0)            # padding / past lens
                if n1 <= n0:
                    assert scale[b, h, blk] == 0
                    continue
                blkx = xf[b, n0:n1, h, :]
                s = np.float32(np.float32(np.abs(blkx).max()) / np.float32(448.0))
                assert scale[b, h, blk] == s
                ratio = (blkx / s).astype(np.float32)
                want = torch.from_numpy(ratio).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
                np.testing.assert_array_equal(c[:n1 - n0], want)
                assert (c[:n1 - n0] & 0x7F).max() == 0x7E   # the absmax encodes to +-448


@pytest.mark.parametrize("N,lens", [(256, None), (300, [211])])
def test_quantize_v_fp8(N, lens):
    w, q, k, v = _tiny(N=N)
    x = bf16_bits(v)
    v8, sv = oracle.quantize_v_fp8(x, lens=lens)
    xf = _f32(x)
    B, _, H, D = xf.shape
    nv = lens[0] if lens else N
    Np = oracle.pad128(N)
    assert v8.shape == (B, H, D, Np)
    for b in range(B):
        for h in range(H):
            amax = np.abs(xf[b, :nv, h, :]).max(axis=0)               # per channel
            s = (amax / np.float32(448.0)).astype(np.float32)
            np.testing.assert_array_equal(sv[b, h], s)
            ratio = (xf[b, :nv, h, :] / s[None, :]).astype(np.float32)  # [n, d]
            want = torch.from_numpy(ratio).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
            np.testing.assert_array_equal(v8[b, h, :, :nv], want.T)   # token-contiguous
            assert np.all(v8[b, h, :, nv:] == 0)
            # every channel's absmax element encodes to +-448
            top = np.abs(v8[b, h, np.arange(D), np.abs(xf[b, :nv, h, :]).argmax(axis=0)])
            assert np.all((top & 0x7F) == 0x7E)


@pytest.mark.parametrize("lens", [None, [100]])
def test_quantize_mxfp4(lens):
    w, q, k, v = _tiny()
    x = bf16_bits(q)
    codes, e8 = oracle.quantize_mxfp4(x, lens=lens)
    xf = _f32(x).astype(np.float64)
    B, N, H, D = xf.shape
    nv = lens[0] if lens else N
    codes_tab = np.arange(8, dtype=np.uint8)
    vals_tab = np.array(E2M1)
    for b in range(B):
        for h in range(H):
            for n in range(0, oracle.pad128(N), 7 if lens is None else 1):
                if n >= nv:
                    assert np.all(codes[b, h, n] == 0) and np.all(e8[b, h, n] == 0)
                    continue
                for g in range(D // 32):
                    grp = xf[b, n, h, g * 32:(g + 1) * 32]
                    amax = np.abs(grp).max()
                    e = int(np.floor(np.log2(amax))) - 2
                    assert e8[b, h, n, g] == e + 127
                    X = 2.0 ** e
                    for i in range(32):
                        byte = codes[b, h, n, g * 16 + i // 2]
                        c = (byte >> (4 * (i % 2))) & 0xF
                        y = grp[i] / X
                        mag = _nearest_even(y, codes_tab, vals_tab, 6.0)
                        assert c == (mag | (0x8 if y < 0 or (y == 0 and math.copysign(1, y) < 0) else 0))


# ------------------------------------------------------------------ Hadamard-rotated MXFP4
def test_fwht128_is_the_sylvester_hadamard_product():
    """On small-integer rows every binary32 sum is exact, so the transform must
    equal x @ H with scipy's Sylvester Hadamard matrix, and applying it twice
    must give 128 x (H H = 128 I)."""
    import scipy.linalg
    rng = np.random.RandomState(3)
    x = rng.randint(-64, 65, size=(9, 128)).astype(np.float32)
    y = oracle.fwht128(x)
    np.testing.assert_array_equal(y, (x.astype(np.float64) @ scipy.linalg.hadamard(128)))
    np.testing.assert_array_equal(oracle.fwht128(y), 128.0 * x)


def test_fwht128_rounding_bound():
    """General BF16 rows: within the rounding of seven binary32 butterfly
    stages of the exact product (each stage adds at most 2^-24 of the row's
    absolute sum)."""
    import scipy.linalg
    w, q, k, v = _tiny()
    x = _f32(bf16_bits(k))[0, :64, 0, :]
    y = oracle.fwht128(x).astype(np.float64)
    exact = x.astype(np.float64) @ scipy.linalg.hadamard(128)
    bound = 7 * 2.0 ** -24 * np.abs(x).astype(np.float64).sum(axis=1, keepdims=True)
    assert np.all(np.abs(y - exact) <= bound)
    assert np.any(y != exact)                       # rounding does occur on these rows


@pytest.mark.parametrize("lens", [None, [100]])
def test_quantize_mxfp4_hadamard(lens):
    """Codes and E8M0 bytes equal the MXFP4 rule applied (independently, in
    numpy) to the rotated rows."""
    w, q, k, v = _tiny()
    x = bf16_bits(k)
    codes, e8 = oracle.quantize_mxfp4_hadamard(x, lens=lens)
    xf = _f32(x)
    B, N, H, D = xf.shape
    nv = lens[0] if lens else N
    codes_tab = np.arange(8, dtype=np.uint8)
    vals_tab = np.array(E2M1)
    for b in range(B):
        for h in range(H):
            rot = oracle.fwht128(xf[b, :, h, :]).astype(np.float64)  # [N, 128]
            for n in range(0, oracle.pad128(N), 11 if lens is None else 1):
                if n >= nv:
                    assert np.all(codes[b, h, n] == 0) and np.all(e8[b, h, n] == 0)
                    continue
                for g in range(D // 32):
                    grp = rot[n, g * 32:(g + 1) * 32]
                    e = int(np.floor(np.log2(np.abs(grp).max()))) - 2
                    assert e8[b, h, n, g] == e + 127
                    for i in range(32):
                        c = (codes[b, h, n, g * 16 + i // 2] >> (4 * (i % 2))) & 0xF
                        y = grp[i] / 2.0 ** e
                        mag = _nearest_even(y, codes_tab, vals_tab, 6.0)
                        assert c == (mag | (0x8 if y < 0 or (y == 0 and math.copysign(1, y) < 0) else 0))


def test_hadamard_rotation_scales_logits_by_128():
    """(QH)(KH)^T = 128 QK^T: exact on integer rows."""
    rng = np.random.RandomState(4)
    qi = rng.randint(-20, 21, size=(5, 128)).astype(np.float32)
    ki = rng.randint(-20, 21, size=(7, 128)).astype(np.float32)
    lhs = oracle.fwht128(qi).astype(np.float64) @ oracle.fwht128(ki).astype(np.float64).T
    np.testing.assert_array_equal(lhs, 128.0 * (qi.astype(np.float64) @ ki.astype(np.float64).T))


def test_hadamard_improves_mxfp4_accuracy():
    """With outlier K channels (4 of 128 scaled x8, the image workload's
    structure) the rotated MXFP4 attention (logit multiplier / 128) is closer
    to unquantized attention than plain MXFP4: the rotation spreads each
    outlier over all channels, so the 32-channel blocks lose less precision."""
    w = Workload("outliers", 1, 2, 256, 256, seed=7, structure="k_channels_x8")
    q, k, v = make_qkv(w)
    qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
    vz = oracle.quantize_v_fp8(vb)
    c = 1.0 / math.sqrt(128)
    oe, _ = oracle.attention_exact(qb, kb, vb)
    o1, _, _ = oracle.attention(1, *oracle.quantize_mxfp4(qb), *oracle.quantize_mxfp4(kb), *vz,
                                Nq=w.Nq, Nk=w.Nk)
    oh, _, _ = oracle.attention(1, *oracle.quantize_mxfp4_hadamard(qb),
                                *oracle.quantize_mxfp4_hadamard(kb), *vz, Nq=w.Nq, Nk=w.Nk,
                                softmax_scale=c / 128)
    cos = lambda a: float((a * oe).sum() / math.sqrt((a * a).sum() * (oe * oe).sum()))  # noqa: E731
    assert cos(oh) > cos(o1) + 0.02


def test_mxfp4_nibble_order_and_scale_closed_form():
    x = np.zeros((1, 1, 1, 128), np.float32)
    x[0, 0, 0, 0] = 6.0 * 2.0 ** 5     # element 0 -> +6 at scale 2^5
    x[0, 0, 0, 1] = -1.0 * 2.0 ** 5    # element 1 -> -1
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    codes, e8 = oracle.quantize_mxfp4(bits)
    assert e8[0, 0, 0, 0] == 127 + 5
    assert codes[0, 0, 0, 0] == (0x7 | (0xA << 4))   # low nibble = element 0
    assert e8[0, 0, 0, 1] == 0 and np.all(codes[0, 0, 0, 16:] == 0)  # all-zero group


# ------------------------------------------------------------------ attention
def _dequant_int8(codes, scale):
    B, H, Np, D = codes.shape
    return codes.astype(np.float64) * np.repeat(scale.astype(np.float64), 128, axis=2)[..., None]


def _dequant_fp8qk(codes, scale):
    tab = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    return tab[codes] * np.repeat(scale.astype(np.float64), 128, axis=2)[..., None]


def _dequant_mxfp4(codes, e8):
    lo = codes & 0xF
    hi = codes >> 4
    c = np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)
    mag = np.array(E2M1)[c & 7] * np.where(c & 8, -1.0, 1.0)
    return mag * np.repeat(np.exp2(e8.astype(np.float64) - 127), 32, axis=-1)


def _dequant_v(v8, sv):
    tab = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).double().numpy()
    return tab[v8] * sv.astype(np.float64)[..., None]     # [B,H,D,Np]


def _quantize_all(q, k, v, fmt, k_lens=None):
    qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
    if fmt == 0:
        qq, qs = oracle.quantize_int8(qb)
        kq, ks = oracle.quantize_int8(kb, lens=k_lens)
        qd, kd = _dequant_int8(qq, qs), _dequant_int8(kq, ks)
    elif fmt == 2:
        qq, qs = oracle.quantize_fp8_qk(qb)
        kq, ks = oracle.quantize_fp8_qk(kb, lens=k_lens)
        qd, kd = _dequant_fp8qk(qq, qs), _dequant_fp8qk(kq, ks)
    else:
        qq, qs = oracle.quantize_mxfp4(qb)
        kq, ks = oracle.quantize_mxfp4(kb, lens=k_lens)
        qd, kd = _dequant_mxfp4(qq, qs), _dequant_mxfp4(kq, ks)
    v8, sv = oracle.quantize_v_fp8(vb, lens=k_lens)
    return (qq, qs, kq, ks, v8, sv), (qd, kd, _dequant_v(v8, sv))


@pytest.mark.parametrize("fmt", [0, 1, 2])
def test_attention_lse_weights_and_output(fmt):
    w, q, k, v = _tiny()
    Nq, Nk, D = w.Nq, w.Nk, w.D
    c = 1.0 / math.sqrt(D)
    qz, (qd, kd, vd) = _quantize_all(q, k, v, fmt)
    o, lse, wts = oracle.attention(fmt, *qz, Nq=Nq, Nk=Nk, want_weights=True)
    z = c * np.einsum("bhid,bhjd->bhij", qd[:, :, :Nq], kd[:, :, :Nk])    # natural-log logits
    # LSE is the logsumexp of the dequantized logits (no FP8 step involved)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(z, axis=-1), rtol=0, atol=1e-9)
    # weights: FP8 rounding of the softmax, within half an E4M3 step (2^-4 relative)
    sm = scipy.special.softmax(z, axis=-1)
    assert np.all(np.abs(wts - sm) <= sm * 2.0 ** -4 + 2.0 ** -18)
    np.testing.assert_allclose(wts.sum(-1), 1.0, atol=2.0 ** -4)
    # each weight is exactly E4M3(p*256)/256/l with the integer maximum (brute force)
    codes, vals = _e4m3_table()
    t = z * L2E
    M = np.ceil(t.max(-1, keepdims=True))
    p = np.exp2(t - M)
    l = p.sum(-1, keepdims=True)
    for (b, h, i) in [(0, 0, 0), (0, 1, 77), (0, 0, 255)]:
        for j in range(0, Nk, 5):
            mag = _nearest_even(p[b, h, i, j] * 256.0, codes, vals, 448.0)
            want = torch.tensor([mag], dtype=torch.uint8).view(torch.float8_e4m3fn).double().item()
            assert wts[b, h, i, j] == pytest.approx(want / 256.0 / l[b, h, i, 0], rel=1e-12)
    # output is the weighted sum of the dequantized V rows
    ref = np.einsum("bhij,bhdj->bhid", wts, vd[..., :Nk])
    np.testing.assert_allclose(o, ref, rtol=1e-10, atol=1e-12)


def test_attention_special_cases():
    w, q, k, v = _tiny()
    Nq, Nk = w.Nq, w.Nk
    # constant V: every output row is the dequantized constant (weights sum ~1 is not enough:
    # O = sum w * v exactly, so O/v = sum w; check against sum of weights)
    vc = torch.full_like(v, 0.75)
    qz, (qd, kd, vd) = _quantize_all(q, k, vc, 0)
    o, lse, wts = oracle.attention(0, *qz, Nq=Nq, Nk=Nk, want_weights=True)
    np.testing.assert_allclose(o, wts.sum(-1, keepdims=True) * vd[:, :, :, :1].transpose(0, 1, 3, 2),
                               rtol=1e-12)
    assert np.all(np.abs(o - 0.75) <= 0.75 * 2.0 ** -4)
    # softmax_scale -> 0: uniform weights, O = mean of dequantized V, LSE = ln Nk
    qz, (qd, kd, vd) = _quantize_all(q, k, v, 0)
    o, lse, wts = oracle.attention(0, *qz, Nq=Nq, Nk=Nk, softmax_scale=1e-30, want_weights=True)
    np.testing.assert_allclose(wts, 1.0 / Nk, rtol=1e-12)
    np.testing.assert_allclose(o, np.broadcast_to(vd[..., :Nk].mean(-1)[:, :, None, :], o.shape),
                               rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(lse, math.log(Nk), rtol=1e-9)
    # a single key: O is that key's value row up to the P8 rounding of p
    o1, lse1, _ = oracle.attention(0, *qz, Nq=Nq, Nk=Nk, k_lens=[1])
    assert np.all(np.abs(o1 - vd[:, :, None, :, 0]) <= np.abs(vd[:, :, None, :, 0]) * 2.0 ** -4 + 1e-12)
    # zero valid keys: empty softmax
    o0, lse0, _ = oracle.attention(0, *qz, Nq=Nq, Nk=Nk, k_lens=[0])
    assert np.all(o0 == 0) and np.all(np.isneginf(lse0))


def test_attention_block_permutation_invariance():
    """Permuting whole 128-key blocks of K/V (their scales move with them)
    leaves every output unchanged."""
    w, q, k, v = _tiny()
    qz, _ = _quantize_all(q, k, v, 0)
    qq, qs, kq, ks, v8, sv = qz
    o, lse, _ = oracle.attention(0, *qz, Nq=w.Nq, Nk=w.Nk)
    perm = [1, 0]
    kq2 = np.concatenate([kq[:, :, p * 128:(p + 1) * 128] for p in perm], axis=2)
    ks2 = ks[:, :, perm]
    v82 = np.concatenate([v8[..., p * 128:(p + 1) * 128] for p in perm], axis=3)
    o2, lse2, _ = oracle.attention(0, qq, qs, kq2, ks2, v82, sv, Nq=w.Nq, Nk=w.Nk)
    np.testing.assert_allclose(o2, o, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(lse2, lse, rtol=1e-13)


def test_attention_ragged_equals_truncated():
    w, q, k, v = _tiny()
    L = 173
    qz, _ = _quantize_all(q, k, v, 0, k_lens=[L])
    o, lse, _ = oracle.attention(0, *qz, Nq=w.Nq, Nk=w.Nk, k_lens=[L])
    qz2, _ = _quantize_all(q, k[:, :L], v[:, :L], 0)
    o2, lse2, _ = oracle.attention(0, *qz2, Nq=w.Nq, Nk=L)
    np.testing.assert_array_equal(o, o2)
    np.testing.assert_array_equal(lse, lse2)


def test_attention_rows_subset():
    w, q, k, v = _tiny()
    qz, _ = _quantize_all(q, k, v, 0)
    o, lse, _ = oracle.attention(0, *qz, Nq=w.Nq, Nk=w.Nk)
    rows = [0, 5, 130, 255]
    o2, lse2, _ = oracle.attention(0, *qz, Nq=w.Nq, Nk=w.Nk, rows=rows)
    np.testing.assert_array_equal(o2, o[:, :, rows])
    np.testing.assert_array_equal(lse2, lse[:, :, rows])


def test_exact_attention_matches_torch_sdpa():
    w, q, k, v = _tiny()
    o, lse = oracle.attention_exact(bf16_bits(q), bf16_bits(k), bf16_bits(v))
    qt, kt, vt = (t.double().permute(0, 2, 1, 3) for t in (q, k, v))
    ref = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt).numpy()
    np.testing.assert_allclose(o, ref, rtol=1e-10, atol=1e-12)
    z = (qt @ kt.transpose(-1, -2)).numpy() / math.sqrt(w.D)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(z, axis=-1), rtol=1e-12)
    # strided views (packed QKV) give the same answer
    qkv = torch.stack([q, k, v], dim=2)  # [B,N,3,H,D]
    o2, _ = oracle.attention_exact(bf16_bits(qkv[:, :, 0]), bf16_bits(qkv[:, :, 1]),
                                   bf16_bits(qkv[:, :, 2]))
    np.testing.assert_array_equal(o2, o)


@pytest.mark.parametrize("fmt,min_cos", [(0, 0.999), (1, 0.95), (2, 0.995)])
def test_quantized_close_to_exact(fmt, min_cos):
    w, q, k, v = _tiny()
    qz, _ = _quantize_all(q, k, v, fmt)
    o, _, _ = oracle.attention(fmt, *qz, Nq=w.Nq, Nk=w.Nk)
    oe, _ = oracle.attention_exact(bf16_bits(q), bf16_bits(k), bf16_bits(v))
    cos = (o * oe).sum() / math.sqrt((o * o).sum() * (oe * oe).sum())
    assert cos >= min_cos


def test_p8_online_equals_final_encoding():
    """The running-integer-maximum encoding equals the final-maximum encoding
    wherever the probability is a normal E4M3 number after the 2^8 scale."""
    rng = np.random.default_rng(3)
    for trial in range(50):
        n = int(rng.integers(1, 1000))
        t = rng.standard_normal(n) * rng.uniform(0.1, 8) + np.linspace(0, rng.uniform(-5, 5), n)
        a = oracle.p8_online(t, 128)
        b = oracle.p8_final(t)
        M = np.ceil(t.max())
        normal = np.exp2(t - M) * 256.0 >= 2.0 ** -6
        np.testing.assert_array_equal(a[normal], b[normal])
        assert np.all(np.abs(a - b) <= 2.0 ** -17)


# ------------------------------------------------------------------ K smoothing
def _bits(x):
    """float array [B,N,H,D] -> BF16 bit patterns (the values must be BF16-exact)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    assert np.array_equal(t.float().numpy(), np.asarray(x, dtype=np.float32)), "not BF16-exact"
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("N", [256, 300])
def test_k_mean_exact_on_dyadic_data(N):
    """On multiples of 1/8 the fixed-point sum loses nothing, so the mean is
    the correctly rounded quotient of the exact sum by the token count."""
    rng = np.random.RandomState(11)
    x = rng.randint(-64, 65, size=(1, N, 2, 128)).astype(np.float32) / 8 + rng.randint(
        -4, 5, size=(1, 1, 2, 128))
    mu = oracle.k_mean(_bits(x))
    want = (x.astype(np.float64).sum(1) / N).astype(np.float32)   # exact sum, one division
    np.testing.assert_array_equal(mu, want)


def test_k_mean_truncation_rule():
    """Contributions are truncated toward zero on the grid 2^(E-40), E the
    exponent of the channel maximum (here E = 10, grid 2^-30)."""
    x = np.zeros((1, 3, 1, 128), np.float32)
    x[0, 0, 0, :] = 2.0 ** 10
    x[0, 1, 0, :] = -(2.0 ** 10)
    x[0, 2, 0, 0] = 3 * 2.0 ** -32      # 0.75 grid steps: truncated to 0
    x[0, 2, 0, 1] = -3 * 2.0 ** -32     # -0.75: toward zero gives 0 (floor would give -1)
    x[0, 2, 0, 2] = 2.0 ** -29          # 2 grid steps: kept
    x[0, 2, 0, 3] = -5 * 2.0 ** -31     # -2.5 steps: -2
    mu = oracle.k_mean(_bits(x))[0, 0]
    assert mu[0] == 0.0 and mu[1] == 0.0 and not np.signbit(mu[1])
    assert mu[2] == np.float32(2.0 * 2.0 ** -30 / 3)
    assert mu[3] == np.float32(-2.0 * 2.0 ** -30 / 3)
    assert np.all(mu[4:] == 0.0)


def test_k_mean_ragged_empty_and_zero():
    rng = np.random.RandomState(12)
    x = rng.randint(-64, 65, size=(3, 200, 1, 128)).astype(np.float32) / 8
    x[:, 150:] = 1000.0                      # past the valid length of batch 0
    x[2, :, :, :5] = 0.0                     # all-zero channels
    mu = oracle.k_mean(_bits(x), lens=[150, 0, 200])
    np.testing.assert_array_equal(mu[0], (x[0, :150].astype(np.float64).sum(0) / 150).astype(np.float32))
    assert np.all(mu[1] == 0.0)              # no valid token
    assert np.all(mu[2, :, :5] == 0.0)


def test_k_mean_error_bound_on_gaussian_data():
    """Truncation moves each term by less than one grid step 2^(E-40) <=
    amax 2^-40, and the two final roundings add at most one binary32 ulp."""
    w, q, k, v = _tiny(N=300)
    kb = bf16_bits(k)
    mu = oracle.k_mean(kb).astype(np.float64)
    kf = _f32(kb).astype(np.float64)
    mean = kf.mean(1)
    amax = np.abs(kf).max(1)
    assert np.all(np.abs(mu - mean) <= amax * 2.0 ** -40 + np.abs(mean) * 2.0 ** -23)


def test_smoothing_is_translation_invariant():
    """Adding a constant to every token of a channel changes the mean by that
    constant and leaves the smoothed codes and scales unchanged (all values
    dyadic, so every step is exact)."""
    rng = np.random.RandomState(13)
    x = rng.randint(-64, 65, size=(1, 256, 2, 128)).astype(np.float32) / 8
    c = rng.randint(-4, 5, size=(1, 1, 2, 128)).astype(np.float32)
    q0, s0, m0 = oracle.quantize_int8_smooth(_bits(x))
    q1, s1, m1 = oracle.quantize_int8_smooth(_bits(x + c))
    np.testing.assert_array_equal(m1, m0 + c[0].transpose(1, 0, 2)[:, 0][None])
    np.testing.assert_array_equal(q1, q0)
    np.testing.assert_array_equal(s1.view(np.uint32), s0.view(np.uint32))
    # without smoothing the offset changes the codes
    assert not np.array_equal(oracle.quantize_int8(_bits(x + c))[0], q0)


def test_smoothing_zero_mean_reduces_to_plain_int8():
    """Channels whose tokens come in +-pairs have mean exactly 0: the smoothed
    quantizer then equals the plain INT8 quantizer."""
    w, q, k, v = _tiny(N=128)
    kf = _f32(bf16_bits(k))
    x = np.concatenate([kf, -kf], axis=1)
    q0, s0 = oracle.quantize_int8(_bits(x))
    q1, s1, m1 = oracle.quantize_int8_smooth(_bits(x))
    assert np.all(m1 == 0.0)
    np.testing.assert_array_equal(q1, q0)
    np.testing.assert_array_equal(s1.view(np.uint32), s0.view(np.uint32))


def test_smoothed_attention_lse_and_accuracy():
    """K with large per-channel offsets (mean ~ N(0, 3^2)): attention over the
    smoothed K, with the per-row term c q^.mean added back to the LSE, matches
    unquantized attention; the term is O(1), so dropping it would fail; and
    smoothing lowers the output error of plain INT8 quantization."""
    w = Workload("offsets", 1, 2, 256, 256, seed=14)
    q, k, v = make_qkv(w)
    k = (k.float() + 3.0 * torch.randn(1, 1, 2, 128, generator=torch.Generator().manual_seed(15))
         ).to(torch.bfloat16)
    qb, kb, vb = bf16_bits(q), bf16_bits(k), bf16_bits(v)
    oe, le = oracle.attention_exact(qb, kb, vb)
    qz = oracle.quantize_int8(qb)
    vz = oracle.quantize_v_fp8(vb)
    kq, ks, mu = oracle.quantize_int8_smooth(kb)
    os_, ls, _ = oracle.attention(0, *qz, kq, ks, *vz, Nq=256, Nk=256, k_mean=mu)
    op, lp, _ = oracle.attention(0, *qz, *oracle.quantize_int8(kb), *vz, Nq=256, Nk=256)
    term = oracle.k_mean_lse_term(*qz, mu, Nq=256)
    assert np.abs(term).max() > 1.0
    # the LSE error is that of INT8 Q (the same in both quantized runs)
    assert np.abs(ls - lp).max() < 0.05
    assert np.abs(ls - le).max() < 0.15
    err = lambda o: float(np.abs(o - oe).max())  # noqa: E731
    assert err(os_) < err(op)


# ------------------------------------------------------------------ MXFP4 V and P
def _e2m1_code(y):
    """Brute-force E2M1 code (sign bit 8) of y: nearest value, ties to the even code."""
    mag = _nearest_even(y, np.arange(8, dtype=np.uint8), np.array(E2M1), 6.0)
    return mag | (0x8 if y < 0 or (y == 0 and math.copysign(1, y) < 0) else 0)


def _dequant_v_mxfp4(codes, e8):
    """[B,H,D,Np/2] codes + [B,H,Np/128,D,4] bytes -> float64 V^T [B,H,D,Np]."""
    lo, hi = codes & 0xF, codes >> 4
    c = np.stack([lo, hi], axis=-1).reshape(*codes.shape[:-1], codes.shape[-1] * 2)
    mag = np.array(E2M1)[c & 7] * np.where(c & 8, -1.0, 1.0)
    B, H, nt, D, _ = e8.shape
    sc = np.exp2(e8.astype(np.float64) - 127).transpose(0, 1, 3, 2, 4).reshape(B, H, D, nt * 4)
    return mag * np.repeat(sc, 32, axis=-1)


@pytest.mark.parametrize("lens", [None, [100]])
def test_quantize_v_mxfp4(lens):
    """Every 32-token block of every channel: E8M0 = floor(log2 amax) - 2
    over the valid tokens (numpy), E2M1 codes by brute-force nearest-even
    search, token 2i in the low nibble, scales tile-major."""
    w, q, k, v = _tiny(N=300)
    x = bf16_bits(v)
    codes, e8 = oracle.quantize_v_mxfp4(x, lens=lens)
    assert codes.shape == (1, 2, 128, 192) and e8.shape == (1, 2, 3, 128, 4)
    vf = _f32(x).astype(np.float64)
    nv = lens[0] if lens else 300
    for h in range(2):
        for d in range(0, 128, 7):
            for blk in range(12):
                n0 = blk * 32
                vals = vf[0, n0:min(n0 + 32, nv), h, d] if n0 < nv else np.zeros(0)
                amax = np.abs(vals).max() if vals.size else 0.0
                byte = 0 if amax == 0 else int(np.floor(np.log2(amax))) - 2 + 127
                assert e8[0, h, blk // 4, d, blk % 4] == byte
                for i in range(32):
                    n = n0 + i
                    c = (codes[0, h, d, n // 2] >> (4 * (n % 2))) & 0xF
                    want = _e2m1_code(vf[0, n, h, d] / 2.0 ** (byte - 127)) if n < nv else 0
                    assert c == want, (h, d, n)


def test_attention_mxfp4_pv_weights_and_output():
    """MXFP4 Q/K, V and P (fmt 4): LSE is the logsumexp of the dequantized
    logits; each weight is the brute-force MXFP4 encoding of p = 2^(t - M)
    (per 32 keys: exponent floor(log2 max p) - 2, E2M1 nearest-even) over l;
    O is the weighted sum of the dequantized MXFP4 V."""
    w, q, k, v = _tiny(N=300)
    Nq = Nk = 300
    qq, qs = oracle.quantize_mxfp4(bf16_bits(q))
    kq, ks = oracle.quantize_mxfp4(bf16_bits(k))
    vc, ve = oracle.quantize_v_mxfp4(bf16_bits(v))
    o, lse, wts = oracle.attention(4, qq, qs, kq, ks, vc, ve, Nq=Nq, Nk=Nk, want_weights=True)
    qd, kd = _dequant_mxfp4(qq, qs), _dequant_mxfp4(kq, ks)
    z = (1 / math.sqrt(128)) * np.einsum("bhid,bhjd->bhij", qd[:, :, :Nq], kd[:, :, :Nk])
    np.testing.assert_allclose(lse, scipy.special.logsumexp(z, axis=-1), rtol=0, atol=1e-9)
    t = z * L2E
    M = np.ceil(t.max(-1, keepdims=True))
    p = np.exp2(t - M)
    l = p.sum(-1)
    for (b, h, i) in [(0, 0, 0), (0, 1, 77), (0, 0, 299)]:
        for j0 in range(0, Nk, 32):
            blk = p[b, h, i, j0:j0 + 32]
            e = int(np.floor(np.log2(blk.max()))) - 2
            for jj, pj in enumerate(blk):
                c = _e2m1_code(pj / 2.0 ** e)
                want = E2M1[c & 7] * 2.0 ** e / l[b, h, i]
                assert wts[b, h, i, j0 + jj] == pytest.approx(want, rel=1e-12, abs=1e-300)
    vd = _dequant_v_mxfp4(vc, ve)
    np.testing.assert_allclose(o, np.einsum("bhij,bhdj->bhid", wts, vd[..., :Nk]),
                               rtol=1e-10, atol=1e-12)
    # the weights still sum to one within the E2M1 half-step (1/4 relative)
    assert np.all(np.abs(wts.sum(-1) - 1.0) <= 0.25)


def test_mxfp4_pv_close_to_exact():
    w, q, k, v = _tiny()
    qz = oracle.quantize_mxfp4(bf16_bits(q))
    kz = oracle.quantize_mxfp4(bf16_bits(k))
    vz = oracle.quantize_v_mxfp4(bf16_bits(v))
    o, _, _ = oracle.attention(4, *qz, *kz, *vz, Nq=w.Nq, Nk=w.Nk)
    oe, _ = oracle.attention_exact(bf16_bits(q), bf16_bits(k), bf16_bits(v))
    cos = (o * oe).sum() / math.sqrt((o * o).sum() * (oe * oe).sum())
    assert cos >= 0.95


# ------------------------------------------------------------------ Q smoothing and dS
def test_qsmooth_block_means_exact_and_ragged():
    """Per 128-token block: on multiples of 1/8 the block mean is the exact
    sum divided by the block's valid-token count (the last block partial,
    tokens past the length left out); padding rows are zero codes."""
    rng = np.random.RandomState(21)
    x = rng.randint(-64, 65, size=(1, 300, 2, 128)).astype(np.float32) / 8
    x += rng.randint(-4, 5, size=(1, 1, 2, 128))
    x[:, 250:] = 1000.0                      # past the valid length
    q8, s, m = oracle.quantize_int8_qsmooth(_bits(x), lens=[250])
    for blk, (n0, n1) in enumerate([(0, 128), (128, 250), (256, 256)]):
        want = (x[0, n0:n1].astype(np.float64).sum(0) / max(n1 - n0, 1)).astype(np.float32)
        np.testing.assert_array_equal(m[0, :, blk], want if n1 > n0 else np.zeros((2, 128), np.float32))
    assert np.all(q8[0, :, 250:] == 0)


def test_qsmooth_block_translation_invariance():
    """Adding a constant per (block, channel) moves that block's mean by it and
    leaves every code and scale unchanged (dyadic values: all steps exact)."""
    rng = np.random.RandomState(22)
    x = rng.randint(-64, 65, size=(1, 256, 2, 128)).astype(np.float32) / 8
    c = np.zeros_like(x)
    c[:, :128] = rng.randint(-4, 5, size=(1, 1, 2, 128))
    c[:, 128:] = rng.randint(-4, 5, size=(1, 1, 2, 128))
    q0, s0, m0 = oracle.quantize_int8_qsmooth(_bits(x))
    q1, s1, m1 = oracle.quantize_int8_qsmooth(_bits(x + c))
    np.testing.assert_array_equal(m1[0, :, 0], m0[0, :, 0] + c[0, 0].astype(np.float32))
    np.testing.assert_array_equal(m1[0, :, 1], m0[0, :, 1] + c[0, 128].astype(np.float32))
    np.testing.assert_array_equal(q1, q0)
    np.testing.assert_array_equal(s1.view(np.uint32), s0.view(np.uint32))


def test_qsmooth_zero_mean_reduces_to_plain_int8():
    w, q, k, v = _tiny(N=64)
    qf = _f32(bf16_bits(q))
    x = np.concatenate([qf, -qf], axis=1)    # one block of +-pairs: mean 0
    q0, s0 = oracle.quantize_int8(_bits(x))
    q1, s1, m1 = oracle.quantize_int8_qsmooth(_bits(x))
    assert np.all(m1 == 0.0)
    np.testing.assert_array_equal(q1, q0)
    np.testing.assert_array_equal(s1.view(np.uint32), s0.view(np.uint32))


@pytest.mark.parametrize("smooth_k", [False, True])
def test_qsmooth_logits_identity(smooth_k):
    """With the dS correction the LSE is the logsumexp of softmax_scale *
    (q^_s + q_grid) . (k^ + mu): the reconstructed Q (block means on their
    16-bit grid) against the dequantized (and, with K smoothing, re-centred)
    K, in numpy from the quantized data."""
    w = Workload("qs", 1, 2, 300, 200, seed=23)
    q, k, v = make_qkv(w)
    g = torch.Generator().manual_seed(24)
    q = (q.float() + 2.0 * torch.randn(1, 1, 2, 128, generator=g)).to(torch.bfloat16)
    k = (k.float() + 2.0 * torch.randn(1, 1, 2, 128, generator=g)).to(torch.bfloat16)
    qq, qs, qm = oracle.quantize_int8_qsmooth(bf16_bits(q))
    if smooth_k:
        kq, ks, mu = oracle.quantize_int8_smooth(bf16_bits(k))
    else:
        (kq, ks), mu = oracle.quantize_int8(bf16_bits(k)), None
    vz = oracle.quantize_v_fp8(bf16_bits(v))
    ds = oracle.delta_s(kq, ks, qm, Nq=300, Nk=200, k_mean=mu)
    o, lse, _ = oracle.attention(0, qq, qs, kq, ks, *vz, Nq=300, Nk=200, delta_s=ds, k_mean=mu)
    qg = oracle.q_grid(qm)
    # the grid keeps the means within half a step of 2^(E-13): 2^-14 of the largest
    assert np.all(np.abs(qg - qm) <= np.abs(qm).max(-1, keepdims=True) * 2.0 ** -14)
    qhat = _dequant_int8(qq, qs)[:, :, :300] + np.repeat(qg, 128, axis=2)[:, :, :300]
    khat = _dequant_int8(kq, ks)[:, :, :200] + (0 if mu is None else mu.astype(np.float64)[:, :, None, :])
    z = (1 / math.sqrt(128)) * np.einsum("bhid,bhjd->bhij", qhat, khat)
    np.testing.assert_allclose(lse, scipy.special.logsumexp(z, axis=-1), rtol=0, atol=1e-9)
    # and the output is close to unquantized attention, closer than without Q smoothing
    oe, _ = oracle.attention_exact(bf16_bits(q), bf16_bits(k), bf16_bits(v))
    o0, _, _ = oracle.attention(0, *oracle.quantize_int8(bf16_bits(q)), kq, ks, *vz, Nq=300,
                                Nk=200, k_mean=mu)
    err = lambda a: float(np.abs(a - oe).max())  # noqa: E731
    assert err(o) < err(o0)


# ------------------------------------------------------------------ binary32 logits (INT8)
def _int8_case(seed, pow2_scales):
    """Quantized INT8 operands built directly: random codes, scales either
    powers of two (so binary32 logits are exact) or general binary32 values."""
    rng = np.random.default_rng(seed)
    B, H, N, D = 1, 2, 256, 128
    q = rng.integers(-127, 128, (B, H, N, D), dtype=np.int8)
    k = rng.integers(-127, 128, (B, H, N, D), dtype=np.int8)
    if pow2_scales:
        qs = (2.0 ** rng.integers(-12, -6, (B, H, 2))).astype(np.float32)
        ks = (2.0 ** rng.integers(-12, -6, (B, H, 2))).astype(np.float32)
    else:
        qs = rng.uniform(0.004, 0.03, (B, H, 2)).astype(np.float32)
        ks = rng.uniform(0.004, 0.03, (B, H, 2)).astype(np.float32)
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    v8 = rng.choice(codes, (B, H, D, N)).astype(np.uint8)
    sv = rng.uniform(0.001, 0.01, (B, H, D)).astype(np.float32)
    return q, qs, k, ks, v8, sv


def test_logits32_equals_binary64_where_binary32_is_exact():
    """With power-of-two scales and c log2(e) = 1/8 the binary32 logits are the
    exact ones, so both modes agree (to the 1e-16 of the binary64 constant):
    the binary32 path forms the same logit, with and without dS."""
    q, qs, k, ks, v8, sv = _int8_case(1, True)
    c = 0.125 / L2E
    o64, l64, w64 = oracle.attention(0, q, qs, k, ks, v8, sv, Nq=256, Nk=256, softmax_scale=c,
                                     want_weights=True)
    o32, l32, w32 = oracle.attention(0, q, qs, k, ks, v8, sv, Nq=256, Nk=256, softmax_scale=c,
                                     want_weights=True, logits32=True)
    np.testing.assert_allclose(o32, o64, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(l32, l64, rtol=1e-12)
    np.testing.assert_array_equal(w32 > 0, w64 > 0)
    np.testing.assert_allclose(w32, w64, rtol=1e-12)
    # with dS: codes within +-7 and scales 2^-4 keep S s_q s_k on the 2^-8 grid
    # below 2^5, and dS (multiples of 2^-8 below 8) keeps the sum exact in binary32
    rng = np.random.default_rng(2)
    q7 = rng.integers(-7, 8, q.shape, dtype=np.int8)
    k7 = rng.integers(-7, 8, k.shape, dtype=np.int8)
    s16 = np.full(qs.shape, 2.0 ** -4, np.float32)
    ds = (rng.integers(-2048, 2048, (1, 2, 2, 256)) / 256.0).astype(np.float64)
    o64, l64, _ = oracle.attention(0, q7, s16, k7, s16, v8, sv, Nq=256, Nk=256, softmax_scale=c,
                                   delta_s=ds)
    o32, l32, _ = oracle.attention(0, q7, s16, k7, s16, v8, sv, Nq=256, Nk=256, softmax_scale=c,
                                   delta_s=ds, logits32=True)
    np.testing.assert_allclose(o32, o64, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(l32, l64, rtol=1e-12)


def test_logits32_within_binary32_rounding_of_binary64():
    """General scales: the binary32 logits differ from the binary64 ones by
    rounding only, so the LSE moves by ~1e-7 and O by the rare E4M3 code that
    crosses a boundary (the rows stay cosine-close)."""
    q, qs, k, ks, v8, sv = _int8_case(3, False)
    for ds in (None, np.random.default_rng(4).normal(0, 2, (1, 2, 2, 256))):
        o64, l64, _ = oracle.attention(0, q, qs, k, ks, v8, sv, Nq=256, Nk=256, delta_s=ds)
        o32, l32, _ = oracle.attention(0, q, qs, k, ks, v8, sv, Nq=256, Nk=256, delta_s=ds,
                                       logits32=True)
        assert np.abs(l32 - l64).max() < 1e-5
        cos = float((o32 * o64).sum() / np.sqrt((o32 * o32).sum() * (o64 * o64).sum()))
        assert cos > 0.99999
        assert not np.array_equal(l32, l64)  # the modes do differ
