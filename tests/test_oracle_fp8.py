"""Pins for the 8-bit (E4M3) oracle, and planted mistakes they must catch.

Facts used:
  * The E4M3 format (OCP 8-bit floating point specification, OFP8): bias 7,
    largest finite 448 = 0x7E, smallest normal 2^-6 = 0x08, smallest
    subnormal 2^-9 = 0x01, 1.0 = 0x38, 0x7F and 0xFF are NaN, 0x80 is -0;
    between two neighbours the spacing is 2^(E-3).
  * A library cast: torch's float8_e4m3fn dtype (all 256 codes decoded,
    round-to-nearest-even encode of values within +-464).
  * Mathematics of the per-slice scaling: the slice maximum maps to +-448;
    multiplying a slice by 2^k leaves its codes unchanged and multiplies its
    descale by 2^k; the dequantised value is within half a step of x.
  * Attention of the dequantised inputs: one key gives O = V^ and L = s;
    scaling descale_q by t equals scaling the softmax scale by t; O is
    linear in descale_v and L does not depend on it.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import oracle.fp8 as of


def _torch_decode_all():
    return torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _finite_codes():
    c = np.arange(256, dtype=np.uint8)
    return c[(c & 0x7F) != 0x7F]


# --------------------------------------------------------------------- pins

def pin_decode_fixed_points(m):
    v = m.e4m3_decode(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x3C, 0x7E, 0x80, 0xB8, 0xFE],
                               dtype=np.uint8))
    want = [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 1.5, 448.0, -0.0, -1.0, -448.0]
    assert np.array_equal(v, np.array(want)), v
    assert np.signbit(v[7])
    nan = m.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))
    assert np.isnan(nan).all()


def pin_decode_library(m):
    ours = m.e4m3_decode(np.arange(256, dtype=np.uint8))
    lib = _torch_decode_all()
    same = (ours == lib) | (np.isnan(ours) & np.isnan(lib))
    assert same.all(), np.nonzero(~same)


def pin_encode_round_trip(m):
    c = _finite_codes()
    back = m.e4m3_encode(m.e4m3_decode(c))
    assert np.array_equal(back, c), np.nonzero(back != c)


def pin_encode_midpoints(m):
    # positive finite codes in value order; midpoints between neighbours go to
    # the even code (mantissa LSB 0); just above/below go to the nearer one
    c = np.arange(0x00, 0x7F, dtype=np.uint8)
    v = m.e4m3_decode(c)
    mid = (v[:-1] + v[1:]) / 2
    even = np.where(c[:-1] % 2 == 0, c[:-1], c[1:])
    assert np.array_equal(m.e4m3_encode(mid), even)
    eps = (v[1:] - v[:-1]) * 1e-3
    assert np.array_equal(m.e4m3_encode(mid - eps), c[:-1])
    assert np.array_equal(m.e4m3_encode(mid + eps), c[1:])
    assert np.array_equal(m.e4m3_encode(-mid), even | 0x80)


def pin_encode_saturation_nan(m):
    big = np.array([448.0, 463.9, 464.0, 470.0, 1e6, np.inf, -500.0, -np.inf])
    assert np.array_equal(m.e4m3_encode(big), np.array([0x7E] * 6 + [0xFE] * 2, dtype=np.uint8))
    assert m.e4m3_encode(np.array([np.nan]))[0] & 0x7F == 0x7F
    assert m.e4m3_encode(np.array([2.0 ** -11]))[0] == 0x00      # below half the smallest step
    assert m.e4m3_encode(np.array([3 * 2.0 ** -11]))[0] == 0x01  # 0.75 step -> 1 step


def pin_encode_library(m):
    g = np.random.default_rng(3)
    y = np.concatenate([g.uniform(-464, 464, 4000), g.normal(0, 1, 4000),
                        g.normal(0, 2.0 ** -7, 4000)]).astype(np.float32)
    lib = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = m.e4m3_encode(y)
    assert np.array_equal(ours, lib), np.nonzero(ours != lib)


def _slices(seed, B=2, H=3, N=37, d=16):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(B, H, N, d, generator=g) * torch.tensor([0.01, 1.0, 30.0]).reshape(1, H, 1, 1))
    return x.to(torch.bfloat16)


def pin_quantize_scaling(m):
    x = _slices(11)
    codes, descale = m.quantize_e4m3(x)
    assert codes.dtype == torch.uint8 and descale.dtype == torch.float32
    vals = torch.from_numpy(m.e4m3_decode(codes.numpy()))
    xf = x.float()
    B, H = x.shape[:2]
    for b in range(B):
        for h in range(H):
            amax = xf[b, h].abs().max()
            # the slice maximum lands on +-448 exactly
            assert vals[b, h].abs().max().item() == 448.0
            assert descale[b, h].item() == (amax / 448.0).item()
    # dequantised value within half a step of x (relative 2^-4 for normal
    # codes; 2^-10 * descale absolute below the smallest normal)
    xh = m.dequantize_e4m3(codes, descale)
    tol = torch.maximum(2.0 ** -4 * xf.double().abs(),
                        2.0 ** -10 * descale.double().reshape(B, H, 1, 1)) * (1 + 1e-6)
    assert ((xh - xf.double()).abs() <= tol).all()


def pin_quantize_power_of_two(m):
    x = _slices(12)
    c0, d0 = m.quantize_e4m3(x)
    c1, d1 = m.quantize_e4m3(x * torch.tensor([1.0, 8.0, 0.25]).reshape(1, 3, 1, 1).to(torch.bfloat16))
    assert torch.equal(c0, c1)
    assert torch.equal(d1, d0 * torch.tensor([1.0, 8.0, 0.25]).reshape(1, 3))
    # slices are independent: changing one leaves the others alone
    y = x.clone()
    y[0, 0] *= 3
    c2, d2 = m.quantize_e4m3(y)
    mask = torch.ones(2, 3, dtype=torch.bool)
    mask[0, 0] = False
    assert torch.equal(c2[mask], c0[mask]) and torch.equal(d2[mask], d0[mask])
    # an all-zero slice: zero codes, zero descale
    z = x.clone()
    z[1, 2] = 0
    c3, d3 = m.quantize_e4m3(z)
    assert (c3[1, 2] == 0).all() and d3[1, 2].item() == 0.0


def pin_transpose_layout(m):
    c = torch.arange(2 * 5 * 3, dtype=torch.uint8).reshape(1, 2, 5, 3)
    t = m.transpose_keys_last(c, 16)
    assert t.shape == (1, 2, 3, 16)
    assert t[0, 1, 2, 4].item() == c[0, 1, 4, 2].item()
    assert (t[..., 5:] == 0).all()


def pin_attention_fp8(m):
    g = torch.Generator().manual_seed(21)
    B, H, N, d = 1, 2, 9, 8
    rnd = lambda: torch.randint(0, 0x70, (B, H, N, d), generator=g, dtype=torch.uint8) | \
        (torch.randint(0, 2, (B, H, N, d), generator=g, dtype=torch.uint8) << 7)
    q8, k8, v8 = rnd(), rnd(), rnd()
    dq = torch.tensor([[0.01, 0.002]]); dk = torch.tensor([[0.03, 0.004]])
    dv = torch.tensor([[0.5, 2.0]])
    dec = lambda c, s: torch.from_numpy(of.e4m3_decode(c.numpy())) * s.double().reshape(B, H, 1, 1)
    # one key: O = V^ of that key, L = its score (written out, not via the oracle)
    O1, L1 = m.attention_fp8(q8[:, :, :1], k8[:, :, :1], v8[:, :, :1], dq, dk, dv, 0.7)
    qh, kh, vh = dec(q8[:, :, :1], dq), dec(k8[:, :, :1], dk), dec(v8[:, :, :1], dv)
    assert torch.allclose(O1, vh, rtol=0, atol=1e-12)
    assert torch.allclose(L1, 0.7 * (qh * kh).sum(-1), rtol=1e-12, atol=1e-12)
    # descale_q * t == scale * t; O linear in descale_v, L independent of it
    Oa, La = m.attention_fp8(q8, k8, v8, dq * 4, dk, dv, 0.3, True)
    Ob, Lb = m.attention_fp8(q8, k8, v8, dq, dk, dv, 1.2, True)
    assert torch.allclose(Oa, Ob, rtol=1e-12, atol=1e-12) and torch.allclose(La, Lb, rtol=1e-12, atol=1e-12)
    Oc, Lc = m.attention_fp8(q8, k8, v8, dq, dk, dv * 3, 1.2, True)
    assert torch.allclose(Oc, 3 * Ob, rtol=1e-12, atol=1e-12) and torch.equal(Lc, Lb)
    # against brute force on the decoded values (pure-Python fsum loops)
    qd, kd, vd = dec(q8, dq), dec(k8, dk), dec(v8, dv)
    Od, Ld = m.attention_fp8(q8, k8, v8, dq, dk, dv, 0.9, True)
    for b in range(B):
        for h in range(H):
            for i in range(N):
                s = [0.9 * math.fsum(qd[b, h, i, t].item() * kd[b, h, k, t].item() for t in range(d))
                     for k in range(i + 1)]
                mx = max(s)
                L = mx + math.log(math.fsum(math.exp(x - mx) for x in s))
                assert abs(Ld[b, h, i].item() - L) < 1e-9
                for t in range(d):
                    o = math.fsum(math.exp(s[k] - L) * vd[b, h, k, t].item() for k in range(i + 1))
                    assert abs(Od[b, h, i, t].item() - o) < 1e-9


ALL_PINS = [pin_decode_fixed_points, pin_decode_library, pin_encode_round_trip,
            pin_encode_midpoints, pin_encode_saturation_nan, pin_encode_library,
            pin_quantize_scaling, pin_quantize_power_of_two, pin_transpose_layout,
            pin_attention_fp8]


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_fp8_oracle_pin(pin):
    pin(of)


# ------------------------------------------------------------------ mutants

def _decode_bias8(codes):
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    e, mm = (c >> 3) & 0xF, c & 7
    v = np.where(e == 0, mm * 2.0 ** -9, (1 + mm / 8) * np.exp2(e - 8.0))
    return np.where(c & 0x80, -v, v)


def _encode_truncate(y):
    y = np.asarray(y, dtype=np.float64)
    a = np.minimum(np.abs(y), 448.0)
    E = np.clip(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6, 8)
    q = np.floor(a / np.exp2(E - 3))
    code = np.where(a < 2.0 ** -6, np.floor(a / 2.0 ** -9), (E + 7) * 8 + (q - 8)).astype(np.int64)
    return np.where(np.signbit(y), code | 0x80, code).astype(np.uint8)


def _encode_half_up(y):
    y = np.asarray(y, dtype=np.float64)
    a = np.minimum(np.abs(y), 448.0)
    E = np.clip(np.floor(np.log2(np.where(a > 0, a, 1.0))), -6, 8)
    q = np.floor(a / np.exp2(E - 3) + 0.5)
    carry = q >= 16
    E, q = np.where(carry, E + 1, E), np.where(carry, 8, q)
    code = np.where(a < 2.0 ** -6, np.floor(a / 2.0 ** -9 + 0.5), (E + 7) * 8 + (q - 8))
    code = np.minimum(code, 0x7E).astype(np.int64)
    return np.where(np.signbit(y), code | 0x80, code).astype(np.uint8)


def _quantize_global_amax(x):
    xf = x.detach().float().numpy()
    amax = np.float32(np.abs(xf).max())
    s = np.float32(448.0) / amax
    codes = of.e4m3_encode((xf * s).astype(np.float32))
    B, H = xf.shape[:2]
    return torch.from_numpy(codes), torch.full((B, H), float(amax / np.float32(448.0)))


def _attention_no_descale_v(q8, k8, v8, dq, dk, dv, scale, causal=False):
    q = of.dequantize_e4m3(q8, dq)
    k = of.dequantize_e4m3(k8, dk)
    v = of.dequantize_e4m3(v8, torch.ones_like(dv))
    return oracle.attention_ref(q, k, v, scale, causal)


def _transpose_no_pad_zero(codes, pitch):
    B, H, N, d = codes.shape
    out = torch.full((B, H, d, pitch), 0x11, dtype=torch.uint8)
    out[:, :, :, :N] = codes.transpose(-1, -2)
    return out


MUTANTS = {
    "decode_bias8": ("e4m3_decode", _decode_bias8),
    "encode_truncate": ("e4m3_encode", _encode_truncate),
    "encode_half_up": ("e4m3_encode", _encode_half_up),
    "quantize_global_amax": ("quantize_e4m3", _quantize_global_amax),
    "quantize_descale_inverted": ("quantize_e4m3", None),
    "attention_no_descale_v": ("attention_fp8", _attention_no_descale_v),
    "transpose_pad_garbage": ("transpose_keys_last", _transpose_no_pad_zero),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_fp8_pins_catch_mutant(name, monkeypatch):
    attr, fn = MUTANTS[name]
    if name == "quantize_descale_inverted":
        orig = of.quantize_e4m3
        fn = lambda x, _o=orig: (lambda c, d: (c, torch.where(d > 0, 1.0 / d, d)))(*_o(x))
    monkeypatch.setattr(of, attr, fn)
    failed = []
    for pin in ALL_PINS:
        try:
            pin(of)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"mutant {name} passed every pin"
