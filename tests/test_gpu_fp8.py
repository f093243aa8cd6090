"""The 8-bit (E4M3) path against the float64 oracle.

Quantisation is integer work decided by fp32 arithmetic both sides perform
in the same precision, so codes and descales must match bit for bit.

The forward is compared with the exact attention of the dequantised inputs
(``oracle.attention_fp8``).  No tolerance is stated for 8-bit inputs; this
one follows from the arithmetic.  The kernel rounds each softmax weight
P~ (in [0, 2^8] relative to its reference maximum, which never exceeds the
row maximum) to E4M3 before the P~ V product: an error of at most 2^-4 P~
for normal codes and at most min(2^-10, P~) below the smallest normal 2^-6.
In units of the normalised weights P_k that is
    e_k = max(2^-4 P_k, min(2^-10 / l_R, P_k)),  l_R = sum_k exp(s_k - max s)
(the kernel's row sum is at least l_R).  The numerator then moves by at
most sum_k e_k |V_kd| and the normaliser (the fp32 sum, corrected by the
rounding error of the largest weight of each 128-key half block) by at most
|O_d| sum_k e_k, over a denominator at least f = 1 - 2^-4 - n_h 2^-10 / l_R
of the true one (n_h half blocks the row sees; a half block whose largest
weight is below 2^-6 corrects by at most 2^-10).  With fp32 accumulation
(2^-12 of sum_k P_k |V_kd|) and the bf16 output (one ulp):
    |O_d - O_ref_d| <= (sum_k e_k |V_kd| + |O_ref_d| sum_k e_k) / f
                       + 2^-12 sum_k P_k |V_kd| + ulp_bf16(O_ref_d).
L comes from the fp32 sum of unrounded weights: |L - L_ref| <= 1e-3 as for
bf16 inputs.  The mean of |error| / bound is also checked (<= 0.25), so a
systematic error well inside the worst case still fails.
"""
import math

import pytest
import torch

import oracle
from exact_attention_forward_04_gb300 import (check_errors, forward_e4m3, quantize_e4m3,
                                              quantize_qkv_e4m3)
from exact_attention_forward_04_gb300.inputs import BY_NAME, make_e4m3_codes, make_qkv, make_workload
from tests.parity import L_TOL, fp8_o_bound as _bound

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _keys_last(codes):
    """[B, H, N, d] -> [B, H, d, P] with zero padding (test glue: a copy)."""
    B, H, N, d = codes.shape
    P = (N + 15) // 16 * 16
    out = torch.zeros(B, H, d, P, dtype=torch.uint8)
    out[..., :N] = codes.transpose(-1, -2)
    return out


def _check(o, lse, O_ref, L_ref, bound, what):
    o64 = o.detach().to("cpu", torch.float64)
    l64 = lse.detach().to("cpu", torch.float64)
    assert torch.isfinite(o64).all() and torch.isfinite(l64).all(), f"{what}: non-finite"
    err = (o64 - O_ref).abs()
    ratio = err / bound
    dL = (l64 - L_ref).abs().max().item()
    worst, mean = ratio.max().item(), ratio.mean().item()
    assert worst <= 1.0, f"{what}: max |dO| {err.max().item():.3e} = x{worst:.2f} of bound"
    assert mean <= 0.25, f"{what}: mean |dO|/bound {mean:.3f}"
    assert dL <= L_TOL, f"{what}: max |dL| {dL:.3e}"
    return worst, mean


# ------------------------------------------------------------ quantisation

@pytest.mark.parametrize("N,d", [(1, 64), (100, 128), (300, 64), (1000, 128), (2048, 128)])
@pytest.mark.parametrize("keys_last", [False, True])
def test_quantize_bit_exact(N, d, keys_last):
    B, H = 2, 3
    q, k, v = make_qkv(B, H, N, d, seed=900 + N + d)
    x = (q.float() * torch.tensor([0.01, 1.0, 40.0]).reshape(1, H, 1, 1)).to(torch.bfloat16)
    x[1, 1] = 0  # an all-zero slice
    codes, ds = quantize_e4m3(x.to(DEV), keys_last=keys_last)
    check_errors()
    ref_codes, ref_ds = oracle.quantize_e4m3(x)
    if keys_last:
        ref_codes = oracle.transpose_keys_last(ref_codes, (N + 15) // 16 * 16)
    assert torch.equal(ds.cpu(), ref_ds), (ds.cpu(), ref_ds)
    got = codes.cpu()
    assert got.shape == ref_codes.shape
    bad = (got != ref_codes).nonzero()
    assert bad.numel() == 0, f"{bad.shape[0]} codes differ, first at {bad[0].tolist()}"


@pytest.mark.parametrize("N,d", [(1, 64), (300, 128), (1000, 64), (2048, 128)])
def test_quantize_qkv_matches_single_calls_and_oracle(N, d):
    B, H = 2, 3
    q, k, v = make_qkv(B, H, N, d, seed=1700 + N + d)
    v = (v.float() * torch.tensor([0.01, 1.0, 40.0]).reshape(1, H, 1, 1)).to(torch.bfloat16)
    k[1, 2] = 0  # an all-zero slice
    qd, kd, vd = (t.to(DEV) for t in (q, k, v))
    q8, k8, vt8, dq, dk, dv = quantize_qkv_e4m3(qd, kd, vd)
    check_errors()
    singles = [quantize_e4m3(t, keys_last=(i == 2)) for i, t in enumerate((qd, kd, vd))]
    for got, one in zip((q8, k8, vt8), singles):
        assert torch.equal(got, one[0])
    for got, one in zip((dq, dk, dv), singles):
        assert torch.equal(got, one[1])
    for i, (t, c, s) in enumerate(((q, q8, dq), (k, k8, dk), (v, vt8, dv))):
        ref_c, ref_s = oracle.quantize_e4m3(t)
        if i == 2:
            ref_c = oracle.transpose_keys_last(ref_c, (N + 15) // 16 * 16)
        assert torch.equal(c.cpu(), ref_c) and torch.equal(s.cpu(), ref_s)


# ------------------------------------------------------- forward on codes

CASES = [(N, causal) for N in (1, 100, 128, 256, 300, 700, 1000) for causal in (False, True)]


@pytest.mark.parametrize("N,causal", CASES)
def test_fwd_e4m3_quantized_inputs(N, causal):
    # bf16 inputs; each side quantises them with its own code
    B, H, d = 1, 2, 128
    q, k, v = make_qkv(B, H, N, d, seed=1300 + N + int(causal))
    scale = 1.0 / math.sqrt(d)
    (q8, dq), (k8, dk), (vt8, dv) = (quantize_e4m3(t.to(DEV), keys_last=(i == 2))
                                     for i, t in enumerate((q, k, v)))
    o, lse = forward_e4m3(q8, k8, vt8, dq, dk, dv, scale=scale, causal=causal)
    check_errors()
    rq, rdq = oracle.quantize_e4m3(q)
    rk, rdk = oracle.quantize_e4m3(k)
    rv, rdv = oracle.quantize_e4m3(v)
    assert torch.equal(q8.cpu(), rq) and torch.equal(k8.cpu(), rk)
    assert torch.equal(vt8.cpu(), oracle.transpose_keys_last(rv, vt8.shape[-1]))
    O_ref, L_ref = oracle.attention_fp8(rq, rk, rv, rdq, rdk, rdv, scale, causal)
    deq = [oracle.dequantize_e4m3(c, s) for c, s in ((rq, rdq), (rk, rdk), (rv, rdv))]
    bound = _bound(*deq, O_ref, scale, causal)
    _check(o, lse, O_ref, L_ref, bound, f"N={N} causal={causal}")


@pytest.mark.parametrize("N,causal", [(N, causal) for N in (1, 100, 256, 300, 1000)
                                      for causal in (False, True)])
def test_fwd_e4m3_head_dim_64(N, causal):
    # head dim 64: 64-byte code rows, zero-padded to the kernel's 128-byte
    # rows by the TMA; each side quantises the same bf16 inputs
    B, H, d = 2, 3, 64
    q, k, v = make_qkv(B, H, N, d, seed=1500 + N + int(causal))
    scale = 1.0 / math.sqrt(d)
    q8, k8, vt8, dq, dk, dv = quantize_qkv_e4m3(q.to(DEV), k.to(DEV), v.to(DEV))
    o, lse = forward_e4m3(q8, k8, vt8, dq, dk, dv, scale=scale, causal=causal)
    check_errors()
    refs = [oracle.quantize_e4m3(t) for t in (q, k, v)]
    assert torch.equal(q8.cpu(), refs[0][0]) and torch.equal(k8.cpu(), refs[1][0])
    O_ref, L_ref = oracle.attention_fp8(refs[0][0], refs[1][0], refs[2][0], refs[0][1],
                                        refs[1][1], refs[2][1], scale, causal)
    deq = [oracle.dequantize_e4m3(c, s) for c, s in refs]
    _check(o, lse, O_ref, L_ref, _bound(*deq, O_ref, scale, causal), f"d=64 N={N} causal={causal}")


@pytest.mark.parametrize("N,causal,max_e,d", [(300, False, 9, 128), (700, True, 12, 128),
                                              (513, False, 14, 128), (700, True, 12, 64),
                                              (513, False, 14, 64)])
def test_fwd_e4m3_random_codes(N, causal, max_e, d):
    # raw codes over a wide exponent range (peaky rows), random descales
    B, H = 1, 2
    (q8, k8, v8), (dq, dk, dv) = make_e4m3_codes(B, H, N, d, seed=77 + N + d, max_exp_field=max_e)
    scale = 0.125
    o, lse = forward_e4m3(q8.to(DEV), k8.to(DEV), _keys_last(v8).to(DEV), dq.to(DEV), dk.to(DEV),
                          dv.to(DEV), scale=scale, causal=causal)
    check_errors()
    O_ref, L_ref = oracle.attention_fp8(q8, k8, v8, dq, dk, dv, scale, causal)
    deq = [oracle.dequantize_e4m3(c, s) for c, s in ((q8, dq), (k8, dk), (v8, dv))]
    _check(o, lse, O_ref, L_ref, _bound(*deq, O_ref, scale, causal), f"codes N={N}")


def test_fwd_e4m3_padding_ignored():
    # columns >= N of the keys-last V are ignored whatever they hold
    B, H, N, d = 1, 1, 100, 128
    (q8, k8, v8), (dq, dk, dv) = make_e4m3_codes(B, H, N, d, seed=5)
    vt = _keys_last(v8)
    vt[..., N:] = 0x7F  # NaN codes in the padding
    o, lse = forward_e4m3(q8.to(DEV), k8.to(DEV), vt.to(DEV), dq.to(DEV), dk.to(DEV), dv.to(DEV),
                          scale=0.1)
    check_errors()
    O_ref, L_ref = oracle.attention_fp8(q8, k8, v8, dq, dk, dv, 0.1, False)
    deq = [oracle.dequantize_e4m3(c, s) for c, s in ((q8, dq), (k8, dk), (v8, dv))]
    _check(o, lse, O_ref, L_ref, _bound(*deq, O_ref, 0.1, False), "padding")


def test_fwd_e4m3_zero_descale():
    # a zero descale (an all-zero slice) makes every score 0: O = mean of V
    B, H, N, d = 1, 2, 300, 128
    (q8, k8, v8), (dq, dk, dv) = make_e4m3_codes(B, H, N, d, seed=6)
    dq[0, 1] = 0.0
    o, lse = forward_e4m3(q8.to(DEV), k8.to(DEV), _keys_last(v8).to(DEV), dq.to(DEV), dk.to(DEV),
                          dv.to(DEV), scale=0.1, causal=True)
    check_errors()
    O_ref, L_ref = oracle.attention_fp8(q8, k8, v8, dq, dk, dv, 0.1, True)
    deq = [oracle.dequantize_e4m3(c, s) for c, s in ((q8, dq), (k8, dk), (v8, dv))]
    _check(o, lse, O_ref, L_ref, _bound(*deq, O_ref, 0.1, True), "zero descale")
    assert torch.allclose(lse[0, 1].cpu().double(), torch.log(torch.arange(1, N + 1).double()),
                          atol=1e-5)


@pytest.mark.parametrize("name,heads,rows", [
    ("b4h16n2048d128", ((0, 0), (3, 15)), (0, 1, 777, 2047)),
    ("b2h32n8192d128_causal", ((1, 31),), (0, 5, 4096, 8191)),
    ("b16h32n1024d64_peaky", ((0, 0), (15, 31)), (0, 1, 255, 256, 1023)),
])
def test_fwd_e4m3_full_size(name, heads, rows):
    # the full workload quantised and run through the library; sampled heads'
    # codes bit-exact and sampled rows against the oracle
    w = BY_NAME[name]
    q, k, v = make_workload(w)
    (q8, dq), (k8, dk), (vt8, dv) = (quantize_e4m3(t.to(DEV), keys_last=(i == 2))
                                     for i, t in enumerate((q, k, v)))
    o, lse = forward_e4m3(q8, k8, vt8, dq, dk, dv, scale=w.scale, causal=w.causal)
    check_errors()
    rows = torch.tensor(rows)
    for (b, h) in heads:
        sl = (slice(b, b + 1), slice(h, h + 1))
        refs = [oracle.quantize_e4m3(t[sl]) for t in (q, k, v)]
        assert torch.equal(q8[sl].cpu(), refs[0][0]) and torch.equal(k8[sl].cpu(), refs[1][0])
        assert torch.equal(vt8[sl].cpu(), oracle.transpose_keys_last(refs[2][0], vt8.shape[-1]))
        for t, (c, s) in zip((dq, dk, dv), refs):
            assert torch.equal(t[sl].cpu(), s)
        deq = [oracle.dequantize_e4m3(c, s) for c, s in refs]
        qd, kd, vd = deq
        O_ref, L_ref = oracle.attention_ref(qd[:, :, rows], kd, vd, w.scale, False) if not w.causal \
            else _causal_rows(qd, kd, vd, w.scale, rows)
        bound = _bound(qd, kd, vd, O_ref, w.scale, w.causal, rows)
        _check(o[sl][:, :, rows], lse[sl][:, :, rows], O_ref, L_ref, bound, f"{name} {(b, h)}")


def _causal_rows(q, k, v, scale, rows):
    O, L = [], []
    for r in rows.tolist():
        o_, l_ = oracle.attention_ref(q[:, :, r:r + 1], k[:, :, :r + 1], v[:, :, :r + 1], scale, False)
        O.append(o_)
        L.append(l_)
    return torch.cat(O, dim=2), torch.cat(L, dim=2)


@pytest.mark.parametrize("N,causal,d", [(200, False, 128), (200, True, 128), (512, True, 128),
                                        (512, True, 64)])
def test_fwd_e4m3_chains_of_short_units(N, causal, d):
    # 608 heads of one or two 256-row tiles: every cluster runs a chain of
    # work units of one or two key blocks (the 8-bit kernel keeps two P~
    # buffers, so its softmax warps run furthest ahead of the epilogue).
    # Each launch must complete, repeat bit for bit, and stay within the
    # bound on sampled heads.
    B, H = 2, 304
    q, k, v = make_qkv(B, H, N, d, seed=4300 + N + int(causal) + d)
    scale = 1.0 / math.sqrt(d)
    q8, k8, vt8, dq, dk, dv = quantize_qkv_e4m3(q.to(DEV), k.to(DEV), v.to(DEV))
    first = None
    for _ in range(5):
        o, lse = forward_e4m3(q8, k8, vt8, dq, dk, dv, scale=scale, causal=causal)
        check_errors()
        if first is None:
            first = (o.clone(), lse.clone())
        else:
            assert torch.equal(o, first[0]) and torch.equal(lse, first[1])
    for b, h in ((0, 0), (0, 151), (1, 76), (1, 303)):
        refs = [oracle.quantize_e4m3(t[b:b + 1, h:h + 1]) for t in (q, k, v)]
        O_ref, L_ref = oracle.attention_fp8(refs[0][0], refs[1][0], refs[2][0], refs[0][1],
                                            refs[1][1], refs[2][1], scale, causal)
        deq = [oracle.dequantize_e4m3(c, s) for c, s in refs]
        _check(o[b:b + 1, h:h + 1], lse[b:b + 1, h:h + 1], O_ref, L_ref,
               _bound(*deq, O_ref, scale, causal), f"N={N} causal={causal} head ({b}, {h})")
