"""The comparison bounds shared by the GPU tests and the benchmark's checks
(tests/parity.py), pinned on the CPU.

- The gradients' term scales A_g of picked rows equal the whole-head sums of
  |terms|, restated here from the gradient formulas.
- The gradient check passes inside its bound and fails beyond it or on a
  non-finite value; the bound covers the gradients computed with P and dS
  rounded to bf16 where the kernels hand them to the tensor core, and
  rounding them to three mantissa bits breaks it.
- The 8-bit O bound covers the error of rounding every softmax weight to
  E4M3 (the oracle's own encoder), and a coarser rounding (one mantissa bit)
  breaks it somewhere, so the bound is not vacuous.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from exact_attention_forward_04_gb300.inputs import make_qkv
from tests.parity import GRAD_A_REL, fp8_o_bound, grad_compare, grad_row_term_scales, half_ulp_bf16

F64 = torch.float64


def _whole_head_term_scales(q, k, v, o, lse, g, scale, causal):
    """|dQ|, |dK|, |dV| term sums over whole heads: with P = exp(scale s - L)
    on visible keys and |dS| <= P (|dO| |V|^T + rowsum |dO| |O|),
    A_dQ = scale |dS| |K|, A_dK = scale |dS|^T |Q|, A_dV = P^T |dO|."""
    B, H, N, _ = q.shape
    out = [torch.empty(q.shape, dtype=F64) for _ in range(3)]
    keep = torch.tril(torch.ones(N, N, dtype=torch.bool)) if causal else torch.ones(N, N, dtype=torch.bool)
    for b in range(B):
        for h in range(H):
            qh, kh, vh, gh, oh = (t[b, h].to(F64) for t in (q, k, v, g, o))
            p = torch.exp(scale * qh @ kh.T - lse[b, h].to(F64)[:, None]) * keep
            ds = p * (gh.abs() @ vh.abs().T + (gh.abs() * oh.abs()).sum(-1, keepdim=True))
            out[0][b, h] = scale * ds @ kh.abs()
            out[1][b, h] = scale * ds.T @ qh.abs()
            out[2][b, h] = p.T @ gh.abs()
    return out


@pytest.mark.parametrize("causal", (False, True))
def test_grad_row_term_scales_match_whole_head(causal):
    B, H, N, d = 1, 2, 37, 16
    q, k, v = make_qkv(B, H, N, d, seed=6101)
    g = make_qkv(B, H, N, d, seed=6102)[0]
    scale = 1.0 / math.sqrt(d)
    O, L = oracle.attention_ref(q, k, v, scale, causal)
    full = _whole_head_term_scales(q, k, v, O, L, g, scale, causal)
    picks = [(0, h, i) for h in (0, 1) for i in (0, 1, 18, 35, 36)]
    rows = grad_row_term_scales(q, k, v, O, L, g, scale, causal, picks, picks)
    idx = torch.tensor(picks)
    for got, ref, nm in zip(rows, full, ("dQ", "dK", "dV")):
        want = ref[idx[:, 0], idx[:, 1], idx[:, 2]]
        assert torch.allclose(got, want, rtol=1e-12, atol=0.0), nm


def test_grad_compare_inside_and_beyond_the_bound():
    ref = torch.tensor([1.0, -2.0, 0.0, 1e-3], dtype=F64)
    A = torch.tensor([4.0, 8.0, 1.0, 1.0], dtype=F64)
    bound = GRAD_A_REL * A + half_ulp_bf16(ref)
    assert grad_compare(ref + 0.9 * bound, ref, A)["ok"]
    bad = ref.clone()
    bad[2] += 1.1 * bound[2]
    r = grad_compare(bad, ref, A)
    assert not r["ok"] and 1.0 < r["max_over_bound"] < 1.2
    nan = ref.clone()
    nan[0] = float("nan")
    assert not grad_compare(nan, ref, A)["ok"]


def _o_with_rounded_weights(q, k, v, scale, causal, rnd):
    """O with every weight exp(s - max s) of a row rounded by rnd in the
    numerator, over the sum of the unrounded weights."""
    B, H, N, _ = q.shape
    out = torch.empty(q.shape, dtype=F64)
    keep = torch.tril(torch.ones(N, N, dtype=torch.bool)) if causal else torch.ones(N, N, dtype=torch.bool)
    for b in range(B):
        for h in range(H):
            s = (scale * q[b, h] @ k[b, h].T).masked_fill(~keep, -math.inf)
            R = torch.exp(s - s.amax(-1, keepdim=True))
            out[b, h] = (rnd(R) @ v[b, h]) / R.sum(-1, keepdim=True)
    return out


def _e4m3(x):
    return torch.from_numpy(oracle.e4m3_decode(oracle.e4m3_encode(x.numpy())))


def _one_mantissa_bit(x):
    m, e = torch.frexp(x)  # x = m 2^e, m in [0.5, 1)
    return torch.ldexp(torch.round(m * 4.0) / 4.0, e)


@pytest.mark.parametrize("causal", (False, True))
def test_fp8_o_bound_covers_e4m3_weights_and_not_coarser_ones(causal):
    B, H, N, d = 1, 2, 300, 64
    q, k, v = make_qkv(B, H, N, d, seed=6201, sigma_q=2.0, sigma_k=2.0)
    deq = [oracle.dequantize_e4m3(*oracle.quantize_e4m3(t)) for t in (q, k, v)]
    deq = [torch.as_tensor(np.asarray(t), dtype=F64) for t in deq]
    scale = 1.0 / math.sqrt(d)
    O_ref, _ = oracle.attention_ref(deq[0], deq[1], deq[2], scale, causal)
    O_ref = O_ref.to(F64)
    bound = fp8_o_bound(deq[0], deq[1], deq[2], O_ref, scale, causal)
    err = (_o_with_rounded_weights(deq[0], deq[1], deq[2], scale, causal, _e4m3) - O_ref).abs()
    assert (err <= bound).all(), f"E4M3 weights: x{(err / bound).max().item():.2f} of the bound"
    err1 = (_o_with_rounded_weights(deq[0], deq[1], deq[2], scale, causal, _one_mantissa_bit)
            - O_ref).abs()
    assert (err1 > bound).any(), "one-bit weights stay inside the bound: the bound is vacuous"


def _bf16(x):
    return x.to(torch.bfloat16).to(F64)


def _mantissa_bits(bits):
    def rnd(x):
        m, e = torch.frexp(x)  # m in [0.5, 1): `bits` bits after the leading one
        return torch.ldexp(torch.round(m * 2.0 ** (bits + 1)) / 2.0 ** (bits + 1), e)
    return rnd


def _grads_with_rounded_p_ds(q, k, v, o, lse, g, scale, causal, rnd):
    """dQ, dK, dV in float64 with P and dS rounded by rnd where the kernels
    hand them to the tensor core as bf16 (P for dV, dS for dQ and dK)."""
    B, H, N, _ = q.shape
    keep = torch.tril(torch.ones(N, N, dtype=torch.bool)) if causal else torch.ones(N, N, dtype=torch.bool)
    out = [torch.empty(q.shape, dtype=F64) for _ in range(3)]
    for b in range(B):
        for h in range(H):
            qh, kh, vh, gh, oh = (t[b, h].to(F64) for t in (q, k, v, g, o))
            p = rnd(torch.exp(scale * qh @ kh.T - lse[b, h].to(F64)[:, None]) * keep)
            ds = rnd(p * (gh @ vh.T - (gh * oh).sum(-1, keepdim=True)))
            out[0][b, h] = scale * ds @ kh
            out[1][b, h] = scale * ds.T @ qh
            out[2][b, h] = p.T @ gh
    return out


@pytest.mark.parametrize("causal", (False, True))
def test_grad_bound_covers_bf16_p_and_ds_and_not_coarser_ones(causal):
    B, H, N, d = 1, 2, 200, 64
    q, k, v = make_qkv(B, H, N, d, seed=6301, sigma_q=2.0, sigma_k=2.0)
    g = make_qkv(B, H, N, d, seed=6302)[0]
    scale = 1.0 / math.sqrt(d)
    O, L = oracle.attention_ref(q, k, v, scale, causal)
    ref = oracle.attention_backward_from_lse(q, k, v, O, L, g, scale, causal)
    A = _whole_head_term_scales(q, k, v, O, L, g, scale, causal)
    sim = _grads_with_rounded_p_ds(q, k, v, O, L, g, scale, causal, _bf16)
    for got, r, a, nm in zip(sim, ref, A, ("dQ", "dK", "dV")):
        res = grad_compare(got, r, a)
        assert res["ok"], f"bf16 P and dS, {nm}: x{res['max_over_bound']:.2f} of the bound"
    coarse = _grads_with_rounded_p_ds(q, k, v, O, L, g, scale, causal, _mantissa_bits(3))
    worst = max(grad_compare(got, r, a)["max_over_bound"] for got, r, a in zip(coarse, ref, A))
    assert worst > 1.0, "P and dS with 3 mantissa bits stay inside the bound: the bound is vacuous"
