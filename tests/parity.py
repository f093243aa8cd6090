"""Comparison helpers for the GPU parity tests.

Tolerances (stated by the workload definition for bf16 inputs):
  max |O - O_ref| <= 1e-2 and max |L - L_ref| <= 1e-3.
The output O must be bf16, and rounding the exact float64 O_ref to bf16
alone already moves it by up to half a bf16 ulp (2^-9 relative, 0.0156 at
|O| >= 4, which peaky rows reach).  The O check is therefore applied
element-wise as |O - O_ref| <= 1e-2 + ulp_bf16(O_ref) / 2; the literal
max |O - O_ref| is always reported beside it.  L is fp32 and checked as stated.
"""
import math

import torch

O_TOL = 1e-2
L_TOL = 1e-3


def half_ulp_bf16(x):
    """Half a bf16 ulp at |x| (float64 tensor); subnormal range clamped."""
    ax = x.abs().clamp_min(2.0 ** -126)
    _, e = torch.frexp(ax)           # ax = m * 2^e, m in [0.5, 1)
    return torch.ldexp(torch.ones_like(ax), (e - 9).to(torch.int32))


def compare(o, lse, O_ref, L_ref):
    """o, lse: GPU outputs (any device); O_ref, L_ref: float64 oracle.
    Returns a dict of error figures and a pass flag."""
    o64 = o.detach().to("cpu", torch.float64)
    l64 = lse.detach().to("cpu", torch.float64)
    O_ref = O_ref.to(torch.float64)
    L_ref = L_ref.to(torch.float64)
    assert o64.shape == O_ref.shape, (o64.shape, O_ref.shape)
    assert l64.shape == L_ref.shape, (l64.shape, L_ref.shape)
    dO = (o64 - O_ref).abs()
    dL = (l64 - L_ref).abs()
    bound = O_TOL + half_ulp_bf16(O_ref)
    finite = bool(torch.isfinite(o64).all() and torch.isfinite(l64).all())
    res = {
        "max_dO": dO.max().item() if dO.numel() else 0.0,
        "max_dO_over_bound": (dO / bound).max().item() if dO.numel() else 0.0,
        "max_dL": dL.max().item() if dL.numel() else 0.0,
        "finite": finite,
    }
    res["ok"] = finite and res["max_dO_over_bound"] <= 1.0 and res["max_dL"] <= L_TOL
    return res


# Gradients (no tolerance is stated for them; this bound is derived): P and
# dS enter the products as bf16, relative rounding <= 2^-9 per term, so an
# element's error scales with the sum of the absolute values of the terms it
# adds, A_g, not with the element itself (dQ and dK cancel to 0 in places):
#   |g - g_ref| <= GRAD_A_REL * A_g + ulp_bf16(g_ref) / 2.
GRAD_A_REL = 2.0 ** -6


def grad_row_term_scales(q, k, v, o, lse, g, scale, causal, q_picks, k_picks):
    """A_g of picked rows (float64): for each query pick (b, h, i) the dQ row's
    sum of |terms|, for each key pick (b, h, j) those of the dK and dV rows,
    with P = exp(scale s - L) from the given L and |dS| bounded by
    P (|dO_i| . |V_j| + sum_t |dO_it O_it|)."""
    d = q.shape[-1]
    aq = torch.empty(len(q_picks), d, dtype=torch.float64)
    ak = torch.empty(len(k_picks), d, dtype=torch.float64)
    av = torch.empty(len(k_picks), d, dtype=torch.float64)
    for n, (b, h, i) in enumerate(q_picks):
        qi, kh, vh = q[b, h, i].double(), k[b, h].double(), v[b, h].double()
        gi, oi = g[b, h, i].double(), o[b, h, i].double()
        p = torch.exp(scale * (kh @ qi) - float(lse[b, h, i]))
        if causal:
            p[i + 1:] = 0.0
        ds_abs = p * (vh.abs() @ gi.abs() + (gi.abs() * oi.abs()).sum())
        aq[n] = scale * (ds_abs @ kh.abs())
    for n, (b, h, j) in enumerate(k_picks):
        qh, gh, oh = q[b, h].double(), g[b, h].double(), o[b, h].double()
        p = torch.exp(scale * (qh @ k[b, h, j].double()) - lse[b, h].double())
        if causal:
            p[:j] = 0.0
        ds_abs = p * (gh.abs() @ v[b, h, j].double().abs() + (gh.abs() * oh.abs()).sum(-1))
        ak[n] = scale * (ds_abs @ qh.abs())
        av[n] = p @ gh.abs()
    return aq, ak, av


def grad_compare(got, ref, a_scale):
    """A gradient (any device) against the float64 oracle under the bound
    above; returns error figures and a pass flag."""
    got = got.detach().to("cpu", torch.float64)
    ref = ref.to(torch.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    bound = GRAD_A_REL * a_scale.to(torch.float64) + half_ulp_bf16(ref)
    err = (got - ref).abs()
    res = {
        "max_err": err.max().item() if err.numel() else 0.0,
        "max_over_bound": (err / bound).max().item() if err.numel() else 0.0,
        "max_rel": (err.max().item() / max(ref.abs().max().item(), 1e-30)) if err.numel() else 0.0,
        "finite": bool(torch.isfinite(got).all()),
    }
    res["ok"] = res["finite"] and res["max_over_bound"] <= 1.0
    return res


def fp8_o_bound(q, k, v, O_ref, scale, causal, rows=None):
    """Per-element bound on |O - O_ref| of the 8-bit forward (float64
    [B, H, R, d]) for dequantised q, k, v (float64 [B, H, N, d]); rows: the
    query rows to cover (default all).  P~ is rounded to E4M3 before the
    P~ V product, an error of at most 2^-4 P~ for normal codes and
    min(2^-10, P~) below 2^-6; in units of the normalised weights
        e_k = max(2^-4 P_k, min(2^-10 / l_R, P_k)),
    over a denominator at least f = 1 - 2^-4 - n_h 2^-10 / l_R (n_h the
    128-key half blocks the row sees), plus fp32 accumulation and the bf16
    output:
        (sum_k e_k |V_kd| + |O_ref_d| sum_k e_k) / f
        + 2^-12 sum_k P_k |V_kd| + ulp_bf16(O_ref_d)."""
    B, H, N, d = q.shape
    rows = torch.arange(N) if rows is None else torch.as_tensor(rows)
    out = torch.empty(B, H, len(rows), d, dtype=torch.float64)
    vis = torch.ones(len(rows), N, dtype=torch.bool)
    if causal:
        vis = torch.arange(N).reshape(1, -1) <= rows.reshape(-1, 1)
    for b in range(B):
        for h in range(H):
            s = scale * (q[b, h, rows] @ k[b, h].T)
            s = s.masked_fill(~vis, -math.inf)
            m = s.amax(-1, keepdim=True)
            R = torch.exp(s - m)
            lR = R.sum(-1, keepdim=True)
            P = R / lR
            e = torch.maximum(2.0 ** -4 * P, torch.minimum(2.0 ** -10 / lR, P))
            n_h = torch.ceil(vis.sum(-1, keepdim=True).double() / 128)
            f = 1 - 2.0 ** -4 - n_h * 2.0 ** -10 / lR
            av = v[b, h].abs()
            out[b, h] = (e @ av + O_ref[b, h].abs() * e.sum(-1, keepdim=True)) / f \
                + 2.0 ** -12 * (P @ av) + 2 * half_ulp_bf16(O_ref[b, h])
    return out


def assert_close(o, lse, O_ref, L_ref, what=""):
    r = compare(o, lse, O_ref, L_ref)
    assert r["ok"], f"{what}: {r}"
    return r
