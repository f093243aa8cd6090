"""Standard (unfused) attention on the GPU (fa_attn_unfused, three kernels
with S and P in device memory) against the float64 oracle: O and L element
by element at the forward's tolerance, and the intermediate S (fp32) and P
(bf16) against the oracle's scores and probabilities.

Bounds on the intermediates (derived here, none is stated):
  * S: products of bf16 inputs (exact in fp32) summed over d <= 128 terms
    by the tensor core in fp32: |S - S_ref| <= 2^-14 * sum_t |scale q_t k_t|
    (d * 2^-24 = 2^-17 per unit of that sum, with room for the adder's
    internal rounding order).
  * P: exp(S - L) in fp32 (ex2.approx), then rounded to bf16 (2^-9
    relative): |P - P_ref| <= 2^-8 P_ref + 2^-24, and exactly 0 at masked
    keys inside the row's 128-row tile.
"""
import math

import pytest
import torch

import oracle
from exact_attention_forward_04_gb300 import (attention_unfused, check_errors, forward,
                                              unfused_intermediates, unfused_workspace_size)
from exact_attention_forward_04_gb300.inputs import BY_NAME, make_qkv, make_workload
from tests.parity import assert_close, compare

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run(q, k, v, scale, causal):
    B, H, N, d = q.shape
    ws = torch.empty(unfused_workspace_size(B, H, N, d), dtype=torch.uint8, device=DEV)
    o, lse = attention_unfused(q.to(DEV), k.to(DEV), v.to(DEV), scale=scale, causal=causal,
                               workspace=ws)
    check_errors()
    return o, lse, ws


SMALL = [(B, H, N, d, causal)
         for (B, H) in ((1, 1), (2, 3))
         for N in (1, 7, 64, 129, 300, 513)
         for d in (64, 128)
         for causal in (False, True)]


@pytest.mark.parametrize("B,H,N,d,causal", SMALL)
def test_unfused_small_shapes(B, H, N, d, causal):
    q, k, v = make_qkv(B, H, N, d, seed=3000 + N + d + int(causal) + 11 * H)
    scale = 1.0 / math.sqrt(d)
    o, lse, ws = _run(q, k, v, scale, causal)
    O_ref, L_ref = oracle.attention_ref(q, k, v, scale, causal)
    assert_close(o, lse, O_ref, L_ref, f"unfused B={B} H={H} N={N} d={d} causal={causal}")


@pytest.mark.parametrize("d", (64, 128))
@pytest.mark.parametrize("causal", (False, True))
def test_unfused_intermediates(d, causal):
    B, H, N = 1, 2, 300
    scale = 1.0 / math.sqrt(d)
    q, k, v = make_qkv(B, H, N, d, seed=3100 + d + int(causal))
    o, lse, ws = _run(q, k, v, scale, causal)
    S, P = unfused_intermediates(ws, B, H, N)
    S, P = S.cpu().double(), P.cpu().double()
    _, _, S_ref, P_ref = oracle.standard_attention(q, k, v, scale, causal)
    rows = torch.arange(N).view(-1, 1)
    keys = torch.arange(N).view(1, -1)
    vis = (keys <= rows) if causal else torch.ones(N, N, dtype=torch.bool)
    # S: every visible score was computed
    absterm = scale * torch.matmul(q.double().abs(), k.double().abs().transpose(-1, -2))
    dS = (S - S_ref).abs()
    assert bool((dS[..., vis] <= 2.0 ** -14 * absterm[..., vis] + 1e-30).all()), \
        f"S max error {dS[..., vis].max().item():.3e}"
    # P: visible keys within the bf16 bound, masked keys of the row's tile 0
    dP = (P - P_ref).abs()
    assert bool((dP[..., vis] <= 2.0 ** -8 * P_ref[..., vis] + 2.0 ** -24).all()), \
        f"P max error {dP[..., vis].max().item():.3e}"
    if causal:
        tile_end = torch.clamp((rows // 128 + 1) * 128, max=N)
        masked_in_tile = (keys > rows) & (keys < tile_end)
        assert bool((P[..., masked_in_tile] == 0).all())


@pytest.mark.parametrize("scale", (-0.3, -0.02, 0.0))
def test_unfused_any_scale(scale):
    q, k, v = make_qkv(1, 2, 200, 128, seed=3200)
    for causal in (False, True):
        o, lse, _ = _run(q, k, v, scale, causal)
        O_ref, L_ref = oracle.attention_ref(q, k, v, scale, causal)
        assert_close(o, lse, O_ref, L_ref, f"unfused scale={scale} causal={causal}")


def test_unfused_peaky_d64():
    q, k, v = make_qkv(2, 2, 384, 64, seed=3300, sigma_q=3.0, sigma_k=3.0)
    o, lse, _ = _run(q, k, v, 0.125, False)
    O_ref, L_ref = oracle.attention_ref(q, k, v, 0.125, False)
    assert_close(o, lse, O_ref, L_ref, "unfused peaky")


def test_unfused_outputs_fully_written_and_deterministic():
    B, H, N, d = 1, 3, 333, 128
    q, k, v = (t.to(DEV) for t in make_qkv(B, H, N, d, seed=3400))
    ws = torch.empty(unfused_workspace_size(B, H, N, d), dtype=torch.uint8, device=DEV)
    o1, l1 = attention_unfused(q, k, v, causal=True, workspace=ws)
    ws.fill_(0xFF)  # NaN patterns in S and P: everything read must be rewritten
    o2, l2 = attention_unfused(q, k, v, causal=True, workspace=ws)
    check_errors()
    assert torch.isfinite(o2.float()).all() and torch.isfinite(l2).all()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_unfused_full_size_bench_workload():
    # the benchmark's unfused leg: B=4, H=16, N=2048, d=128, non-causal
    w = BY_NAME["b4h16n2048d128"]
    q, k, v = make_workload(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o, lse, _ = _run(q, k, v, w.scale, w.causal)
    of, lf = forward(qd, kd, vd, scale=w.scale, causal=w.causal)
    check_errors()
    # against the fused kernel everywhere (both are within the oracle's
    # bound, so they differ by at most twice it)
    r = compare(o, lse, of.cpu().double(), lf.cpu().double())
    assert r["max_dO"] <= 2e-2 and r["max_dL"] <= 2e-3, r
    # against the oracle on three whole heads
    for (b, h) in ((0, 0), (1, 7), (3, 15)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        O_ref, L_ref = oracle.attention_ref(q[sl], k[sl], v[sl], w.scale, w.causal)
        assert_close(o.cpu()[sl], lse.cpu()[sl], O_ref, L_ref, f"unfused head {(b, h)}")


@pytest.mark.parametrize("N,d,causal", [(3000, 64, False), (9000, 128, True), (16500, 64, True)])
def test_unfused_softmax_row_lengths(N, d, causal):
    # the softmax keeps a row in registers up to 16384 keys (register tiles
    # of 4, 8, 16, 32 and 64 elements per thread by length) and uses two
    # passes beyond; these lengths reach the 16- and 64-element tiles and the
    # two-pass kernel.  Sampled rows against the oracle.
    B, H = 1, 1
    q, k, v = make_qkv(B, H, N, d, seed=3600 + N + d)
    scale = 1.0 / math.sqrt(d)
    o, lse, _ = _run(q, k, v, scale, causal)
    rows = sorted({0, 1, 127, 128, 1023, 1024, N // 2, N - 2, N - 1})
    picks = [(0, 0, i) for i in rows]
    O_ref, L_ref = oracle.attention_rows(q, k, v, scale, causal, picks)
    idx = torch.tensor(picks)
    assert_close(o.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]], lse.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]],
                 O_ref, L_ref, f"unfused N={N} d={d} causal={causal}")


def test_unfused_causal_long_sampled_rows():
    # 8K causal, 4 heads: sampled rows (tile edges, first, last) against the oracle
    B, H, N, d = 1, 4, 8192, 128
    q, k, v = make_qkv(B, H, N, d, seed=3500)
    o, lse, _ = _run(q, k, v, 1.0 / math.sqrt(d), True)
    rows = sorted({0, 1, 127, 128, 255, 256, 4095, 4096, 8063, 8064, 8190, 8191})
    picks = [(0, h, i) for h in range(H) for i in rows]
    O_ref, L_ref = oracle.attention_rows(q, k, v, 1.0 / math.sqrt(d), True, picks)
    idx = torch.tensor(picks)
    got_o = o.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]]
    got_l = lse.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]]
    assert_close(got_o, got_l, O_ref, L_ref, "unfused 8K causal sampled rows")
