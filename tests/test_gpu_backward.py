"""The attention backward (fa_bwd) against the float64 oracle.

The kernels recompute P from S and the forward's logsumexp, so the
reference is the oracle's gradient computed the same way from the GPU
forward's own O and L (attention_backward_from_lse); the exact gradient
(attention_backward) is checked with the same bound.

Bound (no tolerance is stated for gradients; this one follows from the
arithmetic): P and dS enter the tensor-core products as bf16 (relative
rounding <= 2^-9 per term), D comes from the bf16 O, and the sums accumulate
in fp32, so an element's error is a small multiple of 2^-9 times the sum of
the absolute values of the terms it adds up, A_g (|dS| built from |dP| and
|D|, then |dS| |K| and so on), not of the element itself: dQ and dK cancel
to 0 in places.  The test allows |g - g_ref| <= 2^-6 A_g + half a bf16 ulp
of g_ref (the output format), element by element, and reports the largest
error relative to max|g_ref|.
"""
import math

import pytest
import torch

import oracle
from exact_attention_forward_04_gb300 import backward, check_errors, forward
from exact_attention_forward_04_gb300.inputs import make_qkv, make_workload, BY_NAME
from tests.parity import grad_compare, grad_row_term_scales

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _term_scales(q, k, v, o, lse, g, scale, causal):
    """A_g for dQ, dK, dV: each gradient's terms in absolute value (float64)."""
    B, H, N, _ = q.shape
    vis = torch.ones(N, N, dtype=torch.bool)
    if causal:
        vis = torch.arange(N).reshape(1, -1) <= torch.arange(N).reshape(-1, 1)
    out = [torch.empty(q.shape, dtype=torch.float64) for _ in range(3)]
    for b in range(B):
        for h in range(H):
            qh, kh, vh, gh, oh = (t[b, h].double() for t in (q, k, v, g, o))
            s_ = scale * (qh @ kh.T)
            p = torch.where(vis, torch.exp(s_ - lse[b, h].double().reshape(-1, 1)),
                            torch.zeros_like(s_))
            ds_abs = p * (gh.abs() @ vh.abs().T + (gh.abs() * oh.abs()).sum(-1, keepdim=True))
            out[0][b, h] = scale * ds_abs @ kh.abs()
            out[1][b, h] = scale * ds_abs.T @ qh.abs()
            out[2][b, h] = p.T @ gh.abs()
    return out


def _grad_check(got, ref, a_scale, what):
    r = grad_compare(got, ref, a_scale)
    assert r["finite"], f"{what}: non-finite"
    assert r["ok"], (f"{what}: max err {r['max_err']:.3e} (x{r['max_over_bound']:.2f} of bound), "
                     f"rel {r['max_rel']:.2e}")
    return r["max_rel"]


def _run(q, k, v, g, scale, causal):
    qd, kd, vd, gd = (t.to(DEV) for t in (q, k, v, g))
    o, lse = forward(qd, kd, vd, scale=scale, causal=causal)
    dq, dk, dv = backward(qd, kd, vd, o, lse, gd, scale=scale, causal=causal)
    check_errors()
    return o.cpu(), lse.cpu(), dq, dk, dv


CASES = [(N, d, causal)
         for N in (1, 100, 128, 300, 700)
         for d in (64, 128)
         for causal in (False, True)]


@pytest.mark.parametrize("N,d,causal", CASES)
def test_backward_elementwise(N, d, causal):
    B, H = 1, 2
    q, k, v = make_qkv(B, H, N, d, seed=7000 + N + d + int(causal))
    g = make_qkv(B, H, N, d, seed=8000 + N + d + int(causal))[0]
    scale = 1.0 / math.sqrt(d)
    o, lse, dq, dk, dv = _run(q, k, v, g, scale, causal)
    ref = oracle.attention_backward_from_lse(q, k, v, o, lse, g, scale, causal)
    exact = oracle.attention_backward(q, k, v, g, scale, causal)
    A = _term_scales(q, k, v, o, lse, g, scale, causal)
    for got, r, e, a, nm in zip((dq, dk, dv), ref, exact, A, ("dQ", "dK", "dV")):
        _grad_check(got, r, a, f"{nm} N={N} d={d} causal={causal}")
        _grad_check(got, e, a, f"{nm} (exact) N={N} d={d} causal={causal}")


def test_backward_scale_zero_and_peaky():
    # scale 0: P uniform over visible keys, so dQ = dK = 0 and dV = P^T dO;
    # peaky inputs (sigma 3) exercise rows dominated by a few keys
    B, H, N, d = 1, 1, 300, 64
    q, k, v = make_qkv(B, H, N, d, seed=31, sigma_q=3.0, sigma_k=3.0)
    g = make_qkv(B, H, N, d, seed=32)[0]
    for scale, causal in ((0.0, True), (0.125, False), (0.125, True)):
        o, lse, dq, dk, dv = _run(q, k, v, g, scale, causal)
        ref = oracle.attention_backward_from_lse(q, k, v, o, lse, g, scale, causal)
        A = _term_scales(q, k, v, o, lse, g, scale, causal)
        for got, r, a, nm in zip((dq, dk, dv), ref, A, ("dQ", "dK", "dV")):
            _grad_check(got, r, a, f"{nm} scale={scale} causal={causal}")
        if scale == 0.0:
            assert dq.abs().max().item() == 0.0 and dk.abs().max().item() == 0.0


def test_backward_deterministic():
    # every gradient tile is accumulated by one CTA in a fixed order: two
    # runs give identical bits
    B, H, N, d = 1, 2, 500, 128
    q, k, v = make_qkv(B, H, N, d, seed=41)
    g = make_qkv(B, H, N, d, seed=42)[0]
    a = _run(q, k, v, g, 0.088, True)
    b = _run(q, k, v, g, 0.088, True)
    assert torch.equal(a[2], b[2]) and torch.equal(a[3], b[3]) and torch.equal(a[4], b[4])


@pytest.mark.parametrize("d", (64, 128))
@pytest.mark.parametrize("causal", (False, True))
def test_backward_many_units_per_cta(d, causal):
    # 2 x 96 heads x 3 query blocks = 576 dQ units, several per persistent
    # CTA (and ring stages reused across unit boundaries); sampled heads,
    # including the last, against the oracle
    B, H, N = 2, 96, 300
    q, k, v = make_qkv(B, H, N, d, seed=9100 + d + int(causal))
    g = make_qkv(B, H, N, d, seed=9200 + d + int(causal))[0]
    scale = 1.0 / math.sqrt(d)
    o, lse, dq, dk, dv = _run(q, k, v, g, scale, causal)
    for (b, h) in ((0, 0), (0, 57), (1, 40), (1, 95)):
        sl = (slice(b, b + 1), slice(h, h + 1))
        args = (q[sl], k[sl], v[sl], o[sl], lse[sl], g[sl], scale, causal)
        ref = oracle.attention_backward_from_lse(*args)
        A = _term_scales(*args)
        for got, r, a, nm in zip((dq, dk, dv), ref, A, ("dQ", "dK", "dV")):
            _grad_check(got[sl], r, a, f"head {(b, h)} {nm} d={d} causal={causal}")


@pytest.mark.parametrize("name,heads", [("b4h16n2048d128", ((0, 0), (3, 15))),
                                        ("b2h32n8192d128_causal", ((1, 31),)),
                                        ("b16h32n1024d64_peaky", ((0, 0), (9, 17), (15, 31)))])
def test_backward_full_size_heads(name, heads):
    # the full workload through the library; whole heads against the oracle
    w = BY_NAME[name]
    q, k, v = make_workload(w)
    g = make_qkv(w.B, w.H, w.N, w.d, seed=w.seed + 100)[0]
    o, lse, dq, dk, dv = _run(q, k, v, g, w.scale, w.causal)
    for (b, h) in heads:
        sl = (slice(b, b + 1), slice(h, h + 1))
        args = (q[sl], k[sl], v[sl], o[sl], lse[sl], g[sl], w.scale, w.causal)
        ref = oracle.attention_backward_from_lse(*args)
        A = _term_scales(*args)
        for got, r, a, nm in zip((dq, dk, dv), ref, A, ("dQ", "dK", "dV")):
            _grad_check(got[sl], r, a, f"{name} head {(b, h)} {nm}")


def test_backward_32k_causal_sampled_rows():
    # the largest workload (B=1, H=32, N=32768, d=128, causal) through the
    # library; dQ rows and dK, dV rows of two heads (tile edges, first, last)
    # against the oracle's row-by-row gradients
    w = BY_NAME["b1h32n32768d128_causal"]
    q, k, v = make_workload(w)
    g = make_qkv(w.B, w.H, w.N, w.d, seed=w.seed + 100)[0]
    o, lse, dq, dk, dv = _run(q, k, v, g, w.scale, w.causal)
    rows = (0, 1, 127, 128, 255, 4096, 16383, 16384, 32639, 32640, 32766, 32767)
    q_picks = [(0, h, i) for h in (0, 31) for i in rows]
    k_picks = q_picks
    ref = oracle.attention_backward_rows(q, k, v, o, lse, g, w.scale, w.causal, q_picks, k_picks)
    A = grad_row_term_scales(q, k, v, o, lse, g, w.scale, w.causal, q_picks, k_picks)
    idx = torch.tensor(q_picks)
    sel = lambda t: t.cpu()[idx[:, 0], idx[:, 1], idx[:, 2]]
    for got, r, a, nm in zip((dq, dk, dv), ref, A, ("dQ", "dK", "dV")):
        _grad_check(sel(got), r, a, f"32K causal sampled {nm} rows")


def test_backward_orders_with_later_work_on_the_stream():
    # fa_bwd runs its dQ walk on a second stream and joins back: work the
    # caller enqueues afterwards on the same stream sees the final dQ
    B, H, N, d = 4, 16, 2048, 128
    q, k, v = (t.to(DEV) for t in make_qkv(B, H, N, d, seed=9300))
    g = make_qkv(B, H, N, d, seed=9301)[0].to(DEV)
    o, lse = forward(q, k, v, causal=False)
    ref = backward(q, k, v, o, lse, g, causal=False)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        for _ in range(3):
            dq, dk, dv = backward(q, k, v, o, lse, g, causal=False, stream=s)
            dq.mul_(2.0)  # enqueued behind fa_bwd on the caller's stream
            dq2 = dq.clone()
    s.synchronize()
    check_errors()
    assert torch.equal(dq2, ref[0] * 2.0)
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])


def test_backward_reads_inputs_written_just_before_it():
    # O and dO are rewritten on the caller's stream right before each call;
    # the statistics kernel and the dK/dV kernel behind it (its programmatic
    # dependent) and the dQ kernel on the forked stream must all see them
    B, H, N, d = 2, 8, 1024, 128
    q, k, v = (t.to(DEV) for t in make_qkv(B, H, N, d, seed=9320))
    o0, lse = forward(q, k, v, causal=True)
    os_ = [o0 * (1.0 + 0.25 * t) for t in range(3)]
    gs = [make_qkv(B, H, N, d, seed=9321 + t)[0].to(DEV) for t in range(3)]
    refs = [backward(q, k, v, o_, lse, g, causal=True) for o_, g in zip(os_, gs)]
    torch.cuda.synchronize()
    o_buf, g_buf = torch.empty_like(o0), torch.empty_like(gs[0])
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    outs = []
    with torch.cuda.stream(s):
        for t in range(3):
            o_buf.copy_(os_[t])
            g_buf.copy_(gs[t])
            outs.append(tuple(x.clone() for x in
                              backward(q, k, v, o_buf, lse, g_buf, causal=True, stream=s)))
    s.synchronize()
    check_errors()
    for t, (got, ref) in enumerate(zip(outs, refs)):
        for a, b, nm in zip(got, ref, ("dQ", "dK", "dV")):
            assert torch.equal(a, b), f"call {t}: {nm} differs from the same inputs run alone"


def test_backward_in_a_cuda_graph():
    # the fork to the second stream and the join are captured with the rest
    B, H, N, d = 2, 8, 1000, 64
    q, k, v = (t.to(DEV) for t in make_qkv(B, H, N, d, seed=9310))
    g = make_qkv(B, H, N, d, seed=9311)[0].to(DEV)
    o, lse = forward(q, k, v, causal=True)
    from exact_attention_forward_04_gb300 import bwd_workspace_size
    ws = torch.empty(bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=DEV)
    ref = backward(q, k, v, o, lse, g, causal=True, workspace=ws)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        backward(q, k, v, o, lse, g, causal=True, workspace=ws, stream=s)  # warm-up on s
        s.synchronize()
        with torch.cuda.graph(graph, stream=s):
            out = backward(q, k, v, o, lse, g, causal=True, workspace=ws, stream=s)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    check_errors()
    for a, b in zip(out, ref):
        assert torch.equal(a, b)
