"""Pins for the float64 oracle: checks against what the pages and the
mathematics fix, independent of the oracle's own code.

Each ``pin_*`` takes the oracle module and raises AssertionError when the
oracle disagrees with a fixed fact.  ``tests/test_oracle_pins.py`` runs them
on the real oracle; ``tests/test_oracle_mutants.py`` plants plausible
mistakes into the oracle and checks that at least one pin fails for each.

Facts used (pages cited by title and section):
  * "Before implementing FlashAttention in Triton: FA1, 2 forward pass",
    "Online Softmax concept": the stream x = [1, 3, 2] read element by
    element or block by block ends with l equal to the safe-softmax
    denominator (fixture tests/golden/online_softmax_stream.json).
  * "FlashAttention: it was data movement, not compute, that made attention
    fast", "Softmax can be computed in pieces": scores 1, 2, 3, 4 split into
    [1, 2] | [3, 4]; naive concatenation sums to 2; the merge scales the
    first block by exp(2 - 4) (fixture tests/golden/block_merge_1234.json).
  * "Before implementing FlashAttention in Triton", FA2 section:
    exp(S_ij - L_i) = P_ij, so every row of exp(S - L) sums to 1.
  * The same page, FA1 and FA2 sections and "Summary": both loop orders give
    the whole-row softmax; the FA2 order reads Q once, K and V T_r times and
    writes O once per head, the FA1 order reads K and V once and moves Q and
    O T_c times.
  * Closed forms: one key gives O = V and L = s; causal row 0 sees only key 0;
    scale 0 gives the mean of the visible V rows and L = ln(#visible); a key
    boosted far above the others takes all the weight.
  * The same 1, 2, 3, 4 example for whole key ranges: each group's own
    logsumexp, 2 + ln(e^-1 + 1) and 4 + ln(e^-1 + 1), merges to the whole
    row's; merge of any split of the keys equals the whole row.
  * Gradients (the pages give no formulas; the backward is the exact
    derivative of the forward): autograd of the library attention, central
    finite differences, one key (P = 1: dV = dO, dQ = dK = 0), and
    invariance under a common shift of all keys (each row of dS sums to 0).
  * "How FlashAttention got past the O(N^2) memory wall", "The
    standard-attention bottleneck": the three steps write S, read it back,
    write P and read it back, N^2 elements each per head, beside Q, K, V
    and O (N d each); for N = 2048, D = 128 and 16-bit elements the
    intensity is about 117 over an 18 MB denominator, and it approaches D
    as N grows (fixture tests/golden/standard_attention_intensity.json).
  * Brute force (pure-Python fsum loops) on tiny inputs, and
    torch.nn.functional.scaled_dot_product_attention in float64 as a
    library special case.
"""
from __future__ import annotations

import json
import math
import os

import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
F64 = torch.float64


def _golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _close(a, b, tol, what):
    a = torch.as_tensor(a, dtype=F64)
    b = torch.as_tensor(b, dtype=F64)
    assert a.shape == b.shape, f"{what}: shape {tuple(a.shape)} vs {tuple(b.shape)}"
    err = (a - b).abs().max().item() if a.numel() else 0.0
    assert math.isfinite(err) and err <= tol, f"{what}: max err {err} > {tol}"


def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, dtype=F64, generator=g) * scale


def _indep_scores(q, k, scale):
    # Written out as an explicit sum over the feature index (not a matmul),
    # so it does not repeat the oracle's expression.
    return scale * (q.unsqueeze(-2) * k.unsqueeze(-3)).sum(-1)


# --------------------------------------------------------------------- pins

def pin_online_stream(o):
    g = _golden("online_softmax_stream.json")
    x = g["x"]
    states = o.online_softmax(x)
    e = math.exp
    want_l = [e(0.0), e(1 - 3) + e(0.0), e(1 - 3) + e(0.0) + e(2 - 3)]
    assert [s[0] for s in states] == g["expected"]["m_sequence"], states
    _close([s[1] for s in states], want_l, 1e-15, "online l sequence")
    m_safe, l_safe = o.safe_softmax_denominator(x)
    assert m_safe == g["expected"]["final_m"]
    _close(l_safe, want_l[-1], 1e-15, "safe-softmax denominator")
    _close(states[-1][1], l_safe, 1e-15, "online l == safe denominator")
    for split in g["block_splits"]:
        m_b, l_b = o.block_softmax_stats(x, split)
        assert m_b == 3.0
        _close(l_b, l_safe, 1e-15, f"blockwise l, splits {split}")


def pin_block_merge_1234(o):
    g = _golden("block_merge_1234.json")
    s = g["scores"]
    cut = g["split"]
    e = math.exp
    # Naive concatenation of per-block softmaxes sums to 2 (page's warning).
    naive = 0.0
    for blk in (s[:cut], s[cut:]):
        mb, lb = o.safe_softmax_denominator(blk)
        naive += sum(e(x - mb) / lb for x in blk)
    _close(naive, g["expected"]["naive_concatenated_probability_sum"], 1e-14,
           "naive concatenation")
    m1, l1 = o.safe_softmax_denominator(s[:cut])
    m2, l2 = o.safe_softmax_denominator(s[cut:])
    assert m1 == g["expected"]["first_block_max"]
    m, l = o.merge_stats(m1, l1, m2, l2)
    assert m == g["expected"]["merged_max"]
    want_l = e(2 - 4) * (e(1 - 2) + e(0)) + (e(3 - 4) + e(0))
    _close(l, want_l, 1e-15, "merged l")
    want_L = 4 + math.log(e(-3) + e(-2) + e(-1) + 1)
    # Through the attention oracle: d = 1, q = 1, keys 1..4, scale 1 gives
    # exactly the scores 1, 2, 3, 4; V = identity exposes the weights.
    q = torch.tensor([[[[1.0]]]], dtype=F64)
    k = torch.tensor(s, dtype=F64).reshape(1, 1, 4, 1)
    v = torch.eye(4, dtype=F64).reshape(1, 1, 4, 4)
    qp = torch.cat([q, torch.zeros(1, 1, 3, 1, dtype=F64)], dim=2)  # N = 4
    O, L = o.attention_ref(qp, k, v, 1.0, False)
    _close(L[0, 0, 0], want_L, 1e-14, "L of scores 1,2,3,4")
    _close(O[0, 0, 0], [e(x - want_L) for x in s], 1e-14, "weights of 1,2,3,4")
    O2, L2 = o.fa2_forward(qp, k, v, 1.0, False, Br=1, Bc=cut)
    _close(L2[0, 0, 0], want_L, 1e-14, "FA2 L with the page's split")
    _close(O2[0, 0, 0], O[0, 0, 0], 1e-14, "FA2 O with the page's split")


def pin_lse_identity(o):
    for causal in (False, True):
        q, k, v = (_rand((2, 3, 37, 16), 11 + i) for i in range(3))
        scale = 0.3
        O, L = o.attention_ref(q, k, v, scale, causal)
        S = _indep_scores(q, k, scale)
        P = torch.exp(S - L.unsqueeze(-1))
        if causal:
            P = torch.tril(P)
        _close(P.sum(-1), torch.ones_like(L), 1e-12, "rows of exp(S-L) sum to 1")
        _close(O, torch.einsum("bhik,bhkd->bhid", P, v), 1e-12, "O = exp(S-L) V")


def pin_blockwise_equals_whole(o):
    for causal in (False, True):
        for N in (1, 37, 130):
            q, k, v = (_rand((1, 2, N, 8), 100 + N + i, 1.5) for i in range(3))
            O, L = o.attention_ref(q, k, v, 0.5, causal)
            for Br, Bc in ((1, 1), (7, 7), (64, 64), (N, N), (16, 7)):
                O2, L2 = o.fa2_forward(q, k, v, 0.5, causal, Br=Br, Bc=Bc)
                _close(O2, O, 1e-12, f"FA2 O Br={Br} Bc={Bc} causal={causal}")
                _close(L2, L, 1e-12, f"FA2 L Br={Br} Bc={Bc} causal={causal}")
            for Br, Bc in ((7, 5), (64, 64)):
                O1, L1 = o.fa1_forward(q, k, v, 0.5, causal, Br=Br, Bc=Bc)
                _close(O1, O, 1e-12, f"FA1 O Br={Br} Bc={Bc} causal={causal}")
                _close(L1, L, 1e-12, f"FA1 L Br={Br} Bc={Bc} causal={causal}")


def pin_traffic_counts(o):
    N, d, Br, Bc = 96, 8, 32, 16
    q, k, v = (_rand((1, 1, N, d), 7 + i) for i in range(3))
    Tr, Tc = math.ceil(N / Br), math.ceil(N / Bc)
    t2 = o.Traffic()
    o.fa2_forward(q, k, v, 1.0, False, Br=Br, Bc=Bc, traffic=t2)
    assert t2.reads["Q"] == N * d, t2.reads
    assert t2.reads["K"] == Tr * N * d and t2.reads["V"] == Tr * N * d, t2.reads
    assert t2.reads["O"] == 0 and t2.writes["O"] == N * d, (t2.reads, t2.writes)
    t1 = o.Traffic()
    o.fa1_forward(q, k, v, 1.0, False, Br=Br, Bc=Bc, traffic=t1)
    assert t1.reads["K"] == N * d and t1.reads["V"] == N * d, t1.reads
    assert t1.reads["Q"] == Tc * N * d, t1.reads
    assert t1.reads["O"] == Tc * N * d and t1.writes["O"] == Tc * N * d


def pin_closed_forms(o):
    # One key: O = V, L = scale q.k
    q, k, v = (_rand((2, 2, 1, 5), 31 + i) for i in range(3))
    O, L = o.attention_ref(q, k, v, 0.7, False)
    _close(O, v, 1e-14, "N=1: O = V")
    _close(L, 0.7 * (q * k).sum(-1), 1e-14, "N=1: L = s")
    # Causal row 0 sees key 0 only; causal row i sees i+1 keys.
    q, k, v = (_rand((1, 1, 9, 4), 41 + i) for i in range(3))
    O, L = o.attention_ref(q, k, v, 1.3, True)
    _close(O[0, 0, 0], v[0, 0, 0], 1e-14, "causal row 0: O = V_0")
    _close(L[0, 0, 0], 1.3 * (q[0, 0, 0] * k[0, 0, 0]).sum(), 1e-14,
           "causal row 0: L = s_00")
    # Scale 0: uniform weights over the visible keys.
    for causal in (False, True):
        O, L = o.attention_ref(q, k, v, 0.0, causal)
        n = torch.arange(1, 10, dtype=F64) if causal else torch.full((9,), 9.0, dtype=F64)
        mean = torch.cumsum(v[0, 0], 0) / n.unsqueeze(1) if causal \
            else v[0, 0].mean(0).expand(9, 4)
        _close(O[0, 0], mean, 1e-14, f"scale 0: mean of visible V (causal={causal})")
        _close(L[0, 0], torch.log(n), 1e-14, f"scale 0: L = ln #visible (causal={causal})")
    # A key boosted by +1000 in score takes all the weight.
    N, d = 6, 3
    q = torch.zeros(1, 1, N, d, dtype=F64)
    q[..., 0] = 1.0
    k = _rand((1, 1, N, d), 51) * 0.1
    k[0, 0, 4, 0] = 1000.0
    v = _rand((1, 1, N, d), 52)
    O, L = o.attention_ref(q, k, v, 1.0, False)
    _close(O[0, 0], v[0, 0, 4].expand(N, d), 1e-12, "boosted key takes all weight")
    _close(L[0, 0], torch.full((N,), 1000.0, dtype=F64), 1e-9, "boosted key L")


def pin_bruteforce(o):
    for causal in (False, True):
        for (N, d) in ((1, 1), (3, 2), (5, 4), (8, 3)):
            q, k, v = (_rand((1, 1, N, d), 61 + N * 10 + d + i, 2.0) for i in range(3))
            O, L = o.attention_ref(q, k, v, 0.9, causal)
            Ob, Lb = o.attention_bruteforce(q[0, 0].tolist(), k[0, 0].tolist(),
                                            v[0, 0].tolist(), 0.9, causal)
            _close(O[0, 0], Ob, 1e-13, f"brute force O N={N} d={d} causal={causal}")
            _close(L[0, 0], Lb, 1e-13, f"brute force L N={N} d={d} causal={causal}")


def pin_library_sdpa(o):
    for causal in (False, True):
        q, k, v = (_rand((2, 3, 45, 16), 71 + i) for i in range(3))
        O, L = o.attention_ref(q, k, v, 0.25, causal)
        Ot = F.scaled_dot_product_attention(q, k, v, scale=0.25, is_causal=causal)
        S = _indep_scores(q, k, 0.25)
        if causal:
            S = S.masked_fill(torch.ones(45, 45, dtype=torch.bool).triu(1), -math.inf)
        _close(O, Ot, 1e-12, f"SDPA O causal={causal}")
        _close(L, torch.logsumexp(S, dim=-1), 1e-12, f"logsumexp L causal={causal}")


def pin_rows_subset(o):
    q, k, v = (_rand((2, 2, 50, 8), 81 + i) for i in range(3))
    for causal in (False, True):
        O, L = o.attention_ref(q, k, v, 0.4, causal)
        picks = [(0, 0, 0), (1, 1, 49), (0, 1, 17), (1, 0, 3), (0, 0, 17)]
        Or, Lr = o.attention_rows(q, k, v, 0.4, causal, picks)
        for n, (b, h, i) in enumerate(picks):
            _close(Or[n], O[b, h, i], 1e-14, f"row {(b, h, i)} O")
            _close(Lr[n], L[b, h, i], 1e-14, f"row {(b, h, i)} L")


def pin_merge_partials(o):
    """Key-range partials and their merge: the page's 1, 2, 3, 4 example in
    closed form, merge of uneven ranges = whole row (with ranges some causal
    rows cannot see), and the two-equal-halves closed form."""
    e = math.exp
    g = _golden("block_merge_1234.json")
    s = g["scores"]
    cut = g["split"]
    q = torch.tensor([[[[1.0]]]], dtype=F64)
    qp = torch.cat([q, torch.zeros(1, 1, 3, 1, dtype=F64)], dim=2)  # N = 4
    k = torch.tensor(s, dtype=F64).reshape(1, 1, 4, 1)
    v = torch.eye(4, dtype=F64).reshape(1, 1, 4, 4)
    parts = [o.attention_keyrange(qp, k, v, 1.0, False, 0, cut),
             o.attention_keyrange(qp, k, v, 1.0, False, cut, 4)]
    # each group on its own: L_1 = 2 + ln(e^-1 + 1), L_2 = 4 + ln(e^-1 + 1)
    _close(parts[0][1][0, 0, 0], 2 + math.log(e(-1) + 1), 1e-14, "L of group [1, 2]")
    _close(parts[1][1][0, 0, 0], 4 + math.log(e(-1) + 1), 1e-14, "L of group [3, 4]")
    _close(parts[0][0][0, 0, 0], [e(1 - 2) / (e(-1) + 1), 1 / (e(-1) + 1), 0, 0], 1e-14,
           "weights of group [1, 2]")
    O, L = o.merge_partials(parts)
    want_L = 4 + math.log(e(-3) + e(-2) + e(-1) + 1)
    _close(L[0, 0, 0], want_L, 1e-14, "merged L of 1, 2, 3, 4")
    _close(O[0, 0, 0], [e(x - want_L) for x in s], 1e-14, "merged weights of 1, 2, 3, 4")
    # uneven ranges, including ones early causal rows cannot see at all
    qr, kr, vr = (_rand((2, 2, 37, 6), 301 + i) for i in range(3))
    bounds = [0, 5, 6, 19, 37]
    for causal in (False, True):
        parts = [o.attention_keyrange(qr, kr, vr, 0.7, causal, a, b)
                 for a, b in zip(bounds[:-1], bounds[1:])]
        Om, Lm = o.merge_partials(parts)
        s_all = _indep_scores(qr, kr, 0.7)
        if causal:
            vis = torch.arange(37).reshape(1, -1) <= torch.arange(37).reshape(-1, 1)
            s_all = s_all.masked_fill(~vis, -math.inf)
        Lw = torch.logsumexp(s_all, dim=-1)
        Ow = torch.einsum("bhik,bhkd->bhid", torch.softmax(s_all, dim=-1), vr)
        _close(Lm, Lw, 1e-12, f"merged L (causal={causal})")
        _close(Om, Ow, 1e-12, f"merged O (causal={causal})")
    # two halves with identical scores: L = L_half + ln 2, O = O_half
    kk = torch.cat([kr[:, :, :10], kr[:, :, :10]], dim=2)
    vv = torch.cat([vr[:, :, :10], vr[:, :, :10]], dim=2)
    a = o.attention_keyrange(qr[:, :, :20], kk, vv, 0.7, False, 0, 10)
    b = o.attention_keyrange(qr[:, :, :20], kk, vv, 0.7, False, 10, 20)
    Om, Lm = o.merge_partials([a, b])
    _close(Lm, a[1] + math.log(2), 1e-13, "two equal halves: L")
    _close(Om, a[0], 1e-13, "two equal halves: O")


def pin_backward(o):
    """Gradients: autograd through the library's attention (float64), central
    finite differences of sum(dO * O) (independent of any autograd), the
    one-key closed form, the common key shift invariance, and the
    from-L restatement."""
    for causal in (False, True):
        q, k, v, g = (_rand((2, 2, 13, 5), 401 + i + 10 * int(causal)) for i in range(4))
        dQ, dK, dV = o.attention_backward(q, k, v, g, 0.45, causal)
        qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
        out = F.scaled_dot_product_attention(qa, ka, va, is_causal=causal, scale=0.45)
        out.backward(g)
        _close(dQ, qa.grad, 1e-12, f"dQ vs autograd (causal={causal})")
        _close(dK, ka.grad, 1e-12, f"dK vs autograd (causal={causal})")
        _close(dV, va.grad, 1e-12, f"dV vs autograd (causal={causal})")
        # from the stored O and L: the same gradients
        O, L = o.attention_ref(q, k, v, 0.45, causal)
        g2 = o.attention_backward_from_lse(q, k, v, O, L, g, 0.45, causal)
        for a, b, nm in zip(g2, (dQ, dK, dV), ("dQ", "dK", "dV")):
            _close(a, b, 1e-12, f"{nm} from L (causal={causal})")

    # central finite differences of f = sum(g * O), a few coordinates each
    q, k, v, g = (_rand((1, 1, 6, 3), 451 + i) for i in range(4))
    dQ, dK, dV = o.attention_backward(q, k, v, g, 0.8, True)

    def f(qq, kk, vv):
        s_ = _indep_scores(qq, kk, 0.8)
        vis = torch.arange(6).reshape(1, -1) <= torch.arange(6).reshape(-1, 1)
        pr = torch.softmax(s_.masked_fill(~vis, -math.inf), dim=-1)
        return (g * torch.einsum("bhik,bhkd->bhid", pr, vv)).sum().item()

    h = 1e-6
    for (which, grad) in ((0, dQ), (1, dK), (2, dV)):
        for (i, t) in ((0, 0), (3, 1), (5, 2), (2, 0)):
            args_p = [q.clone(), k.clone(), v.clone()]
            args_m = [q.clone(), k.clone(), v.clone()]
            args_p[which][0, 0, i, t] += h
            args_m[which][0, 0, i, t] -= h
            fd = (f(*args_p) - f(*args_m)) / (2 * h)
            _close(grad[0, 0, i, t], fd, 1e-7, f"finite difference, tensor {which} ({i},{t})")

    # one key: P = 1, so dV = dO and dQ = dK = 0
    q, k, v, g = (_rand((1, 2, 1, 4), 471 + i) for i in range(4))
    dQ, dK, dV = o.attention_backward(q, k, v, g, 0.3, False)
    _close(dV, g, 1e-15, "one key: dV = dO")
    _close(dQ, torch.zeros_like(dQ), 1e-15, "one key: dQ = 0")
    _close(dK, torch.zeros_like(dK), 1e-15, "one key: dK = 0")

    # every row of dS sums to 0: adding one vector to all keys (P unchanged)
    # leaves dQ, dK and dV unchanged
    q, k, v, g = (_rand((1, 1, 9, 4), 481 + i) for i in range(4))
    shift = _rand((4,), 489)
    a = o.attention_backward(q, k, v, g, 0.6, True)
    b = o.attention_backward(q, k + shift, v, g, 0.6, True)
    for x, y, nm in zip(a, b, ("dQ", "dK", "dV")):
        _close(x, y, 1e-12, f"common key shift: {nm}")


def pin_backward_rows(o):
    """The row-by-row gradients equal autograd through the library's
    attention (float64) on every picked row, with O and L from the oracle's
    forward and from a perturbed copy of them (the rows must use the stored
    O and L as given, like the from-L restatement)."""
    for causal in (False, True):
        q, k, v, g = (_rand((2, 2, 21, 6), 501 + i + 10 * int(causal)) for i in range(4))
        qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
        out = F.scaled_dot_product_attention(qa, ka, va, is_causal=causal, scale=0.35)
        out.backward(g)
        O, L = o.attention_ref(q, k, v, 0.35, causal)
        qp = [(0, 0, 0), (1, 1, 20), (0, 1, 7), (1, 0, 13)]
        kp = [(0, 0, 0), (1, 1, 20), (1, 1, 3), (0, 1, 11)]
        dQ, dK, dV = o.attention_backward_rows(q, k, v, O, L, g, 0.35, causal, qp, kp)
        for n, (b, h, i) in enumerate(qp):
            _close(dQ[n], qa.grad[b, h, i], 1e-12, f"dQ row {(b, h, i)} (causal={causal})")
        for n, (b, h, j) in enumerate(kp):
            _close(dK[n], ka.grad[b, h, j], 1e-12, f"dK row {(b, h, j)} (causal={causal})")
            _close(dV[n], va.grad[b, h, j], 1e-12, f"dV row {(b, h, j)} (causal={causal})")
        # stored O and L perturbed: the rows follow them as the whole-head
        # restatement does
        O2, L2 = O + 0.01 * _rand(O.shape, 531), L + 0.02 * _rand(L.shape, 532)
        full = o.attention_backward_from_lse(q, k, v, O2, L2, g, 0.35, causal)
        dQ, dK, dV = o.attention_backward_rows(q, k, v, O2, L2, g, 0.35, causal, qp, kp)
        for n, (b, h, i) in enumerate(qp):
            _close(dQ[n], full[0][b, h, i], 1e-12, f"dQ row from stored O, L {(b, h, i)}")
        for n, (b, h, j) in enumerate(kp):
            _close(dK[n], full[1][b, h, j], 1e-12, f"dK row from stored O, L {(b, h, j)}")
            _close(dV[n], full[2][b, h, j], 1e-12, f"dV row from stored O, L {(b, h, j)}")


def pin_standard_attention(o):
    # the three steps give the whole-row softmax: brute force on tiny inputs
    for causal in (False, True):
        q, k, v = (_rand((1, 1, 5, 3), 601 + i + 10 * causal) for i in range(3))
        O, L, S, P = o.standard_attention(q, k, v, 0.8, causal)
        qs, ks, vs = (t[0, 0].tolist() for t in (q, k, v))
        Ob, Lb = o.attention_bruteforce(qs, ks, vs, 0.8, causal)
        _close(O[0, 0], torch.tensor(Ob, dtype=F64), 1e-13, f"standard O vs brute force ({causal})")
        _close(L[0, 0], torch.tensor(Lb, dtype=F64), 1e-13, f"standard L vs brute force ({causal})")
    # S as Step 2 writes it, P as Step 3 writes it: rows of P sum to 1, P is
    # 0 at masked keys, and P = exp(S - L)
    q, k, v = (_rand((2, 2, 37, 8), 611 + i, 1.5) for i in range(3))
    for causal in (False, True):
        O, L, S, P = o.standard_attention(q, k, v, 0.5, causal)
        _close(S, _indep_scores(q, k, 0.5), 1e-12, "standard S")
        _close(P.sum(-1), torch.ones_like(L), 1e-12, "rows of P sum to 1")
        if causal:
            upper = torch.triu(torch.ones(37, 37, dtype=torch.bool), 1)
            assert bool((P[..., upper] == 0).all()), "P nonzero at a masked key"
        vis_s = S.masked_fill(torch.triu(torch.ones(37, 37, dtype=torch.bool), 1), -math.inf) \
            if causal else S
        _close(P, torch.exp(vis_s - L.unsqueeze(-1)), 1e-12, "P = exp(S - L)")
    # element transfers of Steps 1-4, per head: Q, K, V read once, S and P
    # written once and read once (N^2 each), O written once
    B, H, N, d = 2, 3, 24, 5
    q, k, v = (_rand((B, H, N, d), 621 + i) for i in range(3))
    t = o.StandardTraffic()
    o.standard_attention(q, k, v, 1.0, False, traffic=t)
    heads = B * H
    assert t.reads == {"Q": heads * N * d, "K": heads * N * d, "V": heads * N * d,
                       "S": heads * N * N, "P": heads * N * N}, t.reads
    assert t.writes == {"S": heads * N * N, "P": heads * N * N, "O": heads * N * d}, t.writes


def pin_standard_intensity(o):
    g = _golden("standard_attention_intensity.json")
    N, D, b = g["N"], g["D"], g["elem_bytes"]
    ai = o.standard_attention_intensity(N, D, b)
    # the page's denominator: 18 MB, exactly 18 MiB for these sizes
    denom = 4.0 * N * N * D / ai
    assert abs(denom - g["page_denominator_megabytes"] * 2 ** 20) < 1e-3, denom
    assert abs(ai - g["page_intensity_approx"]) / g["page_intensity_approx"] < 0.05, ai
    assert ai < g["page_a100_ridge_approx"], ai
    # approaches D as N grows (16-bit elements)
    big = o.standard_attention_intensity(1 << 24, D, 2)
    assert abs(big - D) / D < 1e-4, big


ALL_PINS = [
    pin_online_stream,
    pin_block_merge_1234,
    pin_lse_identity,
    pin_blockwise_equals_whole,
    pin_traffic_counts,
    pin_closed_forms,
    pin_bruteforce,
    pin_library_sdpa,
    pin_rows_subset,
    pin_merge_partials,
    pin_backward,
    pin_backward_rows,
    pin_standard_attention,
    pin_standard_intensity,
]
