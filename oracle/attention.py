"""Float64 CPU oracle for the exact attention forward pass.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
executes this module: only the test suite, the package smoke check and the
benchmark's CPU-baseline / reference arm do.  It shares no code with the CUDA
library (no kernels, headers, helpers, tables or constants); the two meet only
in the seeded bf16 inputs both are handed.

What it computes is the plain definition the pages give for attention, in
float64 on the CPU:

    s_ik = scale * sum_t q_it k_kt          for visible keys k
    L_i  = max_k s_ik + ln sum_k exp(s_ik - max_k s_ik)      (logsumexp)
    O_i  = sum_k exp(s_ik - L_i) v_k

with "visible" meaning every key, or, under the causal mask, key index <=
query index.  The blockwise restatements (FA2 and FA1 loop orders) and the
element-wise online softmax are here as test-only restatements that pin the
plain definition against the pages' own algebra; they are never a model of
the kernel.

Pages restated here (cited by title and section):
  [FA12] "Before implementing FlashAttention in Triton: FA1, 2 forward pass"
         (currybab.bearblog.dev/blog/flash_attention_idea)
  [WALL] "How FlashAttention got past the O(N^2) memory wall"
         (iq-universe.github.io/iq-blog/posts/ch6-kernel)
  [MOVE] "FlashAttention: it was data movement, not compute, that made
         attention fast" (ariser.io)

Readings taken where the pages are silent or disagree:
  * scale: [FA12] writes S = Q K^T with no scale; [WALL] (tiling loop) and
    [MOVE] ("Must the N x N matrix be stored?") divide by sqrt(D).  The scale
    is an explicit argument here.
  * the log in L is the natural log ([FA12] FA2 section pairs it with exp).
  * causal: key index <= query index, square, top-left aligned; masked
    scores are -inf before the exponential.
  * initial state of the running statistics: m = -inf, l = 0, O = 0
    ([WALL] tiling loop); exp(-inf - (-inf)) is taken as 0 for a block in
    which a row sees no key.

Parity unpinned: none.  Every function is pinned by the tests in
``tests/test_oracle_pins.py`` (page examples, closed forms, brute force and a
library special case); ``standard_attention`` and
``standard_attention_intensity`` by brute force, the per-step element counts
of the page's Steps 1-4 and the page's N = 2048, D = 128 worked intensity; ``attention_keyrange`` and ``merge_partials`` by the
page's 1, 2, 3, 4 merge example and by merge-of-ranges = whole row;
``attention_backward`` and ``attention_backward_from_lse`` by autograd of a
library attention, central finite differences, the one-key closed form and
the invariance of every gradient under a common shift of all keys;
``attention_backward_rows`` by autograd of a library attention on every
picked row and by the whole-head restatement with perturbed stored O and L.
"""
from __future__ import annotations

import math

import torch

F64 = torch.float64


# ---------------------------------------------------------------------------
# Softmax statistics ([FA12] "Online Softmax concept"; [WALL] "Online Softmax:
# associativity makes tiling possible"; [MOVE] "Softmax can be computed in
# pieces")
# ---------------------------------------------------------------------------

def safe_softmax_denominator(x):
    """Three-pass safe softmax statistics: the maximum m, then
    l = sum_j exp(x_j - m) ([FA12] "Online Softmax concept", figure part 1)."""
    m = max(x)
    return m, math.fsum(math.exp(xj - m) for xj in x)


def online_softmax(x):
    """Element-wise online softmax ([FA12] "Online Softmax concept",
    recurrence for m^(j) and l^(j); same recurrence in [WALL]).

    Returns the list of states (m^(j), l^(j)) after each element."""
    m, l = -math.inf, 0.0
    states = []
    for xj in x:
        m_new = max(m, xj)
        corr = 0.0 if m == -math.inf else math.exp(m - m_new)
        l = l * corr + math.exp(xj - m_new)
        m = m_new
        states.append((m, l))
    return states


def merge_stats(m_a, l_a, m_b, l_b):
    """Merge the (max, sum) statistics of two disjoint blocks of one row:
    both sums are brought to the common maximum before they are added
    ([FA12] "Online Softmax concept", block form; [MOVE] "Softmax can be
    computed in pieces", the exp(2-4) correction of the 1,2,3,4 example)."""
    m = max(m_a, m_b)
    if m == -math.inf:
        return m, 0.0
    ca = 0.0 if m_a == -math.inf else math.exp(m_a - m)
    cb = 0.0 if m_b == -math.inf else math.exp(m_b - m)
    return m, l_a * ca + l_b * cb


def block_softmax_stats(x, splits):
    """Blockwise online softmax: per block the maximum and sum are taken at
    once, then blocks are merged left to right with ``merge_stats``
    ([FA12] "Online Softmax concept", figure part 3).  ``splits`` are the
    block boundaries, e.g. [1] splits [a, b, c] into [a] | [b, c]."""
    edges = [0] + list(splits) + [len(x)]
    m, l = -math.inf, 0.0
    for lo, hi in zip(edges[:-1], edges[1:]):
        blk = x[lo:hi]
        if not blk:
            continue
        mb, lb = safe_softmax_denominator(blk)
        m, l = merge_stats(m, l, mb, lb)
    return m, l


# ---------------------------------------------------------------------------
# The plain definition ([FA12] "Why it is needed": S = QK^T, P = softmax(S),
# O = PV and the softmax formula; [WALL] tiling loop and [MOVE] for the
# 1/sqrt(D) scale; [FA12] FA2 section for L = m + log l and
# exp(S - L) = P)
# ---------------------------------------------------------------------------

def scores(q, k, scale):
    """S = scale * Q K^T over the last two dims, float64."""
    return scale * torch.matmul(q, k.transpose(-1, -2))


def visible(rows, n_keys, causal):
    """Boolean mask [len(rows), n_keys]: True where query row ``rows[r]`` may
    see key c (all keys, or c <= row under the causal mask)."""
    rows = torch.as_tensor(rows, dtype=torch.long).reshape(-1, 1)
    keys = torch.arange(n_keys, dtype=torch.long).reshape(1, -1)
    if not causal:
        return torch.ones(rows.shape[0], n_keys, dtype=torch.bool)
    return keys <= rows


def logsumexp_rows(s, vis):
    """L_i = max_k s_ik + ln sum_k exp(s_ik - max_k s_ik) over visible keys."""
    s = s.masked_fill(~vis, -math.inf)
    m = s.amax(dim=-1, keepdim=True)
    m_safe = torch.where(torch.isfinite(m), m, torch.zeros_like(m))
    l = torch.exp(s - m_safe).sum(dim=-1, keepdim=True)
    return (m_safe + torch.log(l)).squeeze(-1)


def softmax_weights(s, L, vis):
    """P_ik = exp(s_ik - L_i) on visible keys, 0 elsewhere."""
    p = torch.exp(s - L.unsqueeze(-1))
    return torch.where(vis, p, torch.zeros_like(p))


def _head_rows(q, k, v, scale, causal, rows):
    """O and L for the query rows ``rows`` of one head (q: [N, d] f64)."""
    s = scores(q[rows], k, scale)
    vis = visible(rows, k.shape[0], causal)
    L = logsumexp_rows(s, vis)
    p = softmax_weights(s, L, vis)
    return torch.matmul(p, v), L


def attention_ref(q, k, v, scale, causal=False, rows_per_chunk=512):
    """Exact attention forward in float64.

    q, k, v: [B, H, N, d] tensors of any float dtype (upcast exactly).
    Returns (O [B, H, N, d] float64, L [B, H, N] float64).

    Each query row sees the whole key set at once (an exact per-row softmax,
    never an online one); rows are processed in chunks only to bound memory.
    """
    B, H, N, _ = q.shape
    O = torch.empty(B, H, N, v.shape[-1], dtype=F64)
    L = torch.empty(B, H, N, dtype=F64)
    for b in range(B):
        for h in range(H):
            qh = q[b, h].to(F64)
            kh = k[b, h].to(F64)
            vh = v[b, h].to(F64)
            for r0 in range(0, N, rows_per_chunk):
                rows = torch.arange(r0, min(N, r0 + rows_per_chunk))
                o, l = _head_rows(qh, kh, vh, scale, causal, rows)
                O[b, h, rows] = o
                L[b, h, rows] = l
    return O, L


def attention_keyrange(q, k, v, scale, causal, k_lo, k_hi):
    """Attention of every query row over the keys [k_lo, k_hi) alone (those
    of them the row may see), float64: returns (O_s [B, H, N, d], L_s
    [B, H, N]) with O_s normalised over that range.  A row that sees none of
    these keys gets O_s = 0 and L_s = -inf.  These are the partial results a
    split of the key axis leaves before they are merged ([MOVE] "Softmax can
    be computed in pieces": each group is first computed on its own)."""
    B, H, N, _ = q.shape
    O = torch.zeros(B, H, N, v.shape[-1], dtype=F64)
    L = torch.full((B, H, N), -math.inf, dtype=F64)
    rows = torch.arange(N)
    vis = visible(rows, k.shape[2], causal)[:, k_lo:k_hi]
    for b in range(B):
        for h in range(H):
            s = scores(q[b, h].to(F64), k[b, h, k_lo:k_hi].to(F64), scale)
            l = logsumexp_rows(s, vis)
            p = softmax_weights(s, l, vis)
            O[b, h] = torch.matmul(p, v[b, h, k_lo:k_hi].to(F64))
            L[b, h] = l
    return O, L


def merge_partials(parts):
    """Merge the partial results (O_s, L_s) of disjoint key ranges of the
    same rows into the whole-row result, by the block-merge rule of the
    online softmax ([MOVE] "Softmax can be computed in pieces": the sums of
    each group are brought to the common maximum, exp(m_s - m), before they
    are added; [FA12] "Online Softmax concept"):
        L = m + ln sum_s exp(L_s - m),   m = max_s L_s
        O = sum_s exp(L_s - L) O_s
    A part with L_s = -inf (the row saw none of its keys) weighs 0."""
    Ls = torch.stack([l for _, l in parts])            # [S, ...]
    m = Ls.amax(dim=0)
    m_safe = torch.where(torch.isfinite(m), m, torch.zeros_like(m))
    w = torch.exp(Ls - m_safe)                          # exp(-inf) = 0
    L = m_safe + torch.log(w.sum(dim=0))
    O = torch.zeros_like(parts[0][0])
    for (o, l) in parts:
        ws = torch.exp(l - L)
        ws = torch.where(torch.isfinite(l), ws, torch.zeros_like(ws))
        O = O + ws.unsqueeze(-1) * o
    return O, L


# ---------------------------------------------------------------------------
# Backward pass ([FA12] "FlashAttention 2 forward pass": L lets the backward
# recompute the normalised P from S; [WALL] "v2 and v3": the backward keeps
# only the row statistics and recomputes the blocks it needs; [MOVE] "The
# paradox that recomputing is cheaper").  The pages give no gradient
# formulas: these are the exact derivatives of the forward definition.
# ---------------------------------------------------------------------------

def attention_backward(q, k, v, dO, scale, causal=False):
    """Gradients of the attention forward, float64, for an upstream gradient
    dO of O:  P = softmax(s) on visible keys, O = P V,
        dV = P^T dO,   dP = dO V^T,   D_i = sum_t dO_it O_it,
        dS = P * (dP - D),   dQ = scale dS K,   dK = scale dS^T Q.
    Returns (dQ, dK, dV), each [B, H, N, d] float64."""
    B, H, N, _ = q.shape
    dQ = torch.empty(B, H, N, q.shape[-1], dtype=F64)
    dK = torch.empty(B, H, N, k.shape[-1], dtype=F64)
    dV = torch.empty(B, H, N, v.shape[-1], dtype=F64)
    rows = torch.arange(N)
    vis = visible(rows, N, causal)
    for b in range(B):
        for h in range(H):
            qh, kh, vh, gh = (t[b, h].to(F64) for t in (q, k, v, dO))
            s = scores(qh, kh, scale)
            p = softmax_weights(s, logsumexp_rows(s, vis), vis)
            o = torch.matmul(p, vh)
            dv = torch.matmul(p.transpose(0, 1), gh)
            dp = torch.matmul(gh, vh.transpose(0, 1))
            D = (gh * o).sum(dim=-1, keepdim=True)
            ds = p * (dp - D)
            dQ[b, h] = scale * torch.matmul(ds, kh)
            dK[b, h] = scale * torch.matmul(ds.transpose(0, 1), qh)
            dV[b, h] = dv
    return dQ, dK, dV


def attention_backward_from_lse(q, k, v, O, L, dO, scale, causal=False):
    """The same gradients computed the way the pages' backward does: P is
    recomputed from S and the stored logsumexp L alone (P = exp(s - L)), and
    D = rowsum(dO * O) uses the stored output O.  Equals attention_backward
    when O and L are the exact forward results."""
    B, H, N, _ = q.shape
    dQ = torch.empty(B, H, N, q.shape[-1], dtype=F64)
    dK = torch.empty(B, H, N, k.shape[-1], dtype=F64)
    dV = torch.empty(B, H, N, v.shape[-1], dtype=F64)
    vis = visible(torch.arange(N), N, causal)
    for b in range(B):
        for h in range(H):
            qh, kh, vh, gh, oh = (t[b, h].to(F64) for t in (q, k, v, dO, O))
            s = scores(qh, kh, scale)
            p = softmax_weights(s, L[b, h].to(F64), vis)
            D = (gh * oh).sum(dim=-1, keepdim=True)
            ds = p * (torch.matmul(gh, vh.transpose(0, 1)) - D)
            dQ[b, h] = scale * torch.matmul(ds, kh)
            dK[b, h] = scale * torch.matmul(ds.transpose(0, 1), qh)
            dV[b, h] = torch.matmul(p.transpose(0, 1), gh)
    return dQ, dK, dV


def attention_backward_rows(q, k, v, O, L, dO, scale, causal, q_picks=(), k_picks=()):
    """Selected rows of the gradients, computed as attention_backward_from_lse
    does (P = exp(s - L) from the stored L, D = rowsum(dO * O) from the
    stored O), one row at a time: dQ_i = scale sum_k dS_ik K_k for each query
    pick (b, h, i), and dK_j = scale sum_i dS_ij Q_i, dV_j = sum_i P_ij dO_i
    for each key pick (b, h, j), with dS_ij = P_ij (dO_i . V_j - D_i).  Costs
    O(N d) per row (plus D of the head's rows for key picks), for sizes where
    the whole gradient is too large for the oracle.

    Returns (dQ [len(q_picks), d], dK [len(k_picks), d], dV [len(k_picks), d])
    in float64, in the order given."""
    d = q.shape[-1]
    N = q.shape[2]
    dQ = torch.empty(len(q_picks), d, dtype=F64)
    dK = torch.empty(len(k_picks), d, dtype=F64)
    dV = torch.empty(len(k_picks), d, dtype=F64)
    for n, (b, h, i) in enumerate(q_picks):
        qi = q[b, h, i].to(F64)
        kh, vh = k[b, h].to(F64), v[b, h].to(F64)
        gi, oi = dO[b, h, i].to(F64), O[b, h, i].to(F64)
        s_i = scale * torch.matmul(kh, qi)                       # [N]
        p_i = torch.exp(s_i - float(L[b, h, i]))
        if causal:
            p_i[i + 1:] = 0.0
        ds_i = p_i * (torch.matmul(vh, gi) - torch.dot(gi, oi))
        dQ[n] = scale * torch.matmul(ds_i, kh)
    heads = {}
    for n, (b, h, j) in enumerate(k_picks):
        heads.setdefault((b, h), []).append((n, j))
    for (b, h), items in heads.items():
        qh, gh, oh = q[b, h].to(F64), dO[b, h].to(F64), O[b, h].to(F64)
        D = (gh * oh).sum(dim=-1)                                # [N]
        Lh = L[b, h].to(F64)
        for n, j in items:
            kj, vj = k[b, h, j].to(F64), v[b, h, j].to(F64)
            p_j = torch.exp(scale * torch.matmul(qh, kj) - Lh)   # [N] over queries
            if causal:
                p_j[:j] = 0.0
            ds_j = p_j * (torch.matmul(gh, vj) - D)
            dK[n] = scale * torch.matmul(ds_j, qh)
            dV[n] = torch.matmul(p_j, gh)
    del N
    return dQ, dK, dV


def attention_rows(q, k, v, scale, causal, picks):
    """O and L for selected rows only.

    picks: iterable of (b, h, i).  Returns (O [n, d] float64, L [n] float64)
    in the order given.  Used where the full output is too large for the
    oracle but single rows are cheap."""
    picks = [tuple(int(t) for t in p) for p in picks]
    groups = {}
    for n, (b, h, i) in enumerate(picks):
        groups.setdefault((b, h), []).append((n, i))
    O = torch.empty(len(picks), v.shape[-1], dtype=F64)
    L = torch.empty(len(picks), dtype=F64)
    for (b, h), items in groups.items():
        idx = [n for n, _ in items]
        rows = torch.tensor([i for _, i in items], dtype=torch.long)
        o, l = _head_rows(q[b, h].to(F64), k[b, h].to(F64), v[b, h].to(F64),
                          scale, causal, rows)
        O[idx] = o
        L[idx] = l
    return O, L


# ---------------------------------------------------------------------------
# Blockwise restatements (test-only pins of "blockwise equals whole row")
# ---------------------------------------------------------------------------

class Traffic:
    """Counts elements moved between the slow memory and the on-chip blocks
    by the blockwise restatements, per tensor, so the page's HBM-access
    estimates ([FA12] "Summary", per-head access counts) can be checked."""

    def __init__(self):
        self.reads = {"Q": 0, "K": 0, "V": 0, "O": 0}
        self.writes = {"O": 0}


def _block_visible(r0, r1, c0, c1, causal):
    return visible(torch.arange(r0, r1), c1, causal)[:, c0:c1]


def fa2_forward(q, k, v, scale, causal=False, Br=64, Bc=64, traffic=None):
    """FA2 loop order ([FA12] "FlashAttention 2 forward pass"; [WALL]
    tiling loop): outer loop over query blocks Q_i, inner loop over key/value
    blocks K_j, V_j; running maximum m, running sum l and an unnormalised
    accumulator rescaled by alpha = exp(m_old - m_new); one divide by l at
    the end and L = m + log l.  Under the causal mask, key blocks that lie
    entirely right of the query block are skipped ([WALL] "v2 and v3")."""
    B, H, N, _ = q.shape
    d = v.shape[-1]
    O = torch.empty(B, H, N, d, dtype=F64)
    L = torch.empty(B, H, N, dtype=F64)
    for b in range(B):
        for h in range(H):
            qh, kh, vh = (t[b, h].to(F64) for t in (q, k, v))
            for r0 in range(0, N, Br):
                r1 = min(N, r0 + Br)
                Qi = qh[r0:r1]
                if traffic is not None:
                    traffic.reads["Q"] += Qi.numel()
                m = torch.full((r1 - r0,), -math.inf, dtype=F64)
                l = torch.zeros(r1 - r0, dtype=F64)
                acc = torch.zeros(r1 - r0, d, dtype=F64)
                for c0 in range(0, N, Bc):
                    c1 = min(N, c0 + Bc)
                    if causal and c0 > r1 - 1:
                        break
                    Kj, Vj = kh[c0:c1], vh[c0:c1]
                    if traffic is not None:
                        traffic.reads["K"] += Kj.numel()
                        traffic.reads["V"] += Vj.numel()
                    S = scores(Qi, Kj, scale)
                    S = S.masked_fill(~_block_visible(r0, r1, c0, c1, causal),
                                      -math.inf)
                    m_new = torch.maximum(m, S.amax(dim=1))
                    m_ref = torch.where(torch.isfinite(m_new), m_new,
                                        torch.zeros_like(m_new))
                    P = torch.exp(S - m_ref.unsqueeze(1))
                    alpha = torch.where(torch.isfinite(m), torch.exp(m - m_ref),
                                        torch.zeros_like(m))
                    l = alpha * l + P.sum(dim=1)
                    acc = alpha.unsqueeze(1) * acc + torch.matmul(P, Vj)
                    m = m_new
                O[b, h, r0:r1] = acc / l.unsqueeze(1)
                L[b, h, r0:r1] = m + torch.log(l)
                if traffic is not None:
                    traffic.writes["O"] += acc.numel()
    return O, L


def fa1_forward(q, k, v, scale, causal=False, Br=64, Bc=64, traffic=None):
    """FA1 loop order ([FA12] "FlashAttention 1 forward pass"): outer loop
    over K_j, V_j, inner loop over Q_i.  O_i is kept normalised in the slow
    memory together with l_i and m_i; each block computes its own maximum
    m~, numerator P~ and sum l~, then merges with alpha = exp(m - m_new),
    beta = exp(m~ - m_new):
        l_new = alpha l + beta l~
        O_i  <- diag(l_new)^-1 (diag(l) alpha O_i + beta P~ V_j)."""
    B, H, N, _ = q.shape
    d = v.shape[-1]
    O = torch.zeros(B, H, N, d, dtype=F64)
    Lout = torch.empty(B, H, N, dtype=F64)
    for b in range(B):
        for h in range(H):
            qh, kh, vh = (t[b, h].to(F64) for t in (q, k, v))
            Oh = torch.zeros(N, d, dtype=F64)
            lh = torch.zeros(N, dtype=F64)
            mh = torch.full((N,), -math.inf, dtype=F64)
            for c0 in range(0, N, Bc):
                c1 = min(N, c0 + Bc)
                Kj, Vj = kh[c0:c1], vh[c0:c1]
                if traffic is not None:
                    traffic.reads["K"] += Kj.numel()
                    traffic.reads["V"] += Vj.numel()
                for r0 in range(0, N, Br):
                    r1 = min(N, r0 + Br)
                    if causal and c0 > r1 - 1:
                        continue
                    Qi = qh[r0:r1]
                    Oi, li, mi = Oh[r0:r1], lh[r0:r1], mh[r0:r1]
                    if traffic is not None:
                        traffic.reads["Q"] += Qi.numel()
                        traffic.reads["O"] += Oi.numel()
                    S = scores(Qi, Kj, scale)
                    S = S.masked_fill(~_block_visible(r0, r1, c0, c1, causal),
                                      -math.inf)
                    mt = S.amax(dim=1)
                    mt_ref = torch.where(torch.isfinite(mt), mt,
                                         torch.zeros_like(mt))
                    Pt = torch.exp(S - mt_ref.unsqueeze(1))
                    lt = Pt.sum(dim=1)
                    m_new = torch.maximum(mi, mt)
                    m_ref = torch.where(torch.isfinite(m_new), m_new,
                                        torch.zeros_like(m_new))
                    alpha = torch.where(torch.isfinite(mi), torch.exp(mi - m_ref),
                                        torch.zeros_like(mi))
                    beta = torch.where(torch.isfinite(mt), torch.exp(mt - m_ref),
                                       torch.zeros_like(mt))
                    l_new = alpha * li + beta * lt
                    num = (li * alpha).unsqueeze(1) * Oi \
                        + beta.unsqueeze(1) * torch.matmul(Pt, Vj)
                    safe = torch.where(l_new > 0, l_new, torch.ones_like(l_new))
                    Oh[r0:r1] = num / safe.unsqueeze(1)
                    lh[r0:r1] = l_new
                    mh[r0:r1] = m_new
                    if traffic is not None:
                        traffic.writes["O"] += Oi.numel()
            O[b, h] = Oh
            Lout[b, h] = mh + torch.log(lh)
    return O, Lout


# ---------------------------------------------------------------------------
# Brute force (pure Python, tiny inputs only)
# ---------------------------------------------------------------------------

class StandardTraffic:
    """Counts elements moved between the slow memory and the compute units by
    the standard three-step attention (``standard_attention``), per tensor:
    the traffic the pages charge to writing S and P out and reading them back
    ([WALL] "The standard-attention bottleneck: O(N^2) HBM round trips")."""

    def __init__(self):
        self.reads = {"Q": 0, "K": 0, "V": 0, "S": 0, "P": 0}
        self.writes = {"S": 0, "P": 0, "O": 0}


def standard_attention(q, k, v, scale, causal=False, traffic=None):
    """Standard (unfused) attention in the pages' steps ([WALL] "The
    standard-attention bottleneck", Steps 1-4; [FA12] "Why it is needed"):
      Step 2: S = scale Q K^T, the whole N x N matrix, written out;
      Step 3: S read back, L = logsumexp of each row over its visible keys,
              P = exp(S - L) (0 at masked keys), written out;
      Step 4: P and V read, O = P V written.
    float64; returns (O [B, H, N, d], L [B, H, N], S, P) with S and P
    [B, H, N, N] (S unmasked, as Step 2 writes it).  ``traffic`` (a
    StandardTraffic) counts every element moved, per head: Q, K and S once
    each way as the steps read and write them."""
    B, H, N, _ = q.shape
    d = v.shape[-1]
    O = torch.empty(B, H, N, d, dtype=F64)
    L = torch.empty(B, H, N, dtype=F64)
    S_all = torch.empty(B, H, N, N, dtype=F64)
    P_all = torch.empty(B, H, N, N, dtype=F64)
    vis = visible(torch.arange(N), N, causal)
    for b in range(B):
        for h in range(H):
            qh, kh, vh = (t[b, h].to(F64) for t in (q, k, v))
            S = scores(qh, kh, scale)                       # Step 2
            if traffic is not None:
                traffic.reads["Q"] += qh.numel()
                traffic.reads["K"] += kh.numel()
                traffic.writes["S"] += S.numel()
            l = logsumexp_rows(S, vis)                      # Step 3
            P = softmax_weights(S, l, vis)
            if traffic is not None:
                traffic.reads["S"] += S.numel()
                traffic.writes["P"] += P.numel()
            o = torch.matmul(P, vh)                         # Step 4
            if traffic is not None:
                traffic.reads["P"] += P.numel()
                traffic.reads["V"] += vh.numel()
                traffic.writes["O"] += o.numel()
            O[b, h], L[b, h], S_all[b, h], P_all[b, h] = o, l, S, P
    return O, L, S_all, P_all


def standard_attention_intensity(N, D, elem_bytes=2):
    """The pages' arithmetic intensity of standard attention ([WALL] "The
    standard-attention bottleneck"): the 4 N^2 D flops of S = Q K^T and
    O = P V over 4 N D elements (Q, K, V, O) plus 2 N^2 elements (the N x N
    matrices), each of ``elem_bytes`` bytes:
        AI = 4 N^2 D / (4 N D b + 2 N^2 b).
    As N grows it tends to 2 D / b, i.e. D for 16-bit elements."""
    return 4.0 * N * N * D / (4.0 * N * D * elem_bytes + 2.0 * N * N * elem_bytes)


def attention_bruteforce(q, k, v, scale, causal=False):
    """Pure-Python loops with math.fsum over nested lists [N][d] of floats.
    Returns (O as [N][d] list, L as [N] list).  For N, d of a few units."""
    N, d = len(q), len(q[0])
    O, L = [], []
    for i in range(N):
        keys = [c for c in range(len(k)) if (not causal or c <= i)]
        s = [scale * math.fsum(q[i][t] * k[c][t] for t in range(d)) for c in keys]
        mx = max(s)
        Li = mx + math.log(math.fsum(math.exp(x - mx) for x in s))
        w = [math.exp(x - Li) for x in s]
        O.append([math.fsum(w[n] * v[c][t] for n, c in enumerate(keys))
                  for t in range(len(v[0]))])
        L.append(Li)
    return O, L
