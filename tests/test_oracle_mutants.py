"""Plant plausible mistakes in the oracle (on the CPU) and check that the pin
suite catches each one: a dropped scale, a transposed product, a wrong mask
direction or off-by-one, a missing log or max, a wrong sign, a dropped
normalisation, a wrong value index, a missing correction factor in the
online-softmax recurrence or the block merge, and, in the standard
three-step restatement, an uncounted read-back of S, a softmax that ignores
the mask and an intensity that counts one N x N matrix."""
import math

import pytest
import torch

import oracle
import oracle.attention as oa
from tests.oracle_pins import ALL_PINS


def _scores_noscale(q, k, scale):
    return torch.matmul(q, k.transpose(-1, -2))


def _scores_transposed(q, k, scale):
    return scale * torch.matmul(k, q.transpose(-1, -2)).transpose(-1, -2).flip(-1)


def _visible_strict(rows, n_keys, causal):
    rows = torch.as_tensor(rows, dtype=torch.long).reshape(-1, 1)
    keys = torch.arange(n_keys).reshape(1, -1)
    return (keys < rows) if causal else torch.ones(rows.shape[0], n_keys, dtype=torch.bool)


def _visible_flipped(rows, n_keys, causal):
    rows = torch.as_tensor(rows, dtype=torch.long).reshape(-1, 1)
    keys = torch.arange(n_keys).reshape(1, -1)
    return (keys >= rows) if causal else torch.ones(rows.shape[0], n_keys, dtype=torch.bool)


def _lse_nolog(s, vis):
    s = s.masked_fill(~vis, -math.inf)
    m = s.amax(-1, keepdim=True)
    return (m + torch.exp(s - m).sum(-1, keepdim=True)).squeeze(-1)


def _lse_nomax(s, vis):
    s = s.masked_fill(~vis, -math.inf)
    return torch.log(torch.exp(s).sum(-1))


def _weights_sign(s, L, vis):
    p = torch.exp(L.unsqueeze(-1) - s)
    return torch.where(vis, p, torch.zeros_like(p))


def _weights_unnormalised(s, L, vis):
    s = s.masked_fill(~vis, -math.inf)
    return torch.exp(s - s.amax(-1, keepdim=True))


def _head_rows_v_reversed(q, k, v, scale, causal, rows):
    s = oa.scores(q[rows], k, scale)
    vis = oa.visible(rows, k.shape[0], causal)
    L = oa.logsumexp_rows(s, vis)
    return torch.matmul(oa.softmax_weights(s, L, vis), v.flip(0)), L


def _online_no_correction(x):
    m, l, out = -math.inf, 0.0, []
    for xj in x:
        m = max(m, xj)
        l = l + math.exp(xj - m)
        out.append((m, l))
    return out


def _merge_no_correction(m_a, l_a, m_b, l_b):
    return max(m_a, m_b), l_a + l_b


def _merge_partials_no_max(parts):
    # weights exp(L_s) / sum exp(L_s) without the common maximum is fine in
    # exact arithmetic; the planted mistake drops the renormalisation by L
    Ls = torch.stack([l for _, l in parts])
    L = Ls.amax(dim=0)
    O = sum(torch.exp(l - L).unsqueeze(-1) * o for o, l in parts)
    return O, L


def _merge_partials_plain_sum(parts):
    Ls = torch.stack([l for _, l in parts])
    return sum(o for o, _ in parts), torch.log(torch.exp(Ls).sum(dim=0))


def _bwd_wrapper(kind):
    base = oa.attention_backward

    def fn(q, k, v, dO, scale, causal=False):
        B, H, N, _ = q.shape
        vis = oa.visible(torch.arange(N), N, causal)
        out = []
        for b in range(B):
            for h in range(H):
                qh, kh, vh, gh = (t[b, h].double() for t in (q, k, v, dO))
                s = oa.scores(qh, kh, scale)
                p = oa.softmax_weights(s, oa.logsumexp_rows(s, vis), vis)
                o = p @ vh
                D = (gh * o).sum(-1, keepdim=True)
                if kind == "no_D":
                    D = torch.zeros_like(D)
                ds = p * (gh @ vh.T - D)
                dq = (1.0 if kind == "no_scale" else scale) * ds @ kh
                dk = scale * ds.T @ qh
                dv = (p @ gh) if kind == "dv_untransposed" else p.T @ gh
                out.append((dq, dk, dv))
        stack = lambda i: torch.stack([x[i] for x in out]).reshape(B, H, N, -1)
        return stack(0), stack(1), stack(2)
    return fn


def _standard_no_readback(q, k, v, scale, causal=False, traffic=None):
    # forgets that Step 3 reads S back (counts it once)
    out = oa.StandardTraffic()
    res = _standard_orig(q, k, v, scale, causal, out)
    if traffic is not None:
        out.reads["S"] = 0
        traffic.reads, traffic.writes = out.reads, out.writes
    return res


def _standard_unmasked_p(q, k, v, scale, causal=False, traffic=None):
    # Step 3 takes the softmax over every key, ignoring the mask
    return _standard_orig(q, k, v, scale, False, traffic)


def _intensity_one_matrix(N, D, elem_bytes=2):
    # counts only one N x N matrix in the denominator
    return 4.0 * N * N * D / (4.0 * N * D * elem_bytes + N * N * elem_bytes)


_standard_orig = oa.standard_attention


def _bwd_rows_wrapper(kind):
    # the row-by-row gradients with one planted mistake
    def fn(q, k, v, O, L, dO, scale, causal, q_picks=(), k_picks=()):
        d = q.shape[-1]
        dQ = torch.empty(len(q_picks), d, dtype=torch.float64)
        dK = torch.empty(len(k_picks), d, dtype=torch.float64)
        dV = torch.empty(len(k_picks), d, dtype=torch.float64)
        for n, (b, h, i) in enumerate(q_picks):
            qi, kh, vh = q[b, h, i].double(), k[b, h].double(), v[b, h].double()
            gi, oi = dO[b, h, i].double(), O[b, h, i].double()
            p_i = torch.exp(scale * (kh @ qi) - float(L[b, h, i]))
            if causal:
                p_i[(i if kind == "q_mask_drops_diagonal" else i + 1):] = 0.0
            ds_i = p_i * (vh @ gi - torch.dot(gi, oi))
            dQ[n] = scale * (ds_i @ kh)
        for n, (b, h, j) in enumerate(k_picks):
            qh, gh, oh = q[b, h].double(), dO[b, h].double(), O[b, h].double()
            D = (gh * oh).sum(-1)
            p_j = torch.exp(scale * (qh @ k[b, h, j].double()) - L[b, h].double())
            if causal:
                p_j[:j] = 0.0
            ds_j = p_j * (gh @ v[b, h, j].double() - (0.0 if kind == "k_no_D" else D))
            dK[n] = scale * (ds_j @ qh)
            dV[n] = (ds_j if kind == "dv_from_ds" else p_j) @ gh
        return dQ, dK, dV
    return fn


MUTANTS = {
    "scores_drop_scale": ("scores", _scores_noscale),
    "scores_transposed": ("scores", _scores_transposed),
    "mask_strict": ("visible", _visible_strict),
    "mask_flipped": ("visible", _visible_flipped),
    "lse_missing_log": ("logsumexp_rows", _lse_nolog),
    "lse_missing_max": ("logsumexp_rows", _lse_nomax),
    "weights_wrong_sign": ("softmax_weights", _weights_sign),
    "weights_unnormalised": ("softmax_weights", _weights_unnormalised),
    "values_wrong_index": ("_head_rows", _head_rows_v_reversed),
    "online_no_correction": ("online_softmax", _online_no_correction),
    "merge_no_correction": ("merge_stats", _merge_no_correction),
    "merge_partials_max_only": ("merge_partials", _merge_partials_no_max),
    "merge_partials_plain_sum": ("merge_partials", _merge_partials_plain_sum),
    "backward_no_D": ("attention_backward", _bwd_wrapper("no_D")),
    "backward_dq_no_scale": ("attention_backward", _bwd_wrapper("no_scale")),
    "backward_dv_untransposed": ("attention_backward", _bwd_wrapper("dv_untransposed")),
    "backward_rows_q_mask_drops_diagonal": ("attention_backward_rows", _bwd_rows_wrapper("q_mask_drops_diagonal")),
    "backward_rows_k_no_D": ("attention_backward_rows", _bwd_rows_wrapper("k_no_D")),
    "backward_rows_dv_from_ds": ("attention_backward_rows", _bwd_rows_wrapper("dv_from_ds")),
    "standard_no_s_readback": ("standard_attention", _standard_no_readback),
    "standard_unmasked_p": ("standard_attention", _standard_unmasked_p),
    "intensity_one_matrix": ("standard_attention_intensity", _intensity_one_matrix),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, monkeypatch):
    attr, fn = MUTANTS[name]
    monkeypatch.setattr(oa, attr, fn)
    if hasattr(oracle, attr):
        monkeypatch.setattr(oracle, attr, fn)
    failed = []
    for pin in ALL_PINS:
        try:
            with torch.no_grad():
                pin(oracle)
        except Exception as e:  # AssertionError or a shape error both count
            failed.append((pin.__name__, type(e).__name__))
            break
    assert failed, f"no pin caught the planted mistake {name}"
