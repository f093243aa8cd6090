"""The split key/value forward (fa_fwd_splitkv) against the float64 oracle.

Each query tile's visible key blocks are cut into balanced ranges; every
range leaves a normalised partial (O_s, L_s) in the caller's workspace and a
second kernel merges them.  The final (O, L) is compared element by element
with the plain oracle; the partials themselves are compared with the
oracle's attention over each key range."""
import math

import pytest
import torch

import oracle
from exact_attention_forward_04_gb300 import (check_errors, forward, forward_splitkv,
                                              splitkv_num_splits, splitkv_workspace_size)
from exact_attention_forward_04_gb300.inputs import SPLITKV_WORKLOADS, make_qkv, make_workload
from tests.parity import L_TOL, O_TOL, assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda"
TILE = 256  # query rows per work unit and keys per block


def _ranges(N, causal, splits):
    """Key-block ranges [kb, ke) of each split, per 256-row query tile p:
    the documented balanced cut of the tile's visible blocks."""
    tiles = (N + TILE - 1) // TILE
    out = {}
    for p in range(tiles):
        nkv = p + 1 if causal else tiles
        ns = min(splits, nkv)
        out[p] = [(s * nkv // ns, (s + 1) * nkv // ns) for s in range(ns)]
    return out


CASES = [(N, d, causal, splits)
         for N in (300, 1100, 2100)
         for d in (64, 128)
         for causal in (False, True)
         for splits in (2, 3, 8)]


@pytest.mark.parametrize("N,d,causal,splits", CASES)
def test_splitkv_elementwise(N, d, causal, splits):
    B, H = 1, 2
    q, k, v = make_qkv(B, H, N, d, seed=500 + N + d + 3 * splits + int(causal))
    scale = 1.0 / math.sqrt(d)
    o, lse = forward_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), scale=scale, causal=causal,
                             num_splits=splits)
    check_errors()
    O_ref, L_ref = oracle.attention_ref(q, k, v, scale, causal)
    assert_close(o, lse, O_ref, L_ref, f"splitkv N={N} d={d} causal={causal} splits={splits}")


@pytest.mark.parametrize("causal", (False, True))
def test_splitkv_partials_match_oracle_key_ranges(causal):
    # read the workspace back: every (tile, split) partial against the oracle's
    # attention over exactly that key range
    B, H, N, d, splits = 1, 2, 1100, 128, 3
    q, k, v = make_qkv(B, H, N, d, seed=901 + int(causal))
    scale = 1.0 / math.sqrt(d)
    nbytes = splitkv_workspace_size(B, H, N, d, splits)
    ws = torch.full((nbytes // 4,), float("nan"), dtype=torch.float32, device=DEV)
    o, lse = forward_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), scale=scale, causal=causal,
                             num_splits=splits, workspace=ws)
    check_errors()
    part_o = ws[: splits * B * H * N * d].view(splits, B * H, N, d).double().cpu()
    part_l = ws[splits * B * H * N * d: splits * B * H * N * (d + 1)].view(splits, B * H, N)
    part_l = part_l.double().cpu()
    for p, rngs in _ranges(N, causal, splits).items():
        rows = slice(p * TILE, min(N, (p + 1) * TILE))
        for s, (kb, ke) in enumerate(rngs):
            Os, Ls = oracle.attention_keyrange(q, k, v, scale, causal, kb * TILE, min(N, ke * TILE))
            Os = Os.reshape(B * H, N, d)[:, rows]
            Ls = Ls.reshape(B * H, N)[:, rows]
            err_o = (part_o[s, :, rows] - Os).abs().max().item()
            err_l = (part_l[s, :, rows] - Ls).abs().max().item()
            # the merge is a convex combination of the partials, so each one
            # is held to the bound of the final output
            assert err_o <= O_TOL and err_l <= L_TOL, (p, s, kb, ke, err_o, err_l)


def test_splitkv_auto_and_more_splits_than_blocks():
    B, H, N, d = 1, 1, 1500, 128
    q, k, v = make_qkv(B, H, N, d, seed=77)
    scale = 1.0 / math.sqrt(d)
    O_ref, L_ref = oracle.attention_ref(q, k, v, scale, True)
    n = splitkv_num_splits(B, H, N, True)
    assert 1 <= n <= 8
    for splits in (0, 1, 64):
        o, lse = forward_splitkv(q.to(DEV), k.to(DEV), v.to(DEV), scale=scale, causal=True,
                                 num_splits=splits)
        check_errors()
        assert_close(o, lse, O_ref, L_ref, f"splits={splits}")


@pytest.mark.parametrize("w", SPLITKV_WORKLOADS, ids=[w.name for w in SPLITKV_WORKLOADS])
def test_splitkv_workloads_match_plain_path_and_oracle_rows(w):
    # the full-size workloads in the launch configuration the benchmark times
    # (the library's split choice): sampled rows against the oracle, and the
    # whole output against the one-pass kernel within the bf16 tolerance
    q, k, v = make_workload(w)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    scale = 1.0 / math.sqrt(w.d)
    o, lse = forward_splitkv(qd, kd, vd, scale=scale, causal=w.causal, num_splits=0)
    o1, lse1 = forward(qd, kd, vd, scale=scale, causal=w.causal)
    check_errors()
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    assert (o.float() - o1.float()).abs().max().item() <= 2e-2
    assert (lse - lse1).abs().max().item() <= 2e-3
    g = torch.Generator().manual_seed(w.seed)
    picks = [(0, h, i) for h in range(w.H) for i in (0, 255, 256, w.N // 2, w.N - 1)]
    picks += [(0, int(torch.randint(w.H, (1,), generator=g)), int(torch.randint(w.N, (1,), generator=g)))
              for _ in range(24)]
    O_r, L_r = oracle.attention_rows(q, k, v, scale, w.causal, picks)
    o_c, l_c = o.cpu(), lse.cpu()
    for n, (b, h, i) in enumerate(picks):
        assert_close(o_c[b, h, i], l_c[b, h, i], O_r[n], L_r[n], f"{w.name} row {(b, h, i)}")
