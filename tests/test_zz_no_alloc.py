"""fa_fwd_splitkv_noalloc: the split key/value forward with its partials in
the library's fixed device scratch instead of a caller workspace.

Collected last (file name) so that its use of the shared scratch follows
every other GPU test."""
import ctypes
import math
import os
import re

import pytest
import torch

import oracle
from exact_attention_forward_04_gb300 import (check_errors, forward_splitkv,
                                              forward_splitkv_noalloc, load_library)
from exact_attention_forward_04_gb300.inputs import make_qkv
from tests.parity import assert_close

pytestmark = pytest.mark.gpu

DEV = "cuda"
UNSUPPORTED = -2
SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "exact_attention_forward_04_gb300", "csrc", "fa_fwd.cu")


@pytest.mark.parametrize("d", (64, 128))
@pytest.mark.parametrize("causal", (False, True))
def test_noalloc_matches_oracle_and_workspace_path(d, causal):
    B, H, N, splits = 1, 2, 1100, 3
    q, k, v = make_qkv(B, H, N, d, seed=4242 + d + int(causal))
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    o, lse = forward_splitkv_noalloc(qd, kd, vd, scale=scale, causal=causal, num_splits=splits)
    o2, lse2 = forward_splitkv(qd, kd, vd, scale=scale, causal=causal, num_splits=splits)
    check_errors()
    O_ref, L_ref = oracle.attention_ref(q, k, v, scale, causal)
    assert_close(o, lse, O_ref, L_ref, f"noalloc d={d} causal={causal}")
    # same kernels, same split: identical to the workspace entry point
    assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_noalloc_auto_split():
    B, H, N, d = 1, 1, 2100, 128
    q, k, v = make_qkv(B, H, N, d, seed=99)
    scale = 1.0 / math.sqrt(d)
    o, lse = forward_splitkv_noalloc(q.to(DEV), k.to(DEV), v.to(DEV), scale=scale, causal=False)
    check_errors()
    O_ref, L_ref = oracle.attention_ref(q, k, v, scale, False)
    assert_close(o, lse, O_ref, L_ref, "noalloc auto split")


def test_noalloc_rejects_oversize_without_touching_memory():
    lib = load_library()
    cap = lib.fa_fwd_splitkv_noalloc_capacity()
    assert cap == 64 << 20
    # B=1, H=32, N=8192, d=128, 2 splits: 2 * 262144 rows * 129 * 4 bytes > cap;
    # rejected after validation and before anything runs, so the aligned fake
    # addresses are never dereferenced
    Q, K, V, O, L = (0x10000000 * (i + 1) for i in range(5))
    assert lib.fa_fwd_splitkv_workspace_size(1, 32, 8192, 128, 2) > cap
    st = lib.fa_fwd_splitkv_noalloc(Q, K, V, O, L, 1, 32, 8192, 128, 0.088, 0, 2, None)
    assert st == UNSUPPORTED


def test_noalloc_split_count_above_key_tiles_is_lowered():
    # N = 300 has two 256-key tiles: 8 requested splits run as 2.  With 64
    # heads the partials of 8 splits would not fit the scratch (79 MB) but
    # those of 2 do; results equal the workspace path's with 2 splits.
    B, H, N, d = 1, 64, 300, 128
    lib = load_library()
    assert lib.fa_fwd_splitkv_workspace_size(B, H, N, d, 8) > lib.fa_fwd_splitkv_noalloc_capacity()
    q, k, v = make_qkv(B, H, N, d, seed=4300)
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    scale = 1.0 / math.sqrt(d)
    for causal in (False, True):
        o, lse = forward_splitkv_noalloc(qd, kd, vd, scale=scale, causal=causal, num_splits=8)
        o2, lse2 = forward_splitkv(qd, kd, vd, scale=scale, causal=causal, num_splits=2)
        check_errors()
        assert torch.equal(o, o2) and torch.equal(lse, lse2)
        sl = (slice(0, 1), slice(0, 4))
        O_ref, L_ref = oracle.attention_ref(q[sl], k[sl], v[sl], scale, causal)
        assert_close(o.cpu()[sl], lse.cpu()[sl], O_ref, L_ref, f"lowered split causal={causal}")


def test_noalloc_two_calls_in_a_row_match_workspace_path():
    # the scratch keeps the previous call's partials: a second call on other
    # inputs must not see them
    B, H, N, d = 1, 2, 1500, 64
    scale = 1.0 / math.sqrt(d)
    outs = []
    for seed in (4400, 4401):
        q, k, v = (t.to(DEV) for t in make_qkv(B, H, N, d, seed=seed))
        o, lse = forward_splitkv_noalloc(q, k, v, scale=scale, causal=True, num_splits=4)
        o2, lse2 = forward_splitkv(q, k, v, scale=scale, causal=True, num_splits=4)
        check_errors()
        assert torch.equal(o, o2) and torch.equal(lse, lse2)
        outs.append(o)
    assert not torch.equal(outs[0], outs[1])


def test_noalloc_entry_point_allocates_nothing():
    src = open(SRC).read()
    body = src[src.index("int fa_fwd_splitkv_noalloc("):src.index("size_t fa_fwd_splitkv_noalloc_capacity")]
    assert not re.search(r"cudaMalloc|cudaFree|cuMemAlloc", src)
    assert "cudaGetSymbolAddress" in body
    assert re.search(r"static __device__ __align__\(256\) unsigned char g_noalloc_scratch", src)
