"""Failure detection on the GPU without a fault: a bounded wait that runs out.

fa_selftest_wait_timeout launches one warp that waits, through the kernels'
own bounded-wait code, on a barrier nothing ever arrives at.  The wait must
give up after the given time, fill the device error record, and leave the
context usable: fa_check_errors then reports FA_ERR_TIMEOUT with the site,
clears the record, and the next forward pass is correct.
"""
import ctypes
import math
import time

import pytest

import oracle
from exact_attention_forward_04_gb300 import check_errors, forward, load_library
from exact_attention_forward_04_gb300.inputs import make_qkv
from tests.parity import assert_close

pytestmark = pytest.mark.gpu

FA_OK, FA_ERR_TIMEOUT = 0, -5
SITE = 901


def test_expired_wait_is_reported_and_context_survives():
    import torch
    lib = load_library()
    torch.cuda.synchronize()
    assert lib.fa_check_errors(None) == FA_OK  # nothing pending
    t0 = time.perf_counter()
    assert lib.fa_selftest_wait_timeout(50000, None) == FA_OK  # 50 ms
    assert lib.fa_check_errors(None) == FA_ERR_TIMEOUT
    elapsed = time.perf_counter() - t0
    assert 0.04 <= elapsed < 5.0, elapsed
    rec = (ctypes.c_uint * 4)()
    assert lib.fa_get_last_error_record(rec) == FA_OK
    assert list(rec) == [1, SITE, 0, 0]
    # the record was cleared, and the context still computes correctly
    assert lib.fa_check_errors(None) == FA_OK
    q, k, v = make_qkv(1, 2, 300, 128, seed=77)
    o, lse = forward(q.cuda(), k.cuda(), v.cuda(), causal=True)
    check_errors()
    O_ref, L_ref = oracle.attention_ref(q, k, v, 1.0 / math.sqrt(128), True)
    assert_close(o, lse, O_ref, L_ref, "forward after an expired wait")
