"""Float64 CPU oracle for the exact attention forward pass.

Test infrastructure only: imported by the test suite, the package smoke check
and the benchmark's CPU-baseline / reference arm, never by the product path.
"""
from .attention import (  # noqa: F401
    Traffic,
    attention_backward,
    attention_backward_from_lse,
    attention_backward_rows,
    attention_bruteforce,
    attention_keyrange,
    attention_ref,
    attention_rows,
    block_softmax_stats,
    fa1_forward,
    fa2_forward,
    logsumexp_rows,
    merge_partials,
    merge_stats,
    online_softmax,
    safe_softmax_denominator,
    scores,
    softmax_weights,
    StandardTraffic,
    standard_attention,
    standard_attention_intensity,
    visible,
)
from .fp8 import (  # noqa: F401
    attention_fp8,
    dequantize_e4m3,
    e4m3_decode,
    e4m3_encode,
    quantize_e4m3,
    transpose_keys_last,
)
