"""Float64 CPU oracle for the 8-bit (E4M3) forward variant.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports, calls or
executes this module: only the test suite, the package smoke check and the
benchmark's CPU-baseline / reference arm do.  It shares no code with the CUDA
library.

The pages say only that the third FlashAttention version adds FP8 support
for about twice the BF16 throughput ("How FlashAttention got past the O(N^2)
memory wall", "v2 and v3").  Which format, which operands and what scaling
are left open; the readings taken here (and by the library) are:

  * format: E4M3 as defined by the OCP 8-bit floating point specification
    (OFP8): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; no
    infinities; S.1111.111 is NaN; largest finite value 448 (S.1111.110);
    subnormals are multiples of 2^-9 below 2^-6.
  * rounding: to nearest, ties to even; a finite value beyond +-448 becomes
    +-448 (saturation to the largest finite value).
  * scaling: one scale per (batch, head) slice of each of Q, K and V.
    amax = max |x| over the slice (exact: the inputs are bf16);
    s = fp32(448 / amax) (s = 1 when amax = 0); code = E4M3(fp32(x * s));
    descale = fp32(amax / 448).  The value the attention sees is the
    dequantised x^ = E4M3 value of the code * descale, exactly.
  * the attention itself is the plain definition (``attention_ref``) applied
    to the dequantised Q^, K^, V^ in float64.  The kernel's own 8-bit
    rounding of the softmax weights P~ before the P~ V product is not part
    of this definition: the tests bound it (it is the format's rounding of
    a value in [0, 2^8]).

Parity unpinned: none.  ``tests/test_oracle_fp8.py`` pins the decoder against
the format's fixed points and a library cast of all 256 codes, the encoder
by round trips, midpoints, saturation and a library cast, the quantiser by
its amax and power-of-two invariances, and ``attention_fp8`` by its closed
forms and scale invariances.
"""
from __future__ import annotations

import numpy as np
import torch

from .attention import attention_ref

E4M3_MAX = 448.0
_SUB_STEP = 2.0 ** -9     # spacing of the subnormals
_MIN_NORMAL = 2.0 ** -6


def e4m3_decode(codes):
    """Value of each E4M3 code (uint8 array) as float64; NaN codes give NaN.

    sign = bit 7, exponent field e = bits 6..3, mantissa m = bits 2..0:
    e = 0: (-1)^sign * m * 2^-9; otherwise (-1)^sign * (1 + m/8) * 2^(e-7);
    e = 15 with m = 7 is NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m * _SUB_STEP, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    out = sign * mag
    return np.where((e == 15) & (m == 7), np.nan, out)


def e4m3_encode(y):
    """Nearest E4M3 code (ties to even) of each value of y (float array),
    saturating finite values beyond +-448 to +-448; NaN gives 0x7F (sign
    kept)."""
    y = np.asarray(y, dtype=np.float64)
    neg = np.signbit(y)
    a = np.abs(y)
    nan = np.isnan(a)
    a = np.where(nan, 0.0, np.minimum(a, E4M3_MAX))
    # subnormal range: a multiple of 2^-9, 0..8 (8 is the smallest normal)
    sub = np.rint(a / _SUB_STEP)
    # normal range: exponent E with 2^E <= a < 2^(E+1), step 2^(E-3)
    with np.errstate(divide="ignore"):
        E = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    E = np.clip(E, -6, 8)
    q = np.rint(a / np.exp2(E - 3))          # 8..16
    carry = q >= 16
    E = np.where(carry, E + 1, E)
    q = np.where(carry, 8, q)
    normal_code = (E + 7) * 8 + (q - 8)
    code = np.where(a < _MIN_NORMAL, sub, normal_code).astype(np.int64)
    code = np.minimum(code, 0x7E)            # never the NaN pattern
    code = np.where(nan, 0x7F, code)
    code = np.where(neg, code | 0x80, code)
    return code.astype(np.uint8)


def quantize_e4m3(x):
    """Per-(batch, head) scaled E4M3 codes of x ([B, H, N, d], any float
    dtype holding the values exactly in fp32, e.g. bf16).

    Returns (codes uint8 [B, H, N, d], descale float32 [B, H]).  Every step
    is the fp32 arithmetic the reading fixes: s = fp32(448 / amax),
    fp32(x * s), descale = fp32(amax / 448)."""
    xf = x.detach().to("cpu", torch.float32).numpy()
    B, H = xf.shape[:2]
    amax = np.abs(xf).reshape(B, H, -1).max(axis=-1).astype(np.float32) if xf.size else \
        np.zeros((B, H), np.float32)
    f448 = np.float32(E4M3_MAX)
    with np.errstate(divide="ignore"):
        s = np.where(amax > 0, f448 / amax, np.float32(1.0)).astype(np.float32)
    y = (xf * s[:, :, None, None]).astype(np.float32)
    codes = e4m3_encode(y)
    descale = (amax / f448).astype(np.float32)
    return torch.from_numpy(codes), torch.from_numpy(descale)


def dequantize_e4m3(codes, descale):
    """x^ = value(code) * descale in float64 ([B, H, ...] codes, [B, H])."""
    vals = e4m3_decode(codes.numpy())
    d = descale.numpy().astype(np.float64)
    d = d.reshape(d.shape + (1,) * (vals.ndim - d.ndim))
    return torch.from_numpy(vals * d)


def transpose_keys_last(codes, pitch):
    """[B, H, N, d] codes -> [B, H, d, pitch] with the keys contiguous and the
    columns N..pitch-1 zero: the layout in which the library takes V."""
    B, H, N, d = codes.shape
    out = torch.zeros(B, H, d, pitch, dtype=torch.uint8)
    out[:, :, :, :N] = codes.transpose(-1, -2)
    return out


def attention_fp8(q8, k8, v8, dq, dk, dv, scale, causal=False):
    """Exact attention in float64 of the dequantised inputs: O and L of
    softmax(scale * Q^ K^^T [+ causal]) V^ with X^ = value(x8) * descale_x.

    q8, k8, v8: uint8 codes [B, H, N, d] (V not transposed); dq, dk, dv:
    float32 descales [B, H]."""
    q = dequantize_e4m3(q8, dq)
    k = dequantize_e4m3(k8, dk)
    v = dequantize_e4m3(v8, dv)
    return attention_ref(q, k, v, scale, causal)
