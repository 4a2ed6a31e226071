"""Float64 statement of the FP8 (e4m3) attention forward.  Test infrastructure
only: see the package docstring.

The FA-3 page, section 7.3 "BF16 / FP8 支持", runs both GEMMs of the forward on
e4m3 inputs with fp32 accumulation, and keeps the softmax statistics (the row
max and the running sum) in fp32.  It does not change what is computed: the
result is the exact attention of the values the e4m3 inputs encode.  Here each
input tensor carries one float descale factor, so the value of code ``c`` of
tensor X is ``decode(c) * descale_X``.

The page leaves open how P reaches the second e4m3 GEMM; the reading taken is
that P is rounded to e4m3 per element (round to nearest even, saturating).
That rounding is the one step whose error is not at fp32 level, and
:func:`p_rounding_sigma` gives its size per output element so that a test can
bound it.

E4M3 is the 8-bit format of the OCP 8-bit floating point specification ("E4M3":
1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits; no infinities; only
S.1111.111 is NaN, so the largest finite magnitude is 1.75 * 2^8 = 448).
"""

from __future__ import annotations

import numpy as np

from .attention import attention_f64, causal_offset

E4M3_MAX = 448.0
# Round to nearest with 3 stored mantissa bits: relative error at most 2^-4 for
# normal numbers; spacing 2^-9 (absolute error at most 2^-10) for subnormals,
# which lie below 2^-6.
E4M3_REL_HALF_ULP = 2.0 ** -4
E4M3_MIN_NORMAL = 2.0 ** -6
E4M3_SUBNORMAL_HALF_STEP = 2.0 ** -10


def e4m3_decode(codes):
    """Value of each e4m3 code (uint8 array-like) as float64, from the bit
    fields: exponent field 0 is subnormal, m/8 * 2^-6; otherwise
    (1 + m/8) * 2^(e - 7); code 0x7F / 0xFF is NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where((c >> 7) & 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    mag = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    out = sign * mag
    return np.where((e == 15) & (m == 7), np.nan, out)


def attention_fp8_f64(q8, k8, v8, q_descale, k_descale, v_descale, scale, causal=False):
    """Exact attention of the encoded values: ``(O, LSE)`` in float64, with
    ``q = decode(q8) * q_descale`` (same for K and V) and the float32 ``scale``
    the kernel receives."""
    q = e4m3_decode(q8) * float(q_descale)
    k = e4m3_decode(k8) * float(k_descale)
    v = e4m3_decode(v8) * float(v_descale)
    return attention_f64(q, k, v, scale, causal)


def p_rounding_sigma(q8, k8, v8, q_descale, k_descale, v_descale, scale, causal=False):
    """Standard deviation, per output element, of the error that rounding P to
    e4m3 puts into O = (sum_j p_j v_j) / l when l is summed before the rounding.

    Model: p_j is rounded at a scale where the row's largest p is between 2^6
    and 2^8 (the kernel scales P into that band), so each p_j gets an
    independent error, uniform within half a step: relative 2^-4 for normal
    values, absolute 2^-10 at that scale for subnormal ones. Then
    sigma_i^2 = sum_j v_j^2 var(err p_j) / l^2. Rows without keys get 0.
    Returns an array shaped like O."""
    q = e4m3_decode(q8) * float(q_descale)
    k = e4m3_decode(k8) * float(k_descale)
    v = e4m3_decode(v8) * float(v_descale)
    qh = q.reshape((-1,) + q.shape[-2:])
    kh = k.reshape((-1,) + k.shape[-2:])
    vh = v.reshape((-1,) + v.shape[-2:])
    nq, nk = qh.shape[1], kh.shape[1]
    off = causal_offset(causal, nq, nk)
    out = np.zeros(qh.shape[:2] + (vh.shape[2],))
    rows = np.arange(nq)[:, None]
    cols = np.arange(nk)[None, :]
    for g in range(qh.shape[0]):
        s = float(scale) * (qh[g] @ kh[g].T)
        if off is not None:
            s = np.where(cols > rows + off, -np.inf, s)
        mx = s.max(axis=1, keepdims=True)
        ok = np.isfinite(mx[:, 0])
        p = np.where(np.isfinite(s), np.exp(s - np.where(np.isfinite(mx), mx, 0.0)), 0.0)
        l = p.sum(axis=1, keepdims=True)
        # At the kernel's scale the largest p sits in [2^6, 2^8]; take the
        # smallest factor, for which the most values are subnormal.
        scaled = p * 2.0 ** 6
        var = np.where(scaled >= E4M3_MIN_NORMAL,
                       (E4M3_REL_HALF_ULP * p) ** 2 / 3.0,
                       (E4M3_SUBNORMAL_HALF_STEP / 2.0 ** 6) ** 2 / 3.0)
        var = np.where(p > 0, var, 0.0)
        sig2 = (var @ (vh[g] ** 2)) / np.where(l > 0, l, 1.0) ** 2
        out[g] = np.where(ok[:, None], np.sqrt(sig2), 0.0)
    return out.reshape(q.shape[:-1] + (v.shape[-1],))
