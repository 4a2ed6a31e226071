"""Plain float64 statement of exact scaled-dot-product attention and of the
blockwise (online-softmax / split) algebra.  Test infrastructure only: see the
package docstring.

Conventions (shared with the CUDA library only by documentation, never by code):

* Tensors are ``[..., N, d]``; the leading dimensions are independent heads.
* ``scale`` is the float32 value the caller hands the GPU, upcast exactly.
* ``causal`` selects the mask: ``False``/``0`` none; ``True``/``1``/
  ``"top_left"``: key ``j`` is visible to query ``i`` iff ``j <= i``;
  ``2``/``"bottom_right"``: iff ``j <= i + (Nk - Nq)``, so the last query row
  sees every key.  (The FA-2 page, section "正确性与部署边界", leaves the
  alignment for non-square shapes to the implementation's documentation; both
  readings are offered and coincide when Nq = Nk.)
* A row that sees no key (bottom-right with Nq > Nk) has no softmax; it is
  reported as O = 0, LSE = -inf, the same convention as an empty split.
* LSE is the natural logarithm of the row's softmax denominator, in units of the
  scaled score: ``LSE_i = m_i + ln(l_i)``.
"""

from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


def _as_heads(x):
    """View ``[..., N, d]`` as ``[G, N, d]`` in float64 (exact upcast)."""
    a = np.asarray(x, dtype=np.float64)
    if a.ndim < 2:
        raise ValueError("expected at least [N, d]")
    lead = a.shape[:-2]
    return a.reshape((-1,) + a.shape[-2:]), lead


def causal_offset(causal, nq, nk):
    """Offset ``c`` of the causal mask: key ``j`` is visible to query ``i`` iff
    ``j <= i + c``; ``None`` when there is no mask (see the module docstring)."""
    if causal is None or causal is False or (not isinstance(causal, str) and causal == 0):
        return None
    if causal is True or causal == 1 or causal == "top_left":
        return 0
    if causal == 2 or causal == "bottom_right":
        return nk - nq
    raise ValueError(f"unknown causal mode {causal!r}")


def scores_f64(q, k, scale, causal, rows=None):
    """Scaled, masked score matrix S = scale * Q K^T for one head.

    FA-2 page, section 3.1: the method computes the same dense attention as the
    naive one, so S is the full dot-product matrix.  ``q`` is ``[Nq, d]``,
    ``k`` is ``[Nk, d]``; ``rows`` (optional) selects query rows by their global
    index, which also positions the causal mask (``q`` is the whole head, so
    Nq is its length).  Masked entries are -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    if rows is None:
        rows = np.arange(q.shape[0])
    rows = np.asarray(rows)
    s = float(scale) * (q[rows] @ k.T)
    off = causal_offset(causal, q.shape[0], k.shape[0])
    if off is not None:
        cols = np.arange(k.shape[0])
        s = np.where(cols[None, :] > rows[:, None] + off, NEG_INF, s)
    return s


def _softmax_rows(s, v):
    """O and LSE from a full score block (whole rows), the textbook way.

    m = max_j s_ij;  P = exp(s - m);  l = sum_j P;  O = (P V) / l;  LSE = m + ln l.
    A row with no visible key has no softmax; it is reported as O = 0,
    LSE = -inf (never produced by top-left causal attention with Nk >= 1; the
    first Nq - Nk rows under bottom-right alignment when Nq > Nk).
    """
    m = s.max(axis=1)
    empty = ~np.isfinite(m)
    m_ref = np.where(empty, 0.0, m)
    p = np.exp(s - m_ref[:, None])
    l = p.sum(axis=1)
    o = p @ v
    with np.errstate(divide="ignore", invalid="ignore"):
        o = np.where(empty[:, None], 0.0, o / l[:, None])
        lse = np.where(empty, NEG_INF, m_ref + np.log(l))
    return o, lse


def attention_f64(q, k, v, scale, causal=False, row_block=256):
    """Exact attention forward in float64.

    ``q``: ``[..., Nq, d]``, ``k``: ``[..., Nk, d]``, ``v``: ``[..., Nk, dv]``.
    Returns ``(O [..., Nq, dv], LSE [..., Nq])`` as float64.

    This is the plain definition (FA-2 page, sections 3.1 and 4.1; FA-3 page,
    section 十: the blockwise method reaches the same mathematical result).
    Rows are processed in blocks of ``row_block`` whole rows only to bound
    memory; each block sees every key, so no online rescaling is involved.
    """
    qh, lead = _as_heads(q)
    kh, _ = _as_heads(k)
    vh, _ = _as_heads(v)
    g, nq, _ = qh.shape
    dv = vh.shape[-1]
    o = np.empty((g, nq, dv))
    lse = np.empty((g, nq))
    for h in range(g):
        for r0 in range(0, nq, row_block):
            rows = np.arange(r0, min(r0 + row_block, nq))
            s = scores_f64(qh[h], kh[h], scale, causal, rows)
            o[h, rows], lse[h, rows] = _softmax_rows(s, vh[h])
    return o.reshape(lead + (nq, dv)), lse.reshape(lead + (nq,))


def attention_rows_f64(q, k, v, scale, causal, rows):
    """Exact attention for selected query rows of one head.

    ``q`` ``[Nq, d]``, ``k`` ``[Nk, d]``, ``v`` ``[Nk, dv]``; ``rows`` are global
    query indices (they position the causal mask).  Same definition as
    :func:`attention_f64`; used to check large outputs one row at a time.
    """
    s = scores_f64(q, k, scale, causal, rows)
    return _softmax_rows(s, np.asarray(v, dtype=np.float64))


def attention_varlen_f64(q, k, v, cu_q, cu_k, scale, causal=False):
    """Exact attention over a batch of variable-length sequences.

    The FA-3 page (section 7.2, cuDNN integration) names variable-length
    sequences held as ragged tensors.  Layout: the sequences are packed along
    the token axis, token-major: ``q`` ``[total_q, H, d]``, ``k`` ``[total_k, H,
    d]``, ``v`` ``[total_k, H, dv]``; sequence b owns query tokens
    ``cu_q[b] .. cu_q[b+1]-1`` and key tokens ``cu_k[b] .. cu_k[b+1]-1``.  Each
    sequence is its own attention problem (its queries see only its keys; the
    causal mask is positioned by its own lengths).  Returns ``(O [total_q, H,
    dv], LSE [H, total_q])``.  A sequence with keys but no queries contributes
    nothing; queries with no key give O = 0, LSE = -inf.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    total_q, heads = q.shape[0], q.shape[1]
    dv = v.shape[2]
    o = np.zeros((total_q, heads, dv))
    lse = np.full((heads, total_q), NEG_INF)
    for b in range(len(cu_q) - 1):
        q0, q1 = int(cu_q[b]), int(cu_q[b + 1])
        k0, k1 = int(cu_k[b]), int(cu_k[b + 1])
        if q1 <= q0 or k1 <= k0:
            continue  # no queries, or no keys (O = 0, LSE = -inf already)
        ob, lb = attention_f64(q[q0:q1].transpose(1, 0, 2), k[k0:k1].transpose(1, 0, 2),
                               v[k0:k1].transpose(1, 0, 2), scale, causal)
        o[q0:q1] = ob.transpose(1, 0, 2)
        lse[:, q0:q1] = lb
    return o, lse


def online_softmax_state_f64(s, v, edges):
    """Two-level online softmax over key blocks, as a recurrence.

    FA-3 page, section 二: for each new block x_i of scores
        m_i = max(m_{i-1}, rowmax(x_i))
        l_i = exp(m_{i-1} - m_i) * l_{i-1} + rowsum(exp(x_i - m_i))
        O_i = exp(m_{i-1} - m_i) * O_{i-1} + exp(x_i - m_i) @ V_i
    ``s`` is a scaled, masked score matrix ``[Nq, Nk]`` (-inf = masked);
    ``edges`` are increasing key offsets; block b covers keys
    ``[edges[b], edges[b+1])``.  Returns the unnormalised state ``(m, l, O)``.

    Where every score seen so far in a row is -inf, m stays -inf; the
    exponentials then use 0 as their reference so that exp(-inf - ref) = 0
    instead of NaN (the empty-block rule of the FA-2 page, section
    "接口与实现约束": an empty or fully masked block contributes nothing).
    """
    s = np.asarray(s, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    nq = s.shape[0]
    m = np.full(nq, NEG_INF)
    l = np.zeros(nq)
    o = np.zeros((nq, v.shape[1]))
    for a, b in zip(edges[:-1], edges[1:]):
        if b <= a:
            continue
        x = s[:, a:b]
        m_new = np.maximum(m, x.max(axis=1))
        ref = np.where(np.isfinite(m_new), m_new, 0.0)
        corr = np.exp(m - ref)
        p = np.exp(x - ref[:, None])
        l = corr * l + p.sum(axis=1)
        o = corr[:, None] * o + p @ v[a:b]
        m = m_new
    return m, l, o


def split_states_f64(s, v, bounds, block=None):
    """Partial states of a split along the key axis.

    FA-2 page, section "工程实操 沿键切分的归约与沿查询切分的区别", step 1: each
    key range keeps its own local (m, l, u).  ``bounds`` lists the key ranges
    ``[(a0, b0), (a1, b1), ...]``; an empty range gives m = -inf, l = 0, u = 0.
    Inside a range the recurrence of :func:`online_softmax_state_f64` runs over
    sub-blocks of ``block`` keys (the whole range when ``block`` is None).
    """
    states = []
    for a, b in bounds:
        if block is None or b <= a:
            edges = [a, b]
        else:
            edges = list(range(a, b, block)) + [b]
        states.append(online_softmax_state_f64(s, v, edges))
    return states


def merge_states_f64(states):
    """Merge split partial states into the normalised output and LSE.

    FA-2 page, same section, steps 2-3: take the global max M = max_s m_s,
    rescale each split's l and u by exp(m_s - M), sum, and divide the summed u
    by the summed l.  Returns ``(O, LSE)`` with LSE = M + ln(L).
    """
    ms = np.stack([st[0] for st in states])
    ls = np.stack([st[1] for st in states])
    us = np.stack([st[2] for st in states])
    big_m = ms.max(axis=0)
    ref = np.where(np.isfinite(big_m), big_m, 0.0)
    w = np.exp(ms - ref[None, :])
    big_l = (w * ls).sum(axis=0)
    u = (w[:, :, None] * us).sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        o = np.where(big_l[:, None] > 0, u / big_l[:, None], 0.0)
        lse = np.where(big_l > 0, ref + np.log(big_l), NEG_INF)
    return o, lse


def normalise_then_average_f64(states):
    """The WRONG merge the FA-2 page warns against (same section, step 3):
    normalise each non-empty split by its own l, then average the outputs.
    Kept only so that tests can show it differs from the correct merge.
    """
    outs = [st[2] / st[1][:, None] for st in states if np.all(st[1] > 0)]
    return np.mean(np.stack(outs), axis=0)
