"""Float64 statement of the attention backward (gradients of O with respect to
Q, K, V).  Test infrastructure only: see the package docstring.

The FA-2 page (section "warp之间怎样减少通信" and section "训练与部署
切分与归约的反向一致性") names the training backward: dQ, dK, dV, with dK and dV
accumulated across query rows (a reduction direction the forward does not
have), and prints a gradient of the normalised output with respect to the
scores for its four-key example.  What is differentiated is the plain
definition of the forward (see ``attention.py``):

    S = scale * Q K^T (+ mask),  P = softmax_row(S),  O = P V.

For an upstream gradient dO, the chain rule through the row softmax gives

    dV = P^T dO
    dP = dO V^T
    D_i = sum_j P_ij dP_ij  (= sum_c dO_ic O_ic)
    dS = P * (dP - D)        (elementwise; row i uses D_i)
    dQ = scale * dS K
    dK = scale * dS^T Q

Masked entries have P = 0, so they receive no gradient; a row that sees no key
(bottom-right with Nq > Nk) has P = 0 and contributes nothing.
"""

from __future__ import annotations

import numpy as np

from .attention import causal_offset


def attention_backward_f64(q, k, v, do, scale, causal=False):
    """Gradients ``(dq, dk, dv)`` in float64 for ``q [..., Nq, d]``, ``k``, ``v``
    ``[..., Nk, d]`` and the upstream gradient ``do [..., Nq, d]``."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    lead = q.shape[:-2]
    qh = q.reshape((-1,) + q.shape[-2:])
    kh = k.reshape((-1,) + k.shape[-2:])
    vh = v.reshape((-1,) + v.shape[-2:])
    doh = do.reshape((-1,) + do.shape[-2:])
    nq, nk = qh.shape[1], kh.shape[1]
    off = causal_offset(causal, nq, nk)
    rows = np.arange(nq)[:, None]
    cols = np.arange(nk)[None, :]
    dq = np.zeros_like(qh)
    dk = np.zeros_like(kh)
    dv = np.zeros_like(vh)
    for g in range(qh.shape[0]):
        s = float(scale) * (qh[g] @ kh[g].T)
        if off is not None:
            s = np.where(cols > rows + off, -np.inf, s)
        m = s.max(axis=1, keepdims=True)
        seen = np.isfinite(m)
        e = np.where(seen, np.exp(s - np.where(seen, m, 0.0)), 0.0)
        l = e.sum(axis=1, keepdims=True)
        p = np.where(l > 0, e / np.where(l > 0, l, 1.0), 0.0)
        dv[g] = p.T @ doh[g]
        dp = doh[g] @ vh[g].T
        dd = (p * dp).sum(axis=1, keepdims=True)
        ds = p * (dp - dd)
        dq[g] = float(scale) * (ds @ kh[g])
        dk[g] = float(scale) * (ds.T @ qh[g])
    return (dq.reshape(lead + qh.shape[1:]), dk.reshape(lead + kh.shape[1:]),
            dv.reshape(lead + vh.shape[1:]))
