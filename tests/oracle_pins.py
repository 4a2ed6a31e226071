"""Pins for the float64 oracle: checks against values printed on the pages,
closed forms, invariants, a library routine and brute force.

Every pin is a function ``pin_xxx(orc)`` taking the oracle module (or a mutant
of it) and raising ``AssertionError`` on a mismatch.  ``tests/test_oracle.py``
runs them on the real oracle; ``tests/test_oracle_mutants.py`` runs them on
copies of the oracle with planted mistakes and expects each mutant to fail at
least one pin.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        return json.load(f)


def _printed_tol(g):
    # A value printed with n decimals is within 0.5e-n of the exact one.
    return 0.5 * 10.0 ** (-g["printed_decimals"]) + 1e-12


def _example_as_attention(g):
    """The four-key example as a one-query, d=1 attention with scale 1:
    q = [1], k_j = score_j, v_j = value_j, so s_j = q . k_j = score_j."""
    q = np.array([[1.0]])
    k = np.array(g["scores"], dtype=np.float64)[:, None]
    v = np.array(g["values"], dtype=np.float64)[:, None]
    return q, k, v


# --------------------------------------------------------------------------
# Printed values (FA-2 page, split worked example and its gradient)
# --------------------------------------------------------------------------

def pin_split_example_block_states(orc):
    g = _golden("split_example.json")
    s = np.array([g["scores"]])
    v = np.array(g["values"])[:, None]
    states = orc.split_states_f64(s, v, [tuple(b) for b in g["blocks"]])
    tol = _printed_tol(g)
    for (m, l, u), want in zip(states, g["block_states"]):
        assert abs(m[0] - want["m"]) <= tol, (m, want)
        assert abs(l[0] - want["l"]) <= tol, (l, want)
        assert abs(u[0, 0] - want["u"]) <= tol, (u, want)


def pin_split_example_merge(orc):
    g = _golden("split_example.json")
    s = np.array([g["scores"]])
    v = np.array(g["values"])[:, None]
    states = orc.split_states_f64(s, v, [tuple(b) for b in g["blocks"]])
    o, _ = orc.merge_states_f64(states)
    tol = _printed_tol(g)
    assert abs(o[0, 0] - g["merged_output"]) <= tol, o
    wrong = orc.normalise_then_average_f64(states)
    assert abs(wrong[0, 0] - g["normalise_then_average_output"]) <= tol, wrong
    assert abs(wrong[0, 0] - o[0, 0]) > 1.0


def pin_split_example_full_attention(orc):
    g = _golden("split_example.json")
    q, k, v = _example_as_attention(g)
    o, lse = orc.attention_f64(q, k, v, 1.0, causal=False)
    assert abs(o[0, 0] - g["merged_output"]) <= _printed_tol(g), o
    # The merge of the two block states must give the same LSE as the whole row.
    s = np.array([g["scores"]])
    _, lse_m = orc.merge_states_f64(
        orc.split_states_f64(s, v, [tuple(b) for b in g["blocks"]]))
    assert abs(lse[0] - lse_m[0]) <= 1e-12, (lse, lse_m)


def pin_split_example_gradient(orc):
    """Central differences of the oracle's output with respect to each score
    reproduce the printed gradient (FA-2 page, split gradient section)."""
    g = _golden("split_gradient.json")
    q, k, v = _example_as_attention(g)
    h = 1e-5
    grad = []
    for j in range(k.shape[0]):
        kp = k.copy()
        km = k.copy()
        kp[j, 0] += h
        km[j, 0] -= h
        yp = orc.attention_f64(q, kp, v, 1.0)[0][0, 0]
        ym = orc.attention_f64(q, km, v, 1.0)[0][0, 0]
        grad.append((yp - ym) / (2 * h))
    tol = _printed_tol(g) + 1e-8
    for got, want in zip(grad, g["d_output_d_scores"]):
        assert abs(got - want) <= tol, (grad, g["d_output_d_scores"])
    assert abs(sum(grad)) <= 1e-8


# --------------------------------------------------------------------------
# Split / online-softmax algebra (FA-3 page section 二; FA-2 page split section)
# --------------------------------------------------------------------------

def _tile_split_bounds(nk, block, num_splits):
    """Contiguous ranges of whole blocks, ceil(T/S) blocks per split; trailing
    splits may be empty (the empty-tail rule of the FA-2 split section)."""
    t = -(-nk // block)
    per = -(-t // num_splits)
    out = []
    for s in range(num_splits):
        a = min(s * per * block, nk)
        b = min((s + 1) * per * block, nk)
        out.append((a, max(a, b)))
    return out


def pin_split_invariance(orc):
    rng = np.random.default_rng(7)
    for nk in (1, 4, 5, 13, 64, 130):
        q = rng.standard_normal((9, 8))
        k = rng.standard_normal((nk, 8))
        v = rng.standard_normal((nk, 5))
        for causal in (False, True):
            o_ref, lse_ref = orc.attention_f64(q, k, v, 0.3, causal)
            s = orc.scores_f64(q, k, 0.3, causal)
            for block in (1, 2, 4, 16):
                for ns in (1, 2, 3, 4, 16, 64):
                    bounds = _tile_split_bounds(nk, block, ns)
                    o, lse = orc.merge_states_f64(
                        orc.split_states_f64(s, v, bounds, block=block))
                    assert np.allclose(o, o_ref, rtol=0, atol=1e-12)
                    assert np.allclose(lse, lse_ref, rtol=0, atol=1e-12)
            # Unaligned split points, including empty ranges in the middle.
            cuts = sorted(rng.integers(0, nk + 1, size=3).tolist())
            bounds = [(0, cuts[0]), (cuts[0], cuts[1]), (cuts[1], cuts[1]),
                      (cuts[1], cuts[2]), (cuts[2], nk)]
            o, lse = orc.merge_states_f64(orc.split_states_f64(s, v, bounds))
            assert np.allclose(o, o_ref, rtol=0, atol=1e-12)
            assert np.allclose(lse, lse_ref, rtol=0, atol=1e-12)


def pin_empty_split_state(orc):
    s = np.array([[0.5, 1.5, -2.0]])
    v = np.array([[1.0], [2.0], [3.0]])
    (m, l, u), = orc.split_states_f64(s, v, [(3, 3)])
    assert m[0] == -np.inf and l[0] == 0.0 and u[0, 0] == 0.0
    # A range whose scores are all masked is empty in the same way, with no NaN.
    sm = np.array([[0.5, -np.inf, -np.inf]])
    (m, l, u), = orc.split_states_f64(sm, v, [(1, 3)], block=1)
    assert m[0] == -np.inf and l[0] == 0.0 and u[0, 0] == 0.0
    o, lse = orc.merge_states_f64(orc.split_states_f64(sm, v, [(0, 1), (1, 3)]))
    assert o[0, 0] == 1.0 and lse[0] == 0.5


def pin_online_recurrence(orc):
    rng = np.random.default_rng(11)
    q = rng.standard_normal((6, 4))
    k = rng.standard_normal((23, 4))
    v = rng.standard_normal((23, 3))
    for causal in (False, True):
        s = orc.scores_f64(q, k, 0.7, causal)
        o_ref, lse_ref = orc.attention_f64(q, k, v, 0.7, causal)
        for edges in ([0, 23], [0, 1, 2, 23], [0, 5, 5, 12, 23], list(range(24))):
            m, l, u = orc.online_softmax_state_f64(s, v, edges)
            assert np.allclose(u / l[:, None], o_ref, rtol=0, atol=1e-12)
            assert np.allclose(m + np.log(l), lse_ref, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Closed forms and invariants
# --------------------------------------------------------------------------

def pin_single_key(orc):
    rng = np.random.default_rng(3)
    q = rng.standard_normal((2, 3, 5, 16))
    k = rng.standard_normal((2, 3, 1, 16))
    v = rng.standard_normal((2, 3, 1, 8))
    for causal in (False, True):
        o, lse = orc.attention_f64(q, k, v, 0.25, causal)
        assert np.allclose(o, np.broadcast_to(v, o.shape), rtol=0, atol=1e-14)
        s = 0.25 * np.einsum("bhid,bhjd->bhi", q, k)
        assert np.allclose(lse, s, rtol=0, atol=1e-13)


def pin_zero_query(orc):
    rng = np.random.default_rng(4)
    k = rng.standard_normal((1, 2, 37, 8))
    v = rng.standard_normal((1, 2, 37, 4))
    q = np.zeros((1, 2, 6, 8))
    o, lse = orc.attention_f64(q, k, v, 0.5, causal=False)
    assert np.allclose(o, v.mean(axis=2, keepdims=True).repeat(6, axis=2), atol=1e-14)
    assert np.allclose(lse, math.log(37), atol=1e-14)
    # Causal with Q = 0: row i averages the first i+1 values, LSE = ln(i+1).
    o, lse = orc.attention_f64(q, k, v, 0.5, causal=True)
    for i in range(6):
        assert np.allclose(o[:, :, i], v[:, :, : i + 1].mean(axis=2), atol=1e-14)
        assert np.allclose(lse[:, :, i], math.log(i + 1), atol=1e-14)


def pin_causal_first_row(orc):
    rng = np.random.default_rng(5)
    q = rng.standard_normal((9, 8))
    k = rng.standard_normal((12, 8))
    v = rng.standard_normal((12, 8))
    o, lse = orc.attention_f64(q, k, v, 0.4, causal=True)
    assert np.allclose(o[0], v[0], atol=1e-14)
    assert abs(lse[0] - 0.4 * float(q[0] @ k[0])) < 1e-13


def pin_rows_sum_to_one(orc):
    rng = np.random.default_rng(6)
    q = rng.standard_normal((17, 8))
    k = rng.standard_normal((29, 8))
    for causal in (False, True):
        s = orc.scores_f64(q, k, 0.9, causal)
        _, lse = orc.attention_f64(q, k, np.eye(29), 0.9, causal)
        p = np.exp(s - lse[:, None])
        assert np.allclose(p.sum(axis=1), 1.0, atol=1e-13)
        # With V = I the output is P itself.
        o, _ = orc.attention_f64(q, k, np.eye(29), 0.9, causal)
        assert np.allclose(o, p, atol=1e-13)
        if causal:
            assert np.all(np.triu(o, 1)[:, :17] == 0.0)


def pin_shift_invariance(orc):
    """S + c 1^T leaves O unchanged and moves LSE by c (follows from the FA-3
    page's recurrence: every term carries the same factor exp(c)).  Realised
    as K' = K + 1 w^T, which shifts row i by scale * q_i . w."""
    rng = np.random.default_rng(8)
    q = rng.standard_normal((10, 8))
    k = rng.standard_normal((21, 8))
    v = rng.standard_normal((21, 6))
    w = 3.0 * rng.standard_normal(8)
    for causal in (False, True):
        o1, lse1 = orc.attention_f64(q, k, v, 0.6, causal)
        o2, lse2 = orc.attention_f64(q, k + w[None, :], v, 0.6, causal)
        assert np.allclose(o1, o2, atol=1e-12)
        assert np.allclose(lse2 - lse1, 0.6 * (q @ w), atol=1e-12)


def pin_huge_scores(orc):
    """Huge scores must not overflow (FA-2 page, section 正确性与部署边界: test
    huge scores and tiny denominators separately).  Scores near 1e3 shifted by
    -1e3 give the same O and an LSE lower by exactly 1e3."""
    rng = np.random.default_rng(9)
    s_small = rng.standard_normal((4, 11))
    v = rng.standard_normal((11, 3))
    q = np.concatenate([s_small, np.ones((4, 1))], axis=1)
    k_small = np.concatenate([np.eye(11), np.zeros((11, 1))], axis=1)
    k_big = np.concatenate([np.eye(11), np.full((11, 1), 1000.0)], axis=1)
    o1, lse1 = orc.attention_f64(q, k_small, v, 1.0)
    o2, lse2 = orc.attention_f64(q, k_big, v, 1.0)
    assert np.all(np.isfinite(o2)) and np.all(np.isfinite(lse2))
    assert np.allclose(o1, o2, atol=1e-12)
    assert np.allclose(lse2 - lse1, 1000.0, atol=1e-9)
    # Tiny denominators: one key far above the rest makes l close to 1 and the
    # others' weights ~1e-40; the output is then that key's value.
    s = np.array([[0.0, -92.0, -95.0]])
    (m, l, u), = orc.split_states_f64(s, np.array([[1.0], [2.0], [3.0]]), [(0, 3)])
    assert m[0] == 0.0 and abs(l[0] - 1.0) < 1e-39
    o, _ = orc.attention_f64(np.array([[1.0]]), np.array([[0.0], [-92.0], [-95.0]]),
                             np.array([[1.0], [2.0], [3.0]]), 1.0)
    assert abs(o[0, 0] - 1.0) < 1e-38


def pin_key_permutation(orc):
    rng = np.random.default_rng(10)
    q = rng.standard_normal((7, 8))
    k = rng.standard_normal((19, 8))
    v = rng.standard_normal((19, 4))
    perm = rng.permutation(19)
    o1, lse1 = orc.attention_f64(q, k, v, 0.5)
    o2, lse2 = orc.attention_f64(q, k[perm], v[perm], 0.5)
    assert np.allclose(o1, o2, atol=1e-13) and np.allclose(lse1, lse2, atol=1e-13)


def pin_row_subset(orc):
    rng = np.random.default_rng(12)
    q = rng.standard_normal((40, 8))
    k = rng.standard_normal((33, 8))
    v = rng.standard_normal((33, 5))
    rows = np.array([0, 3, 17, 32, 39])
    for causal in (False, True):
        o, lse = orc.attention_f64(q, k, v, 0.35, causal, row_block=7)
        o_r, lse_r = orc.attention_rows_f64(q, k, v, 0.35, causal, rows)
        assert np.array_equal(o_r, o[rows]) or np.allclose(o_r, o[rows], atol=1e-14)
        assert np.allclose(lse_r, lse[rows], atol=1e-14)


# --------------------------------------------------------------------------
# Library routine and brute force
# --------------------------------------------------------------------------

def pin_torch_sdpa_float64(orc):
    """The FA-2 page (section 5.1) names torch SDPA as the error reference; its
    CPU float64 kernel is an independent implementation of the same op."""
    import torch

    rng = np.random.default_rng(13)
    for (nq, nk, d, dv) in ((33, 33, 16, 16), (20, 47, 8, 12), (47, 20, 8, 8)):
        q = rng.standard_normal((2, 3, nq, d))
        k = rng.standard_normal((2, 3, nk, d))
        v = rng.standard_normal((2, 3, nk, dv))
        modes = [False, True] + (["bottom_right"] if nq <= nk else [])
        for causal in modes:
            mask = None
            if causal is True:
                mask = torch.ones(nq, nk, dtype=torch.bool).tril()
            elif causal == "bottom_right":
                mask = torch.ones(nq, nk, dtype=torch.bool).tril(diagonal=nk - nq)
            ref = torch.nn.functional.scaled_dot_product_attention(
                torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
                attn_mask=mask, scale=0.45)
            o, _ = orc.attention_f64(q, k, v, 0.45, causal)
            assert np.allclose(o, ref.numpy(), rtol=0, atol=1e-12)
            sref = torch.from_numpy(q) @ torch.from_numpy(k).transpose(-1, -2) * 0.45
            if causal:
                sref = sref.masked_fill(~mask, float("-inf"))
            _, lse = orc.attention_f64(q, k, v, 0.45, causal)
            assert np.allclose(lse, torch.logsumexp(sref, dim=-1).numpy(), atol=1e-12)


def _brute(q, k, v, scale, causal, offset=0):
    """Per-element loops; with ``causal`` key j is visible to query i iff
    j <= i + offset.  A row with no visible key gives O = 0, LSE = -inf."""
    nq, nk = len(q), len(k)
    o, lse = [], []
    for i in range(nq):
        s = []
        for j in range(nk):
            if causal and j > i + offset:
                continue
            s.append((j, scale * math.fsum(a * b for a, b in zip(q[i], k[j]))))
        if not s:
            o.append([0.0] * len(v[0]))
            lse.append(-math.inf)
            continue
        m = max(x for _, x in s)
        e = [(j, math.exp(x - m)) for j, x in s]
        den = math.fsum(w for _, w in e)
        o.append([math.fsum(w * v[j][c] for j, w in e) / den for c in range(len(v[0]))])
        lse.append(m + math.log(den))
    return o, lse


def pin_brute_force(orc):
    rng = np.random.default_rng(14)
    for (nq, nk, d, dv) in ((1, 1, 1, 1), (3, 5, 2, 3), (8, 8, 4, 4), (6, 2, 3, 2), (5, 7, 4, 1)):
        q = rng.standard_normal((nq, d))
        k = rng.standard_normal((nk, d))
        v = rng.standard_normal((nk, dv))
        for causal in (False, True):
            o, lse = orc.attention_f64(q, k, v, 0.8, causal)
            ob, lb = _brute(q.tolist(), k.tolist(), v.tolist(), 0.8, causal)
            assert np.allclose(o, np.array(ob), rtol=0, atol=1e-14)
            assert np.allclose(lse, np.array(lb), rtol=0, atol=1e-14)


def pin_brute_force_bottom_right(orc):
    """Bottom-right alignment against per-element loops with offset Nk - Nq,
    including Nq > Nk (rows that see no key)."""
    rng = np.random.default_rng(15)
    for (nq, nk, d, dv) in ((3, 5, 2, 3), (5, 3, 2, 2), (1, 6, 3, 2), (7, 7, 2, 2), (6, 1, 2, 3)):
        q = rng.standard_normal((nq, d))
        k = rng.standard_normal((nk, d))
        v = rng.standard_normal((nk, dv))
        o, lse = orc.attention_f64(q, k, v, 0.8, "bottom_right")
        ob, lb = _brute(q.tolist(), k.tolist(), v.tolist(), 0.8, True, nk - nq)
        assert np.allclose(o, np.array(ob), rtol=0, atol=1e-14)
        lb = np.array(lb)
        assert np.array_equal(np.isinf(lse), np.isinf(lb))
        assert np.allclose(lse[np.isfinite(lb)], lb[np.isfinite(lb)], rtol=0, atol=1e-14)


def pin_bottom_right_rows(orc):
    """Closed forms of the bottom-right mask (key j visible to query i iff
    j <= i + Nk - Nq): for Nq = Nk it is the top-left mask; the last query row
    sees every key; with Nq > Nk the first Nq - Nk rows see nothing (O = 0,
    LSE = -inf) and the next one sees key 0 only (O = V_0, LSE = its score)."""
    rng = np.random.default_rng(16)
    q = rng.standard_normal((13, 6))
    k = rng.standard_normal((13, 6))
    v = rng.standard_normal((13, 4))
    a = orc.attention_f64(q, k, v, 0.5, "bottom_right")
    b = orc.attention_f64(q, k, v, 0.5, True)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    # Nq < Nk: last row = non-causal last row; first row = attention over keys 0..Nk-Nq.
    q5 = q[:5]
    o, lse = orc.attention_f64(q5, k, v, 0.5, 2)
    o_nc, lse_nc = orc.attention_f64(q5, k, v, 0.5, False)
    assert np.allclose(o[4], o_nc[4], atol=1e-15) and np.isclose(lse[4], lse_nc[4], atol=1e-15)
    o0, lse0 = orc.attention_f64(q5[:1], k[:9], v[:9], 0.5, False)
    assert np.allclose(o[0], o0[0], atol=1e-15) and np.isclose(lse[0], lse0[0], atol=1e-15)
    # Nq > Nk: rows 0..Nq-Nk-1 see nothing, row Nq-Nk sees key 0 only.
    k3, v3 = k[:3], v[:3]
    o, lse = orc.attention_f64(q[:7], k3, v3, 0.5, "bottom_right")
    assert np.array_equal(o[:4], np.zeros((4, 4))) and np.all(lse[:4] == -np.inf)
    assert np.allclose(o[4], v3[0], atol=1e-15)
    assert np.isclose(lse[4], 0.5 * float(q[4] @ k3[0]), atol=1e-15)
    o_nc, lse_nc = orc.attention_f64(q[:7], k3, v3, 0.5, False)
    assert np.allclose(o[6], o_nc[6], atol=1e-15)


def pin_varlen_equal_lengths(orc):
    """Packed sequences of equal length are a dense batch: the varlen oracle on
    token-major packing equals the batched oracle on [B, H, N, d]."""
    rng = np.random.default_rng(17)
    B, H, N, M, d = 3, 2, 9, 11, 4
    q = rng.standard_normal((B, H, N, d))
    k = rng.standard_normal((B, H, M, d))
    v = rng.standard_normal((B, H, M, 5))
    pack = lambda x: x.transpose(0, 2, 1, 3).reshape(-1, x.shape[1], x.shape[3])  # noqa: E731
    cu_q = np.arange(B + 1) * N
    cu_k = np.arange(B + 1) * M
    for causal in (False, True, "bottom_right"):
        o, lse = orc.attention_varlen_f64(pack(q), pack(k), pack(v), cu_q, cu_k, 0.6, causal)
        o_d, lse_d = orc.attention_f64(q, k, v, 0.6, causal)
        assert np.allclose(o, pack(o_d), rtol=0, atol=1e-15)
        assert np.allclose(lse, lse_d.transpose(1, 0, 2).reshape(H, -1), rtol=0, atol=1e-15)


def pin_varlen_brute_force(orc):
    """Ragged lengths (including a sequence with no query and one with no key)
    against per-element loops run sequence by sequence, head by head."""
    rng = np.random.default_rng(18)
    lq = [3, 0, 1, 5, 2]
    lk = [4, 2, 6, 3, 0]
    H, d, dv = 2, 3, 2
    cu_q = np.concatenate([[0], np.cumsum(lq)])
    cu_k = np.concatenate([[0], np.cumsum(lk)])
    q = rng.standard_normal((cu_q[-1], H, d))
    k = rng.standard_normal((cu_k[-1], H, d))
    v = rng.standard_normal((cu_k[-1], H, dv))
    for causal, off_of in ((False, None), (True, lambda a, b: 0), ("bottom_right", lambda a, b: b - a)):
        o, lse = orc.attention_varlen_f64(q, k, v, cu_q, cu_k, 0.7, causal)
        for b in range(len(lq)):
            for h in range(H):
                qs = q[cu_q[b]:cu_q[b + 1], h].tolist()
                ks = k[cu_k[b]:cu_k[b + 1], h].tolist()
                vs = v[cu_k[b]:cu_k[b + 1], h].tolist()
                if not qs:
                    continue
                if not ks:
                    assert np.all(o[cu_q[b]:cu_q[b + 1], h] == 0)
                    assert np.all(lse[h, cu_q[b]:cu_q[b + 1]] == -np.inf)
                    continue
                off = 0 if off_of is None else off_of(len(qs), len(ks))
                ob, lb = _brute(qs, ks, vs, 0.7, off_of is not None, off)
                assert np.allclose(o[cu_q[b]:cu_q[b + 1], h], np.array(ob), rtol=0, atol=1e-14)
                lb = np.array(lb)
                got = lse[h, cu_q[b]:cu_q[b + 1]]
                assert np.array_equal(np.isinf(got), np.isinf(lb))
                assert np.allclose(got[np.isfinite(lb)], lb[np.isfinite(lb)], rtol=0, atol=1e-14)


def pin_varlen_independence(orc):
    """Sequences do not see each other: changing one sequence's keys and values
    leaves every other sequence's output unchanged, bit for bit."""
    rng = np.random.default_rng(19)
    cu_q = np.array([0, 4, 9, 12])
    cu_k = np.array([0, 6, 8, 15])
    q = rng.standard_normal((12, 2, 3))
    k = rng.standard_normal((15, 2, 3))
    v = rng.standard_normal((15, 2, 4))
    o1, l1 = orc.attention_varlen_f64(q, k, v, cu_q, cu_k, 0.5, True)
    k2, v2 = k.copy(), v.copy()
    k2[6:8] += 3.0
    v2[6:8] -= 1.0
    o2, l2 = orc.attention_varlen_f64(q, k2, v2, cu_q, cu_k, 0.5, True)
    keep = np.r_[0:4, 9:12]
    assert np.array_equal(o1[keep], o2[keep]) and np.array_equal(l1[:, keep], l2[:, keep])
    assert not np.allclose(o1[4:9], o2[4:9])



# --------------------------------------------------------------------------
# FP8 (e4m3) inputs: the decoder, the attention of the encoded values, and the
# size of the error that rounding P to e4m3 adds (module ``oracle.fp8``).
# --------------------------------------------------------------------------

def pin_e4m3_hand_values(f8):
    """Codes whose values follow from the E4M3 bit fields by hand: sign,
    exponent bias 7, subnormals m/8 * 2^-6, no infinities, NaN only at
    S.1111.111 (so 0x7E = 1.75 * 2^8 = 448 is the largest finite value)."""
    want = {0x00: 0.0, 0x38: 1.0, 0x40: 2.0, 0x3C: 1.5, 0x30: 0.5, 0xB8: -1.0,
            0x7E: 448.0, 0xFE: -448.0, 0x78: 256.0, 0x77: 240.0, 0x01: 2.0 ** -9,
            0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x0F: 1.875 * 2.0 ** -6}
    got = f8.e4m3_decode(np.array(list(want), dtype=np.uint8))
    assert np.array_equal(got, np.array(list(want.values()))), got
    assert np.isnan(f8.e4m3_decode(np.array([0x7F, 0xFF], dtype=np.uint8))).all()
    assert np.signbit(f8.e4m3_decode(np.array([0x80], dtype=np.uint8))[0])


def pin_e4m3_vs_torch(f8):
    """All 256 codes against torch's float8_e4m3fn conversion (an independent
    library implementation of the same format)."""
    import torch
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = f8.e4m3_decode(codes.numpy())
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    assert np.array_equal(got[ok], ref[ok])


def _codes(rng, shape, scale):
    """e4m3 codes of N(0,1) * scale values (rounded by torch, saturating)."""
    import torch
    x = torch.from_numpy(rng.standard_normal(shape) * scale)
    return x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def pin_fp8_single_key(f8):
    """Nk = 1: O is the single value row, LSE its scaled score (exact)."""
    rng = np.random.default_rng(31)
    q8, k8, v8 = _codes(rng, (3, 1, 8), 16), _codes(rng, (3, 1, 8), 16), _codes(rng, (3, 1, 8), 16)
    o, lse = f8.attention_fp8_f64(q8, k8, v8, 0.25, 0.125, 0.5, 0.3)
    q = f8.e4m3_decode(q8) * 0.25
    k = f8.e4m3_decode(k8) * 0.125
    v = f8.e4m3_decode(v8) * 0.5
    assert np.allclose(o, v, rtol=0, atol=1e-15)
    assert np.allclose(lse[..., 0], 0.3 * (q * k).sum(-1)[..., 0], rtol=1e-14, atol=1e-14)


def pin_fp8_descales(f8):
    """The Q and K descales multiply the scores (the same as scaling ``scale``),
    and the V descale multiplies O and leaves LSE alone."""
    rng = np.random.default_rng(37)
    q8, k8, v8 = (_codes(rng, (2, 9, 16), 8) for _ in range(3))
    o1, l1 = f8.attention_fp8_f64(q8, k8, v8, 0.5, 0.25, 1.0, 0.2, True)
    o2, l2 = f8.attention_fp8_f64(q8, k8, v8, 1.0, 1.0, 1.0, 0.025, True)
    o3, l3 = f8.attention_fp8_f64(q8, k8, v8, 0.5, 0.25, 3.0, 0.2, True)
    assert np.allclose(o1, o2, rtol=1e-12, atol=1e-12) and np.allclose(l1, l2, rtol=1e-12, atol=1e-12)
    assert np.allclose(o3, 3.0 * o1, rtol=1e-12, atol=1e-12) and np.array_equal(l3, l1)


def pin_p_sigma_closed_forms(f8):
    """One key: p = 1 (normal), sigma = 2^-4/sqrt(3) |v|. Two keys with equal
    scores: p = (1, 1), l = 2, sigma = 2^-4/sqrt(3) sqrt(v1^2 + v2^2) / 2."""
    h = 2.0 ** -4 / math.sqrt(3.0)
    one = np.array([[[0x38]]], dtype=np.uint8)
    v8 = np.array([[[0x40, 0xC4]]], dtype=np.uint8)  # 2.0, -3.0
    sig = f8.p_rounding_sigma(one, one, v8, 1.0, 1.0, 1.0, 1.0)
    assert np.allclose(sig, h * np.array([[[2.0, 3.0]]]), rtol=1e-14, atol=0)
    k8 = np.array([[[0x38], [0x38]]], dtype=np.uint8)
    v8 = np.array([[[0x40], [0x44]]], dtype=np.uint8)  # 2.0, 3.0
    sig = f8.p_rounding_sigma(one, k8, v8, 1.0, 1.0, 1.0, 1.0)
    assert np.allclose(sig, h * math.sqrt(4.0 + 9.0) / 2.0, rtol=1e-14, atol=0)


def pin_p_sigma_simulated(f8):
    """Against a simulation of the model it states: independent errors uniform
    within half a step on every p_j (relative 2^-4 when p_j * 2^6 is normal,
    absolute 2^-16 below), 4000 draws; the sample standard deviation of the
    error in O agrees with sigma within 10 %."""
    rng = np.random.default_rng(41)
    q8, k8, v8 = _codes(rng, (1, 3, 8), 4), _codes(rng, (1, 40, 8), 4), _codes(rng, (1, 40, 8), 4)
    sig = f8.p_rounding_sigma(q8, k8, v8, 1.0, 1.0, 1.0, 0.35)
    q = f8.e4m3_decode(q8)[0]
    k = f8.e4m3_decode(k8)[0]
    v = f8.e4m3_decode(v8)[0]
    s = 0.35 * q @ k.T
    p = np.exp(s - s.max(axis=1, keepdims=True))
    l = p.sum(axis=1, keepdims=True)
    normal = p * 2.0 ** 6 >= 2.0 ** -6
    half = np.where(normal, 2.0 ** -4 * p, 2.0 ** -16)
    u = rng.uniform(-1.0, 1.0, size=(4000,) + p.shape)
    err = np.einsum("tqk,kd->tqd", u * half, v) / l
    assert np.allclose(err.std(axis=0), sig[0], rtol=0.1, atol=0)



# --------------------------------------------------------------------------
# Backward (module ``oracle.backward``): gradients of O with respect to Q, K, V.
# --------------------------------------------------------------------------

def pin_bwd_printed_gradient(bw, orc):
    """The FA-2 page's printed score gradient (split-gradient section): with the
    four-key example as a one-query, d = 1 attention (q = 1, k_j = score_j,
    v_j = value_j, scale 1) and dO = 1, dK_j = dO * dS_j * q is the gradient of
    the output with respect to score j."""
    g = _golden("split_gradient.json")
    q, k, v = _example_as_attention(g)
    dq, dk, dv = bw.attention_backward_f64(q, k, v, np.ones((1, 1)), 1.0)
    tol = _printed_tol(g) + 1e-8
    assert np.allclose(dk[:, 0], g["d_output_d_scores"], rtol=0, atol=tol), dk[:, 0]
    # dV_j = p_j; dQ = sum_j dS_j k_j.
    p = np.exp(np.array(g["scores"]) - max(g["scores"]))
    p /= p.sum()
    assert np.allclose(dv[:, 0], p, rtol=0, atol=1e-15)
    assert np.allclose(dq[0, 0], (dk[:, 0] * np.array(g["scores"])).sum(), rtol=0, atol=1e-14)


def _loss(orc, q, k, v, do, scale, causal):
    return float((orc.attention_f64(q, k, v, scale, causal)[0] * do).sum())


def pin_bwd_finite_differences(bw, orc):
    """Central differences of L = sum(dO * O) from the forward oracle, along
    random directions in Q, K and V, for no mask and both causal alignments."""
    rng = np.random.default_rng(43)
    for causal, nq, nk in ((False, 5, 7), (True, 6, 6), ("bottom_right", 4, 9), ("bottom_right", 7, 3)):
        q = rng.standard_normal((2, nq, 3))
        k = rng.standard_normal((2, nk, 3))
        v = rng.standard_normal((2, nk, 4))
        do = rng.standard_normal((2, nq, 4))
        dq, dk, dv = bw.attention_backward_f64(q, k, v, do, 0.7, causal)
        h = 1e-6
        for x, gx, which in ((q, dq, 0), (k, dk, 1), (v, dv, 2)):
            u = rng.standard_normal(x.shape)
            args = [q, k, v]
            args[which] = x + h * u
            lp = _loss(orc, *args, do, 0.7, causal)
            args[which] = x - h * u
            lm = _loss(orc, *args, do, 0.7, causal)
            assert abs((lp - lm) / (2 * h) - (gx * u).sum()) <= 1e-7, (causal, which)


def pin_bwd_torch_autograd(bw, orc):
    """Against torch's float64 autograd through scaled_dot_product_attention on
    the CPU, with an explicit boolean mask for the causal cases."""
    import torch
    rng = np.random.default_rng(47)
    for causal, nq, nk in ((False, 9, 11), (True, 8, 8), ("bottom_right", 5, 12)):
        q = rng.standard_normal((2, 3, nq, 6))
        k = rng.standard_normal((2, 3, nk, 6))
        v = rng.standard_normal((2, 3, nk, 5))
        do = rng.standard_normal((2, 3, nq, 5))
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        mask = None
        if causal:
            off = 0 if causal is True else nk - nq
            mask = torch.ones(nq, nk, dtype=torch.bool).tril(off)
        out = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=0.45)
        out.backward(torch.tensor(do))
        dq, dk, dv = bw.attention_backward_f64(q, k, v, do, 0.45, causal)
        for got, want in ((dq, tq.grad), (dk, tk.grad), (dv, tv.grad)):
            assert np.allclose(got, want.numpy(), rtol=1e-10, atol=1e-12), causal


def pin_bwd_closed_forms(bw, orc):
    """One key: P = 1, so dV = sum of dO over the queries and dQ = dK = 0. Key
    gradients sum to zero over the keys (each row of dS sums to zero)."""
    rng = np.random.default_rng(53)
    q = rng.standard_normal((4, 3))
    k = rng.standard_normal((1, 3))
    v = rng.standard_normal((1, 2))
    do = rng.standard_normal((4, 2))
    dq, dk, dv = bw.attention_backward_f64(q, k, v, do, 0.9)
    assert np.allclose(dv[0], do.sum(axis=0), rtol=0, atol=1e-14)
    assert np.abs(dq).max() <= 1e-14 and np.abs(dk).max() <= 1e-14
    k = rng.standard_normal((6, 3))
    v = rng.standard_normal((6, 2))
    dq, dk, dv = bw.attention_backward_f64(q, k, v, do, 0.9, True)
    assert np.abs(dk.sum(axis=0)).max() <= 1e-12


BWD_PINS = [
    pin_bwd_printed_gradient,
    pin_bwd_finite_differences,
    pin_bwd_torch_autograd,
    pin_bwd_closed_forms,
]

FP8_PINS = [
    pin_e4m3_hand_values,
    pin_e4m3_vs_torch,
    pin_fp8_single_key,
    pin_fp8_descales,
    pin_p_sigma_closed_forms,
    pin_p_sigma_simulated,
]

ALL_PINS = [
    pin_split_example_block_states,
    pin_split_example_merge,
    pin_split_example_full_attention,
    pin_split_example_gradient,
    pin_split_invariance,
    pin_empty_split_state,
    pin_online_recurrence,
    pin_single_key,
    pin_zero_query,
    pin_causal_first_row,
    pin_rows_sum_to_one,
    pin_shift_invariance,
    pin_huge_scores,
    pin_key_permutation,
    pin_row_subset,
    pin_torch_sdpa_float64,
    pin_brute_force,
    pin_brute_force_bottom_right,
    pin_bottom_right_rows,
    pin_varlen_equal_lengths,
    pin_varlen_brute_force,
    pin_varlen_independence,
]
