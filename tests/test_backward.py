"""GPU parity of the backward (fa_bwd) against the float64 gradient oracle.

Tolerance, from the arithmetic: the inputs are exact bf16, and every product is
accumulated in fp32. Three quantities are rounded on the GPU: P and dS to bf16
before their MMAs, and O to bf16 (the forward's output) before D = rowsum(dO O).
Each rounding is about 2^-9 relative, and the gradients are rounded to bf16 at
the end. Each gradient element sums many such terms, so the per-tensor bound is
relative L2 <= 1e-2 (about 2.5x the bf16 unit 2^-8). The largest element error is
bounded by 1e-2 of the tensor's largest magnitude, plus 1e-3.
"""

import math

import numpy as np
import pytest
import torch

import exact_attention_80_gb300 as fa
import oracle
import oracle.backward as obw
from exact_attention_80_gb300.inputs import f32, make_grad_output, make_qkv, to_f64

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
MAX_REL = 1e-2


def check_grad(got, ref, what):
    got = got.float().cpu().numpy().astype(np.float64)
    scale = float(np.abs(ref).max())
    err = np.abs(got - ref)
    assert err.max() <= MAX_REL * scale + 1e-3, (what, "max", float(err.max()), scale)
    # A zero reference (one key: dQ = dK = 0) has no relative L2; the element
    # bound above is the whole check there.
    den = float(np.linalg.norm(ref))
    if den > 0:
        assert float(np.linalg.norm(got - ref)) <= REL_L2 * den, (what, "rel-L2", float(np.linalg.norm(got - ref)) / den)


def run_bwd(B, H, Nq, Nk, causal, seed, d=128):
    q, k, v = make_qkv(B, H, Nq, Nk, d, seed)
    do = make_grad_output(B, H, Nq, d, seed + 1)
    scale = f32(1.0 / math.sqrt(d))
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.attention(qc, kc, vc, causal=causal, scale=scale)
    dq, dk, dv = fa.attention_backward(qc, kc, vc, o, lse, doc, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    ref = obw.attention_backward_f64(to_f64(q), to_f64(k), to_f64(v), to_f64(do), scale, causal)
    return (dq, dk, dv), ref


CASES = [
    # B, H, Nq, Nk, causal
    (1, 1, 128, 128, False),
    (1, 2, 300, 333, False),
    (1, 2, 300, 333, True),
    (2, 3, 257, 511, True),
    (1, 2, 384, 384, "bottom_right"),
    (1, 2, 700, 200, "bottom_right"),   # rows without keys
    (1, 1, 100, 300, True),             # keys no query sees: dK = dV = 0
    (1, 2, 1, 1000, False),
    (1, 1, 1000, 1, False),
    (2, 2, 1024, 1024, False),
]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("B,H,Nq,Nk,causal", CASES)
def test_backward_parity(B, H, Nq, Nk, causal, d):
    got, ref = run_bwd(B, H, Nq, Nk, causal, 8100 + Nq + Nk + d, d)
    for g, r, name in zip(got, ref, ("dq", "dk", "dv")):
        check_grad(g, r, f"{name} B{B} H{H} Nq{Nq} Nk{Nk} {causal} d{d}")


@pytest.mark.parametrize("d", [64, 128, 256])
def test_backward_negative_scores_key_tail(d):
    """Every score near -200 (Q along u, K against it): LSE is about -190, so an
    unmasked missing key of the ragged last key tile (its S reads 0) would give
    exp(190) = inf in fp32 and NaN in dQ. The missing keys are masked.

    dV takes the usual bounds. dQ_i = scale sum_j dS_ij K_j, and every K_j
    carries the common part -c u while sum_j dS_ij = 0, so the bf16 rounding of
    dS (2^-9) is amplified by about c / sqrt(d), 4 to 5, against dQ's own size; dK
    sees the same part of Q. Rounding P, dS and O to bf16 in a float64 model of
    this input gives 2.6 % (dQ) and 0.75 % (dK) of the largest element: dQ takes
    5e-2 and dK 2e-2, for both the element bound and the relative L2."""
    B, H, Nq, Nk = 1, 2, 200, 300
    q, k, v = make_qkv(B, H, Nq, Nk, d, 8301)
    do = make_grad_output(B, H, Nq, d, 8302)
    scale = f32(1.0 / math.sqrt(d))
    u = torch.zeros(d)
    u[:8] = 1.0 / math.sqrt(8.0)
    c = math.sqrt(200.0 / scale)
    q = (q.float() + c * u).to(torch.bfloat16)
    k = (k.float() - c * u).to(torch.bfloat16)
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.attention(qc, kc, vc, scale=scale)
    assert lse.max().item() < -150.0
    dq, dk, dv = fa.attention_backward(qc, kc, vc, o, lse, doc, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    rq, rk, rv = obw.attention_backward_f64(to_f64(q), to_f64(k), to_f64(v), to_f64(do), scale)
    for g, name in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        assert torch.isfinite(g).all(), name
    check_grad(dv, rv, "dv negative scores")
    for g, r, tol, name in ((dq, rq, 5e-2, "dq"), (dk, rk, 2e-2, "dk")):
        got = g.float().cpu().numpy().astype(np.float64)
        err = np.abs(got - r)
        assert err.max() <= tol * np.abs(r).max(), (name, float(err.max()))
        assert np.linalg.norm(got - r) <= tol * np.linalg.norm(r), name


@pytest.fixture(scope="module")
def head_pool():
    from oracle.parallel import HeadPool

    with HeadPool() as pool:
        yield pool


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("causal", [True, False])
def test_backward_full_size_every_head(head_pool, causal, d):
    """The C2 shape (B=8, H=32, N=2048) at d = 128 and 64, as the bench times
    it: dQ, dK and dV of every head against the oracle (run per head in worker
    processes), each head held to the per-tensor bounds."""
    B, H, N = 8, 32, 2048
    q, k, v = make_qkv(B, H, N, N, d, 8201)
    do = make_grad_output(B, H, N, d, 8202)
    scale = f32(1.0 / math.sqrt(d))
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.attention(qc, kc, vc, causal=causal, scale=scale)
    dq, dk, dv = fa.attention_backward(qc, kc, vc, o, lse, doc, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    got = [t.reshape(B * H, N, d).cpu() for t in (dq, dk, dv)]
    qh, kh, vh, doh = (t.reshape(B * H, N, d) for t in (q, k, v, do))
    tasks = ((i, qh[i].float().numpy(), kh[i].float().numpy(), vh[i].float().numpy(),
              doh[i].float().numpy(), scale, causal) for i in range(B * H))
    seen = 0
    for i, *ref in head_pool.backward_heads(tasks):
        for g, r, name in zip(got, ref, ("dq", "dk", "dv")):
            check_grad(g[i], r, f"{name} head {i} causal={causal}")
        seen += 1
    assert seen == B * H


@pytest.mark.parametrize("causal", [True, False])
def test_backward_d256_sampled_heads(head_pool, causal):
    """Head dim 256 at the bench's shape (B=2, H=16, N=4096): two CTAs per key
    tile, one per half of the head dim, and one Q/dO stage. dQ, dK and dV of
    three heads spread over the grid against the oracle."""
    B, H, N, d = 2, 16, 4096, 256
    q, k, v = make_qkv(B, H, N, N, d, 8401)
    do = make_grad_output(B, H, N, d, 8402)
    scale = f32(1.0 / math.sqrt(d))
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.attention(qc, kc, vc, causal=causal, scale=scale)
    dq, dk, dv = fa.attention_backward(qc, kc, vc, o, lse, doc, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    got = [t.reshape(B * H, N, d).cpu() for t in (dq, dk, dv)]
    qh, kh, vh, doh = (t.reshape(B * H, N, d) for t in (q, k, v, do))
    heads = (0, 17, B * H - 1)
    tasks = ((i, qh[i].float().numpy(), kh[i].float().numpy(), vh[i].float().numpy(),
              doh[i].float().numpy(), scale, causal) for i in heads)
    seen = 0
    for i, *ref in head_pool.backward_heads(tasks):
        for g, r, name in zip(got, ref, ("dq", "dk", "dv")):
            check_grad(g[i], r, f"d256 {name} head {i} causal={causal}")
        seen += 1
    assert seen == len(heads)
