"""A seeded sweep of small shapes against the oracle.

The fixed parity cases pick their ragged tails and masks by hand. This sweep
draws shapes from a fixed seed instead: head dims 64, 128 and 256, query and key
lengths from 1 to about 700 (so tails fall anywhere in a tile and Nq may exceed
Nk), all three masks, and for split-KV a random split count. Each case is
compared with the float64 oracle on the whole output, with the same tolerances
as the other parity tests, and e4m3 cases within the e4m3 P-rounding bound. The
backward and packed variable-length batches get sweeps of their own.
"""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import exact_attention_80_gb300 as fa  # noqa: E402
import oracle  # noqa: E402
import oracle.backward as obw  # noqa: E402
import oracle.fp8 as ofp8  # noqa: E402
from exact_attention_80_gb300.inputs import (f32, make_grad_output, make_qkv, make_qkv_fp8,  # noqa: E402
                                            make_varlen, to_f64)

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _needs_cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")


MAX_ABS = 2e-2
REL_L2 = 5e-3
LSE_ABS = 1e-3
MASKS = (False, True, "bottom_right")


def _draw(n, seed, dims=(64, 128, 256)):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        d = int(rng.choice(dims))
        Nq = int(rng.integers(1, 700))
        Nk = int(rng.integers(1, 700))
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        causal = MASKS[int(rng.integers(0, 3))]
        out.append((B, H, Nq, Nk, d, causal, 9300 + 7 * i))
    return out


def _check(o_gpu, lse_gpu, o_ref, lse_ref, what):
    o = o_gpu.float().cpu().numpy().astype(np.float64)
    lse = lse_gpu.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    err = np.abs(o - o_ref)
    rel = float(np.linalg.norm((o - o_ref).ravel()) / max(np.linalg.norm(o_ref.ravel()), 1e-30))
    empty = ~np.isfinite(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: -inf LSE rows differ"
    assert float(err.max()) <= MAX_ABS, f"{what}: max-abs {float(err.max()):.3e}"
    # rel-L2 is meaningless when every row is empty (o_ref = 0).
    assert rel <= REL_L2 or not (~empty).any(), f"{what}: rel-L2 {rel:.3e}"
    if (~empty).any():
        assert float(np.abs(lse[~empty] - lse_ref[~empty]).max()) <= LSE_ABS, f"{what}: LSE"


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,seed", _draw(24, 20261203))
def test_random_shape_forward(B, H, Nq, Nk, d, causal, seed):
    q, k, v = make_qkv(B, H, Nq, Nk, d, seed)
    scale = f32(1.0 / math.sqrt(d))
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    o_ref, lse_ref = oracle.attention_f64(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    _check(o, lse, o_ref, lse_ref, f"B{B} H{H} Nq{Nq} Nk{Nk} d{d} {causal}")


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,seed", _draw(12, 20261204))
def test_random_shape_splitkv(B, H, Nq, Nk, d, causal, seed):
    S = 1 + seed % 9  # 1 .. 9 splits, some of them empty for short Nk
    q, k, v = make_qkv(B, H, Nq, Nk, d, seed)
    scale = f32(1.0 / math.sqrt(d))
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale, num_splits=S)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    o_ref, lse_ref = oracle.attention_f64(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    _check(o, lse, o_ref, lse_ref, f"B{B} H{H} Nq{Nq} Nk{Nk} d{d} {causal} S{S}")


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,seed", _draw(12, 20261205))
def test_random_shape_fp8(B, H, Nq, Nk, d, causal, seed):
    descales = (2.0 ** -5, 2.0 ** -5, 2.0 ** -5)
    q8, k8, v8 = make_qkv_fp8(B, H, Nq, Nk, d, seed, descales)
    scale = f32(1.0 / math.sqrt(d))
    o, lse = fa.attention_fp8(q8.cuda(), k8.cuda(), v8.cuda(), *descales, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    qn, kn, vn = q8.numpy(), k8.numpy(), v8.numpy()
    o_ref, lse_ref = ofp8.attention_fp8_f64(qn, kn, vn, *descales, scale, causal)
    sigma = ofp8.p_rounding_sigma(qn, kn, vn, *descales, scale, causal)
    o64 = o.float().cpu().numpy().astype(np.float64)
    err = np.abs(o64 - o_ref)
    bound = 6.0 * sigma + 2.0 ** -8 * np.abs(o_ref) + 1e-3
    assert (err <= bound).all(), f"B{B} H{H} Nq{Nq} Nk{Nk} d{d} {causal}: e4m3 bound"
    lse64 = lse.float().cpu().numpy().astype(np.float64)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isneginf(lse64), ~fin)
    if fin.any():
        assert np.abs(lse64[fin] - lse_ref[fin]).max() <= LSE_ABS


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,seed", _draw(12, 20261206))
def test_random_shape_backward(B, H, Nq, Nk, d, causal, seed):
    """dQ, dK, dV within the backward tests' bounds (max error 1e-2 of the largest
    reference entry + 1e-3, relative L2 1e-2)."""
    q, k, v = make_qkv(B, H, Nq, Nk, d, seed)
    do = make_grad_output(B, H, Nq, d, seed + 1)
    scale = f32(1.0 / math.sqrt(d))
    qc, kc, vc, doc = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, lse = fa.attention(qc, kc, vc, causal=causal, scale=scale)
    got = fa.attention_backward(qc, kc, vc, o, lse, doc, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    ref = obw.attention_backward_f64(to_f64(q), to_f64(k), to_f64(v), to_f64(do), scale, causal)
    for g, r, name in zip(got, ref, ("dq", "dk", "dv")):
        g = g.float().cpu().numpy().astype(np.float64)
        top = float(np.abs(r).max())
        assert float(np.abs(g - r).max()) <= 1e-2 * top + 1e-3, (name, B, H, Nq, Nk, d, causal)
        den = float(np.linalg.norm(r))
        if den > 0:
            assert float(np.linalg.norm(g - r)) <= 1e-2 * den, (name, B, H, Nq, Nk, d, causal)


def _draw_varlen(n, seed):
    rng = np.random.default_rng(seed)
    out = []
    for i in range(n):
        nseq = int(rng.integers(1, 7))
        lq = [int(x) for x in rng.integers(0, 400, nseq)]
        lk = [int(x) for x in rng.integers(0, 400, nseq)]
        if sum(lq) == 0:
            lq[0] = 1
        if sum(lk) == 0:
            lk[0] = 1
        out.append((lq, lk, int(rng.choice((64, 128, 256))), MASKS[int(rng.integers(0, 3))], 9600 + 11 * i))
    return out


@pytest.mark.parametrize("lq,lk,d,causal,seed", _draw_varlen(10, 20261207))
def test_random_varlen_batch(lq, lk, d, causal, seed):
    """Packed variable-length batches with random per-sequence lengths (empty
    sequences included) against the oracle, sequence by sequence."""
    H = 2
    q, k, v, cu_q, cu_k = make_varlen(lq, lk, H, d, seed)
    scale = f32(1.0 / math.sqrt(d))
    o = torch.empty(q.shape, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((H, q.shape[0]), dtype=torch.float32, device="cuda")
    fa.fa_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), o, lse, cu_q.cuda(), cu_k.cuda(), max(lq), causal, scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    o_ref, lse_ref = oracle.attention_varlen_f64(to_f64(q), to_f64(k), to_f64(v), cu_q.numpy(),
                                                cu_k.numpy(), scale, causal)
    _check(o, lse, o_ref, lse_ref, f"lq={lq} lk={lk} d={d} {causal}")
