"""GPU parity of the e4m3 forward (fa_fwd_fp8) against the float64 oracle of
the encoded values.

Tolerance, from the arithmetic (the FA-3 page, section 7.3, keeps the softmax
statistics in fp32; P is rounded to e4m3 for the PV GEMM):
* S is exact up to fp32 accumulation (products of e4m3 values are exact in
  fp32), so the LSE meets the same bound as the bf16 path, 1e-3.
* O carries the rounding of P to e4m3, error sigma_i per element from
  ``oracle.fp8.p_rounding_sigma`` (independent half-step errors, relative 2^-4
  on normal values), plus the bf16 rounding of O (relative 2^-8 at most, 2^-9
  on average). Per element: |err| <= 6 sigma + 2^-8 |O| + 1e-3. Over a tensor,
  to catch a bias that per-element bounds would let through: rms(err) <=
  1.25 * sqrt(mean(sigma^2 + (2^-9 O)^2 / 3)) + 1e-5.
"""

import math

import numpy as np
import pytest
import torch

import exact_attention_80_gb300 as fa
import oracle
import oracle.fp8 as ofp8
from exact_attention_80_gb300.inputs import f32, make_qkv_fp8

pytestmark = pytest.mark.gpu

LSE_TOL = 1e-3


def check_fp8(o, lse, o_ref, lse_ref, sigma, what):
    o = o.float().cpu().numpy().astype(np.float64)
    lse = lse.float().cpu().numpy().astype(np.float64)
    err = np.abs(o - o_ref)
    bound = 6.0 * sigma + 2.0 ** -8 * np.abs(o_ref) + 1e-3
    worst = np.unravel_index(np.argmax(err - bound), err.shape)
    assert (err <= bound).all(), (what, "element", worst, err[worst], bound[worst])
    rms = math.sqrt(float(np.mean(err ** 2)))
    model = math.sqrt(float(np.mean(sigma ** 2 + (2.0 ** -9 * o_ref) ** 2 / 3.0)))
    assert rms <= 1.25 * model + 1e-5, (what, "rms", rms, model)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isneginf(lse), ~fin), what
    if fin.any():
        assert np.abs(lse[fin] - lse_ref[fin]).max() <= LSE_TOL, what
    return rms, model


def run_fp8(B, H, Nq, Nk, causal, seed, descales=(2.0 ** -5, 2.0 ** -5, 2.0 ** -5), d=128,
            num_splits=1):
    q8, k8, v8 = make_qkv_fp8(B, H, Nq, Nk, d, seed, descales)
    scale = f32(1.0 / math.sqrt(d))
    o, lse = fa.attention_fp8(q8.cuda(), k8.cuda(), v8.cuda(), *descales, causal=causal, scale=scale,
                              num_splits=num_splits)
    torch.cuda.synchronize()
    return q8.numpy(), k8.numpy(), v8.numpy(), scale, o, lse


CASES = [
    # B, H, Nq, Nk, causal: tiles, a ragged tail, both masks, Nq != Nk
    (1, 2, 256, 256, False),
    (1, 2, 300, 333, False),
    (1, 2, 300, 333, True),
    (2, 3, 1000, 1500, False),
    (1, 2, 700, 2000, "bottom_right"),
    (1, 1, 1, 1, False),
    (1, 1, 129, 1, False),
    (1, 4, 2048, 2048, True),
]


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("B,H,Nq,Nk,causal", CASES)
def test_fp8_parity(B, H, Nq, Nk, causal, d):
    """d = 128 (128-byte swizzle rows) and d = 64 (64-byte rows, 64-byte
    swizzle)."""
    descales = (2.0 ** -5, 2.0 ** -5, 2.0 ** -5)
    q8, k8, v8, scale, o, lse = run_fp8(B, H, Nq, Nk, causal, 5100 + Nq + Nk + d, descales, d=d)
    o_ref, lse_ref = ofp8.attention_fp8_f64(q8, k8, v8, *descales, scale, causal)
    sigma = ofp8.p_rounding_sigma(q8, k8, v8, *descales, scale, causal)
    check_fp8(o, lse, o_ref, lse_ref, sigma, f"d{d} B{B} H{H} Nq{Nq} Nk{Nk} {causal}")


def test_fp8_descales():
    """Non-power-of-two descales, different per tensor, with codes that use
    e4m3's whole range (|code value| up to 448)."""
    descales = (0.0123, 0.0071, 0.3)
    q8, k8, v8, scale, o, lse = run_fp8(1, 3, 400, 900, False, 5201, descales)
    assert np.abs(ofp8.e4m3_decode(k8)).max() == ofp8.E4M3_MAX
    o_ref, lse_ref = ofp8.attention_fp8_f64(q8, k8, v8, *descales, scale, False)
    sigma = ofp8.p_rounding_sigma(q8, k8, v8, *descales, scale, False)
    check_fp8(o, lse, o_ref, lse_ref, sigma, "descales")


def test_fp8_full_size_sampled_heads():
    """The C2 shape (B=8, H=32, N=2048, d=128) in e4m3, as the bench times it:
    every row of three heads against the oracle."""
    B, H, N, d = 8, 32, 2048, 128
    descales = (2.0 ** -5, 2.0 ** -5, 2.0 ** -5)
    q8, k8, v8, scale, o, lse = run_fp8(B, H, N, N, False, 5301, descales, d)
    for b, h in ((0, 0), (3, 17), (7, 31)):
        o_ref, lse_ref = ofp8.attention_fp8_f64(q8[b, h], k8[b, h], v8[b, h], *descales, scale)
        sigma = ofp8.p_rounding_sigma(q8[b, h], k8[b, h], v8[b, h], *descales, scale)
        check_fp8(o[b, h], lse[b, h], o_ref, lse_ref, sigma, f"head {b},{h}")


def test_fp8_matches_bf16_path_on_the_same_values():
    """The e4m3 codes decoded to bf16 (exact: e4m3 values are bf16 values) run
    through the bf16 kernel give the same LSE to fp32 rounding, and an O within
    the e4m3 P-rounding bound of it."""
    descales = (1.0, 1.0, 1.0)
    q8, k8, v8, scale, o8, lse8 = run_fp8(1, 2, 512, 777, True, 5401, descales)
    to_bf16 = lambda c: torch.from_numpy(ofp8.e4m3_decode(c)).to(torch.bfloat16).cuda()  # noqa: E731
    o16, lse16 = fa.attention(to_bf16(q8), to_bf16(k8), to_bf16(v8), causal=True, scale=scale)
    torch.cuda.synchronize()
    assert (lse8 - lse16).abs().max().item() <= 1e-4
    o_ref, _ = oracle.attention_f64(ofp8.e4m3_decode(q8), ofp8.e4m3_decode(k8), ofp8.e4m3_decode(v8),
                                    scale, True)
    sigma = ofp8.p_rounding_sigma(q8, k8, v8, 1.0, 1.0, 1.0, scale, True)
    diff = (o8.float() - o16.float()).abs().cpu().numpy()
    assert (diff <= 6.0 * sigma + 2.0 ** -7 * np.abs(o_ref) + 2e-3).all()


@pytest.mark.parametrize("S", [2, 3, 16, 64])
@pytest.mark.parametrize("causal", [False, True, "bottom_right"])
def test_fp8_splitkv(S, causal):
    """fa_fwd_fp8_splitkv + fa_combine against the oracle, with the plain e4m3
    bound (the split only regroups fp32 sums). Splits past the keys are empty."""
    descales = (2.0 ** -5, 0.02, 0.3)
    Nq, Nk = 200, 3000
    q8, k8, v8, scale, o, lse = run_fp8(1, 2, Nq, Nk, causal, 5500 + S, descales, num_splits=S)
    o_ref, lse_ref = ofp8.attention_fp8_f64(q8, k8, v8, *descales, scale, causal)
    sigma = ofp8.p_rounding_sigma(q8, k8, v8, *descales, scale, causal)
    check_fp8(o, lse, o_ref, lse_ref, sigma, f"splits={S} {causal}")


def test_fp8_decode_shape_split():
    """The C5 decode shape (B=1, H=8, Nq=128, Nk=131072) in e4m3 with 16 splits:
    one head's every row against the oracle."""
    B, H, Nq, Nk, d = 1, 8, 128, 131072, 128
    descales = (2.0 ** -5, 2.0 ** -5, 2.0 ** -5)
    q8, k8, v8, scale, o, lse = run_fp8(B, H, Nq, Nk, False, 5601, descales, d, num_splits=16)
    h = 5
    o_ref, lse_ref = ofp8.attention_fp8_f64(q8[0, h], k8[0, h], v8[0, h], *descales, scale)
    sigma = ofp8.p_rounding_sigma(q8[0, h], k8[0, h], v8[0, h], *descales, scale)
    check_fp8(o[0, h], lse[0, h], o_ref, lse_ref, sigma, "c5 head 5")


@pytest.mark.parametrize("S,Nq", [(2, 128), (7, 100), (40, 1)])
def test_fp8_dual_range_split(S, Nq):
    """e4m3 split-KV with one query tile (two splits per CTA), odd split counts
    and splits without keys, against the oracle."""
    descales = (2.0 ** -5, 0.02, 0.3)
    q8, k8, v8, scale, o, lse = run_fp8(2, 2, Nq, 4000, "bottom_right", 5700 + S, descales,
                                        num_splits=S)
    o_ref, lse_ref = ofp8.attention_fp8_f64(q8, k8, v8, *descales, scale, "bottom_right")
    sigma = ofp8.p_rounding_sigma(q8, k8, v8, *descales, scale, "bottom_right")
    check_fp8(o, lse, o_ref, lse_ref, sigma, f"dual S={S} Nq={Nq}")


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("causal", [False, True, "bottom_right"])
def test_fp8_persistent_ctas(d, causal):
    """More query units than four waves of CTAs (B=2, H=160, Nq=300, Nk=333:
    640 units, each head's last tile ragged), so fa_fwd_fp8 runs persistent
    CTAs that walk several units each; every element against the oracle."""
    B, H, Nq, Nk = 2, 160, 300, 333
    assert fa.fa_fwd_grid_ctas(B, H, Nq, d, 1) >= 4 * torch.cuda.get_device_properties(0).multi_processor_count
    descales = (2.0 ** -5, 0.02, 0.3)
    q8, k8, v8, scale, o, lse = run_fp8(B, H, Nq, Nk, causal, 5950 + d, descales, d=d)
    o_ref, lse_ref = ofp8.attention_fp8_f64(q8, k8, v8, *descales, scale, causal)
    sigma = ofp8.p_rounding_sigma(q8, k8, v8, *descales, scale, causal)
    check_fp8(o, lse, o_ref, lse_ref, sigma, f"persistent d{d} {causal}")


def test_fp8_persistent_rows_without_keys():
    """e4m3 persistent CTAs over units with no key step, or keys in the
    second tile only (bottom-right, Nq = 700 > Nk = 200, 960 units)."""
    B, H, Nq, Nk, d = 1, 320, 700, 200, 128
    descales = (2.0 ** -5, 2.0 ** -5, 2.0 ** -5)
    q8, k8, v8, scale, o, lse = run_fp8(B, H, Nq, Nk, "bottom_right", 5960, descales, d=d)
    o_ref, lse_ref = ofp8.attention_fp8_f64(q8, k8, v8, *descales, scale, "bottom_right")
    sigma = ofp8.p_rounding_sigma(q8, k8, v8, *descales, scale, "bottom_right")
    check_fp8(o, lse, o_ref, lse_ref, sigma, "persistent, rows without keys")


@pytest.mark.parametrize("S,Nq", [(3, 200), (2, 128), (7, 100), (40, 1)])
def test_fp8_splitkv_d64(S, Nq):
    """d = 64 e4m3 through split-KV + merge: two query tiles per CTA (Nq = 200)
    and dual-range CTAs (Nq <= 128), odd split counts and splits without keys."""
    descales = (0.0123, 0.0071, 0.3)
    q8, k8, v8, scale, o, lse = run_fp8(2, 2, Nq, 4000, "bottom_right", 5800 + S + Nq, descales, d=64,
                                        num_splits=S)
    o_ref, lse_ref = ofp8.attention_fp8_f64(q8, k8, v8, *descales, scale, "bottom_right")
    sigma = ofp8.p_rounding_sigma(q8, k8, v8, *descales, scale, "bottom_right")
    check_fp8(o, lse, o_ref, lse_ref, sigma, f"d64 S={S} Nq={Nq}")


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_full_size_d64_sampled_heads(causal):
    """The batched shape at d = 64 (B=8, H=32, N=2048) in e4m3, as the bench
    times it: every row of three heads, spread over the grid, against the
    oracle."""
    B, H, N, d = 8, 32, 2048, 64
    descales = (2.0 ** -5, 2.0 ** -5, 2.0 ** -5)
    q8, k8, v8, scale, o, lse = run_fp8(B, H, N, N, causal, 5901, descales, d)
    for b, h in ((0, 0), (3, 17), (7, 31)):
        o_ref, lse_ref = ofp8.attention_fp8_f64(q8[b, h], k8[b, h], v8[b, h], *descales, scale, causal)
        sigma = ofp8.p_rounding_sigma(q8[b, h], k8[b, h], v8[b, h], *descales, scale, causal)
        check_fp8(o[b, h], lse[b, h], o_ref, lse_ref, sigma, f"d64 head {b},{h} causal={causal}")


D256_CASES = [
    # B, H, Nq, Nk, causal: the d = 256 kernel (one 128-row tile per CTA, key
    # tiles of 96): tails in both, both masks, Nq != Nk
    (1, 2, 128, 96, False),
    (1, 2, 300, 333, False),
    (1, 2, 300, 333, True),
    (2, 2, 700, 1000, "bottom_right"),
    (1, 1, 1, 1, False),
    (1, 2, 1000, 300, True),
]


@pytest.mark.parametrize("B,H,Nq,Nk,causal", D256_CASES)
def test_fp8_parity_d256(B, H, Nq, Nk, causal):
    descales = (2.0 ** -5, 2.0 ** -5, 2.0 ** -5)
    q8, k8, v8, scale, o, lse = run_fp8(B, H, Nq, Nk, causal, 5500 + Nq + Nk, descales, d=256)
    o_ref, lse_ref = ofp8.attention_fp8_f64(q8, k8, v8, *descales, scale, causal)
    sigma = ofp8.p_rounding_sigma(q8, k8, v8, *descales, scale, causal)
    check_fp8(o, lse, o_ref, lse_ref, sigma, f"d256 B{B} H{H} Nq{Nq} Nk{Nk} {causal}")


@pytest.mark.parametrize("S", [2, 5])
def test_fp8_splitkv_d256(S):
    """d = 256 e4m3 through split-KV + merge, non-power-of-two descales."""
    descales = (0.0123, 0.0071, 0.3)
    q8, k8, v8, scale, o, lse = run_fp8(1, 3, 200, 1500, "bottom_right", 5600 + S, descales, d=256,
                                        num_splits=S)
    o_ref, lse_ref = ofp8.attention_fp8_f64(q8, k8, v8, *descales, scale, "bottom_right")
    sigma = ofp8.p_rounding_sigma(q8, k8, v8, *descales, scale, "bottom_right")
    check_fp8(o, lse, o_ref, lse_ref, sigma, f"d256 splits={S}")


def test_fp8_full_size_d256_sampled_heads():
    """The large-head-dim workload's shape (B=8, H=16, N=8191, d=256, causal) in
    e4m3, as the bench times it: every row of three heads against the oracle."""
    B, H, N, d = 8, 16, 8191, 256
    descales = (2.0 ** -5, 2.0 ** -5, 2.0 ** -5)
    q8, k8, v8, scale, o, lse = run_fp8(B, H, N, N, True, 5701, descales, d)
    for b, h in ((0, 0), (4, 9), (7, 15)):
        o_ref, lse_ref = ofp8.attention_fp8_f64(q8[b, h], k8[b, h], v8[b, h], *descales, scale, True)
        sigma = ofp8.p_rounding_sigma(q8[b, h], k8[b, h], v8[b, h], *descales, scale, True)
        check_fp8(o[b, h], lse[b, h], o_ref, lse_ref, sigma, f"d256 head {b},{h}")
