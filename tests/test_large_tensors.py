"""Tensors past 2^31 elements (more than 4 GiB of bf16), on the GPU.

The kernels address rows, partial states, token-major sequences and the
backward's dQ accumulator with 64-bit offsets; tensor-map coordinates stay
small (column, row within a head, head). These cases put the last heads (or
sequences) of each tensor beyond element 2^31, and the split-KV partial states
beyond element 2^32, and compare the heads on either side of that boundary,
plus the first and the last, with the float64 oracle. Query lengths are not
multiples of the tile, so the ragged tail is stored at those offsets too.

Inputs are drawn on the device by the seeded device generators of
``exact_attention_80_gb300.inputs`` (too large to draw on the host); only the
checked heads are copied back for the oracle.
"""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import exact_attention_80_gb300 as fa  # noqa: E402
import oracle  # noqa: E402
import oracle.backward as obw  # noqa: E402
import oracle.fp8 as ofp8  # noqa: E402
from exact_attention_80_gb300.inputs import f32, make_device_e4m3, make_device_normal  # noqa: E402

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
REL_L2 = 5e-3
LSE_ABS = 1e-3

# One head of Nq = 1000 rows at d = 128 is 128,000 elements, so head 16777
# straddles element 2^31 and head 16799 lies past it.
H, NQ, D = 16800, 1000, 128
HEADS = (0, 16776, 16777, 16778, H - 1)


@pytest.fixture(autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    fa.load_library()
    fa.fa_device_status(clear=True)
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


def _check_head(o, lse, o_ref, lse_ref, what):
    o, lse = _f64(o), lse.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    assert float(np.abs(o - o_ref).max()) <= MAX_ABS, what
    rel = float(np.linalg.norm(o - o_ref) / np.linalg.norm(o_ref))
    assert rel <= REL_L2, (what, rel)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isneginf(lse), ~fin), what
    assert float(np.abs(lse[fin] - lse_ref[fin]).max()) <= LSE_ABS, what


def _qkv(Nk, seed):
    dev = torch.device("cuda", 0)
    q = make_device_normal((1, H, NQ, D), seed, dev)
    k = make_device_normal((1, H, Nk, D), seed + 1, dev)
    v = make_device_normal((1, H, Nk, D), seed + 2, dev)
    assert q.numel() > 2 ** 31
    return q, k, v


@pytest.mark.parametrize("causal", [False, True])
def test_forward_past_2g_elements(causal):
    """Persistent forward (four waves of short units) over a 4.3 GB Q and O."""
    q, k, v = _qkv(300, 7100)
    scale = f32(1.0 / math.sqrt(D))
    o, lse = fa.attention(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    assert bool(torch.isfinite(o).all())
    for h in HEADS:
        o_ref, lse_ref = oracle.attention_f64(_f64(q[0, h]), _f64(k[0, h]), _f64(v[0, h]), scale, causal)
        _check_head(o[0, h], lse[0, h], o_ref, lse_ref, f"head {h} causal={causal}")


def test_splitkv_partials_past_2_to_32():
    """Split-KV partial states of 4.4e9 floats (17.5 GB), then the merge."""
    q, k, v = _qkv(500, 7200)
    S = 2
    nbytes = fa.fa_splitkv_workspace_bytes(1, H, NQ, D, S)
    assert nbytes // 4 > 2 ** 32
    ws = torch.empty(nbytes // 4, dtype=torch.float32, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((1, H, NQ), dtype=torch.float32, device=q.device)
    scale = f32(1.0 / math.sqrt(D))
    fa.fa_fwd_splitkv(q, k, v, ws, S, False, scale)
    fa.fa_combine(ws, o, lse, 1, H, NQ, D, S)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    for h in HEADS:
        o_ref, lse_ref = oracle.attention_f64(_f64(q[0, h]), _f64(k[0, h]), _f64(v[0, h]), scale, False)
        _check_head(o[0, h], lse[0, h], o_ref, lse_ref, f"head {h}")


def test_backward_past_2g_elements():
    """dQ, dK, dV with Q, O, dO, dQ of 4.3 GB and an 8.7 GB dQ accumulator, at the
    backward tests' bounds (max error 1e-2 of the largest reference entry + 1e-3,
    relative L2 1e-2)."""
    q, k, v = _qkv(200, 7300)
    do = make_device_normal((1, H, NQ, D), 7303, q.device)
    scale = f32(1.0 / math.sqrt(D))
    o, lse = fa.attention(q, k, v, causal=True, scale=scale)
    dq, dk, dv = fa.attention_backward(q, k, v, o, lse, do, causal=True, scale=scale)
    del o, lse
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    for h in HEADS:
        ref = obw.attention_backward_f64(_f64(q[0, h]), _f64(k[0, h]), _f64(v[0, h]), _f64(do[0, h]),
                                         scale, True)
        for g, r, name in zip((dq[0, h], dk[0, h], dv[0, h]), ref, ("dq", "dk", "dv")):
            g = _f64(g)
            assert float(np.abs(g - r).max()) <= 1e-2 * float(np.abs(r).max()) + 1e-3, (name, h)
            assert float(np.linalg.norm(g - r)) <= 1e-2 * float(np.linalg.norm(r)), (name, h)


def test_varlen_past_2g_elements():
    """265 packed sequences, token-major, 2.2e9 query elements: sequence 262
    straddles element 2^31 and the last two start past it. Bottom-right mask
    with lq > lk, so the first rows of each sequence see no key."""
    Hv, lq, lk = 64, 1000, 256
    nseq = 265
    dev = torch.device("cuda", 0)
    q = make_device_normal((nseq * lq, Hv, D), 7400, dev)
    k = make_device_normal((nseq * lk, Hv, D), 7401, dev)
    v = make_device_normal((nseq * lk, Hv, D), 7402, dev)
    assert q.numel() > 2 ** 31
    cu_q = torch.arange(0, nseq + 1, dtype=torch.int32, device=dev) * lq
    cu_k = torch.arange(0, nseq + 1, dtype=torch.int32, device=dev) * lk
    scale = f32(1.0 / math.sqrt(D))
    o, lse = fa.attention_varlen(q, k, v, cu_q, cu_k, lq, causal="bottom_right", scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    first_past = (2 ** 31) // (lq * Hv * D)  # the sequence that straddles element 2^31
    for b in (0, first_past, first_past + 1, nseq - 1):
        sq, sk = slice(b * lq, (b + 1) * lq), slice(b * lk, (b + 1) * lk)
        qs, ks, vs = (_f64(t[s]).transpose(1, 0, 2) for t, s in ((q, sq), (k, sk), (v, sk)))
        o_ref, lse_ref = oracle.attention_f64(qs, ks, vs, scale, "bottom_right")
        _check_head(o[sq].transpose(0, 1), lse[:, sq], o_ref, lse_ref, f"sequence {b}")


def test_fp8_forward_past_2g_bytes():
    """e4m3 Q of 2.15e9 bytes, within the e4m3 P-rounding bound."""
    dev = torch.device("cuda", 0)
    ds = 2.0 ** -5
    q8 = make_device_e4m3((1, H, NQ, D), 7500, dev, ds)
    k8 = make_device_e4m3((1, H, 300, D), 7501, dev, ds)
    v8 = make_device_e4m3((1, H, 300, D), 7502, dev, ds)
    assert q8.numel() > 2 ** 31
    scale = f32(1.0 / math.sqrt(D))
    o, lse = fa.attention_fp8(q8, k8, v8, ds, ds, ds, causal=False, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    for h in HEADS:
        qn, kn, vn = (t[0, h].cpu().numpy() for t in (q8, k8, v8))
        o_ref, lse_ref = ofp8.attention_fp8_f64(qn, kn, vn, ds, ds, ds, scale, False)
        sigma = ofp8.p_rounding_sigma(qn, kn, vn, ds, ds, ds, scale, False)
        err = np.abs(_f64(o[0, h]) - o_ref)
        assert (err <= 6.0 * sigma + 2.0 ** -8 * np.abs(o_ref) + 1e-3).all(), h
        lse64 = lse[0, h].cpu().numpy().astype(np.float64)
        assert float(np.abs(lse64 - lse_ref).max()) <= LSE_ABS, h
