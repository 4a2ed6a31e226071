"""GPU parity of the variable-length forward (fa_fwd_varlen) against the float64
oracle's per-sequence statement, on packed token-major inputs.

Same acceptance as the dense path: on O, max-abs <= 2e-2 and relative L2
<= 5e-3; on LSE, max-abs <= 1e-3 (rows that see no key: -inf on both sides).
"""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import exact_attention_80_gb300 as fa  # noqa: E402
import oracle  # noqa: E402
from exact_attention_80_gb300.inputs import f32, make_qkv, make_varlen, to_f64  # noqa: E402

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
REL_L2 = 5e-3
LSE_ABS = 1e-3


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    fa.load_library()
    fa.fa_device_status(clear=True)


def check(o_gpu, lse_gpu, o_ref, lse_ref, what):
    o = o_gpu.float().cpu().numpy().astype(np.float64)
    lse = lse_gpu.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    max_abs = float(np.abs(o - o_ref).max()) if o.size else 0.0
    rel = float(np.linalg.norm((o - o_ref).ravel()) / max(np.linalg.norm(o_ref.ravel()), 1e-30))
    empty = ~np.isfinite(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: -inf LSE rows differ"
    lse_err = float(np.abs(lse[~empty] - lse_ref[~empty]).max()) if (~empty).any() else 0.0
    assert max_abs <= MAX_ABS, f"{what}: max-abs {max_abs:.3e}"
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e}"
    assert lse_err <= LSE_ABS, f"{what}: LSE err {lse_err:.3e}"


def run(q, k, v, cu_q, cu_k, causal, scale):
    max_q = int((cu_q[1:] - cu_q[:-1]).max())
    o, lse = fa.attention_varlen(q.cuda(), k.cuda(), v.cuda(), cu_q.cuda(), cu_k.cuda(),
                                 max(max_q, 1), causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    return o, lse


RAGGED = [
    # query lengths, key lengths (one entry per sequence)
    ([1, 127, 128, 129, 300, 0, 513], [5, 127, 256, 129, 1, 17, 513]),
    ([256, 70, 1000], [256, 3000, 40]),
    ([64, 0, 200], [0, 64, 200]),  # a sequence with queries but no key
]


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True, "bottom_right"])
@pytest.mark.parametrize("case", range(len(RAGGED)))
def test_varlen_ragged(d, causal, case):
    lq, lk = RAGGED[case]
    q, k, v, cu_q, cu_k = make_varlen(lq, lk, 3, d, 900 + 7 * case + d)
    scale = f32(1.0 / math.sqrt(d))
    o, lse = run(q, k, v, cu_q, cu_k, causal, scale)
    o_ref, lse_ref = oracle.attention_varlen_f64(to_f64(q), to_f64(k), to_f64(v), cu_q.numpy(),
                                                cu_k.numpy(), scale, causal)
    check(o, lse, o_ref, lse_ref, f"lq={lq} lk={lk} d={d} causal={causal}")


@pytest.mark.parametrize("d", [64, 128, 256])
def test_varlen_equal_lengths_match_dense_path(d):
    """Equal-length sequences packed token-major give the dense API's result."""
    B, H, N = 3, 2, 333
    q, k, v = make_qkv(B, H, N, N, d, 77 + d)
    scale = f32(1.0 / math.sqrt(d))
    pack = lambda x: x.transpose(1, 2).reshape(B * N, H, d).contiguous()  # noqa: E731
    cu = torch.arange(B + 1, dtype=torch.int32) * N
    for causal in (False, True):
        o_v, lse_v = run(pack(q), pack(k), pack(v), cu, cu, causal, scale)
        o_d, lse_d = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale)
        torch.cuda.synchronize()
        assert torch.equal(o_v, pack(o_d.cpu()).cuda())
        assert torch.equal(lse_v, lse_d.transpose(0, 1).reshape(H, B * N))


def test_varlen_leaves_tokens_past_the_batch():
    """Tokens past cu_seqlens_q[B] are not written (sentinels survive)."""
    d, H = 128, 2
    q, k, v, cu_q, cu_k = make_varlen([100, 50], [80, 120], H, d, 31)
    total_q = q.shape[0] + 40
    qp = torch.zeros((total_q, H, d), dtype=torch.bfloat16)
    qp[: q.shape[0]] = q
    o = torch.full((total_q, H, d), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((H, total_q), 5.0, dtype=torch.float32, device="cuda")
    fa.fa_fwd_varlen(qp.cuda(), k.cuda(), v.cuda(), o, lse, cu_q.cuda(), cu_k.cuda(), 100)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    assert torch.all(o[q.shape[0]:] == 7.0) and torch.all(lse[:, q.shape[0]:] == 5.0)


def test_varlen_bad_offsets_reported_not_used():
    """Offsets that are not a valid partition (decreasing; a query length above
    max_seqlen_q) are found on the device: nothing of those sequences is read
    or written, and fa_device_status reports FA_ERR_SEQLENS."""
    d, H = 64, 1
    q, k, v, _, _ = make_varlen([40, 40, 40], [40, 40, 40], H, d, 5)
    o = torch.full((120, H, d), 3.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((H, 120), 2.0, dtype=torch.float32, device="cuda")
    bad_q = torch.tensor([0, 40, 20, 120], dtype=torch.int32, device="cuda")  # decreasing
    cu_k = torch.tensor([0, 40, 80, 120], dtype=torch.int32, device="cuda")
    fa.fa_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), o, lse, bad_q, cu_k, 100)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_ERR_SEQLENS
    # Sequence 1 (40 -> 20) is skipped; sequence 0 is computed.
    assert torch.all(o[:40] != 3.0)
    long_q = torch.tensor([0, 40, 80, 120], dtype=torch.int32, device="cuda")
    o.fill_(3.0)
    fa.fa_fwd_varlen(q.cuda(), k.cuda(), v.cuda(), o, lse, long_q, cu_k, 30)  # 40 > 30
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_ERR_SEQLENS
    assert torch.all(o == 3.0)
