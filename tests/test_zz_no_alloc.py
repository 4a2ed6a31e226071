"""fa_fwd_splitkv_static, the entry point that allocates nothing.

It serves callers that may not call cudaMalloc (device memory owned and
budgeted by a host framework's own allocator; serving loops where an
allocation could stall the device). It keeps the split partial states in the
library's static device buffer instead of a caller workspace. These tests call
it through the C ABI and check, on two calls in a row, that it gives what the
workspace path (fa_fwd_splitkv + fa_combine) gives and what the float64 oracle
gives, within the parity tolerances used everywhere else. This file is
collected last on purpose.
"""

import ctypes
import math

import pytest

torch = pytest.importorskip("torch")

import exact_attention_80_gb300 as fa  # noqa: E402
from exact_attention_80_gb300.inputs import f32, make_qkv  # noqa: E402

MAX_ABS = 2e-2
REL_L2 = 5e-3
LSE_ABS = 1e-3
FA_ERR_SCRATCH = 10
STATIC_BYTES = 16 * 1024 * 1024

P = ctypes.c_void_p


def _static_fn():
    lib = fa.load_library()
    fn = lib.fa_fwd_splitkv_static
    i, f = ctypes.c_int, ctypes.c_float
    fn.argtypes = [P, P, P, P, P, i, i, i, i, i, f, i, i, P]
    fn.restype = i
    return fn


def test_rejects_partial_states_beyond_the_static_buffer():
    """Checked on the host before any CUDA call (fake pointers are never used)."""
    fn = _static_fn()
    fake = 0x10000
    # 1 x 8 heads x 128 rows x (128 + 2) floats x 64 splits = 34 MB > 16 MiB
    assert fa.fa_splitkv_workspace_bytes(1, 8, 128, 128, 64) > STATIC_BYTES
    st = fn(P(fake), P(fake), P(fake), P(fake), P(fake), 1, 8, 128, 4096, 128, 0.088, 0, 64, P(0))
    assert st == FA_ERR_SCRATCH
    assert fa.fa_status_string(st).startswith("FA_ERR_SCRATCH")
    assert fn(P(fake), P(fake), P(fake), P(0), P(fake), 1, 8, 128, 4096, 128, 0.088, 0, 4, P(0)) == 1
    assert fn(P(fake), P(fake), P(fake), P(fake), P(fake), 1, 8, 128, 4096, 96, 0.088, 0, 4, P(0)) == 4
    assert fn(P(fake), P(fake), P(fake), P(fake), P(fake), 1, 8, 128, 4096, 128, 0.088, 0, 0, P(0)) == 5


def test_refuses_misaligned_outputs_before_any_launch():
    """A misaligned o or lse, an unknown mask or a bad scale is refused on the
    host with the status fa_fwd would give, before the size test and before any
    CUDA call, so no work is queued (fake pointers are never used)."""
    fn = _static_fn()
    fake = 0x10000
    args = (1, 8, 128, 4096, 128)
    assert fn(P(fake), P(fake), P(fake), P(fake + 8), P(fake), *args, 0.088, 0, 4, P(0)) == 2
    assert fn(P(fake), P(fake), P(fake), P(fake), P(fake + 2), *args, 0.088, 0, 4, P(0)) == 2
    assert fn(P(fake), P(fake + 8), P(fake), P(fake), P(fake), *args, 0.088, 0, 4, P(0)) == 2
    assert fn(P(fake), P(fake), P(fake), P(fake), P(fake), *args, 0.088, 7, 4, P(0)) == 11
    assert fn(P(fake), P(fake), P(fake), P(fake), P(fake), *args, -1.0, 0, 4, P(0)) == 9
    # ... and the misaligned output is refused even when the partial states
    # would not fit the buffer either.
    assert fn(P(fake), P(fake), P(fake), P(fake + 8), P(fake), 1, 8, 128, 4096, 128, 0.088, 0, 64,
              P(0)) == 2


def _compare_oracle(o, lse, q, k, v, scale, causal):
    """Element by element against the float64 oracle."""
    import numpy as np

    import oracle
    from exact_attention_80_gb300.inputs import to_f64

    o_ref, lse_ref = oracle.attention_f64(to_f64(q.cpu()), to_f64(k.cpu()), to_f64(v.cpu()), scale,
                                          causal)
    got = o.float().cpu().numpy().astype(np.float64)
    max_abs = float(np.abs(got - o_ref).max())
    rel = float(np.linalg.norm(got - o_ref) / np.linalg.norm(o_ref))
    lerr = float(np.abs(lse.cpu().numpy() - lse_ref).max())
    assert max_abs <= MAX_ABS and rel <= REL_L2 and lerr <= LSE_ABS, (max_abs, rel, lerr)


def _compare(o, lse, o_ref, lse_ref):
    a, b = o.float(), o_ref.float()
    max_abs = (a - b).abs().max().item()
    rel = ((a - b).norm() / b.norm()).item()
    lerr = (lse - lse_ref).abs().max().item()
    assert max_abs <= MAX_ABS and rel <= REL_L2 and lerr <= LSE_ABS, (max_abs, rel, lerr)


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Nq,Nk,d,causal,splits", [
    (1, 8, 128, 8192, 128, False, 16),
    (2, 3, 300, 1000, 64, True, 4),
    (1, 2, 200, 777, 256, True, 3),
])
def test_static_scratch_matches_workspace_path(B, H, Nq, Nk, d, causal, splits):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    assert fa.fa_splitkv_workspace_bytes(B, H, Nq, d, splits) <= STATIC_BYTES
    fn = _static_fn()
    q, k, v = (t.cuda() for t in make_qkv(B, H, Nq, Nk, d, 90 + Nq + d))
    scale = f32(1.0 / math.sqrt(d))
    o_ref, lse_ref = fa.attention(q, k, v, causal=causal, scale=scale, num_splits=splits)
    stream = P(torch.cuda.current_stream().cuda_stream)
    for _ in range(2):  # two calls in a row share and reuse the static buffer
        o = torch.full_like(o_ref, float("nan"))
        lse = torch.full_like(lse_ref, float("nan"))
        st = fn(P(q.data_ptr()), P(k.data_ptr()), P(v.data_ptr()), P(o.data_ptr()),
                P(lse.data_ptr()), B, H, Nq, Nk, d, scale, int(causal), splits, stream)
        assert st == 0, fa.fa_status_string(st)
        torch.cuda.synchronize()
        assert fa.fa_device_status(clear=True) == fa.FA_OK
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        _compare(o, lse, o_ref, lse_ref)
        _compare_oracle(o, lse, q, k, v, scale, causal)
