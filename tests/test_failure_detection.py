"""Failure detection without a GPU fault: a bounded wait that nothing will
satisfy runs out, the kernel leaves through its abort path, the host reads
FA_ERR_TIMEOUT, and the same CUDA context then computes correctly.

The test hook (fa_test_fwd_withheld_q) withholds the Q tile loads, so the MMA
issuer's wait for Q can never complete; every wait is bounded, no MMA is issued
and no copy is left in flight."""

import ctypes
import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import exact_attention_80_gb300 as fa  # noqa: E402
import oracle  # noqa: E402
from exact_attention_80_gb300.inputs import f32, make_qkv, to_f64  # noqa: E402

P = ctypes.c_void_p
FA_ERR_SHAPE = 3
FA_ERR_TIMEOUT = 8


def _hook():
    lib = fa.load_library()
    fn = lib.fa_test_fwd_withheld_q
    i = ctypes.c_int
    fn.argtypes = [P, P, P, P, P, i, i, i, i, i, ctypes.c_longlong, P]
    fn.restype = i
    return fn


def test_hook_rejects_unbounded_or_tiny_limits():
    """Checked on the host before any CUDA call."""
    fn = _hook()
    fake = 0x10000
    for limit in (0, 1000, (1 << 31) + 1):
        assert fn(P(fake), P(fake), P(fake), P(fake), P(fake), 1, 1, 8, 8, 128, limit, P(0)) == FA_ERR_SHAPE


@pytest.mark.gpu
@pytest.mark.parametrize("d,persistent", [(128, False), (256, False), (128, True), (64, True)])
def test_bounded_wait_times_out_and_context_survives(d, persistent):
    """persistent: enough query units (four per SM) that the launch runs
    persistent CTAs, whose control warps carry the ring across units; their
    abort path is the one exercised."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    fn = _hook()
    B, H, Nq, Nk = 1, 2, 256, 300
    if persistent:
        sms = torch.cuda.get_device_properties(0).multi_processor_count
        Nq = 300                      # two 256-row units per head, the second ragged
        H = 2 * sms                   # 4 x SMs units
        assert fa.fa_fwd_grid_ctas(B, H, Nq, d, 1) >= 4 * sms
    q, k, v = (t.cuda() for t in make_qkv(B, H, Nq, Nk, d, 5150 + d))
    o = torch.full((B, H, Nq, d), 7.0, dtype=torch.bfloat16, device="cuda")
    lse = torch.full((B, H, Nq), 7.0, dtype=torch.float32, device="cuda")
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    stream = P(torch.cuda.current_stream().cuda_stream)
    st = fn(P(q.data_ptr()), P(k.data_ptr()), P(v.data_ptr()), P(o.data_ptr()), P(lse.data_ptr()),
            B, H, Nq, Nk, d, 1 << 22, stream)
    assert st == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == FA_ERR_TIMEOUT
    assert torch.all(o == 7.0) and torch.all(lse == 7.0)  # the aborted kernel wrote nothing
    # The context is intact: a normal call right after is correct.
    scale = f32(1.0 / math.sqrt(d))
    o2, lse2 = fa.attention(q, k, v, causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    o_ref, lse_ref = oracle.attention_f64(to_f64(q.cpu()), to_f64(k.cpu()), to_f64(v.cpu()), scale, True)
    err = np.abs(o2.float().cpu().numpy() - o_ref)
    assert err.max() <= 2e-2
    assert np.abs(lse2.cpu().numpy() - lse_ref).max() <= 1e-3
