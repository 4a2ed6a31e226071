"""Stream order with the forward kernels' dependent launch.

Every forward kernel and the split merge are launched with programmatic stream
serialization: a launch may be scheduled while the kernel before it in the
stream finishes, and waits for that kernel's completion before it reads or
writes memory. These tests chain calls that depend on each other's data on one
stream, with no synchronisation between them, and compare bit for bit with the
same calls separated by device-wide synchronisation.
"""

import pytest

torch = pytest.importorskip("torch")

import exact_attention_80_gb300 as fa  # noqa: E402
from exact_attention_80_gb300.inputs import make_qkv  # noqa: E402

pytestmark = pytest.mark.gpu


def _dev_qkv(B, H, Nq, Nk, d, seed):
    return tuple(t.cuda() for t in make_qkv(B, H, Nq, Nk, d, seed))


@pytest.mark.parametrize("B,H,N,d", [(2, 160, 300, 128), (1, 4, 1000, 64), (2, 8, 500, 256)])
def test_chained_forwards_read_the_previous_output(B, H, N, d):
    """o_{i+1} = attention(o_i, k, v): each forward's queries are the previous
    forward's output, launched back to back (persistent, one-unit and one-tile
    kernels)."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    q, k, v = _dev_qkv(B, H, N, N, d, 6100 + d)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    outs = [torch.empty_like(q) for _ in range(6)]
    src = q
    for o in outs:  # no synchronisation between the calls
        fa.fa_fwd(src, k, v, o, lse, True)
        src = o
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    src = q
    for o in outs:
        ref = torch.empty_like(q)
        fa.fa_fwd(src, k, v, ref, lse, True)
        torch.cuda.synchronize()
        assert torch.equal(ref, o)
        src = ref


def test_forward_after_a_kernel_that_rewrites_its_inputs():
    """A PyTorch kernel rewrites Q and V right before each forward on the same
    stream; the forward sees the new values."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    B, H, N, d = 2, 160, 300, 128
    q, k, v = _dev_qkv(B, H, N, N, d, 6200)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    got = []
    for i in range(4):
        q.mul_(0.5)
        v.add_(1.0)
        fa.fa_fwd(q, k, v, o, lse, False)
        got.append((o.clone(), lse.clone()))
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    q2, k2, v2 = _dev_qkv(B, H, N, N, d, 6200)
    for i in range(4):
        q2.mul_(0.5)
        v2.add_(1.0)
        torch.cuda.synchronize()
        o2 = torch.empty_like(q2)
        lse2 = torch.empty_like(lse)
        fa.fa_fwd(q2, k2, v2, o2, lse2, False)
        torch.cuda.synchronize()
        assert torch.equal(got[i][0], o2) and torch.equal(got[i][1], lse2)


def test_split_merge_then_forward_chain():
    """Split-KV partials, their merge, then a forward whose queries are the
    merged output, repeated back to back on one stream."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    B, H, Nq, Nk, d, S = 1, 16, 64, 4000, 128, 8
    q, k, v = _dev_qkv(B, H, Nq, Nk, d, 6300)
    ws = torch.empty(fa.fa_splitkv_workspace_bytes(B, H, Nq, d, S) // 4, device="cuda")
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")

    def chain(sync):
        src, res = q, []
        for _ in range(3):
            m = torch.empty_like(q)
            fa.fa_fwd_splitkv(src, k, v, ws, S, False)
            if sync:
                torch.cuda.synchronize()
            fa.fa_combine(ws, m, lse, B, H, Nq, d, S)
            if sync:
                torch.cuda.synchronize()
            o = torch.empty_like(q)
            fa.fa_fwd(m, k, v, o, lse, False)
            if sync:
                torch.cuda.synchronize()
            res += [m, o]
            src = o
        torch.cuda.synchronize()
        return res

    fast = chain(False)
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    slow = chain(True)
    for a, b in zip(fast, slow):
        assert torch.equal(a, b)
