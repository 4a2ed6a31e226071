"""The Python binding checks every tensor before it hands a bare pointer to the
library: outputs and workspaces of the wrong dtype, shape, layout or size are
refused. CPU only: the library's compute entry points are replaced by stubs
that launch nothing (its host-only size functions are the real ones), and CPU
tensors stand in for device tensors."""

import pytest

import exact_attention_80_gb300 as fa

torch = pytest.importorskip("torch")


class _StubLib:
    """Compute entry points that return FA_OK without doing anything."""

    def __init__(self, real):
        self._real = real
        self.calls = []

    def __getattr__(self, name):
        if name in ("fa_splitkv_workspace_bytes", "fa_bwd_workspace_bytes", "fa_status_string"):
            return getattr(self._real, name)

        def stub(*args):
            self.calls.append(name)
            return 0
        stub.argtypes = None
        return stub


@pytest.fixture
def stub(monkeypatch):
    if torch.cuda.is_available():
        pytest.skip("CPU tensors stand in for device tensors only where no GPU exists")
    real = fa.load_library()
    lib = _StubLib(real)
    monkeypatch.setattr(fa, "load_library", lambda: lib)
    monkeypatch.setattr(torch.Tensor, "is_cuda", property(lambda self: True))
    return lib


def bf16(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


def f32(*shape):
    return torch.zeros(shape, dtype=torch.float32)


B, H, NQ, NK, D = 2, 3, 130, 200, 128


def test_forward_outputs_checked(stub):
    q, k, v = bf16(B, H, NQ, D), bf16(B, H, NK, D), bf16(B, H, NK, D)
    fa.fa_fwd(q, k, v, bf16(B, H, NQ, D), f32(B, H, NQ), stream=0)
    assert stub.calls == ["fa_fwd"]
    with pytest.raises(ValueError):
        fa.fa_fwd(q, k, v, bf16(B, H, NQ, 64), f32(B, H, NQ), stream=0)
    with pytest.raises(ValueError):
        fa.fa_fwd(q, k, v, bf16(B, H, NQ + 1, D), f32(B, H, NQ), stream=0)
    with pytest.raises(TypeError):
        fa.fa_fwd(q, k, v, f32(B, H, NQ, D), f32(B, H, NQ), stream=0)
    with pytest.raises(TypeError):
        fa.fa_fwd(q, k, v, bf16(B, H, NQ, D), bf16(B, H, NQ), stream=0)
    with pytest.raises(ValueError):
        fa.fa_fwd(q, k, v, bf16(B, H, D, NQ).transpose(2, 3), f32(B, H, NQ), stream=0)
    with pytest.raises(TypeError):
        fa.fa_fwd(q, k, v, None, f32(B, H, NQ), stream=0)
    assert stub.calls == ["fa_fwd"]  # nothing refused reached the library


def test_split_and_combine_workspace_checked(stub):
    q, k, v = bf16(B, H, NQ, D), bf16(B, H, NK, D), bf16(B, H, NK, D)
    S = 3
    nbytes = fa.fa_splitkv_workspace_bytes(B, H, NQ, D, S)
    ws = f32(nbytes // 4)
    fa.fa_fwd_splitkv(q, k, v, ws, S, stream=0)
    fa.fa_combine(ws, bf16(B, H, NQ, D), f32(B, H, NQ), B, H, NQ, D, S, stream=0)
    assert stub.calls == ["fa_fwd_splitkv", "fa_combine"]
    with pytest.raises(ValueError):
        fa.fa_fwd_splitkv(q, k, v, f32(nbytes // 4 - 1), S, stream=0)
    with pytest.raises(TypeError):
        fa.fa_fwd_splitkv(q, k, v, torch.zeros(nbytes // 4, dtype=torch.float64), S, stream=0)
    with pytest.raises(ValueError):
        fa.fa_combine(f32(nbytes // 4 - 4), bf16(B, H, NQ, D), f32(B, H, NQ), B, H, NQ, D, S, stream=0)
    with pytest.raises(ValueError):
        fa.fa_combine(ws, bf16(B, H, NQ, D), f32(B, H, NQ + 2), B, H, NQ, D, S, stream=0)
    assert stub.calls == ["fa_fwd_splitkv", "fa_combine"]


def test_e4m3_outputs_checked(stub):
    d = 128
    q8 = torch.zeros((B, H, NQ, d), dtype=torch.uint8)
    k8 = torch.zeros((B, H, NK, d), dtype=torch.uint8)
    fa.fa_fwd_fp8(q8, k8, k8, 1.0, 1.0, 1.0, bf16(B, H, NQ, d), f32(B, H, NQ), stream=0)
    nbytes = fa.fa_splitkv_workspace_bytes(B, H, NQ, d, 4)
    fa.fa_fwd_fp8_splitkv(q8, k8, k8, 1.0, 1.0, 1.0, f32(nbytes // 4), 4, stream=0)
    assert stub.calls == ["fa_fwd_fp8", "fa_fwd_fp8_splitkv"]
    with pytest.raises(ValueError):
        fa.fa_fwd_fp8(q8, k8, k8, 1.0, 1.0, 1.0, bf16(B, H, NK, d), f32(B, H, NQ), stream=0)
    with pytest.raises(ValueError):
        fa.fa_fwd_fp8_splitkv(q8, k8, k8, 1.0, 1.0, 1.0, f32(16), 4, stream=0)


def test_backward_tensors_checked(stub):
    q, k, v = bf16(B, H, NQ, D), bf16(B, H, NK, D), bf16(B, H, NK, D)
    o, do, lse = bf16(B, H, NQ, D), bf16(B, H, NQ, D), f32(B, H, NQ)
    dq, dk, dv = bf16(B, H, NQ, D), bf16(B, H, NK, D), bf16(B, H, NK, D)
    ws = f32(fa.fa_bwd_workspace_bytes(B, H, NQ, D) // 4)
    fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, stream=0)
    assert stub.calls == ["fa_bwd"]
    bad = [
        dict(dq=bf16(B, H, NK, D)),                       # dq shaped like k
        dict(dk=bf16(B, H, NQ, D)),                       # dk shaped like q
        dict(dv=bf16(B, H, NK, 64)),
        dict(dout=bf16(B, H, NQ, 64)),
        dict(lse=f32(B, H, NK)),
        dict(workspace=f32(ws.numel() - 1)),              # one float short
        dict(workspace=f32(B * H * NQ * (D + 1))),        # unpadded rows: too small
    ]
    args = dict(o=o, dout=do, lse=lse, dq=dq, dk=dk, dv=dv, workspace=ws)
    for change in bad:
        a = dict(args, **change)
        with pytest.raises((ValueError, TypeError)):
            fa.fa_bwd(q, k, v, a["o"], a["dout"], a["lse"], a["dq"], a["dk"], a["dv"], a["workspace"],
                      stream=0)
    assert stub.calls == ["fa_bwd"]


def test_varlen_tensors_checked(stub):
    h, d = 2, 64
    q, k = bf16(150, h, d), bf16(200, h, d)
    cu = torch.tensor([0, 100, 150], dtype=torch.int32)
    cu_k = torch.tensor([0, 80, 200], dtype=torch.int32)
    fa.fa_fwd_varlen(q, k, k, bf16(150, h, d), f32(h, 150), cu, cu_k, 100, stream=0)
    assert stub.calls == ["fa_fwd_varlen"]
    with pytest.raises(ValueError):
        fa.fa_fwd_varlen(q, k, k, bf16(150, h, d), f32(150, h), cu, cu_k, 100, stream=0)
    with pytest.raises(ValueError):
        fa.fa_fwd_varlen(q, k, k, bf16(149, h, d), f32(h, 150), cu, cu_k, 100, stream=0)
    with pytest.raises(ValueError):
        fa.fa_fwd_varlen(q, k, bf16(199, h, d), bf16(150, h, d), f32(h, 150), cu, cu_k, 100, stream=0)
    assert stub.calls == ["fa_fwd_varlen"]


def test_static_scratch_outputs_checked(stub):
    q, k = bf16(1, 2, 64, 128), bf16(1, 2, 300, 128)
    fa.fa_fwd_splitkv_static(q, k, k, bf16(1, 2, 64, 128), f32(1, 2, 64), 4, stream=0)
    with pytest.raises(ValueError):
        fa.fa_fwd_splitkv_static(q, k, k, bf16(1, 2, 64, 128), f32(1, 2, 63), 4, stream=0)
    assert stub.calls == ["fa_fwd_splitkv_static"]


@pytest.mark.parametrize("BH,chunks", [(256, 8), (256, 1), (256, 2), (256, 3), (256, 12), (3, 8),
                                       (1, 8), (7, 5), (5, 5), (1000, 64)])
def test_head_slices_cover_the_heads(BH, chunks):
    """fa_fwd_from_host's slices: consecutive, non-empty, covering [0, BH), at
    most `chunks` of them; with three or more, the last two are no larger than
    the ones before them."""
    b = fa.head_slices(BH, chunks)
    assert 1 <= len(b) <= min(chunks, BH)
    assert b[0][0] == 0 and b[-1][1] == BH
    assert all(h0 < h1 for h0, h1 in b)
    assert all(b[i][1] == b[i + 1][0] for i in range(len(b) - 1))
    sizes = [h1 - h0 for h0, h1 in b]
    if min(chunks, BH) >= 3 and BH >= 4 * chunks:
        assert sizes[-1] <= sizes[-2] <= min(sizes[:-2])
        assert sizes[-1] < max(sizes)
