"""The forward calls captured in a CUDA graph.

A serving loop captures its launches once and replays them. The calls here
take only pointers and sizes and allocate nothing once warmed up, so they may
be captured. The split-KV merge is launched with programmatic stream
serialization after the split kernel, which a capture turns into a
programmatic graph edge. Each case captures a few calls in one graph, copies new
inputs into the captured buffers, replays, and checks bit for bit against the
same calls made eagerly on those inputs, and a few heads against the float64
oracle.
"""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import exact_attention_80_gb300 as fa  # noqa: E402
import oracle  # noqa: E402
from exact_attention_80_gb300.inputs import f32, make_qkv, to_f64  # noqa: E402

pytestmark = pytest.mark.gpu

MAX_ABS = 2e-2
LSE_ABS = 1e-3
STATIC_BYTES = 16 * 1024 * 1024  # FA_STATIC_SCRATCH_BYTES (include/fa.h)


def _check_heads(q, k, v, o, lse, scale, causal, heads):
    for b, h in heads:
        o_ref, lse_ref = oracle.attention_f64(to_f64(q[b, h]), to_f64(k[b, h]), to_f64(v[b, h]), scale, causal)
        assert np.abs(o[b, h].float().cpu().numpy() - o_ref).max() <= MAX_ABS
        assert np.abs(lse[b, h].cpu().numpy() - lse_ref).max() <= LSE_ABS


def _static_fits(B, H, Nq, d):
    return fa.fa_splitkv_workspace_bytes(B, H, Nq, d, 2) <= STATIC_BYTES


def _calls(q, k, v, outs, ws, splits, causal, scale, stream):
    o1, l1, o2, l2, o3, l3 = outs
    B, H, Nq, d = q.shape
    fa.fa_fwd(q, k, v, o1, l1, causal, scale, stream=stream)
    fa.fa_fwd_splitkv(q, k, v, ws, splits, causal, scale, stream=stream)
    fa.fa_combine(ws, o2, l2, B, H, Nq, d, splits, stream=stream)
    if _static_fits(B, H, Nq, d):  # the library's scratch holds the partial states
        fa.fa_fwd_splitkv_static(q, k, v, o3, l3, 2, causal, scale, stream=stream)


@pytest.mark.parametrize("B,H,Nq,Nk,splits,causal", [
    (2, 160, 300, 333, 3, True),          # persistent forward; split CTAs of two tiles
    (1, 16, 64, 4000, 8, "bottom_right"),  # decode shape: dual-range split CTAs; static scratch
])
def test_graph_replay_matches_eager(B, H, Nq, Nk, splits, causal):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    d = 128
    scale = f32(1.0 / math.sqrt(d))
    dev = torch.device("cuda", 0)
    q, k, v = (t.to(dev) for t in make_qkv(B, H, Nq, Nk, d, 8100 + Nq))
    mk = lambda: (torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=dev),  # noqa: E731
                  torch.empty((B, H, Nq), dtype=torch.float32, device=dev))
    outs = [t for _ in range(3) for t in mk()]
    ws = torch.empty(fa.fa_splitkv_workspace_bytes(B, H, Nq, d, splits) // 4, device=dev)

    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize()  # inputs and outputs made on the default stream
    with torch.cuda.stream(stream):
        _calls(q, k, v, outs, ws, splits, causal, scale, stream)  # warm-up (kernel attributes, scratch)
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        _calls(q, k, v, outs, ws, splits, causal, scale, torch.cuda.current_stream(dev))

    # New inputs into the captured buffers, then replay.
    q2, k2, v2 = (t.to(dev) for t in make_qkv(B, H, Nq, Nk, d, 8200 + Nq))
    q.copy_(q2)
    k.copy_(k2)
    v.copy_(v2)
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    replayed = [t.clone() for t in outs]
    torch.cuda.synchronize()  # the clones are read before the eager calls overwrite the outputs

    # The same calls made eagerly on the new inputs.
    with torch.cuda.stream(stream):
        _calls(q, k, v, outs, ws, splits, causal, scale, stream)
    stream.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    # Outputs the calls wrote (the allocation-free call runs only where its
    # partial states fit the library's scratch; unwritten buffers hold stale
    # bits, NaN patterns included).
    written = 6 if _static_fits(B, H, Nq, d) else 4
    for a, b in zip(replayed[:written], outs[:written]):
        assert torch.equal(a, b)

    qc, kc, vc = q.cpu(), k.cpu(), v.cpu()
    heads = [(0, 0), (B - 1, H - 1)]
    for i in range(3 if _static_fits(B, H, Nq, d) else 2):
        _check_heads(qc, kc, vc, replayed[2 * i].cpu(), replayed[2 * i + 1].cpu(), scale, causal, heads)


def test_graph_replay_backward_fp8_varlen():
    """The backward, the e4m3 forward and the variable-length forward captured
    in one graph (caller-owned outputs and workspaces), replayed on new inputs
    and compared bit for bit with the same calls made eagerly."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    from exact_attention_80_gb300.inputs import make_grad_output, make_qkv_fp8, make_varlen

    dev = torch.device("cuda", 0)
    B, H, N, d = 2, 4, 300, 128
    scale = f32(1.0 / math.sqrt(d))
    ds = 2.0 ** -5
    lq, lk = [100, 0, 257, 33], [90, 5, 300, 200]
    # Captured buffers: inputs are refilled in place before the replay.
    q, k, v = (t.to(dev) for t in make_qkv(B, H, N, N, d, 8300))
    do = make_grad_output(B, H, N, d, 8301).to(dev)
    q8, k8, v8 = (t.to(dev) for t in make_qkv_fp8(B, H, N, N, d, 8302))
    qv, kv, vv, cu_q, cu_k = make_varlen(lq, lk, H, d, 8303)
    qv, kv, vv, cu_q, cu_k = (t.to(dev) for t in (qv, kv, vv, cu_q, cu_k))
    o, lse = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=dev)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fa_bwd_workspace_bytes(B, H, N, d) // 4, dtype=torch.float32, device=dev)
    o8, lse8 = torch.empty_like(q), torch.empty((B, H, N), dtype=torch.float32, device=dev)
    ov = torch.empty_like(qv)
    lsev = torch.empty((H, qv.shape[0]), dtype=torch.float32, device=dev)
    outs = (o, lse, dq, dk, dv, o8, lse8, ov, lsev)

    def calls(st):
        fa.fa_fwd(q, k, v, o, lse, True, scale, stream=st)
        fa.fa_bwd(q, k, v, o, do, lse, dq, dk, dv, ws, True, scale, stream=st)
        fa.fa_fwd_fp8(q8, k8, v8, ds, ds, ds, o8, lse8, False, scale, stream=st)
        fa.fa_fwd_varlen(qv, kv, vv, ov, lsev, cu_q, cu_k, max(lq), "bottom_right", scale, stream=st)

    stream = torch.cuda.Stream(dev)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        calls(stream)  # warm-up
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        calls(torch.cuda.current_stream(dev))

    q.copy_(make_qkv(B, H, N, N, d, 8400)[0].to(dev))
    do.copy_(make_grad_output(B, H, N, d, 8401).to(dev))
    q8.copy_(make_qkv_fp8(B, H, N, N, d, 8402)[0].to(dev))
    vv.copy_(make_varlen(lq, lk, H, d, 8403)[2].to(dev))
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    replayed = [t.clone() for t in outs]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        calls(stream)
    stream.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    for name, a, b in zip(("o", "lse", "dq", "dk", "dv", "o8", "lse8", "ov", "lsev"), replayed, outs):
        assert torch.equal(a, b), name
    # The replay ran on the new inputs: its output differs from the warm-up's.
    o_ref, _ = oracle.attention_f64(to_f64(q[0, 0].cpu()), to_f64(k[0, 0].cpu()), to_f64(v[0, 0].cpu()),
                                    scale, True)
    assert np.abs(replayed[0][0, 0].float().cpu().numpy() - o_ref).max() <= MAX_ABS
