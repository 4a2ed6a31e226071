"""GB300 (sm_103a) exact attention (forward, split-KV merge, e4m3 forward,
backward): Python binding of ``libfa_gb300.so``.

The functions below carry the names of the C ABI in ``include/fa.h`` and only
marshal arguments: every step of the computation runs in the library's CUDA
kernels. PyTorch supplies device memory and the current CUDA stream. The
library receives bare pointers and cannot see a buffer's size, so the binding
checks every tensor's dtype, shape, device and layout before the call. There is
no fallback: if the library is missing or a call fails, an exception says so.
"""

from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfa_gb300.so")

FA_OK = 0
FA_ERR_SEQLENS = 12
STATUS_NAMES = {
    0: "FA_OK", 1: "FA_ERR_NULL", 2: "FA_ERR_ALIGN", 3: "FA_ERR_SHAPE", 4: "FA_ERR_HEADDIM",
    5: "FA_ERR_SPLITS", 6: "FA_ERR_WORKSPACE", 7: "FA_ERR_CUDA", 8: "FA_ERR_TIMEOUT",
    9: "FA_ERR_SCALE", 10: "FA_ERR_SCRATCH", 11: "FA_ERR_CAUSAL", 12: "FA_ERR_SEQLENS",
    13: "FA_ERR_TILE",
}
# Causal mask modes (include/fa.h): key j visible to query i iff j <= i (top-left)
# or j <= i + Nk - Nq (bottom-right).
CAUSAL_NONE, CAUSAL_TOP_LEFT, CAUSAL_BOTTOM_RIGHT = 0, 1, 2
_CAUSAL_NAMES = {"none": 0, "top_left": 1, "bottom_right": 2}
FA_MAX_SPLITS = 256

_lib = None


class FAError(RuntimeError):
    """A library call returned a status other than FA_OK."""

    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {fa_status_string(status)}")


def load_library() -> ctypes.CDLL:
    """Load the in-tree CUDA library (build it with ``exact_attention_80_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it with `python -m exact_attention_80_gb300.build`")
    try:  # make torch's CUDA runtime the one the library binds to
        import torch  # noqa: F401
    except ImportError:
        pass
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_fwd.restype = i
    lib.fa_fwd_rows.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
    lib.fa_fwd_rows.restype = i
    lib.fa_splitkv_workspace_bytes.argtypes = [i, i, i, i, i]
    lib.fa_splitkv_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_fwd_splitkv.argtypes = [vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
    lib.fa_fwd_splitkv.restype = i
    lib.fa_combine.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
    lib.fa_combine.restype = i
    lib.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp]
    lib.fa_fwd_varlen.restype = i
    lib.fa_fwd_fp8.argtypes = [vp, vp, vp, f, f, f, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_fwd_fp8.restype = i
    lib.fa_fwd_fp8_splitkv.argtypes = [vp, vp, vp, f, f, f, vp, i, i, i, i, i, f, i, i, vp]
    lib.fa_fwd_fp8_splitkv.restype = i
    lib.fa_bwd_workspace_bytes.argtypes = [i, i, i, i]
    lib.fa_bwd_workspace_bytes.restype = ctypes.c_size_t
    lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
    lib.fa_bwd.restype = i
    lib.fa_fwd_grid_ctas.argtypes = [i, i, i, i, i]
    lib.fa_fwd_grid_ctas.restype = ctypes.c_longlong
    lib.fa_device_status.argtypes = [vp, i]
    lib.fa_device_status.restype = i
    lib.fa_status_string.argtypes = [i]
    lib.fa_status_string.restype = ctypes.c_char_p
    _lib = lib
    return lib


def fa_status_string(status: int) -> str:
    return load_library().fa_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != FA_OK:
        raise FAError(status, what)


def _stream_handle(stream):
    import torch

    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _need(t, name, shape, dtype, device):
    """Raise unless ``t`` is a contiguous tensor of ``dtype`` and ``shape`` on
    ``device``: the library writes through a bare pointer."""
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.device != device or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous tensor on {device}")
    if tuple(t.shape) != tuple(int(x) for x in shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")


def _need_workspace(t, nbytes: int, name: str, device):
    """Raise unless ``t`` is a contiguous float32 tensor on ``device`` of at least
    ``nbytes`` bytes (0: the arguments are out of range, for the library to
    reject)."""
    import torch

    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32, got {t.dtype}")
    if t.device != device or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous tensor on {device}")
    if nbytes > 0 and t.numel() * 4 < nbytes:
        raise ValueError(f"{name} holds {t.numel() * 4} bytes; the call needs {nbytes}")


def _bhnd(q, k, v):
    import torch

    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype != torch.bfloat16:
            raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
        if t.dim() != 4 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CUDA tensor [B, H, N, d]")
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k and v must be on the same device")
    B, H, Nq, d = q.shape
    if k.shape[:2] != (B, H) or k.shape[3] != d or v.shape != k.shape:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    return int(B), int(H), int(Nq), int(k.shape[2]), int(d)


def _need_o_lse(o, lse, B, H, Nq, d, device):
    import torch

    _need(o, "o", (B, H, Nq, d), torch.bfloat16, device)
    _need(lse, "lse", (B, H, Nq), torch.float32, device)


def causal_code(causal) -> int:
    """The C-ABI causal value: ``False``/``True`` (top-left), 0/1/2, or one of
    ``"none"``, ``"top_left"``, ``"bottom_right"``. Other values pass through as
    given, for the library to reject (FA_ERR_CAUSAL)."""
    if isinstance(causal, str):
        if causal not in _CAUSAL_NAMES:
            raise ValueError(f"unknown causal mode {causal!r}")
        return _CAUSAL_NAMES[causal]
    if isinstance(causal, bool):
        return CAUSAL_TOP_LEFT if causal else CAUSAL_NONE
    return int(causal)


def default_scale(d: int) -> float:
    """1/sqrt(d) rounded once to float32 (the value the kernel receives)."""
    return float(ctypes.c_float(d ** -0.5).value)


def fa_fwd(q, k, v, o, lse, causal=False, scale: float | None = None, stream=None):
    """Fused forward into caller-owned ``o`` (bf16 [B,H,Nq,d]) and ``lse`` (fp32 [B,H,Nq])."""
    B, H, Nq, Nk, d = _bhnd(q, k, v)
    _need_o_lse(o, lse, B, H, Nq, d, q.device)
    scale = default_scale(d) if scale is None else float(scale)
    st = load_library().fa_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
                               scale, causal_code(causal), _stream_handle(stream))
    _check(st, "fa_fwd")


def fa_fwd_rows(q, k, v, o, lse, rows_per_cta: int, causal=False, scale: float | None = None,
                stream=None):
    """:func:`fa_fwd` with ``rows_per_cta`` query rows per CTA (include/fa.h,
    fa_fwd_rows: 64, 128 or 256 at d <= 128, 128 at d = 256)."""
    B, H, Nq, Nk, d = _bhnd(q, k, v)
    _need_o_lse(o, lse, B, H, Nq, d, q.device)
    scale = default_scale(d) if scale is None else float(scale)
    st = load_library().fa_fwd_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
                                    scale, causal_code(causal), int(rows_per_cta),
                                    _stream_handle(stream))
    _check(st, "fa_fwd_rows")


def _bhnd8(q, k, v):
    import torch

    ok_types = (torch.uint8, torch.float8_e4m3fn)
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.dtype not in ok_types:
            raise TypeError(f"{name} must hold e4m3 codes (uint8 or float8_e4m3fn), got {t.dtype}")
        if t.dim() != 4 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError(f"{name} must be a contiguous CUDA tensor [B, H, N, d]")
    if k.device != q.device or v.device != q.device:
        raise ValueError("q, k and v must be on the same device")
    B, H, Nq, d = q.shape
    if k.shape[:2] != (B, H) or k.shape[3] != d or v.shape != k.shape:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)}")
    return int(B), int(H), int(Nq), int(k.shape[2]), int(d)


def fa_fwd_fp8(q, k, v, q_descale: float, k_descale: float, v_descale: float, o, lse,
               causal=False, scale: float | None = None, stream=None):
    """Fused forward on e4m3 inputs (include/fa.h, fa_fwd_fp8): ``q``, ``k``, ``v``
    hold e4m3 codes [B,H,N,d] (uint8 or float8_e4m3fn), the value of a code being
    its e4m3 value times the tensor's descale; ``o`` bf16 [B,H,Nq,d] and ``lse``
    fp32 [B,H,Nq] are written."""
    B, H, Nq, Nk, d = _bhnd8(q, k, v)
    _need_o_lse(o, lse, B, H, Nq, d, q.device)
    scale = default_scale(d) if scale is None else float(scale)
    st = load_library().fa_fwd_fp8(_ptr(q), _ptr(k), _ptr(v), float(q_descale), float(k_descale),
                                   float(v_descale), _ptr(o), _ptr(lse), B, H, Nq, Nk, d, scale,
                                   causal_code(causal), _stream_handle(stream))
    _check(st, "fa_fwd_fp8")


def fa_fwd_fp8_splitkv(q, k, v, q_descale: float, k_descale: float, v_descale: float, workspace,
                       num_splits: int, causal=False, scale: float | None = None, stream=None):
    """Split-KV forward on e4m3 inputs into ``workspace`` (fp32, at least
    ``fa_splitkv_workspace_bytes`` bytes); merge with :func:`fa_combine`."""
    B, H, Nq, Nk, d = _bhnd8(q, k, v)
    _need_workspace(workspace, fa_splitkv_workspace_bytes(B, H, Nq, d, int(num_splits)), "workspace",
                    q.device)
    scale = default_scale(d) if scale is None else float(scale)
    st = load_library().fa_fwd_fp8_splitkv(_ptr(q), _ptr(k), _ptr(v), float(q_descale),
                                           float(k_descale), float(v_descale), _ptr(workspace), B, H,
                                           Nq, Nk, d, scale, causal_code(causal), int(num_splits),
                                           _stream_handle(stream))
    _check(st, "fa_fwd_fp8_splitkv")


def attention_fp8(q, k, v, q_descale: float = 1.0, k_descale: float = 1.0, v_descale: float = 1.0,
                  causal=False, scale: float | None = None, num_splits: int = 1, stream=None):
    """Allocate bf16 ``o`` and fp32 ``lse`` and run :func:`fa_fwd_fp8`, or, with
    ``num_splits > 1``, :func:`fa_fwd_fp8_splitkv` and :func:`fa_combine`."""
    import torch

    B, H, Nq, Nk, d = _bhnd8(q, k, v)
    o = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if num_splits == 1:
        fa_fwd_fp8(q, k, v, q_descale, k_descale, v_descale, o, lse, causal, scale, stream)
    else:
        ws = torch.empty(fa_splitkv_workspace_bytes(B, H, Nq, d, num_splits) // 4,
                         dtype=torch.float32, device=q.device)
        fa_fwd_fp8_splitkv(q, k, v, q_descale, k_descale, v_descale, ws, num_splits, causal, scale,
                           stream)
        fa_combine(ws, o, lse, B, H, Nq, d, num_splits, stream)
    return o, lse


def fa_bwd_workspace_bytes(B: int, H: int, Nq: int, d: int) -> int:
    return int(load_library().fa_bwd_workspace_bytes(B, H, Nq, d))


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, causal=False,
           scale: float | None = None, stream=None):
    """Backward into caller-owned ``dq``, ``dk``, ``dv`` (bf16, shaped like q, k,
    v), from bf16 ``o`` and ``dout`` and the forward's fp32 ``lse``; ``workspace``
    fp32 of at least ``fa_bwd_workspace_bytes`` bytes (include/fa.h, fa_bwd)."""
    import torch

    B, H, Nq, Nk, d = _bhnd(q, k, v)
    dev = q.device
    _need(o, "o", (B, H, Nq, d), torch.bfloat16, dev)
    _need(dout, "dout", (B, H, Nq, d), torch.bfloat16, dev)
    _need(lse, "lse", (B, H, Nq), torch.float32, dev)
    _need(dq, "dq", (B, H, Nq, d), torch.bfloat16, dev)
    _need(dk, "dk", (B, H, Nk, d), torch.bfloat16, dev)
    _need(dv, "dv", (B, H, Nk, d), torch.bfloat16, dev)
    _need_workspace(workspace, fa_bwd_workspace_bytes(B, H, Nq, d), "workspace", dev)
    scale = default_scale(d) if scale is None else float(scale)
    st = load_library().fa_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq),
                               _ptr(dk), _ptr(dv), _ptr(workspace), B, H, Nq, Nk, d, scale,
                               causal_code(causal), _stream_handle(stream))
    _check(st, "fa_bwd")


def attention_backward(q, k, v, o, lse, dout, causal=False, scale: float | None = None,
                       stream=None):
    """Allocate ``(dq, dk, dv)`` and the workspace and run :func:`fa_bwd`."""
    import torch

    B, H, Nq, Nk, d = _bhnd(q, k, v)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(max(1, fa_bwd_workspace_bytes(B, H, Nq, d) // 4), dtype=torch.float32,
                     device=q.device)
    fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, ws, causal, scale, stream)
    return dq, dk, dv


def fa_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, causal=False,
                  scale: float | None = None, stream=None):
    """Forward over packed variable-length sequences: ``q``/``o`` bf16
    [total_q, H, d], ``k``/``v`` bf16 [total_k, H, d], ``lse`` fp32 [H, total_q],
    ``cu_seqlens_*`` int32 [B+1] on the device (include/fa.h, fa_fwd_varlen)."""
    import torch

    for t in (q, k, v, o):
        if t.dtype != torch.bfloat16 or t.dim() != 3 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("q, k, v, o must be contiguous CUDA bf16 [tokens, H, d]")
    for t in (cu_seqlens_q, cu_seqlens_k):
        if t.dtype != torch.int32 or t.dim() != 1 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("cu_seqlens must be contiguous CUDA int32 [B+1]")
    if lse.dtype != torch.float32 or not lse.is_contiguous() or not lse.is_cuda:
        raise ValueError("lse must be contiguous CUDA fp32 [H, total_q]")
    if any(t.device != q.device for t in (k, v, o, lse, cu_seqlens_q, cu_seqlens_k)):
        raise ValueError("every tensor must be on q's device")
    total_q, H, d = (int(x) for x in q.shape)
    total_k = int(k.shape[0])
    if tuple(o.shape) != tuple(q.shape) or tuple(k.shape) != (total_k, H, d) or v.shape != k.shape:
        raise ValueError(f"shape mismatch q{tuple(q.shape)} k{tuple(k.shape)} v{tuple(v.shape)} "
                         f"o{tuple(o.shape)}")
    if tuple(lse.shape) != (H, total_q):
        raise ValueError(f"lse must have shape {(H, total_q)}, got {tuple(lse.shape)}")
    B = int(cu_seqlens_q.shape[0]) - 1
    if int(cu_seqlens_k.shape[0]) != B + 1 or B < 1:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must both have B+1 >= 2 entries")
    scale = default_scale(d) if scale is None else float(scale)
    st = load_library().fa_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                      _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B, H, total_q,
                                      total_k, int(max_seqlen_q), d, scale, causal_code(causal),
                                      _stream_handle(stream))
    _check(st, "fa_fwd_varlen")


def attention_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, causal=False,
                     scale: float | None = None, stream=None):
    """Allocate ``o`` [total_q, H, d] and ``lse`` [H, total_q] and run
    :func:`fa_fwd_varlen`. Returns ``(o, lse)``."""
    import torch

    o = torch.empty_like(q)
    lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    fa_fwd_varlen(q, k, v, o, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q, causal, scale, stream)
    return o, lse


def fa_splitkv_workspace_bytes(B: int, H: int, Nq: int, d: int, num_splits: int) -> int:
    return int(load_library().fa_splitkv_workspace_bytes(B, H, Nq, d, num_splits))


def fa_fwd_splitkv(q, k, v, workspace, num_splits: int, causal=False,
                   scale: float | None = None, stream=None):
    """Split-KV partial states into ``workspace`` (see include/fa.h for the layout)."""
    B, H, Nq, Nk, d = _bhnd(q, k, v)
    _need_workspace(workspace, fa_splitkv_workspace_bytes(B, H, Nq, d, int(num_splits)), "workspace",
                    q.device)
    scale = default_scale(d) if scale is None else float(scale)
    st = load_library().fa_fwd_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(workspace), B, H, Nq, Nk,
                                       d, scale, causal_code(causal), int(num_splits),
                                       _stream_handle(stream))
    _check(st, "fa_fwd_splitkv")


def fa_combine(workspace, o, lse, B: int, H: int, Nq: int, d: int, num_splits: int,
               stream=None):
    """Merge partial states from ``workspace`` into ``o`` and ``lse``."""
    _need_o_lse(o, lse, B, H, Nq, d, o.device if hasattr(o, "device") else None)
    _need_workspace(workspace, fa_splitkv_workspace_bytes(int(B), int(H), int(Nq), int(d), int(num_splits)),
                    "workspace", o.device)
    st = load_library().fa_combine(_ptr(workspace), _ptr(o), _ptr(lse), int(B), int(H), int(Nq),
                                   int(d), int(num_splits), _stream_handle(stream))
    _check(st, "fa_combine")


def fa_fwd_grid_ctas(B: int, H: int, Nq: int, d: int, num_splits: int = 1) -> int:
    return int(load_library().fa_fwd_grid_ctas(B, H, Nq, d, num_splits))


def fa_device_status(clear: bool = True, stream=None) -> int:
    """Synchronises the stream and returns the device status (FA_OK or FA_ERR_TIMEOUT)."""
    return int(load_library().fa_device_status(_stream_handle(stream), int(bool(clear))))


def attention(q, k, v, causal=False, scale: float | None = None, num_splits: int = 1,
              stream=None):
    """Allocate outputs and run the forward; ``num_splits > 1`` takes the split-KV +
    combine path. Returns ``(o, lse)``."""
    import torch

    B, H, Nq, Nk, d = _bhnd(q, k, v)
    o = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=q.device)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if num_splits == 1:
        fa_fwd(q, k, v, o, lse, causal, scale, stream)
    else:
        nbytes = fa_splitkv_workspace_bytes(B, H, Nq, d, num_splits)
        if nbytes == 0:
            raise FAError(5, "fa_splitkv_workspace_bytes")
        ws = torch.empty(nbytes // 4, dtype=torch.float32, device=q.device)
        fa_fwd_splitkv(q, k, v, ws, num_splits, causal, scale, stream)
        fa_combine(ws, o, lse, B, H, Nq, d, num_splits, stream)
    return o, lse


def fa_fwd_splitkv_static(q, k, v, o, lse, num_splits: int, causal=False,
                          scale: float | None = None, stream=None):
    """Split-KV forward + merge into caller-owned ``o``/``lse`` with no workspace
    argument: the partial states live in the library's static device buffer
    (``FA_STATIC_SCRATCH_BYTES``), so nothing is allocated. For callers that may
    not allocate device memory; calls that overlap on the GPU share that buffer
    and race (see include/fa.h)."""
    B, H, Nq, Nk, d = _bhnd(q, k, v)
    _need_o_lse(o, lse, B, H, Nq, d, q.device)
    scale = default_scale(d) if scale is None else float(scale)
    lib = load_library()
    fn = lib.fa_fwd_splitkv_static
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, i, vp]
    fn.restype = i
    st = fn(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d, scale,
            causal_code(causal), int(num_splits), _stream_handle(stream))
    _check(st, "fa_fwd_splitkv_static")


_SIDE_STREAMS = {}


def _side_streams(device):
    """Two streams per device, for host-to-device and device-to-host copies."""
    import torch

    key = torch.device(device).index
    if key not in _SIDE_STREAMS:
        _SIDE_STREAMS[key] = (torch.cuda.Stream(device=device), torch.cuda.Stream(device=device))
    return _SIDE_STREAMS[key]


def head_slices(BH: int, chunks: int):
    """The ``(h0, h1)`` bounds :func:`fa_fwd_from_host` cuts ``BH`` heads into:
    at most ``chunks`` non-empty slices of consecutive heads covering
    ``[0, BH)``. With three or more, the last two slices get a half and a
    quarter of the others' share: the last slice's kernel and copy back run
    after every copy in has finished, so a smaller last slice leaves less of
    the call uncovered."""
    chunks = max(1, min(int(chunks), BH))
    weights = [1.0] * (chunks - 2) + [0.5, 0.25] if chunks >= 3 else [1.0] * chunks
    total = sum(weights)
    bounds, acc, prev = [], 0.0, 0
    for w in weights:
        acc += w
        cur = min(BH, int(round(BH * acc / total)))
        if cur > prev:
            bounds.append((prev, cur))
            prev = cur
    if prev < BH:
        bounds.append((prev, BH))
    return bounds


def fa_fwd_from_host(q_host, k_host, v_host, o_host, lse_host, q, k, v, o, lse, causal=False,
                     scale: float | None = None, chunks: int = 4, stream=None):
    """The forward of :func:`fa_fwd` on inputs and outputs in pinned host memory.

    ``q_host``, ``k_host``, ``v_host`` (bf16 [B,H,N,d]) are copied into the
    device tensors ``q``, ``k``, ``v`` of the same shapes, the forward writes the
    device ``o``, ``lse``, and they are copied back into ``o_host``, ``lse_host``.
    The (b, h) heads are cut into at most ``chunks`` slices of consecutive heads
    (:func:`head_slices`; contiguous in every tensor, each slice runs as one
    forward over its heads) so that the copies of one slice overlap the kernel
    of another:
    host-to-device copies on one side stream, the kernels on ``stream``,
    device-to-host copies on another. Every call starts after the work already
    queued on ``stream`` and ``stream`` waits for the last copy back, so a caller
    synchronises on ``stream`` alone.
    """
    import torch

    B, H, Nq, Nk, d = _bhnd(q, k, v)
    _need_o_lse(o, lse, B, H, Nq, d, q.device)
    cpu = torch.device("cpu")
    for name, t, dev_t in (("q_host", q_host, q), ("k_host", k_host, k), ("v_host", v_host, v),
                           ("o_host", o_host, o), ("lse_host", lse_host, lse)):
        _need(t, name, tuple(dev_t.shape), dev_t.dtype, cpu)
        if not t.is_pinned():
            raise ValueError(f"{name} must be in pinned host memory")
    BH = B * H
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    s_in, s_out = _side_streams(q.device)
    s_in.wait_stream(stream)
    # Heads flattened: [1, B*H, N, d] views (contiguous tensors, checked above).
    flat = lambda t: t.view(1, BH, *t.shape[2:])  # noqa: E731
    qh, kh, vh, oh, lh = (flat(t) for t in (q_host, k_host, v_host, o_host, lse_host))
    qd, kd, vd, od, ld = (flat(t) for t in (q, k, v, o, lse))
    bounds = head_slices(BH, chunks)
    done_out = None
    for h0, h1 in bounds:
        with torch.cuda.stream(s_in):
            for src, dst in ((qh, qd), (kh, kd), (vh, vd)):
                dst[:, h0:h1].copy_(src[:, h0:h1], non_blocking=True)
            ev_in = torch.cuda.Event()
            ev_in.record(s_in)
        stream.wait_event(ev_in)
        fa_fwd(qd[:, h0:h1], kd[:, h0:h1], vd[:, h0:h1], od[:, h0:h1], ld[:, h0:h1], causal, scale, stream)
        ev_c = torch.cuda.Event()
        ev_c.record(stream)
        s_out.wait_event(ev_c)
        with torch.cuda.stream(s_out):
            oh[:, h0:h1].copy_(od[:, h0:h1], non_blocking=True)
            lh[:, h0:h1].copy_(ld[:, h0:h1], non_blocking=True)
            done_out = torch.cuda.Event()
            done_out.record(s_out)
    stream.wait_event(done_out)
