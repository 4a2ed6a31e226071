"""Seeded synthetic inputs, the one module both the CUDA path's callers and the
float64 oracle's callers use. It holds no attention arithmetic: it only draws
numbers and rounds them to bf16.

Recipe (the workloads of the five benchmark configurations):

* Q, K, V are drawn i.i.d. N(0, 1) in float32 from ``torch.Generator`` seeded
  with ``seed``, in the order Q, K, V, then rounded to bf16 (round to nearest
  even, torch's conversion). The same bf16 bits go to the GPU and, upcast
  exactly, to the oracle.
* ``outlier_frac`` > 0 (the large-head-dim configuration): for each (b, h),
  ``floor(outlier_frac * Nk)`` distinct key rows, chosen by a seeded
  permutation (drawn after V, same generator), are multiplied by
  ``outlier_scale`` in float32 before the bf16 rounding. A factor of 8 is a
  power of two, so it commutes with the rounding.
"""

from __future__ import annotations

import itertools
import math

import torch

CONFIG_SEED_BASE = 1000


def make_qkv(B: int, H: int, Nq: int, Nk: int, d: int, seed: int,
             outlier_frac: float = 0.0, outlier_scale: float = 8.0):
    """Return bf16 CPU tensors ``(q [B,H,Nq,d], k [B,H,Nk,d], v [B,H,Nk,d])``."""
    g = torch.Generator().manual_seed(int(seed))
    q = torch.randn((B, H, Nq, d), generator=g, dtype=torch.float32)
    k = torch.randn((B, H, Nk, d), generator=g, dtype=torch.float32)
    v = torch.randn((B, H, Nk, d), generator=g, dtype=torch.float32)
    if outlier_frac > 0.0:
        count = int(math.floor(outlier_frac * Nk))
        for b in range(B):
            for h in range(H):
                rows = torch.randperm(Nk, generator=g)[:count]
                k[b, h, rows] *= outlier_scale
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16)


def make_varlen(lq, lk, H: int, d: int, seed: int):
    """Packed variable-length inputs: bf16 CPU tensors ``q [sum lq, H, d]``,
    ``k``/``v [sum lk, H, d]`` (token-major, drawn N(0, 1) in the order Q, K, V
    like :func:`make_qkv`) and int32 prefix offsets ``cu_q``, ``cu_k`` [B+1]."""
    g = torch.Generator().manual_seed(int(seed))
    tq, tk = int(sum(lq)), int(sum(lk))
    q = torch.randn((tq, H, d), generator=g, dtype=torch.float32)
    k = torch.randn((tk, H, d), generator=g, dtype=torch.float32)
    v = torch.randn((tk, H, d), generator=g, dtype=torch.float32)
    cu_q = torch.tensor([0] + list(itertools.accumulate(lq)), dtype=torch.int32)
    cu_k = torch.tensor([0] + list(itertools.accumulate(lk)), dtype=torch.int32)
    return q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16), cu_q, cu_k


def make_qkv_fp8(B: int, H: int, Nq: int, Nk: int, d: int, seed: int,
                 descales=(2.0 ** -5, 2.0 ** -5, 2.0 ** -5)):
    """e4m3 inputs: Q, K, V drawn N(0, 1) in float32 as in :func:`make_qkv`, each
    divided by its descale, clamped to +-448 (e4m3's largest magnitude; torch's
    cast does not saturate) and rounded to e4m3 by torch (nearest even).
    Returns uint8 CPU tensors of e4m3 codes ``(q8, k8, v8)``; the value each code
    stands for is its e4m3 value times the descale."""
    import torch

    g = torch.Generator().manual_seed(int(seed))
    out = []
    for shape, ds in zip(((B, H, Nq, d), (B, H, Nk, d), (B, H, Nk, d)), descales):
        x = (torch.randn(shape, generator=g, dtype=torch.float32) / float(ds)).clamp(-448.0, 448.0)
        out.append(x.to(torch.float8_e4m3fn).view(torch.uint8))
    return tuple(out)


def make_grad_output(B: int, H: int, Nq: int, d: int, seed: int):
    """Upstream gradient dO for the backward: N(0, 1) in float32 from its own
    seeded generator, rounded to bf16; a CPU tensor [B, H, Nq, d]."""
    g = torch.Generator().manual_seed(int(seed))
    return torch.randn((B, H, Nq, d), generator=g, dtype=torch.float32).to(torch.bfloat16)


def make_device_normal(shape, seed: int, device, dtype=None, chunk: int = 1 << 28):
    """A tensor of i.i.d. N(0, 1) draws made on ``device`` by a seeded device
    generator, in float32 and rounded to ``dtype`` (bf16 by default), filled
    ``chunk`` elements at a time so that no float32 copy of the whole tensor is
    held. For sizes too large to draw on the host; only the rows a test checks
    are copied back for the oracle."""
    dtype = torch.bfloat16 if dtype is None else dtype
    g = torch.Generator(device=device).manual_seed(int(seed))
    t = torch.empty(shape, dtype=dtype, device=device)
    flat = t.view(-1)
    for i in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - i)
        flat[i:i + n] = torch.randn(n, generator=g, dtype=torch.float32, device=device).to(dtype)
    return t


def make_device_e4m3(shape, seed: int, device, descale: float, chunk: int = 1 << 28):
    """e4m3 codes (uint8) made on ``device`` by the recipe of
    :func:`make_qkv_fp8` (N(0, 1) / descale, clamped to +-448, rounded by
    torch), from a seeded device generator, ``chunk`` elements at a time."""
    g = torch.Generator(device=device).manual_seed(int(seed))
    t = torch.empty(shape, dtype=torch.uint8, device=device)
    flat = t.view(-1)
    for i in range(0, flat.numel(), chunk):
        n = min(chunk, flat.numel() - i)
        x = (torch.randn(n, generator=g, dtype=torch.float32, device=device) / float(descale)).clamp(-448.0, 448.0)
        flat[i:i + n] = x.to(torch.float8_e4m3fn).view(torch.uint8)
    return t


def to_f64(t):
    """Exact upcast of a (bf16) torch tensor to a float64 numpy array."""
    return t.to(torch.float64).numpy()


def f32(x: float) -> float:
    """Round a Python float to the nearest float32 (the value a kernel receives)."""
    return float(torch.tensor(x, dtype=torch.float32).item())


# The five benchmark workloads (shape, mask, scale, seed).
CONFIGS = {
    "c1": dict(B=1, H=1, Nq=128, Nk=128, d=64, causal=False, seed=CONFIG_SEED_BASE + 0),
    "c2": dict(B=8, H=32, Nq=2048, Nk=2048, d=128, causal=False, seed=CONFIG_SEED_BASE + 1),
    "c2_causal": dict(B=8, H=32, Nq=2048, Nk=2048, d=128, causal=True, seed=CONFIG_SEED_BASE + 1),
    "c3": dict(B=1, H=8, Nq=8192, Nk=8192, d=128, causal=False, seed=CONFIG_SEED_BASE + 2),
    "c3_causal": dict(B=1, H=8, Nq=8192, Nk=8192, d=128, causal=True, seed=CONFIG_SEED_BASE + 2),
    "c4": dict(B=8, H=16, Nq=8191, Nk=8191, d=256, causal=True, seed=CONFIG_SEED_BASE + 3,
               outlier_frac=0.01),
    "c5": dict(B=1, H=8, Nq=128, Nk=131072, d=128, causal=False, seed=CONFIG_SEED_BASE + 4),
}


def config_inputs(name: str):
    c = CONFIGS[name]
    return make_qkv(c["B"], c["H"], c["Nq"], c["Nk"], c["d"], c["seed"],
                    outlier_frac=c.get("outlier_frac", 0.0))


def metric_flops(B: int, H: int, Nq: int, Nk: int, d: int, causal) -> float:
    """The benchmark's FLOP count: 4*B*H*Nq*Nk*d, halved for a (top-left)
    causal mask. For the bottom-right mask, whose shapes are not square, it is
    4*B*H*d times the number of visible (query, key) pairs."""
    if causal == "bottom_right" or causal == 2:
        pairs = sum(max(0, min(Nk, i + Nk - Nq + 1)) for i in range(Nq))
        return 4.0 * B * H * d * pairs
    f = 4.0 * B * H * Nq * Nk * d
    return f / 2 if causal else f
