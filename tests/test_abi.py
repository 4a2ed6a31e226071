"""The C-ABI library on the CPU: it builds, loads, exports every symbol that
include/fa.h declares, and rejects bad arguments with the documented status
before any CUDA work. No kernel is launched here."""

import ctypes
import json
import math
import os
import re

import pytest

import exact_attention_80_gb300 as fa
from exact_attention_80_gb300 import build as fa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")

FAKE = 0x10000  # 16-byte aligned, never dereferenced: validation fails first
P = ctypes.c_void_p


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(fa.LIB_PATH):
        fa_build.build()
    return fa.load_library()


def declared_functions():
    with open(HEADER, encoding="utf-8") as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_api():
    names = declared_functions()
    for want in ("fa_fwd", "fa_fwd_splitkv", "fa_combine", "fa_splitkv_workspace_bytes",
                 "fa_status_string", "fa_fwd_grid_ctas", "fa_device_status", "fa_fwd_varlen",
                 "fa_fwd_fp8", "fa_fwd_fp8_splitkv", "fa_bwd", "fa_bwd_workspace_bytes",
                 "fa_fwd_rows"):
        assert want in names


def test_header_is_plain_c(tmp_path):
    """include/fa.h is a C interface: it compiles as C11 with warnings as errors."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no gcc")
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(fa_build.nvcc_path())), "include")
    src = tmp_path / "c_client.c"
    src.write_text('#include "fa.h"\nint main(void) { return fa_status_string(FA_OK) == 0; }\n')
    r = subprocess.run([gcc, "-std=c11", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in include/fa.h but not exported"


def test_status_strings(lib):
    for code, name in fa.STATUS_NAMES.items():
        assert fa.fa_status_string(code).startswith(name)


def _fwd(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, B=1, H=1, Nq=8, Nk=8, d=64,
         scale=0.125, causal=0):
    return lib.fa_fwd(P(q), P(k), P(v), P(o), P(lse), B, H, Nq, Nk, d, scale, causal, P(0))


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), 1), (dict(k=0), 1), (dict(v=0), 1), (dict(o=0), 1), (dict(lse=0), 1),
    (dict(B=0), 3), (dict(H=0), 3), (dict(Nq=0), 3), (dict(Nk=0), 3), (dict(Nk=-5), 3),
    (dict(B=1 << 16, H=1 << 16), 3),
    (dict(d=32), 4), (dict(d=96), 4), (dict(d=512), 4), (dict(d=0), 4),
    (dict(scale=0.0), 9), (dict(scale=-0.1), 9), (dict(scale=float("nan")), 9),
    (dict(scale=float("inf")), 9),
    (dict(q=FAKE + 8), 2), (dict(k=FAKE + 4), 2), (dict(v=FAKE + 2), 2), (dict(o=FAKE + 8), 2),
    (dict(lse=FAKE + 2), 2),
    (dict(causal=3), 11), (dict(causal=-1), 11),
])
def test_fwd_rejects(lib, kw, code):
    assert _fwd(lib, **kw) == code


def _split(lib, ws=FAKE, S=4, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, B=1, H=1, Nq=8, Nk=8, d=64, scale=0.125, causal=0)
    a.update(kw)
    return lib.fa_fwd_splitkv(P(a["q"]), P(a["k"]), P(a["v"]), P(ws), a["B"], a["H"], a["Nq"],
                              a["Nk"], a["d"], a["scale"], a["causal"], S, P(0))


@pytest.mark.parametrize("kw,code", [
    (dict(ws=0), 6), (dict(ws=FAKE + 4), 6), (dict(S=0), 5), (dict(S=257), 5),
    (dict(d=80), 4), (dict(q=0), 1), (dict(Nq=0), 3), (dict(scale=0.0), 9), (dict(causal=7), 11),
])
def test_splitkv_rejects(lib, kw, code):
    assert _split(lib, **kw) == code


@pytest.mark.parametrize("args,code", [
    ((0, FAKE, FAKE, 1, 1, 8, 64, 2), 6), ((FAKE, 0, FAKE, 1, 1, 8, 64, 2), 1),
    ((FAKE, FAKE, 0, 1, 1, 8, 64, 2), 1), ((FAKE, FAKE, FAKE, 0, 1, 8, 64, 2), 3),
    ((FAKE, FAKE, FAKE, 1, 1, 8, 48, 2), 4), ((FAKE, FAKE, FAKE, 1, 1, 8, 64, 0), 5),
    ((FAKE + 8, FAKE, FAKE, 1, 1, 8, 64, 2), 6), ((FAKE, FAKE + 8, FAKE, 1, 1, 8, 64, 2), 2),
])
def test_combine_rejects(lib, args, code):
    ws, o, lse, B, H, Nq, d, S = args
    assert lib.fa_combine(P(ws), P(o), P(lse), B, H, Nq, d, S, P(0)) == code


def _varlen(lib, q=FAKE, k=FAKE, v=FAKE, o=FAKE, lse=FAKE, cq=FAKE, ck=FAKE, B=2, H=1, tq=64,
            tk=64, maxq=32, d=64, scale=0.125, causal=0):
    return lib.fa_fwd_varlen(P(q), P(k), P(v), P(o), P(lse), P(cq), P(ck), B, H, tq, tk, maxq, d,
                             scale, causal, P(0))


@pytest.mark.parametrize("kw,code", [
    (dict(cq=0), 1), (dict(ck=0), 1), (dict(o=0), 1), (dict(q=0), 1),
    (dict(cq=FAKE + 2), 2), (dict(ck=FAKE + 1), 2), (dict(o=FAKE + 8), 2),
    (dict(maxq=0), 3), (dict(maxq=65), 3), (dict(tq=0), 3), (dict(B=0), 3),
    (dict(d=96), 4), (dict(scale=0.0), 9), (dict(causal=4), 11),
])
def test_varlen_rejects(lib, kw, code):
    assert _varlen(lib, **kw) == code


def _fp8(lib, q=FAKE, k=FAKE, v=FAKE, qd=0.03125, kd=0.03125, vd=0.03125, o=FAKE, lse=FAKE, B=1,
         H=1, Nq=8, Nk=8, d=128, scale=0.088, causal=0):
    return lib.fa_fwd_fp8(P(q), P(k), P(v), qd, kd, vd, P(o), P(lse), B, H, Nq, Nk, d, scale,
                          causal, P(0))


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), 1), (dict(v=0), 1), (dict(o=0), 1), (dict(lse=0), 1),
    (dict(Nq=0), 3), (dict(B=0), 3),
    (dict(d=32), 4), (dict(d=96), 4), (dict(d=512), 4),
    (dict(qd=0.0), 9), (dict(kd=-1.0), 9), (dict(vd=float("nan")), 9), (dict(vd=float("inf")), 9),
    (dict(scale=0.0), 9), (dict(qd=1e-30, kd=1e-30), 9), (dict(qd=1e30, kd=1e30), 9),
    (dict(q=FAKE + 8), 2), (dict(o=FAKE + 8), 2), (dict(lse=FAKE + 2), 2),
    (dict(causal=3), 11),
])
def test_fp8_rejects(lib, kw, code):
    assert _fp8(lib, **kw) == code


@pytest.mark.parametrize("kw,code", [
    (dict(ws=0), 6), (dict(ws=FAKE + 4), 6), (dict(S=0), 5), (dict(S=257), 5), (dict(d=96), 4),
    (dict(q=0), 1), (dict(vd=0.0), 9), (dict(causal=5), 11), (dict(Nk=0), 3),
])
def test_fp8_splitkv_rejects(lib, kw, code):
    a = dict(q=FAKE, k=FAKE, v=FAKE, qd=0.03125, kd=0.03125, vd=0.03125, ws=FAKE, B=1, H=1, Nq=8,
             Nk=8, d=128, scale=0.088, causal=0, S=4)
    a.update(kw)
    assert lib.fa_fwd_fp8_splitkv(P(a["q"]), P(a["k"]), P(a["v"]), a["qd"], a["kd"], a["vd"],
                                  P(a["ws"]), a["B"], a["H"], a["Nq"], a["Nk"], a["d"], a["scale"],
                                  a["causal"], a["S"], P(0)) == code


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), 1), (dict(o=0), 1), (dict(do=0), 1), (dict(lse=0), 1), (dict(dq=0), 1),
    (dict(dk=0), 1), (dict(dv=0), 1), (dict(ws=0), 6), (dict(ws=FAKE + 4), 6),
    (dict(d=96), 4), (dict(d=512), 4), (dict(Nq=0), 3), (dict(scale=0.0), 9), (dict(causal=3), 11),
    (dict(dq=FAKE + 8), 2), (dict(o=FAKE + 2), 2), (dict(lse=FAKE + 2), 2),
    (dict(Nq=2**31 - 100), 3), (dict(Nk=2**31 - 100), 3),  # no room to round up to 128-row tiles
])
def test_bwd_rejects(lib, kw, code):
    a = dict(q=FAKE, k=FAKE, v=FAKE, o=FAKE, do=FAKE, lse=FAKE, dq=FAKE, dk=FAKE, dv=FAKE, ws=FAKE,
             B=1, H=1, Nq=8, Nk=8, d=128, scale=0.088, causal=0)
    a.update(kw)
    assert lib.fa_bwd(P(a["q"]), P(a["k"]), P(a["v"]), P(a["o"]), P(a["do"]), P(a["lse"]), P(a["dq"]),
                      P(a["dk"]), P(a["dv"]), P(a["ws"]), a["B"], a["H"], a["Nq"], a["Nk"], a["d"],
                      a["scale"], a["causal"], P(0)) == code
    assert fa.fa_bwd_workspace_bytes(2, 3, 77, 128) == 2 * 3 * 128 * 130 * 4
    assert fa.fa_bwd_workspace_bytes(1, 1, 129, 128) == 256 * 130 * 4
    assert fa.fa_bwd_workspace_bytes(2, 3, 77, 64) == 2 * 3 * 128 * 66 * 4
    assert fa.fa_bwd_workspace_bytes(2, 3, 77, 256) == 2 * 3 * 128 * 258 * 4
    assert fa.fa_bwd_workspace_bytes(2, 3, 77, 96) == 0


def test_workspace_bytes(lib):
    for (B, H, Nq, d, S) in ((1, 8, 128, 128, 64), (2, 3, 77, 64, 1), (8, 16, 8191, 256, 3)):
        assert fa.fa_splitkv_workspace_bytes(B, H, Nq, d, S) == S * B * H * Nq * (d + 2) * 4
    assert fa.fa_splitkv_workspace_bytes(1, 1, 1, 100, 1) == 0
    assert fa.fa_splitkv_workspace_bytes(1, 1, 1, 64, 0) == 0
    assert fa.fa_splitkv_workspace_bytes(0, 1, 1, 64, 1) == 0


def test_cta_counts_match_printed_schedule(lib):
    """The FA-2 page's printed CTA counts (batch*heads*ceil(seq/tile)) and the
    library's grid: 256-row CTAs for d<=128, 128-row CTAs for d=256."""
    with open(os.path.join(ROOT, "tests", "golden", "cta_schedule.json"), encoding="utf-8") as f:
        g = json.load(f)
    for b, h, n, tile, ctas in g["rows"]:
        assert b * h * math.ceil(n / tile) == ctas
    by_tile = {(r[0], r[1], r[2], r[3]): r[4] for r in g["rows"]}
    assert fa.fa_fwd_grid_ctas(1, 8, 8192, 128) == by_tile[(1, 8, 8192, 256)]
    assert fa.fa_fwd_grid_ctas(1, 8, 8192, 64) == by_tile[(1, 8, 8192, 256)]
    assert fa.fa_fwd_grid_ctas(1, 8, 8192, 256) == by_tile[(1, 8, 8192, 128)]
    # Splits multiply the grid; with one query tile per head, two splits share a
    # CTA (one per query-tile slot).
    assert fa.fa_fwd_grid_ctas(1, 8, 128, 128, 64) == 8 * 32
    assert fa.fa_fwd_grid_ctas(1, 8, 128, 128, 19) == 8 * 10
    assert fa.fa_fwd_grid_ctas(1, 8, 129, 128, 4) == 8 * 4
    assert fa.fa_fwd_grid_ctas(1, 8, 128, 256, 4) == 8 * 4
    assert fa.fa_fwd_grid_ctas(1, 8, 8192, 128, 1) > g["heads_only_ctas"]["ctas"]
    assert fa.fa_fwd_grid_ctas(1, 8, 128, 100, 1) == -1


def test_valid_call_without_gpu_reports_cuda_error(lib):
    torch = pytest.importorskip("torch")
    if torch.cuda.is_available():
        pytest.skip("would launch on fake pointers; only meaningful without a GPU")
    assert _fwd(lib) == 7
    assert lib.fa_device_status(P(0), 1) == 7


def test_python_binding_rejects_bad_tensors():
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 8, 64, dtype=torch.float32)
    with pytest.raises(TypeError):
        fa.fa_fwd(q, q, q, q, q)
    qb = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fa_fwd(qb, qb, qb, qb, qb)  # CPU tensors are refused before any call


def test_bench_fill_splits(lib):
    """The bench's split count for one CTA per SM follows the grid the library
    reports: two splits per CTA with one query tile, one otherwise."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    assert bench.fill_splits(fa, 1, 8, 128, 128, 152) == 38   # C5: 8 heads x 19 pairs
    assert bench.fill_splits(fa, 1, 8, 128, 64, 152) == 38
    assert bench.fill_splits(fa, 1, 8, 256, 128, 152) == 19   # two query tiles per CTA
    assert bench.fill_splits(fa, 1, 8, 128, 256, 152) == 19   # d = 256: no dual-range CTAs
    assert bench.fill_splits(fa, 1, 200, 128, 128, 152) == 1


def test_rows_per_cta_refused_before_any_cuda_call(lib):
    """fa_fwd_rows offers 64, 128 or 256 query rows per CTA at d <= 128 and 128
    at d = 256; anything else is FA_ERR_TILE (13), checked on the host (fake
    pointers are never used)."""
    fn = lib.fa_fwd_rows
    i, f = ctypes.c_int, ctypes.c_float
    fn.argtypes = [P, P, P, P, P, i, i, i, i, i, f, i, i, P]
    fn.restype = i
    fake = P(0x10000)
    for d, rows in ((128, 32), (128, 384), (64, 192), (256, 256), (128, 0), (256, 64), (64, -64)):
        assert fn(fake, fake, fake, fake, fake, 1, 8, 1024, 1024, d, 0.1, 0, rows, P(0)) == 13, (d, rows)
    assert lib.fa_status_string(13).decode().startswith("FA_ERR_TILE")
    # A head dim outside the set is still FA_ERR_HEADDIM, and bad pointers keep their codes.
    assert fn(fake, fake, fake, fake, fake, 1, 8, 1024, 1024, 96, 0.1, 0, 128, P(0)) == 4
    assert fn(fake, fake, fake, P(0), fake, 1, 8, 1024, 1024, 128, 0.1, 0, 128, P(0)) == 1
