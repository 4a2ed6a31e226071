"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle on
the same seeded bf16 inputs.

Acceptance (bf16 inputs, fp32 accumulation): on O, max-abs error <= 2e-2 and
relative L2 error <= 5e-3; on LSE, max-abs error <= 1e-3.  Small shapes and
the full benchmark workloads alike are compared element by element on their
whole outputs.
"""

import math

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import exact_attention_80_gb300 as fa  # noqa: E402
import oracle  # noqa: E402
from exact_attention_80_gb300.inputs import CONFIGS, config_inputs, f32, make_qkv, to_f64  # noqa: E402

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


def check(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    o = o_gpu.float().cpu().numpy().astype(np.float64)
    lse = lse_gpu.cpu().numpy().astype(np.float64)
    assert np.all(np.isfinite(o)), f"{what}: non-finite O"
    err = np.abs(o - o_ref)
    max_abs = float(err.max())
    rel = float(np.linalg.norm((o - o_ref).ravel()) / max(np.linalg.norm(o_ref.ravel()), 1e-30))
    # Rows that see no key (bottom-right mask with Nq > Nk) have LSE = -inf on
    # both sides; the finite rows are compared.
    empty = ~np.isfinite(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: -inf LSE rows differ"
    lse_err = float(np.abs(lse[~empty] - lse_ref[~empty]).max()) if (~empty).any() else 0.0
    assert max_abs <= MAX_ABS, f"{what}: max-abs {max_abs:.3e}"
    assert rel <= REL_L2, f"{what}: rel-L2 {rel:.3e}"
    assert lse_err <= LSE_ABS, f"{what}: LSE err {lse_err:.3e}"
    return max_abs, rel, lse_err


def run_gpu(q, k, v, causal, scale, num_splits=1):
    o, lse = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=causal, scale=scale,
                          num_splits=num_splits)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    return o, lse


def run_gpu_rows(q, k, v, causal, scale, rows_per_cta):
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    B, H, Nq, d = q.shape
    o = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    fa.fa_fwd_rows(qc, kc, vc, o, lse, rows_per_cta, causal, scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status(clear=True) == fa.FA_OK
    return o, lse


SMALL = [
    # B, H, Nq, Nk, d, causal
    (1, 1, 128, 128, 64, False),
    (2, 3, 300, 333, 64, False),
    (2, 3, 300, 333, 64, True),
    (1, 2, 257, 511, 128, False),
    (1, 2, 257, 511, 128, True),
    (2, 2, 384, 384, 128, True),
    (1, 2, 200, 190, 256, False),
    (1, 2, 200, 190, 256, True),
    (1, 1, 1, 1, 128, False),
    (1, 1, 1, 1000, 128, False),
    (1, 1, 1000, 1, 64, False),
    (1, 1, 300, 100, 128, True),   # Nq > Nk: rows past Nk see every key
    (1, 1, 100, 300, 128, True),   # Nq < Nk: top-left alignment
    (1, 1, 513, 129, 256, True),
    (3, 1, 640, 640, 64, True),
    # bottom-right alignment: key j visible to query i iff j <= i + Nk - Nq
    (1, 1, 300, 100, 128, "bottom_right"),  # Nq > Nk: the first 200 rows see no key
    (1, 1, 100, 300, 128, "bottom_right"),
    (2, 3, 257, 511, 64, "bottom_right"),
    (1, 2, 200, 190, 256, "bottom_right"),
    (1, 2, 190, 200, 256, "bottom_right"),
    (1, 1, 1, 1000, 128, "bottom_right"),  # one new query over a 1000-key cache
    (1, 1, 513, 129, 64, "bottom_right"),
    (3, 1, 640, 640, 64, "bottom_right"),  # Nq = Nk: same as top-left
]


@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", SMALL)
def test_small_shapes_elementwise(B, H, Nq, Nk, d, causal):
    seed = 7 + Nq + 3 * Nk + d
    q, k, v = make_qkv(B, H, Nq, Nk, d, seed)
    scale = f32(1.0 / math.sqrt(d))
    o, lse = run_gpu(q, k, v, causal, scale)
    o_ref, lse_ref = oracle.attention_f64(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    check(o, lse, o_ref, lse_ref, f"{(B, H, Nq, Nk, d, causal)}")


@pytest.mark.parametrize("d", [64, 128, 256])
def test_outlier_keys_and_other_scales(d):
    q, k, v = make_qkv(2, 2, 191, 191, d, 99, outlier_frac=0.01)
    for scale in (f32(0.5 / math.sqrt(d)), f32(2.0 / math.sqrt(d))):
        for causal in (False, True):
            o, lse = run_gpu(q, k, v, causal, scale)
            o_ref, lse_ref = oracle.attention_f64(to_f64(q), to_f64(k), to_f64(v), scale, causal)
            check(o, lse, o_ref, lse_ref, f"d={d} scale={scale} causal={causal}")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("splits", [1, 3])
def test_dominant_key_weight_matches_rounded_p(d, splits):
    """Rows dominated by one key whose p is not a power of two relative to the
    exponent reference: key 0 sets the reference (score 20), key 200 in a later
    key tile scores 25, less than 8 base-2 units above it, so its p = 2^7.2 is
    rounded to bf16 for the PV product (relative error up to 2^-8). O must
    still equal that key's V (values in [4, 8)) up to the bf16 output rounding:
    the kernel divides O by the weights the product used. With O divided by
    the unrounded sum, an element could be off by up to 2^-8 of its value
    before the output rounding, and land a whole bf16 step away."""
    Nq, Nk = 128, 400
    g = torch.Generator().manual_seed(600 + d)
    q = torch.zeros(1, 1, Nq, d)
    q[..., 0] = 1.0
    k = torch.randn(1, 1, Nk, d, generator=g) * 0.5
    k[0, 0, 0, 0] = 20.0
    k[0, 0, 200, 0] = 25.0
    v = torch.randn(1, 1, Nk, d, generator=g)
    mag = 4.0 + 4.0 * torch.rand(d, generator=g)
    v[0, 0, 200] = torch.where(torch.rand(d, generator=g) < 0.5, -mag, mag)
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    o, lse = run_gpu(q, k, v, False, 1.0, num_splits=splits)
    o_ref, lse_ref = oracle.attention_f64(to_f64(q), to_f64(k), to_f64(v), 1.0, False)
    got = o.float().cpu().numpy().astype(np.float64)
    half_ulp = np.exp2(np.floor(np.log2(np.abs(o_ref))) - 8)  # bf16: 8 significand bits
    assert np.all(np.abs(got - o_ref) <= half_ulp + 1e-3)
    assert np.abs(lse.cpu().numpy() - lse_ref).max() <= LSE_ABS
    check(o, lse, o_ref, lse_ref, f"dominant key d={d}")


def test_worked_example_on_gpu():
    """The FA-2 page's four-key example as a real kernel call: d=64, scale 1,
    q = e0, K rows = score_j * e0, V rows = value_j * e0 (all exact in bf16)."""
    scores = [1.0, 2.0, 4.0, 0.0]
    values = [2.0, 5.0, 1.0, 9.0]
    q = torch.zeros(1, 1, 1, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    v = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    q[0, 0, 0, 0] = 1.0
    for j in range(4):
        k[0, 0, j, 0] = scores[j]
        v[0, 0, j, 0] = values[j]
    for splits in (1, 2, 3, 4):
        o, lse = run_gpu(q, k, v, False, 1.0, num_splits=splits)
        assert abs(o[0, 0, 0, 0].item() - 1.612955) <= MAX_ABS
        assert torch.all(o[0, 0, 0, 1:] == 0)
        want_lse = math.log(sum(math.exp(s) for s in scores))
        assert abs(lse[0, 0, 0].item() - want_lse) <= LSE_ABS


def _split_bounds(Nk, bn, S):
    T = -(-Nk // bn)
    per = -(-T // S)
    out = []
    for s in range(S):
        a = min(s * per, T)
        b = min(a + per, T)
        out.append((min(a * bn, Nk), min(b * bn, Nk)))
    return out


@pytest.mark.parametrize("d", [64, 128, 256])
def test_split_partials_match_oracle_states(d):
    """Each split's (m, l, O) workspace entries against the oracle's partial
    state over the same key range (documented split rule in include/fa.h)."""
    B, H, Nq, Nk, S = 1, 2, 130, 1100, 4
    bn = 96 if d == 256 else 128  # keys per KV tile (include/fa.h, fa_fwd_splitkv)
    q, k, v = make_qkv(B, H, Nq, Nk, d, 5 + d)
    scale = f32(1.0 / math.sqrt(d))
    for causal in (False, True):
        nbytes = fa.fa_splitkv_workspace_bytes(B, H, Nq, d, S)
        ws = torch.full((nbytes // 4,), float("nan"), dtype=torch.float32, device="cuda")
        fa.fa_fwd_splitkv(q.cuda(), k.cuda(), v.cuda(), ws, S, causal, scale)
        torch.cuda.synchronize()
        rows = B * H * Nq
        w = ws.cpu().numpy().astype(np.float64)
        wo = w[: S * rows * d].reshape(S, B * H, Nq, d)
        wm = w[S * rows * d: S * rows * (d + 1)].reshape(S, B * H, Nq)
        wl = w[S * rows * (d + 1):].reshape(S, B * H, Nq)
        bounds = _split_bounds(Nk, bn, S)
        qf, kf, vf = to_f64(q), to_f64(k), to_f64(v)
        for h in range(B * H):
            s_full = oracle.scores_f64(qf.reshape(-1, Nq, d)[h], kf.reshape(-1, Nk, d)[h], scale,
                                       causal)
            states = oracle.split_states_f64(s_full, vf.reshape(-1, Nk, d)[h], bounds)
            for sidx, (m_ref, l_ref, u_ref) in enumerate(states):
                fin = np.isfinite(m_ref)
                assert np.array_equal(np.isfinite(wm[sidx, h]), fin)
                assert np.all(wl[sidx, h][~fin] == 0) and np.all(wo[sidx, h][~fin] == 0)
                if fin.any():
                    assert np.abs(wm[sidx, h][fin] - m_ref[fin]).max() <= 1e-4
                    assert np.abs(wl[sidx, h][fin] / l_ref[fin] - 1).max() <= 1e-3
                    o_n = wo[sidx, h][fin] / wl[sidx, h][fin][:, None]
                    o_r = u_ref[fin] / l_ref[fin][:, None]
                    assert np.abs(o_n - o_r).max() <= MAX_ABS


def test_combine_of_printed_block_states():
    """fa_combine fed the two printed block states (m, l, u) of the FA-2 page's
    split example as a 2-split workspace must give 1.612955."""
    d, S = 64, 2
    ws = torch.zeros(S * (d + 2), dtype=torch.float32)
    for s, (m, l, u) in enumerate([(2.0, 1.367879, 5.735759), (4.0, 1.018316, 1.164841)]):
        ws[s * d] = u
        ws[S * d + s] = m
        ws[S * d + S + s] = l
    o = torch.empty(1, 1, 1, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 1, 1, dtype=torch.float32, device="cuda")
    fa.fa_combine(ws.cuda(), o, lse, 1, 1, 1, d, S)
    torch.cuda.synchronize()
    assert abs(o[0, 0, 0, 0].item() - 1.612955) <= 1e-2
    assert abs(lse.item() - (4.0 + math.log(1.367879 * math.exp(-2.0) + 1.018316))) <= 1e-4


@pytest.mark.parametrize("d", [64, 128, 256])
def test_combine_of_oracle_partials(d):
    """fa_combine alone, fed oracle-made partial states (with empty splits)."""
    rng = np.random.default_rng(d)
    BH, Nq, Nk = 3, 45, 200
    q = rng.standard_normal((BH, Nq, d))
    k = rng.standard_normal((BH, Nk, d))
    v = rng.standard_normal((BH, Nk, d))
    bounds = [(0, 50), (50, 50), (50, 120), (120, 200), (200, 200)]
    S = len(bounds)
    ws = np.zeros((S * BH * Nq * (d + 2),), dtype=np.float32)
    wo = ws[: S * BH * Nq * d].reshape(S, BH, Nq, d)
    wm = ws[S * BH * Nq * d: S * BH * Nq * (d + 1)].reshape(S, BH, Nq)
    wl = ws[S * BH * Nq * (d + 1):].reshape(S, BH, Nq)
    o_ref = np.zeros((BH, Nq, d))
    lse_ref = np.zeros((BH, Nq))
    for h in range(BH):
        s_full = oracle.scores_f64(q[h], k[h], 0.1, False)
        states = oracle.split_states_f64(s_full, v[h], bounds)
        for s, (m, l, u) in enumerate(states):
            wm[s, h], wl[s, h], wo[s, h] = m, l, u
        o_ref[h], lse_ref[h] = oracle.merge_states_f64(states)
    o = torch.empty(1, BH, Nq, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, BH, Nq, dtype=torch.float32, device="cuda")
    fa.fa_combine(torch.from_numpy(ws).cuda(), o, lse, 1, BH, Nq, d, S)
    torch.cuda.synchronize()
    check(o[0], lse[0], o_ref, lse_ref, "combine")


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("S", [1, 3, 7, 33, 100, 256])
def test_combine_split_counts(d, S):
    """fa_combine over split counts from 1 to the maximum (256), fed oracle
    partial states of contiguous key ranges, some of them empty; 2 x 37 rows,
    so the last block of rows is ragged."""
    rng = np.random.default_rng(1000 * d + S)
    BH, Nq, Nk = 2, 37, 300
    q = rng.standard_normal((BH, Nq, d))
    k = rng.standard_normal((BH, Nk, d))
    v = rng.standard_normal((BH, Nk, d))
    cuts = np.sort(rng.integers(0, Nk + 1, size=S - 1))
    edges = [0, *cuts.tolist(), Nk]
    bounds = [(edges[s], edges[s + 1]) for s in range(S)]
    ws = np.zeros((S * BH * Nq * (d + 2),), dtype=np.float32)
    wo = ws[: S * BH * Nq * d].reshape(S, BH, Nq, d)
    wm = ws[S * BH * Nq * d: S * BH * Nq * (d + 1)].reshape(S, BH, Nq)
    wl = ws[S * BH * Nq * (d + 1):].reshape(S, BH, Nq)
    o_ref = np.zeros((BH, Nq, d))
    lse_ref = np.zeros((BH, Nq))
    for h in range(BH):
        s_full = oracle.scores_f64(q[h], k[h], 0.08, False)
        states = oracle.split_states_f64(s_full, v[h], bounds)
        for s, (m, l, u) in enumerate(states):
            wm[s, h], wl[s, h], wo[s, h] = m, l, u
        o_ref[h], lse_ref[h] = oracle.merge_states_f64(states)
    o = torch.empty(1, BH, Nq, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, BH, Nq, dtype=torch.float32, device="cuda")
    fa.fa_combine(torch.from_numpy(ws).cuda(), o, lse, 1, BH, Nq, d, S)
    torch.cuda.synchronize()
    check(o[0], lse[0], o_ref, lse_ref, f"combine S={S}")


@pytest.mark.parametrize("causal", [False, True, "bottom_right"])
def test_split_invariance(causal):
    """Output semantics do not change with the split count (FA-2 page, split
    section: 1, 2, 3, 4 splits including empty tails), plus 16 and 64."""
    B, H, Nq, Nk, d = 1, 2, 256, 4000, 128
    q, k, v = make_qkv(B, H, Nq, Nk, d, 4242)
    scale = f32(1.0 / math.sqrt(d))
    o_ref, lse_ref = oracle.attention_f64(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    outs = []
    for S in (1, 2, 3, 4, 16, 64):
        o, lse = run_gpu(q, k, v, causal, scale, num_splits=S)
        check(o, lse, o_ref, lse_ref, f"splits={S}")
        outs.append(o.float())
    for x in outs[1:]:
        assert (x - outs[0]).abs().max().item() <= MAX_ABS


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("S", [2, 3, 5, 40])
@pytest.mark.parametrize("Nq,causal", [(1, False), (77, False), (128, True), (100, "bottom_right"),
                                       (64, "bottom_right")])
def test_dual_range_split(d, S, Nq, causal):
    """Split-KV with one query tile runs two splits per CTA (each query-tile
    slot holds the same rows with its own split): odd split counts leave the
    last CTA's second slot without a split, and 40 splits over 4000 keys leave
    splits without keys. Element by element against the oracle."""
    B, H, Nk = 2, 3, 4000
    q, k, v = make_qkv(B, H, Nq, Nk, d, 7100 + S + Nq)
    scale = f32(1.0 / math.sqrt(d))
    o_ref, lse_ref = oracle.attention_f64(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    o, lse = run_gpu(q, k, v, causal, scale, num_splits=S)
    check(o, lse, o_ref, lse_ref, f"dual d={d} S={S} Nq={Nq} {causal}")
    assert fa.fa_fwd_grid_ctas(B, H, Nq, d, S) == B * H * ((S + 1) // 2)


@pytest.mark.parametrize("d", [64, 128, 256])
def test_bottom_right_rows_without_keys_split(d):
    """Bottom-right with Nq > Nk through split-KV + combine: rows that see no key
    in any split come out as O = 0, LSE = -inf; the others match the oracle."""
    B, H, Nq, Nk = 1, 2, 300, 170
    q, k, v = make_qkv(B, H, Nq, Nk, d, 515 + d)
    scale = f32(1.0 / math.sqrt(d))
    o_ref, lse_ref = oracle.attention_f64(to_f64(q), to_f64(k), to_f64(v), scale, "bottom_right")
    assert np.all(lse_ref[..., : Nq - Nk] == -np.inf)
    for S in (1, 2, 3):
        o, lse = run_gpu(q, k, v, "bottom_right", scale, num_splits=S)
        check(o, lse, o_ref, lse_ref, f"d={d} splits={S}")


def test_guard_bands_untouched():
    """Writes stay inside O and LSE: sentinel-filled bands after both survive."""
    B, H, Nq, Nk, d = 1, 3, 130, 200, 128
    q, k, v = make_qkv(B, H, Nq, Nk, d, 31)
    pad = 4096
    o_buf = torch.full((B * H * Nq * d + pad,), 7.0, dtype=torch.bfloat16, device="cuda")
    l_buf = torch.full((B * H * Nq + pad,), 7.0, dtype=torch.float32, device="cuda")
    o = o_buf[: B * H * Nq * d].view(B, H, Nq, d)
    lse = l_buf[: B * H * Nq].view(B, H, Nq)
    for causal in (False, True):
        fa.fa_fwd(q.cuda(), k.cuda(), v.cuda(), o, lse, causal=causal)
        torch.cuda.synchronize()
        assert torch.all(o_buf[B * H * Nq * d:] == 7.0)
        assert torch.all(l_buf[B * H * Nq:] == 7.0)


def test_deterministic():
    q, k, v = make_qkv(2, 2, 700, 900, 128, 77)
    a = run_gpu(q, k, v, True, None)
    b = run_gpu(q, k, v, True, None)
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_shift_invariance_on_gpu():
    """K' = K + 1 w^T shifts every score of row i by scale*q_i.w: O unchanged,
    LSE moved; compared against the oracle on the rounded K'."""
    B, H, Nq, Nk, d = 1, 2, 200, 300, 64
    q, k, v = make_qkv(B, H, Nq, Nk, d, 55)
    w = torch.linspace(-2, 2, d)
    k2 = (k.float() + w).to(torch.bfloat16)
    scale = f32(1.0 / math.sqrt(d))
    o1, _ = run_gpu(q, k, v, False, scale)
    o2, lse2 = run_gpu(q, k2, v, False, scale)
    o_ref, lse_ref = oracle.attention_f64(to_f64(q), to_f64(k2), to_f64(v), scale, False)
    check(o2, lse2, o_ref, lse_ref, "shifted")
    assert (o1.float() - o2.float()).abs().max().item() <= 2 * MAX_ABS


@pytest.mark.parametrize("chunks", [1, 3, 4, 5, 12])
def test_forward_from_pinned_host_buffers(chunks):
    """fa_fwd_from_host (copies of one slice of consecutive (b, h) heads
    overlapping the kernel of another, on three streams; slices that cross
    batch entries, uneven ones, one head each) gives bit for bit what fa_fwd
    gives on device-resident inputs, and matches the oracle; a second call
    reuses the staging buffers."""
    B, H, Nq, Nk, d = 4, 3, 300, 333, 128
    q, k, v = make_qkv(B, H, Nq, Nk, d, 4040 + chunks)
    scale = f32(1.0 / math.sqrt(d))
    o_dev, lse_dev = run_gpu(q, k, v, True, scale)
    qp, kp, vp = q.pin_memory(), k.pin_memory(), v.pin_memory()
    op = torch.empty((B, H, Nq, d), dtype=torch.bfloat16).pin_memory()
    lp = torch.empty((B, H, Nq), dtype=torch.float32).pin_memory()
    qd, kd, vd = (torch.empty(t.shape, dtype=t.dtype, device="cuda") for t in (q, k, v))
    od = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device="cuda")
    ld = torch.empty((B, H, Nq), dtype=torch.float32, device="cuda")
    for _ in range(2):
        op.fill_(float("nan"))
        lp.fill_(float("nan"))
        fa.fa_fwd_from_host(qp, kp, vp, op, lp, qd, kd, vd, od, ld, True, scale, chunks=chunks)
        torch.cuda.current_stream().synchronize()
        assert fa.fa_device_status(clear=True) == fa.FA_OK
        assert torch.equal(op, o_dev.cpu()) and torch.equal(lp, lse_dev.cpu())
    o_ref, lse_ref = oracle.attention_f64(to_f64(q), to_f64(k), to_f64(v), scale, True)
    check(op, lp, o_ref, lse_ref, f"from host, {chunks} chunks")


# ---------------------------------------------------------------- full sizes
#
# Every benchmark workload is compared with the oracle on its whole output,
# element by element, in the launch configuration the benchmark times: every
# row of every head (the large-head-dim workload included) and, for the
# split-KV workload, every split count the benchmark sweeps. The oracle runs
# per head in spawn-started worker processes (heads are independent problems).


@pytest.fixture(scope="module")
def head_pool():
    from oracle.parallel import HeadPool

    with HeadPool() as pool:
        yield pool


class WholeCheck:
    """The acceptance test of `check`, accumulated over a tensor head by head:
    max-abs and LSE errors over every element, relative L2 over the whole
    tensor."""

    def __init__(self, what):
        self.what = what
        self.max_abs = 0.0
        self.lse_err = 0.0
        self.err2 = 0.0
        self.ref2 = 0.0
        self.heads = 0

    def add(self, o, lse, o_ref, lse_ref, head):
        o = np.asarray(o, dtype=np.float64)
        lse = np.asarray(lse, dtype=np.float64)
        assert np.all(np.isfinite(o)), f"{self.what}: non-finite O in head {head}"
        diff = o - o_ref
        self.max_abs = max(self.max_abs, float(np.abs(diff).max()))
        self.err2 += float(np.square(diff).sum())
        self.ref2 += float(np.square(o_ref).sum())
        empty = ~np.isfinite(lse_ref)
        assert np.array_equal(np.isneginf(lse), empty), f"{self.what}: -inf LSE rows differ, head {head}"
        if (~empty).any():
            self.lse_err = max(self.lse_err, float(np.abs(lse[~empty] - lse_ref[~empty]).max()))
        self.heads += 1

    def finish(self, heads):
        assert self.heads == heads
        rel = math.sqrt(self.err2 / max(self.ref2, 1e-300))
        assert self.max_abs <= MAX_ABS, f"{self.what}: max-abs {self.max_abs:.3e}"
        assert rel <= REL_L2, f"{self.what}: rel-L2 {rel:.3e}"
        assert self.lse_err <= LSE_ABS, f"{self.what}: LSE err {self.lse_err:.3e}"
        return self.max_abs, rel, self.lse_err


def whole_tensor_check(pool, c, inputs, splits=(1,), rows_per_cta=None):
    """Runs the GPU path once per split count (or, with ``rows_per_cta``,
    fa_fwd_rows) and compares each whole output with the oracle, head by
    head."""
    q, k, v = inputs
    B, H, Nq, Nk, d, causal = c["B"], c["H"], c["Nq"], c["Nk"], c["d"], c["causal"]
    scale = f32(1.0 / math.sqrt(d))
    outs = {}
    for S in splits:
        if rows_per_cta is None:
            o, lse = run_gpu(q, k, v, causal, scale, num_splits=S)
        else:
            o, lse = run_gpu_rows(q, k, v, causal, scale, rows_per_cta)
        outs[S] = (o.float().cpu().numpy().reshape(B * H, Nq, d), lse.cpu().numpy().reshape(B * H, Nq))
        del o, lse
    qh, kh, vh = (t.reshape(B * H, -1, d) for t in (q, k, v))
    tasks = ((h, qh[h].float().numpy(), kh[h].float().numpy(), vh[h].float().numpy(), scale, causal)
             for h in range(B * H))
    checks = {S: WholeCheck(f"{c.get('name', '')} B={B} H={H} Nq={Nq} Nk={Nk} d={d} {causal} splits={S}")
              for S in splits}
    for h, o_ref, lse_ref in pool.heads(tasks):
        for S in splits:
            checks[S].add(outs[S][0][h], outs[S][1][h], o_ref, lse_ref, h)
    return {S: checks[S].finish(B * H) for S in splits}


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("causal", [False, True, "bottom_right"])
def test_persistent_ctas_ragged(head_pool, d, causal):
    """More query units than four waves of CTAs (B=2, H=160, Nq=300, Nk=333:
    640 units of 256 rows, each head's last tile ragged), so fa_fwd runs
    persistent CTAs that walk several units each: every head against the
    oracle, and bit for bit the output of one unit per CTA (fa_fwd_rows with
    256 rows)."""
    B, H, Nq, Nk = 2, 160, 300, 333
    c = dict(B=B, H=H, Nq=Nq, Nk=Nk, d=d, causal=causal, name="persistent")
    q, k, v = make_qkv(B, H, Nq, Nk, d, 7100 + d)
    whole_tensor_check(head_pool, c, (q, k, v))
    scale = f32(1.0 / math.sqrt(d))
    o1, l1 = run_gpu(q, k, v, causal, scale)
    o2, l2 = run_gpu_rows(q, k, v, causal, scale, 256)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d", [128, 64])
@pytest.mark.parametrize("B,H,Nq,Nk,causal", [
    (8, 80, 1, 1000, False),          # one query row per head: tile 1 of every unit idle
    (2, 320, 129, 129, True),         # a one-row second tile
    (4, 80, 512, 77, "bottom_right"),  # fewer keys than one key tile
])
def test_persistent_ctas_small_units(head_pool, B, H, Nq, Nk, causal, d):
    """Persistent launches (at least four waves of units) whose units are
    short or partly idle; every head against the oracle and bit for bit one
    unit per CTA."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert fa.fa_fwd_grid_ctas(B, H, Nq, d, 1) >= 4 * sms
    c = dict(B=B, H=H, Nq=Nq, Nk=Nk, d=d, causal=causal, name="persistent, short units")
    q, k, v = make_qkv(B, H, Nq, Nk, d, 7400 + Nq + d)
    whole_tensor_check(head_pool, c, (q, k, v))
    scale = f32(1.0 / math.sqrt(d))
    o1, l1 = run_gpu(q, k, v, causal, scale)
    o2, l2 = run_gpu_rows(q, k, v, causal, scale, 256)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d", [128, 64])
def test_persistent_ctas_rows_without_keys(head_pool, d):
    """Persistent CTAs over units in which one or both tiles see no key
    (bottom-right alignment with Nq = 700 > Nk = 200: rows 0-499 see none, so
    the first unit of each head has no key step at all and the second has keys
    only in its second tile): 960 units, every head against the oracle (O = 0
    and LSE = -inf on rows that see no key) and bit for bit one unit per CTA."""
    B, H, Nq, Nk = 1, 320, 700, 200
    c = dict(B=B, H=H, Nq=Nq, Nk=Nk, d=d, causal="bottom_right", name="persistent, rows without keys")
    q, k, v = make_qkv(B, H, Nq, Nk, d, 7300 + d)
    whole_tensor_check(head_pool, c, (q, k, v))
    scale = f32(1.0 / math.sqrt(d))
    o1, l1 = run_gpu(q, k, v, "bottom_right", scale)
    o2, l2 = run_gpu_rows(q, k, v, "bottom_right", scale, 256)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("name", ["c1", "c2", "c2_causal", "c3", "c3_causal", "c4"])
def test_full_size_whole_tensor(head_pool, name):
    """Whole O and LSE of each benchmark workload against the oracle (C4 with its
    1 % of key rows scaled x8)."""
    c = dict(CONFIGS[name], name=name)
    whole_tensor_check(head_pool, c, config_inputs(name))


def test_full_size_splitkv_whole_tensor(head_pool):
    """The split-KV workload through fa_fwd_splitkv + fa_combine at every split
    count the benchmark sweeps: the printed 1, 2, 3, 4, 16, 64 and the largest
    count whose grid fits one CTA per SM."""
    c = dict(CONFIGS["c5"], name="c5")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    fill = max(S for S in range(1, fa.FA_MAX_SPLITS + 1)
               if fa.fa_fwd_grid_ctas(c["B"], c["H"], c["Nq"], c["d"], S) <= sms)
    whole_tensor_check(head_pool, c, config_inputs("c5"), splits=sorted({1, 2, 3, 4, 16, 64, fill}))


def test_full_size_bottom_right_prefill(head_pool):
    """The benchmark's chunked-prefill workload: 4096 new queries over 8192 keys
    with the bottom-right causal mask, B=1, H=32, d=128."""
    c = dict(B=1, H=32, Nq=4096, Nk=8192, d=128, causal="bottom_right", name="prefill")
    whole_tensor_check(head_pool, c, make_qkv(1, 32, 4096, 8192, 128, 1006))


@pytest.mark.parametrize("name", ["c3", "c3_causal"])
def test_full_size_one_tile_per_cta(head_pool, name):
    """The long-sequence workload's query-tile sweep point of 128 rows per CTA
    (fa_fwd_rows): whole O and LSE against the oracle."""
    c = dict(CONFIGS[name], name=name + " rows=128")
    whole_tensor_check(head_pool, c, config_inputs(name), rows_per_cta=128)


@pytest.mark.parametrize("name", ["c3", "c3_causal"])
def test_full_size_64_row_tiles(head_pool, name):
    """The sweep point of 64 rows per CTA (fa_fwd_rows; M = 64 MMAs): whole O
    and LSE of the long-sequence workload against the oracle."""
    c = dict(CONFIGS[name], name=name + " rows=64")
    whole_tensor_check(head_pool, c, config_inputs(name), rows_per_cta=64)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True, "bottom_right"])
@pytest.mark.parametrize("Nq,Nk", [(389, 457), (1, 300), (63, 64), (700, 200), (200, 1)])
def test_64_row_tiles(d, causal, Nq, Nk):
    """64 query rows per CTA: ragged shapes (a tail in the 64-row tile and in
    the key tile, one query row, rows that see no key) against the oracle, and
    bit for bit fa_fwd's output (a row's arithmetic does not depend on the
    MMA height that computes it)."""
    B, H = 2, 3
    q, k, v = make_qkv(B, H, Nq, Nk, d, 970 + d + Nq)
    scale = f32(1.0 / math.sqrt(d))
    o, lse = run_gpu_rows(q, k, v, causal, scale, 64)
    oo, ll = oracle.attention_f64(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    check(o, lse, oo, ll, f"rows=64 d={d} {causal} Nq={Nq} Nk={Nk}")
    o_ref, lse_ref = run_gpu(q, k, v, causal, scale)
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("causal", [False, True, "bottom_right"])
def test_rows_per_cta_equal_fa_fwd(d, causal):
    """A row's arithmetic does not depend on which CTA or tile slot computes
    it: fa_fwd_rows gives fa_fwd's output bit for bit on ragged shapes, for
    every offered tile size, and matches the oracle."""
    B, H, Nq, Nk = 2, 3, 389, 457
    q, k, v = make_qkv(B, H, Nq, Nk, d, 960 + d)
    scale = f32(1.0 / math.sqrt(d))
    o_ref, lse_ref = run_gpu(q, k, v, causal, scale)
    for rows in ((128, 256) if d <= 128 else (128,)):
        o, lse = run_gpu_rows(q, k, v, causal, scale, rows)
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), rows
    oo, ll = oracle.attention_f64(to_f64(q), to_f64(k), to_f64(v), scale, causal)
    check(o, lse, oo, ll, f"rows d={d} {causal}")
