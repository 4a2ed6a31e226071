"""Planted mistakes in the oracle must each fail at least one pin.

Each mutant is a copy of ``oracle/attention.py`` with one textual change (a
dropped term, a wrong sign or index, a transposed operand, a shifted mask), run
on the CPU.  A mutant that passes every pin would mean the pins cannot tell
that mistake from the correct oracle.
"""

import os
import types

import warnings

import pytest

import oracle
from oracle_pins import ALL_PINS, BWD_PINS, FP8_PINS

SRC = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                   "oracle", "attention.py")
SRC_FP8 = os.path.join(os.path.dirname(SRC), "fp8.py")
SRC_BWD = os.path.join(os.path.dirname(SRC), "backward.py")

MUTANTS = [
    ("dropped scale", "s = float(scale) * (q[rows] @ k.T)", "s = (q[rows] @ k.T)"),
    ("keys used as queries", "s = float(scale) * (q[rows] @ k.T)",
     "s = float(scale) * (k[rows % k.shape[0]] @ k.T)"),
    ("mask includes diagonal", "cols[None, :] > rows[:, None] + off", "cols[None, :] >= rows[:, None] + off"),
    ("mask flipped", "cols[None, :] > rows[:, None] + off", "cols[None, :] < rows[:, None] + off"),
    ("bottom-right offset sign", "return nk - nq", "return nq - nk"),
    ("bottom-right as top-left", "return nk - nq", "return 0"),
    ("varlen keys of the next sequence", "k[k0:k1].transpose(1, 0, 2),", "k[k0:k1 + 1].transpose(1, 0, 2),"),
    ("varlen values shifted", "v[k0:k1].transpose(1, 0, 2), scale, causal)", "v[k0 + 1:k1 + 1].transpose(1, 0, 2), scale, causal)"),
    ("lse sign", "lse = np.where(empty, NEG_INF, m_ref + np.log(l))",
     "lse = np.where(empty, NEG_INF, m_ref - np.log(l))"),
    ("lse drops max", "lse = np.where(empty, NEG_INF, m_ref + np.log(l))",
     "lse = np.where(empty, NEG_INF, np.log(l))"),
    ("min instead of max", "m = s.max(axis=1)", "m = s.min(axis=1)"),
    ("no normalisation", "o = np.where(empty[:, None], 0.0, o / l[:, None])",
     "o = np.where(empty[:, None], 0.0, o)"),
    ("values reversed", "o = p @ v\n", "o = p @ v[::-1]\n"),
    ("dropped l rescale", "l = corr * l + p.sum(axis=1)", "l = l + p.sum(axis=1)"),
    ("dropped O rescale", "o = corr[:, None] * o + p @ v[a:b]", "o = o + p @ v[a:b]"),
    ("rescale sign", "corr = np.exp(m - ref)", "corr = np.exp(ref - m)"),
    ("block off by one", "x = s[:, a:b]", "x = s[:, a:b + 1]"),
    ("merge weight sign", "w = np.exp(ms - ref[None, :])", "w = np.exp(ref[None, :] - ms)"),
    ("merge drops l weight", "big_l = (w * ls).sum(axis=0)", "big_l = ls.sum(axis=0)"),
    ("merge lse drops max", "lse = np.where(big_l > 0, ref + np.log(big_l), NEG_INF)",
     "lse = np.where(big_l > 0, np.log(big_l), NEG_INF)"),
    ("wrong merge is right", "outs = [st[2] / st[1][:, None] for st in states if np.all(st[1] > 0)]\n    return np.mean(np.stack(outs), axis=0)",
     "return merge_states_f64(states)[0]"),
]


def _load_mutant(find, repl):
    with open(SRC, encoding="utf-8") as f:
        src = f.read()
    assert src.count(find) == 1, f"mutation anchor not unique: {find!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(find, repl), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,find,repl", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(name, find, repl):
    mod = _load_mutant(find, repl)
    caught = []
    warnings.simplefilter("ignore", RuntimeWarning)
    for pin in ALL_PINS:
        try:
            pin(mod)
        except Exception as e:  # AssertionError, or a crash from a broken shape
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"mutant '{name}' passed every pin"


FP8_MUTANTS = [
    ("exponent bias 6", "np.exp2(e - 7.0)", "np.exp2(e - 6.0)"),
    ("subnormal scale 2^-7", "m / 8.0 * 2.0 ** -6", "m / 8.0 * 2.0 ** -7"),
    ("no implicit one", "(1.0 + m / 8.0) * np.exp2(e - 7.0)", "(m / 8.0) * np.exp2(e - 7.0)"),
    ("four mantissa bits", "(1.0 + m / 8.0)", "(1.0 + m / 16.0)"),
    ("sign ignored", "sign = np.where((c >> 7) & 1, -1.0, 1.0)", "sign = 1.0"),
    ("e5m2 fields", "e = (c >> 3) & 0xF", "e = (c >> 2) & 0x1F"),
    ("top exponent as NaN", "(e == 15) & (m == 7)", "(e == 15)"),
    ("q descale dropped", "q = e4m3_decode(q8) * float(q_descale)\n    k = e4m3_decode(k8) * float(k_descale)\n    v = e4m3_decode(v8) * float(v_descale)\n    return",
     "q = e4m3_decode(q8)\n    k = e4m3_decode(k8) * float(k_descale)\n    v = e4m3_decode(v8) * float(v_descale)\n    return"),
    ("v descale squared", "v = e4m3_decode(v8) * float(v_descale)\n    return", "v = e4m3_decode(v8) * float(v_descale) ** 2\n    return"),
    ("sigma without the 1/3", "(E4M3_REL_HALF_ULP * p) ** 2 / 3.0", "(E4M3_REL_HALF_ULP * p) ** 2"),
    ("sigma over l, not l^2", "/ np.where(l > 0, l, 1.0) ** 2", "/ np.where(l > 0, l, 1.0)"),
    ("sigma relative to the max", "(E4M3_REL_HALF_ULP * p) ** 2 / 3.0", "(E4M3_REL_HALF_ULP * 1.0) ** 2 / 3.0"),
]


def _load_fp8_mutant(find, repl):
    with open(SRC_FP8, encoding="utf-8") as f:
        src = f.read()
    assert src.count(find) == 1, f"mutation anchor not unique: {find!r}"
    src = src.replace(find, repl).replace("from .attention import", "from oracle.attention import")
    mod = types.ModuleType("oracle_fp8_mutant")
    exec(compile(src, "oracle_fp8_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,find,repl", FP8_MUTANTS, ids=[m[0] for m in FP8_MUTANTS])
def test_fp8_mutant_is_caught(name, find, repl):
    mod = _load_fp8_mutant(find, repl)
    caught = []
    warnings.simplefilter("ignore", RuntimeWarning)
    for pin in FP8_PINS:
        try:
            pin(mod)
        except Exception as e:
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"mutant '{name}' passed every pin"


BWD_MUTANTS = [
    ("dV with the keys reversed", "dv[g] = p.T @ doh[g]", "dv[g] = p[:, ::-1].T @ doh[g]"),
    ("dP from K instead of V", "dp = doh[g] @ vh[g].T", "dp = doh[g] @ np.resize(kh[g], vh[g].shape).T"),
    ("D dropped", "ds = p * (dp - dd)", "ds = p * dp"),
    ("D sign", "ds = p * (dp - dd)", "ds = p * (dp + dd)"),
    ("D from the row max", "dd = (p * dp).sum(axis=1, keepdims=True)", "dd = dp.max(axis=1, keepdims=True)"),
    ("dQ without scale", "dq[g] = float(scale) * (ds @ kh[g])", "dq[g] = ds @ kh[g]"),
    ("dK without scale", "dk[g] = float(scale) * (ds.T @ qh[g])", "dk[g] = ds.T @ qh[g]"),
    ("dK from dS, not its transpose", "dk[g] = float(scale) * (ds.T @ qh[g])", "dk[g] = float(scale) * (ds[::-1, ::-1].T @ qh[g])[:kh.shape[1]]"),
    ("mask ignored", "            s = np.where(cols > rows + off, -np.inf, s)\n", "            pass\n"),
    ("unnormalised P", "p = np.where(l > 0, e / np.where(l > 0, l, 1.0), 0.0)", "p = e"),
]


def _load_bwd_mutant(find, repl):
    with open(SRC_BWD, encoding="utf-8") as f:
        src = f.read()
    assert src.count(find) == 1, f"mutation anchor not unique: {find!r}"
    src = src.replace(find, repl).replace("from .attention import", "from oracle.attention import")
    mod = types.ModuleType("oracle_bwd_mutant")
    exec(compile(src, "oracle_bwd_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,find,repl", BWD_MUTANTS, ids=[m[0] for m in BWD_MUTANTS])
def test_bwd_mutant_is_caught(name, find, repl):
    mod = _load_bwd_mutant(find, repl)
    caught = []
    warnings.simplefilter("ignore", RuntimeWarning)
    for pin in BWD_PINS:
        try:
            pin(mod, oracle)
        except Exception as e:
            caught.append((pin.__name__, type(e).__name__))
    assert caught, f"mutant '{name}' passed every pin"
