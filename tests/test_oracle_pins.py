"""Pins for the float64 oracle: it is checked against things other than itself.

Each pin is a closed form, an exact rational brute force, an invariant, a
textbook special case, a hand-worked example (tests/golden/hand_examples.json)
or a figure the pages print (tests/golden/page_figures.json). The planted-
mistake tests at the bottom mutate the oracle on the CPU and check that some pin
fails, so a dropped term, a wrong weight, a wrong mask or a swapped operand in
the oracle cannot pass unnoticed.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from oracle import tsa_oracle as O
from fixed_state_recurrence_phi_b300.inputs import np_qkv

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def _order_slices(d, n):
    out, off = [], 0
    for m in range(n):
        w = math.comb(d + m - 1, m)
        out.append(slice(off, off + w))
        off += w
    return out


# ---------------------------------------------------------------------------
# pins (plain functions so the planted-mistake tests can re-run them)
# ---------------------------------------------------------------------------

def pin_widths():
    """Width of the m-th state is C(d+m-1, m) (Expanding Attention, abstract)."""
    for d in range(1, 33):
        for m in range(0, 5):
            mons = O.monomials(d, m)
            assert len(mons) == math.comb(d + m - 1, m), (d, m)
            assert len(set(mons)) == len(mons)
            assert all(list(t) == sorted(t) for t in mons)
        assert O.feature_dim(d, 4) == sum(math.comb(d + m - 1, m) for m in range(4))
    # the workload widths: 1+16+136 = 153, 1+16+136+816 = 969, 1+32+528 = 561
    assert O.feature_dim(16, 3) == 153
    assert O.feature_dim(16, 4) == 969
    assert O.feature_dim(32, 3) == 561
    assert O.feature_dim(16, 5) == 4845 == 969 + math.comb(19, 4)
    x = np.random.default_rng(1).standard_normal((3, 7))
    assert O.phi(x, 4).shape == (3, O.feature_dim(7, 4))


def pin_page_state_size():
    g = _load("page_figures.json")["state_elems_per_head_n3"]
    assert O.state_elems(g["d_k"], g["d_v"], g["n_terms"]) == g["value"] == (1 + 16 + 136) * 65


def pin_phi_closed_form():
    """<phi_m(q), phi_m(k)> = (q.k)^m / m! and |phi_m(k)|^2 = |k|^(2m) / m!."""
    rng = np.random.default_rng(7)
    for d in (3, 16, 32):
        n = 5 if d < 32 else 4
        q = rng.standard_normal((20, d)); k = rng.standard_normal((20, d))
        fq, fk = O.phi(q, n), O.phi(k, n)
        x = np.sum(q * k, axis=1)
        kk = np.sum(k * k, axis=1)
        for m, sl in enumerate(_order_slices(d, n)):
            ip = np.sum(fq[:, sl] * fk[:, sl], axis=1)
            ref = x ** m / math.factorial(m)
            assert np.allclose(ip, ref, rtol=1e-12, atol=1e-12), (d, m)
            nrm = np.sum(fk[:, sl] ** 2, axis=1)
            assert np.allclose(nrm, kk ** m / math.factorial(m), rtol=1e-12), (d, m)


def pin_phi_full_tensor_power():
    """The symmetric packing equals the full d^m tensor power with 1/m!:
    sum over all ordered tuples of q_i1..q_im k_i1..k_im / m!."""
    rng = np.random.default_rng(3)
    d, n = 4, 5
    q = rng.standard_normal(d); k = rng.standard_normal(d)
    fq, fk = O.phi(q, n), O.phi(k, n)
    for m, sl in enumerate(_order_slices(d, n)):
        full = 0.0
        for t in itertools.product(range(d), repeat=m):
            full += np.prod([q[i] for i in t]) * np.prod([k[i] for i in t])
        assert abs(np.dot(fq[sl], fk[sl]) - full / math.factorial(m)) < 1e-12


def pin_svd_width():
    """Stacked vec(k^{(x)m}) over many keys has rank C(d+m-1, m), the bound the
    abstract says SVD confirms; the packed features have full column rank."""
    rng = np.random.default_rng(11)
    d = 16
    for m in (1, 2, 3):
        w = math.comb(d + m - 1, m)
        K = rng.standard_normal((w + 200, d))
        T = K
        for _ in range(m - 1):
            T = np.einsum("ni,nj->nij", T, K).reshape(K.shape[0], -1)
        assert T.shape[1] == d ** m
        assert np.linalg.matrix_rank(T) == w
    K = rng.standard_normal((400, d))
    assert np.linalg.matrix_rank(O.phi(K, 3)) == O.feature_dim(d, 3)


def pin_taylor_kernel():
    x = np.linspace(-1, 1, 201)
    assert np.all(O.taylor_kernel(x, 1) == 1.0)
    assert np.allclose(O.taylor_kernel(x, 2), 1 + x, atol=0)
    assert np.allclose(O.taylor_kernel(x, 3), 1 + x + x * x / 2, atol=1e-16)
    assert np.allclose(O.taylor_kernel(x, 20), np.exp(x), rtol=1e-15, atol=0)
    for n in range(1, 9):  # Lagrange remainder bound
        err = np.abs(np.exp(x) - O.taylor_kernel(x, n))
        assert np.all(err <= np.exp(np.abs(x)) * np.abs(x) ** n / math.factorial(n) + 1e-15)


def _frac_state_entry(e):
    return float(Fraction(e["rat"])) / (math.sqrt(2.0) ** e["inv_sqrt2"])


def pin_hand_examples():
    g = _load("hand_examples.json")
    for name in ("d1_n3", "d2_n3"):
        ex = g[name]
        n = ex["n_terms"]
        q = np.array([[float(Fraction(s)) for s in r] for r in ex["q"]])
        k = np.array([[float(Fraction(s)) for s in r] for r in ex["k"]])
        v = np.array([[float(Fraction(s)) for s in r] for r in ex["v"]])
        want = np.array([[float(Fraction(s)) for s in r] for r in ex["out"]])
        want_S = np.array([[_frac_state_entry(e) for e in r] for r in ex["state"]])
        assert np.allclose(O.attention_direct(q, k, v, n), want, rtol=1e-14, atol=1e-15), name
        out, S = O.prefill_recurrent(q, k, v, n)
        assert np.allclose(out, want, rtol=1e-14, atol=1e-15), name
        assert np.allclose(S, want_S, rtol=1e-14, atol=1e-15), name
        outc, Sc = O.prefill_chunked(q, k, v, n, 2)
        assert np.allclose(outc, want, rtol=1e-14, atol=1e-15), name
        assert np.allclose(Sc, want_S, rtol=1e-14, atol=1e-15), name


def _rand_frac(rng, shape, den=4, lo=-4, hi=4):
    return [[Fraction(int(rng.integers(lo, hi + 1)), den) for _ in range(shape[1])]
            for _ in range(shape[0])]


def pin_brute_force():
    """Exact rational agreement of the direct form, the symmetric recurrence and
    the full tensor-power recurrence; the float oracle within rounding of it."""
    rng = np.random.default_rng(5)
    for (d, N, dv, n) in [(1, 4, 2, 3), (2, 5, 2, 3), (3, 6, 1, 4), (2, 6, 3, 2), (3, 4, 2, 3)]:
        q = _rand_frac(rng, (N, d)); k = _rand_frac(rng, (N, d))
        v = _rand_frac(rng, (N, dv), den=2)
        a = O.brute_direct(q, k, v, n)
        b = O.brute_recurrent_symmetric(q, k, v, n)
        c = O.brute_recurrent_full(q, k, v, n)
        assert a == b == c, (d, N, dv, n)
        fa = np.array([[float(x) for x in r] for r in a])
        to = lambda M: np.array([[float(x) for x in r] for r in M])
        assert np.allclose(O.attention_direct(to(q), to(k), to(v), n), fa, rtol=1e-13, atol=1e-13)
        assert np.allclose(O.prefill_recurrent(to(q), to(k), to(v), n)[0], fa, rtol=1e-13, atol=1e-13)


def pin_recurrent_equals_direct():
    """Abstract: the recursion is lossless w.r.t. the truncated kernel (2.2e-16
    in float64). Pinned to the order of magnitude: relative <= 1e-14."""
    fig = _load("page_figures.json")["recurrence_vs_truncated_kernel_f64"]["value"]
    for (N, d, dv, n, seed) in [(256, 16, 64, 3, 0), (300, 16, 64, 4, 1), (200, 32, 128, 3, 2)]:
        q, k, v = np_qkv(N, d, dv, seed)
        a = O.attention_direct(q, k, v, n)
        r, _ = O.prefill_recurrent(q, k, v, n)
        rel = np.abs(a - r).max() / np.abs(a).max()
        assert rel <= 50 * fig, rel


def pin_chunk_additivity():
    """Abstract: states additive across chunks (5.7e-14). Chunk states summed vs
    the whole-sequence state; chunked output vs recurrent output."""
    fig = _load("page_figures.json")["chunk_additivity"]["value"]
    q, k, v = np_qkv(500, 16, 64, 4)
    out, S = O.prefill_recurrent(q, k, v, 3)
    for C in (1, 7, 64, 128, 500):
        cs = O.chunk_states(k, v, 3, C)
        assert len(cs) == -(-500 // C)
        assert np.abs(sum(cs) - S).max() <= 10 * fig
        oc, Sc = O.prefill_chunked(q, k, v, 3, C)
        assert np.abs(oc - out).max() / np.abs(out).max() <= 1e-14
        assert np.abs(Sc - S).max() <= 10 * fig
    # merge of two segments' states equals the state of the concatenation
    _, S1 = O.prefill_recurrent(q[:200], k[:200], v[:200], 3)
    _, S2 = O.prefill_recurrent(q[200:], k[200:], v[200:], 3)
    assert np.abs(O.state_merge(S1, S2) - S).max() <= 10 * fig
    # continuing from saved states equals one pass over the concatenation
    o2, S12 = O.prefill_recurrent(q[200:], k[200:], v[200:], 3, S0=S1)
    assert np.abs(o2 - out[200:]).max() <= 1e-14 and np.abs(S12 - S).max() <= 10 * fig


def pin_special_cases():
    q, k, v = np_qkv(200, 16, 8, 9)
    # n = 1: every weight is 1, so out_i is the running mean of v_0..v_i
    run_mean = np.cumsum(v, axis=0) / np.arange(1, 201)[:, None]
    assert np.allclose(O.attention_direct(q, k, v, 1), run_mean, rtol=1e-13, atol=1e-14)
    assert np.allclose(O.prefill_recurrent(q, k, v, 1)[0], run_mean, rtol=1e-13, atol=1e-14)
    # n = 20 on unit q, k: the truncation error e/20! ~ 1e-18 is below rounding,
    # so the result is exact causal softmax attention (textbook, via np.exp)
    sm = O.softmax_attention(q, k, v)
    assert np.abs(O.attention_direct(q, k, v, 20) - sm).max() <= 1e-14
    # exact softmax by a second, independent route: the first row is v_0 and
    # row i is a convex combination of v_0..v_i
    assert np.allclose(sm[0], v[0], atol=1e-15)


def pin_error_falls_with_n():
    """Accuracy improves with n on unit-normalised q, k (abstract; trade-offs
    bullet); without normalisation adding terms stops helping."""
    q, k, v = np_qkv(256, 16, 64, 0)
    sm = O.softmax_attention(q, k, v)
    errs = [np.abs(O.attention_direct(q, k, v, n) - sm).max() for n in range(1, 7)]
    assert all(a > b for a, b in zip(errs, errs[1:])), errs
    assert errs[-1] < 1e-4
    # scaled by 4, |q.k| reaches ~14: no order from 1 to 8 gets near softmax
    bad = [np.abs(O.attention_direct(4 * q, 4 * k, v, n) - O.softmax_attention(4 * q, 4 * k, v)).max()
           for n in range(1, 9)]
    assert min(bad) > 0.5, bad


def pin_state_invariants():
    q, k, v = np_qkv(321, 16, 64, 6)
    _, S = O.prefill_recurrent(q, k, v, 3)
    dv = 64
    assert S[0, dv] == 321.0                               # token count
    assert np.allclose(S[0, :dv], v.sum(0), atol=1e-12)    # sum of values
    assert np.allclose(S[1:17, dv], k.sum(0), atol=1e-12)  # order-1 normaliser = sum of keys
    # order-2 normaliser entries: sum_j k_ja k_jb / sqrt(a!)
    ent = [(a, b) for a in range(16) for b in range(a, 16)]
    want = np.array([np.sum(k[:, a] * k[:, b]) / (math.sqrt(2) if a == b else 1.0) for a, b in ent])
    assert np.allclose(S[17:153, dv], want, atol=1e-12)


def pin_decode_consistency():
    q, k, v = np_qkv(129, 16, 64, 8)
    out_all, S_all = O.prefill_recurrent(q, k, v, 3)
    _, S = O.prefill_recurrent(q[:128], k[:128], v[:128], 3)
    o, S2 = O.decode_step(q[128], k[128], v[128], S, 3)
    assert np.abs(o - out_all[128]).max() <= 1e-14
    assert np.abs(S2 - S_all).max() <= 1e-12


PINS = [pin_widths, pin_page_state_size, pin_phi_closed_form, pin_phi_full_tensor_power,
        pin_svd_width, pin_taylor_kernel, pin_hand_examples, pin_brute_force,
        pin_recurrent_equals_direct, pin_chunk_additivity, pin_special_cases,
        pin_error_falls_with_n, pin_state_invariants, pin_decode_consistency]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin()


# ---------------------------------------------------------------------------
# planted mistakes: each mutation of the oracle must make some pin fail
# ---------------------------------------------------------------------------

def _phi_no_sqrt(x, n):
    x = np.asarray(x, np.float64); d = x.shape[-1]; cols = []
    for m in range(n):
        for idx in O.monomials(d, m):
            val = np.prod([x[..., i] for i in idx], axis=0) if idx else np.ones(x.shape[:-1])
            cols.append(val / O._alpha_factorial(idx))          # wrong: a! instead of sqrt(a!)
    return np.stack(cols, axis=-1)


def _taylor_dropped_term(x, n):
    x = np.asarray(x, np.float64); out = np.zeros_like(x)
    for m in range(n - 1):                                          # wrong: drops the last term
        out = out + x ** m / math.factorial(m)
    return out


def _direct_exclusive(q, k, v, n, row_block=1024):
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    N = q.shape[0]
    w = O.taylor_kernel(q @ k.T, n) * (np.arange(N)[None, :] < np.arange(N)[:, None] + 0)  # wrong: j < i
    w[0, 0] = 1.0
    return (w @ v) / w.sum(axis=1, keepdims=True)


def _recurrent_read_before_update(q, k, v, n, S0=None):
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    N, d_v = v.shape
    fq, fk = O.phi(q, n), O.phi(k, n)
    S = np.zeros((fq.shape[1], d_v + 1)); S[0, d_v] = 1e-300
    out = np.empty((N, d_v))
    vv = np.concatenate([v, np.ones((N, 1))], axis=1)
    for t in range(N):
        r = fq[t] @ S                                               # wrong: reads before the update
        out[t] = r[:d_v] / r[d_v]
        S += np.outer(fk[t], vv[t])
    return out, S


def _chunked_swapped(q, k, v, n, C, S0=None):
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    N, d_v = v.shape
    S = np.zeros((O.feature_dim(q.shape[1], n), d_v + 1)); out = np.empty((N, d_v))
    for c0 in range(0, N, C):
        c1 = min(N, c0 + C); L = c1 - c0
        vv = np.concatenate([v[c0:c1], np.ones((L, 1))], axis=1)
        inter = O.phi(k[c0:c1], n) @ S                              # wrong: phi(K) in the readout
        w = O.taylor_kernel(q[c0:c1] @ k[c0:c1].T, n) * (np.arange(L)[None, :] <= np.arange(L)[:, None])
        r = inter + w @ vv
        out[c0:c1] = r[:, :d_v] / r[:, d_v:]
        S = S + O.phi(k[c0:c1], n).T @ vv
    return out, S


def _monomials_no_repeat(d, m):
    return list(itertools.combinations(range(d), m))               # wrong: drops x_i^2 terms


MUTATIONS = [
    ("phi", _phi_no_sqrt),
    ("taylor_kernel", _taylor_dropped_term),
    ("attention_direct", _direct_exclusive),
    ("prefill_recurrent", _recurrent_read_before_update),
    ("prefill_chunked", _chunked_swapped),
    ("monomials", _monomials_no_repeat),
]


@pytest.mark.parametrize("name,bad", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, bad):
    monkeypatch.setattr(O, name, bad)
    caught = 0
    for pin in PINS:
        try:
            with np.errstate(all="ignore"):
                pin()
        except (AssertionError, ValueError, ZeroDivisionError, FloatingPointError):
            caught += 1
    assert caught > 0, f"no pin caught the planted mistake in {name}"
