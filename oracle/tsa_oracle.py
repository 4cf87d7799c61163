"""Float64 CPU oracle for truncated-Taylor, fixed-state causal attention.

TEST INFRASTRUCTURE ONLY. This module is the checker, not the product: only the
test suite, the package's smoke check and the benchmark's CPU-baseline leg may
import it. It shares no code, tables or constants with the CUDA library, and it
imports nothing from the package.

What is computed (the plain definition, per attention head):

    T_n(x) = sum_{m=0}^{n-1} x^m / m!                 (truncated exp, x = q.k)
    out_i  = sum_{j<=i} T_n(q_i.k_j) v_j / sum_{j<=i} T_n(q_i.k_j)

Sources (web pages on the method; cited by title and section):
  [EA]  "Expanding Attention: A Taylor-Series Route to Linear-Time Transformers
        with a Fixed Number of Recurrent States" (wpnews.pro), the quoted arXiv
        2610.20637v1 abstract: truncate the exponential kernel to n Taylor terms,
        factor each term as a tensor-power inner product, fold the causal history
        into n states updated by one rank-one outer product per token; states are
        additive across chunks; the m-th state is C(d+m-1, m) wide.
  [AX]  "arXiv Introduces New Linear-Time Transformer Method via Taylor Series
        Expansion and Fixed-State Recurrence" (zicq.com), sections "Technical
        Mechanism Analysis" (items 1-2: lossless recursion, additive states) and
        "Engineering Trade-offs and Performance" (width, n=3 optimum, q/k
        normalisation).
  [HN]  Hacker News thread on the paper (item 46888355): the comment explaining
        the "+1" column of the state as the softmax normaliser, and the comment
        giving the chunk algebra (Q'K)V = Q'(KV).

Readings taken where the pages are silent (each is also listed in the design
notes): no 1/sqrt(d) score scale (x = q.k on unit vectors); "n terms" means orders
0..n-1; the causal mask is inclusive (j <= i); the normaliser column carries
sum_j T_n with no epsilon; the multinomial weight is split symmetrically,
phi_m(x)_a = x^a / sqrt(a!), so that <phi_m(q), phi_m(k)> = (q.k)^m / m!;
monomials are ordered as itertools.combinations_with_replacement yields them,
orders concatenated in ascending m.

State layout used here (canonical): S has shape [D, d_v + 1]; column d_v is the
normaliser z = sum_j phi(k_j).

Every function below is pinned by tests/test_oracle_pins.py against closed forms,
exact rational brute force, invariants and the figures the pages print.
"""
from __future__ import annotations

import itertools
import math
from fractions import Fraction

import numpy as np

__all__ = [
    "monomials", "feature_dim", "state_elems", "phi", "taylor_kernel",
    "attention_direct", "prefill_recurrent", "chunk_states", "prefill_chunked",
    "decode_step", "state_merge", "softmax_attention",
    "brute_direct", "brute_recurrent_symmetric", "brute_recurrent_full",
]


# ---------------------------------------------------------------------------
# Feature map: symmetric tensor powers ([EA] abstract; [AX] trade-offs: width
# C(d+m-1, m) per order)
# ---------------------------------------------------------------------------

def monomials(d: int, m: int) -> list[tuple[int, ...]]:
    """Index tuples i_1 <= ... <= i_m of the degree-m monomials in d variables.

    Their number is C(d+m-1, m), the width the pages give for the m-th state.
    """
    return list(itertools.combinations_with_replacement(range(d), m))


def _alpha_factorial(idx: tuple[int, ...]) -> int:
    """a! = prod_i a_i! for the multi-index a whose counts come from idx."""
    out = 1
    for i in set(idx):
        out *= math.factorial(idx.count(i))
    return out


def feature_dim(d: int, n: int) -> int:
    """D = sum_{m<n} C(d+m-1, m): total feature width for n Taylor terms."""
    return sum(len(monomials(d, m)) for m in range(n))


def state_elems(d: int, d_v: int, n: int) -> int:
    """Elements per head of the fixed state: D * (d_v + 1) (+1: normaliser)."""
    return feature_dim(d, n) * (d_v + 1)


def phi(x: np.ndarray, n: int) -> np.ndarray:
    """Concatenated symmetric feature map [phi_0 | phi_1 | ... | phi_{n-1}].

    phi_m(x)_a = x^a / sqrt(a!) for each multi-index |a| = m, so that
    <phi_m(q), phi_m(k)> = sum_{|a|=m} q^a k^a / a! = (q.k)^m / m!
    (multinomial theorem). x: [..., d] -> [..., D], float64.
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    cols = []
    for m in range(n):
        for idx in monomials(d, m):
            val = np.ones(x.shape[:-1], dtype=np.float64)
            for i in idx:
                val = val * x[..., i]
            cols.append(val / math.sqrt(_alpha_factorial(idx)))
    return np.stack(cols, axis=-1)


def taylor_kernel(x: np.ndarray, n: int) -> np.ndarray:
    """T_n(x) = sum_{m=0}^{n-1} x^m / m!, the n-term truncation of exp(x)."""
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros_like(x)
    for m in range(n):
        out = out + x ** m / math.factorial(m)
    return out


# ---------------------------------------------------------------------------
# Attention in its three forms
# ---------------------------------------------------------------------------

def attention_direct(q, k, v, n: int, row_block: int = 1024) -> np.ndarray:
    """Direct O(N^2) causal attention with the truncated kernel.

    out_i = sum_{j<=i} T_n(q_i.k_j) v_j / sum_{j<=i} T_n(q_i.k_j).
    Rows are processed in blocks only to bound memory; each row is the plain
    definition. q, k: [N, d]; v: [N, d_v] -> [N, d_v].
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    N = q.shape[0]
    out = np.empty((N, v.shape[1]), dtype=np.float64)
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        w = taylor_kernel(q[r0:r1] @ k[:r1].T, n)            # [rows, r1]
        w = w * (np.arange(r1)[None, :] <= np.arange(r0, r1)[:, None])
        out[r0:r1] = (w @ v[:r1]) / w.sum(axis=1, keepdims=True)
    return out


def prefill_recurrent(q, k, v, n: int, S0=None):
    """Recurrent form: one rank-one state update per token, then the readout.

    S <- S + phi(k_t) [v_t; 1]^T ;  r = phi(q_t)^T S ;  out_t = r[:d_v] / r[d_v]
    ([EA] abstract: n states, each updated by one rank-one outer product per
    token; [HN] the +1 column carries the softmax normaliser). The inclusive
    mask (update before readout) is the reading taken for causality.
    Returns (out [N, d_v], S [D, d_v + 1]).
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    N, d_v = v.shape
    fq, fk = phi(q, n), phi(k, n)
    D = fq.shape[1]
    S = np.zeros((D, d_v + 1)) if S0 is None else np.array(S0, np.float64, copy=True)
    out = np.empty((N, d_v))
    vv = np.concatenate([v, np.ones((N, 1))], axis=1)
    for t in range(N):
        S += np.outer(fk[t], vv[t])
        r = fq[t] @ S
        out[t] = r[:d_v] / r[d_v]
    return out, S


def chunk_states(k, v, n: int, C: int) -> list[np.ndarray]:
    """State contribution of each chunk of C tokens: phi(K_c)^T [V_c, 1].

    Additivity across chunks ([EA] abstract; [AX] "Technical Mechanism
    Analysis" item 2) says these sum to the whole-sequence state.
    """
    k = np.asarray(k, np.float64); v = np.asarray(v, np.float64)
    N = k.shape[0]
    out = []
    for c0 in range(0, N, C):
        fk = phi(k[c0:c0 + C], n)
        vv = np.concatenate([v[c0:c0 + C], np.ones((fk.shape[0], 1))], axis=1)
        out.append(fk.T @ vv)
    return out


def prefill_chunked(q, k, v, n: int, C: int, S0=None):
    """Chunked form: (Q'K)V inside a chunk, Q'(KV) across chunks ([HN] chunk
    algebra comment; [EA] additivity makes prefill a scan over chunks).

    For chunk c: inter = phi(Q_c) S_{<c}; intra = mask(T_n(Q_c K_c^T)) [V_c, 1];
    out = (inter + intra)[:, :d_v] / (inter + intra)[:, d_v];
    S_{<c+1} = S_{<c} + phi(K_c)^T [V_c, 1].
    Returns (out [N, d_v], S [D, d_v + 1]).
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    N, d_v = v.shape
    D = feature_dim(q.shape[1], n)
    S = np.zeros((D, d_v + 1)) if S0 is None else np.array(S0, np.float64, copy=True)
    out = np.empty((N, d_v))
    for c0 in range(0, N, C):
        c1 = min(N, c0 + C)
        qc, kc = q[c0:c1], k[c0:c1]
        vv = np.concatenate([v[c0:c1], np.ones((c1 - c0, 1))], axis=1)
        inter = phi(qc, n) @ S
        L = c1 - c0
        w = taylor_kernel(qc @ kc.T, n) * (np.arange(L)[None, :] <= np.arange(L)[:, None])
        r = inter + w @ vv
        out[c0:c1] = r[:, :d_v] / r[:, d_v:d_v + 1]
        S = S + phi(kc, n).T @ vv
    return out, S


def decode_step(q, k, v, S, n: int):
    """One decode token for one head: S' = S + phi(k)[v; 1]^T, then the readout
    out = (phi(q)^T S')[:d_v] / (phi(q)^T S')[d_v]. Cost independent of the
    context length ([EA] abstract, constant per-token decoding).
    q, k: [d]; v: [d_v]; S: [D, d_v + 1]. Returns (out [d_v], S').
    """
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    S2 = np.asarray(S, np.float64) + np.outer(phi(k, n), np.append(v, 1.0))
    r = phi(q, n) @ S2
    return r[:-1] / r[-1], S2


def state_merge(a, b):
    """States of two consecutive segments combine by addition ([EA] abstract)."""
    return np.asarray(a, np.float64) + np.asarray(b, np.float64)


def softmax_attention(q, k, v, row_block: int = 1024) -> np.ndarray:
    """Exact causal softmax attention with weights exp(q.k) (the comparator the
    pages measure error and speed against). Max-subtracted per row."""
    q = np.asarray(q, np.float64); k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    N = q.shape[0]
    out = np.empty((N, v.shape[1]))
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        s = q[r0:r1] @ k[:r1].T
        mask = np.arange(r1)[None, :] <= np.arange(r0, r1)[:, None]
        s = np.where(mask, s, -np.inf)
        w = np.exp(s - s.max(axis=1, keepdims=True))
        out[r0:r1] = (w @ v[:r1]) / w.sum(axis=1, keepdims=True)
    return out


# ---------------------------------------------------------------------------
# Exact rational brute force (tiny inputs; d <= 3, N <= 6)
# ---------------------------------------------------------------------------

def _dot(a, b):
    return sum((x * y for x, y in zip(a, b)), Fraction(0))


def brute_direct(q, k, v, n: int):
    """Direct form in exact rationals: weights sum_{m<n} (q.k)^m / m!."""
    N = len(q)
    out = []
    for i in range(N):
        w = [sum((_dot(q[i], k[j]) ** m / math.factorial(m) for m in range(n)),
                 Fraction(0)) for j in range(i + 1)]
        den = sum(w, Fraction(0))
        out.append([sum((w[j] * v[j][c] for j in range(i + 1)), Fraction(0)) / den
                    for c in range(len(v[0]))])
    return out


def brute_recurrent_symmetric(q, k, v, n: int):
    """Recurrent form in exact rationals with the multinomial weight kept whole
    on the key side: query feature q^a, key feature k^a / a!, over symmetric
    multi-indices a (all rational, no square roots)."""
    d = len(q[0]); dv = len(v[0])
    feats = [idx for m in range(n) for idx in monomials(d, m)]

    def mono(x, idx):
        p = Fraction(1)
        for i in idx:
            p *= x[i]
        return p

    S = [[Fraction(0)] * (dv + 1) for _ in feats]
    out = []
    for t in range(len(q)):
        vv = list(v[t]) + [Fraction(1)]
        for a, idx in enumerate(feats):
            g = mono(k[t], idx) / _alpha_factorial(idx)
            for c in range(dv + 1):
                S[a][c] += g * vv[c]
        r = [sum((mono(q[t], idx) * S[a][c] for a, idx in enumerate(feats)), Fraction(0))
             for c in range(dv + 1)]
        out.append([r[c] / r[dv] for c in range(dv)])
    return out


def brute_recurrent_full(q, k, v, n: int):
    """Recurrent form in exact rationals over the full (non-symmetric) tensor
    power: all d^m ordered index tuples, query q^{(x)m}, key k^{(x)m} / m!."""
    d = len(q[0]); dv = len(v[0])
    feats = [(m, idx) for m in range(n) for idx in itertools.product(range(d), repeat=m)]

    def mono(x, idx):
        p = Fraction(1)
        for i in idx:
            p *= x[i]
        return p

    S = [[Fraction(0)] * (dv + 1) for _ in feats]
    out = []
    for t in range(len(q)):
        vv = list(v[t]) + [Fraction(1)]
        for a, (m, idx) in enumerate(feats):
            g = mono(k[t], idx) / math.factorial(m)
            for c in range(dv + 1):
                S[a][c] += g * vv[c]
        r = [sum((mono(q[t], idx) * S[a][c] for a, (m, idx) in enumerate(feats)),
                 Fraction(0)) for c in range(dv + 1)]
        out.append([r[c] / r[dv] for c in range(dv)])
    return out
