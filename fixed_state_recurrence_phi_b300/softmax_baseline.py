"""The exact causal softmax attention that the truncated-Taylor path is timed
against: causal prefill and one KV-cache decode step on the same GPU.

The pages state their speed results against exact softmax attention: prefill
time growing as N^2.28 against N^0.91 for the states, a crossover near
N = 728, 20.8x at N = 8192, and per-token decode latency growing as N^1.04
against a constant for the states, 76.0x at N = 65536 ("Expanding Attention:
A Taylor-Series Route to Linear-Time Transformers with a Fixed Number of
Recurrent States", abstract; "arXiv Introduces New Linear-Time Transformer
Method ...", Technical Mechanism Analysis, items 3 and 4).

This module is that comparator, not part of the method's path: it calls the
library's own attention kernels (torch scaled_dot_product_attention on its
cuDNN, flash or memory-efficient backend, never the math backend, which
materialises the N x N scores) so that the comparison is against the fastest
exact softmax this GPU has. The weights are exp(q.k) with scale 1, the
function whose Taylor series the method truncates. On CPU tensors the math
backend runs instead; that is only for checking the conventions without a GPU.

The library's fast kernels do not all take d_k != d_v. Zero-padding q and k
to d_v columns leaves every q.k unchanged, so the padded call computes the
same attention; `select` times the backends in both forms on
the inputs at hand and keeps the fastest, so the comparator is never
handicapped by a form the library runs slowly at that size.
"""
from __future__ import annotations

import statistics
import warnings

import torch
import torch.nn.functional as F
from torch.nn.attention import SDPBackend, sdpa_kernel

FAST_BACKENDS = (SDPBackend.CUDNN_ATTENTION, SDPBackend.FLASH_ATTENTION, SDPBackend.EFFICIENT_ATTENTION)
BACKEND_NAMES = {SDPBackend.CUDNN_ATTENTION: "cudnn", SDPBackend.FLASH_ATTENTION: "flash",
                 SDPBackend.EFFICIENT_ATTENTION: "efficient", SDPBackend.MATH: "math"}


def pad_columns(x: torch.Tensor, width: int) -> torch.Tensor:
    """x with zero columns appended up to `width` (inner products unchanged)."""
    return x if x.shape[-1] == width else F.pad(x, (0, width - x.shape[-1]))


class SoftmaxAttention:
    """Exact softmax attention with weights exp(q.k) on one backend and form.

    backend: an SDPBackend (None: the fast backends in the library's order on
    CUDA, the math backend on CPU). padded: q and k are zero-padded to d_v
    columns before the call (the caller stores keys padded, see `keys`).
    """

    def __init__(self, backend=None, padded: bool = False):
        self.backend = backend
        self.padded = padded

    @property
    def name(self) -> str:
        b = "default" if self.backend is None else BACKEND_NAMES[self.backend]
        return f"{b}{', q and k zero-padded to d_v' if self.padded else ''}"

    def _backends(self, device):
        if self.backend is not None:
            return [self.backend]
        return list(FAST_BACKENDS) if device.type == "cuda" else [SDPBackend.MATH]

    def attend(self, q, k, v, causal: bool):
        """softmax(q k^T) v with scale 1, causal or not, on this backend."""
        with sdpa_kernel(self._backends(q.device)):
            return F.scaled_dot_product_attention(q, k, v, is_causal=causal, scale=1.0)

    def keys(self, x: torch.Tensor, d_v: int) -> torch.Tensor:
        """q or k rows in the form this comparator stores and calls with."""
        return pad_columns(x, d_v) if self.padded else x

    def cache(self, k: torch.Tensor, v: torch.Tensor):
        """A KV cache ([B, H, N, *]) holding these keys and values in this
        comparator's form (its own copies)."""
        return self.keys(k, v.shape[-1]).clone(), v.clone()

    def prefill(self, q, k, v) -> torch.Tensor:
        """Causal attention over [B, H, N, *]: out_i = sum_{j<=i} e^{q_i.k_j} v_j
        / sum_{j<=i} e^{q_i.k_j}. q and k as returned by `keys`."""
        return self.attend(q, k, v, causal=True)

    def decode_step(self, q1, k1, v1, k_cache, v_cache, pos: int) -> torch.Tensor:
        """One decode step with a KV cache: write token `pos`'s k and v into the
        caches ([B, H, >pos, *]), then attend q1 ([B, H, d]) over tokens 0..pos.
        Returns [B, H, d_v]."""
        k_cache[:, :, pos, : k1.shape[-1]] = k1
        v_cache[:, :, pos] = v1
        qq = self.keys(q1, v_cache.shape[-1])[:, :, None]
        kk, vv = k_cache[:, :, : pos + 1], v_cache[:, :, : pos + 1]
        return self.attend(qq, kk, vv, causal=False)[:, :, 0]


def candidates(device) -> list:
    """Every (backend, form) the comparator may run on this device."""
    if device.type != "cuda":
        return [SoftmaxAttention(SDPBackend.MATH, p) for p in (False, True)]
    return [SoftmaxAttention(b, p) for b in FAST_BACKENDS for p in (False, True)]


def select(q, k, v, causal: bool = True, reps: int = 5):
    """The fastest comparator for these inputs ([B, H, L, *] queries against
    [B, H, S, *] keys and values on CUDA; causal for a prefill, not causal for
    the single query of a decode step) among the library's fast backends,
    unpadded and padded, each timed with CUDA events on the current stream
    (median of `reps` calls after one untimed call). Returns (comparator,
    {name: ms or the refusal}). Backends that refuse the shapes or dtype are
    skipped; ValueError if none takes them."""
    d_v = v.shape[-1]
    stream = torch.cuda.current_stream(q.device)
    tried, best, best_ms = {}, None, float("inf")
    for c in candidates(q.device):
        qq, kk = c.keys(q, d_v), c.keys(k, d_v)
        try:
            with warnings.catch_warnings():   # a refusal is expected here, not news
                warnings.simplefilter("ignore", UserWarning)
                c.attend(qq, kk, v, causal)
            torch.cuda.synchronize(q.device)
        except RuntimeError as e:
            tried[c.name] = f"refused: {str(e).splitlines()[0][:80]}"
            continue
        evs = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            c.attend(qq, kk, v, causal)
            b.record(stream)
            evs.append((a, b))
        torch.cuda.synchronize(q.device)
        ms = statistics.median(a.elapsed_time(b) for a, b in evs)
        tried[c.name] = round(ms, 4)
        if ms < best_ms:
            best, best_ms = c, ms
        del qq, kk
    if best is None:
        raise ValueError(f"no softmax attention backend takes these inputs: {tried}")
    return best, tried
