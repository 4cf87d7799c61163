"""Seeded synthetic inputs and the named workloads.

This module is shared by the tests, the benchmark and the smoke check. It holds
no arithmetic of the attention method itself: it only draws Gaussian rows,
scales q and k rows to unit length (the caller-side precondition the pages
state: query/key normalisation keeps the Taylor argument |q.k| <= 1) and rounds
to the storage dtype.

Recipe (all workloads): q, k rows ~ N(0, I_d) scaled to unit L2 norm; v ~ N(0, 1);
generated in float32, then rounded to the workload's dtype (round-to-nearest-even
for bfloat16). Both the CUDA path and the oracle consume the rounded values.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d_k: int
    d_v: int
    n_terms: int
    dtype: str          # "f32" or "bf16"
    decode_steps: int
    seed: int


# The five workloads: a single-head parity case, the 8192-token prefill point,
# long-context decode, a fourth-order case and a wide head.
WORKLOADS = {
    "single_head_N256": Workload("single_head_N256", 1, 1, 256, 16, 64, 3, "f32", 64, 0),
    "prefill_B1_H8_N8192": Workload("prefill_B1_H8_N8192", 1, 8, 8192, 16, 64, 3, "f32", 0, 2),
    "decode_B64_H16_N65536": Workload("decode_B64_H16_N65536", 64, 16, 65536, 16, 64, 3, "bf16", 1024, 3),
    "order4_B4_H16_N32768": Workload("order4_B4_H16_N32768", 4, 16, 32768, 16, 64, 4, "bf16", 256, 4),
    "wide_B2_H32_N65536": Workload("wide_B2_H32_N65536", 2, 32, 65536, 32, 128, 3, "bf16", 0, 5),
}


def _mix(*parts: int) -> int:
    """Deterministic 63-bit seed from a tuple of small integers (splitmix64)."""
    h = 0x9E3779B97F4A7C15
    for p in parts:
        h = (h ^ (p & 0xFFFFFFFFFFFFFFFF)) & 0xFFFFFFFFFFFFFFFF
        h = (h + 0x9E3779B97F4A7C15) & 0xFFFFFFFFFFFFFFFF
        z = h
        z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & 0xFFFFFFFFFFFFFFFF
        z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & 0xFFFFFFFFFFFFFFFF
        h = z ^ (z >> 31)
    return h & 0x7FFFFFFFFFFFFFFF


def np_qkv(N: int, d_k: int, d_v: int, seed, dtype=np.float64):
    """Host (numpy) inputs for one head: unit q, k rows and Gaussian v."""
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((N, d_k))
    k = rng.standard_normal((N, d_k))
    v = rng.standard_normal((N, d_v))
    q /= np.linalg.norm(q, axis=1, keepdims=True)
    k /= np.linalg.norm(k, axis=1, keepdims=True)
    return q.astype(dtype), k.astype(dtype), v.astype(dtype)


def torch_qkv(B: int, H: int, N: int, d_k: int, d_v: int, dtype: str, seed: int,
              phase: int = 0, device="cpu"):
    """Inputs [B, H, N, d] on `device`, drawn with a seeded torch generator in
    float32 (per batch row, to bound temporaries), q/k rows unit-normalised,
    then rounded to `dtype` ("f32" or "bf16")."""
    import torch
    tdt = {"f32": torch.float32, "bf16": torch.bfloat16}[dtype]
    g = torch.Generator(device=device)
    q = torch.empty((B, H, N, d_k), dtype=tdt, device=device)
    k = torch.empty((B, H, N, d_k), dtype=tdt, device=device)
    v = torch.empty((B, H, N, d_v), dtype=tdt, device=device)
    for b in range(B):
        g.manual_seed(_mix(seed, phase, b))
        qb = torch.randn((H, N, d_k), generator=g, device=device, dtype=torch.float32)
        kb = torch.randn((H, N, d_k), generator=g, device=device, dtype=torch.float32)
        vb = torch.randn((H, N, d_v), generator=g, device=device, dtype=torch.float32)
        qb = qb / torch.linalg.vector_norm(qb, dim=-1, keepdim=True)
        kb = kb / torch.linalg.vector_norm(kb, dim=-1, keepdim=True)
        q[b].copy_(qb); k[b].copy_(kb); v[b].copy_(vb)
        del qb, kb, vb
    return q, k, v
