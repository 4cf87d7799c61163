"""Shared pieces of the GPU parity tests: running the CUDA path through the C
ABI, running the oracle on host copies of the same inputs, and the error
measure.

Tolerance (stated with the workloads): normwise relative error per (b, h) head,
max|gpu - oracle| / max|oracle|, at most 1e-4 for fp32 inputs and 2e-2 for bf16
inputs (fp32 accumulation and fp32 states either way).
"""
from __future__ import annotations

import numpy as np
import torch

from fixed_state_recurrence_phi_b300 import tsa as T
from fixed_state_recurrence_phi_b300.inputs import torch_qkv
from oracle import tsa_oracle as O

TOL = {"f32": 1e-4, "bf16": 2e-2}


def rel_err(g, r) -> float:
    g = np.asarray(g, np.float64); r = np.asarray(r, np.float64)
    den = np.abs(r).max()
    return float(np.abs(g - r).max() / (den if den > 0 else 1.0))


def host(x) -> np.ndarray:
    return x.detach().float().cpu().numpy().astype(np.float64)


def gpu_prefill(cfg, q, k, v, states=None, accumulate=False):
    """Run tsa_prefill on device tensors; returns (out, states)."""
    N = q.shape[2]
    out = torch.empty((cfg.B, cfg.H, N, cfg.d_v), dtype=q.dtype, device=q.device)
    if states is None:
        states = T.new_states(cfg, q.device)
    T.prefill(cfg, N, q, k, v, out, states, accumulate=accumulate)
    T.sync_status()   # a kernel that gave up on a wait reports it here
    return out, states


def canonical(cfg, states) -> np.ndarray:
    return host(T.canonical_states(cfg, states))


def check_head(cfg, out_g, S_g, out_r, S_r, tol, what=""):
    """Compare one head's outputs and state (value part and normaliser column
    separately, each normwise)."""
    dv = cfg.d_v
    e_out = rel_err(out_g, out_r)
    e_S = rel_err(S_g[:, :dv], S_r[:, :dv])
    e_z = rel_err(S_g[:, dv], S_r[:, dv])
    assert e_out <= tol, f"{what} out err {e_out:.3e} > {tol}"
    assert e_S <= tol, f"{what} state err {e_S:.3e} > {tol}"
    assert e_z <= tol, f"{what} normaliser err {e_z:.3e} > {tol}"
    return e_out, e_S, e_z


def make_inputs(cfg, N, seed, phase=0, device="cuda"):
    return torch_qkv(cfg.B, cfg.H, N, cfg.d_k, cfg.d_v, cfg.dtype, seed, phase, device)


def sample_heads(B, H, k=2, seed=0):
    heads = {(0, 0), (B - 1, H - 1)}
    rng = np.random.default_rng(seed)
    while len(heads) < min(B * H, 2 + k):
        heads.add((int(rng.integers(B)), int(rng.integers(H))))
    return sorted(heads)


def oracle_prefill(q, k, v, n, S0=None, chunked=None):
    """Oracle prefill for one head; the chunked form (pinned equal to the
    recurrent one) is used for long sequences to keep the run short."""
    if chunked:
        return O.prefill_chunked(q, k, v, n, chunked, S0=S0)
    return O.prefill_recurrent(q, k, v, n, S0=S0)
