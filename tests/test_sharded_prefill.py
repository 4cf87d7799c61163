"""The sequence-sharded prefill's host logic on CPU ranks (gloo): segments in
rank order, the all-gather of the segment sums, each rank's prefix, and the
final state every rank ends with. The per-rank arithmetic here is the
float64 oracle (the library's own kernels need a GPU; the GPU test of the same
routine is tests/test_gpu_sharded.py): the sharded result must equal the
oracle run on the whole sequence."""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from fixed_state_recurrence_phi_b300.sharded import shard_bounds  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class OracleOps:
    """The sharded prefill's steps done by the oracle on [B, H, n, d] float64
    tensors, states in the oracle's layout [B, H, D, d_v + 1]."""

    def __init__(self, n_terms):
        from oracle import tsa_oracle as O
        self.O, self.n = O, n_terms

    def new_states(self, cfg, like):
        return torch.zeros_like(like)

    def segment_sum(self, cfg, n, k, v, states):
        for b in range(k.shape[0]):
            for h in range(k.shape[1]):
                S = self.O.chunk_states(k[b, h].numpy(), v[b, h].numpy(), self.n, n)[0]
                states[b, h] = torch.from_numpy(S)

    def prefill(self, cfg, n, q, k, v, out, states, accumulate):
        for b in range(q.shape[0]):
            for h in range(q.shape[1]):
                S0 = states[b, h].numpy() if accumulate else None
                o, S = self.O.prefill_recurrent(q[b, h].numpy(), k[b, h].numpy(), v[b, h].numpy(), self.n, S0=S0)
                if n:
                    out[b, h] = torch.from_numpy(o)
                states[b, h] = torch.from_numpy(S)

    def merge(self, cfg, a, b):
        a += b

    def zero(self, cfg, states):
        states.zero_()


def _inputs(B, H, N, d, dv, seed):
    from fixed_state_recurrence_phi_b300.inputs import np_qkv
    q = np.zeros((B, H, N, d)); k = np.zeros((B, H, N, d)); v = np.zeros((B, H, N, dv))
    for b in range(B):
        for h in range(H):
            q[b, h], k[b, h], v[b, h] = np_qkv(N, d, dv, seed=[seed, b, h])
    return q, k, v


def _rank_main(rank, ws, port, N, n_pre, result_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        from fixed_state_recurrence_phi_b300.sharded import sharded_prefill
        from oracle import tsa_oracle as O
        B, H, d, dv, n = 1, 2, 4, 3, 3
        q, k, v = _inputs(B, H, n_pre + N, d, dv, seed=77)
        D = O.feature_dim(d, n)
        S0 = torch.zeros((B, H, D, dv + 1), dtype=torch.float64)
        for b in range(B):
            for h in range(H):   # the state before the sharded sequence: a prefix of n_pre tokens
                _, S = O.prefill_recurrent(q[b, h, :n_pre], k[b, h, :n_pre], v[b, h, :n_pre], n)
                S0[b, h] = torch.from_numpy(S)
        a, e = shard_bounds(N, ws, rank)
        seg = lambda x: torch.from_numpy(np.ascontiguousarray(x[:, :, n_pre + a:n_pre + e]))
        qs, ks, vs = seg(q), seg(k), seg(v)
        out = torch.zeros((B, H, e - a, dv), dtype=torch.float64)
        st = S0.clone()
        sharded_prefill(None, qs, ks, vs, out, st, accumulate=n_pre > 0, ops=OracleOps(n))
        worst_o = worst_s = 0.0
        for b in range(B):
            for h in range(H):
                o_ref, S_ref = O.prefill_recurrent(q[b, h], k[b, h], v[b, h], n)
                if e > a:
                    worst_o = max(worst_o, float(np.abs(out[b, h].numpy() - o_ref[n_pre + a:n_pre + e]).max()))
                worst_s = max(worst_s, float(np.abs(st[b, h].numpy() - S_ref).max() / np.abs(S_ref).max()))
        with open(os.path.join(result_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{worst_o} {worst_s}")
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("ws,N,n_pre", [(2, 300, 0), (2, 257, 40), (3, 2, 10)])
def test_sharded_prefill_equals_whole_sequence(ws, N, n_pre, tmp_path):
    mp.start_processes(_rank_main, args=(ws, _free_port(), N, n_pre, str(tmp_path)), nprocs=ws,
                       start_method="spawn", join=True)
    for r in range(ws):
        worst_o, worst_s = map(float, open(tmp_path / f"r{r}.txt").read().split())
        assert worst_o <= 1e-12, (r, worst_o)
        assert worst_s <= 1e-12, (r, worst_s)


def test_shard_bounds_cover_in_order():
    for N in (0, 1, 5, 128, 1001):
        for ws in (1, 2, 3, 8):
            spans = [shard_bounds(N, ws, r) for r in range(ws)]
            assert spans[0][0] == 0 and spans[-1][1] == N
            assert all(spans[i][1] == spans[i + 1][0] for i in range(ws - 1))
            lens = [e - a for a, e in spans]
            assert max(lens) - min(lens) <= 1
    with pytest.raises(ValueError):
        shard_bounds(10, 2, 2)
