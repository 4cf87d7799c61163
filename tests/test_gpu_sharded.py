"""The state sum of a segment (tsa_prefill_states) and the sequence-sharded
prefill built on it, against the float64 oracle.

tsa_prefill_states is checked on every path's span pass (fp32 split-operand
tensor cores, bf16 value-sliced tensor cores, CUDA cores), from zero and
added to existing states. The sharded prefill runs as two processes that
share this machine's one GPU for their kernels and exchange the segment sums
over gloo (through host memory): every rank's outputs and the final state
must match the oracle on the whole sequence. The kernels of the two processes
never wait on each other; the only exchange is the host-side all-gather."""
import os
import socket
import sys

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def G():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fixed_state_recurrence_phi_b300 import build
    build.build()
    import gpu_helpers
    return gpu_helpers


@pytest.mark.parametrize("d,dv,n,dtype,N", [
    (16, 64, 3, "f32", 1000),    # fp32 tensor-core span pass
    (16, 64, 4, "bf16", 700),    # bf16, value slices (the shape the CTA-pair prefill takes)
    (32, 128, 3, "bf16", 300),
    (16, 64, 4, "f32", 333),     # CUDA-core span pass
    (16, 32, 2, "bf16", 5),
])
def test_prefill_states_matches_oracle(G, d, dv, n, dtype, N):
    T, O = G.T, G.O
    cfg = T.Config(1, 3, d, dv, n, dtype)
    q, k, v = G.make_inputs(cfg, N + 50, seed=600 + d + dv + n)
    sl = lambda x, a, b: x[:, :, a:b].contiguous()
    tol = G.TOL[dtype]
    # from zero
    st = T.new_states(cfg)
    st.fill_(7.0)
    T.prefill_states(cfg, N, sl(k, 50, N + 50), sl(v, 50, N + 50), st)
    T.sync_status()
    Sg = G.canonical(cfg, st)
    kh, vh, qh = G.host(k), G.host(v), G.host(q)
    for h in range(3):
        S_r = O.chunk_states(kh[0, h, 50:], vh[0, h, 50:], n, N)[0]
        assert G.rel_err(Sg[0, h][:, :dv], S_r[:, :dv]) <= tol, h
        assert G.rel_err(Sg[0, h][:, dv], S_r[:, dv]) <= tol, h
    # added to the state of a 50-token prefix (from a prefill)
    _, st2 = G.gpu_prefill(cfg, sl(q, 0, 50), sl(k, 0, 50), sl(v, 0, 50))
    T.prefill_states(cfg, N, sl(k, 50, N + 50), sl(v, 50, N + 50), st2, accumulate=True)
    T.sync_status()
    Sg2 = G.canonical(cfg, st2)
    for h in range(3):
        _, S_r = O.prefill_recurrent(qh[0, h], kh[0, h], vh[0, h], n)
        assert G.rel_err(Sg2[0, h][:, :dv], S_r[:, :dv]) <= tol, h
        assert G.rel_err(Sg2[0, h][:, dv], S_r[:, dv]) <= tol, h


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, shape, result_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    torch.cuda.set_device(0)
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        import gpu_helpers as G
        from fixed_state_recurrence_phi_b300.sharded import shard_bounds, sharded_prefill
        T, O = G.T, G.O
        B, H, d, dv, n, dtype, N = shape
        cfg = T.Config(B, H, d, dv, n, dtype)
        q, k, v = G.make_inputs(cfg, N, seed=41)        # the whole sequence, the same on every rank
        a, e = shard_bounds(N, ws, rank)
        sl = lambda x: x[:, :, a:e].contiguous()
        out = torch.empty((B, H, e - a, dv), dtype=q.dtype, device="cuda")
        st = T.new_states(cfg)
        sharded_prefill(cfg, sl(q), sl(k), sl(v), out, st)
        T.sync_status()
        Sg = G.canonical(cfg, st)
        og = G.host(out)
        qh, kh, vh = G.host(q), G.host(k), G.host(v)
        worst = 0.0
        for b in range(B):
            for h in range(H):
                o_r, S_r = O.prefill_recurrent(qh[b, h], kh[b, h], vh[b, h], n)
                e_o, e_s, e_z = G.check_head(cfg, og[b, h], Sg[b, h], o_r[a:e], S_r, G.TOL[dtype],
                                             f"rank {rank} head {(b, h)}")
                worst = max(worst, e_o, e_s, e_z)
        with open(os.path.join(result_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"ok {worst}")
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("shape", [
    (1, 4, 16, 64, 3, "f32", 1500),
    (1, 2, 16, 64, 4, "bf16", 900),
])
def test_sharded_prefill_two_processes(G, shape, tmp_path):
    mp.start_processes(_rank_main, args=(2, _free_port(), shape, str(tmp_path)), nprocs=2,
                       start_method="spawn", join=True)
    for r in range(2):
        assert open(tmp_path / f"r{r}.txt").read().startswith("ok"), r
