"""Order 4 (n = 5 Taylor terms) at d_k = 16: 4,845 features, a 1.26 MB state
per head at d_v = 64, which the CUDA-core kernels keep in global memory (in
place in the caller's state, or in each span's scratch slot). Every head
against the float64 oracle: one span and several, fp32 and bf16, d_v 32 and
64, from zero and continuing a prefix, ragged tails, the states-only call,
decode steps, and the padding rows staying zero."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def G():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from fixed_state_recurrence_phi_b300 import build
    build.build()
    import gpu_helpers
    return gpu_helpers


def _sl(x, a, b):
    return x[:, :, a:b].contiguous()


@pytest.mark.parametrize("dtype,dv,N", [("f32", 64, 300), ("bf16", 64, 300), ("f32", 32, 70),
                                        ("f32", 64, 1), ("bf16", 32, 129)])
def test_order5_prefill_every_head(G, dtype, dv, N):
    T, O = G.T, G.O
    cfg = T.Config(1, 2, 16, dv, 5, dtype)
    plan = T.prefill_plan(cfg, N)
    assert plan["path"] == T.TSA_PATH_SIMT and plan["n_slices"] == 1
    q, k, v = G.make_inputs(cfg, N, seed=500 + dv + N)
    out, st = G.gpu_prefill(cfg, q, k, v)
    og, Sg = G.host(out), G.canonical(cfg, st)
    qh, kh, vh = G.host(q), G.host(k), G.host(v)
    for h in range(2):
        o_r, S_r = O.prefill_recurrent(qh[0, h], kh[0, h], vh[0, h], 5)
        G.check_head(cfg, og[0, h], Sg[0, h], o_r, S_r, G.TOL[dtype], f"n5 {dtype} dv{dv} N{N} h{h}")


def test_order5_several_spans_and_accumulate(G):
    """A prefix of 129 tokens, then 520 more continuing it (several spans:
    the span pass, the scan over the span slots and the output pass all run
    on the global state)."""
    T, O = G.T, G.O
    cfg = T.Config(1, 3, 16, 64, 5, "f32")
    P, L = 129, 520
    assert T.prefill_plan(cfg, L)["n_spans"] > 1
    q, k, v = G.make_inputs(cfg, P + L, seed=531)
    _, st = G.gpu_prefill(cfg, _sl(q, 0, P), _sl(k, 0, P), _sl(v, 0, P))
    out, st = G.gpu_prefill(cfg, _sl(q, P, P + L), _sl(k, P, P + L), _sl(v, P, P + L), states=st,
                            accumulate=True)
    og, Sg = G.host(out), G.canonical(cfg, st)
    qh, kh, vh = G.host(q), G.host(k), G.host(v)
    for h in range(3):
        o_r, S_r = O.prefill_recurrent(qh[0, h], kh[0, h], vh[0, h], 5)
        G.check_head(cfg, og[0, h], Sg[0, h], o_r[P:], S_r, G.TOL["f32"], f"n5 acc h{h}")
    # the padding rows of the state stay exactly zero
    D, Dp = T.feature_dim(16, 5), T.state_pad_dim(16, 5)
    s3 = st.view(3, Dp * 65)
    assert torch.count_nonzero(s3[:, :Dp * 64].view(3, Dp, 64)[:, D:]) == 0
    assert torch.count_nonzero(s3[:, Dp * 64:][:, D:]) == 0


def test_order5_states_only_and_decode(G):
    T, O = G.T, G.O
    cfg = T.Config(2, 2, 16, 64, 5, "bf16")
    N, steps = 400, 6
    q, k, v = G.make_inputs(cfg, N + steps, seed=532)
    _, st = G.gpu_prefill(cfg, _sl(q, 0, N), _sl(k, 0, N), _sl(v, 0, N))
    st2 = T.new_states(cfg)
    T.prefill_states(cfg, N, _sl(k, 0, N), _sl(v, 0, N), st2)
    torch.cuda.synchronize()
    assert G.rel_err(G.canonical(cfg, st2), G.canonical(cfg, st)) <= 1e-5
    outs = []
    for t in range(N, N + steps):
        o1 = torch.empty((2, 2, 64), dtype=q.dtype, device="cuda")
        T.decode_step(cfg, q[:, :, t].contiguous(), k[:, :, t].contiguous(), v[:, :, t].contiguous(), o1, st)
        outs.append(G.host(o1))
    T.sync_status()
    qh, kh, vh = G.host(q), G.host(k), G.host(v)
    Sg = G.canonical(cfg, st)
    for b in range(2):
        for h in range(2):
            o_r, S_r = O.prefill_recurrent(qh[b, h], kh[b, h], vh[b, h], 5)
            got = np.stack([o[b, h] for o in outs])
            G.check_head(cfg, got, Sg[b, h], o_r[N:], S_r, G.TOL["bf16"], f"n5 decode ({b},{h})")
