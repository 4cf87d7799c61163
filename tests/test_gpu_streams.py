"""Kernels of different paths running at once on two CUDA streams: the bf16
append form (three CTAs per SM, 128 TMEM columns each) on one, the fp32
three-launch prefill (span pass, scan, output pass with programmatic launch
dependencies, 512 TMEM columns a CTA) on the other, so that their CTAs share
SMs and contend for tensor memory. Every result must be bitwise the one the
same call gives alone (the kernels are deterministic), and the concurrent
results are also checked against the oracle on sampled heads."""
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


def test_append_form_and_fp32_prefill_on_two_streams(G):
    T, O = G.T, G.O
    sl = lambda x, a, b: x[:, :, a:b].contiguous()
    # stream A: 32-token appends to 512 bf16 heads that continue a 200-token prefix
    ca = T.Config(16, 32, 16, 64, 3, "bf16")
    P, L = 200, 32
    qa, ka, va = G.make_inputs(ca, P + L, seed=801)
    _, st0 = G.gpu_prefill(ca, sl(qa, 0, P), sl(ka, 0, P), sl(va, 0, P))
    assert T.prefill_plan(ca, L)["ctas_per_sm"] == 3
    aq, ak, av = sl(qa, P, P + L), sl(ka, P, P + L), sl(va, P, P + L)
    # stream B: the 8-head 8192-token fp32 prefill (several spans)
    cb = T.Config(1, 8, 16, 64, 3, "f32")
    N = 8192
    assert T.prefill_plan(cb, N)["n_spans"] > 1
    qb, kb, vb = G.make_inputs(cb, N, seed=802)

    # alone, on the current stream
    ref_oa, ref_sa = G.gpu_prefill(ca, aq, ak, av, states=st0.clone(), accumulate=True)
    ref_ob, ref_sb = G.gpu_prefill(cb, qb, kb, vb)

    # at once: several calls on each stream, interleaved in issue order
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    sa.wait_stream(torch.cuda.current_stream())
    sb.wait_stream(torch.cuda.current_stream())
    reps = 6
    outs_a = [torch.empty_like(ref_oa) for _ in range(reps)]
    sts_a = [st0.clone() for _ in range(reps)]
    outs_b = [torch.empty_like(ref_ob) for _ in range(reps)]
    sts_b = [T.new_states(cb) for _ in range(reps)]
    torch.cuda.synchronize()
    for r in range(reps):
        T.prefill(cb, N, qb, kb, vb, outs_b[r], sts_b[r], stream=sb)
        T.prefill(ca, L, aq, ak, av, outs_a[r], sts_a[r], accumulate=True, stream=sa)
    torch.cuda.synchronize()
    T.sync_status()
    for r in range(reps):
        assert torch.equal(outs_a[r], ref_oa) and torch.equal(sts_a[r], ref_sa), r
        assert torch.equal(outs_b[r], ref_ob) and torch.equal(sts_b[r], ref_sb), r

    # and the concurrent results against the oracle on sampled heads
    Sa, oa = G.canonical(ca, sts_a[-1]), G.host(outs_a[-1])
    qh, kh, vh = G.host(qa), G.host(ka), G.host(va)
    for b, h in G.sample_heads(16, 32, k=2, seed=3):
        o_r, S_r = O.prefill_recurrent(qh[b, h], kh[b, h], vh[b, h], 3)
        G.check_head(ca, oa[b, h], Sa[b, h], o_r[P:], S_r, G.TOL["bf16"], f"append ({b},{h})")
    Sb, ob = G.canonical(cb, sts_b[-1]), G.host(outs_b[-1])
    qh, kh, vh = G.host(qb), G.host(kb), G.host(vb)
    for h in (0, 7):
        o_r, S_r = G.oracle_prefill(qh[0, h], kh[0, h], vh[0, h], 3, chunked=128)
        G.check_head(cb, ob[0, h], Sb[0, h], o_r, S_r, G.TOL["f32"], f"fp32 head {h}")
